#!/usr/bin/env python
"""Benchmark: paged decode attention (append + decode per layer) on one GB300.

Workload (default): the mixed batch -- 32 rows, 31 lengths uniform on
16..512 plus one 4096-token row, 64-token blocks, 12 query / 2 KV heads,
head_dim 128, fp16, 28 layers each with its own pool, shuffled physical
blocks, seed 0.  One step = for every layer, append the row's new token into
its slot, then decode attention over the row's true length.  The step is one
CUDA graph of 56 launches.

Prints one JSON line (rank 0).  ``value`` is algorithmic bytes per step
(KV + q + out + table + seq_lens + appended tokens) / device time per step,
in GB/s.  ``roofline`` is for the decode kernel alone (a graph of 28 decode
launches timed the same way) against the measured HBM copy bandwidth.
``e2e`` repeats the step through the public API with the step's inputs copied
from pinned host memory (one packed buffer, one copy) and the outputs copied
back inside the timed region.
``cpu_baseline`` times the fp64 oracle on a bounded sample on the host cores.

--impl reference times the oracle itself as the reference arm (rank 0 only).
Multi-GPU runs (torchrun) are independent replicas: every rank runs the same
workload on its own GPU (weak scaling), no collective on the data path.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "decode-attention KV GB/s and % of HBM roofline; rows·layers/s at batch 32"
FALLBACK_HBM_GBS = 6800.0
CPU_SAMPLE_SECONDS = 10.0  # the oracle's timed sample: layer passes until this much time
REFERENCE_STEP_LAYERS = 4  # reference arm: layers of the workload per timed step


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=["mixed", "uniform", "shared", "long", "tiny"],
                    default="mixed")
    ap.add_argument("--layers", type=int, default=28)
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-comparator", action="store_true")
    ap.add_argument("--no-configs", action="store_true",
                    help="skip the per-config lines (tiny, uniform, shared, long)")
    return ap.parse_args()


# ---------------------------------------------------------------------------
# distributed plumbing (replicas only)

def dist_setup(args):
    import torch
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    pg = None
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
        pg = dist
    elif torch.cuda.is_available():
        torch.cuda.set_device(0)
    return rank, world, pg


def barrier(pg):
    if pg is not None:
        pg.barrier()


def max_over_ranks(pg, x: float) -> float:
    if pg is None:
        return x
    import torch
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    pg.all_reduce(t, op=pg.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(pg, x: float) -> float:
    if pg is None:
        return x
    import torch
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    pg.all_reduce(t, op=pg.ReduceOp.SUM)
    return float(t.item())


# ---------------------------------------------------------------------------
# clocks during the timed region

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.15)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return None
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        smax = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        power = [float(r[3]) for r in rows if r[3].replace(".", "").isdigit()]
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": reasons, "samples": len(rows),
                "power_w_max": max(power) if power else None}


# ---------------------------------------------------------------------------

def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        try:
            d = json.load(open(p))
            return float(d["hbm_gbs"]), "measured"
        except (KeyError, ValueError):
            pass
    return FALLBACK_HBM_GBS, "fallback"


def load_tensor_peak():
    """Dense fp16/bf16 tensor peak: the measured cuBLAS bf16 burst figure (the
    fp16 rate is the same on this part), else the recipe's fallback."""
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            m = json.load(f)
        v = m.get("bf16_tflops")
        if v:
            return float(v), "measured (bf16 burst)"
    except (OSError, ValueError):
        pass
    return 1900.0, "fallback"


def decode_source_hash() -> str:
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "paged_kv_cache_06_gb300", "csrc")
    for name in sorted(os.listdir(csrc)):
        if (name.startswith("decode") and name.endswith((".cu", ".cuh"))) or \
                name in ("ptx.cuh", "pkv_internal.cuh", "tmap.cu", "fp8_codec.cuh"):
            h.update(open(os.path.join(csrc, name), "rb").read())
    return h.hexdigest()[:16]


def load_traffic(workload: str):
    """dram bytes per decode launch from a committed ncu summary, only if it was
    taken on the current decode kernel source."""
    p = os.path.join(ROOT, "profiles", f"decode_{workload}_traffic.json")
    if not os.path.exists(p):
        return None
    try:
        d = json.load(open(p))
    except ValueError:
        return None
    if d.get("decode_source_hash") != decode_source_hash():
        return None
    return d.get("dram_bytes_per_launch")


def make_case(args):
    from paged_kv_cache_06_gb300 import workloads as wl
    if args.workload == "mixed":
        return wl.mixed(seed=args.seed, layers=args.layers)
    if args.workload == "uniform":
        return wl.uniform(seed=args.seed, layers=args.layers)
    return wl.WORKLOADS[args.workload](seed=args.seed)


CONFIG_DESC = {
    "tiny": "4 rows of 1 / 17 / 64 / 200 tokens, 16-token blocks, one append per row",
    "uniform": "32 rows x 1024 tokens, 64-token blocks",
    "mixed": "31 rows U{16..512} + 1 row of 4096, 64-token blocks",
    "shared": "96 rows log-uniform on [16, 8192], 16-token blocks, the first 592 tokens "
              "(37 blocks) shared by every row",
    "long": "4 rows x 32769 tokens (one append at 32768), 64-token blocks",
    "uniform_fp8": "uniform, FP8 (E4M3) pools with one scale per KV head",
    "long_fp8": "long, FP8 (E4M3) pools with one scale per KV head",
}


def workload_config(case, args):
    from paged_kv_cache_06_gb300 import workloads as wl
    b = wl.algorithmic_bytes(case)
    desc = CONFIG_DESC[args.workload]
    return {
        "workload": args.workload, "rows": case.rows, "layers": case.layers,
        "lengths": desc, "tokens_per_layer": int(case.seq_lens.sum()),
        "block_size": case.block_size, "q_heads": case.q_heads, "kv_heads": case.kv_heads,
        "head_dim": case.head_dim, "seed": args.seed,
        "step": "per layer: paged_attention_append_decode (append + decode, one launch, PDL); "
                "the step is one CUDA graph",
        "bytes_per_step": case.layers * (b["decode_layer"] + b["append_layer"]),
        "l2": f"inputs larger than L2: {case.layers * b['kv_logical'] / 1e6:.0f} MB of KV per step "
              "vs 129 MB L2, each layer its own pool",
        "parallelism": "replicas",
    }


def cpu_oracle_sample(case, seconds: float = CPU_SAMPLE_SECONDS, threads: int = 0):
    """Time the fp64 oracle (append + decode) on whole layers of the workload,
    cycling through its layers until ``seconds`` have passed; ``threads`` 0
    means every host core."""
    import oracle
    from paged_kv_cache_06_gb300 import workloads as wl
    threads = threads or oracle.default_threads()
    b = wl.algorithmic_bytes(case)
    t0 = time.perf_counter()
    passes = 0
    while True:
        l = passes % case.layers
        kp, vp = oracle.paged_append(case.k_pool[l], case.v_pool[l], case.block_tables,
                                     case.positions, case.k_new[l], case.v_new[l])
        oracle.paged_decode(case.q[l], kp, vp, case.block_tables, case.seq_lens, case.scale,
                            num_threads=threads)
        passes += 1
        dt = time.perf_counter() - t0
        if dt >= seconds:
            break
    nbytes = passes * (b["decode_layer"] + b["append_layer"])
    return nbytes / dt / 1e9, threads, dt, passes


# ---------------------------------------------------------------------------

def measure_configs(args, dev, peak, peak_kind):
    """Every workload configuration as its own timed step (fused append +
    decode per launch, programmatic dependent launch between launches, one
    CUDA graph).  Single-layer configurations are timed over several copies
    of their pool, one per launch, so that the step reads more than L2 holds
    (a real model's layers each have their own pool); the tiny one stays in
    L2 whatever the copies.  The shared-prefix roofline counts each distinct
    block once (a block that many rows read is served from L2 after its first
    read); its logical bytes are reported beside it."""
    import torch
    from paged_kv_cache_06_gb300 import ops
    from paged_kv_cache_06_gb300 import workloads as wl
    copies = {"tiny": 28, "uniform": 1, "shared": 4, "long": 4, "uniform_fp8": 1, "long_fp8": 4}
    out_cfg = {}
    for name in ("tiny", "uniform", "shared", "long", "uniform_fp8", "long_fp8"):
        fp8 = name.endswith("_fp8")
        base = name[:-4] if fp8 else name
        if base == "uniform":
            case = wl.uniform(seed=args.seed, layers=args.layers)
        else:
            case = wl.WORKLOADS[base](seed=args.seed)
        b = wl.algorithmic_bytes(case)
        if fp8:
            # E4M3 codes drawn like the pools' values (scales near 1/8)
            gen8 = torch.Generator().manual_seed(args.seed + 8)
            k8 = [torch.from_numpy(wl.fp8_codes(gen8, case.k_pool[l].shape)) for l in range(case.layers)]
            v8 = [torch.from_numpy(wl.fp8_codes(gen8, case.v_pool[l].shape)) for l in range(case.layers)]
        d = wl.to_device(case, dev)
        n = case.layers * copies[name]
        if fp8:
            del d["k_pool"], d["v_pool"]
            kp = [k8[l % case.layers].to(dev) for l in range(n)]
            vp = [v8[l % case.layers].to(dev) for l in range(n)]
            del k8, v8
        else:
            kp = [d["k_pool"][l % case.layers].clone() if copies[name] > 1 else d["k_pool"][l]
                  for l in range(n)]
            vp = [d["v_pool"][l % case.layers].clone() if copies[name] > 1 else d["v_pool"][l]
                  for l in range(n)]
            del d["k_pool"], d["v_pool"]
        rows, hq, hk, hd = case.rows, case.q_heads, case.kv_heads, case.head_dim
        ws = ops.alloc_workspace(rows, hq, hk, hd, case.max_seq_len, case.block_size, device=dev)
        out = torch.zeros(n, rows, hq, hd, dtype=torch.float16, device=dev)
        has_append = bool((case.positions >= 0).any())
        ks8 = torch.full((hk,), 0.12, dtype=torch.float32, device=dev)
        vs8 = torch.full((hk,), 0.12, dtype=torch.float32, device=dev)

        def step():
            # positions < 0 (the shared-prefix rows) append nothing
            for l in range(n):
                li = l % case.layers
                if fp8:
                    ops.append_decode_fp8(out[l], d["q"][li], kp[l], vp[l], ks8, vs8,
                                          d["block_tables"], d["seq_lens"], d["positions"],
                                          d["k_new"][li], d["v_new"][li], case.scale,
                                          case.max_seq_len, ws, pdl=True)
                else:
                    ops.append_decode(out[l], d["q"][li], kp[l], vp[l], d["block_tables"],
                                      d["seq_lens"], d["positions"], d["k_new"][li],
                                      d["v_new"][li], case.scale, case.max_seq_len, ws, pdl=True)

        step()
        torch.cuda.synchronize()
        s = torch.cuda.Stream(device=dev)
        s.wait_stream(torch.cuda.current_stream())
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(s):
            with torch.cuda.graph(g, stream=s):
                step()
        torch.cuda.current_stream().wait_stream(s)
        for _ in range(args.warmup):
            g.replay()
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(args.steps):
            g.replay()
        e1.record()
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1) / args.steps
        per_launch = ms * 1e-3 / n
        logical = b["decode_layer"] + b["append_layer"]
        unique = b["decode_layer_unique"] + b["append_layer"]
        if fp8:
            # one byte per cached element; the new token comes in as fp16 and goes out as codes
            n_app = int((case.positions >= 0).sum())
            logical = (b["kv_logical"] // 2 + b["q_out"] + b["table"]
                       + n_app * hk * hd * (2 + 1) * 2)
        roof_bytes = unique if name == "shared" else logical
        achieved = roof_bytes / per_launch / 1e9
        entry = {
            "workload": CONFIG_DESC[name], "rows": rows, "block_size": case.block_size,
            "launches_per_step": n, "ms_per_step": round(ms, 5),
            "us_per_launch": round(per_launch * 1e6, 3),
            "bytes_per_launch": roof_bytes,
            "GBps": round(achieved, 2),
            "rows_layers_per_s": round(rows * n / (ms * 1e-3), 1),
            "roofline": {"bound": "hbm", "achieved": round(achieved, 2), "peak": peak,
                         "unit": "GB/s", "frac": round(achieved / peak, 4),
                         "peak_source": peak_kind},
            "what": ("append + decode (one fused launch)" if has_append else "decode")
                    + (" over FP8 pools" if fp8 else "")
                    + (f", {copies[name]} pool copies" if copies[name] > 1 else ""),
        }
        if name == "shared":
            entry["kv_logical_bytes"] = b["kv_logical"]
            entry["kv_unique_bytes"] = b["kv_unique"]
            entry["GBps_logical"] = round(logical / per_launch / 1e9, 2)
        if name == "tiny":
            entry["note"] = "0.29 MB per launch: L2-resident; a launch-latency figure"
        if fp8 and base in out_cfg:
            # the same workload on fp16 pools: time and bandwidth ratios
            entry["vs_fp16"] = {"time_ratio": round(out_cfg[base]["us_per_launch"] / entry["us_per_launch"], 3),
                                "GBps_ratio": round(entry["GBps"] / out_cfg[base]["GBps"], 3)}
        out_cfg[name] = entry
        del g, kp, vp, d, out, ws
        torch.cuda.empty_cache()
    return out_cfg


def run_ours(args, rank, world, pg):
    import torch
    from paged_kv_cache_06_gb300 import ops
    from paged_kv_cache_06_gb300 import workloads as wl

    dev = torch.device("cuda", torch.cuda.current_device())
    ops.lib()  # fails loudly if the CUDA library cannot be built or loaded
    case = make_case(args)
    b = wl.algorithmic_bytes(case)
    d = wl.to_device(case, dev)
    # A step's inputs sit in one device buffer, as typed views 256-byte
    # aligned, so a caller moves them with one host-to-device copy.
    in_names = ("q", "k_new", "v_new", "block_tables", "seq_lens", "positions")
    in_bytes = [d[n].numel() * d[n].element_size() for n in in_names]
    packed = torch.empty(sum((n + 255) // 256 * 256 for n in in_bytes), dtype=torch.uint8, device=dev)
    off = 0
    for n, nb in zip(in_names, in_bytes):
        view = packed[off:off + nb].view(d[n].dtype).view(d[n].shape)
        view.copy_(d[n])
        d[n] = view
        off += (nb + 255) // 256 * 256
    L = case.layers
    rows, hq, hk, hd = case.rows, case.q_heads, case.kv_heads, case.head_dim
    msl = case.max_seq_len
    ws = ops.alloc_workspace(rows, hq, hk, hd, msl, case.block_size, device=dev)
    plan_buf = ops.alloc_plan(rows, hq, hk, hd, msl, case.block_size, device=dev)
    out = torch.zeros(L, rows, hq, hd, dtype=torch.float16, device=dev)

    def make_plan():
        ops.plan(plan_buf, d["block_tables"], d["seq_lens"], d["positions"], hq, hk, hd,
                 case.block_size, case.num_blocks, msl)

    def step():
        # One layer = one fused launch (append the new token, decode); each
        # block derives the step's split itself before its dependency wait,
        # and layers overlap through programmatic dependent launch.
        for l in range(L):
            ops.append_decode(out[l], d["q"][l], d["k_pool"][l], d["v_pool"][l],
                              d["block_tables"], d["seq_lens"], d["positions"], d["k_new"][l],
                              d["v_new"][l], case.scale, msl, ws, pdl=True)

    def step_planned():
        # The step's work split is planned once; then one fused launch per
        # layer, each overlapping the previous one through programmatic
        # dependent launch (the first follows the plan without it, since it
        # reads the plan early).
        make_plan()
        for l in range(L):
            ops.decode_planned(out[l], d["q"][l], d["k_pool"][l], d["v_pool"][l],
                               d["block_tables"], d["seq_lens"], case.scale, msl, plan_buf, ws,
                               positions=d["positions"], k_new=d["k_new"][l], v_new=d["v_new"][l],
                               pdl=l > 0)


    def step_unfused():
        for l in range(L):
            ops.append(d["k_pool"][l], d["v_pool"][l], d["block_tables"], d["positions"],
                       d["k_new"][l], d["v_new"][l])
            ops.decode(out[l], d["q"][l], d["k_pool"][l], d["v_pool"][l], d["block_tables"],
                       d["seq_lens"], case.scale, msl, ws)

    def decode_only():
        make_plan()
        for l in range(L):
            ops.decode_planned(out[l], d["q"][l], d["k_pool"][l], d["v_pool"][l],
                               d["block_tables"], d["seq_lens"], case.scale, msl, plan_buf, ws)

    def capture(fn):
        fn()  # eager warm-up (also validates arguments)
        torch.cuda.synchronize()
        s = torch.cuda.Stream(device=dev)
        s.wait_stream(torch.cuda.current_stream())
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(s):
            with torch.cuda.graph(g, stream=s):
                fn()
        torch.cuda.current_stream().wait_stream(s)
        torch.cuda.synchronize()
        return g

    def time_graph(g, k, w, clocks=None):
        for _ in range(w):
            g.replay()
        barrier(pg)
        torch.cuda.synchronize()
        if clocks:
            clocks.start()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(k):
            g.replay()
        e1.record()
        torch.cuda.synchronize()
        cl = clocks.stop() if clocks else None
        barrier(pg)
        return e0.elapsed_time(e1) / k, cl

    g_step = capture(step)
    clocks = ClockSampler(torch.cuda.current_device())
    ms_local, clk = time_graph(g_step, args.steps, args.warmup, clocks)
    ms = max_over_ranks(pg, ms_local)
    bytes_step = L * (b["decode_layer"] + b["append_layer"])
    total_bytes = sum_over_ranks(pg, bytes_step)
    value = total_bytes / (ms * 1e-3) / 1e9

    # The dominant kernel is the fused append+decode launch; the step is made
    # of nothing else, so its average launch time is the step time / layers.
    per_launch_s = ms * 1e-3 / L
    bytes_launch = b["decode_layer"] + b["append_layer"]
    achieved = bytes_launch / per_launch_s / 1e9
    peak, peak_kind = load_peaks()
    traffic = load_traffic(args.workload)
    # Same step without fusion or overlap, and the decode kernel alone.
    g_unf = capture(step_unfused)
    ms_unf, _ = time_graph(g_unf, args.steps, args.warmup)
    del g_unf
    g_pl = capture(step_planned)
    ms_pl, _ = time_graph(g_pl, args.steps, args.warmup)
    del g_pl
    g_dec = capture(decode_only)
    ms_dec, _ = time_graph(g_dec, args.steps, args.warmup)

    # The same step over FP8 (E4M3) pools with one scale per KV head: per
    # layer one fused launch (quantising append + FP8 decode) with PDL, and
    # for reference the two separate launches without PDL.
    gen8 = torch.Generator().manual_seed(args.seed + 8)
    kp8 = [torch.from_numpy(wl.fp8_codes(gen8, case.k_pool[l].shape)).to(dev) for l in range(L)]
    vp8 = [torch.from_numpy(wl.fp8_codes(gen8, case.v_pool[l].shape)).to(dev) for l in range(L)]
    ks8 = torch.full((hk,), 0.12, dtype=torch.float32, device=dev)
    vs8 = torch.full((hk,), 0.12, dtype=torch.float32, device=dev)

    def step_fp8():
        for l in range(L):
            ops.append_decode_fp8(out[l], d["q"][l], kp8[l], vp8[l], ks8, vs8, d["block_tables"],
                                  d["seq_lens"], d["positions"], d["k_new"][l], d["v_new"][l],
                                  case.scale, msl, ws, pdl=True)

    def step_fp8_unfused():
        for l in range(L):
            ops.append_fp8(kp8[l], vp8[l], ks8, vs8, d["block_tables"], d["positions"],
                           d["k_new"][l], d["v_new"][l])
            ops.decode_fp8(out[l], d["q"][l], kp8[l], vp8[l], ks8, vs8, d["block_tables"],
                           d["seq_lens"], case.scale, msl, ws)

    g8 = capture(step_fp8)
    ms8, _ = time_graph(g8, args.steps, args.warmup)
    del g8
    g8u = capture(step_fp8_unfused)
    ms8u, _ = time_graph(g8u, args.steps, args.warmup)
    del g8u, kp8, vp8

    # Chunked prefill: 8 rows whose newest 512 tokens (the pages' chunk size)
    # are the chunk, at 4096 tokens of context, one layer's pool.
    pcase = wl.custom([4096] * 8, 64, seed=args.seed + 3, layers=1, append=False, nan_fill=False)
    pd = wl.to_device(pcase, dev)
    pchunk = 512
    pqs = torch.arange(0, pchunk * (pcase.rows + 1), pchunk, dtype=torch.int32, device=dev)
    pgen = torch.Generator().manual_seed(args.seed + 4)
    pq = torch.randn(pcase.rows * pchunk, hq, hd, generator=pgen).to(torch.float16).to(dev)
    pout = torch.empty_like(pq)
    pws = ops.alloc_prefill_workspace(pcase.rows, hq, hk, hd, pcase.block_size, device=dev)

    def step_prefill():
        ops.prefill(pout, pq, pd["k_pool"][0], pd["v_pool"][0], pd["block_tables"],
                    pd["seq_lens"], pqs, pcase.scale, pcase.max_seq_len, workspace=pws)

    g_pf = capture(step_prefill)
    ms_pf, _ = time_graph(g_pf, args.steps, args.warmup)
    del g_pf
    # causal FLOPs: query i of a chunk sees (context - chunk + i + 1) keys;
    # 2 flops per multiply-add, QK^T and PV, every query head
    vis = sum(4096 - pchunk + i + 1 for i in range(pchunk))
    pf_flops = pcase.rows * hq * vis * hd * 2 * 2
    tf_peak, tf_kind = load_tensor_peak()
    n_app = int((case.positions >= 0).sum())
    bytes8 = (b["kv_logical"] // 2 + b["q_out"] + b["table"]
              + n_app * hk * hd * (2 + 1) * 2)  # append: fp16 in, one byte out, K and V

    result = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f16",
        "data": "synthetic (seeded N(0,1) fp16 values, seeded lengths and block permutation)",
        "config": workload_config(case, args),
        "rows_layers_per_s": round(world * rows * L / (ms * 1e-3), 1),
        "rows_heads_per_s": round(world * rows * hq * L / (ms * 1e-3), 1),
        "hbm_frac_of_measured": round(value / world / peak, 4),
        "hbm_frac_of_nominal_8TBs": round(value / world / 8000.0, 4),
        "roofline": {"bound": "hbm", "achieved": round(achieved, 2), "peak": peak,
                     "unit": "GB/s", "frac": round(achieved / peak, 4),
                     "traffic": traffic, "peak_source": peak_kind,
                     "kernel": "paged_attention_append_decode (fused, PDL)",
                     "bytes_per_launch": bytes_launch,
                     "launch_us": round(per_launch_s * 1e6, 3)},
        "planned_step": {"ms_per_step": round(ms_pl, 5),
                         "value": round(total_bytes / (ms_pl * 1e-3) / 1e9 if world == 1 else 0, 2),
                         "what": "paged_attention_plan once, then per layer "
                                 "paged_attention_decode_planned (fused append + decode, PDL "
                                 "from layer 1)"},
        "unfused_step": {"ms_per_step": round(ms_unf, 5),
                         "value": round(total_bytes / (ms_unf * 1e-3) / 1e9 if world == 1 else 0, 2),
                         "what": "per layer paged_kv_append + paged_attention_decode, no PDL"},
        "decode_only": {"ms_per_step": round(ms_dec, 5),
                        "us_per_launch": round(ms_dec * 1e3 / L, 3),
                        "GBps": round(b["decode_layer"] / (ms_dec * 1e-3 / L) / 1e9, 2)},
        "prefill": {"what": "paged_attention_prefill, 8 rows x 512-token chunk at 4096 context, "
                            "12 query / 2 KV heads, tcgen05 fp16 in / fp32 accumulate in TMEM",
                    "ms_per_launch": round(ms_pf, 5),
                    "prompt_tokens_per_s": round(pcase.rows * pchunk / (ms_pf * 1e-3), 1),
                    "roofline": {"bound": "tensor",
                                 "achieved": round(pf_flops / (ms_pf * 1e-3) / 1e12, 2),
                                 "peak": tf_peak, "unit": "TFLOP/s",
                                 "frac": round(pf_flops / (ms_pf * 1e-3) / 1e12 / tf_peak, 4),
                                 "peak_source": tf_kind, "flops_per_launch": pf_flops}},
        "fp8_step": {"ms_per_step": round(ms8, 5),
                     "value": round(L * bytes8 / (ms8 * 1e-3) / 1e9, 2), "unit": "GB/s",
                     "bytes_per_layer": bytes8,
                     "what": "per layer paged_attention_append_decode_fp8 with PDL "
                             "(E4M3 pools, one scale per KV head)",
                     "unfused_ms_per_step": round(ms8u, 5),
                     "unfused_what": "per layer paged_kv_append_fp8 + paged_attention_decode_fp8, "
                                     "no PDL"},
        "gpu_launches": args.steps * L,
        "clocks": clk,
    }

    if not args.no_configs and args.workload == "mixed":
        cfgs = measure_configs(args, dev, peak, peak_kind)
        cfgs["mixed"] = {"workload": CONFIG_DESC["mixed"], "rows": rows, "block_size": case.block_size,
                         "launches_per_step": L, "ms_per_step": round(ms, 5),
                         "us_per_launch": round(per_launch_s * 1e6, 3),
                         "bytes_per_launch": bytes_launch, "GBps": round(achieved, 2),
                         "roofline": {"bound": "hbm", "achieved": round(achieved, 2), "peak": peak,
                                      "unit": "GB/s", "frac": round(achieved / peak, 4),
                                      "peak_source": peak_kind},
                         "what": "the headline step above"}
        result["configs"] = cfgs
        result["gpu_launches"] += args.steps * sum(
            c["launches_per_step"] for k, c in cfgs.items() if k != "mixed")

    # Padded comparator: the same rows in a [rows][4096] slab, full width read.
    if not args.no_comparator and args.workload == "mixed":
        width = int(case.seq_lens.max())
        slabs = []
        for l in range(L):
            ks, vs = wl.padded_slab(case, l, width=width, fill_bits=0)
            slabs.append((torch.from_numpy(ks.view(np.float16)).to(dev),
                          torch.from_numpy(vs.view(np.float16)).to(dev)))
        wsp = ops.alloc_workspace(rows, hq, hk, hd, width, case.block_size, device=dev)

        def padded():
            for l in range(L):
                ops.padded_decode(out[l], d["q"][l], slabs[l][0], slabs[l][1], d["seq_lens"],
                                  case.scale, wsp)

        g_pad = capture(padded)
        ms_pad, _ = time_graph(g_pad, args.steps, args.warmup)
        result["comparator"] = {
            "padded_decode_ms_per_step": round(ms_pad, 5),
            "paged_decode_ms_per_step": round(ms_dec, 5),
            "paged_speedup": round(ms_pad / ms_dec, 3),
            "padded_bytes_read_per_layer": rows * width * hk * hd * 2 * 2,
        }
        del slabs, g_pad

    # End to end through the public API: per-step inputs from pinned host memory.
    if not args.no_e2e:
        # q, new tokens, tables, lengths and positions: one pinned buffer, one copy
        h_in = torch.empty_like(packed, device="cpu").pin_memory()
        h_in.copy_(packed)
        h_out = torch.empty_like(out, device="cpu").pin_memory()
        h2d = h_in.numel()
        d2h = h_out.numel() * h_out.element_size()

        def e2e_step():
            packed.copy_(h_in, non_blocking=True)
            g_step.replay()
            h_out.copy_(out, non_blocking=True)

        for _ in range(args.warmup):
            e2e_step()
        barrier(pg)
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(args.steps):
            e2e_step()
        e1.record()
        torch.cuda.synchronize()
        barrier(pg)
        ms_e2e = max_over_ranks(pg, e0.elapsed_time(e1) / args.steps)
        result["e2e"] = {"value": round(total_bytes / (ms_e2e * 1e-3) / 1e9, 2), "unit": "GB/s",
                         "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                         "ms_per_step": round(ms_e2e, 5)}

    if rank == 0 and not args.no_cpu_baseline:
        gbs, threads, dt, passes = cpu_oracle_sample(case)
        gbs1, _, dt1, passes1 = cpu_oracle_sample(case, seconds=CPU_SAMPLE_SECONDS / 4, threads=1)
        result["cpu_baseline"] = {
            "value": round(gbs, 5), "unit": "GB/s", "cores": threads, "kind": "oracle",
            "sample": f"{passes} layer passes (append + decode, fp64 C, OpenMP) over the "
                      f"{L} layers of the same workload, {dt:.1f} s",
            "single_thread": {"value": round(gbs1, 5), "unit": "GB/s",
                              "sample": f"{passes1} layer passes on one core, {dt1:.1f} s"}}
    return result


def run_reference(args, rank, world, pg):
    """The oracle as the reference arm: rank 0 only, on the host cores."""
    if rank != 0:
        return None
    import oracle
    from paged_kv_cache_06_gb300 import workloads as wl
    oracle.build()
    case = make_case(args)
    layers = min(REFERENCE_STEP_LAYERS, case.layers)
    b = wl.algorithmic_bytes(case)
    threads = oracle.default_threads()

    def step():
        for l in range(layers):
            kp, vp = oracle.paged_append(case.k_pool[l], case.v_pool[l], case.block_tables,
                                         case.positions, case.k_new[l], case.v_new[l])
            oracle.paged_decode(case.q[l], kp, vp, case.block_tables, case.seq_lens, case.scale,
                                num_threads=threads)

    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    ms = (time.perf_counter() - t0) * 1e3 / args.steps
    nbytes = layers * (b["decode_layer"] + b["append_layer"])
    value = nbytes / (ms * 1e-3) / 1e9
    sample = (f"each step: first {layers} of {case.layers} layers of the workload "
              f"(append + decode), fp64 C oracle, OpenMP")
    cfg = workload_config(case, args)
    return {
        "impl": "reference", "metric": METRIC, "value": round(value, 5), "unit": "GB/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded N(0,1) fp16 values, seeded lengths and block permutation)",
        "config": cfg,
        "rows_layers_per_s": round(case.rows * layers / (ms * 1e-3), 2),
        "cpu_baseline": {"value": round(value, 5), "unit": "GB/s", "cores": threads,
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": round(value, 5), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }


def main():
    args = parse_args()
    if args.impl == "reference":
        # Rank 0 alone times the oracle; other ranks exit without work.
        rank = int(os.environ.get("RANK", "0"))
        world = int(os.environ.get("WORLD_SIZE", "1"))
        res = run_reference(args, rank, world, None)
        if rank == 0 and res is not None:
            print(json.dumps(res), flush=True)
        return
    rank, world, pg = dist_setup(args)
    res = run_ours(args, rank, world, pg)
    if rank == 0 and res is not None:
        print(json.dumps(res), flush=True)
    if pg is not None:
        pg.destroy_process_group()


if __name__ == "__main__":
    main()
