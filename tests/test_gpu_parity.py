"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle.

Append and block-table indexing must be bit-exact; attention outputs must
satisfy |gpu - oracle| <= 2e-3 + 2e-3 * |oracle| elementwise (fp16 output of
fp32 arithmetic; the pages report the paged kernel's fp16 outputs differing
from the contiguous kernel's by roughly 1e-3 relative).
"""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_06_gb300 import ops
from paged_kv_cache_06_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

ATOL = 2e-3
RTOL = 2e-3
DEV_ERR_BLOCK_ID, DEV_ERR_SEQ_LEN, DEV_ERR_POSITION = 1, 2, 4


def assert_close(gpu: torch.Tensor, ref: np.ndarray, what: str = ""):
    g = gpu.float().cpu().numpy().astype(np.float64)
    assert g.shape == ref.shape, (g.shape, ref.shape)
    assert np.all(np.isfinite(g)), f"{what}: non-finite output"
    err = np.abs(g - ref)
    bound = ATOL + RTOL * np.abs(ref)
    bad = err > bound
    if bad.any():
        i = np.unravel_index(np.argmax(err - bound), err.shape)
        pytest.fail(f"{what}: {int(bad.sum())} of {bad.size} outside tolerance; worst at {i}: "
                    f"gpu {g[i]!r} oracle {ref[i]!r}")


def bits(t: torch.Tensor) -> np.ndarray:
    return t.cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def oracle_after_append(case, layer, rows=None):
    """Oracle pools after this step's append, and the oracle decode of ``rows``."""
    kp, vp = case.k_pool[layer], case.v_pool[layer]
    if case.has_append:
        kp, vp = oracle.paged_append(kp, vp, case.block_tables, case.positions,
                                     case.k_new[layer], case.v_new[layer])
    sub = case if rows is None else wl.row_subset(case, rows)
    ref = oracle.paged_decode(sub.q[layer], kp, vp, sub.block_tables, sub.seq_lens, case.scale,
                              num_threads=oracle.default_threads())
    return kp, vp, ref


def run_gpu(case, layer=0, dev_err=None, max_seq_len=None, append=True):
    d = wl.to_device(case)
    kp, vp = d["k_pool"][layer], d["v_pool"][layer]
    if append and case.has_append:
        ops.append(kp, vp, d["block_tables"], d["positions"], d["k_new"][layer], d["v_new"][layer],
                   dev_err=dev_err)
    msl = case.max_seq_len if max_seq_len is None else max_seq_len
    ws = ops.alloc_workspace(case.rows, case.q_heads, case.kv_heads, case.head_dim, msl,
                             case.block_size)
    out = torch.full((case.rows, case.q_heads, case.head_dim), float("nan"),
                     dtype=torch.float16, device="cuda")
    ops.decode(out, d["q"][layer], kp, vp, d["block_tables"], d["seq_lens"], case.scale, msl, ws,
               dev_err=dev_err)
    torch.cuda.synchronize()
    return out, kp, vp, d, ws


# --- append ---------------------------------------------------------------------

@pytest.mark.parametrize("lengths,bs", [([1, 17, 64, 200], 16), ([5, 64, 65, 1], 64),
                                        ([3, 9, 2, 30], 1), ([100, 7], 7)])
def test_append_is_bit_exact_over_the_whole_pool(cuda_device, lengths, bs):
    case = wl.custom(lengths, bs, seed=1, nan_fill=True, extra_blocks=3)
    d = wl.to_device(case)
    ops.append(d["k_pool"][0], d["v_pool"][0], d["block_tables"], d["positions"], d["k_new"][0],
               d["v_new"][0])
    ek, ev = oracle.paged_append(case.k_pool[0], case.v_pool[0], case.block_tables,
                                 case.positions, case.k_new[0], case.v_new[0])
    assert np.array_equal(bits(d["k_pool"][0]), ek)
    assert np.array_equal(bits(d["v_pool"][0]), ev)


def test_append_skips_negative_positions(cuda_device):
    case = wl.custom([4, 8], 4, seed=2, nan_fill=True)
    case.positions[0] = -1
    d = wl.to_device(case)
    ops.append(d["k_pool"][0], d["v_pool"][0], d["block_tables"], d["positions"], d["k_new"][0],
               d["v_new"][0])
    ek, ev = oracle.paged_append(case.k_pool[0], case.v_pool[0], case.block_tables,
                                 case.positions, case.k_new[0], case.v_new[0])
    assert np.array_equal(bits(d["k_pool"][0]), ek)


# --- decode vs oracle -------------------------------------------------------------

def test_tiny_config_append_then_decode(cuda_device):
    case = wl.tiny(nan_fill=True)
    out, kp, vp, _, _ = run_gpu(case)
    ek, ev, ref = oracle_after_append(case, 0)
    assert np.array_equal(bits(kp), ek) and np.array_equal(bits(vp), ev)
    assert_close(out, ref, "tiny")


@pytest.mark.parametrize("lengths,bs,hq,hk", [
    ([1, 2, 3, 300, 255, 256, 257, 513], 16, 12, 2),   # split boundaries, ragged tails
    ([0, 1, 1000, 0, 47], 64, 12, 2),                  # zero-length rows
    ([700, 33, 64, 65], 32, 16, 2),                    # group of 8
    ([129, 5, 600], 64, 8, 8),                         # group of 1
    ([77, 300], 7, 4, 1),                              # odd block size, one KV head
    ([1500, 20, 2049], 128, 12, 2),                    # large blocks
    ([3000, 17], 1024, 12, 2),                         # largest supported block size
    ([40, 41, 42], 1, 12, 2),                          # one-token blocks
])
def test_decode_matches_oracle(cuda_device, lengths, bs, hq, hk):
    case = wl.custom(lengths, bs, seed=sum(lengths) % 97, nan_fill=True, extra_blocks=2,
                     q_heads=hq, kv_heads=hk)
    out, *_ = run_gpu(case)
    _, _, ref = oracle_after_append(case, 0)
    assert_close(out, ref, f"lengths={lengths} bs={bs}")


def test_one_token_row_returns_v_bit_exact(cuda_device):
    case = wl.custom([1, 1, 1], 16, seed=3, nan_fill=True)
    out, *_ = run_gpu(case)
    group = case.q_heads // case.kv_heads
    got = bits(out)
    for r in range(case.rows):
        for h in range(case.q_heads):
            assert np.array_equal(got[r, h], case.v_new[0, r, h // group])


def test_zero_length_rows_are_zero(cuda_device):
    case = wl.custom([0, 5, 0], 16, seed=4, nan_fill=True)
    out, *_ = run_gpu(case)
    o = out.float().cpu().numpy()
    assert np.all(o[0] == 0) and np.all(o[2] == 0) and np.all(np.isfinite(o[1]))


def test_bit_identical_under_permutation_of_physical_blocks(cuda_device):
    case = wl.custom([333, 64, 1, 700], 16, seed=5, nan_fill=True, extra_blocks=9)
    out_a, *_ = run_gpu(case)
    rng = np.random.default_rng(1)
    perm = rng.permutation(case.num_blocks)
    kp = np.empty_like(case.k_pool); vp = np.empty_like(case.v_pool)
    kp[:, perm] = case.k_pool; vp[:, perm] = case.v_pool
    bt = np.where(case.block_tables >= 0, perm[np.maximum(case.block_tables, 0)], -1).astype(np.int32)
    import dataclasses
    moved = dataclasses.replace(case, k_pool=kp, v_pool=vp, block_tables=bt)
    out_b, *_ = run_gpu(moved)
    assert torch.equal(out_a.view(torch.int16), out_b.view(torch.int16))


def test_workspace_reuse_gives_identical_results(cuda_device):
    case = wl.custom([900, 5, 2000, 64], 64, seed=6, nan_fill=True)
    out, kp, vp, d, ws = run_gpu(case)
    for _ in range(3):
        out2 = torch.empty_like(out)
        ops.decode(out2, d["q"][0], kp, vp, d["block_tables"], d["seq_lens"], case.scale,
                   case.max_seq_len, ws)
        assert torch.equal(out.view(torch.int16), out2.view(torch.int16))


@pytest.mark.parametrize("lengths,hq,hk", [
    ([8192], 4, 2),                    # group of 2: each unit split over 76 blocks
    ([3000, 2000], 2, 2),              # group of 1: 46-47 pieces, then 31
    ([1000, 1000, 1000, 1000], 2, 2),  # group of 1: 19 pieces per unit, landed merges
    ([1100, 1100], 8, 2),              # group of 4: 38 pieces per unit
    ([4096, 40, 900], 8, 2),           # group of 4: ~62 pieces on the long row, ~15 on the last
])
def test_units_split_over_many_blocks_small_groups(cuda_device, lengths, hq, hk):
    """A unit's merge over many pieces, for every record size: landed in shared
    memory when its records fit, else read from the workspace; repeated calls
    on one workspace stay bit-identical (arrival words re-armed)."""
    case = wl.custom(lengths, 16, seed=len(lengths) + hq, nan_fill=True, q_heads=hq, kv_heads=hk)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out, kp, vp, d, ws = run_gpu(case, dev_err=err)
    _, _, ref = oracle_after_append(case, 0)
    assert_close(out, ref, f"lengths={lengths} hq={hq} hk={hk}")
    for _ in range(3):
        out2 = torch.full_like(out, float("nan"))
        ops.decode(out2, d["q"][0], kp, vp, d["block_tables"], d["seq_lens"], case.scale,
                   case.max_seq_len, ws, dev_err=err)
        assert torch.equal(out.view(torch.int16), out2.view(torch.int16))
    assert int(err.item()) == 0


def test_padded_comparator_matches_oracle(cuda_device):
    case = wl.custom([12, 300, 1, 257], 16, seed=7, nan_fill=True)
    _, _, ref = oracle_after_append(case, 0)
    width = 512
    ks, vs = wl.padded_slab(case, 0, width=width, fill_bits=0)
    f16 = lambda a: torch.from_numpy(a.view(np.float16)).cuda()
    out = torch.full((case.rows, case.q_heads, case.head_dim), float("nan"), dtype=torch.float16,
                     device="cuda")
    ws = ops.alloc_workspace(case.rows, case.q_heads, case.kv_heads, case.head_dim, width, 16)
    ops.padded_decode(out, f16(case.q[0]), f16(ks), f16(vs),
                      torch.from_numpy(case.seq_lens).cuda(), case.scale, ws)
    torch.cuda.synchronize()
    assert_close(out, ref, "padded comparator")
    # the oracle's own contiguous form agrees on the same slab
    cont = oracle.contiguous_decode(case.q[0], ks, vs, case.seq_lens, case.scale)
    assert np.allclose(cont, ref, rtol=1e-12, atol=1e-12)


# --- full-size workloads, every row, in the launch the benchmark times ----------

def run_fused(case, layer=0, pdl=True):
    """One layer through paged_attention_append_decode with programmatic
    dependent launch, as the benchmark launches it (rows with a negative
    position append nothing)."""
    d = wl.to_device(case)
    kp, vp = d["k_pool"][layer], d["v_pool"][layer]
    ws = ops.alloc_workspace(case.rows, case.q_heads, case.kv_heads, case.head_dim,
                             case.max_seq_len, case.block_size)
    out = torch.full((case.rows, case.q_heads, case.head_dim), float("nan"),
                     dtype=torch.float16, device="cuda")
    ops.append_decode(out, d["q"][layer], kp, vp, d["block_tables"], d["seq_lens"],
                      d["positions"], d["k_new"][layer], d["v_new"][layer], case.scale,
                      case.max_seq_len, ws, pdl=pdl)
    torch.cuda.synchronize()
    return out, kp, vp


@pytest.mark.parametrize("name", ["uniform", "mixed", "shared", "long"])
def test_full_size_workloads_every_row(cuda_device, name):
    if name in ("uniform", "mixed"):
        case = wl.WORKLOADS[name](layers=1)
    else:
        case = wl.WORKLOADS[name]()
    out, kp, vp = run_fused(case)
    ek, ev, ref = oracle_after_append(case, 0)
    assert np.array_equal(bits(kp), ek) and np.array_equal(bits(vp), ev), f"{name}: pools"
    assert_close(out, ref, name)


def test_mixed_28_layer_pdl_graph_every_row(cuda_device):
    # Exactly the benchmark's step: 28 fused launches with programmatic
    # dependent launch, captured in one CUDA graph and replayed.
    case = wl.mixed(layers=28)
    d = wl.to_device(case)
    ws = ops.alloc_workspace(case.rows, 12, 2, 128, case.max_seq_len, 64)
    outs = torch.zeros(case.layers, case.rows, 12, 128, dtype=torch.float16, device="cuda")
    k0 = [d["k_pool"][l].clone() for l in range(case.layers)]
    v0 = [d["v_pool"][l].clone() for l in range(case.layers)]

    def step(pdl):
        for l in range(case.layers):
            ops.append_decode(outs[l], d["q"][l], d["k_pool"][l], d["v_pool"][l],
                              d["block_tables"], d["seq_lens"], d["positions"], d["k_new"][l],
                              d["v_new"][l], case.scale, case.max_seq_len, ws, pdl=pdl)

    step(False)
    torch.cuda.synchronize()
    eager = outs.clone()
    for l in range(case.layers):  # the pools as they were before the step
        d["k_pool"][l].copy_(k0[l])
        d["v_pool"][l].copy_(v0[l])
    outs.fill_(float("nan"))
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            step(True)
    torch.cuda.current_stream().wait_stream(s)
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    assert torch.equal(eager.view(torch.int16), outs.view(torch.int16))
    for layer in (case.layers // 2, case.layers - 1):
        ek, ev, ref = oracle_after_append(case, layer)
        assert np.array_equal(bits(d["k_pool"][layer]), ek), f"layer {layer} k pool"
        assert np.array_equal(bits(d["v_pool"][layer]), ev), f"layer {layer} v pool"
        assert_close(outs[layer], ref, f"pdl graph layer {layer}")


# --- device-side error reporting (never a fault) -----------------------------------

def test_bad_table_entries_are_flagged_and_skipped(cuda_device):
    case = wl.custom([40, 40], 16, seed=8, nan_fill=True, append=False)
    case.block_tables[1, 1] = case.num_blocks + 5      # out of range, and read
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out, *_ = run_gpu(case, dev_err=err)
    assert ops.check_error(err) & DEV_ERR_BLOCK_ID
    _, _, ref0 = oracle_after_append(case, 0, rows=[0])
    assert_close(out[:1], ref0, "row with a valid table")
    assert ops.check_error(err) == 0                    # cleared by the read


def test_seq_len_above_bound_is_clamped_and_flagged(cuda_device):
    case = wl.custom([64, 10], 16, seed=9, nan_fill=False, append=False)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    d = wl.to_device(case)
    d["seq_lens"][1] = 10_000
    ws = ops.alloc_workspace(2, 12, 2, 128, 64, 16)
    out = torch.empty(2, 12, 128, dtype=torch.float16, device="cuda")
    ops.decode(out, d["q"][0], d["k_pool"][0], d["v_pool"][0], d["block_tables"], d["seq_lens"],
               case.scale, 64, ws, dev_err=err)
    assert ops.check_error(err) & DEV_ERR_SEQ_LEN


def test_append_position_past_table_is_flagged(cuda_device):
    case = wl.custom([4], 4, seed=10, nan_fill=True)
    d = wl.to_device(case)
    d["positions"][0] = 4 * case.max_blocks_per_row      # logical block past the table
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    before = bits(d["k_pool"][0]).copy()
    ops.append(d["k_pool"][0], d["v_pool"][0], d["block_tables"], d["positions"], d["k_new"][0],
               d["v_new"][0], dev_err=err)
    assert ops.check_error(err) & DEV_ERR_POSITION
    assert np.array_equal(bits(d["k_pool"][0]), before)


# --- graph capture of a multi-layer step ----------------------------------------

def test_cuda_graph_of_layers_matches_eager(cuda_device):
    case = wl.mixed(layers=3)
    d = wl.to_device(case)
    ws = ops.alloc_workspace(case.rows, 12, 2, 128, case.max_seq_len, 64)
    outs = torch.zeros(case.layers, case.rows, 12, 128, dtype=torch.float16, device="cuda")

    def step():
        for l in range(case.layers):
            ops.append(d["k_pool"][l], d["v_pool"][l], d["block_tables"], d["positions"],
                       d["k_new"][l], d["v_new"][l])
            ops.decode(outs[l], d["q"][l], d["k_pool"][l], d["v_pool"][l], d["block_tables"],
                       d["seq_lens"], case.scale, case.max_seq_len, ws)

    step()
    torch.cuda.synchronize()
    eager = outs.clone()
    outs.zero_()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            step()
    torch.cuda.current_stream().wait_stream(s)
    for _ in range(2):
        g.replay()
    torch.cuda.synchronize()
    assert torch.equal(eager.view(torch.int16), outs.view(torch.int16))
    rows = [int(np.argmax(case.seq_lens)), 3]
    _, _, ref = oracle_after_append(case, 2, rows=rows)
    assert_close(outs[2][rows], ref, "graph layer 2")


# --- fused append + decode ---------------------------------------------------

def _fused_vs_separate(case, pdl=False):
    d1 = wl.to_device(case)
    d2 = wl.to_device(case)
    ws1 = ops.alloc_workspace(case.rows, case.q_heads, case.kv_heads, case.head_dim,
                              case.max_seq_len, case.block_size)
    ws2 = ops.alloc_workspace(case.rows, case.q_heads, case.kv_heads, case.head_dim,
                              case.max_seq_len, case.block_size)
    o1 = torch.full((case.rows, case.q_heads, case.head_dim), float("nan"), dtype=torch.float16,
                    device="cuda")
    o2 = torch.full_like(o1, float("nan"))
    ops.append(d1["k_pool"][0], d1["v_pool"][0], d1["block_tables"], d1["positions"],
               d1["k_new"][0], d1["v_new"][0])
    ops.decode(o1, d1["q"][0], d1["k_pool"][0], d1["v_pool"][0], d1["block_tables"],
               d1["seq_lens"], case.scale, case.max_seq_len, ws1)
    ops.append_decode(o2, d2["q"][0], d2["k_pool"][0], d2["v_pool"][0], d2["block_tables"],
                      d2["seq_lens"], d2["positions"], d2["k_new"][0], d2["v_new"][0], case.scale,
                      case.max_seq_len, ws2, pdl=pdl)
    torch.cuda.synchronize()
    return o1, o2, d1, d2


@pytest.mark.parametrize("lengths,bs", [([1, 17, 64, 200], 16), ([5, 64, 65, 1, 4096, 300], 64),
                                        ([700, 33, 64, 65], 32), ([77, 300], 7)])
def test_append_decode_equals_append_then_decode(cuda_device, lengths, bs):
    case = wl.custom(lengths, bs, seed=11, nan_fill=True, extra_blocks=2)
    o1, o2, d1, d2 = _fused_vs_separate(case)
    assert torch.equal(d1["k_pool"].view(torch.int16), d2["k_pool"].view(torch.int16))
    assert torch.equal(d1["v_pool"].view(torch.int16), d2["v_pool"].view(torch.int16))
    assert torch.equal(o1.view(torch.int16), o2.view(torch.int16))
    _, _, ref = oracle_after_append(case, 0)
    assert_close(o2, ref, "fused append+decode")


def test_append_decode_position_before_the_end_and_past_it(cuda_device):
    # positions < seq_len - 1 overwrite an older slot that is attended to;
    # positions >= seq_len are written but not attended to.
    case = wl.custom([40, 100, 33], 16, seed=12, nan_fill=False, append=False)
    case.positions[:] = [10, 100, 50]
    case.block_tables[1, 6] = case.num_blocks - 1 if case.block_tables[1, 6] < 0 else case.block_tables[1, 6]
    o1, o2, d1, d2 = _fused_vs_separate(case)
    assert torch.equal(d1["k_pool"].view(torch.int16), d2["k_pool"].view(torch.int16))
    assert torch.equal(o1.view(torch.int16), o2.view(torch.int16))


def test_append_decode_pdl_graph_of_layers_matches_eager(cuda_device):
    case = wl.mixed(layers=4)
    d = wl.to_device(case)
    ws = ops.alloc_workspace(case.rows, 12, 2, 128, case.max_seq_len, 64)
    outs = torch.zeros(case.layers, case.rows, 12, 128, dtype=torch.float16, device="cuda")

    def step(pdl):
        for l in range(case.layers):
            ops.append_decode(outs[l], d["q"][l], d["k_pool"][l], d["v_pool"][l],
                              d["block_tables"], d["seq_lens"], d["positions"], d["k_new"][l],
                              d["v_new"][l], case.scale, case.max_seq_len, ws, pdl=pdl)

    step(False)
    torch.cuda.synchronize()
    eager = outs.clone()
    outs.zero_()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            step(True)
    torch.cuda.current_stream().wait_stream(s)
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    assert torch.equal(eager.view(torch.int16), outs.view(torch.int16))
    rows = [int(np.argmax(case.seq_lens)), 5]
    _, _, ref = oracle_after_append(case, 3, rows=rows)
    assert_close(outs[3][rows], ref, "pdl graph layer 3")


def test_many_rows_use_the_split_kernel(cuda_device):
    # more rows than the staged kernel takes: the split kernel serves them
    lengths = (np.arange(1100) % 37 + 1).tolist()
    case = wl.custom(lengths, 16, seed=13, nan_fill=True)
    out, *_ = run_gpu(case)
    rows = [0, 36, 555, 1099]
    _, _, ref = oracle_after_append(case, 0, rows=rows)
    assert_close(out[rows], ref, "1100 rows")
