"""GPU parity of the planned decode path (paged_attention_plan once per step,
paged_attention_decode_planned per layer) against the fp64 oracle, and
against the unplanned entry points, which run the same kernel on the same
split: the planned results must be bit-identical to them.
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
DEV_ERR_BLOCK_ID, DEV_ERR_SEQ_LEN, DEV_ERR_PLAN = 1, 2, 0x10


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


def make_plan(case, d, msl, append=True, dev_err=None):
    pb = ops.alloc_plan(case.rows, case.q_heads, case.kv_heads, case.head_dim, msl,
                        case.block_size)
    ops.plan(pb, d["block_tables"], d["seq_lens"], d["positions"] if append else None,
             case.q_heads, case.kv_heads, case.head_dim, case.block_size, case.num_blocks, msl,
             dev_err=dev_err)
    return pb


CASES = [
    ([1, 17, 64, 200], 16, 12, 2),
    ([1, 2, 3, 300, 255, 256, 257, 513], 16, 12, 2),
    ([0, 1, 1000, 0, 47], 64, 12, 2),
    ([700, 33, 64, 65], 32, 16, 2),
    ([129, 5, 600], 64, 8, 8),
    ([1500, 20, 2049], 128, 12, 2),
    ([4096] + [100] * 20, 64, 12, 2),
]


@pytest.mark.parametrize("lengths,bs,hq,hk", CASES)
def test_planned_append_decode_matches_oracle_and_unplanned(cuda_device, lengths, bs, hq, hk):
    case = wl.custom(lengths, bs, seed=len(lengths) + bs, nan_fill=True, extra_blocks=2,
                     q_heads=hq, kv_heads=hk)
    msl = case.max_seq_len
    d = wl.to_device(case)
    kp, vp = d["k_pool"][0].clone(), d["v_pool"][0].clone()
    ws = ops.alloc_workspace(case.rows, hq, hk, 128, msl, bs)
    pb = make_plan(case, d, msl)
    out = torch.full((case.rows, hq, 128), float("nan"), dtype=torch.float16, device="cuda")
    ops.decode_planned(out, d["q"][0], kp, vp, d["block_tables"], d["seq_lens"], case.scale, msl,
                       pb, ws, positions=d["positions"], k_new=d["k_new"][0], v_new=d["v_new"][0])
    # unplanned fused call on fresh pools
    kp2, vp2 = d["k_pool"][0].clone(), d["v_pool"][0].clone()
    out2 = torch.full_like(out, float("nan"))
    ops.append_decode(out2, d["q"][0], kp2, vp2, d["block_tables"], d["seq_lens"], d["positions"],
                      d["k_new"][0], d["v_new"][0], case.scale, msl, ws)
    torch.cuda.synchronize()
    ek, ev = oracle.paged_append(case.k_pool[0], case.v_pool[0], case.block_tables,
                                 case.positions, case.k_new[0], case.v_new[0])
    assert np.array_equal(bits(kp), ek) and np.array_equal(bits(vp), ev)
    ref = oracle.paged_decode(case.q[0], ek, ev, case.block_tables, case.seq_lens, case.scale,
                              num_threads=oracle.default_threads())
    assert_close(out, ref, f"planned lengths={lengths} bs={bs}")
    assert np.array_equal(bits(out), bits(out2)), "planned and unplanned calls differ"


def test_planned_decode_without_append(cuda_device):
    case = wl.custom([300, 1, 77, 1024, 5], 16, seed=11, nan_fill=True, append=False)
    msl = case.max_seq_len
    d = wl.to_device(case)
    ws = ops.alloc_workspace(case.rows, 12, 2, 128, msl, 16)
    pb = make_plan(case, d, msl, append=False)
    out = torch.full((case.rows, 12, 128), float("nan"), dtype=torch.float16, device="cuda")
    ops.decode_planned(out, d["q"][0], d["k_pool"][0], d["v_pool"][0], d["block_tables"],
                       d["seq_lens"], case.scale, msl, pb, ws)
    out2 = torch.full_like(out, float("nan"))
    ops.decode(out2, d["q"][0], d["k_pool"][0], d["v_pool"][0], d["block_tables"], d["seq_lens"],
               case.scale, msl, ws)
    torch.cuda.synchronize()
    ref = oracle.paged_decode(case.q[0], case.k_pool[0], case.v_pool[0], case.block_tables,
                              case.seq_lens, case.scale, num_threads=oracle.default_threads())
    assert_close(out, ref, "planned decode")
    assert np.array_equal(bits(out), bits(out2))


def test_planned_layers_of_a_step_share_one_plan(cuda_device):
    """The bench's step: one plan, then layer 0 without PDL and layers 1.. with
    PDL, captured in a CUDA graph; every row of every layer against the oracle."""
    case = wl.mixed(layers=4, nan_fill=True)
    msl = case.max_seq_len
    d = wl.to_device(case)
    ws = ops.alloc_workspace(case.rows, 12, 2, 128, msl, case.block_size)
    pb = ops.alloc_plan(case.rows, 12, 2, 128, msl, case.block_size)
    out = torch.full((case.layers, case.rows, 12, 128), float("nan"), dtype=torch.float16,
                     device="cuda")
    kp = d["k_pool"].clone()
    vp = d["v_pool"].clone()

    def step():
        ops.plan(pb, d["block_tables"], d["seq_lens"], d["positions"], 12, 2, 128,
                 case.block_size, case.num_blocks, msl)
        for l in range(case.layers):
            ops.decode_planned(out[l], d["q"][l], kp[l], vp[l], d["block_tables"], d["seq_lens"],
                               case.scale, msl, pb, ws, positions=d["positions"],
                               k_new=d["k_new"][l], v_new=d["v_new"][l], pdl=l > 0)

    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            step()
    torch.cuda.current_stream().wait_stream(s)
    for _ in range(3):  # the appends are idempotent: the same token into the same slot
        g.replay()
    torch.cuda.synchronize()
    for l in range(case.layers):
        ek, ev = oracle.paged_append(case.k_pool[l], case.v_pool[l], case.block_tables,
                                     case.positions, case.k_new[l], case.v_new[l])
        assert np.array_equal(bits(kp[l]), ek) and np.array_equal(bits(vp[l]), ev)
        ref = oracle.paged_decode(case.q[l], ek, ev, case.block_tables, case.seq_lens, case.scale,
                                  num_threads=oracle.default_threads())
        assert_close(out[l], ref, f"layer {l}")


def test_planned_fp8_matches_unplanned(cuda_device):
    case = wl.custom([1, 17, 300, 64, 513, 2000], 16, seed=5, nan_fill=False, extra_blocks=1)
    msl = case.max_seq_len
    d = wl.to_device(case)
    gen = torch.Generator().manual_seed(9)
    k8 = torch.from_numpy(wl.fp8_codes(gen, case.k_pool[0].shape)).cuda()
    v8 = torch.from_numpy(wl.fp8_codes(gen, case.v_pool[0].shape)).cuda()
    ks = torch.tensor([0.11, 0.13], dtype=torch.float32, device="cuda")
    vs = torch.tensor([0.12, 0.09], dtype=torch.float32, device="cuda")
    ws = ops.alloc_workspace(case.rows, 12, 2, 128, msl, 16)
    pb = make_plan(case, d, msl)
    out = torch.full((case.rows, 12, 128), float("nan"), dtype=torch.float16, device="cuda")
    k8a, v8a = k8.clone(), v8.clone()
    ops.decode_planned(out, d["q"][0], k8a, v8a, d["block_tables"], d["seq_lens"], case.scale, msl,
                       pb, ws, positions=d["positions"], k_new=d["k_new"][0], v_new=d["v_new"][0],
                       k_scale=ks, v_scale=vs)
    out2 = torch.full_like(out, float("nan"))
    k8b, v8b = k8.clone(), v8.clone()
    ops.append_decode_fp8(out2, d["q"][0], k8b, v8b, ks, vs, d["block_tables"], d["seq_lens"],
                          d["positions"], d["k_new"][0], d["v_new"][0], case.scale, msl, ws)
    torch.cuda.synchronize()
    assert torch.equal(k8a, k8b) and torch.equal(v8a, v8b)
    assert np.array_equal(bits(out), bits(out2))
    ref = oracle.paged_decode_fp8(case.q[0], k8a.cpu().numpy(), v8a.cpu().numpy(),
                                  ks.cpu().numpy(), vs.cpu().numpy(), case.block_tables,
                                  case.seq_lens, case.scale, num_threads=oracle.default_threads())
    assert_close(out, ref, "planned fp8")


def test_plan_for_another_launch_size_is_refused_on_the_device(cuda_device):
    """A plan made for fewer blocks than the launch uses sets PKV_DEV_ERR_PLAN
    and the call writes nothing."""
    case = wl.custom([3000, 40], 64, seed=3, nan_fill=True, append=False)
    d = wl.to_device(case)
    big = case.max_seq_len
    ws = ops.alloc_workspace(case.rows, 12, 2, 128, big, 64)
    pb = ops.alloc_plan(case.rows, 12, 2, 128, big, 64)
    small = torch.tensor([16, 16], dtype=torch.int32, device="cuda")
    ops.plan(pb, d["block_tables"], small, None, 12, 2, 128, 64, case.num_blocks, 16)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = torch.full((case.rows, 12, 128), float("nan"), dtype=torch.float16, device="cuda")
    ops.decode_planned(out, d["q"][0], d["k_pool"][0], d["v_pool"][0], d["block_tables"],
                       d["seq_lens"], case.scale, big, pb, ws, dev_err=err)
    assert ops.check_error(err) & DEV_ERR_PLAN
    assert torch.isnan(out.float()).all()


def test_plan_flags_bad_table_entries(cuda_device):
    case = wl.custom([200, 90], 16, seed=4, nan_fill=True, append=False)
    case.block_tables[1, 2] = case.num_blocks + 5
    d = wl.to_device(case)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    pb = make_plan(case, d, case.max_seq_len, append=False, dev_err=err)
    ws = ops.alloc_workspace(case.rows, 12, 2, 128, case.max_seq_len, 16)
    out = torch.zeros((case.rows, 12, 128), dtype=torch.float16, device="cuda")
    ops.decode_planned(out, d["q"][0], d["k_pool"][0], d["v_pool"][0], d["block_tables"],
                       d["seq_lens"], case.scale, case.max_seq_len, pb, ws)
    assert ops.check_error(err) & DEV_ERR_BLOCK_ID
    ref = oracle.paged_decode(case.q[0][:1], case.k_pool[0], case.v_pool[0],
                              case.block_tables[:1], case.seq_lens[:1], case.scale)
    assert_close(out[:1], ref, "row with good table entries")
