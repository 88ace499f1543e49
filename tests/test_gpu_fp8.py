"""GPU parity for the FP8 (E4M3, one scale per KV head) pools.

The append must match the oracle's quantisation bit for bit over the whole
pool; the decode must satisfy |gpu - oracle| <= 2e-3 + 2e-3 * |oracle| like
the fp16 decode (the kernel converts E4M3 to fp16 exactly and applies the
scales in fp32).
"""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_06_gb300 import ops
from paged_kv_cache_06_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

ATOL = RTOL = 2e-3


def dev_u8(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def dev_f16(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.float16).cuda()


def dev_i32(a):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).cuda()


def dev_f32(a):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).cuda()


def assert_close(gpu, ref, what=""):
    g = gpu.float().cpu().numpy().astype(np.float64)
    assert np.all(np.isfinite(g)), what
    err = np.abs(g - ref)
    bound = ATOL + RTOL * np.abs(ref)
    bad = err > bound
    if bad.any():
        i = np.unravel_index(np.argmax(err - bound), err.shape)
        pytest.fail(f"{what}: {int(bad.sum())} outside tolerance; worst at {i}: gpu {g[i]} oracle {ref[i]}")


def fp8_case(lengths, bs, seed, extra=3):
    case = wl.custom(lengths, bs, seed=seed, append=True, nan_fill=False, extra_blocks=extra)
    gen = torch.Generator().manual_seed(seed + 1000)
    shape = case.k_pool[0].shape
    kp8, vp8 = wl.fp8_codes(gen, shape), wl.fp8_codes(gen, shape)
    ks = np.array([0.11, 0.16], dtype=np.float32)
    vs = np.array([0.09, 0.13], dtype=np.float32)
    return case, kp8, vp8, ks, vs


@pytest.mark.parametrize("lengths,bs", [([1, 17, 64, 200], 16), ([5, 64, 65, 1, 300], 64)])
def test_append_fp8_is_bit_exact_over_the_whole_pool(cuda_device, lengths, bs):
    case, kp8, vp8, ks, vs = fp8_case(lengths, bs, seed=3)
    # scales chosen so that some values saturate and some fall to subnormals
    ks = np.array([0.004, 0.3], dtype=np.float32)
    ek, ev = oracle.paged_append_fp8(kp8, vp8, ks, vs, case.block_tables, case.positions,
                                     case.k_new[0], case.v_new[0])
    gk, gv = dev_u8(kp8), dev_u8(vp8)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    ops.append_fp8(gk, gv, dev_f32(ks), dev_f32(vs), dev_i32(case.block_tables), dev_i32(case.positions),
                   dev_f16(case.k_new[0]), dev_f16(case.v_new[0]), dev_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert np.array_equal(gk.cpu().numpy(), ek) and np.array_equal(gv.cpu().numpy(), ev)
    assert (ek == 0x7E).any() or (ek == 0xFE).any()  # saturation was exercised


@pytest.mark.parametrize("lengths,bs", [
    ([1, 17, 64, 200], 16),
    ([5, 64, 65, 1, 4096, 300], 64),
    ([16] * 40, 16),
    ([0, 33, 2000], 32),
    # ranges longer than the ring: stream mode, units split within and across blocks
    ([20000, 3000, 17, 9000], 64),
    # stream mode with several short units in every block's range
    ([300] * 200 + [8000], 16),
])
def test_decode_fp8_matches_oracle(cuda_device, lengths, bs):
    case, kp8, vp8, ks, vs = fp8_case(lengths, bs, seed=len(lengths) + bs)
    ref = oracle.paged_decode_fp8(case.q[0], kp8, vp8, ks, vs, case.block_tables, case.seq_lens,
                                  case.scale, num_threads=oracle.default_threads())
    ws = ops.alloc_workspace(case.rows, case.q_heads, case.kv_heads, case.head_dim, case.max_seq_len,
                             bs)
    out = torch.full((case.rows, case.q_heads, case.head_dim), float("nan"), dtype=torch.float16,
                     device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    ops.decode_fp8(out, dev_f16(case.q[0]), dev_u8(kp8), dev_u8(vp8), dev_f32(ks), dev_f32(vs),
                   dev_i32(case.block_tables), dev_i32(case.seq_lens), case.scale, case.max_seq_len,
                   ws, dev_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert_close(out, ref, f"fp8 decode {lengths}")


def test_append_then_decode_fp8_full_mixed_shape(cuda_device):
    """The mixed batch-32 shape (31 rows of 16..512 tokens and one of 4096,
    block size 64): quantised append of the step's tokens, then decode,
    against the oracle doing the same two steps."""
    case = wl.mixed(seed=0, layers=1)
    gen = torch.Generator().manual_seed(77)
    shape = case.k_pool[0].shape
    kp8, vp8 = wl.fp8_codes(gen, shape), wl.fp8_codes(gen, shape)
    ks = np.array([0.12, 0.1], dtype=np.float32)
    vs = np.array([0.08, 0.14], dtype=np.float32)
    ek, ev = oracle.paged_append_fp8(kp8, vp8, ks, vs, case.block_tables, case.positions,
                                     case.k_new[0], case.v_new[0])
    rows = [0, 1, int(np.argmax(case.seq_lens)), case.rows - 1]
    sub = wl.row_subset(case, rows)
    ref = oracle.paged_decode_fp8(sub.q[0], ek, ev, ks, vs, sub.block_tables, sub.seq_lens,
                                  case.scale, num_threads=oracle.default_threads())
    gk, gv = dev_u8(kp8), dev_u8(vp8)
    gks, gvs = dev_f32(ks), dev_f32(vs)
    bt, sl = dev_i32(case.block_tables), dev_i32(case.seq_lens)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    ops.append_fp8(gk, gv, gks, gvs, bt, dev_i32(case.positions), dev_f16(case.k_new[0]),
                   dev_f16(case.v_new[0]), dev_err=err)
    ws = ops.alloc_workspace(case.rows, 12, 2, 128, case.max_seq_len, case.block_size)
    out = torch.empty((case.rows, 12, 128), dtype=torch.float16, device="cuda")
    ops.decode_fp8(out, dev_f16(case.q[0]), gk, gv, gks, gvs, bt, sl, case.scale, case.max_seq_len, ws,
                   dev_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert np.array_equal(gk.cpu().numpy(), ek) and np.array_equal(gv.cpu().numpy(), ev)
    assert_close(out[rows], ref, "mixed fp8")


def test_decode_fp8_bad_block_is_flagged(cuda_device):
    case, kp8, vp8, ks, vs = fp8_case([40, 20], 16, seed=5)
    bt = case.block_tables.copy()
    bt[0, 1] = case.num_blocks + 3
    ws = ops.alloc_workspace(case.rows, 12, 2, 128, case.max_seq_len, 16)
    out = torch.empty((case.rows, 12, 128), dtype=torch.float16, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    ops.decode_fp8(out, dev_f16(case.q[0]), dev_u8(kp8), dev_u8(vp8), dev_f32(ks), dev_f32(vs),
                   dev_i32(bt), dev_i32(case.seq_lens), case.scale, case.max_seq_len, ws, dev_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) & 1
    ref = oracle.paged_decode_fp8(case.q[0][1:], kp8, vp8, ks, vs, case.block_tables[1:],
                                  case.seq_lens[1:], case.scale)
    assert_close(out[1:], ref, "row without the bad entry")


@pytest.mark.parametrize("lengths,bs,pdl", [
    ([1, 17, 64, 200], 16, False),
    ([5, 64, 65, 1, 4096, 300], 64, True),
    ([16] * 40, 16, True),
    ([0, 33, 2000], 32, False),
    ("mixed", 64, True),
    ([20000, 3000, 17, 9000], 64, True),
])
def test_append_decode_fp8_fused_equals_the_two_calls(cuda_device, lengths, bs, pdl):
    """One fused launch: the pools end bit-identical to the oracle's FP8
    append, the outputs bit-identical to paged_kv_append_fp8 followed by
    paged_attention_decode_fp8, and within tolerance of the oracle."""
    if lengths == "mixed":
        case = wl.mixed(seed=2, layers=1)
        gen = torch.Generator().manual_seed(91)
        shape = case.k_pool[0].shape
        kp8, vp8 = wl.fp8_codes(gen, shape), wl.fp8_codes(gen, shape)
        ks = np.array([0.12, 0.1], dtype=np.float32)
        vs = np.array([0.08, 0.14], dtype=np.float32)
    else:
        case, kp8, vp8, ks, vs = fp8_case(lengths, bs, seed=7 + bs)
    ek, ev = oracle.paged_append_fp8(kp8, vp8, ks, vs, case.block_tables, case.positions,
                                     case.k_new[0], case.v_new[0])
    rows = sorted({0, case.rows - 1, int(np.argmax(case.seq_lens)), case.rows // 2})
    sub = wl.row_subset(case, rows)
    ref = oracle.paged_decode_fp8(sub.q[0], ek, ev, ks, vs, sub.block_tables, sub.seq_lens,
                                  case.scale, num_threads=oracle.default_threads())
    gks, gvs = dev_f32(ks), dev_f32(vs)
    bt, sl, pos = dev_i32(case.block_tables), dev_i32(case.seq_lens), dev_i32(case.positions)
    q, kn, vn = dev_f16(case.q[0]), dev_f16(case.k_new[0]), dev_f16(case.v_new[0])
    ws = ops.alloc_workspace(case.rows, case.q_heads, case.kv_heads, case.head_dim, case.max_seq_len,
                             case.block_size)
    shape = (case.rows, case.q_heads, case.head_dim)
    # the two calls
    k2, v2 = dev_u8(kp8), dev_u8(vp8)
    out2 = torch.full(shape, float("nan"), dtype=torch.float16, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    ops.append_fp8(k2, v2, gks, gvs, bt, pos, kn, vn, dev_err=err)
    ops.decode_fp8(out2, q, k2, v2, gks, gvs, bt, sl, case.scale, case.max_seq_len, ws, dev_err=err)
    # the fused launch
    k1, v1 = dev_u8(kp8), dev_u8(vp8)
    out1 = torch.full(shape, float("nan"), dtype=torch.float16, device="cuda")
    ops.append_decode_fp8(out1, q, k1, v1, gks, gvs, bt, sl, pos, kn, vn, case.scale,
                          case.max_seq_len, ws, pdl=pdl, dev_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert np.array_equal(k1.cpu().numpy(), ek) and np.array_equal(v1.cpu().numpy(), ev)
    assert torch.equal(out1.view(torch.int16), out2.view(torch.int16))
    assert_close(out1[rows], ref, f"fused fp8 {lengths}")


def test_append_decode_fp8_rejects_what_it_does_not_take(cuda_device):
    case, kp8, vp8, ks, vs = fp8_case([40, 20], 16, seed=5)
    ws = ops.alloc_workspace(case.rows, 12, 2, 128, case.max_seq_len, 16)
    out = torch.empty((case.rows, 12, 128), dtype=torch.float16, device="cuda")
    args = (out, dev_f16(case.q[0]), dev_u8(kp8), dev_u8(vp8), dev_f32(ks), dev_f32(vs),
            dev_i32(case.block_tables), dev_i32(case.seq_lens), dev_i32(case.positions),
            dev_f16(case.k_new[0]), dev_f16(case.v_new[0]), case.scale, case.max_seq_len)
    with pytest.raises(ops.PagedKVError):
        ops.append_decode_fp8(*args, ws[:16])  # workspace too small
    lib = ops.lib()
    st = lib.paged_attention_append_decode_fp8(
        ops._ptr(out), ops._ptr(args[1]), ops._ptr(args[2]), ops._ptr(args[3]), ops._ptr(args[4]),
        ops._ptr(args[5]), ops._ptr(args[6]), ops._ptr(args[7]), ops._ptr(args[8]),
        ops._ptr(args[9]), ops._ptr(args[10]), case.rows, 12, 2, 128, 16, float(case.scale),
        case.block_tables.shape[1], case.num_blocks, case.max_seq_len, ops._ptr(ws), ws.numel(),
        0x2, None, None)
    assert st != 0  # unknown flag
