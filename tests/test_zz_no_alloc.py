"""paged_attention_decode_noalloc: decode for callers that cannot allocate.

Some callers cannot give the library a device workspace: a plug-in inside a
host framework that owns all device memory through its own pool, or a serving
loop that forbids cudaMalloc after start-up because it can synchronise the
device.  For them the library keeps its split-K scratch in one static device
array.  These checks call that entry point through the C ABI and compare it
with the workspace-taking entry point on two calls in a row (the array keeps
the previous call's contents, so the second call checks that the entry point
re-arms it).  Both run the same kernel on the same work split, so the outputs
must be bit-identical; the calls must also leave the device's free memory
unchanged.

The file name sorts last so a run that stops at the first failure has already
run every other test; it also passes when run alone in a fresh process.
"""
import numpy as np
import pytest
import torch

from paged_kv_cache_06_gb300 import ops
from paged_kv_cache_06_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

ATOL = 2e-3
RTOL = 2e-3
NOALLOC_BYTES = 8 << 20  # PKV_NOALLOC_WORKSPACE_BYTES
PKV_ERR_WORKSPACE = 3


def _close(a: torch.Tensor, b: torch.Tensor):
    x = a.float().cpu().numpy()
    y = b.float().cpu().numpy()
    assert np.all(np.isfinite(x))
    assert np.all(np.abs(x - y) <= ATOL + RTOL * np.abs(y))
    # the same kernel on the same split: bit for bit
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def _reference_and_inputs(case):
    d = wl.to_device(case)
    kp, vp = d["k_pool"][0], d["v_pool"][0]
    if case.has_append:
        ops.append(kp, vp, d["block_tables"], d["positions"], d["k_new"][0], d["v_new"][0])
    ws = ops.alloc_workspace(case.rows, case.q_heads, case.kv_heads, case.head_dim,
                             case.max_seq_len, case.block_size)
    ref = torch.empty(case.rows, case.q_heads, case.head_dim, dtype=torch.float16, device="cuda")
    ops.decode(ref, d["q"][0], kp, vp, d["block_tables"], d["seq_lens"], case.scale,
               case.max_seq_len, ws)
    torch.cuda.synchronize()
    return d, kp, vp, ref


def test_noalloc_matches_workspace_entry_point_on_two_calls_in_a_row(cuda_device):
    case = wl.mixed(layers=1)
    assert ops.workspace_size(case.rows, 12, 2, 128, case.max_seq_len, 64) <= NOALLOC_BYTES
    d, kp, vp, ref = _reference_and_inputs(case)
    outs = [torch.full_like(ref, float("nan")) for _ in range(3)]
    # the first call may set up the array's address on this device
    ops.decode_noalloc(outs[0], d["q"][0], kp, vp, d["block_tables"], d["seq_lens"], case.scale,
                       case.max_seq_len)
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    alloc0 = torch.cuda.memory_allocated()
    for out in outs[1:]:
        ops.decode_noalloc(out, d["q"][0], kp, vp, d["block_tables"], d["seq_lens"], case.scale,
                           case.max_seq_len)
        torch.cuda.synchronize()
    assert torch.cuda.mem_get_info()[0] == free0
    assert torch.cuda.memory_allocated() == alloc0
    for out in outs:
        _close(out, ref)


def test_noalloc_after_a_different_shape(cuda_device):
    # The shared array still holds the mixed case's partials; a new shape must
    # not read them.
    case = wl.custom([700, 1, 300, 5000, 64], 64, seed=3, nan_fill=True)
    d, kp, vp, ref = _reference_and_inputs(case)
    for _ in range(2):
        out = torch.full_like(ref, float("nan"))
        ops.decode_noalloc(out, d["q"][0], kp, vp, d["block_tables"], d["seq_lens"], case.scale,
                           case.max_seq_len)
        torch.cuda.synchronize()
        _close(out, ref)


def test_noalloc_rejects_sizes_beyond_its_scratch(cuda_device):
    bs, msl = 16, 4096
    for rows in (256, 512, 1024, 2048, 4096, 8192):
        if ops.workspace_size(rows, 12, 2, 128, msl, bs) > NOALLOC_BYTES:
            break
    assert ops.workspace_size(rows, 12, 2, 128, msl, bs) > NOALLOC_BYTES
    mbpr = msl // bs
    q = torch.zeros(rows, 12, 128, dtype=torch.float16, device="cuda")
    pool = torch.zeros(1, bs, 2, 128, dtype=torch.float16, device="cuda")
    bt = torch.zeros(rows, mbpr, dtype=torch.int32, device="cuda")
    sl = torch.ones(rows, dtype=torch.int32, device="cuda")
    out = torch.empty_like(q)
    with pytest.raises(ops.PagedKVError) as e:
        ops.decode_noalloc(out, q, pool, pool, bt, sl, 0.088, msl)
    assert e.value.status == PKV_ERR_WORKSPACE
