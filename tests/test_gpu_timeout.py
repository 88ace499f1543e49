"""The decode merge's bounded wait, made to run out on purpose (no fault).

A split unit's merge polls the records of the unit's other pieces.  A test
hook caps those polls and adds a device word that nothing writes to what every
poll waits for, so every merge gives up: the call must still finish (in
milliseconds, not the production limit of about a second), flag
PKV_DEV_ERR_TIMEOUT in the error word, and leave the device usable: after the
workspace is zero-filled again, the next call matches the oracle.
"""
import time

import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_06_gb300 import ops
from paged_kv_cache_06_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

DEV_ERR_TIMEOUT = 0x8
ATOL = RTOL = 2e-3


@pytest.mark.parametrize("name", ["mixed", "uniform"])  # burst-mode and stream-mode blocks
def test_merge_poll_runs_out_and_the_next_call_is_exact(cuda_device, name):
    case = wl.WORKLOADS[name](layers=1)
    d = wl.to_device(case)
    kp, vp = d["k_pool"][0], d["v_pool"][0]
    ws = ops.alloc_workspace(case.rows, case.q_heads, case.kv_heads, case.head_dim,
                             case.max_seq_len, case.block_size)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    stuck = torch.zeros(1, dtype=torch.int32, device="cuda")  # nothing ever writes it
    out = torch.full((case.rows, case.q_heads, case.head_dim), float("nan"),
                     dtype=torch.float16, device="cuda")
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    try:
        ops.debug_set_decode_hooks(1024, stuck)
        ops.decode(out, d["q"][0], kp, vp, d["block_tables"], d["seq_lens"], case.scale,
                   case.max_seq_len, ws, dev_err=err)
        torch.cuda.synchronize()
    finally:
        ops.debug_set_decode_hooks(0, None)
    elapsed = time.perf_counter() - t0
    assert ops.check_error(err) & DEV_ERR_TIMEOUT
    assert elapsed < 2.0, elapsed
    # the context is still usable; the workspace is zero-filled again first
    ws.zero_()
    out.fill_(float("nan"))
    ops.decode(out, d["q"][0], kp, vp, d["block_tables"], d["seq_lens"], case.scale,
               case.max_seq_len, ws, dev_err=err)
    torch.cuda.synchronize()
    assert ops.check_error(err) == 0
    ref = oracle.paged_decode(case.q[0], case.k_pool[0], case.v_pool[0], case.block_tables,
                              case.seq_lens, case.scale, num_threads=oracle.default_threads())
    g = out.float().cpu().numpy().astype(np.float64)
    assert np.all(np.abs(g - ref) <= ATOL + RTOL * np.abs(ref))
