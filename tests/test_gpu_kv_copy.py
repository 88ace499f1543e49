"""GPU parity for the copy-on-write block copy and the prefill scatter.

Both are pure data movement, so the whole pools must match the oracle's bit
for bit.  The integration test drives the host block manager through a
shared prefix, a copy-on-write and an append, then checks decode against the
oracle run through the same steps.
"""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_06_gb300 import ops
from paged_kv_cache_06_gb300 import workloads as wl
from paged_kv_cache_06_gb300.block_manager import BlockManager

pytestmark = pytest.mark.gpu

DEV_ERR_BLOCK_ID, DEV_ERR_POSITION = 1, 4
HK, D = 2, 128


def bits(t: torch.Tensor) -> np.ndarray:
    return t.cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def dev(a, dtype=None):
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16)).view(torch.float16).cuda()
    return torch.from_numpy(a.astype(np.int32)).cuda()


def pools(gen, nb, bs):
    return wl._randn_fp16(gen, (nb, bs, HK, D)), wl._randn_fp16(gen, (nb, bs, HK, D))


def err_tensor():
    return torch.zeros(1, dtype=torch.int32, device="cuda")


# --- copy-on-write block copy ------------------------------------------------------

@pytest.mark.parametrize("bs,n", [(16, 1), (16, 37), (64, 9), (1, 5), (128, 3)])
def test_copy_blocks_bit_exact_over_the_whole_pool(cuda_device, bs, n):
    gen = torch.Generator().manual_seed(bs * 100 + n)
    nb = 2 * n + 7
    kp, vp = pools(gen, nb, bs)
    perm = torch.randperm(nb, generator=gen).numpy()
    src, dst = perm[:n], perm[n:2 * n]
    ek, ev = oracle.copy_blocks(kp, vp, src, dst)
    gk, gv = dev(kp), dev(vp)
    err = err_tensor()
    ops.copy_blocks(gk, gv, dev(src), dev(dst), dev_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert np.array_equal(bits(gk), ek) and np.array_equal(bits(gv), ev)


def test_copy_blocks_shared_source_and_self_copy(cuda_device):
    """One source cloned into several blocks; a pair with src == dst is a no-op."""
    gen = torch.Generator().manual_seed(5)
    kp, vp = pools(gen, 12, 16)
    src, dst = np.array([3, 3, 3, 7]), np.array([0, 5, 9, 7])
    ek, ev = oracle.copy_blocks(kp, vp, src, dst)
    gk, gv = dev(kp), dev(vp)
    ops.copy_blocks(gk, gv, dev(src), dev(dst))
    torch.cuda.synchronize()
    assert np.array_equal(bits(gk), ek) and np.array_equal(bits(gv), ev)


def test_copy_blocks_empty_list_is_a_no_op(cuda_device):
    gen = torch.Generator().manual_seed(6)
    kp, vp = pools(gen, 4, 16)
    gk, gv = dev(kp), dev(vp)
    empty = torch.zeros(0, dtype=torch.int32, device="cuda")
    ops.copy_blocks(gk, gv, empty, empty)
    torch.cuda.synchronize()
    assert np.array_equal(bits(gk), kp) and np.array_equal(bits(gv), vp)


def test_copy_blocks_bad_id_is_flagged_and_skipped(cuda_device):
    gen = torch.Generator().manual_seed(7)
    nb = 10
    kp, vp = pools(gen, nb, 16)
    src, dst = np.array([1, 2, 3]), np.array([4, nb, 5])
    ek, ev = oracle.copy_blocks(kp, vp, src[[0, 2]], dst[[0, 2]])
    gk, gv = dev(kp), dev(vp)
    err = err_tensor()
    ops.copy_blocks(gk, gv, dev(src), dev(dst), dev_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) & DEV_ERR_BLOCK_ID
    assert np.array_equal(bits(gk), ek) and np.array_equal(bits(gv), ev)


# --- prefill scatter --------------------------------------------------------------

def _scatter_case(gen, lengths, bs, dst_start=None, width=None, spare=5):
    lengths = np.asarray(lengths, dtype=np.int32)
    rows = len(lengths)
    width = int(lengths.max()) if width is None else width
    ds = np.zeros(rows, np.int32) if dst_start is None else np.asarray(dst_start, np.int32)
    need = [(int(d + l) + bs - 1) // bs for d, l in zip(ds, lengths)]
    mbpr = max(1, max(need))
    nb = sum(need) + spare
    perm = torch.randperm(nb, generator=gen).numpy().astype(np.int32)
    bt = np.full((rows, mbpr), -1, np.int32)
    k = 0
    for r in range(rows):
        bt[r, :need[r]] = perm[k:k + need[r]]
        k += need[r]
    kp, vp = pools(gen, nb, bs)
    ks = wl._randn_fp16(gen, (rows, width, HK, D))
    vs = wl._randn_fp16(gen, (rows, width, HK, D))
    ss = (width - lengths).astype(np.int32)  # left padding
    return kp, vp, bt, ss, ds, lengths, ks, vs


@pytest.mark.parametrize("lengths,bs,dst", [
    ([1, 17, 64, 200, 0], 16, None),
    ([5, 64, 65, 1], 64, [0, 3, 64, 127]),
    ([300, 33], 1, [7, 0]),
    ([16] * 40, 16, None),
])
def test_prefill_scatter_bit_exact_over_the_whole_pool(cuda_device, lengths, bs, dst):
    gen = torch.Generator().manual_seed(len(lengths) * 1000 + bs)
    kp, vp, bt, ss, ds, ln, ks, vs = _scatter_case(gen, lengths, bs, dst)
    ek, ev = oracle.prefill_scatter(kp, vp, bt, ss, ds, ln, ks, vs)
    gk, gv = dev(kp), dev(vp)
    err = err_tensor()
    ops.prefill_scatter(gk, gv, dev(bt), dev(ss), dev(ds), dev(ln), dev(ks), dev(vs), dev_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert np.array_equal(bits(gk), ek) and np.array_equal(bits(gv), ev)


def test_prefill_scatter_position_past_table_is_flagged(cuda_device):
    gen = torch.Generator().manual_seed(11)
    kp, vp, bt, ss, ds, ln, ks, vs = _scatter_case(gen, [20, 20], 16)
    # Row 1 starts one token before the end of its two-block table: tokens past
    # position 31 have no block and are skipped; row 0 is unaffected.
    ds_bad = np.array([0, 31], np.int32)
    # Expected: row 0 in full, and row 1's first token at position 31.
    ek, ev = oracle.prefill_scatter(kp, vp, bt[:1], ss[:1], ds[:1], ln[:1], ks[:1], vs[:1])
    ek, ev = oracle.prefill_scatter(ek, ev, bt[1:], ss[1:], ds_bad[1:], np.array([1], np.int32),
                                    ks[1:], vs[1:])
    gk, gv = dev(kp), dev(vp)
    err = err_tensor()
    ops.prefill_scatter(gk, gv, dev(bt), dev(ss), dev(ds_bad), dev(ln), dev(ks), dev(vs),
                        dev_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) & DEV_ERR_POSITION
    assert np.array_equal(bits(gk), ek) and np.array_equal(bits(gv), ev)


def test_prefill_scatter_source_range_past_width_is_flagged(cuda_device):
    gen = torch.Generator().manual_seed(12)
    kp, vp, bt, ss, ds, ln, ks, vs = _scatter_case(gen, [8, 8], 16)
    ss_bad = np.array([0, 1], np.int32)  # row 1: columns 1..8 of a width-8 source
    ek, ev = oracle.prefill_scatter(kp, vp, bt[:1], ss_bad[:1], ds[:1], ln[:1], ks[:1], vs[:1])
    gk, gv = dev(kp), dev(vp)
    err = err_tensor()
    ops.prefill_scatter(gk, gv, dev(bt), dev(ss_bad), dev(ds), dev(ln), dev(ks), dev(vs),
                        dev_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) & DEV_ERR_POSITION
    assert np.array_equal(bits(gk), ek) and np.array_equal(bits(gv), ev)


# --- shared prefix, copy-on-write, append, decode --------------------------------

def test_prefix_cow_append_decode_matches_oracle(cuda_device):
    """Two sequences share a 112-token prefix; the first one's prompt ends inside
    the last shared block, so its next append must clone that block first.  The
    other sequence must still see the original block."""
    bs, hq = 16, 12
    gen = torch.Generator().manual_seed(21)
    bm = BlockManager(32, bs, 16)
    pid, pids = bm.register_prefix(112)                   # 7 whole blocks
    bm.admit(0, 100, 4, prefix_id=pid)                    # ends inside shared block 6
    bm.admit(1, 130, 4, prefix_id=pid)                    # private tail after the prefix
    kp, vp = pools(gen, 32, bs)

    # Prefill: the prefix once (into its own blocks), then each prompt's private tail.
    pre_k = wl._randn_fp16(gen, (1, 112, HK, D))
    pre_v = wl._randn_fp16(gen, (1, 112, HK, D))
    pre_bt = np.full((1, 16), -1, np.int32)
    pre_bt[0, :7] = pids
    tail_k = wl._randn_fp16(gen, (2, 18, HK, D))
    tail_v = wl._randn_fp16(gen, (2, 18, HK, D))
    bt, lens = bm.tables([0, 1])
    t_ss, t_ds, t_ln = np.array([18, 0], np.int32), np.array([100, 112], np.int32), \
        np.array([0, 18], np.int32)

    pk, pv = oracle.prefill_scatter(kp, vp, pre_bt, [0], [0], [112], pre_k, pre_v)
    ek, ev = oracle.prefill_scatter(pk, pv, bt, t_ss, t_ds, t_ln, tail_k, tail_v)
    gk, gv = dev(kp), dev(vp)
    err = err_tensor()
    ops.prefill_scatter(gk, gv, dev(pre_bt), dev([0]), dev([0]), dev([112]), dev(pre_k),
                        dev(pre_v), dev_err=err)
    ops.prefill_scatter(gk, gv, dev(bt), dev(t_ss), dev(t_ds), dev(t_ln), dev(tail_k),
                        dev(tail_v), dev_err=err)

    # One decode step for both sequences.
    pos0, cow0 = bm.append_slot(0)
    pos1, cow1 = bm.append_slot(1)
    assert cow0 is not None and cow0[0] == pids[6] and cow1 is None
    src, dst = np.array([cow0[0]]), np.array([cow0[1]])
    ek, ev = oracle.copy_blocks(ek, ev, src, dst)
    ops.copy_blocks(gk, gv, dev(src), dev(dst), dev_err=err)
    bt, lens = bm.tables([0, 1])
    positions = np.array([pos0, pos1], np.int32)
    k_new = wl._randn_fp16(gen, (2, HK, D))
    v_new = wl._randn_fp16(gen, (2, HK, D))
    ek, ev = oracle.paged_append(ek, ev, bt, positions, k_new, v_new)
    gbt = dev(bt)
    ops.append(gk, gv, gbt, dev(positions), dev(k_new), dev(v_new), dev_err=err)
    q = wl._randn_fp16(gen, (2, hq, D))
    scale = wl.default_scale(D)
    ref = oracle.paged_decode(q, ek, ev, bt, lens, scale)
    msl = int(lens.max())
    ws = ops.alloc_workspace(2, hq, HK, D, msl, bs)
    out = torch.empty((2, hq, D), dtype=torch.float16, device="cuda")
    ops.decode(out, dev(q), gk, gv, gbt, dev(lens), scale, msl, ws, dev_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert np.array_equal(bits(gk), ek) and np.array_equal(bits(gv), ev)
    # The shared block still holds the prefix for sequence 1: the append went
    # to the clone.
    b = int(pids[6])
    assert np.array_equal(bits(gk)[b], pk[b]) and np.array_equal(bits(gv)[b], pv[b])
    assert not np.array_equal(bits(gk)[cow0[1]], pk[b])
    g = out.float().cpu().numpy().astype(np.float64)
    assert np.all(np.abs(g - ref) <= 2e-3 + 2e-3 * np.abs(ref))
