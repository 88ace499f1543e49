"""GPU parity for chunked-prefill paged attention (causal within each chunk).

|gpu - oracle| <= 2e-3 + 2e-3 * |oracle| elementwise, as for decode.
"""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_06_gb300 import ops
from paged_kv_cache_06_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

ATOL = RTOL = 2e-3


def assert_close(gpu, ref, what=""):
    g = gpu.float().cpu().numpy().astype(np.float64)
    assert np.all(np.isfinite(g)), what
    err = np.abs(g - ref)
    bound = ATOL + RTOL * np.abs(ref)
    bad = err > bound
    if bad.any():
        i = np.unravel_index(np.argmax(err - bound), err.shape)
        pytest.fail(f"{what}: {int(bad.sum())} of {bad.size} outside tolerance; worst at {i}: "
                    f"gpu {g[i]} oracle {ref[i]}")


def prefill_case(lengths, chunks, bs, seed):
    case = wl.custom(lengths, bs, seed=seed, append=False, nan_fill=True, extra_blocks=2)
    gen = torch.Generator().manual_seed(seed + 500)
    qs = np.concatenate([[0], np.cumsum(chunks)]).astype(np.int32)
    q = wl._randn_fp16(gen, (int(qs[-1]), case.q_heads, case.head_dim))
    return case, q, qs


def run(case, q, qs, dev_err=None, tables=None, workspace=None, stream=None, sync=True):
    d = wl.to_device(case)
    bt = d["block_tables"] if tables is None else torch.from_numpy(tables).cuda()
    gq = torch.from_numpy(q.view(np.int16)).view(torch.float16).cuda()
    out = torch.full(gq.shape, float("nan"), dtype=torch.float16, device="cuda")
    qst = torch.from_numpy(qs).cuda()
    if stream is not None:
        stream.wait_stream(torch.cuda.current_stream())
    ops.prefill(out, gq, d["k_pool"][0], d["v_pool"][0], bt, d["seq_lens"], qst, case.scale,
                case.max_seq_len, dev_err=dev_err, workspace=workspace, stream=stream)
    if sync:
        torch.cuda.synchronize()
        return out
    return out, (d, gq, qst, bt)  # keep the inputs alive until the caller synchronises


@pytest.mark.parametrize("lengths,chunks,bs", [
    ([100], [100], 16),                      # whole prompt, ragged last tile
    ([64, 300, 16], [17, 130, 16], 16),      # chunks at the end of longer rows
    ([1, 65, 200, 5], [1, 64, 65, 0], 64),   # a row with no queries
    ([640], [512], 32),                      # one 512-token chunk after 128 cached tokens
    ([300, 129], [200, 129], 128),           # 128-token pages: one copy per K tile
    ([260], [150], 48),                      # a page size that is no power of two
    ([192], [128], 16),                      # every unit cut in two; the end piece starts past
                                             #   the first 64 queries' last key
    ([8192], [128], 64),                     # one query tile per head, its keys cut over ~13 blocks
    ([3000, 20, 2500], [700, 20, 300], 16),  # long and short units cut at arbitrary steps
    ([20] * 60, [5] * 60, 16),               # many short units per block
])
def test_prefill_matches_oracle(cuda_device, lengths, chunks, bs):
    case, q, qs = prefill_case(lengths, chunks, bs, seed=sum(chunks) + bs)
    ref = oracle.paged_prefill(q, case.k_pool[0], case.v_pool[0], case.block_tables, case.seq_lens,
                               qs, case.scale, num_threads=oracle.default_threads())
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = run(case, q, qs, dev_err=err)
    assert int(err.item()) == 0
    assert_close(out, ref, f"prefill {lengths} {chunks}")


def test_prefill_512_chunks_on_4096_rows_sampled(cuda_device):
    """Two rows of 4096 tokens whose last 512 form the chunk (block size 64):
    every query of the first and last 64-query tile, and a sample between."""
    case, q, qs = prefill_case([4096, 4096], [512, 512], 64, seed=11)
    out = run(case, q, qs)
    idx = np.r_[0:64, 448:576, 960:1024, 200:201, 700:701]
    ref_all = oracle.paged_prefill(q, case.k_pool[0], case.v_pool[0], case.block_tables,
                                   case.seq_lens, qs, case.scale, num_threads=oracle.default_threads())
    assert_close(out[torch.from_numpy(idx)], ref_all[idx], "512-token chunks")


def test_prefill_benchmark_launch_every_query(cuda_device):
    # The benchmark's prefill launch: 8 rows whose newest 512 tokens are the
    # chunk, at 4096 tokens of context, 64-token blocks, seeds as there;
    # every query of every row against the oracle.
    case = wl.custom([4096] * 8, 64, seed=3, layers=1, append=False, nan_fill=False)
    chunk = 512
    qs = np.arange(0, chunk * (case.rows + 1), chunk, dtype=np.int32)
    gen = torch.Generator().manual_seed(4)
    q = torch.randn(case.rows * chunk, case.q_heads, case.head_dim, generator=gen).to(torch.float16)
    qbits = q.view(torch.int16).numpy().view(np.uint16)
    out = run(case, qbits, qs)
    ref = oracle.paged_prefill(qbits, case.k_pool[0], case.v_pool[0], case.block_tables,
                               case.seq_lens, qs, case.scale, num_threads=oracle.default_threads())
    assert_close(out, ref, "benchmark prefill launch")


def test_prefill_calls_on_separate_workspaces_overlap(cuda_device):
    # Two prefill calls, each with its own caller workspace, enqueued on two
    # streams at once (neither waits for the other): both match the oracle.
    # Then the same two back to back on one stream through the library-owned
    # scratch (no workspace).
    c1, q1, qs1 = prefill_case([3000, 20, 2500], [700, 20, 300], 16, seed=31)
    c2, q2, qs2 = prefill_case([8192], [128], 64, seed=32)
    ws1 = ops.alloc_prefill_workspace(c1.rows, c1.q_heads, c1.kv_heads, c1.head_dim, c1.block_size)
    ws2 = ops.alloc_prefill_workspace(c2.rows, c2.q_heads, c2.kv_heads, c2.head_dim, c2.block_size)
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    o1, keep1 = run(c1, q1, qs1, workspace=ws1, stream=s1, sync=False)
    o2, keep2 = run(c2, q2, qs2, workspace=ws2, stream=s2, sync=False)
    torch.cuda.synchronize()
    refs = []
    for c, q, qs, o in ((c1, q1, qs1, o1), (c2, q2, qs2, o2)):
        ref = oracle.paged_prefill(q, c.k_pool[0], c.v_pool[0], c.block_tables, c.seq_lens, qs,
                                   c.scale, num_threads=oracle.default_threads())
        assert_close(o, ref, "overlapping call")
        refs.append(ref)
    del keep1, keep2
    for c, q, qs, ref in ((c1, q1, qs1, refs[0]), (c2, q2, qs2, refs[1])):
        assert_close(run(c, q, qs), ref, "library-owned scratch")


def test_prefill_bit_identical_under_block_permutation(cuda_device):
    case, q, qs = prefill_case([300, 77], [120, 77], 16, seed=13)
    out1 = run(case, q, qs)
    # move every block to a new physical id
    nb = case.num_blocks
    perm = np.random.default_rng(1).permutation(nb).astype(np.int32)
    kp = np.empty_like(case.k_pool[0]); vp = np.empty_like(case.v_pool[0])
    kp[perm] = case.k_pool[0]; vp[perm] = case.v_pool[0]
    bt = np.where(case.block_tables >= 0, perm[np.maximum(case.block_tables, 0)], -1).astype(np.int32)
    case2 = wl.DecodeCase(**{**case.__dict__, "k_pool": kp[None], "v_pool": vp[None],
                             "block_tables": bt})
    out2 = run(case2, q, qs)
    assert torch.equal(out1.view(torch.int16), out2.view(torch.int16))


def test_prefill_bad_chunk_is_flagged_and_skipped(cuda_device):
    case, q, qs = prefill_case([10, 40], [12, 8], 16, seed=14)  # row 0: chunk longer than the row
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = run(case, q, qs, dev_err=err)
    assert int(err.item()) & 2
    ref = oracle.paged_prefill(q[12:], case.k_pool[0], case.v_pool[0], case.block_tables[1:],
                               case.seq_lens[1:], qs[1:] - 12, case.scale)
    assert_close(out[12:], ref, "the valid row")
    assert torch.isnan(out[:12].float()).all()  # skipped row untouched


def test_prefill_repeated_calls_are_bit_identical(cuda_device):
    """Units cut over several blocks merge the same way on every call (the
    arrival words are left at zero for the next call)."""
    case, q, qs = prefill_case([4000, 900], [256, 300], 32, seed=15)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    first = run(case, q, qs, dev_err=err)
    for _ in range(3):
        again = run(case, q, qs, dev_err=err)
        assert torch.equal(first.view(torch.int16), again.view(torch.int16))
    assert int(err.item()) == 0


def test_prefill_output_aligned_to_16_bytes_only(cuda_device):
    """An output that is 16- but not 32-byte aligned takes 16-byte stores."""
    case, q, qs = prefill_case([700, 300], [300, 129], 32, seed=16)
    d = wl.to_device(case)
    gq = torch.from_numpy(q.view(np.int16)).view(torch.float16).cuda()
    big = torch.full((gq.numel() + 8,), float("nan"), dtype=torch.float16, device="cuda")
    out = big[8:].view(gq.shape)
    assert out.data_ptr() % 32 == 16
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    ops.prefill(out, gq, d["k_pool"][0], d["v_pool"][0], d["block_tables"], d["seq_lens"],
                torch.from_numpy(qs).cuda(), case.scale, case.max_seq_len, dev_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert torch.isnan(big[:8].float()).all()
    ref = oracle.paged_prefill(q, case.k_pool[0], case.v_pool[0], case.block_tables, case.seq_lens,
                               qs, case.scale, num_threads=oracle.default_threads())
    assert_close(out, ref, "16-byte aligned output")


def test_prefill_1024_rows_of_short_chunks(cuda_device):
    """The most rows the kernel takes, with tiny ragged chunks (some empty):
    many whole units per block and rows skipped by the walk."""
    rng = np.random.default_rng(17)
    lengths = rng.integers(1, 40, size=1024)
    chunks = np.minimum(lengths, rng.integers(0, 4, size=1024))
    case, q, qs = prefill_case(lengths.tolist(), chunks.tolist(), 16, seed=17)
    ref = oracle.paged_prefill(q, case.k_pool[0], case.v_pool[0], case.block_tables, case.seq_lens,
                               qs, case.scale, num_threads=oracle.default_threads())
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = run(case, q, qs, dev_err=err)
    assert int(err.item()) == 0
    assert_close(out, ref, "1024 rows")


def test_prefill_more_than_1024_rows_is_rejected(cuda_device):
    case, q, qs = prefill_case([3] * 1025, [1] * 1025, 16, seed=18)
    with pytest.raises(ops.PagedKVError) as e:
        run(case, q, qs)
    assert e.value.status == 2  # PKV_ERR_UNSUPPORTED
