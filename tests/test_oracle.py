"""Pins for the fp64 oracle: it is checked against things other than itself.

Each test ties one part of the oracle to a fact fixed by the pages or by
mathematics, chosen so a plausible slip (wrong fp16 decode, dropped
normalisation, wrong query-head -> KV-head map, wrong table index, reading
past the row's length, wrong merge weight) fails at least one of them.
"""
import json
import math
import os

import numpy as np
import pytest
import scipy.special

import oracle
from oracle import brute
from paged_kv_cache_06_gb300 import workloads as wl

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _f16(a):
    return np.asarray(a, dtype=np.float16).view(np.uint16)


def _rand_case(seed, lengths, bs, hq=4, hk=2, d=8, extra=3, nan=True):
    return wl.custom(lengths, bs, seed=seed, append=False, nan_fill=nan, extra_blocks=extra,
                     q_heads=hq, kv_heads=hk, head_dim=d)


# --- fp16 decoding -----------------------------------------------------------

def test_half_decode_matches_numpy_for_every_bit_pattern():
    bits = np.arange(1 << 16, dtype=np.uint16)
    ours = oracle.half_to_double(bits)
    ref = bits.view(np.float16).astype(np.float64)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], ref[~nan])
    # signed zero is kept
    assert math.copysign(1.0, ours[0x8000]) == -1.0


# --- brute force ---------------------------------------------------------------

@pytest.mark.parametrize("seed,lengths,bs", [
    (1, [1, 2, 3], 1), (2, [5, 0, 7], 2), (3, [4, 9], 3), (4, [8, 8, 1, 13], 4), (5, [6], 5)])
def test_oracle_matches_pure_python_brute_force(seed, lengths, bs):
    c = _rand_case(seed, lengths, bs)
    ours = oracle.paged_decode(c.q[0], c.k_pool[0], c.v_pool[0], c.block_tables, c.seq_lens, c.scale)
    ref = np.array(brute.paged_decode(c.q[0].tolist(), c.k_pool[0].tolist(), c.v_pool[0].tolist(),
                                      c.block_tables.tolist(), c.seq_lens.tolist(), c.scale))
    ref = ref.reshape(ours.shape)
    np.testing.assert_allclose(ours, ref, rtol=1e-12, atol=1e-12)


def test_golden_hand_worked_decode():
    g = json.load(open(os.path.join(GOLDEN, "decode_hand.json")))
    out = oracle.paged_decode(_f16(g["q"]), _f16(g["k_pool"]), _f16(g["v_pool"]),
                              np.array(g["block_tables"], np.int32),
                              np.array(g["seq_lens"], np.int32), g["scale"])
    np.testing.assert_allclose(out, np.array(g["expected"]), rtol=1e-14, atol=1e-14)


# --- closed forms and special cases --------------------------------------------

def test_one_token_row_returns_v_exactly():
    c = _rand_case(7, [1, 1, 1], 4)
    out = oracle.paged_decode(c.q[0], c.k_pool[0], c.v_pool[0], c.block_tables, c.seq_lens, c.scale)
    group = c.q_heads // c.kv_heads
    for r in range(c.rows):
        pb = c.block_tables[r, 0]
        for h in range(c.q_heads):
            v = oracle.half_to_double(c.v_pool[0, pb, 0, h // group])
            assert np.array_equal(out[r, h], v)


def test_constant_v_returns_that_v():
    c = _rand_case(8, [9, 30], 4, nan=False)
    v = c.v_pool.copy()
    const = _f16(np.linspace(-2, 2, c.head_dim))
    v[...] = const  # every token of every head carries the same V
    out = oracle.paged_decode(c.q[0], c.k_pool[0], v[0], c.block_tables, c.seq_lens, c.scale)
    np.testing.assert_allclose(out, np.broadcast_to(oracle.half_to_double(const), out.shape),
                               rtol=1e-14, atol=1e-15)


def test_equal_keys_give_the_plain_mean_of_v():
    c = _rand_case(9, [11, 4], 3, nan=False)
    k = c.k_pool.copy()
    k[...] = _f16(np.full(c.head_dim, 0.75))
    out = oracle.paged_decode(c.q[0], k[0], c.v_pool[0], c.block_tables, c.seq_lens, c.scale)
    group = c.q_heads // c.kv_heads
    for r in range(c.rows):
        toks = [(c.block_tables[r, t // 3], t % 3) for t in range(c.seq_lens[r])]
        for h in range(c.q_heads):
            vs = np.stack([oracle.half_to_double(c.v_pool[0, pb, s, h // group]) for pb, s in toks])
            np.testing.assert_allclose(out[r, h], np.mean(vs, axis=0), rtol=1e-13, atol=1e-14)


def test_zero_scale_gives_the_plain_mean_of_v():
    c = _rand_case(10, [7], 2, nan=False)
    out = oracle.paged_decode(c.q[0], c.k_pool[0], c.v_pool[0], c.block_tables, c.seq_lens, 0.0)
    group = c.q_heads // c.kv_heads
    toks = [(c.block_tables[0, t // 2], t % 2) for t in range(7)]
    for h in range(c.q_heads):
        vs = np.stack([oracle.half_to_double(c.v_pool[0, pb, s, h // group]) for pb, s in toks])
        np.testing.assert_allclose(out[0, h], vs.mean(axis=0), rtol=1e-13, atol=1e-14)


def test_two_tokens_follow_the_logistic_closed_form():
    # softmax of two scores is (1 - sigma(s1 - s0), sigma(s1 - s0))
    c = _rand_case(11, [2], 1, nan=False)
    out = oracle.paged_decode(c.q[0], c.k_pool[0], c.v_pool[0], c.block_tables, c.seq_lens, c.scale)
    group = c.q_heads // c.kv_heads
    b0, b1 = c.block_tables[0, 0], c.block_tables[0, 1]
    for h in range(c.q_heads):
        kvh = h // group
        qv = oracle.half_to_double(c.q[0, 0, h])
        k0 = oracle.half_to_double(c.k_pool[0, b0, 0, kvh])
        k1 = oracle.half_to_double(c.k_pool[0, b1, 0, kvh])
        v0 = oracle.half_to_double(c.v_pool[0, b0, 0, kvh])
        v1 = oracle.half_to_double(c.v_pool[0, b1, 0, kvh])
        w1 = scipy.special.expit(c.scale * (np.dot(qv, k1) - np.dot(qv, k0)))
        np.testing.assert_allclose(out[0, h], v0 + w1 * (v1 - v0), rtol=1e-12, atol=1e-13)


def test_dominant_score_selects_its_token_without_overflow():
    # a huge score must not overflow: the result is that token's V
    c = _rand_case(12, [5], 5, hq=2, hk=1, d=8, nan=False)
    q = c.q.copy(); k = c.k_pool.copy()
    q[...] = _f16(np.full(8, 8.0))
    k[0, c.block_tables[0, 0]] = _f16(np.zeros(8))
    k[0, c.block_tables[0, 0], 3] = _f16(np.full(8, 60000.0))
    out = oracle.paged_decode(q[0], k[0], c.v_pool[0], c.block_tables, c.seq_lens, 1.0)
    v = oracle.half_to_double(c.v_pool[0, c.block_tables[0, 0], 3, 0])
    assert np.all(np.isfinite(out))
    np.testing.assert_allclose(out[0, 0], v, rtol=0, atol=1e-300)


def test_gqa_maps_contiguous_query_head_groups_to_kv_heads():
    # Hq=6, Hk=3: heads {0,1}->kv0, {2,3}->kv1, {4,5}->kv2.
    c = _rand_case(13, [6, 3], 2, hq=6, hk=3, d=8, nan=False)
    v = c.v_pool.copy()
    for kvh in range(3):
        v[0, :, :, kvh] = _f16(np.full(8, float(kvh + 1)))
    out = oracle.paged_decode(c.q[0], c.k_pool[0], v[0], c.block_tables, c.seq_lens, c.scale)
    for h in range(6):
        np.testing.assert_allclose(out[:, h], h // 2 + 1.0, rtol=1e-14)


def test_zero_length_row_is_all_zeros():
    c = _rand_case(14, [0, 5, 0], 2)
    out = oracle.paged_decode(c.q[0], c.k_pool[0], c.v_pool[0], c.block_tables, c.seq_lens, c.scale)
    assert np.all(out[0] == 0) and np.all(out[2] == 0)
    assert np.all(np.isfinite(out[1]))


# --- invariants fixed by the pages -------------------------------------------

def test_output_invariant_under_permutation_of_physical_block_ids():
    # blocks are interchangeable: moving every block to another id and
    # rewriting the tables accordingly changes nothing, bit for bit.
    c = _rand_case(15, [13, 7, 1, 20], 4, extra=5)
    rng = np.random.default_rng(0)
    perm = rng.permutation(c.num_blocks)          # new id of old block b = perm[b]
    kp = np.empty_like(c.k_pool[0]); vp = np.empty_like(c.v_pool[0])
    kp[perm] = c.k_pool[0]; vp[perm] = c.v_pool[0]
    bt = np.where(c.block_tables >= 0, perm[np.maximum(c.block_tables, 0)], -1).astype(np.int32)
    a = oracle.paged_decode(c.q[0], c.k_pool[0], c.v_pool[0], c.block_tables, c.seq_lens, c.scale)
    b = oracle.paged_decode(c.q[0], kp, vp, bt, c.seq_lens, c.scale)
    assert np.array_equal(a, b)


def test_paged_equals_contiguous_slab():
    c = wl.custom([1, 17, 64, 200], 16, seed=16, append=True, nan_fill=True)
    kp, vp = oracle.paged_append(c.k_pool[0], c.v_pool[0], c.block_tables, c.positions,
                                 c.k_new[0], c.v_new[0])
    paged = oracle.paged_decode(c.q[0], kp, vp, c.block_tables, c.seq_lens, c.scale)
    ks, vs = wl.padded_slab(c, 0, width=256, fill_bits=wl.FP16_NAN_BITS)
    cont = oracle.contiguous_decode(c.q[0], ks, vs, c.seq_lens, c.scale)
    assert np.all(np.isfinite(paged))
    assert np.array_equal(paged, cont)


def test_unread_slots_do_not_matter():
    # NaN in every slot past each row's length (and in spare blocks) leaves the
    # result finite and equal to the same rows with ordinary filler.
    a = _rand_case(17, [3, 9, 16], 4, nan=True)
    b = _rand_case(17, [3, 9, 16], 4, nan=False)
    # same draws for the used tokens: copy used slots from a into b's pools
    for r in range(a.rows):
        for t in range(a.seq_lens[r]):
            pb, s = a.block_tables[r, t // 4], t % 4
            b.k_pool[0, pb, s] = a.k_pool[0, pb, s]
            b.v_pool[0, pb, s] = a.v_pool[0, pb, s]
    oa = oracle.paged_decode(a.q[0], a.k_pool[0], a.v_pool[0], a.block_tables, a.seq_lens, a.scale)
    ob = oracle.paged_decode(a.q[0], b.k_pool[0], b.v_pool[0], a.block_tables, a.seq_lens, a.scale)
    assert np.all(np.isfinite(oa))
    assert np.array_equal(oa, ob)


@pytest.mark.parametrize("chunk", [1, 3, 16, 64, 1000])
def test_blockwise_logsumexp_merge_equals_single_pass(chunk):
    c = wl.custom([1, 17, 64, 200], 16, seed=18, append=False, nan_fill=True)
    single = oracle.paged_decode(c.q[0], c.k_pool[0], c.v_pool[0], c.block_tables, c.seq_lens, c.scale)
    merged, lse = oracle.blockwise_decode(c.q[0], c.k_pool[0], c.v_pool[0], c.block_tables,
                                          c.seq_lens, c.scale, chunk)
    np.testing.assert_allclose(merged, single, rtol=1e-12, atol=1e-13)
    # lse is log sum exp of the scores, pinned against scipy's logsumexp
    r, h = 3, 7
    kvh = h // (c.q_heads // c.kv_heads)
    qv = oracle.half_to_double(c.q[0, r, h])
    s = [c.scale * np.dot(qv, oracle.half_to_double(c.k_pool[0, c.block_tables[r, t // 16], t % 16, kvh]))
         for t in range(c.seq_lens[r])]
    assert abs(lse[r, h] - scipy.special.logsumexp(s)) < 1e-11


def test_thread_count_does_not_change_results():
    c = wl.custom([33, 7, 120, 64, 5], 16, seed=19, append=False, nan_fill=True)
    a = oracle.paged_decode(c.q[0], c.k_pool[0], c.v_pool[0], c.block_tables, c.seq_lens, c.scale, 1)
    b = oracle.paged_decode(c.q[0], c.k_pool[0], c.v_pool[0], c.block_tables, c.seq_lens, c.scale, 4)
    assert np.array_equal(a, b)


def test_bad_table_entry_is_an_error_not_a_read():
    c = _rand_case(20, [5], 2)
    bt = c.block_tables.copy()
    bt[0, 1] = c.num_blocks  # out of range, and it is read (token 2..3)
    with pytest.raises(oracle.OracleError):
        oracle.paged_decode(c.q[0], c.k_pool[0], c.v_pool[0], bt, c.seq_lens, c.scale)
    bt[0, 1] = -1
    with pytest.raises(oracle.OracleError):
        oracle.paged_decode(c.q[0], c.k_pool[0], c.v_pool[0], bt, c.seq_lens, c.scale)


# --- append --------------------------------------------------------------------

def test_golden_hand_worked_append():
    g = json.load(open(os.path.join(GOLDEN, "append_hand.json")))
    nb, bs, hk, d = g["num_blocks"], g["block_size"], g["kv_heads"], g["head_dim"]
    kp = np.full((nb, bs, hk, d), wl.FP16_NAN_BITS, np.uint16)
    vp = kp.copy()
    k2, v2 = oracle.paged_append(kp, vp, np.array(g["block_tables"], np.int32),
                                 np.array(g["positions"], np.int32), _f16(g["k_new"]), _f16(g["v_new"]))
    ek, ev = kp.copy(), vp.copy()
    for w in g["expected_writes"]:
        ek[w["block"], w["slot"], 0] = _f16(w["k"])
        ev[w["block"], w["slot"], 0] = _f16(w["v"])
    assert np.array_equal(k2, ek) and np.array_equal(v2, ev)


def test_append_writes_only_the_target_slots():
    c = wl.tiny(nan_fill=True)
    kp, vp = oracle.paged_append(c.k_pool[0], c.v_pool[0], c.block_tables, c.positions,
                                 c.k_new[0], c.v_new[0])
    changed = np.argwhere(np.any(kp != c.k_pool[0], axis=(2, 3)))
    expect = sorted((int(c.block_tables[r, p // 16]), int(p % 16)) for r, p in enumerate(c.positions))
    assert sorted(map(tuple, changed.tolist())) == expect
    for r, p in enumerate(c.positions):
        pb = c.block_tables[r, p // 16]
        assert np.array_equal(kp[pb, p % 16], c.k_new[0, r])
        assert np.array_equal(vp[pb, p % 16], c.v_new[0, r])


def test_append_position_beyond_table_is_an_error():
    c = wl.custom([4], 4, seed=21, append=True, nan_fill=True)
    with pytest.raises(oracle.OracleError):
        oracle.paged_append(c.k_pool[0], c.v_pool[0], c.block_tables, np.array([4], np.int32),
                            c.k_new[0], c.v_new[0])


# --- copy-on-write block copy and prefill scatter -----------------------------

def test_golden_copy_on_write_pairs_in_order():
    g = json.load(open(os.path.join(GOLDEN, "cow_prefill_hand.json")))
    nb, bs, hk, d = g["num_blocks"], g["block_size"], g["kv_heads"], g["head_dim"]
    base = np.arange(nb * bs * hk * d, dtype=np.float32).reshape(nb, bs, hk, d)
    kp, vp = _f16(base), _f16(-base)
    k2, v2 = oracle.copy_blocks(kp, vp, g["cow"]["src"], g["cow"]["dst"])
    ek, ev = kp.copy(), vp.copy()
    for s, t in zip(g["cow"]["src"], g["cow"]["dst"]):
        ek[t] = ek[s]
        ev[t] = ev[s]
    assert np.array_equal(k2, ek) and np.array_equal(v2, ev)
    assert np.array_equal(k2[[1, 2, 4, 5]], kp[[1, 2, 4, 5]])


def test_copy_on_write_then_repoint_keeps_decode_exact():
    # cloning a shared block and repointing one row at the clone changes nothing
    c = wl.custom([20, 20], 8, seed=30, append=False, nan_fill=True, extra_blocks=4,
                  shared_tokens=16)
    shared = c.block_tables[1, 1]
    spare = c.num_blocks - 1
    kp, vp = oracle.copy_blocks(c.k_pool[0], c.v_pool[0], [shared], [spare])
    bt = c.block_tables.copy()
    bt[1, 1] = spare
    a = oracle.paged_decode(c.q[0], c.k_pool[0], c.v_pool[0], c.block_tables, c.seq_lens, c.scale)
    b = oracle.paged_decode(c.q[0], kp, vp, bt, c.seq_lens, c.scale)
    assert np.array_equal(a, b)


def test_copy_blocks_rejects_bad_ids():
    c = wl.custom([4], 4, seed=31, nan_fill=True)
    with pytest.raises(oracle.OracleError):
        oracle.copy_blocks(c.k_pool[0], c.v_pool[0], [0], [c.num_blocks])


def test_golden_prefill_scatter_drops_left_padding():
    g = json.load(open(os.path.join(GOLDEN, "cow_prefill_hand.json")))
    pf = g["prefill"]
    nb, bs, hk, d = g["num_blocks"], g["block_size"], g["kv_heads"], g["head_dim"]
    kp = np.full((nb, bs, hk, d), wl.FP16_NAN_BITS, np.uint16)
    ks = _f16(pf["k_src"])
    bt = np.array(pf["block_tables"], np.int32)
    # row 1 targets a -1 entry: an error, nothing written
    with pytest.raises(oracle.OracleError):
        oracle.prefill_scatter(kp, kp, bt, pf["src_start"], pf["dst_start"], pf["lengths"], ks, ks)
    lengths = [pf["lengths"][0], 0]
    k2, _ = oracle.prefill_scatter(kp, kp, bt, pf["src_start"], pf["dst_start"], lengths, ks, ks)
    ek = kp.copy()
    for w in pf["expected_writes_row0"]:
        ek[w["block"], w["slot"], 0] = _f16(w["k"])
    assert np.array_equal(k2, ek)


def test_prefill_scatter_then_gather_recovers_the_prompts():
    c = wl.custom([37, 5, 64, 1], 16, seed=32, append=False, nan_fill=True)
    rng = np.random.default_rng(3)
    width = 70
    ks = rng.standard_normal((c.rows, width, c.kv_heads, c.head_dim)).astype(np.float16)
    vs = rng.standard_normal((c.rows, width, c.kv_heads, c.head_dim)).astype(np.float16)
    lengths = c.seq_lens.copy()
    src_start = (width - lengths).astype(np.int32)      # left padded
    dst_start = np.zeros(c.rows, np.int32)
    kp, vp = oracle.prefill_scatter(c.k_pool[0], c.v_pool[0], c.block_tables, src_start, dst_start,
                                    lengths, ks, vs)
    import dataclasses
    c2 = dataclasses.replace(c, k_pool=kp[None], v_pool=vp[None])
    for r in range(c.rows):
        k, v = wl.logical_tokens(c2, 0, r)
        assert np.array_equal(k, ks[r, src_start[r]:].view(np.uint16))
        assert np.array_equal(v, vs[r, src_start[r]:].view(np.uint16))


# --- FP8 (E4M3) pools ----------------------------------------------------------
# The pages name FP8 KV without fixing a format ("PagedAttention", section
# "Checking it on a real system"); the oracle takes OCP E4M3 with one scale
# per KV head.  These pins tie it to the format's definition, to PyTorch's
# independent float8_e4m3fn conversion, and to the fp16 oracle.

def test_fp8_decode_matches_format_definition_values():
    c = oracle.fp8_e4m3_to_double
    expect = {0x00: 0.0, 0x01: 2.0 ** -9, 0x07: 7 * 2.0 ** -9, 0x08: 2.0 ** -6, 0x38: 1.0,
              0x39: 1.125, 0x3F: 1.875, 0x40: 2.0, 0x7E: 448.0, 0xFE: -448.0, 0xB8: -1.0}
    for code, v in expect.items():
        assert c([code])[0] == v, hex(code)
    assert np.isnan(c([0x7F, 0xFF])).all()
    assert math.copysign(1.0, c([0x80])[0]) == -1.0
    pos = c(np.arange(0x7F))
    assert np.all(np.diff(pos) > 0)  # finite non-negative codes increase


def test_fp8_decode_matches_torch_for_every_code():
    torch = pytest.importorskip("torch")
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).double().numpy()
    ours = oracle.fp8_e4m3_to_double(codes)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], ref[~nan])


def test_fp8_encode_rounds_to_nearest_even_and_saturates():
    enc = oracle.fp8_e4m3_from_float
    assert list(enc([1.0625, 1.1875, 1.03125])) == [0x38, 0x3A, 0x38]   # ties to even, below tie
    assert list(enc([2.0 ** -10, 1.5 * 2.0 ** -10, 2.0 ** -11])) == [0x00, 0x01, 0x00]
    assert list(enc([448.0, 449.0, 1000.0, -1e30])) == [0x7E, 0x7E, 0x7E, 0xFE]
    assert list(enc([-0.0, 0.0])) == [0x80, 0x00]
    finite = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], dtype=np.uint8)
    assert np.array_equal(enc(oracle.fp8_e4m3_to_double(finite).astype(np.float32)), finite)


def test_fp8_encode_matches_torch_in_range():
    torch = pytest.importorskip("torch")
    g = torch.Generator().manual_seed(3)
    y = torch.randn(20000, generator=g) * torch.exp2(torch.randint(-12, 9, (20000,), generator=g).float())
    y = y[y.abs() <= 448].float()
    ref = y.to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(oracle.fp8_e4m3_from_float(y.numpy()), ref)


def test_fp8_quantize_divides_in_binary32_first():
    x = np.array([0.1, -3.0, 250.0, 1e-4], dtype=np.float16)
    s = np.float32(0.37)
    expect = oracle.fp8_e4m3_from_float(x.astype(np.float32) / s)
    assert np.array_equal(oracle.fp8_quantize(x, s), expect)


def test_fp8_quantize_matches_torch_on_many_draws_and_near_ties():
    # The quotient x / s is formed in binary32 and then rounded to E4M3
    # (nearest, ties to even).  PyTorch does the same independently:
    # (x.float() / s).to(float8_e4m3fn).  Compared on 2e5 fp16 draws over many
    # binades and on fp16 values whose quotient lies within a few binary32
    # ulps of an E4M3 rounding tie, where a quotient formed in double
    # precision (or rounded twice) would pick the other neighbour.  Only
    # quotients inside the E4M3 range are compared: beyond it the oracle
    # saturates and PyTorch's conversion does not.
    torch = pytest.importorskip("torch")
    g = torch.Generator().manual_seed(11)
    xs = []
    for _ in range(4):
        e = torch.randint(-14, 16, (50000,), generator=g).float()
        xs.append((torch.randn(50000, generator=g) * torch.exp2(e)).to(torch.float16))
    # near ties: midpoints between neighbouring positive E4M3 values, times s,
    # rounded to fp16, and the fp16 values one and two steps either side
    codes = np.arange(0x01, 0x7E, dtype=np.uint8)
    vals = oracle.fp8_e4m3_to_double(codes)
    mids = (vals[:-1] + vals[1:]) / 2
    for s in (np.float32(0.37), np.float32(0.0123), np.float32(1.0), np.float32(3.3)):
        base = torch.from_numpy(mids * float(s)).to(torch.float16)
        near = [base]
        bits16 = base.view(torch.int16)
        for k in (-2, -1, 1, 2):
            near.append((bits16 + k).view(torch.float16))
        near = torch.cat(near)
        near = torch.cat([near, -near])
        for x in xs + [near]:
            q = x.float() / torch.tensor(s)
            keep = torch.isfinite(q) & (q.abs() <= 448)
            x = x[keep]
            ref = (x.float() / torch.tensor(s)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
            ours = oracle.fp8_quantize(x.view(torch.int16).numpy().view(np.float16), s)
            assert np.array_equal(ours, ref), f"scale {s}: {int((ours != ref).sum())} of {ref.size} differ"


def test_fp8_append_writes_quantised_slots_only():
    rng = np.random.default_rng(4)
    nb, bs, hk, d, rows = 6, 16, 2, 8, 3
    kp = rng.integers(0, 0x7E, (nb, bs, hk, d), dtype=np.uint8)
    vp = rng.integers(0, 0x7E, (nb, bs, hk, d), dtype=np.uint8)
    bt = np.array([[4, 1], [0, 5], [2, 3]], dtype=np.int32)
    pos = np.array([17, 3, -1], dtype=np.int32)
    kn = _f16(rng.standard_normal((rows, hk, d)))
    vn = _f16(rng.standard_normal((rows, hk, d)))
    ks = np.array([0.05, 0.2], dtype=np.float32)
    vs = np.array([0.1, 0.01], dtype=np.float32)
    k2, v2 = oracle.paged_append_fp8(kp, vp, ks, vs, bt, pos, kn, vn)
    ek, ev = kp.copy(), vp.copy()
    for r, (b, o) in enumerate([(1, 1), (0, 3)]):
        for h in range(hk):
            ek[b, o, h] = oracle.fp8_quantize(kn[r, h].view(np.float16), ks[h])
            ev[b, o, h] = oracle.fp8_quantize(vn[r, h].view(np.float16), vs[h])
    assert np.array_equal(k2, ek) and np.array_equal(v2, ev)


def test_fp8_decode_equals_fp16_decode_on_exactly_representable_pools():
    # E4M3 values times a power-of-two scale are exact in fp16 (within its
    # range), so the FP8 decode must equal the fp16 oracle on those values.
    rng = np.random.default_rng(5)
    lengths, bs, hq, hk, d = [1, 17, 40], 16, 4, 2, 8
    case = _rand_case(9, lengths, bs, hq=hq, hk=hk, d=d, nan=False)
    nb = case.k_pool[0].shape[0]
    finite = np.array([c for c in range(256) if (c & 0x7F) != 0x7F and (c & 0x78) >= 0x20], dtype=np.uint8)
    kp8 = rng.choice(finite, (nb, bs, hk, d))
    vp8 = rng.choice(finite, (nb, bs, hk, d))
    ks = np.array([0.25, 2.0], dtype=np.float32)
    vs = np.array([0.5, 0.125], dtype=np.float32)
    kf = (oracle.fp8_e4m3_to_double(kp8) * ks[None, None, :, None]).astype(np.float16)
    vf = (oracle.fp8_e4m3_to_double(vp8) * vs[None, None, :, None]).astype(np.float16)
    assert np.array_equal(kf.astype(np.float64), oracle.fp8_e4m3_to_double(kp8) * ks[None, None, :, None])
    a = oracle.paged_decode_fp8(case.q[0], kp8, vp8, ks, vs, case.block_tables, case.seq_lens, case.scale)
    b = oracle.paged_decode(case.q[0], kf, vf, case.block_tables, case.seq_lens, case.scale)
    assert np.max(np.abs(a - b)) <= 1e-12


def test_fp8_decode_scales_output_with_v_scale():
    rng = np.random.default_rng(6)
    case = _rand_case(11, [5, 30], 16, hq=4, hk=2, d=8, nan=False)
    nb = case.k_pool[0].shape[0]
    kp8 = rng.integers(0x20, 0x60, (nb, 16, 2, 8), dtype=np.uint8)
    vp8 = rng.integers(0x20, 0x60, (nb, 16, 2, 8), dtype=np.uint8)
    ks = np.array([0.3, 0.7], dtype=np.float32)
    a = oracle.paged_decode_fp8(case.q[0], kp8, vp8, ks, np.array([1.0, 1.0], np.float32),
                                case.block_tables, case.seq_lens, case.scale)
    b = oracle.paged_decode_fp8(case.q[0], kp8, vp8, ks, np.array([3.0, 0.5], np.float32),
                                case.block_tables, case.seq_lens, case.scale)
    assert np.allclose(b[:, :2], 3.0 * a[:, :2], rtol=1e-13, atol=0)
    assert np.allclose(b[:, 2:], 0.5 * a[:, 2:], rtol=1e-13, atol=0)


# --- chunked prefill (several queries per row, causal within the chunk) ---------

def _prefill_case(seed, lengths, chunks, bs, hq=4, hk=2, d=8):
    c = _rand_case(seed, lengths, bs, hq=hq, hk=hk, d=d, nan=True)
    rng = np.random.default_rng(seed)
    qs = np.concatenate([[0], np.cumsum(chunks)]).astype(np.int32)
    q = _f16(rng.standard_normal((int(qs[-1]), hq, d)))
    return c, q, qs


@pytest.mark.parametrize("seed,lengths,chunks,bs", [
    (1, [5, 9], [5, 3], 4), (2, [7, 1, 12], [2, 1, 12], 4), (3, [20], [7], 8)])
def test_prefill_matches_pure_python_brute_force(seed, lengths, chunks, bs):
    c, q, qs = _prefill_case(seed, lengths, chunks, bs)
    ours = oracle.paged_prefill(q, c.k_pool[0], c.v_pool[0], c.block_tables, c.seq_lens, qs, c.scale)
    ref = np.array(brute.paged_prefill(q.tolist(), c.k_pool[0].tolist(), c.v_pool[0].tolist(),
                                       c.block_tables.tolist(), c.seq_lens.tolist(), qs.tolist(),
                                       c.scale)).reshape(ours.shape)
    np.testing.assert_allclose(ours, ref, rtol=1e-12, atol=1e-12)


def test_prefill_chunk_of_one_is_decode():
    c, q, qs = _prefill_case(4, [1, 17, 40], [1, 1, 1], 16)
    ours = oracle.paged_prefill(q, c.k_pool[0], c.v_pool[0], c.block_tables, c.seq_lens, qs, c.scale)
    dec = oracle.paged_decode(q, c.k_pool[0], c.v_pool[0], c.block_tables, c.seq_lens, c.scale)
    np.testing.assert_allclose(ours, dec, rtol=0, atol=0)


def test_prefill_whole_prompt_is_causal_self_attention():
    # A chunk that is the whole prompt: masked softmax(q k^T) v over the
    # gathered tokens, computed with dense matrix products.
    L, bs, hq, hk, d = 37, 8, 4, 2, 8
    c, q, qs = _prefill_case(5, [L], [L], bs, hq, hk, d)
    ours = oracle.paged_prefill(q, c.k_pool[0], c.v_pool[0], c.block_tables, c.seq_lens, qs, c.scale)
    K = np.empty((L, hk, d)); V = np.empty((L, hk, d))
    for t in range(L):
        pb = c.block_tables[0, t // bs]
        K[t] = oracle.half_to_double(c.k_pool[0][pb, t % bs])
        V[t] = oracle.half_to_double(c.v_pool[0][pb, t % bs])
    Q = oracle.half_to_double(q)
    mask = np.tril(np.ones((L, L), dtype=bool))
    for h in range(hq):
        kvh = h // (hq // hk)
        s = c.scale * Q[:, h, :] @ K[:, kvh, :].T
        s = np.where(mask, s, -np.inf)
        p = scipy.special.softmax(s, axis=1)
        np.testing.assert_allclose(ours[:, h, :], p @ V[:, kvh, :], rtol=1e-12, atol=1e-13)


def test_prefill_last_query_equals_decode_of_the_row():
    c, q, qs = _prefill_case(6, [33, 64, 9], [8, 16, 9], 16)
    ours = oracle.paged_prefill(q, c.k_pool[0], c.v_pool[0], c.block_tables, c.seq_lens, qs, c.scale)
    last = q[qs[1:] - 1]
    dec = oracle.paged_decode(last, c.k_pool[0], c.v_pool[0], c.block_tables, c.seq_lens, c.scale)
    np.testing.assert_allclose(ours[qs[1:] - 1], dec, rtol=0, atol=0)


def test_prefill_rejects_chunk_longer_than_row():
    c, q, qs = _prefill_case(7, [4, 6], [5, 1], 4)
    with pytest.raises(oracle.OracleError):
        oracle.paged_prefill(q, c.k_pool[0], c.v_pool[0], c.block_tables, c.seq_lens, qs, c.scale)
