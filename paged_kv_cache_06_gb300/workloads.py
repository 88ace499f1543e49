"""Seeded synthetic workloads for paged decode attention.

This module only *generates inputs*: row lengths, a block-table layout and
fp16 values.  It holds none of the attention arithmetic, so the CUDA path and
the fp64 oracle can both be fed from it without sharing any of the method.

Shapes follow the serving workloads of the "Paged attention" page
(danielfleming.xyz): Qwen2.5-1.5B heads (12 query heads over 2 KV heads,
head_dim 128, fp16, 28 layers), 32 batch rows, prompts up to 4096 tokens,
64-token blocks; and the "PagedAttention" page (deepconcepts.dev): 16-token
blocks and a shared system-prompt prefix shared in whole blocks.

Every draw comes from one CPU ``torch.Generator`` seeded with ``seed`` in a
fixed order (lengths, block permutation, then per layer q, cached K, cached V,
new K, new V), values drawn as fp32 N(0,1) and rounded to fp16, so a case is
bit-identical on every machine.

Layout produced:
  * pools ``[layers][num_blocks][block_size][kv_heads][head_dim]`` fp16
    (as uint16 bit patterns), one pool per layer, separate K and V;
  * ``block_tables [rows][max_blocks_per_row]`` int32, -1 where unused, the
    same table for every layer (a block id names the same slot range in every
    layer's pool);
  * ``seq_lens [rows]`` = tokens in the row *including* this step's new token;
  * ``positions [rows]`` = where this step's new token goes (seq_len - 1), or
    -1 for cases without an append;
  * before the append the pool slot at ``positions[r]`` holds filler (NaN in
    ``nan_fill`` mode), so only a correct append makes decode right.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Dict, List, Optional

import numpy as np
import torch

Q_HEADS = 12
KV_HEADS = 2
HEAD_DIM = 128
FP16_NAN_BITS = 0x7E00


def default_scale(head_dim: int = HEAD_DIM) -> float:
    """1/sqrt(head_dim) rounded to fp32 (the value passed to the kernel)."""
    return float(np.float32(1.0 / math.sqrt(head_dim)))


@dataclasses.dataclass
class DecodeCase:
    name: str
    block_size: int
    num_blocks: int
    layers: int
    q_heads: int
    kv_heads: int
    head_dim: int
    seq_lens: np.ndarray        # int32 [rows]
    positions: np.ndarray       # int32 [rows], -1 = no append
    block_tables: np.ndarray    # int32 [rows][max_blocks_per_row]
    q: np.ndarray               # uint16 [layers][rows][Hq][D]
    k_pool: np.ndarray          # uint16 [layers][nb][bs][Hk][D]  (before append)
    v_pool: np.ndarray
    k_new: np.ndarray           # uint16 [layers][rows][Hk][D]
    v_new: np.ndarray
    scale: float
    shared_blocks: int = 0      # leading table entries shared by every row
    nan_fill: bool = False

    @property
    def rows(self) -> int:
        return int(self.seq_lens.shape[0])

    @property
    def max_blocks_per_row(self) -> int:
        return int(self.block_tables.shape[1])

    @property
    def max_seq_len(self) -> int:
        return int(self.seq_lens.max()) if self.rows else 0

    @property
    def has_append(self) -> bool:
        return bool((self.positions >= 0).any())

    def blocks_per_row(self) -> np.ndarray:
        return (self.seq_lens.astype(np.int64) + self.block_size - 1) // self.block_size

    def unique_blocks(self) -> int:
        used = set()
        for r, n in enumerate(self.blocks_per_row()):
            used.update(int(x) for x in self.block_tables[r, :n])
        return len(used)


def _randn_fp16(gen: torch.Generator, shape) -> np.ndarray:
    t = torch.randn(tuple(shape), generator=gen, dtype=torch.float32).to(torch.float16)
    return t.numpy().view(np.uint16)


def fp8_codes(gen: torch.Generator, shape) -> np.ndarray:
    """Seeded random E4M3 codes for FP8 pools: a random sign bit, exponent
    field uniform in 3..10 and mantissa field uniform in 0..7, so that with a
    scale near 1/8 the stored values have magnitudes like N(0, 1) draws.
    Pure bit assembly: no quantisation happens here."""
    shape = tuple(shape)
    sign = torch.randint(0, 2, shape, generator=gen, dtype=torch.int32)
    expo = torch.randint(3, 11, shape, generator=gen, dtype=torch.int32)
    mant = torch.randint(0, 8, shape, generator=gen, dtype=torch.int32)
    return ((sign << 7) | (expo << 3) | mant).to(torch.uint8).numpy()


def _assign_tables(lengths: np.ndarray, block_size: int, perm: np.ndarray,
                   max_blocks_per_row: int, shared_ids: Optional[np.ndarray] = None
                   ) -> np.ndarray:
    """Give each row ceil(L/bs) physical ids, taken from ``perm`` in order.

    With ``shared_ids`` the first entries of every row point at those shared
    ids (only as many as the row's length needs); the remainder are private.
    """
    rows = lengths.shape[0]
    tables = np.full((rows, max_blocks_per_row), -1, dtype=np.int32)
    cursor = 0
    n_shared = 0 if shared_ids is None else shared_ids.shape[0]
    for r in range(rows):
        need = (int(lengths[r]) + block_size - 1) // block_size
        k = min(need, n_shared)
        if k:
            tables[r, :k] = shared_ids[:k]
        priv = need - k
        tables[r, k:need] = perm[cursor:cursor + priv]
        cursor += priv
    return tables


def _make_case(name: str, lengths: np.ndarray, block_size: int, num_blocks: int,
               layers: int, gen: torch.Generator, perm_blocks: int,
               append: bool, nan_fill: bool, shared_tokens: int = 0,
               max_blocks_per_row: Optional[int] = None,
               q_heads: int = Q_HEADS, kv_heads: int = KV_HEADS,
               head_dim: int = HEAD_DIM) -> DecodeCase:
    rows = lengths.shape[0]
    bs = block_size
    need = (lengths.astype(np.int64) + bs - 1) // bs
    if max_blocks_per_row is None:
        max_blocks_per_row = int(max(1, need.max() if rows else 1))
    perm = torch.randperm(perm_blocks, generator=gen).numpy().astype(np.int32)
    shared_ids = None
    n_shared_blocks = shared_tokens // bs
    if n_shared_blocks:
        shared_ids = perm[:n_shared_blocks]
        perm = perm[n_shared_blocks:]
    tables = _assign_tables(lengths, bs, perm, max_blocks_per_row, shared_ids)
    positions = (lengths.astype(np.int32) - 1) if append else np.full(rows, -1, np.int32)
    positions = np.where(lengths > 0, positions, -1).astype(np.int32)

    q = np.empty((layers, rows, q_heads, head_dim), dtype=np.uint16)
    fill = FP16_NAN_BITS if nan_fill else None
    kp = np.empty((layers, num_blocks, bs, kv_heads, head_dim), dtype=np.uint16)
    vp = np.empty_like(kp)
    kn = np.empty((layers, rows, kv_heads, head_dim), dtype=np.uint16)
    vn = np.empty_like(kn)
    for layer in range(layers):
        q[layer] = _randn_fp16(gen, (rows, q_heads, head_dim))
        if fill is not None:
            kp[layer].fill(fill)
            vp[layer].fill(fill)
        else:
            kp[layer] = _randn_fp16(gen, kp.shape[1:])
            vp[layer] = _randn_fp16(gen, vp.shape[1:])
        # Shared prefix tokens: one draw, written into the shared blocks.
        if n_shared_blocks:
            ks = _randn_fp16(gen, (n_shared_blocks * bs, kv_heads, head_dim))
            vs = _randn_fp16(gen, (n_shared_blocks * bs, kv_heads, head_dim))
            for lb in range(n_shared_blocks):
                pb = int(shared_ids[lb])
                kp[layer, pb] = ks[lb * bs:(lb + 1) * bs]
                vp[layer, pb] = vs[lb * bs:(lb + 1) * bs]
        for r in range(rows):
            L = int(lengths[r])
            first_private = min(int(need[r]), n_shared_blocks) * bs
            n_priv = max(0, L - first_private)
            if n_priv == 0:
                continue
            kt = _randn_fp16(gen, (n_priv, kv_heads, head_dim))
            vt = _randn_fp16(gen, (n_priv, kv_heads, head_dim))
            for lb in range(first_private // bs, int(need[r])):
                pb = int(tables[r, lb])
                t0 = lb * bs
                n = min(bs, L - t0)
                kp[layer, pb, :n] = kt[t0 - first_private:t0 - first_private + n]
                vp[layer, pb, :n] = vt[t0 - first_private:t0 - first_private + n]
        kn[layer] = _randn_fp16(gen, (rows, kv_heads, head_dim))
        vn[layer] = _randn_fp16(gen, (rows, kv_heads, head_dim))
        # The appended position holds filler until the append runs.
        for r in range(rows):
            pos = int(positions[r])
            if pos < 0:
                continue
            pb = int(tables[r, pos // bs])
            if fill is not None:
                kp[layer, pb, pos % bs] = fill
                vp[layer, pb, pos % bs] = fill
    return DecodeCase(name=name, block_size=bs, num_blocks=num_blocks, layers=layers,
                      q_heads=q_heads, kv_heads=kv_heads, head_dim=head_dim,
                      seq_lens=lengths.astype(np.int32), positions=positions,
                      block_tables=tables, q=q, k_pool=kp, v_pool=vp, k_new=kn, v_new=vn,
                      scale=default_scale(head_dim), shared_blocks=n_shared_blocks,
                      nan_fill=nan_fill)


# ---------------------------------------------------------------------------
# The five named workloads.

def tiny(seed: int = 0, nan_fill: bool = True) -> DecodeCase:
    """1 layer; rows of 1, 17, 64, 200 tokens; 16-token blocks; 64-block pool;
    one append per row (at L-1) before decode."""
    gen = torch.Generator().manual_seed(seed)
    lengths = np.array([1, 17, 64, 200], dtype=np.int32)
    return _make_case("tiny", lengths, 16, 64, 1, gen, 64, append=True, nan_fill=nan_fill)


def uniform(seed: int = 0, layers: int = 28, nan_fill: bool = False) -> DecodeCase:
    """32 rows of 1024 tokens, 64-token blocks, 512-block pool per layer."""
    gen = torch.Generator().manual_seed(seed)
    lengths = np.full(32, 1024, dtype=np.int32)
    return _make_case("uniform", lengths, 64, 512, layers, gen, 512, append=True,
                      nan_fill=nan_fill)


def mixed_lengths(gen: torch.Generator) -> np.ndarray:
    """31 lengths uniform on the integers 16..512 plus one 4096-token row at a
    seeded index (the pages' ragged draw with one long prompt)."""
    short = torch.randint(16, 513, (31,), generator=gen).numpy()
    where = int(torch.randint(0, 32, (1,), generator=gen).item())
    return np.insert(short, where, 4096).astype(np.int32)


def mixed(seed: int = 0, layers: int = 28, nan_fill: bool = False) -> DecodeCase:
    """32 rows: 31 lengths U{16..512} and one of 4096; 64-token blocks; pool
    holding exactly the blocks needed; 28 layers."""
    gen = torch.Generator().manual_seed(seed)
    lengths = mixed_lengths(gen)
    nb = int(((lengths.astype(np.int64) + 63) // 64).sum())
    return _make_case("mixed", lengths, 64, nb, layers, gen, nb, append=True,
                      nan_fill=nan_fill)


SHARED_PREFIX_TOKENS = 592  # 37 whole 16-token blocks


def shared_lengths(gen: torch.Generator, rows: int = 96) -> np.ndarray:
    """Log-uniform lengths on [16, 8192]: floor(exp(U(ln 16, ln 8192)))."""
    u = torch.rand(rows, generator=gen, dtype=torch.float64).numpy()
    lo, hi = math.log(16.0), math.log(8192.0)
    return np.floor(np.exp(lo + u * (hi - lo))).astype(np.int32)


def shared(seed: int = 0, nan_fill: bool = False, rows: int = 96) -> DecodeCase:
    """96 rows, log-uniform lengths in [16, 8192], 16-token blocks, the first
    37 table entries of every row pointing at the same 37 physical blocks."""
    gen = torch.Generator().manual_seed(seed)
    lengths = shared_lengths(gen, rows)
    bs = 16
    nshared = SHARED_PREFIX_TOKENS // bs
    need = (lengths.astype(np.int64) + bs - 1) // bs
    nb = nshared + int(np.maximum(need - nshared, 0).sum())
    return _make_case("shared", lengths, bs, nb, 1, gen, nb, append=False,
                      nan_fill=nan_fill, shared_tokens=SHARED_PREFIX_TOKENS)


def long(seed: int = 0, nan_fill: bool = False, cached: int = 32768, rows: int = 4) -> DecodeCase:
    """4 rows with 32768 cached tokens; one append at position 32768, then
    decode over 32769 tokens (513 blocks of 64)."""
    gen = torch.Generator().manual_seed(seed)
    lengths = np.full(rows, cached + 1, dtype=np.int32)
    bs = 64
    nb = int(((lengths.astype(np.int64) + bs - 1) // bs).sum())
    return _make_case("long", lengths, bs, nb, 1, gen, nb, append=True, nan_fill=nan_fill)


def custom(lengths, block_size: int, seed: int = 0, layers: int = 1, append: bool = True,
           nan_fill: bool = True, extra_blocks: int = 0, max_blocks_per_row: Optional[int] = None,
           q_heads: int = Q_HEADS, kv_heads: int = KV_HEADS, head_dim: int = HEAD_DIM,
           shared_tokens: int = 0) -> DecodeCase:
    """Any lengths / block size; pool = blocks needed + ``extra_blocks``."""
    gen = torch.Generator().manual_seed(seed)
    lengths = np.asarray(lengths, dtype=np.int32)
    need = (lengths.astype(np.int64) + block_size - 1) // block_size
    n_sh = shared_tokens // block_size
    nb = n_sh + int(np.maximum(need - n_sh, 0).sum()) + extra_blocks
    nb = max(nb, 1)
    return _make_case("custom", lengths, block_size, nb, layers, gen, nb, append=append,
                      nan_fill=nan_fill, shared_tokens=shared_tokens,
                      max_blocks_per_row=max_blocks_per_row, q_heads=q_heads,
                      kv_heads=kv_heads, head_dim=head_dim)


WORKLOADS = {
    "tiny": tiny,
    "uniform": uniform,
    "mixed": mixed,
    "shared": shared,
    "long": long,
}


def logical_tokens(case: DecodeCase, layer: int, r: int):
    """Row r's K and V in logical order after the append, as [L][Hk][D] bits.

    Input plumbing for building a padded slab; the table is read exactly as
    the layout above defines it (block table[r][t // bs], slot t % bs).
    """
    L = int(case.seq_lens[r])
    bs = case.block_size
    k = np.empty((L, case.kv_heads, case.head_dim), dtype=np.uint16)
    v = np.empty_like(k)
    for lb in range((L + bs - 1) // bs):
        pb = int(case.block_tables[r, lb])
        n = min(bs, L - lb * bs)
        k[lb * bs:lb * bs + n] = case.k_pool[layer, pb, :n]
        v[lb * bs:lb * bs + n] = case.v_pool[layer, pb, :n]
    pos = int(case.positions[r])
    if pos >= 0:
        k[pos] = case.k_new[layer, r]
        v[pos] = case.v_new[layer, r]
    return k, v


def padded_slab(case: DecodeCase, layer: int, width: Optional[int] = None,
                fill_bits: int = 0):
    """The same rows in a contiguous [rows][width][Hk][D] slab (the layout of
    the "Continuous batching" page's cache), padded with ``fill_bits``."""
    width = case.max_seq_len if width is None else width
    ks = np.full((case.rows, width, case.kv_heads, case.head_dim), fill_bits, dtype=np.uint16)
    vs = np.full_like(ks, fill_bits)
    for r in range(case.rows):
        k, v = logical_tokens(case, layer, r)
        ks[r, :k.shape[0]] = k
        vs[r, :v.shape[0]] = v
    return ks, vs


def algorithmic_bytes(case: DecodeCase) -> Dict[str, int]:
    """Bytes the method must move per layer (decode) and per step.

    KV: sum_r L_r * Hk * D * 2 B * 2 (K and V); plus q and out (rows*Hq*D*2 B
    each), the table entries read (4 B * ceil(L/bs)) and seq_lens (4 B/row).
    ``kv_unique`` counts each distinct physical block's used slots once.
    """
    L = case.seq_lens.astype(np.int64)
    tok_bytes = case.kv_heads * case.head_dim * 2 * 2
    kv = int(L.sum()) * tok_bytes
    # unique: every distinct block counted at the max slots any row uses in it
    used: Dict[int, int] = {}
    bs = case.block_size
    for r in range(case.rows):
        for lb in range(int((L[r] + bs - 1) // bs)):
            pb = int(case.block_tables[r, lb])
            n = int(min(bs, L[r] - lb * bs))
            used[pb] = max(used.get(pb, 0), n)
    kv_unique = sum(used.values()) * tok_bytes
    qo = 2 * case.rows * case.q_heads * case.head_dim * 2
    table = int(((L + bs - 1) // bs).sum()) * 4 + 4 * case.rows
    append = int((case.positions >= 0).sum()) * case.kv_heads * case.head_dim * 2 * 2 * 2
    return {
        "kv_logical": kv,
        "kv_unique": kv_unique,
        "q_out": qo,
        "table": table,
        "decode_layer": kv + qo + table,
        "decode_layer_unique": kv_unique + qo + table,
        "append_layer": append,
    }


def to_device(case: DecodeCase, device="cuda") -> Dict[str, "torch.Tensor"]:
    """Copy a case's arrays to the device as fp16 / int32 torch tensors."""
    def f16(a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.float16)).to(device)

    def i32(a):
        return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).to(device)

    return {
        "q": f16(case.q), "k_pool": f16(case.k_pool), "v_pool": f16(case.v_pool),
        "k_new": f16(case.k_new), "v_new": f16(case.v_new),
        "block_tables": i32(case.block_tables), "seq_lens": i32(case.seq_lens),
        "positions": i32(case.positions),
    }


def row_subset(case: DecodeCase, rows) -> DecodeCase:
    """The same case restricted to some rows (pools unchanged)."""
    rows = np.asarray(rows)
    return dataclasses.replace(case, seq_lens=case.seq_lens[rows].copy(),
                               positions=case.positions[rows].copy(),
                               block_tables=case.block_tables[rows].copy(),
                               q=case.q[:, rows].copy(), k_new=case.k_new[:, rows].copy(),
                               v_new=case.v_new[:, rows].copy())
