"""Pure-Python brute force for paged decode attention -- TEST INFRASTRUCTURE.

An independent restatement used only to pin the C oracle on tiny inputs.  It
differs from the C oracle on purpose in every step a mistake could hide in:

  * fp16 bits are decoded by ``struct`` ('e' format), not by the C bit
    arithmetic;
  * the block table is walked per physical block (block by block, slot by
    slot) instead of per logical token;
  * the softmax is exp(s) / sum exp(s) without subtracting the maximum
    (valid for the small scores of tiny test inputs);
  * tokens are summed in reverse logical order.

Source: "PagedAttention" (deepconcepts.dev), "PagedAttention": logical block
n of a sequence lives in the physical block its table lists; the attention
result is that of ordinary attention over the sequence's tokens.
"""
from __future__ import annotations

import math
import struct


def half_bits_to_float(bits: int) -> float:
    return struct.unpack("<e", struct.pack("<H", int(bits) & 0xFFFF))[0]


def paged_decode(q, k_pool, v_pool, block_tables, seq_lens, scale):
    """q: nested [rows][Hq][D] uint16 bits; pools [nb][bs][Hk][D]; returns floats."""
    rows = len(q)
    hq = len(q[0])
    d = len(q[0][0])
    bs = len(k_pool[0])
    hk = len(k_pool[0][0])
    group = hq // hk
    out = []
    for r in range(rows):
        L = int(seq_lens[r])
        # Collect (K, V) vectors block by block.
        toks = []
        nblk = (L + bs - 1) // bs
        for lb in range(nblk):
            pb = int(block_tables[r][lb])
            used = min(bs, L - lb * bs)
            for slot in range(used):
                toks.append((pb, slot))
        row_out = []
        for h in range(hq):
            kvh = h // group
            qv = [half_bits_to_float(x) for x in q[r][h]]
            weights = []
            for (pb, slot) in toks:
                kv = k_pool[pb][slot][kvh]
                s = 0.0
                for i in range(d):
                    s += qv[i] * half_bits_to_float(kv[i])
                weights.append(math.exp(scale * s))
            z = math.fsum(weights)
            o = [0.0] * d
            for idx in range(len(toks) - 1, -1, -1):
                pb, slot = toks[idx]
                vv = v_pool[pb][slot][kvh]
                w = weights[idx] / z
                for i in range(d):
                    o[i] += w * half_bits_to_float(vv[i])
            row_out.append(o)
        out.append(row_out)
    return out


def paged_prefill(q, k_pool, v_pool, block_tables, seq_lens, q_start, scale):
    """Causal chunk attention, brute force: q nested [total][Hq][D] bits.

    For each query the visible tokens are gathered block by block, the
    softmax is taken without max subtraction and summed in reverse order,
    as in paged_decode above."""
    out = []
    rows = len(seq_lens)
    for r in range(rows):
        lo, hi = int(q_start[r]), int(q_start[r + 1])
        C = hi - lo
        for i in range(C):
            pos = int(seq_lens[r]) - C + i
            # a decode of this single query over tokens 0..pos
            out.append(paged_decode([q[lo + i]], k_pool, v_pool, [block_tables[r]], [pos + 1],
                                    scale)[0])
    return out
