"""The FP8 decode's per-lane dim orders, checked on the CPU.

The FP8 attend builds its tensor-core fragments straight from the E4M3 bytes
of a staged granule (16 token rows of 128 bytes, 16-byte chunk c of row r
stored at r*128 + 16*(c ^ (r % 8))).  It takes the dims of the QK product in
a per-lane order (lane (g, t) reads bytes 32t .. 32t+31 of K rows g and g+8;
its word ks feeds k-step ks) and loads the queries in the same order, and it
lets row g of PV m-tile i stand for output dim 16g + 2i and row g + 8 for
16g + 2i + 1 (each lane reads chunk g of V rows 2t, 2t+1, 8+2t, 9+2t and
pairs their bytes across tokens), undoing that order when it stores the
output.

This test restates those reads lane by lane, assembles the m16n8k16 operand
matrices from the fragments in the layout the PTX ISA gives for
mma.sync.m16n8k16 (A row-major 16x16, B column-major 16x8, C 16x8; lane l has
groupID l // 4 and threadID_in_group l % 4), and checks that the products
equal K.Q^T and P^T.V exactly: every dim is used once, by matching K and Q
elements, and every output lands on its own dim and head.  Small integers
keep the float arithmetic exact.
"""
import numpy as np


def swizzled_box(rows):
    """16 x 128 bytes -> the 2 KB staged box (128-byte swizzle)."""
    box = np.zeros(2048, dtype=np.int64)
    for r in range(16):
        for c in range(8):
            pos = r * 128 + 16 * (c ^ (r % 8))
            box[pos:pos + 16] = rows[r, 16 * c:16 * c + 16]
    return box


def chunk(box, r, c):
    """The 16 bytes of chunk c of row r, read back from the swizzled box."""
    pos = r * 128 + 16 * (c ^ (r % 8))
    return box[pos:pos + 16]


def test_qk_dim_order_pairs_k_with_q():
    rng = np.random.default_rng(0)
    K = rng.integers(-8, 9, size=(16, 128))  # 16 tokens x 128 dims
    Q = rng.integers(-8, 9, size=(8, 128))   # 8 heads x 128 dims
    kbox = swizzled_box(K)
    S = np.zeros((16, 8), dtype=np.int64)
    for ks in range(8):
        A = np.full((16, 16), 10**9, dtype=np.int64)  # sentinel: every element must be written
        B = np.full((16, 8), 10**9, dtype=np.int64)
        for lane in range(32):
            g, t = lane // 4, lane % 4
            h, j = ks // 4, ks % 4
            # bytes 32t + 16h .. +15 of rows g and g + 8: chunk 2t + h
            w0 = chunk(kbox, g, 2 * t + h)[4 * j:4 * j + 4]
            w1 = chunk(kbox, g + 8, 2 * t + h)[4 * j:4 * j + 4]
            # low half of a word -> cols 2t, 2t+1; high half -> cols 8+2t, 9+2t
            A[g, 2 * t:2 * t + 2] = w0[0:2]
            A[g, 8 + 2 * t:8 + 2 * t + 2] = w0[2:4]
            A[g + 8, 2 * t:2 * t + 2] = w1[0:2]
            A[g + 8, 8 + 2 * t:8 + 2 * t + 2] = w1[2:4]
            # queries: halves 32t .. 32t+31 of head g; word 2ks -> b0 b1, word 2ks+1 -> b2 b3
            q = Q[g, 32 * t:32 * t + 32]
            B[2 * t:2 * t + 2, g] = q[4 * ks:4 * ks + 2]
            B[8 + 2 * t:8 + 2 * t + 2, g] = q[4 * ks + 2:4 * ks + 4]
        assert (A != 10**9).all() and (B != 10**9).all()
        S += A @ B
    assert np.array_equal(S, K @ Q.T)


def test_pv_dim_order_and_the_output_store():
    rng = np.random.default_rng(1)
    V = rng.integers(-8, 9, size=(16, 128))  # 16 tokens x 128 dims
    P = rng.integers(0, 5, size=(16, 8))     # 16 tokens x 8 heads
    vbox = swizzled_box(V)
    out = np.full((8, 128), 10**9, dtype=np.int64)
    for i in range(8):  # m-tile
        A = np.full((16, 16), 10**9, dtype=np.int64)
        for lane in range(32):
            g, t = lane // 4, lane % 4
            x, y = chunk(vbox, 2 * t, g), chunk(vbox, 2 * t + 1, g)
            z, w = chunk(vbox, 8 + 2 * t, g), chunk(vbox, 9 + 2 * t, g)
            # bytes 2i, 2i+1 of each row, paired across tokens: (x, y) then (z, w)
            A[g, 2 * t], A[g, 2 * t + 1] = x[2 * i], y[2 * i]
            A[g + 8, 2 * t], A[g + 8, 2 * t + 1] = x[2 * i + 1], y[2 * i + 1]
            A[g, 8 + 2 * t], A[g, 9 + 2 * t] = z[2 * i], w[2 * i]
            A[g + 8, 8 + 2 * t], A[g + 8, 9 + 2 * t] = z[2 * i + 1], w[2 * i + 1]
        assert (A != 10**9).all()
        D = A @ P  # 16 (rows) x 8 (heads); B = P^T fragments in their usual order
        for lane in range(32):
            g, t = lane // 4, lane % 4
            o = (D[g, 2 * t], D[g, 2 * t + 1], D[g + 8, 2 * t], D[g + 8, 2 * t + 1])
            # the output store: dims 16g + 2i (o0, o1) and 16g + 2i + 1 (o2, o3)
            d = 16 * g + 2 * i
            out[2 * t, d], out[2 * t, d + 1] = o[0], o[2]
            out[2 * t + 1, d], out[2 * t + 1, d + 1] = o[1], o[3]
    assert (out != 10**9).all()
    assert np.array_equal(out, P.T @ V)
