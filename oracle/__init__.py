"""fp64 CPU oracle for paged KV-cache attention -- TEST INFRASTRUCTURE ONLY.

Only the tests, the smoke check and the benchmark's CPU-baseline leg may
import this package.  The CUDA library never loads it and shares no code with
it; the only thing both sides share is the seeded input generator, which holds
none of the method's arithmetic.

The arithmetic lives in ``pkv_oracle.c`` (plain C, double precision) and is
loaded here through ctypes; ``brute.py`` is an independent pure-Python brute
force used to pin it on tiny inputs.  fp16 tensors cross this boundary as
numpy ``uint16`` arrays holding raw binary16 bit patterns (or as numpy
``float16`` arrays, which are viewed as such).

Citations (page title, section):
  * "PagedAttention" (deepconcepts.dev), "PagedAttention" and the closing note
    on FlashAttention: paged attention computes exactly ordinary attention;
    block-wise softmax recombination is exact.
  * "Paged attention" (danielfleming.xyz), "What changed": decode touches
    just the blocks a row's table names, up to its true length.
  * "SLM paged attention" (aicassindra.com), "The architecture": a row's
    table turns position / block_size into a physical block; the final block
    may be partly filled.

Parity pins: every function here is pinned by tests in ``tests/test_oracle.py``
(brute force, closed forms, invariants); none is "parity unpinned".
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "pkv_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

ORACLE_OK = 0
ORACLE_BAD_ARG = 1
ORACLE_BAD_TABLE = 5


class OracleError(RuntimeError):
    pass


def build(force: bool = False) -> str:
    """Compile pkv_oracle.c into liboracle.so beside it (gcc, -O2, OpenMP)."""
    stale = (not os.path.exists(_LIB_PATH)
             or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC))
    if force or stale:
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp",
               "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB_PATH)
            P = ctypes.c_void_p
            I = ctypes.c_int
            D = ctypes.c_double
            lib.oracle_half_to_double.argtypes = [ctypes.c_uint16]
            lib.oracle_half_to_double.restype = D
            lib.oracle_half_array_to_double.argtypes = [P, P, ctypes.c_int64]
            lib.oracle_half_array_to_double.restype = None
            lib.oracle_paged_decode.argtypes = [P, P, P, P, P, P, I, I, I, I, I, D, I, I, I]
            lib.oracle_paged_decode.restype = I
            lib.oracle_contiguous_decode.argtypes = [P, P, P, P, P, I, I, I, I, I, D, I]
            lib.oracle_contiguous_decode.restype = I
            lib.oracle_blockwise_decode.argtypes = [P, P, P, P, P, P, P, I, I, I, I, I, D, I, I, I]
            lib.oracle_blockwise_decode.restype = I
            lib.oracle_paged_append.argtypes = [P, P, P, P, P, P, I, I, I, I, I, I]
            lib.oracle_paged_append.restype = I
            lib.oracle_copy_blocks.argtypes = [P, P, P, P, I, I, I, I, I]
            lib.oracle_copy_blocks.restype = I
            lib.oracle_prefill_scatter.argtypes = [P, P, P, P, P, P, P, P, I, I, I, I, I, I, I]
            lib.oracle_prefill_scatter.restype = I
            lib.oracle_fp8_e4m3_to_double.argtypes = [ctypes.c_uint8]
            lib.oracle_fp8_e4m3_to_double.restype = D
            lib.oracle_fp8_e4m3_from_float.argtypes = [ctypes.c_float]
            lib.oracle_fp8_e4m3_from_float.restype = ctypes.c_uint8
            lib.oracle_fp8_quantize_array.argtypes = [P, P, ctypes.c_int64, ctypes.c_float]
            lib.oracle_fp8_quantize_array.restype = None
            lib.oracle_paged_append_fp8.argtypes = [P, P, P, P, P, P, P, P, I, I, I, I, I, I]
            lib.oracle_paged_append_fp8.restype = I
            lib.oracle_paged_decode_fp8.argtypes = [P, P, P, P, P, P, P, P, I, I, I, I, I, D, I, I, I]
            lib.oracle_paged_decode_fp8.restype = I
            lib.oracle_paged_prefill.argtypes = [P, P, P, P, P, P, P, I, I, I, I, I, D, I, I, I]
            lib.oracle_paged_prefill.restype = I
            _lib = lib
    return _lib


def _bits(a) -> np.ndarray:
    """fp16 array (float16 or uint16 bit patterns) -> contiguous uint16."""
    a = np.asarray(a)
    if a.dtype == np.float16:
        a = a.view(np.uint16)
    if a.dtype != np.uint16:
        raise TypeError(f"expected float16/uint16 bits, got {a.dtype}")
    return np.ascontiguousarray(a)


def _i32(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.int32))


def _ptr(a: np.ndarray):
    return ctypes.c_void_p(a.ctypes.data)


def _check(rc: int, what: str):
    if rc != ORACLE_OK:
        raise OracleError(f"{what}: oracle status {rc}")


def half_to_double(bits) -> np.ndarray:
    """Exact binary16 -> float64 widening (written from the IEEE definition)."""
    b = _bits(bits)
    out = np.empty(b.shape, dtype=np.float64)
    _load().oracle_half_array_to_double(_ptr(out), _ptr(b), b.size)
    return out


def default_threads() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1


def paged_decode(q, k_pool, v_pool, block_tables, seq_lens, scale: float,
                 num_threads: int = 1) -> np.ndarray:
    """fp64 attention per row over its table-listed tokens in logical order.

    q: [rows][Hq][D]; pools: [num_blocks][bs][Hk][D]; block_tables:
    [rows][max_blocks_per_row]; seq_lens: [rows].  Returns [rows][Hq][D] f64.
    """
    q = _bits(q); kp = _bits(k_pool); vp = _bits(v_pool)
    bt = _i32(block_tables); sl = _i32(seq_lens)
    rows, hq, d = q.shape
    nb, bs, hk, d2 = kp.shape
    assert d2 == d and vp.shape == kp.shape and bt.shape[0] == rows and sl.shape == (rows,)
    out = np.zeros((rows, hq, d), dtype=np.float64)
    rc = _load().oracle_paged_decode(_ptr(out), _ptr(q), _ptr(kp), _ptr(vp), _ptr(bt), _ptr(sl),
                                     rows, hq, hk, d, bs, float(scale), bt.shape[1], nb,
                                     int(num_threads))
    _check(rc, "paged_decode")
    return out


def contiguous_decode(q, k_slab, v_slab, seq_lens, scale: float,
                      num_threads: int = 1) -> np.ndarray:
    """fp64 attention over a padded contiguous slab [rows][W][Hk][D]."""
    q = _bits(q); ks = _bits(k_slab); vs = _bits(v_slab); sl = _i32(seq_lens)
    rows, hq, d = q.shape
    r2, w, hk, d2 = ks.shape
    assert r2 == rows and d2 == d and vs.shape == ks.shape
    out = np.zeros((rows, hq, d), dtype=np.float64)
    rc = _load().oracle_contiguous_decode(_ptr(out), _ptr(q), _ptr(ks), _ptr(vs), _ptr(sl),
                                          rows, w, hq, hk, d, float(scale), int(num_threads))
    _check(rc, "contiguous_decode")
    return out


def blockwise_decode(q, k_pool, v_pool, block_tables, seq_lens, scale: float,
                     chunk_tokens: int):
    """Chunked softmax with exact log-sum-exp recombination; returns (o, lse)."""
    q = _bits(q); kp = _bits(k_pool); vp = _bits(v_pool)
    bt = _i32(block_tables); sl = _i32(seq_lens)
    rows, hq, d = q.shape
    nb, bs, hk, _ = kp.shape
    out = np.zeros((rows, hq, d), dtype=np.float64)
    lse = np.zeros((rows, hq), dtype=np.float64)
    rc = _load().oracle_blockwise_decode(_ptr(out), _ptr(lse), _ptr(q), _ptr(kp), _ptr(vp),
                                         _ptr(bt), _ptr(sl), rows, hq, hk, d, bs, float(scale),
                                         bt.shape[1], nb, int(chunk_tokens))
    _check(rc, "blockwise_decode")
    return out, lse


def paged_append(k_pool, v_pool, block_tables, positions, k_new, v_new):
    """Return copies of the pools with each row's new token written to its slot."""
    kp = _bits(k_pool).copy(); vp = _bits(v_pool).copy()
    bt = _i32(block_tables); pos = _i32(positions)
    kn = _bits(k_new); vn = _bits(v_new)
    nb, bs, hk, d = kp.shape
    rows = pos.shape[0]
    assert kn.shape == (rows, hk, d) and vn.shape == kn.shape
    rc = _load().oracle_paged_append(_ptr(kp), _ptr(vp), _ptr(bt), _ptr(pos), _ptr(kn), _ptr(vn),
                                     rows, hk, d, bs, bt.shape[1] if bt.ndim == 2 else 0, nb)
    _check(rc, "paged_append")
    return kp, vp


def copy_blocks(k_pool, v_pool, src_ids, dst_ids):
    """Return copies of the pools with block dst_ids[i] := block src_ids[i] (in order)."""
    kp = _bits(k_pool).copy(); vp = _bits(v_pool).copy()
    src = _i32(src_ids); dst = _i32(dst_ids)
    nb, bs, hk, d = kp.shape
    rc = _load().oracle_copy_blocks(_ptr(kp), _ptr(vp), _ptr(src), _ptr(dst), int(src.shape[0]),
                                    bs, hk, d, nb)
    _check(rc, "copy_blocks")
    return kp, vp


def prefill_scatter(k_pool, v_pool, block_tables, src_start, dst_start, lengths, k_src, v_src):
    """Return copies of the pools with each row's prompt tokens laid into its blocks."""
    kp = _bits(k_pool).copy(); vp = _bits(v_pool).copy()
    bt = _i32(block_tables); ss = _i32(src_start); ds = _i32(dst_start); ln = _i32(lengths)
    ks = _bits(k_src); vs = _bits(v_src)
    nb, bs, hk, d = kp.shape
    rows, width = ks.shape[0], ks.shape[1]
    rc = _load().oracle_prefill_scatter(_ptr(kp), _ptr(vp), _ptr(bt), _ptr(ss), _ptr(ds), _ptr(ln),
                                        _ptr(ks), _ptr(vs), rows, width, hk, d, bs, bt.shape[1], nb)
    _check(rc, "prefill_scatter")
    return kp, vp


# --- FP8 (E4M3) pools, one scale per KV head ------------------------------------

def fp8_e4m3_to_double(codes) -> np.ndarray:
    """Exact E4M3 decode of uint8 codes (written from the format definition)."""
    c = np.asarray(codes, dtype=np.uint8)
    L = _load()
    return np.vectorize(lambda v: L.oracle_fp8_e4m3_to_double(int(v)), otypes=[np.float64])(c) \
        if c.size else np.zeros(c.shape)


def fp8_e4m3_from_float(values) -> np.ndarray:
    """Nearest E4M3 codes of float32 values (ties to even, saturating at 448)."""
    v = np.asarray(values, dtype=np.float32)
    L = _load()
    return np.vectorize(lambda x: L.oracle_fp8_e4m3_from_float(float(x)), otypes=[np.uint8])(v) \
        if v.size else np.zeros(v.shape, dtype=np.uint8)


def fp8_quantize(x_fp16, scale: float) -> np.ndarray:
    """Codes of fp16 values quantised with one scale (binary32 x / scale, then encode)."""
    b = _bits(x_fp16)
    out = np.empty(b.shape, dtype=np.uint8)
    _load().oracle_fp8_quantize_array(_ptr(out), _ptr(b), b.size, float(np.float32(scale)))
    return out


def _f32(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.float32))


def _u8(a) -> np.ndarray:
    a = np.asarray(a)
    if a.dtype != np.uint8:
        raise TypeError(f"expected uint8 fp8 codes, got {a.dtype}")
    return np.ascontiguousarray(a)


def paged_append_fp8(k_pool8, v_pool8, k_scale, v_scale, block_tables, positions, k_new, v_new):
    """Copies of the FP8 pools with each row's new token quantised into its slot."""
    kp = _u8(k_pool8).copy(); vp = _u8(v_pool8).copy()
    ks = _f32(k_scale); vs = _f32(v_scale)
    bt = _i32(block_tables); pos = _i32(positions)
    kn = _bits(k_new); vn = _bits(v_new)
    nb, bs, hk, d = kp.shape
    rows = pos.shape[0]
    assert kn.shape == (rows, hk, d) and vn.shape == kn.shape and ks.shape == (hk,)
    rc = _load().oracle_paged_append_fp8(_ptr(kp), _ptr(vp), _ptr(ks), _ptr(vs), _ptr(bt), _ptr(pos),
                                         _ptr(kn), _ptr(vn), rows, hk, d, bs,
                                         bt.shape[1] if bt.ndim == 2 else 0, nb)
    _check(rc, "paged_append_fp8")
    return kp, vp


def paged_decode_fp8(q, k_pool8, v_pool8, k_scale, v_scale, block_tables, seq_lens, scale: float,
                     num_threads: int = 1) -> np.ndarray:
    """fp64 attention over FP8 pools dequantised with one scale per KV head."""
    q = _bits(q); kp = _u8(k_pool8); vp = _u8(v_pool8)
    ks = _f32(k_scale); vs = _f32(v_scale)
    bt = _i32(block_tables); sl = _i32(seq_lens)
    rows, hq, d = q.shape
    nb, bs, hk, d2 = kp.shape
    assert d2 == d and vp.shape == kp.shape and ks.shape == (hk,) and vs.shape == (hk,)
    out = np.zeros((rows, hq, d), dtype=np.float64)
    rc = _load().oracle_paged_decode_fp8(_ptr(out), _ptr(q), _ptr(kp), _ptr(vp), _ptr(ks), _ptr(vs),
                                         _ptr(bt), _ptr(sl), rows, hq, hk, d, bs, float(scale),
                                         bt.shape[1], nb, int(num_threads))
    _check(rc, "paged_decode_fp8")
    return out


# --- chunked prefill: several queries per row, causal within the chunk ----------

def paged_prefill(q, k_pool, v_pool, block_tables, seq_lens, q_start, scale: float,
                  num_threads: int = 1) -> np.ndarray:
    """fp64 causal attention of each row's chunk of newest tokens.

    q: [total][Hq][D] (rows' chunks packed in order, q_start[r]..q_start[r+1]);
    query i of row r sits at position seq_lens[r] - chunk + i and attends to
    the row's tokens 0..that position.  Returns [total][Hq][D] float64.
    """
    q = _bits(q); kp = _bits(k_pool); vp = _bits(v_pool)
    bt = _i32(block_tables); sl = _i32(seq_lens); qs = _i32(q_start)
    total, hq, d = q.shape
    nb, bs, hk, d2 = kp.shape
    rows = sl.shape[0]
    assert d2 == d and qs.shape == (rows + 1,) and int(qs[-1]) == total
    out = np.zeros((total, hq, d), dtype=np.float64)
    rc = _load().oracle_paged_prefill(_ptr(out), _ptr(q), _ptr(kp), _ptr(vp), _ptr(bt), _ptr(sl),
                                      _ptr(qs), rows, hq, hk, d, bs, float(scale), bt.shape[1], nb,
                                      int(num_threads))
    _check(rc, "paged_prefill")
    return out
