"""Thin ctypes binding over libpagedkv's C ABI (include/paged_kv.h).

Argument marshalling only: each function checks the tensors' device, dtype
and contiguity, derives the sizes from their shapes and calls the C entry
point of the same name with raw pointers and the current CUDA stream.  Every
step of the computation runs in the library's CUDA kernels; there is no CPU
fallback, and calling an op without the built library raises.

Tensors (torch, on the GPU):
  k_pool, v_pool  fp16 [num_blocks][block_size][kv_heads][head_dim]
  block_tables    int32 [rows][max_blocks_per_row]
  seq_lens        int32 [rows];  positions int32 [rows]
  q, out          fp16 [rows][q_heads][head_dim]
  k_new, v_new    fp16 [rows][kv_heads][head_dim]
"""
from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional

import torch

from . import build as _build

_lock = threading.Lock()
_lib = None

PKV_OK = 0
STATUS_NAMES = {}


class PagedKVError(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        super().__init__(f"{fn} failed: {status_string(status)} ({status})")


def lib() -> ctypes.CDLL:
    """Load libpagedkv.so (building it first if it is missing or stale)."""
    global _lib
    with _lock:
        if _lib is None:
            path = _build.build()
            if not os.path.exists(path):
                raise RuntimeError(f"libpagedkv.so missing at {path}")
            L = ctypes.CDLL(path)
            _declare(L)
            _lib = L
    return _lib


def _declare(L: ctypes.CDLL) -> None:
    P, I, F, S = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
    L.pkv_status_string.argtypes = [I]
    L.pkv_status_string.restype = ctypes.c_char_p
    L.pkv_abi_version.argtypes = []
    L.pkv_abi_version.restype = I
    L.paged_kv_append.argtypes = [P, P, P, P, P, P, I, I, I, I, I, I, P, P]
    L.paged_kv_append.restype = I
    L.paged_attention_workspace_size.argtypes = [I, I, I, I, I, I]
    L.paged_attention_workspace_size.restype = S
    L.paged_attention_decode.argtypes = [P, P, P, P, P, P, I, I, I, I, I, F, I, I, I, P, S, P, P]
    L.paged_attention_decode.restype = I
    L.paged_attention_padded_decode.argtypes = [P, P, P, P, P, I, I, I, I, I, F, P, S, P, P]
    L.paged_attention_padded_decode.restype = I
    L.pkv_check_error.argtypes = [P, P, P]
    L.pkv_check_error.restype = I
    L.paged_attention_decode_noalloc.argtypes = [P, P, P, P, P, P, I, I, I, I, I, F, I, I, I, P, P]
    L.paged_attention_decode_noalloc.restype = I
    L.paged_attention_append_decode.argtypes = [P, P, P, P, P, P, P, P, P, I, I, I, I, I, F, I, I, I,
                                                P, S, ctypes.c_uint, P, P]
    L.paged_attention_append_decode.restype = I
    L.paged_kv_append_fp8.argtypes = [P, P, P, P, P, P, P, P, I, I, I, I, I, I, P, P]
    L.paged_kv_append_fp8.restype = I
    L.paged_attention_decode_fp8.argtypes = [P, P, P, P, P, P, P, P, I, I, I, I, I, F, I, I, I, P,
                                             S, P, P]
    L.paged_attention_decode_fp8.restype = I
    L.paged_attention_append_decode_fp8.argtypes = [P, P, P, P, P, P, P, P, P, P, P, I, I, I, I, I,
                                                    F, I, I, I, P, S, ctypes.c_uint, P, P]
    L.paged_attention_append_decode_fp8.restype = I
    L.paged_attention_prefill.argtypes = [P, P, P, P, P, P, P, I, I, I, I, I, I, F, I, I, I, P, S,
                                          P, P]
    L.paged_attention_prefill.restype = I
    L.paged_attention_prefill_workspace_size.argtypes = [I, I, I, I, I]
    L.paged_attention_prefill_workspace_size.restype = S
    L.paged_kv_copy_blocks.argtypes = [P, P, P, P, I, I, I, I, I, P, P]
    L.paged_kv_copy_blocks.restype = I
    L.paged_kv_prefill_scatter.argtypes = [P, P, P, P, P, P, P, P, I, I, I, I, I, I, I, P, P]
    L.paged_kv_prefill_scatter.restype = I
    L.paged_attention_plan_size.argtypes = [I, I, I, I, I, I]
    L.paged_attention_plan_size.restype = S
    L.paged_attention_plan.argtypes = [P, S, P, P, P, I, I, I, I, I, I, I, I, P, P]
    L.paged_attention_plan.restype = I
    L.paged_attention_decode_planned.argtypes = [P, P, P, P, P, P, P, P, P, P, P, I, I, I, I, I, F,
                                                 I, I, I, P, S, P, S, ctypes.c_uint, P, P]
    L.paged_attention_decode_planned.restype = I
    L.pkv_debug_set_decode_hooks.argtypes = [ctypes.c_uint, P]
    L.pkv_debug_set_decode_hooks.restype = I


def status_string(status: int) -> str:
    return lib().pkv_status_string(int(status)).decode()


def _check(fn: str, status: int) -> None:
    if status != PKV_OK:
        raise PagedKVError(fn, status)


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _need(t: torch.Tensor, name: str, dtype: torch.dtype, ndim: int) -> None:
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be on a CUDA device")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dims, got {tuple(t.shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def _need_err(dev_err: Optional[torch.Tensor]) -> None:
    if dev_err is not None:
        _need(dev_err, "dev_err", torch.int32, 1)


def append(k_pool, v_pool, block_tables, positions, k_new, v_new, dev_err=None, stream=None):
    """paged_kv_append: write each row's new token into its slot."""
    for t, n, dt, nd in ((k_pool, "k_pool", torch.float16, 4), (v_pool, "v_pool", torch.float16, 4),
                         (block_tables, "block_tables", torch.int32, 2),
                         (positions, "positions", torch.int32, 1),
                         (k_new, "k_new", torch.float16, 3), (v_new, "v_new", torch.float16, 3)):
        _need(t, n, dt, nd)
    _need_err(dev_err)
    nb, bs, hk, d = k_pool.shape
    rows = positions.shape[0]
    st = lib().paged_kv_append(_ptr(k_pool), _ptr(v_pool), _ptr(block_tables), _ptr(positions),
                               _ptr(k_new), _ptr(v_new), rows, hk, d, bs, block_tables.shape[1], nb,
                               _ptr(dev_err), _stream(stream))
    _check("paged_kv_append", st)


def copy_blocks(k_pool, v_pool, src_ids, dst_ids, dev_err=None, stream=None):
    """paged_kv_copy_blocks: block dst_ids[i] := block src_ids[i] in both pools."""
    for t, n, dt, nd in ((k_pool, "k_pool", torch.float16, 4), (v_pool, "v_pool", torch.float16, 4),
                         (src_ids, "src_ids", torch.int32, 1), (dst_ids, "dst_ids", torch.int32, 1)):
        _need(t, n, dt, nd)
    _need_err(dev_err)
    if src_ids.shape != dst_ids.shape:
        raise ValueError("src_ids and dst_ids must have the same length")
    nb, bs, hk, d = k_pool.shape
    st = lib().paged_kv_copy_blocks(_ptr(k_pool), _ptr(v_pool), _ptr(src_ids), _ptr(dst_ids),
                                    src_ids.shape[0], bs, hk, d, nb, _ptr(dev_err), _stream(stream))
    _check("paged_kv_copy_blocks", st)


def prefill_scatter(k_pool, v_pool, block_tables, src_start, dst_start, lengths, k_src, v_src,
                    dev_err=None, stream=None):
    """paged_kv_prefill_scatter: copy each row's prompt K/V into its blocks."""
    for t, n, dt, nd in ((k_pool, "k_pool", torch.float16, 4), (v_pool, "v_pool", torch.float16, 4),
                         (block_tables, "block_tables", torch.int32, 2),
                         (src_start, "src_start", torch.int32, 1),
                         (dst_start, "dst_start", torch.int32, 1),
                         (lengths, "lengths", torch.int32, 1),
                         (k_src, "k_src", torch.float16, 4), (v_src, "v_src", torch.float16, 4)):
        _need(t, n, dt, nd)
    _need_err(dev_err)
    nb, bs, hk, d = k_pool.shape
    rows, width = k_src.shape[0], k_src.shape[1]
    st = lib().paged_kv_prefill_scatter(_ptr(k_pool), _ptr(v_pool), _ptr(block_tables),
                                        _ptr(src_start), _ptr(dst_start), _ptr(lengths), _ptr(k_src),
                                        _ptr(v_src), rows, width, hk, d, bs, block_tables.shape[1],
                                        nb, _ptr(dev_err), _stream(stream))
    _check("paged_kv_prefill_scatter", st)


def append_fp8(k_pool, v_pool, k_scale, v_scale, block_tables, positions, k_new, v_new,
               dev_err=None, stream=None):
    """paged_kv_append_fp8: quantise each row's new token into its FP8 slot."""
    for t, n, dt, nd in ((k_pool, "k_pool", torch.uint8, 4), (v_pool, "v_pool", torch.uint8, 4),
                         (k_scale, "k_scale", torch.float32, 1), (v_scale, "v_scale", torch.float32, 1),
                         (block_tables, "block_tables", torch.int32, 2),
                         (positions, "positions", torch.int32, 1),
                         (k_new, "k_new", torch.float16, 3), (v_new, "v_new", torch.float16, 3)):
        _need(t, n, dt, nd)
    _need_err(dev_err)
    nb, bs, hk, d = k_pool.shape
    st = lib().paged_kv_append_fp8(_ptr(k_pool), _ptr(v_pool), _ptr(k_scale), _ptr(v_scale),
                                   _ptr(block_tables), _ptr(positions), _ptr(k_new), _ptr(v_new),
                                   positions.shape[0], hk, d, bs, block_tables.shape[1], nb,
                                   _ptr(dev_err), _stream(stream))
    _check("paged_kv_append_fp8", st)


def decode_fp8(out, q, k_pool, v_pool, k_scale, v_scale, block_tables, seq_lens, scale: float,
               max_seq_len: int, workspace, dev_err=None, stream=None):
    """paged_attention_decode_fp8: attention over FP8 pools with per-head scales."""
    for t, n, dt, nd in ((out, "out", torch.float16, 3), (q, "q", torch.float16, 3),
                         (k_pool, "k_pool", torch.uint8, 4), (v_pool, "v_pool", torch.uint8, 4),
                         (k_scale, "k_scale", torch.float32, 1), (v_scale, "v_scale", torch.float32, 1),
                         (block_tables, "block_tables", torch.int32, 2),
                         (seq_lens, "seq_lens", torch.int32, 1)):
        _need(t, n, dt, nd)
    _need_err(dev_err)
    rows, hq, d = q.shape
    nb, bs, hk, _ = k_pool.shape
    st = lib().paged_attention_decode_fp8(
        _ptr(out), _ptr(q), _ptr(k_pool), _ptr(v_pool), _ptr(k_scale), _ptr(v_scale),
        _ptr(block_tables), _ptr(seq_lens), rows, hq, hk, d, bs, float(scale),
        block_tables.shape[1], nb, int(max_seq_len), _ptr(workspace), workspace.numel(),
        _ptr(dev_err), _stream(stream))
    _check("paged_attention_decode_fp8", st)


def prefill_workspace_size(rows: int, q_heads: int, kv_heads: int, head_dim: int,
                           block_size: int) -> int:
    return int(lib().paged_attention_prefill_workspace_size(rows, q_heads, kv_heads, head_dim,
                                                            block_size))


def alloc_prefill_workspace(rows, q_heads, kv_heads, head_dim, block_size, device="cuda"):
    """A zero-filled prefill workspace (uint8, 256-byte aligned by the allocator)."""
    n = prefill_workspace_size(rows, q_heads, kv_heads, head_dim, block_size)
    if n == 0:
        raise ValueError("invalid sizes for a prefill workspace")
    return torch.zeros(n, dtype=torch.uint8, device=device)


def prefill(out, q, k_pool, v_pool, block_tables, seq_lens, q_start, scale: float,
            max_seq_len: int, dev_err=None, stream=None, workspace=None):
    """paged_attention_prefill: causal attention of each row's chunk of new tokens.

    workspace: from alloc_prefill_workspace (calls on separate workspaces may
    overlap), or None for library-owned memory (calls without a workspace on
    one device must not overlap: issue them on one stream, or order the
    streams).
    """
    for t, n, dt, nd in ((out, "out", torch.float16, 3), (q, "q", torch.float16, 3),
                         (k_pool, "k_pool", torch.float16, 4), (v_pool, "v_pool", torch.float16, 4),
                         (block_tables, "block_tables", torch.int32, 2),
                         (seq_lens, "seq_lens", torch.int32, 1), (q_start, "q_start", torch.int32, 1)):
        _need(t, n, dt, nd)
    _need_err(dev_err)
    if workspace is not None:
        _need(workspace, "workspace", torch.uint8, 1)
    total, hq, d = q.shape
    nb, bs, hk, _ = k_pool.shape
    rows = seq_lens.shape[0]
    if q_start.shape[0] != rows + 1:
        raise ValueError("q_start must have rows + 1 entries")
    st = lib().paged_attention_prefill(
        _ptr(out), _ptr(q), _ptr(k_pool), _ptr(v_pool), _ptr(block_tables), _ptr(seq_lens),
        _ptr(q_start), rows, total, hq, hk, d, bs, float(scale), block_tables.shape[1], nb,
        int(max_seq_len), _ptr(workspace), 0 if workspace is None else workspace.numel(),
        _ptr(dev_err), _stream(stream))
    _check("paged_attention_prefill", st)


def workspace_size(rows: int, q_heads: int, kv_heads: int, head_dim: int, max_seq_len: int,
                   block_size: int) -> int:
    return int(lib().paged_attention_workspace_size(rows, q_heads, kv_heads, head_dim, max_seq_len,
                                                    block_size))


def alloc_workspace(rows, q_heads, kv_heads, head_dim, max_seq_len, block_size, device="cuda"):
    """Zero-filled workspace of the size the C ABI asks for."""
    n = workspace_size(rows, q_heads, kv_heads, head_dim, max_seq_len, block_size)
    if n == 0:
        raise ValueError("unsupported sizes for paged_attention_decode")
    return torch.zeros(n, dtype=torch.uint8, device=device)


def decode(out, q, k_pool, v_pool, block_tables, seq_lens, scale: float, max_seq_len: int,
           workspace, dev_err=None, stream=None):
    """paged_attention_decode: attention of each row's query over its paged tokens."""
    for t, n, dt, nd in ((out, "out", torch.float16, 3), (q, "q", torch.float16, 3),
                         (k_pool, "k_pool", torch.float16, 4), (v_pool, "v_pool", torch.float16, 4),
                         (block_tables, "block_tables", torch.int32, 2),
                         (seq_lens, "seq_lens", torch.int32, 1),
                         (workspace, "workspace", torch.uint8, 1)):
        _need(t, n, dt, nd)
    _need_err(dev_err)
    rows, hq, d = q.shape
    nb, bs, hk, _ = k_pool.shape
    st = lib().paged_attention_decode(_ptr(out), _ptr(q), _ptr(k_pool), _ptr(v_pool),
                                      _ptr(block_tables), _ptr(seq_lens), rows, hq, hk, d, bs,
                                      float(scale), block_tables.shape[1], nb, int(max_seq_len),
                                      _ptr(workspace), workspace.numel(), _ptr(dev_err),
                                      _stream(stream))
    _check("paged_attention_decode", st)


PKV_FLAG_PDL = 0x1


def append_decode(out, q, k_pool, v_pool, block_tables, seq_lens, positions, k_new, v_new,
                  scale: float, max_seq_len: int, workspace, pdl: bool = False, dev_err=None,
                  stream=None):
    """paged_attention_append_decode: append each row's new token, then decode
    (one fused launch where supported; ``pdl`` overlaps it with the previous
    kernel under the contract stated in include/paged_kv.h)."""
    for t, n, dt, nd in ((out, "out", torch.float16, 3), (q, "q", torch.float16, 3),
                         (k_pool, "k_pool", torch.float16, 4), (v_pool, "v_pool", torch.float16, 4),
                         (block_tables, "block_tables", torch.int32, 2),
                         (seq_lens, "seq_lens", torch.int32, 1),
                         (positions, "positions", torch.int32, 1),
                         (k_new, "k_new", torch.float16, 3), (v_new, "v_new", torch.float16, 3),
                         (workspace, "workspace", torch.uint8, 1)):
        _need(t, n, dt, nd)
    _need_err(dev_err)
    rows, hq, d = q.shape
    nb, bs, hk, _ = k_pool.shape
    st = lib().paged_attention_append_decode(
        _ptr(out), _ptr(q), _ptr(k_pool), _ptr(v_pool), _ptr(block_tables), _ptr(seq_lens),
        _ptr(positions), _ptr(k_new), _ptr(v_new), rows, hq, hk, d, bs, float(scale),
        block_tables.shape[1], nb, int(max_seq_len), _ptr(workspace), workspace.numel(),
        PKV_FLAG_PDL if pdl else 0, _ptr(dev_err), _stream(stream))
    _check("paged_attention_append_decode", st)


def append_decode_fp8(out, q, k_pool, v_pool, k_scale, v_scale, block_tables, seq_lens, positions,
                      k_new, v_new, scale: float, max_seq_len: int, workspace, pdl: bool = False,
                      dev_err=None, stream=None):
    """paged_attention_append_decode_fp8: quantise and append each row's new
    token into FP8 pools, then decode, in one launch (``pdl`` as for
    append_decode)."""
    for t, n, dt, nd in ((out, "out", torch.float16, 3), (q, "q", torch.float16, 3),
                         (k_pool, "k_pool", torch.uint8, 4), (v_pool, "v_pool", torch.uint8, 4),
                         (k_scale, "k_scale", torch.float32, 1), (v_scale, "v_scale", torch.float32, 1),
                         (block_tables, "block_tables", torch.int32, 2),
                         (seq_lens, "seq_lens", torch.int32, 1),
                         (positions, "positions", torch.int32, 1),
                         (k_new, "k_new", torch.float16, 3), (v_new, "v_new", torch.float16, 3),
                         (workspace, "workspace", torch.uint8, 1)):
        _need(t, n, dt, nd)
    _need_err(dev_err)
    rows, hq, d = q.shape
    nb, bs, hk, _ = k_pool.shape
    st = lib().paged_attention_append_decode_fp8(
        _ptr(out), _ptr(q), _ptr(k_pool), _ptr(v_pool), _ptr(k_scale), _ptr(v_scale),
        _ptr(block_tables), _ptr(seq_lens), _ptr(positions), _ptr(k_new), _ptr(v_new), rows, hq,
        hk, d, bs, float(scale), block_tables.shape[1], nb, int(max_seq_len), _ptr(workspace),
        workspace.numel(), PKV_FLAG_PDL if pdl else 0, _ptr(dev_err), _stream(stream))
    _check("paged_attention_append_decode_fp8", st)


def padded_decode(out, q, k_slab, v_slab, seq_lens, scale: float, workspace, dev_err=None,
                  stream=None):
    """paged_attention_padded_decode: the full-width masked comparator."""
    for t, n, dt, nd in ((out, "out", torch.float16, 3), (q, "q", torch.float16, 3),
                         (k_slab, "k_slab", torch.float16, 4), (v_slab, "v_slab", torch.float16, 4),
                         (seq_lens, "seq_lens", torch.int32, 1),
                         (workspace, "workspace", torch.uint8, 1)):
        _need(t, n, dt, nd)
    _need_err(dev_err)
    rows, hq, d = q.shape
    _, width, hk, _ = k_slab.shape
    st = lib().paged_attention_padded_decode(_ptr(out), _ptr(q), _ptr(k_slab), _ptr(v_slab),
                                             _ptr(seq_lens), rows, width, hq, hk, d, float(scale),
                                             _ptr(workspace), workspace.numel(), _ptr(dev_err),
                                             _stream(stream))
    _check("paged_attention_padded_decode", st)


def decode_noalloc(out, q, k_pool, v_pool, block_tables, seq_lens, scale: float,
                   max_seq_len: int, dev_err=None, stream=None):
    """paged_attention_decode_noalloc: decode with the library's static scratch
    (for callers that cannot allocate a workspace; see include/paged_kv.h)."""
    for t, n, dt, nd in ((out, "out", torch.float16, 3), (q, "q", torch.float16, 3),
                         (k_pool, "k_pool", torch.float16, 4), (v_pool, "v_pool", torch.float16, 4),
                         (block_tables, "block_tables", torch.int32, 2),
                         (seq_lens, "seq_lens", torch.int32, 1)):
        _need(t, n, dt, nd)
    _need_err(dev_err)
    rows, hq, d = q.shape
    nb, bs, hk, _ = k_pool.shape
    st = lib().paged_attention_decode_noalloc(_ptr(out), _ptr(q), _ptr(k_pool), _ptr(v_pool),
                                              _ptr(block_tables), _ptr(seq_lens), rows, hq, hk, d,
                                              bs, float(scale), block_tables.shape[1], nb,
                                              int(max_seq_len), _ptr(dev_err), _stream(stream))
    _check("paged_attention_decode_noalloc", st)


def plan_size(rows: int, q_heads: int, kv_heads: int, head_dim: int, max_seq_len: int,
              block_size: int) -> int:
    return int(lib().paged_attention_plan_size(rows, q_heads, kv_heads, head_dim, max_seq_len,
                                               block_size))


def alloc_plan(rows, q_heads, kv_heads, head_dim, max_seq_len, block_size, device="cuda"):
    """A plan buffer of the size the C ABI asks for."""
    n = plan_size(rows, q_heads, kv_heads, head_dim, max_seq_len, block_size)
    if n == 0:
        raise ValueError("unsupported sizes for paged_attention_plan")
    return torch.empty(n, dtype=torch.uint8, device=device)


def plan(plan_buf, block_tables, seq_lens, positions, q_heads: int, kv_heads: int, head_dim: int,
         block_size: int, num_blocks: int, max_seq_len: int, dev_err=None, stream=None):
    """paged_attention_plan: the work split of one decode step, shared by its
    layers (``positions`` may be None when the step appends nothing)."""
    for t, n, dt, nd in ((plan_buf, "plan", torch.uint8, 1),
                         (block_tables, "block_tables", torch.int32, 2),
                         (seq_lens, "seq_lens", torch.int32, 1)):
        _need(t, n, dt, nd)
    if positions is not None:
        _need(positions, "positions", torch.int32, 1)
    _need_err(dev_err)
    rows = seq_lens.shape[0]
    st = lib().paged_attention_plan(_ptr(plan_buf), plan_buf.numel(), _ptr(block_tables),
                                    _ptr(seq_lens), _ptr(positions), rows, q_heads, kv_heads,
                                    head_dim, block_size, block_tables.shape[1], num_blocks,
                                    int(max_seq_len), _ptr(dev_err), _stream(stream))
    _check("paged_attention_plan", st)


def decode_planned(out, q, k_pool, v_pool, block_tables, seq_lens, scale: float, max_seq_len: int,
                   plan_buf, workspace, positions=None, k_new=None, v_new=None, k_scale=None,
                   v_scale=None, pdl: bool = False, dev_err=None, stream=None):
    """paged_attention_decode_planned: one layer of a planned step (append +
    decode when ``positions`` is given; FP8 pools when the scales are)."""
    fp8 = k_scale is not None
    pool_dt = torch.uint8 if fp8 else torch.float16
    for t, n, dt, nd in ((out, "out", torch.float16, 3), (q, "q", torch.float16, 3),
                         (k_pool, "k_pool", pool_dt, 4), (v_pool, "v_pool", pool_dt, 4),
                         (block_tables, "block_tables", torch.int32, 2),
                         (seq_lens, "seq_lens", torch.int32, 1),
                         (plan_buf, "plan", torch.uint8, 1),
                         (workspace, "workspace", torch.uint8, 1)):
        _need(t, n, dt, nd)
    if fp8:
        _need(k_scale, "k_scale", torch.float32, 1)
        _need(v_scale, "v_scale", torch.float32, 1)
    if positions is not None:
        _need(positions, "positions", torch.int32, 1)
        _need(k_new, "k_new", torch.float16, 3)
        _need(v_new, "v_new", torch.float16, 3)
    _need_err(dev_err)
    rows, hq, d = q.shape
    nb, bs, hk, _ = k_pool.shape
    st = lib().paged_attention_decode_planned(
        _ptr(out), _ptr(q), _ptr(k_pool), _ptr(v_pool), _ptr(k_scale), _ptr(v_scale),
        _ptr(block_tables), _ptr(seq_lens), _ptr(positions), _ptr(k_new), _ptr(v_new), rows, hq,
        hk, d, bs, float(scale), block_tables.shape[1], nb, int(max_seq_len), _ptr(plan_buf),
        plan_buf.numel(), _ptr(workspace), workspace.numel(), PKV_FLAG_PDL if pdl else 0,
        _ptr(dev_err), _stream(stream))
    _check("paged_attention_decode_planned", st)


def check_error(dev_err: torch.Tensor, stream=None) -> int:
    """Synchronise, read and clear the device error word (PKV_DEV_ERR_* bits)."""
    _need(dev_err, "dev_err", torch.int32, 1)
    host = ctypes.c_int32(0)
    st = lib().pkv_check_error(_ptr(dev_err), _stream(stream), ctypes.byref(host))
    _check("pkv_check_error", st)
    return int(host.value)


def debug_set_decode_hooks(poll_limit: int = 0, stuck_word: Optional[torch.Tensor] = None) -> None:
    """pkv_debug_set_decode_hooks: cap the merge's polls and/or make every
    merge also wait on a device word (a word that nothing writes makes each
    merge give up and flag PKV_DEV_ERR_TIMEOUT).  (0, None) restores normal
    operation.  Test hook."""
    if stuck_word is not None:
        _need(stuck_word, "stuck_word", torch.int32, 1)
    _check("pkv_debug_set_decode_hooks",
           lib().pkv_debug_set_decode_hooks(int(poll_limit), _ptr(stuck_word)))
