"""Python handle on the native host block manager (pkv_bm_* in the C ABI).

Free list, per-sequence block tables, reserve on admit, shared prefix
blocks with reference counts and copy-on-write bookkeeping, as described on
the "Paged attention" page (danielfleming.xyz, "What changed") and the "SLM
paged attention" page (aicassindra.com, "The architecture", "End-to-end
flow").  All logic is in C++; this is marshalling only.
"""
from __future__ import annotations

import ctypes
from typing import Optional, Tuple

import numpy as np

from .ops import PagedKVError, lib


class Stats(ctypes.Structure):
    _fields_ = [("num_blocks", ctypes.c_int32), ("free_blocks", ctypes.c_int32),
                ("used_blocks", ctypes.c_int32), ("shared_blocks", ctypes.c_int32),
                ("sequences", ctypes.c_int32), ("prefixes", ctypes.c_int32),
                ("live_tokens", ctypes.c_int64), ("reserved_slots", ctypes.c_int64),
                ("cow_copies", ctypes.c_int64)]

    def as_dict(self):
        return {name: getattr(self, name) for name, _ in self._fields_}


_declared = False


def _L():
    global _declared
    L = lib()
    if not _declared:
        P, I, I32, I64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_int32, ctypes.c_int64
        PI32 = ctypes.POINTER(ctypes.c_int32)
        L.pkv_bm_create.argtypes = [I, I, I, ctypes.POINTER(P)]
        L.pkv_bm_destroy.argtypes = [P]
        L.pkv_bm_destroy.restype = None
        L.pkv_bm_register_prefix.argtypes = [P, I, PI32, P]
        L.pkv_bm_release_prefix.argtypes = [P, I32]
        L.pkv_bm_admit.argtypes = [P, I64, I, I, I32, I]
        L.pkv_bm_append_slot.argtypes = [P, I64, PI32, PI32, PI32]
        L.pkv_bm_free.argtypes = [P, I64]
        L.pkv_bm_table.argtypes = [P, I64, P, PI32]
        L.pkv_bm_stats.argtypes = [P, ctypes.POINTER(Stats)]
        L.pkv_bm_refcount.argtypes = [P, I32, PI32]
        L.pkv_bm_inject_pop_failure.argtypes = [P, I]
        for fn in ("pkv_bm_create", "pkv_bm_register_prefix", "pkv_bm_release_prefix",
                   "pkv_bm_admit", "pkv_bm_append_slot", "pkv_bm_free", "pkv_bm_table",
                   "pkv_bm_stats", "pkv_bm_refcount", "pkv_bm_inject_pop_failure"):
            getattr(L, fn).restype = I
        _declared = True
    return L


def _check(fn: str, st: int) -> None:
    if st != 0:
        raise PagedKVError(fn, st)


class BlockManager:
    def __init__(self, num_blocks: int, block_size: int, max_blocks_per_row: int):
        self._h = ctypes.c_void_p()
        _check("pkv_bm_create", _L().pkv_bm_create(num_blocks, block_size, max_blocks_per_row,
                                                   ctypes.byref(self._h)))
        self.num_blocks = num_blocks
        self.block_size = block_size
        self.max_blocks_per_row = max_blocks_per_row

    def close(self):
        if self._h:
            _L().pkv_bm_destroy(self._h)
            self._h = ctypes.c_void_p()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def register_prefix(self, prefix_tokens: int) -> Tuple[int, np.ndarray]:
        pid = ctypes.c_int32(-1)
        ids = np.full(max(1, prefix_tokens // self.block_size), -1, dtype=np.int32)
        _check("pkv_bm_register_prefix",
               _L().pkv_bm_register_prefix(self._h, prefix_tokens, ctypes.byref(pid),
                                           ids.ctypes.data_as(ctypes.c_void_p)))
        return pid.value, ids[:prefix_tokens // self.block_size]

    def release_prefix(self, prefix_id: int) -> None:
        _check("pkv_bm_release_prefix", _L().pkv_bm_release_prefix(self._h, prefix_id))

    def admit(self, seq_id: int, prompt_len: int, max_new_tokens: int,
              prefix_id: int = -1, reserve: bool = True) -> None:
        _check("pkv_bm_admit", _L().pkv_bm_admit(self._h, seq_id, prompt_len, max_new_tokens,
                                                 prefix_id, int(bool(reserve))))

    def try_admit(self, *a, **k) -> bool:
        try:
            self.admit(*a, **k)
            return True
        except PagedKVError as e:
            if e.status == 6:  # PKV_ERR_NO_BLOCKS
                return False
            raise

    def append_slot(self, seq_id: int) -> Tuple[int, Optional[Tuple[int, int]]]:
        """Position of the sequence's next token and the (src, dst) block copy
        that copy-on-write requires first, if any."""
        pos, src, dst = ctypes.c_int32(), ctypes.c_int32(), ctypes.c_int32()
        _check("pkv_bm_append_slot", _L().pkv_bm_append_slot(self._h, seq_id, ctypes.byref(pos),
                                                             ctypes.byref(src), ctypes.byref(dst)))
        return pos.value, ((src.value, dst.value) if src.value >= 0 else None)

    def free(self, seq_id: int) -> None:
        _check("pkv_bm_free", _L().pkv_bm_free(self._h, seq_id))

    def table(self, seq_id: int) -> Tuple[np.ndarray, int]:
        row = np.empty(self.max_blocks_per_row, dtype=np.int32)
        n = ctypes.c_int32()
        _check("pkv_bm_table", _L().pkv_bm_table(self._h, seq_id,
                                                 row.ctypes.data_as(ctypes.c_void_p),
                                                 ctypes.byref(n)))
        return row, n.value

    def tables(self, seq_ids) -> Tuple[np.ndarray, np.ndarray]:
        """Dense int32 [rows][max_blocks_per_row] table and seq_lens for a batch."""
        t = np.empty((len(seq_ids), self.max_blocks_per_row), dtype=np.int32)
        lens = np.empty(len(seq_ids), dtype=np.int32)
        for i, s in enumerate(seq_ids):
            t[i], lens[i] = self.table(s)
        return t, lens

    def stats(self) -> dict:
        st = Stats()
        _check("pkv_bm_stats", _L().pkv_bm_stats(self._h, ctypes.byref(st)))
        return st.as_dict()

    def refcount(self, block_id: int) -> int:
        c = ctypes.c_int32()
        _check("pkv_bm_refcount", _L().pkv_bm_refcount(self._h, block_id, ctypes.byref(c)))
        return c.value

    def inject_pop_failure(self, pops: int) -> None:
        _check("pkv_bm_inject_pop_failure", _L().pkv_bm_inject_pop_failure(self._h, pops))
