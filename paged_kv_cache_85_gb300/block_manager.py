"""Host-side KV-cache block allocator (wrapper over ``include/pkv_block_manager.h``).

Hands out the physical blocks of the paged cache to sequences, with
reference counts and prefix caching by chained content hashes, and builds the
``block_tables`` / ``context_lens`` / ``slot_mapping`` arrays a decode step
passes to ``store_kvcache`` and ``paged_attn_decode``.  All logic runs in the
library's C++; this class only marshals arguments (no GPU needed).
"""

from __future__ import annotations

import ctypes

import numpy as np

from . import PkvError, load_library

_configured = False


def _lib():
    global _configured
    lib = load_library()
    if not _configured:
        P, i32, i64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64
        lib.pkv_bm_create.restype = i32
        lib.pkv_bm_create.argtypes = [i64, i32, ctypes.POINTER(P)]
        lib.pkv_bm_destroy.restype = None
        lib.pkv_bm_destroy.argtypes = [P]
        lib.pkv_bm_can_allocate.restype = i32
        lib.pkv_bm_can_allocate.argtypes = [P, i64]
        lib.pkv_bm_allocate.restype = i32
        lib.pkv_bm_allocate.argtypes = [P, i64, P, i64, ctypes.POINTER(i64)]
        lib.pkv_bm_can_append.restype = i32
        lib.pkv_bm_can_append.argtypes = [P, i64]
        lib.pkv_bm_append.restype = i32
        lib.pkv_bm_append.argtypes = [P, i64, ctypes.c_int32, ctypes.POINTER(i64)]
        lib.pkv_bm_append_batch.restype = i32
        lib.pkv_bm_append_batch.argtypes = [P, P, P, i32, P]
        lib.pkv_bm_deallocate.restype = i32
        lib.pkv_bm_deallocate.argtypes = [P, i64]
        lib.pkv_bm_num_free_blocks.restype = i64
        lib.pkv_bm_num_free_blocks.argtypes = [P]
        lib.pkv_bm_seq_len.restype = i64
        lib.pkv_bm_seq_len.argtypes = [P, i64]
        lib.pkv_bm_ref_count.restype = ctypes.c_int32
        lib.pkv_bm_ref_count.argtypes = [P, ctypes.c_int32]
        lib.pkv_bm_block_table.restype = i64
        lib.pkv_bm_block_table.argtypes = [P, i64, P, i64]
        lib.pkv_bm_slots.restype = i32
        lib.pkv_bm_slots.argtypes = [P, i64, i64, i64, P]
        lib.pkv_bm_decode_batch.restype = i32
        lib.pkv_bm_decode_batch.argtypes = [P, P, i32, i32, P, P, P]
        _configured = True
    return lib


def _check(lib, status):
    if status != 0:
        raise PkvError(status, lib.pkv_last_error().decode(errors="replace"))


def _ptr(a: np.ndarray):
    return ctypes.c_void_p(a.ctypes.data)


class BlockManager:
    """Allocator over ``num_blocks`` blocks of ``block_size`` token slots."""

    def __init__(self, num_blocks: int, block_size: int):
        self._lib = _lib()
        h = ctypes.c_void_p()
        _check(self._lib, self._lib.pkv_bm_create(num_blocks, block_size, ctypes.byref(h)))
        self._h = h
        self.num_blocks = num_blocks
        self.block_size = block_size

    def close(self):
        if self._h:
            self._lib.pkv_bm_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def can_allocate(self, num_tokens: int) -> bool:
        return bool(self._lib.pkv_bm_can_allocate(self._h, num_tokens))

    def allocate(self, seq_id: int, tokens) -> int:
        """Allocate a prompt with prefix caching; returns the number of cached tokens."""
        t = np.ascontiguousarray(tokens, dtype=np.int32)
        cached = ctypes.c_int64()
        _check(self._lib, self._lib.pkv_bm_allocate(self._h, seq_id, _ptr(t), t.size,
                                                    ctypes.byref(cached)))
        return cached.value

    def can_append(self, seq_id: int) -> bool:
        return bool(self._lib.pkv_bm_can_append(self._h, seq_id))

    def append(self, seq_id: int, token: int) -> int:
        """Append one token; returns the flat slot for its K/V."""
        slot = ctypes.c_int64()
        _check(self._lib, self._lib.pkv_bm_append(self._h, seq_id, int(token), ctypes.byref(slot)))
        return slot.value

    def append_batch(self, seq_ids, tokens) -> np.ndarray:
        """One decode step: append tokens[i] to seq_ids[i]; returns their slots (all or nothing)."""
        ids = np.ascontiguousarray(seq_ids, dtype=np.int64)
        toks = np.ascontiguousarray(tokens, dtype=np.int32)
        if ids.shape != toks.shape:
            raise ValueError("append_batch: seq_ids and tokens differ in length")
        slots = np.empty(ids.size, dtype=np.int64)
        _check(self._lib, self._lib.pkv_bm_append_batch(self._h, _ptr(ids), _ptr(toks), ids.size,
                                                        _ptr(slots)))
        return slots

    def deallocate(self, seq_id: int):
        _check(self._lib, self._lib.pkv_bm_deallocate(self._h, seq_id))

    @property
    def num_free_blocks(self) -> int:
        return int(self._lib.pkv_bm_num_free_blocks(self._h))

    def seq_len(self, seq_id: int) -> int:
        return int(self._lib.pkv_bm_seq_len(self._h, seq_id))

    def ref_count(self, block_id: int) -> int:
        return int(self._lib.pkv_bm_ref_count(self._h, block_id))

    def block_table(self, seq_id: int) -> np.ndarray:
        n = self._lib.pkv_bm_block_table(self._h, seq_id, None, 0)
        if n < 0:
            raise KeyError(seq_id)
        out = np.empty(n, dtype=np.int32)
        self._lib.pkv_bm_block_table(self._h, seq_id, _ptr(out), n)
        return out

    def slots(self, seq_id: int, t0: int, t1: int) -> np.ndarray:
        out = np.empty(max(t1 - t0, 0), dtype=np.int64)
        _check(self._lib, self._lib.pkv_bm_slots(self._h, seq_id, t0, t1, _ptr(out)))
        return out

    def decode_batch(self, seq_ids, MBS: int):
        """(block_tables [n, MBS] int32, context_lens [n] int32, slot_mapping [n] int64)."""
        ids = np.ascontiguousarray(seq_ids, dtype=np.int64)
        n = ids.size
        tables = np.empty((n, MBS), dtype=np.int32)
        lens = np.empty(n, dtype=np.int32)
        slots = np.empty(n, dtype=np.int64)
        _check(self._lib, self._lib.pkv_bm_decode_batch(self._h, _ptr(ids), n, MBS, _ptr(tables),
                                                        _ptr(lens), _ptr(slots)))
        return tables, lens, slots
