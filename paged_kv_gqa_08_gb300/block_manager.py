"""Python handle on libpagedattn's host block manager (pa_bm_* calls).

Argument marshalling only: the allocation, prefix matching and reference
counting run in the library.  Token ids, block tables, lengths and slots are
host numpy arrays.
"""
from __future__ import annotations

import ctypes
from typing import Sequence

import numpy as np

from . import _check, load_library

_I64 = ctypes.c_int64
_I32 = ctypes.c_int32


def _arr(a, dtype) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=dtype))


class BlockManager:
    """Blocks of ``block_size`` tokens over a cache of ``num_blocks`` pages."""

    def __init__(self, num_blocks: int, block_size: int):
        self._lib = load_library()
        h = ctypes.c_void_p()
        _check("pa_bm_create", self._lib.pa_bm_create(num_blocks, block_size, ctypes.byref(h)))
        self._h = h
        self.num_blocks = num_blocks
        self.block_size = block_size

    def close(self) -> None:
        if self._h:
            self._lib.pa_bm_destroy(self._h)
            self._h = ctypes.c_void_p()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def can_allocate(self, token_ids: Sequence[int]) -> int:
        """Leading blocks the prompt would reuse, or -1 when it does not fit."""
        t = _arr(token_ids, np.int32)
        out = _I64()
        _check("pa_bm_can_allocate", self._lib.pa_bm_can_allocate(self._h, t.ctypes.data, t.size, ctypes.byref(out)))
        return out.value

    def allocate(self, seq_id: int, token_ids: Sequence[int]) -> int:
        """Register a sequence; returns the number of prompt tokens already cached."""
        t = _arr(token_ids, np.int32)
        out = _I64()
        _check("pa_bm_allocate", self._lib.pa_bm_allocate(self._h, seq_id, t.ctypes.data, t.size, ctypes.byref(out)))
        return out.value

    def append_token(self, seq_id: int, token_id: int) -> None:
        _check("pa_bm_append_token", self._lib.pa_bm_append_token(self._h, seq_id, int(token_id)))

    def hash_blocks(self, seq_id: int, num_computed_tokens: int) -> None:
        _check("pa_bm_hash_blocks", self._lib.pa_bm_hash_blocks(self._h, seq_id, num_computed_tokens))

    def free(self, seq_id: int) -> None:
        _check("pa_bm_free", self._lib.pa_bm_free(self._h, seq_id))

    def block_tables(self, seq_ids: Sequence[int], max_pages_per_seq: int, pad_page: int = 0):
        """(block_tables int32 [n, max_pages_per_seq], context_lens int32 [n])."""
        ids = _arr(seq_ids, np.int64)
        bt = np.empty((ids.size, max_pages_per_seq), dtype=np.int32)
        lens = np.empty(ids.size, dtype=np.int32)
        _check("pa_bm_block_tables", self._lib.pa_bm_block_tables(
            self._h, ids.ctypes.data, ids.size, max_pages_per_seq, pad_page, bt.ctypes.data, lens.ctypes.data))
        return bt, lens

    def slot_mapping(self, seq_ids: Sequence[int], num_new_tokens: Sequence[int]) -> np.ndarray:
        ids = _arr(seq_ids, np.int64)
        nn = _arr(num_new_tokens, np.int32)
        assert nn.size == ids.size
        out = np.empty(int(nn.sum()), dtype=np.int64)
        _check("pa_bm_slot_mapping", self._lib.pa_bm_slot_mapping(
            self._h, ids.ctypes.data, ids.size, nn.ctypes.data, out.ctypes.data))
        return out

    def num_free_blocks(self) -> int:
        n = _I64()
        _check("pa_bm_query", self._lib.pa_bm_query(self._h, ctypes.byref(n), None, None))
        return n.value

    def counts(self):
        """(free blocks, sequences, registered block hashes)."""
        a, b, c = _I64(), _I64(), _I64()
        _check("pa_bm_query", self._lib.pa_bm_query(self._h, ctypes.byref(a), ctypes.byref(b), ctypes.byref(c)))
        return a.value, b.value, c.value

    def ref_count(self, block_id: int) -> int:
        r = _I32()
        _check("pa_bm_block_ref_count", self._lib.pa_bm_block_ref_count(self._h, block_id, ctypes.byref(r)))
        return r.value

    def seq_info(self, seq_id: int):
        """(tokens, cached tokens, blocks) of one sequence."""
        a, b, c = _I64(), _I64(), _I32()
        _check("pa_bm_seq_info", self._lib.pa_bm_seq_info(self._h, seq_id, ctypes.byref(a), ctypes.byref(b),
                                                           ctypes.byref(c)))
        return a.value, b.value, c.value
