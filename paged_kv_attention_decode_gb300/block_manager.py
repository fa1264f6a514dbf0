"""ctypes binding of the host block manager (include/pa_block_manager.h,
built into libpagedattn.so): which physical block holds each 16-token
logical block of every sequence, with prefix sharing, copy-on-write and
truncation.  Argument marshalling only; the logic is the C++ in
csrc/pa_block_manager.cpp.
"""
from __future__ import annotations

import ctypes

import numpy as np

from ._binding import load_library

_p = ctypes.c_void_p
_i32 = ctypes.c_int32
_i64 = ctypes.c_int64
_u64 = ctypes.c_uint64
_I32P = ctypes.POINTER(ctypes.c_int32)

OK, INVALID_ARG, NO_SPACE, CAPACITY = 0, 1, 5, 6
_NAMES = {OK: "PA_BM_OK", INVALID_ARG: "PA_BM_ERR_INVALID_ARG", NO_SPACE: "PA_BM_ERR_NO_SPACE",
          CAPACITY: "PA_BM_ERR_CAPACITY"}

_SIGNATURES = {
    "pa_bm_create": (_p, [_i32, _i32, _i32]),
    "pa_bm_destroy": (None, [_p]),
    "pa_bm_num_free_blocks": (_i32, [_p]),
    "pa_bm_add_sequence": (ctypes.c_int, [_p, _i64, _u64, _p, _i32, _I32P]),
    "pa_bm_append_tokens": (ctypes.c_int, [_p, _i64, _p, _i32]),
    "pa_bm_allocate_slots": (ctypes.c_int, [_p, _i64, _i32, _I32P, _I32P, _I32P]),
    "pa_bm_truncate": (ctypes.c_int, [_p, _i64, _i32]),
    "pa_bm_fork": (ctypes.c_int, [_p, _i64, _i64]),
    "pa_bm_free_sequence": (ctypes.c_int, [_p, _i64]),
    "pa_bm_seq_len": (_i32, [_p, _i64]),
    "pa_bm_block_table": (_i32, [_p, _i64, _p, _i32]),
    "pa_bm_block_ref": (_i32, [_p, _i32]),
    "pa_bm_block_cached": (_i32, [_p, _i32]),
    "pa_bm_build_step": (ctypes.c_int, [_p, _p, _p, _i32, _p, _i32, _p, _p, _p, _i64]),
}

_bound = None


def _lib():
    global _bound
    if _bound is None:
        lib = load_library()
        for name, (res, args) in _SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _bound = lib
    return _bound


class BlockManagerError(RuntimeError):
    def __init__(self, what: str, status: int):
        super().__init__(f"{what} failed: {_NAMES.get(status, status)}")
        self.status = status


def _i32arr(x) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(x, dtype=np.int32).reshape(-1))


class BlockManager:
    """Free list + allocate_slots + prefix caching over a pool of blocks."""

    def __init__(self, num_blocks: int, block_size: int = 16, prefix_caching: bool = True):
        self._h = _lib().pa_bm_create(num_blocks, block_size, int(bool(prefix_caching)))
        if not self._h:
            raise BlockManagerError("pa_bm_create", INVALID_ARG)
        self.num_blocks = num_blocks
        self.block_size = block_size

    def close(self) -> None:
        if self._h:
            _lib().pa_bm_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def _check(self, rc: int, what: str) -> None:
        if rc != OK:
            raise BlockManagerError(what, rc)

    @property
    def num_free_blocks(self) -> int:
        return int(_lib().pa_bm_num_free_blocks(self._h))

    def add_sequence(self, seq_id: int, prompt, extra_key: int = 0) -> int:
        """Register a sequence; returns the number of prompt tokens already cached."""
        toks = _i32arr(prompt)
        cached = ctypes.c_int32(0)
        self._check(_lib().pa_bm_add_sequence(self._h, seq_id, extra_key & (2**64 - 1), toks.ctypes.data,
                                              toks.size, ctypes.byref(cached)), "pa_bm_add_sequence")
        return cached.value

    def append_tokens(self, seq_id: int, tokens) -> None:
        toks = _i32arr(tokens)
        self._check(_lib().pa_bm_append_tokens(self._h, seq_id, toks.ctypes.data, toks.size),
                    "pa_bm_append_tokens")

    def allocate_slots(self, seq_id: int, num_new: int):
        """Slots for the next num_new known tokens.  Returns the copy-on-write
        pair (src, dst) or None; raises BlockManagerError(NO_SPACE) when the
        pool is short (nothing changed)."""
        src, dst, n = ctypes.c_int32(0), ctypes.c_int32(0), ctypes.c_int32(0)
        self._check(_lib().pa_bm_allocate_slots(self._h, seq_id, num_new, ctypes.byref(src), ctypes.byref(dst),
                                                ctypes.byref(n)), "pa_bm_allocate_slots")
        return (src.value, dst.value) if n.value else None

    def truncate(self, seq_id: int, new_len: int) -> None:
        self._check(_lib().pa_bm_truncate(self._h, seq_id, new_len), "pa_bm_truncate")

    def fork(self, parent_id: int, child_id: int) -> None:
        self._check(_lib().pa_bm_fork(self._h, parent_id, child_id), "pa_bm_fork")

    def free_sequence(self, seq_id: int) -> None:
        self._check(_lib().pa_bm_free_sequence(self._h, seq_id), "pa_bm_free_sequence")

    def seq_len(self, seq_id: int) -> int:
        return int(_lib().pa_bm_seq_len(self._h, seq_id))

    def block_table(self, seq_id: int) -> np.ndarray:
        n = self.seq_len(seq_id)
        if n < 0:
            raise BlockManagerError("pa_bm_block_table", INVALID_ARG)
        out = np.zeros(-(-n // self.block_size) + 1, dtype=np.int32)
        k = _lib().pa_bm_block_table(self._h, seq_id, out.ctypes.data, out.size)
        if k < 0:
            raise BlockManagerError("pa_bm_block_table", CAPACITY)
        return out[:k].copy()

    def block_ref(self, block: int) -> int:
        return int(_lib().pa_bm_block_ref(self._h, block))

    def block_cached(self, block: int) -> bool:
        return bool(_lib().pa_bm_block_cached(self._h, block))

    def build_step(self, seq_ids, q_lens, max_blocks: int):
        """Host arrays of one device step: (block_tables [B, max_blocks] int32,
        seq_lens int32, cu_q_lens int32 [B+1], slot_mapping int64)."""
        ids = np.ascontiguousarray(np.asarray(seq_ids, dtype=np.int64).reshape(-1))
        ql = _i32arr(q_lens)
        B = ids.size
        tables = np.empty((B, max_blocks), dtype=np.int32)
        lens = np.empty(B, dtype=np.int32)
        cu = np.empty(B + 1, dtype=np.int32)
        slots = np.empty(max(1, int(ql.sum())), dtype=np.int64)
        self._check(_lib().pa_bm_build_step(self._h, ids.ctypes.data, ql.ctypes.data, B, tables.ctypes.data,
                                            max_blocks, lens.ctypes.data, cu.ctypes.data, slots.ctypes.data,
                                            slots.size), "pa_bm_build_step")
        return tables, lens, cu, slots[: int(ql.sum())]
