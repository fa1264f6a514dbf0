"""CPU oracle for paged KV attention: TEST INFRASTRUCTURE ONLY.

A plain fp64 C implementation (``oracle.c``) of what the paged attention path
computes, loaded through ctypes.  Only ``tests/``, the package smoke check
and the benchmark's CPU-baseline leg may import this package; the product path
never does, and nothing here imports the product package.

All functions take numpy arrays.  Half-precision data is passed as its raw
16-bit patterns (``uint16``) together with a dtype name (``"f16"`` or
``"bf16"``); results are fp64.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

from . import build as _build

_DT = {"f16": 0, "bf16": 1}
_ERR = {1: "invalid argument", 2: "block table entry out of range",
        3: "slot out of range", 4: "out of memory"}
_lib = None

_p = ctypes.c_void_p
_i32 = ctypes.c_int
_i64 = ctypes.c_int64


def _load():
    global _lib
    if _lib is None:
        path = _build.build()
        lib = ctypes.CDLL(path)
        lib.oracle_decode_values.argtypes = [_p, _p, _i64, _i32]
        lib.oracle_slot_mapping.argtypes = [_p, _p, _i32, _p, _p, _i32, _i32, _i32]
        lib.oracle_kv_write.argtypes = [_p, _p, _p, _p, _p, _i64, _i32, _i32, _i32, _i32]
        lib.oracle_paged_attention_decode.argtypes = [
            _p, _p, _p, _p, _p, _i32, _p, _i32, _i32, _i32, _i32, _i32, _i32,
            ctypes.c_double, _i32, _p, _i64, _i32]
        lib.oracle_paged_attention_prefill.argtypes = [
            _p, _p, _p, _p, _p, _i32, _p, _p, _i32, _i32, _i32, _i32, _i32, _i32,
            ctypes.c_double, _i32, _p, _i64, _i32]
        lib.oracle_num_threads.argtypes = [_i32]
        lib.oracle_decode_e4m3.argtypes = [_p, _p, _i64]
        lib.oracle_encode_e4m3.argtypes = [_p, _p, _i64]
        lib.oracle_kv_write_fp8.argtypes = [_p, _p, _p, _p, _p, _i64, _i32, _i32, _i32, _i32, _i32,
                                            ctypes.c_float, ctypes.c_float]
        lib.oracle_paged_attention_decode_fp8.argtypes = [
            _p, _p, _p, _p, _p, _i32, _p, _i32, _i32, _i32, _i32, _i32, _i32,
            ctypes.c_double, _i32, ctypes.c_double, ctypes.c_double, _p, _i64, _i32]
        lib.oracle_paged_attention_prefill_fp8.argtypes = [
            _p, _p, _p, _p, _p, _i32, _p, _p, _i32, _i32, _i32, _i32, _i32, _i32,
            ctypes.c_double, _i32, ctypes.c_double, ctypes.c_double, _p, _i64, _i32]
        for f in ("oracle_decode_values", "oracle_slot_mapping", "oracle_kv_write",
                  "oracle_paged_attention_decode", "oracle_paged_attention_prefill",
                  "oracle_num_threads", "oracle_decode_e4m3", "oracle_encode_e4m3",
                  "oracle_kv_write_fp8", "oracle_paged_attention_decode_fp8",
                  "oracle_paged_attention_prefill_fp8"):
            getattr(lib, f).restype = _i32
        _lib = lib
    return _lib


def _ptr(a):
    return a.ctypes.data_as(ctypes.c_void_p) if a is not None else None


def _check(rc):
    if rc:
        raise ValueError("oracle: " + _ERR.get(rc, "error %d" % rc))


def _c(a, dt):
    return np.ascontiguousarray(a, dtype=dt)


def num_threads(requested: int = 0) -> int:
    return int(_load().oracle_num_threads(requested))


def decode_values(bits: np.ndarray, dtype: str) -> np.ndarray:
    """Decode raw fp16/bf16 bit patterns to fp64."""
    bits = _c(bits, np.uint16)
    out = np.empty(bits.shape, dtype=np.float64)
    _check(_load().oracle_decode_values(_ptr(bits), _ptr(out), bits.size, _DT[dtype]))
    return out


def slot_mapping(block_tables, seq_lens, q_lens, block_size: int, num_blocks: int) -> np.ndarray:
    """Physical slot of every new token (the last q_lens[b] positions of each sequence)."""
    bt = _c(block_tables, np.int32)
    sl = _c(seq_lens, np.int32)
    ql = _c(q_lens, np.int32)
    out = np.empty(int(ql.sum()), dtype=np.int64)
    _check(_load().oracle_slot_mapping(_ptr(out), _ptr(bt), bt.shape[1], _ptr(sl), _ptr(ql),
                                       sl.size, block_size, num_blocks))
    return out


def kv_write(key_bits, value_bits, k_cache_bits, v_cache_bits, slots) -> None:
    """In-place: k_cache[slot // bs, slot % bs] = key[t] (and V) for every slot >= 0."""
    key_bits = _c(key_bits, np.uint16)
    value_bits = _c(value_bits, np.uint16)
    slots = _c(slots, np.int64)
    assert k_cache_bits.dtype == np.uint16 and k_cache_bits.flags.c_contiguous
    assert v_cache_bits.dtype == np.uint16 and v_cache_bits.flags.c_contiguous
    NB, bs, H, D = k_cache_bits.shape
    _check(_load().oracle_kv_write(_ptr(key_bits), _ptr(value_bits), _ptr(k_cache_bits),
                                   _ptr(v_cache_bits), _ptr(slots), slots.size, NB, H, D, bs))


def paged_attention_decode(q_bits, k_cache_bits, v_cache_bits, block_tables, seq_lens,
                           scale: float, dtype: str, num_q_heads: int | None = None,
                           select=None, threads: int = 0) -> np.ndarray:
    """fp64 decode attention: q [B, Hq, D] -> out [n, Hq, D] (n = B or len(select))."""
    q_bits = _c(q_bits, np.uint16)
    B, Hq, D = q_bits.shape
    NB, bs, Hkv, D2 = k_cache_bits.shape
    assert D2 == D
    kc = _c(k_cache_bits, np.uint16)
    vc = _c(v_cache_bits, np.uint16)
    bt = _c(block_tables, np.int32)
    sl = _c(seq_lens, np.int32)
    sel = None if select is None else _c(select, np.int64)
    n = B if sel is None else sel.size
    out = np.empty((n, Hq, D), dtype=np.float64)
    _check(_load().oracle_paged_attention_decode(
        _ptr(out), _ptr(q_bits), _ptr(kc), _ptr(vc), _ptr(bt), bt.shape[1], _ptr(sl), B, NB,
        Hq, Hkv, D, bs, float(scale), _DT[dtype], _ptr(sel), 0 if sel is None else sel.size,
        threads))
    return out


def paged_attention_prefill(q_bits, k_cache_bits, v_cache_bits, block_tables, seq_lens, q_lens,
                            scale: float, dtype: str, select=None, threads: int = 0) -> np.ndarray:
    """fp64 causal varlen attention: q [T, Hq, D] -> out [n, Hq, D] (n = T or len(select))."""
    q_bits = _c(q_bits, np.uint16)
    T, Hq, D = q_bits.shape
    NB, bs, Hkv, D2 = k_cache_bits.shape
    assert D2 == D
    kc = _c(k_cache_bits, np.uint16)
    vc = _c(v_cache_bits, np.uint16)
    bt = _c(block_tables, np.int32)
    sl = _c(seq_lens, np.int32)
    ql = _c(q_lens, np.int32)
    assert int(ql.sum()) == T
    sel = None if select is None else _c(select, np.int64)
    n = T if sel is None else sel.size
    out = np.empty((n, Hq, D), dtype=np.float64)
    _check(_load().oracle_paged_attention_prefill(
        _ptr(out), _ptr(q_bits), _ptr(kc), _ptr(vc), _ptr(bt), bt.shape[1], _ptr(sl), _ptr(ql),
        sl.size, NB, Hq, Hkv, D, bs, float(scale), _DT[dtype], _ptr(sel),
        0 if sel is None else sel.size, threads))
    return out


# ---------------------------------------------------------------------------
# FP8 (E4M3) KV cache
# ---------------------------------------------------------------------------

def decode_e4m3(codes) -> np.ndarray:
    """E4M3 (FN) codes -> fp64 values."""
    codes = _c(codes, np.uint8)
    out = np.empty(codes.shape, dtype=np.float64)
    _check(_load().oracle_decode_e4m3(_ptr(codes), _ptr(out), codes.size))
    return out


def encode_e4m3(values) -> np.ndarray:
    """fp32 values -> nearest E4M3 codes (ties to even, saturating at +-448)."""
    values = _c(values, np.float32)
    out = np.empty(values.shape, dtype=np.uint8)
    _check(_load().oracle_encode_e4m3(_ptr(values), _ptr(out), values.size))
    return out


def kv_write_fp8(key_bits, value_bits, k_cache_codes, v_cache_codes, slots, src_dtype: str,
                 k_scale: float, v_scale: float) -> None:
    """In place, for every slot >= 0 and head h:
    cache[slot // bs, h, slot % bs] = e4m3(float(x) * float32(1 / scale)).
    The E4M3 pools are head-major [NB, Hkv, bs, D]."""
    key_bits = _c(key_bits, np.uint16)
    value_bits = _c(value_bits, np.uint16)
    slots = _c(slots, np.int64)
    assert k_cache_codes.dtype == np.uint8 and k_cache_codes.flags.c_contiguous
    assert v_cache_codes.dtype == np.uint8 and v_cache_codes.flags.c_contiguous
    NB, H, bs, D = k_cache_codes.shape
    k_inv = float(np.float32(1.0) / np.float32(k_scale))
    v_inv = float(np.float32(1.0) / np.float32(v_scale))
    _check(_load().oracle_kv_write_fp8(_ptr(key_bits), _ptr(value_bits), _ptr(k_cache_codes),
                                       _ptr(v_cache_codes), _ptr(slots), slots.size, NB, H, D, bs,
                                       _DT[src_dtype], k_inv, v_inv))


def paged_attention_decode_fp8(q_bits, k_cache_codes, v_cache_codes, block_tables, seq_lens, scale: float,
                               q_dtype: str, k_scale: float, v_scale: float, select=None,
                               threads: int = 0) -> np.ndarray:
    """fp64 decode attention over a head-major E4M3 cache [NB, Hkv, bs, D]
    (values = code * scale)."""
    q_bits = _c(q_bits, np.uint16)
    B, Hq, D = q_bits.shape
    NB, Hkv, bs, D2 = k_cache_codes.shape
    assert D2 == D
    kc = _c(k_cache_codes, np.uint8)
    vc = _c(v_cache_codes, np.uint8)
    bt = _c(block_tables, np.int32)
    sl = _c(seq_lens, np.int32)
    sel = None if select is None else _c(select, np.int64)
    n = B if sel is None else sel.size
    out = np.empty((n, Hq, D), dtype=np.float64)
    _check(_load().oracle_paged_attention_decode_fp8(
        _ptr(out), _ptr(q_bits), _ptr(kc), _ptr(vc), _ptr(bt), bt.shape[1], _ptr(sl), B, NB, Hq, Hkv, D, bs,
        float(scale), _DT[q_dtype], float(k_scale), float(v_scale), _ptr(sel),
        0 if sel is None else sel.size, threads))
    return out


def paged_attention_prefill_fp8(q_bits, k_cache_codes, v_cache_codes, block_tables, seq_lens, q_lens,
                                scale: float, q_dtype: str, k_scale: float, v_scale: float, select=None,
                                threads: int = 0) -> np.ndarray:
    """fp64 causal varlen attention over a head-major E4M3 cache [NB, Hkv, bs, D]
    (values = code * scale): q [T, Hq, D] -> out [n, Hq, D] (n = T or len(select))."""
    q_bits = _c(q_bits, np.uint16)
    T, Hq, D = q_bits.shape
    NB, Hkv, bs, D2 = k_cache_codes.shape
    assert D2 == D
    kc = _c(k_cache_codes, np.uint8)
    vc = _c(v_cache_codes, np.uint8)
    bt = _c(block_tables, np.int32)
    sl = _c(seq_lens, np.int32)
    ql = _c(q_lens, np.int32)
    assert int(ql.sum()) == T
    sel = None if select is None else _c(select, np.int64)
    n = T if sel is None else sel.size
    out = np.empty((n, Hq, D), dtype=np.float64)
    _check(_load().oracle_paged_attention_prefill_fp8(
        _ptr(out), _ptr(q_bits), _ptr(kc), _ptr(vc), _ptr(bt), bt.shape[1], _ptr(sl), _ptr(ql), sl.size, NB,
        Hq, Hkv, D, bs, float(scale), _DT[q_dtype], float(k_scale), float(v_scale), _ptr(sel),
        0 if sel is None else sel.size, threads))
    return out
