"""ctypes binding of libpagedattn.so (declared in include/pagedattn.h).

Argument marshalling only: shape/dtype/device checks, ``data_ptr()`` and the
current CUDA stream go in, a status code comes out.  Every step of the path
runs in the library's kernels; there is no fallback of any kind.  Scratch
space is allocated here with torch (caller-owned memory for the library).
"""
from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_NAME = "libpagedattn.so"

PA_BLOCK_SIZE = 16
PA_DEFAULT_PARTITION = 512
_DTYPES = {torch.float16: 0, torch.bfloat16: 1}
_STATUS = {0: "PA_OK", 1: "PA_ERR_INVALID_ARG", 2: "PA_ERR_UNSUPPORTED",
           3: "PA_ERR_WORKSPACE_TOO_SMALL", 4: "PA_ERR_CUDA"}

_p = ctypes.c_void_p
_i32 = ctypes.c_int
_f32 = ctypes.c_float
_sz = ctypes.c_size_t

_SIGNATURES = {
    "pa_version": (_i32, []),
    "pa_status_string": (ctypes.c_char_p, [_i32]),
    "pa_slot_mapping": (_i32, [_p, _p, _i32, _p, _p, _i32, _i32, _i32, _i32, _p]),
    "pa_paged_kv_write": (_i32, [_p, _p, _p, _p, _p, _i32, _i32, _i32, _i32, _i32, _i32, _p]),
    "pa_decode_workspace_bytes": (_sz, [_i32, _i32, _i32, _i32, _i32]),
    "pa_paged_attention_decode": (_i32, [_p, _p, _p, _p, _p, _i32, _p, _i32, _i32, _i32, _f32,
                                         _i32, _i32, _i32, _i32, _i32, _p, _sz, _i32, _p]),
    "pa_prefill_workspace_bytes": (_sz, [_i32, _i32, _i32, _i32, _i32]),
    "pa_paged_attention_prefill": (_i32, [_p, _p, _p, _p, _p, _i32, _p, _p, _i32, _i32, _i32,
                                          _i32, _i32, _f32, _i32, _i32, _i32, _i32, _p, _sz,
                                          _i32, _p]),
    "pa_get_device_error": (_i32, [ctypes.POINTER(_i32), _i32, _p]),
    "pa_paged_attention_decode_noalloc": (_i32, [_p, _p, _p, _p, _p, _i32, _p, _i32, _i32, _i32, _f32,
                                                 _i32, _i32, _i32, _i32, _i32, _i32, _p]),
    "pa_paged_kv_write_fp8": (_i32, [_p, _p, _p, _p, _p, _i32, _i32, _i32, _i32, _i32, _i32, _f32, _f32, _p]),
    "pa_paged_attention_decode_fp8": (_i32, [_p, _p, _p, _p, _p, _i32, _p, _i32, _i32, _i32, _f32, _f32, _f32,
                                             _i32, _i32, _i32, _i32, _i32, _p, _sz, _i32, _p]),
    "pa_prefill_fp8_workspace_bytes": (_sz, [_i32, _i32, _i32, _i32, _i32, _i32, _i32, ctypes.c_int64]),
    "pa_paged_attention_prefill_fp8": (_i32, [_p, _p, _p, _p, _p, _i32, _p, _p, _i32, _i32, _i32, _i32, _i32,
                                              _f32, _f32, _f32, _i32, _i32, _i32, _i32, _p, _sz, _i32, _p]),
    "pa_copy_blocks": (_i32, [_p, _p, _p, _i32, _i32, _i32, _i32, _i32, _p]),
    "pa_decode_partition": (_i32, [_i32, _i32]),
    "pa_selftest_wait_timeout": (_i32, [_p]),
    "pa_paged_kv_gather": (_i32, [_p, _p, _p, _p, _p, _i32, _p, _p, _i32, _i32, _i32, _i32, _i32, _i32, _p]),
}


class PagedAttnError(RuntimeError):
    """A libpagedattn call returned a nonzero status, or the library is missing."""


_lib = None


def library_path() -> str:
    return os.path.join(_HERE, _LIB_NAME)


def load_library():
    """Load libpagedattn.so from the package directory (raises if it is not built)."""
    global _lib
    if _lib is not None:
        return _lib
    path = library_path()
    if not os.path.exists(path):
        raise PagedAttnError(
            f"{path} is missing: build it first (python -c 'import __graft_entry__ as g; g.build()')")
    lib = ctypes.CDLL(path)
    for name, (res, args) in _SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def _check(rc: int, what: str) -> None:
    if rc != 0:
        raise PagedAttnError(f"{what} failed: {_STATUS.get(rc, rc)}")


def _stream(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return int(stream.cuda_stream) if hasattr(stream, "cuda_stream") else int(stream)


def _dt(t: torch.Tensor) -> int:
    if t.dtype not in _DTYPES:
        raise PagedAttnError(f"unsupported dtype {t.dtype}")
    return _DTYPES[t.dtype]


def _need(cond: bool, msg: str) -> None:
    if not cond:
        raise PagedAttnError(msg)


def _cuda(*ts):
    for t in ts:
        if t is not None:
            _need(t.is_cuda and t.is_contiguous(), "tensors must be contiguous CUDA tensors")


def _ptr(t):
    return None if t is None else t.data_ptr()


# --------------------------------------------------------------------------

def slot_mapping(block_tables: torch.Tensor, seq_lens: torch.Tensor, cu_q_lens, num_tokens: int,
                 num_blocks: int, out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """int64 slot of every new token (the last q_len positions of each sequence)."""
    _cuda(block_tables, seq_lens, cu_q_lens)
    _need(block_tables.dtype == torch.int32 and seq_lens.dtype == torch.int32, "int32 tables")
    B = seq_lens.shape[0]
    if out is None:
        out = torch.empty(num_tokens, dtype=torch.int64, device=seq_lens.device)
    _cuda(out)
    rc = load_library().pa_slot_mapping(out.data_ptr(), block_tables.data_ptr(), block_tables.shape[1],
                                        seq_lens.data_ptr(), _ptr(cu_q_lens), B, num_tokens,
                                        num_blocks, PA_BLOCK_SIZE, _stream(stream))
    _check(rc, "pa_slot_mapping")
    return out


def paged_kv_write(key: torch.Tensor, value: torch.Tensor, k_cache: torch.Tensor,
                   v_cache: torch.Tensor, slot_mapping: torch.Tensor, stream=None) -> None:
    """In place: k_cache/v_cache[slot // 16, slot % 16] = key/value rows (slot < 0: skipped)."""
    _cuda(key, value, k_cache, v_cache, slot_mapping)
    _need(slot_mapping.dtype == torch.int64, "slot_mapping must be int64")
    NB, bs, H, D = k_cache.shape
    T = key.shape[0]
    _need(tuple(key.shape) == (T, H, D) and value.shape == key.shape, "key/value shape")
    _need(v_cache.shape == k_cache.shape and k_cache.dtype == key.dtype == value.dtype == v_cache.dtype,
          "cache shape/dtype")
    _need(slot_mapping.numel() >= T, "slot_mapping too short")
    rc = load_library().pa_paged_kv_write(key.data_ptr(), value.data_ptr(), k_cache.data_ptr(),
                                          v_cache.data_ptr(), slot_mapping.data_ptr(), T, NB, H, D,
                                          bs, _dt(key), _stream(stream))
    _check(rc, "pa_paged_kv_write")


def selftest_wait_timeout(stream=None) -> None:
    """Enqueue the failure-path self-test (a bounded wait that runs out after
    about a second and records PA_DEVERR_TIMEOUT)."""
    _check(load_library().pa_selftest_wait_timeout(_stream(stream)), "pa_selftest_wait_timeout")


def decode_partition(max_seq_len: int, partition_size: int = 0) -> int:
    """Partition length (tokens) a decode call uses; 0 selects the automatic one."""
    n = int(load_library().pa_decode_partition(max_seq_len, partition_size))
    _need(n > 0, "invalid max_seq_len or partition_size")
    return n


def decode_workspace_bytes(num_seqs: int, num_q_heads: int, head_dim: int, max_seq_len: int,
                           partition_size: int = 0) -> int:
    return int(load_library().pa_decode_workspace_bytes(num_seqs, num_q_heads, head_dim, max_seq_len,
                                                        partition_size))


def prefill_workspace_bytes(num_seqs: int, num_tokens: int, num_q_heads: int, head_dim: int,
                            max_seq_len: int) -> int:
    return int(load_library().pa_prefill_workspace_bytes(num_seqs, num_tokens, num_q_heads, head_dim,
                                                         max_seq_len))


def prefill_fp8_workspace_bytes(num_seqs: int, num_tokens: int, num_q_heads: int, num_kv_heads: int,
                                head_dim: int, max_seq_len: int, max_blocks_per_seq: int,
                                chunk_kv_tokens: int) -> int:
    return int(load_library().pa_prefill_fp8_workspace_bytes(num_seqs, num_tokens, num_q_heads, num_kv_heads,
                                                             head_dim, max_seq_len, max_blocks_per_seq,
                                                             chunk_kv_tokens))


def count_chunk_kv_tokens(seq_lens: torch.Tensor, cu_q_lens: torch.Tensor) -> int:
    """Sum of seq_lens over the rows with more than 8 new tokens (the FP8
    prefill copy's size argument), from host copies of the two arrays."""
    sl = seq_lens.detach().to("cpu", torch.int64)
    cu = cu_q_lens.detach().to("cpu", torch.int64)
    return int(sl[(cu[1:] - cu[:-1]) > 8].sum())


def _workspace(nbytes: int, device, workspace):
    if nbytes == 0:
        return workspace
    if workspace is not None and workspace.numel() * workspace.element_size() >= nbytes:
        return workspace
    return torch.empty(nbytes, dtype=torch.uint8, device=device)


def paged_attention_decode(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                           block_tables: torch.Tensor, seq_lens: torch.Tensor, scale: float,
                           max_seq_len: int | None = None, out: torch.Tensor | None = None,
                           partition_size: int = 0, workspace: torch.Tensor | None = None,
                           stream=None) -> torch.Tensor:
    """Decode attention: q [B, Hq, D] -> out [B, Hq, D] over the paged cache."""
    _cuda(q, k_cache, v_cache, block_tables, seq_lens, out, workspace)
    B, Hq, D = q.shape
    NB, bs, Hkv, D2 = k_cache.shape
    _need(D2 == D and v_cache.shape == k_cache.shape, "cache shape")
    _need(block_tables.dtype == torch.int32 and seq_lens.dtype == torch.int32, "int32 tables")
    if max_seq_len is None:
        max_seq_len = int(seq_lens.max().item()) if B else 0
    if out is None:
        out = torch.empty_like(q)
    nbytes = decode_workspace_bytes(B, Hq, D, max_seq_len, partition_size)
    workspace = _workspace(nbytes, q.device, workspace)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    rc = load_library().pa_paged_attention_decode(
        out.data_ptr(), q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(), block_tables.data_ptr(),
        block_tables.shape[1], seq_lens.data_ptr(), B, max_seq_len, NB, float(scale), Hq, Hkv, D, bs,
        partition_size, _ptr(workspace), ws_bytes, _dt(q), _stream(stream))
    _check(rc, "pa_paged_attention_decode")
    return out


def paged_attention_prefill(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                            block_tables: torch.Tensor, seq_lens: torch.Tensor,
                            cu_q_lens: torch.Tensor, scale: float, max_q_len: int,
                            max_seq_len: int, out: torch.Tensor | None = None,
                            workspace: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Causal varlen attention of new query rows over the paged cache.

    Chunks of at most PA_VERIFY_MAX_Q (8) queries -- decodes and speculative
    verify steps -- run in the decode kernel, longer chunks in the prefill
    kernels."""
    _cuda(q, k_cache, v_cache, block_tables, seq_lens, cu_q_lens, out, workspace)
    T, Hq, D = q.shape
    NB, bs, Hkv, D2 = k_cache.shape
    _need(D2 == D and v_cache.shape == k_cache.shape, "cache shape")
    B = seq_lens.shape[0]
    _need(cu_q_lens.shape[0] == B + 1 and cu_q_lens.dtype == torch.int32, "cu_q_lens")
    if out is None:
        out = torch.empty_like(q)
    nbytes = prefill_workspace_bytes(B, T, Hq, D, max_seq_len)
    workspace = _workspace(nbytes, q.device, workspace)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    rc = load_library().pa_paged_attention_prefill(
        out.data_ptr(), q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(), block_tables.data_ptr(),
        block_tables.shape[1], seq_lens.data_ptr(), cu_q_lens.data_ptr(), B, T, max_q_len, max_seq_len,
        NB, float(scale), Hq, Hkv, D, bs, _ptr(workspace), ws_bytes, _dt(q), _stream(stream))
    _check(rc, "pa_paged_attention_prefill")
    return out


def copy_blocks(k_cache: torch.Tensor, v_cache: torch.Tensor, pairs: torch.Tensor, stream=None) -> None:
    """In place: block pairs[i, 1] of both pools receives block pairs[i, 0]
    (the copy-on-write step; pairs is a device int32 [n, 2] tensor)."""
    _cuda(k_cache, v_cache, pairs)
    _need(pairs.dtype == torch.int32 and pairs.dim() == 2 and pairs.shape[1] == 2, "pairs: int32 [n, 2]")
    _need(v_cache.shape == k_cache.shape and v_cache.dtype == k_cache.dtype, "cache shape/dtype")
    NB, bs, H, D = k_cache.shape
    rc = load_library().pa_copy_blocks(k_cache.data_ptr(), v_cache.data_ptr(), pairs.data_ptr(), pairs.shape[0],
                                       NB, H, D, k_cache.element_size(), _stream(stream))
    _check(rc, "pa_copy_blocks")


def paged_kv_gather(k_cache: torch.Tensor, v_cache: torch.Tensor, block_tables: torch.Tensor,
                    seq_lens: torch.Tensor, max_seq_len: int, stream=None):
    """Test support: every sequence's live K/V rows, gathered through its block
    table into contiguous [sum(seq_lens), Hkv, D] tensors.  16-bit pools are
    [NB, 16, Hkv, D]; one-byte (FP8) pools are head-major [NB, Hkv, 16, D]."""
    _cuda(k_cache, v_cache, block_tables, seq_lens)
    _need(block_tables.dtype == torch.int32 and seq_lens.dtype == torch.int32, "int32 tables")
    _need(v_cache.shape == k_cache.shape and v_cache.dtype == k_cache.dtype, "cache shape/dtype")
    if k_cache.element_size() == 1:
        NB, H, bs, D = k_cache.shape
    else:
        NB, bs, H, D = k_cache.shape
    B = seq_lens.shape[0]
    cu = torch.zeros(B + 1, dtype=torch.int32, device=seq_lens.device)
    torch.cumsum(seq_lens, 0, out=cu[1:])
    total = int(cu[-1])
    k_out = torch.empty(total, H, D, dtype=k_cache.dtype, device=k_cache.device)
    v_out = torch.empty_like(k_out)
    rc = load_library().pa_paged_kv_gather(k_out.data_ptr(), v_out.data_ptr(), k_cache.data_ptr(),
                                           v_cache.data_ptr(), block_tables.data_ptr(), block_tables.shape[1],
                                           seq_lens.data_ptr(), cu.data_ptr(), B, max_seq_len, NB, H, D,
                                           k_cache.element_size(), _stream(stream))
    _check(rc, "pa_paged_kv_gather")
    return k_out, v_out


def device_error(clear: bool = True, stream=None) -> int:
    """Device error word (PA_DEVERR_* bits); synchronises the stream."""
    code = ctypes.c_int(0)
    _check(load_library().pa_get_device_error(ctypes.byref(code), int(clear), _stream(stream)),
           "pa_get_device_error")
    return code.value


# --------------------------------------------------------------------------
# FP8 (E4M3) cache
# --------------------------------------------------------------------------

def _u8(t: torch.Tensor) -> torch.Tensor:
    _need(t.element_size() == 1, "FP8 caches hold one byte per element")
    return t


def paged_kv_write_fp8(key: torch.Tensor, value: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                       slot_mapping: torch.Tensor, k_scale: float, v_scale: float, stream=None) -> None:
    """In place: E4M3 codes of key/value * (1 / scale) into the head-major FP8
    pools [NB, Hkv, 16, D] (slot < 0: skipped)."""
    _cuda(key, value, k_cache, v_cache, slot_mapping)
    _u8(k_cache), _u8(v_cache)
    _need(slot_mapping.dtype == torch.int64, "slot_mapping must be int64")
    NB, H, bs, D = k_cache.shape
    T = key.shape[0]
    _need(tuple(key.shape) == (T, H, D) and value.shape == key.shape and v_cache.shape == k_cache.shape,
          "key/value/cache shapes")
    rc = load_library().pa_paged_kv_write_fp8(key.data_ptr(), value.data_ptr(), k_cache.data_ptr(),
                                              v_cache.data_ptr(), slot_mapping.data_ptr(), T, NB, H, D, bs,
                                              _dt(key), float(k_scale), float(v_scale), _stream(stream))
    _check(rc, "pa_paged_kv_write_fp8")


def paged_attention_decode_fp8(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                               block_tables: torch.Tensor, seq_lens: torch.Tensor, scale: float, k_scale: float,
                               v_scale: float, max_seq_len: int | None = None, out: torch.Tensor | None = None,
                               partition_size: int = 0, workspace: torch.Tensor | None = None,
                               stream=None) -> torch.Tensor:
    """Decode attention over head-major FP8 (E4M3) pools [NB, Hkv, 16, 128]:
    q [B, Hq, 128] -> out [B, Hq, 128]."""
    _cuda(q, k_cache, v_cache, block_tables, seq_lens, out, workspace)
    _u8(k_cache), _u8(v_cache)
    B, Hq, D = q.shape
    NB, Hkv, bs, D2 = k_cache.shape
    _need(D2 == D and v_cache.shape == k_cache.shape, "cache shape")
    if max_seq_len is None:
        max_seq_len = int(seq_lens.max().item()) if B else 0
    if out is None:
        out = torch.empty_like(q)
    nbytes = decode_workspace_bytes(B, Hq, D, max_seq_len, partition_size)
    workspace = _workspace(nbytes, q.device, workspace)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    rc = load_library().pa_paged_attention_decode_fp8(
        out.data_ptr(), q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(), block_tables.data_ptr(),
        block_tables.shape[1], seq_lens.data_ptr(), B, max_seq_len, NB, float(scale), float(k_scale),
        float(v_scale), Hq, Hkv, D, bs, partition_size, _ptr(workspace), ws_bytes, _dt(q), _stream(stream))
    _check(rc, "pa_paged_attention_decode_fp8")
    return out


def paged_attention_prefill_fp8(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                                block_tables: torch.Tensor, seq_lens: torch.Tensor, cu_q_lens: torch.Tensor,
                                scale: float, k_scale: float, v_scale: float, max_q_len: int, max_seq_len: int,
                                out: torch.Tensor | None = None, workspace: torch.Tensor | None = None,
                                stream=None, chunk_kv_tokens: int | None = None) -> torch.Tensor:
    """Causal varlen attention of new query rows over head-major FP8 (E4M3)
    pools [NB, Hkv, 16, 128] (decodes, speculative-verify rows and prefill
    chunks in one call).  `chunk_kv_tokens` sizes the chunks' 16-bit copy
    (see `count_chunk_kv_tokens()`); when it is None and a chunk can be longer than
    8 queries, it is computed from host copies of seq_lens and cu_q_lens."""
    _cuda(q, k_cache, v_cache, block_tables, seq_lens, cu_q_lens, out, workspace)
    _u8(k_cache), _u8(v_cache)
    T, Hq, D = q.shape
    NB, Hkv, bs, D2 = k_cache.shape
    _need(D2 == D and v_cache.shape == k_cache.shape, "cache shape")
    B = seq_lens.shape[0]
    _need(cu_q_lens.shape[0] == B + 1 and cu_q_lens.dtype == torch.int32, "cu_q_lens")
    if out is None:
        out = torch.empty_like(q)
    if max_q_len > 8 and B > 0 and T > 0:
        if chunk_kv_tokens is None:
            chunk_kv_tokens = count_chunk_kv_tokens(seq_lens, cu_q_lens)
        nbytes = prefill_fp8_workspace_bytes(B, T, Hq, Hkv, D, max_seq_len, block_tables.shape[1],
                                             chunk_kv_tokens)
    else:
        nbytes = prefill_workspace_bytes(B, T, Hq, D, max_seq_len)
    workspace = _workspace(nbytes, q.device, workspace)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    rc = load_library().pa_paged_attention_prefill_fp8(
        out.data_ptr(), q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(), block_tables.data_ptr(),
        block_tables.shape[1], seq_lens.data_ptr(), cu_q_lens.data_ptr(), B, T, max_q_len, max_seq_len, NB,
        float(scale), float(k_scale), float(v_scale), Hq, Hkv, D, bs, _ptr(workspace), ws_bytes, _dt(q),
        _stream(stream))
    _check(rc, "pa_paged_attention_prefill_fp8")
    return out
