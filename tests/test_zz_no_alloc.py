"""The decode entry point that allocates nothing.

Some callers cannot allocate device memory when they run a decode step: an
inference runtime that gave all remaining HBM to its KV block pool, or a
plugin whose host framework forbids device allocation by extensions.  For
them pa_paged_attention_decode_noalloc keeps the split-context partials in a
fixed scratch array inside the library instead of a caller workspace.  These
tests call it through the C ABI and hold its output to the ordinary decode
entry point's, within the decode tolerance, on two calls in a row with
different inputs (the scratch array is shared by every call and keeps the
previous call's contents).  This file is collected last on purpose.
"""
import ctypes

import numpy as np
import pytest
import torch

import paged_kv_attention_decode_gb300 as pa
from paged_kv_attention_decode_gb300 import _binding
from paged_kv_attention_decode_gb300 import workloads as W

pytestmark = pytest.mark.gpu
DEV = "cuda"
TOL = {"f16": 2e-3, "bf16": 1.6e-2}
SCRATCH = 32 << 20   # PA_NOALLOC_SCRATCH_BYTES


def _noalloc(lib, out, w, bt, sl, max_len, partition=0):
    stream = torch.cuda.current_stream().cuda_stream
    return lib.pa_paged_attention_decode_noalloc(
        out.data_ptr(), w.q.data_ptr(), w.k_cache.data_ptr(), w.v_cache.data_ptr(), bt.data_ptr(),
        bt.shape[1], sl.data_ptr(), w.batch, max_len, w.num_blocks, ctypes.c_float(w.scale),
        w.num_q_heads, w.num_kv_heads, w.head_dim, 16, partition, 0 if w.dtype == "f16" else 1, stream)


def test_noalloc_matches_the_workspace_entry_point_on_two_calls():
    lib = _binding.load_library()
    cases = [W.make("llama7b_decode", device=DEV),
             W.build_workload(name="second", seq_lens=np.arange(1, 40) * 97, q_lens=1, num_q_heads=32,
                              num_kv_heads=8, head_dim=128, dtype="bf16", seed=77, device=DEV)]
    for w in cases:
        bt = torch.from_numpy(w.block_tables).to(DEV)
        sl = torch.from_numpy(w.seq_lens).to(DEV)
        need = pa.decode_workspace_bytes(w.batch, w.num_q_heads, w.head_dim, w.max_seq_len, 0)
        assert 0 < need <= SCRATCH
        ref = pa.paged_attention_decode(w.q, w.k_cache, w.v_cache, bt, sl, w.scale, w.max_seq_len)
        out = torch.full_like(w.q, float("nan"))
        assert _noalloc(lib, out, w, bt, sl, w.max_seq_len) == 0
        torch.cuda.synchronize()
        assert torch.isfinite(out.float()).all()
        err = float((out.float() - ref.float()).abs().max())
        assert err <= TOL[w.dtype], err
        del w
    assert pa.device_error() == 0


def test_noalloc_rejects_sizes_beyond_its_scratch():
    lib = _binding.load_library()
    w = W.build_workload(name="big", seq_lens=[16], q_lens=1, num_q_heads=64, num_kv_heads=8,
                         head_dim=128, dtype="bf16", seed=1, device=DEV)
    bt = torch.from_numpy(w.block_tables).to(DEV)
    sl = torch.from_numpy(w.seq_lens).to(DEV)
    out = torch.zeros_like(w.q)
    # 64 heads x 1024 partitions of 16 tokens x (128 + 2) floats = 34 MB > 32 MiB
    assert pa.decode_workspace_bytes(1, 64, 128, 16 * 1024, 16) > SCRATCH
    assert _noalloc(lib, out, w, bt, sl, 16 * 1024, partition=16) == 3   # PA_ERR_WORKSPACE_TOO_SMALL
    torch.cuda.synchronize()
    assert torch.count_nonzero(out) == 0
