"""The decode entry point that allocates nothing.

Some callers cannot allocate device memory when they run a decode step: an
inference runtime that gave all remaining HBM to its KV block pool, or a
plugin whose host framework forbids device allocation by extensions.  For
them pa_paged_attention_decode_noalloc keeps the split-context partials in a
fixed scratch array inside the library instead of a caller workspace.

These tests call it through the C ABI.  Its outputs must be bit-identical to
the ordinary decode entry point's (the same kernels with the same
partitioning) and within the decode tolerance of the fp64 oracle on a sample
of sequences.  The calls come in a row with different inputs and no other
kernel between them: the scratch array is shared by every call and keeps the
previous call's contents, and a call's work list must not be rewritten by the
next call while it still runs.  This file is collected last on purpose.
"""
import ctypes
import os
import subprocess
import sys

import numpy as np
import pytest
import torch

import oracle
import paged_kv_attention_decode_gb300 as pa
from paged_kv_attention_decode_gb300 import _binding
from paged_kv_attention_decode_gb300 import workloads as W
from tests._gpu_util import TOL, bits, max_err, snapshot

pytestmark = pytest.mark.gpu
DEV = "cuda"
SCRATCH = 32 << 20   # PA_NOALLOC_SCRATCH_BYTES
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _noalloc(lib, out, w, bt, sl, max_len, partition=0, num_seqs=None):
    stream = torch.cuda.current_stream().cuda_stream
    return lib.pa_paged_attention_decode_noalloc(
        out.data_ptr(), w.q.data_ptr(), w.k_cache.data_ptr(), w.v_cache.data_ptr(), bt.data_ptr(),
        bt.shape[1], sl.data_ptr(), w.batch if num_seqs is None else num_seqs, max_len, w.num_blocks,
        ctypes.c_float(w.scale), w.num_q_heads, w.num_kv_heads, w.head_dim, 16, partition,
        0 if w.dtype == "f16" else 1, stream)


def _oracle_sample(w, count, seed):
    seqs = np.sort(np.random.default_rng(seed).choice(w.batch, min(count, w.batch), replace=False))
    kc, vc, tables = snapshot(w, seqs)
    q = bits(w.q[torch.from_numpy(seqs).to(DEV)])
    ref = oracle.paged_attention_decode(q, kc, vc, tables, w.seq_lens[seqs], w.scale, w.dtype)
    return seqs, ref


def test_noalloc_matches_the_workspace_entry_point_and_the_oracle_on_calls_in_a_row():
    lib = _binding.load_library()
    rng = np.random.default_rng(5)
    cases = [
        # several partitions per sequence (split context + reduce), fp16 MHA
        W.make("llama7b_decode", device=DEV),
        # one partition each (no reduce between this call and the next), bf16 GQA 4:1
        W.build_workload(name="one_part_a", seq_lens=rng.integers(200, 513, 96), q_lens=1, num_q_heads=32,
                         num_kv_heads=8, head_dim=128, dtype="bf16", seed=77, device=DEV),
        # one partition each, fewer sequences, fp16 GQA 2:1 at head_dim 64
        W.build_workload(name="one_part_b", seq_lens=rng.integers(1, 400, 11), q_lens=1, num_q_heads=16,
                         num_kv_heads=8, head_dim=64, dtype="f16", seed=78, device=DEV),
    ]
    args = []
    for w in cases:
        bt = torch.from_numpy(w.block_tables).to(DEV)
        sl = torch.from_numpy(w.seq_lens).to(DEV)
        need = pa.decode_workspace_bytes(w.batch, w.num_q_heads, w.head_dim, w.max_seq_len, 0)
        assert 0 < need <= SCRATCH
        ref = pa.paged_attention_decode(w.q, w.k_cache, w.v_cache, bt, sl, w.scale, w.max_seq_len)
        args.append((w, bt, sl, ref))
    # the oracle's view of a sample of each case, before anything else runs
    samples = [_oracle_sample(w, 6, 40 + i) for i, w in enumerate(cases)]
    outs = [torch.full_like(w.q, float("nan")) for w in cases]
    torch.cuda.synchronize()
    # three calls queued back to back, then the last two again in reverse order
    for order in ([0, 1, 2], [2, 1]):
        for i in order:
            w, bt, sl, _ = args[i]
            assert _noalloc(lib, outs[i], w, bt, sl, w.max_seq_len) == 0
        torch.cuda.synchronize()
        for i in order:
            w, _, _, ref = args[i]
            assert torch.equal(outs[i].view(torch.int16), ref.view(torch.int16)), w.name
            seqs, oref = samples[i]
            err = max_err(outs[i][torch.from_numpy(seqs).to(DEV)], oref)
            assert err <= TOL[w.dtype], (w.name, err)
            outs[i].fill_(float("nan"))
        torch.cuda.synchronize()
    assert pa.device_error() == 0


def test_noalloc_with_no_sequences_only_sets_up():
    lib = _binding.load_library()
    w = W.build_workload(name="empty", seq_lens=[16], q_lens=1, num_q_heads=8, num_kv_heads=8,
                         head_dim=128, dtype="f16", seed=2, device=DEV)
    bt = torch.from_numpy(w.block_tables).to(DEV)
    sl = torch.from_numpy(w.seq_lens).to(DEV)
    out = torch.zeros_like(w.q)
    torch.cuda.synchronize()
    assert _noalloc(lib, out, w, bt, sl, 16, num_seqs=0) == 0
    torch.cuda.synchronize()
    assert torch.count_nonzero(out) == 0


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


_LAZY_PROBE = r"""
import ctypes
import torch
from paged_kv_attention_decode_gb300 import _binding
lib = _binding.load_library()
torch.zeros(1, device="cuda")
torch.cuda.synchronize()
def call():
    return lib.pa_paged_attention_decode_noalloc(None, None, None, None, None, 1, None, 0, 16, 1,
                                                 ctypes.c_float(0.1), 8, 8, 128, 16, 0, 0, None)
f0 = torch.cuda.mem_get_info()[0]
rc1 = call()
f1 = torch.cuda.mem_get_info()[0]
rc2 = call()
f2 = torch.cuda.mem_get_info()[0]
print(rc1, rc2, f0 - f1, f1 - f2)
"""


def test_first_call_reserves_the_scratch_under_lazy_module_loading():
    """With lazy module loading the scratch array is reserved by the first call
    on a device, not when the library is loaded: a runtime that hands all free
    memory to its KV pool must make that call (num_seqs = 0 does only the
    set-up) before.  A fresh process, so that no earlier test loaded it."""
    env = dict(os.environ, CUDA_MODULE_LOADING="LAZY")
    r = subprocess.run([sys.executable, "-c", _LAZY_PROBE], cwd=ROOT, env=env, capture_output=True, text=True,
                       timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    rc1, rc2, first, second = (int(x) for x in r.stdout.split()[-4:])
    assert rc1 == 0 and rc2 == 0
    assert first >= SCRATCH, first          # the first call reserved the array
    assert abs(second) < (2 << 20), second  # later calls reserve nothing
