"""Full-size workloads, in the launch configuration the benchmark times
(default 512-token partitions): the whole step runs on the GPU, and the fp64
oracle checks the slot mapping and the written rows bit-exactly and the
attention output of a sample of sequences (rows) within tolerance."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_attention_decode_gb300 as pa
from paged_kv_attention_decode_gb300 import workloads as W
from tests._gpu_util import TOL, bits, gpu_step, max_err, oracle_rows, snapshot

pytestmark = [pytest.mark.gpu, pytest.mark.slow]
DEV = "cuda"


def _check_cache(w, slots):
    ref = oracle.slot_mapping(w.block_tables, w.seq_lens, w.q_lens, 16, w.num_blocks)
    assert np.array_equal(slots.cpu().numpy(), ref)
    flat_k = w.k_cache.view(-1, w.num_kv_heads, w.head_dim)
    flat_v = w.v_cache.view(-1, w.num_kv_heads, w.head_dim)
    assert torch.equal(flat_k[slots].view(torch.int16), w.key.view(torch.int16))
    assert torch.equal(flat_v[slots].view(torch.int16), w.value.view(torch.int16))


@pytest.mark.parametrize("name,sample", [
    ("llama7b_decode", None), ("llama7b_ctx4096", 16), ("gqa_prefix", 48), ("long_context", None),
])
def test_full_decode_config(name, sample):
    w = W.make(name, device=DEV)
    rng = np.random.default_rng(12)
    seqs = np.arange(w.batch) if sample is None else np.sort(rng.choice(w.batch, sample, replace=False))
    snap = snapshot(w, seqs)
    slots, out = gpu_step(w)
    _check_cache(w, slots)
    rows, ref = oracle_rows(w, seqs, snap)
    err = max_err(out[torch.from_numpy(rows).to(DEV)], ref)
    assert err <= TOL[w.dtype], err
    assert pa.device_error() == 0
    del w
    torch.cuda.empty_cache()


def test_full_mixed_step():
    w = W.make("mixed", device=DEV)
    rng = np.random.default_rng(13)
    pre = np.nonzero(w.q_lens > 1)[0]
    dec = np.sort(rng.choice(np.nonzero(w.q_lens == 1)[0], 64, replace=False))
    seqs = np.sort(np.concatenate([pre, dec]))
    snap = snapshot(w, seqs)
    slots, out = gpu_step(w)
    _check_cache(w, slots)

    def pick(b, ql):
        if ql == 1:
            return [0]
        fixed = [0, 1, 15, 16, 63, 64, 65, ql // 2, ql - 2, ql - 1]
        extra = np.random.default_rng(b).choice(ql, 6, replace=False).tolist()
        return sorted(set(fixed + extra))

    rows, ref = oracle_rows(w, seqs, snap, q_rows_per_seq=pick)
    err = max_err(out[torch.from_numpy(rows).to(DEV)], ref)
    assert err <= TOL["bf16"], err
    assert pa.device_error() == 0
    del w
    torch.cuda.empty_cache()


def test_full_prefill():
    """The prefill-only workload the benchmark times (16 chunks of 1536 on
    prefixes up to 4096; the tcgen05 kernel alone on the GPU, items in the
    cost-sorted snake order): chunk edges, tile edges and random rows of every
    chunk against the oracle."""
    w = W.make("prefill", device=DEV)
    seqs = np.arange(w.batch)
    snap = snapshot(w, seqs)
    slots, out = gpu_step(w)
    _check_cache(w, slots)

    def pick(b, ql):
        fixed = [0, 1, 31, 32, 63, 64, 127, 128, ql // 2, ql - 33, ql - 32, ql - 2, ql - 1]
        extra = np.random.default_rng(100 + b).choice(ql, 4, replace=False).tolist()
        return sorted(set(fixed + extra))

    rows, ref = oracle_rows(w, seqs, snap, q_rows_per_seq=pick)
    err = max_err(out[torch.from_numpy(rows).to(DEV)], ref)
    assert err <= TOL["bf16"], err
    assert pa.device_error() == 0
    del w
    torch.cuda.empty_cache()


def test_full_spec_verify():
    # 64 verify rows of 4 queries (3 drafts) on contexts up to 4K: every row
    w = W.make("spec_verify", device=DEV)
    seqs = np.arange(w.batch)
    snap = snapshot(w, seqs)
    slots, out = gpu_step(w)
    _check_cache(w, slots)
    rows, ref = oracle_rows(w, seqs, snap)
    err = max_err(out[torch.from_numpy(rows).to(DEV)], ref)
    assert err <= TOL[w.dtype], err
    assert pa.device_error() == 0
    del w
    torch.cuda.empty_cache()
