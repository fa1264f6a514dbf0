"""GPU parity of speculative-decoding verify rows ("vLLM-Ascend 原理",
section 4 "推测解码": the drafts and the last accepted token form a short
mini-prefill whose k/v are written as it runs; rejected drafts are rolled back
by cutting the sequence length).  Chunks of 1..8 queries run in the decode
kernel; the fp64 oracle is the same causal definition as for any prefill."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_attention_decode_gb300 as pa
from paged_kv_attention_decode_gb300 import workloads as W
from tests._gpu_util import TOL, bits, gpu_step, max_err, oracle_rows, snapshot

pytestmark = pytest.mark.gpu
DEV = "cuda"

# (q_len, cached context before the step): every q_len 1..8; contexts inside
# one block, across block and 512-token partition boundaries (split context,
# partitions that some queries of the chunk cannot see), and q_len == seq_len.
CASES = [(1, 0), (2, 0), (8, 0), (3, 13), (4, 16), (5, 509), (8, 505), (6, 511), (7, 512), (2, 1024),
         (8, 1400), (4, 2047), (1, 700), (3, 1), (8, 33), (5, 3000)]


@pytest.mark.parametrize("Hq,Hkv,D,dtype", [
    (32, 8, 128, "bf16"), (8, 8, 128, "f16"), (16, 2, 128, "f16"), (6, 2, 64, "bf16"), (8, 4, 64, "f16"),
    (14, 2, 128, "bf16"), (12, 2, 64, "f16"),
    (32, 2, 128, "bf16"), (32, 1, 64, "f16"),      # 16 and 32 heads per kv head
])
def test_verify_rows_parity(Hq, Hkv, D, dtype):
    q_lens = [c[0] for c in CASES]
    seq_lens = [c[0] + c[1] for c in CASES]
    w = W.build_workload(name="verify", seq_lens=seq_lens, q_lens=q_lens, num_q_heads=Hq, num_kv_heads=Hkv,
                         head_dim=D, dtype=dtype, seed=Hq * 3 + D, device=DEV, poison=True, pool_slack=0.3)
    seqs = np.arange(w.batch)
    snap = snapshot(w, seqs)
    _, out = gpu_step(w, prefill=True)
    assert pa.device_error() == 0
    rows, ref = oracle_rows(w, seqs, snap)
    err = max_err(out[torch.from_numpy(rows).to(DEV)], ref)
    assert err <= TOL[dtype], err


def test_verify_rows_next_to_prefill_chunks():
    # one call: long chunks (tensor-core prefill), verify rows and decodes
    q_lens = [300, 4, 1, 9, 8, 1, 130, 2]
    ctx = [100, 600, 40, 0, 1030, 2, 0, 77]
    w = W.build_workload(name="verify_mixed", seq_lens=np.add(q_lens, ctx), q_lens=q_lens, num_q_heads=32,
                         num_kv_heads=8, head_dim=128, dtype="bf16", seed=5, device=DEV, poison=True)
    seqs = np.arange(w.batch)
    snap = snapshot(w, seqs)
    _, out = gpu_step(w, prefill=True)
    assert pa.device_error() == 0
    rows, ref = oracle_rows(w, seqs, snap)
    err = max_err(out[torch.from_numpy(rows).to(DEV)], ref)
    assert err <= TOL["bf16"], err


def test_verify_row_equals_decodes_of_its_queries():
    # query i of a chunk of L sits at position n - L + i: it must equal a
    # decode over the first n - L + i + 1 positions of the same cache
    w = W.make("spec_verify", device=DEV, batch=24, drafts=5)
    _, out = gpu_step(w, prefill=True)
    assert pa.device_error() == 0
    bt = torch.from_numpy(w.block_tables).to(DEV)
    L = int(w.q_lens[0])
    cu = torch.from_numpy(w.cu_q_lens).to(DEV)
    for i in range(L):
        sl = torch.from_numpy(w.seq_lens - (L - 1 - i)).to(DEV)
        qi = w.q[cu[:-1].long() + i].contiguous()
        dec = pa.paged_attention_decode(qi, w.k_cache, w.v_cache, bt, sl, w.scale, w.max_seq_len)
        torch.cuda.synchronize()
        diff = float((out[cu[:-1].long() + i].float() - dec.float()).abs().max())
        assert diff <= TOL["bf16"], (i, diff)


def test_rollback_by_truncation():
    """Verify 1 + k tokens, accept a of the drafts, cut seq_len back, then
    decode the next token into the first rejected slot: positions past the
    cut must not count, whatever the rejected slots hold."""
    k = 5
    ctx = np.array([29, 500, 1021, 60, 7, 250], dtype=np.int32)    # drafts cross blocks and a partition
    accepted = np.array([0, 5, 2, 3, 1, 4], dtype=np.int32)
    w = W.build_workload(name="verify_rollback", seq_lens=ctx + k + 1, q_lens=k + 1, num_q_heads=16,
                         num_kv_heads=4, head_dim=128, dtype="f16", seed=77, device=DEV, pool_slack=0.5)
    _, out = gpu_step(w, prefill=True)
    assert pa.device_error() == 0

    # truncate: keep the last accepted token and the accepted drafts
    new_len = ctx + 1 + accepted
    bt = torch.from_numpy(w.block_tables).to(DEV)
    flat_k = w.k_cache.view(-1, w.num_kv_heads, w.head_dim)
    flat_v = w.v_cache.view(-1, w.num_kv_heads, w.head_dim)
    # rejected slots may hold anything now
    for b in range(w.batch):
        for pos in range(int(new_len[b]), int(ctx[b] + k + 1)):
            slot = int(w.block_tables[b, pos // 16]) * 16 + pos % 16
            flat_k[slot] = float("nan")
            flat_v[slot] = float("nan")
    # next step: one decode token per sequence at position new_len
    gen = torch.Generator(device=DEV)
    gen.manual_seed(79)
    q = torch.randn(w.batch, 16, 128, generator=gen, device=DEV).half()
    key = torch.randn(w.batch, 4, 128, generator=gen, device=DEV).half()
    val = torch.randn(w.batch, 4, 128, generator=gen, device=DEV).half()
    sl = torch.from_numpy(new_len + 1).to(DEV)
    slots = pa.slot_mapping(bt, sl, None, w.batch, w.num_blocks)
    pa.paged_kv_write(key, val, w.k_cache, w.v_cache, slots)
    dec = pa.paged_attention_decode(q, w.k_cache, w.v_cache, bt, sl, w.scale, int(new_len.max()) + 1)
    torch.cuda.synchronize()
    assert pa.device_error() == 0

    # oracle on the live prefix only: positions 0 .. new_len (inclusive of the new token)
    used = np.unique(np.concatenate([w.block_tables[b, : -(-int(new_len[b] + 1) // 16)] for b in range(w.batch)]))
    idx = torch.from_numpy(used.astype(np.int64)).to(DEV)
    kc = bits(w.k_cache.index_select(0, idx))
    vc = bits(w.v_cache.index_select(0, idx))
    remap = {int(x): i for i, x in enumerate(used)}
    tables = np.zeros((w.batch, w.max_blocks_per_seq), dtype=np.int32)
    for b in range(w.batch):
        live = w.block_tables[b, : -(-int(new_len[b] + 1) // 16)]
        tables[b, : live.size] = [remap[int(x)] for x in live]
    ref = oracle.paged_attention_decode(bits(q), kc, vc, tables, (new_len + 1).astype(np.int32), w.scale, "f16")
    err = max_err(dec, ref)
    assert err <= TOL["f16"], err


def test_short_chunk_longer_than_max_q_len_is_flagged():
    # a chunk of 3 queries while the caller promised max_q_len = 2: zero rows
    # and PA_DEVERR_SEQ_LEN, the other rows unaffected
    w = W.build_workload(name="verify_bad", seq_lens=[40, 50], q_lens=[2, 3], num_q_heads=8, num_kv_heads=2,
                         head_dim=64, dtype="f16", seed=3, device=DEV)
    bt = torch.from_numpy(w.block_tables).to(DEV)
    sl = torch.from_numpy(w.seq_lens).to(DEV)
    cu = torch.from_numpy(w.cu_q_lens).to(DEV)
    seqs = np.arange(2)
    snap = snapshot(w, seqs)
    slots = pa.slot_mapping(bt, sl, cu, w.num_tokens, w.num_blocks)
    pa.paged_kv_write(w.key, w.value, w.k_cache, w.v_cache, slots)
    pa.device_error()
    out = pa.paged_attention_prefill(w.q, w.k_cache, w.v_cache, bt, sl, cu, w.scale, 2, w.max_seq_len)
    assert pa.device_error() == 4
    assert float(out[2:].float().abs().max()) == 0.0
    rows, ref = oracle_rows(w, seqs[:1], (snap[0], snap[1], snap[2][:1]))
    assert max_err(out[:2], ref) <= TOL["f16"]
