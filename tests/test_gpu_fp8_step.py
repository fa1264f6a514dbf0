"""GPU parity of a whole continuous-batching step over an FP8 (E4M3) cache:
prefill chunks on cached prefixes, speculative-verify rows and decode rows in
one call ("vLLM-Ascend 原理", section 4 "量化": the cache itself is quantised,
so every row kind dequantises what it reads through the block table).

The step runs through the library (slot mapping, quantising write, varlen
attention); the fp64 oracle writes the same codes into a copy of the pools
and attends.  The write is bit-exact; attention is within the tolerance of
the query dtype.  Dead pool slots hold the E4M3 NaN code, so a read of a slot
a row must not see makes the output non-finite.
"""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_attention_decode_gb300 as pa
from paged_kv_attention_decode_gb300 import workloads as W
from tests._gpu_util import TOL, bits

pytestmark = pytest.mark.gpu
DEV = "cuda"

# (context length, new tokens): chunks on prefixes (some longer than one
# 128-key tile, one starting at position 0), verify rows, decodes
STEP = [(300, 300), (1000, 37), (213, 9), (700, 513), (50, 2), (1500, 8), (90, 4), (2049, 1), (16, 1),
        (1, 1), (129, 128)]


def u8(t):
    return t.detach().contiguous().cpu().numpy().view(np.uint8)


def run_step(w):
    """slot mapping -> E4M3 write -> varlen attention through the library;
    returns (out, k_ref, v_ref) with the oracle's copy of the written pools."""
    sc = w.meta["kv_scale"]
    bt = torch.from_numpy(w.block_tables).to(DEV)
    sl = torch.from_numpy(w.seq_lens).to(DEV)
    cu = torch.from_numpy(w.cu_q_lens).to(DEV)
    k_ref, v_ref = u8(w.k_cache), u8(w.v_cache)
    slots = pa.slot_mapping(bt, sl, cu, w.num_tokens, w.num_blocks)
    pa.paged_kv_write_fp8(w.key, w.value, w.k_cache, w.v_cache, slots, sc, sc)
    out = pa.paged_attention_prefill_fp8(w.q, w.k_cache, w.v_cache, bt, sl, cu, w.scale, sc, sc, w.max_q_len,
                                         w.max_seq_len)
    torch.cuda.synchronize()
    ref_slots = oracle.slot_mapping(w.block_tables, w.seq_lens, w.q_lens, 16, w.num_blocks)
    assert np.array_equal(slots.cpu().numpy(), ref_slots)
    oracle.kv_write_fp8(bits(w.key), bits(w.value), k_ref, v_ref, ref_slots, w.dtype, sc, sc)
    assert np.array_equal(u8(w.k_cache), k_ref) and np.array_equal(u8(w.v_cache), v_ref)
    return out, k_ref, v_ref


def check(w, out, k_ref, v_ref):
    sc = w.meta["kv_scale"]
    ref = oracle.paged_attention_prefill_fp8(bits(w.q), k_ref, v_ref, w.block_tables, w.seq_lens, w.q_lens,
                                             w.scale, w.dtype, sc, sc)
    got = out.double().cpu().numpy()
    assert np.all(np.isfinite(got)), "non-finite output"
    err = float(np.max(np.abs(got - ref)))
    assert err <= TOL[w.dtype], err
    assert pa.device_error() == 0


@pytest.mark.parametrize("Hq,Hkv,dtype", [
    (8, 8, "f16"), (8, 8, "bf16"), (32, 8, "bf16"), (16, 2, "f16"), (24, 3, "bf16"), (32, 1, "f16"),
    (20, 4, "f16"), (64, 1, "bf16"),
])
def test_fp8_varlen_step(Hq, Hkv, dtype):
    lens = [n for n, _ in STEP]
    qlens = [c for _, c in STEP]
    w = W.build_workload(name="f8step", seq_lens=lens, q_lens=qlens, num_q_heads=Hq, num_kv_heads=Hkv,
                         head_dim=128, dtype=dtype, seed=Hq * 3 + Hkv, device=DEV, poison=True, pool_slack=0.3,
                         cache_dtype="fp8")
    check(w, *run_step(w))


@pytest.mark.parametrize("Hq,Hkv,dtype", [(8, 8, "bf16"), (32, 8, "f16"), (16, 1, "bf16")])
def test_fp8_verify_and_decode_rows_only(Hq, Hkv, dtype):
    # every row at most 8 queries: the call runs the decode kernel alone (one
    # or two tiles of 8 (query, head) columns per kv head)
    lens = [5, 17, 600, 1024, 33, 2, 4100, 8]
    qlens = [5, 8, 3, 1, 2, 2, 7, 8]
    w = W.build_workload(name="f8ver", seq_lens=lens, q_lens=qlens, num_q_heads=Hq, num_kv_heads=Hkv,
                         head_dim=128, dtype=dtype, seed=Hq + 5 * Hkv, device=DEV, poison=True, pool_slack=0.3,
                         cache_dtype="fp8")
    check(w, *run_step(w))


def test_fp8_chunks_alone_on_many_tiles():
    # prefill chunks only, several query-tile pairs each, long prefixes
    lens = [3000, 2100, 640]
    qlens = [900, 1100, 640]
    w = W.build_workload(name="f8chunks", seq_lens=lens, q_lens=qlens, num_q_heads=32, num_kv_heads=8,
                         head_dim=128, dtype="bf16", seed=71, device=DEV, poison=True, pool_slack=0.2,
                         cache_dtype="fp8")
    check(w, *run_step(w))


def test_fp8_chunks_that_do_not_fit_the_copy_are_skipped():
    """Chunks take 16-bit copy blocks in sequence order.  With room for the
    first chunk's 19 blocks only, the second chunk (63 blocks) and every later
    one are skipped: their rows keep what was there and PA_DEVERR_WORKSPACE is
    set.  The first chunk and the decode rows are still exact."""
    lens, qlens = [300, 1000, 213, 50, 700], [300, 37, 9, 1, 1]
    w = W.build_workload(name="f8cap", seq_lens=lens, q_lens=qlens, num_q_heads=16, num_kv_heads=4,
                         head_dim=128, dtype="bf16", seed=19, device=DEV, poison=True, pool_slack=0.3,
                         cache_dtype="fp8")
    sc = w.meta["kv_scale"]
    bt = torch.from_numpy(w.block_tables).to(DEV)
    sl = torch.from_numpy(w.seq_lens).to(DEV)
    cu = torch.from_numpy(w.cu_q_lens).to(DEV)
    k_ref, v_ref = u8(w.k_cache), u8(w.v_cache)
    slots = pa.slot_mapping(bt, sl, cu, w.num_tokens, w.num_blocks)
    pa.paged_kv_write_fp8(w.key, w.value, w.k_cache, w.v_cache, slots, sc, sc)
    oracle.kv_write_fp8(bits(w.key), bits(w.value), k_ref, v_ref,
                        oracle.slot_mapping(w.block_tables, w.seq_lens, w.q_lens, 16, w.num_blocks), w.dtype, sc, sc)
    B, T, mb = w.batch, w.num_tokens, w.max_blocks_per_seq
    per = 2 * 16 * w.num_kv_heads * 128 * 2
    slack = min(B, T // 9) * per                      # the size function's one partial block per chunk
    fixed = pa.prefill_fp8_workspace_bytes(B, T, w.num_q_heads, w.num_kv_heads, 128, w.max_seq_len, mb, 0) - slack
    ws = torch.empty(fixed + 19 * per, dtype=torch.uint8, device=DEV)
    out = torch.full_like(w.q, 7.0)
    pa.device_error()
    pa.paged_attention_prefill_fp8(w.q, w.k_cache, w.v_cache, bt, sl, cu, w.scale, sc, sc, w.max_q_len,
                                   w.max_seq_len, out=out, workspace=ws, chunk_kv_tokens=0)
    assert pa.device_error() == 16                    # PA_DEVERR_WORKSPACE
    ref = oracle.paged_attention_prefill_fp8(bits(w.q), k_ref, v_ref, w.block_tables, w.seq_lens, w.q_lens,
                                             w.scale, w.dtype, sc, sc)
    got = out.double().cpu().numpy()
    cu_np = w.cu_q_lens
    done = np.r_[cu_np[0]:cu_np[1], cu_np[3]:cu_np[5]]     # chunk 0 and the two decode rows
    skipped = np.r_[cu_np[1]:cu_np[3]]
    assert float(np.max(np.abs(got[done] - ref[done]))) <= TOL["bf16"]
    assert np.all(got[skipped] == 7.0)


def test_fp8_bad_block_id_in_a_chunk_is_masked_and_flagged():
    """A live table entry outside the pool in a long chunk's cached prefix:
    its copy block is marked not loaded, the prefill kernel masks it and sets
    PA_DEVERR_BLOCK_ID, the chunk's rows stay finite, and the other rows match
    the oracle."""
    lens, qlens = [300, 1000, 50, 700], [300, 37, 1, 1]
    w = W.build_workload(name="f8bad", seq_lens=lens, q_lens=qlens, num_q_heads=16, num_kv_heads=4,
                         head_dim=128, dtype="bf16", seed=23, device=DEV, poison=True, pool_slack=0.3,
                         cache_dtype="fp8")
    sc = w.meta["kv_scale"]
    bt = torch.from_numpy(w.block_tables).to(DEV)
    sl = torch.from_numpy(w.seq_lens).to(DEV)
    cu = torch.from_numpy(w.cu_q_lens).to(DEV)
    k_ref, v_ref = u8(w.k_cache), u8(w.v_cache)
    slots = pa.slot_mapping(bt, sl, cu, w.num_tokens, w.num_blocks)
    pa.paged_kv_write_fp8(w.key, w.value, w.k_cache, w.v_cache, slots, sc, sc)
    oracle.kv_write_fp8(bits(w.key), bits(w.value), k_ref, v_ref,
                        oracle.slot_mapping(w.block_tables, w.seq_lens, w.q_lens, 16, w.num_blocks), w.dtype, sc, sc)
    tables = w.block_tables.copy()
    tables[1, 10] = w.num_blocks + 3                # tokens 160-175 of the 1000-token sequence (its prefix)
    pa.device_error()
    out = pa.paged_attention_prefill_fp8(w.q, w.k_cache, w.v_cache, torch.from_numpy(tables).to(DEV), sl, cu,
                                         w.scale, sc, sc, w.max_q_len, w.max_seq_len)
    torch.cuda.synchronize()
    assert pa.device_error() == 1                   # PA_DEVERR_BLOCK_ID
    got = out.double().cpu().numpy()
    cu_np = w.cu_q_lens
    assert np.all(np.isfinite(got[cu_np[1]:cu_np[2]]))
    ref = oracle.paged_attention_prefill_fp8(bits(w.q), k_ref, v_ref, w.block_tables, w.seq_lens, w.q_lens,
                                             w.scale, w.dtype, sc, sc)
    others = np.r_[cu_np[0]:cu_np[1], cu_np[2]:cu_np[4]]
    assert float(np.max(np.abs(got[others] - ref[others]))) <= TOL["bf16"]


def test_fp8_prefill_rejects_other_head_dims():
    q = torch.zeros(4, 4, 64, device=DEV, dtype=torch.float16)
    kc = torch.zeros(4, 4, 16, 64, device=DEV, dtype=torch.uint8)
    bt = torch.zeros(1, 1, device=DEV, dtype=torch.int32)
    sl = torch.full((1,), 4, device=DEV, dtype=torch.int32)
    cu = torch.tensor([0, 4], device=DEV, dtype=torch.int32)
    with pytest.raises(pa.PagedAttnError):
        pa.paged_attention_prefill_fp8(q, kc, kc, bt, sl, cu, 0.1, 1.0, 1.0, 4, 4)


@pytest.mark.slow
@pytest.mark.parametrize("name", ["mixed_fp8", "prefill_fp8"])
def test_fp8_full_step_sampled(name):
    """The continuous-batching workload (4 chunks of 1536 on prefixes up to
    4096 and 2048 decodes, 32/8 heads) and the prefill-only one (16 chunks)
    with an E4M3 cache, as the benchmark times them: the whole step on the
    GPU; the oracle checks the slots and written codes bit for bit and a
    sample of rows (spread over every chunk, and 64 decodes) within tolerance."""
    w = W.make(name, device=DEV)
    sc = w.meta["kv_scale"]
    rng = np.random.default_rng(14)
    pre = np.nonzero(w.q_lens > 1)[0]
    decs = np.nonzero(w.q_lens == 1)[0]
    dec = np.sort(rng.choice(decs, 64, replace=False)) if decs.size else decs
    seqs = np.sort(np.concatenate([pre, dec]))
    # compact copy of the blocks those sequences use (their tables renumbered)
    used = np.unique(np.concatenate([w.block_tables[b, : -(-int(w.seq_lens[b]) // 16)] for b in seqs]))
    idx = torch.from_numpy(used.astype(np.int64)).to(DEV)
    k_snap, v_snap = u8(w.k_cache.index_select(0, idx)), u8(w.v_cache.index_select(0, idx))
    remap = {int(x): i for i, x in enumerate(used)}
    tables = np.zeros((len(seqs), w.max_blocks_per_seq), np.int32)
    for r, b in enumerate(seqs):
        lb = w.block_tables[b, : -(-int(w.seq_lens[b]) // 16)]
        tables[r, : lb.size] = [remap[int(x)] for x in lb]
    bt = torch.from_numpy(w.block_tables).to(DEV)
    sl = torch.from_numpy(w.seq_lens).to(DEV)
    cu = torch.from_numpy(w.cu_q_lens).to(DEV)
    slots = pa.slot_mapping(bt, sl, cu, w.num_tokens, w.num_blocks)
    pa.paged_kv_write_fp8(w.key, w.value, w.k_cache, w.v_cache, slots, sc, sc)
    out = pa.paged_attention_prefill_fp8(w.q, w.k_cache, w.v_cache, bt, sl, cu, w.scale, sc, sc, w.max_q_len,
                                         w.max_seq_len)
    torch.cuda.synchronize()
    assert np.array_equal(slots.cpu().numpy(), oracle.slot_mapping(w.block_tables, w.seq_lens, w.q_lens, 16,
                                                                   w.num_blocks))
    cu_np = w.cu_q_lens
    rows = np.concatenate([np.arange(cu_np[b], cu_np[b + 1]) for b in seqs]).astype(np.int64)
    rows_t = torch.from_numpy(rows).to(DEV)
    ql = w.q_lens[seqs]
    s2 = oracle.slot_mapping(tables, w.seq_lens[seqs], ql, 16, len(used))
    oracle.kv_write_fp8(bits(w.key[rows_t]), bits(w.value[rows_t]), k_snap, v_snap, s2, "bf16", sc, sc)
    # rows to compare: chunk edges and a spread inside each chunk, every decode
    sel, keep, base = [], [], 0
    for r, b in enumerate(seqs):
        n = int(ql[r])
        pick = [0] if n == 1 else sorted(set([0, 1, 63, 64, 127, 128, n // 2, n - 2, n - 1] +
                                             np.random.default_rng(int(b)).choice(n, 8, replace=False).tolist()))
        for i in pick:
            sel.append(base + i)
            keep.append(rows[base + i])
        base += n
    ref = oracle.paged_attention_prefill_fp8(bits(w.q[rows_t]), k_snap, v_snap, tables, w.seq_lens[seqs], ql,
                                             w.scale, "bf16", sc, sc, select=np.array(sel))
    got = out[torch.from_numpy(np.array(keep)).to(DEV)].double().cpu().numpy()
    assert np.all(np.isfinite(got))
    err = float(np.max(np.abs(got - ref)))
    assert err <= TOL["bf16"], err
    assert pa.device_error() == 0
    del w
    torch.cuda.empty_cache()
