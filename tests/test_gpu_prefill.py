"""GPU parity of chunked-prefill (causal, varlen, on cached prefixes) and of
the mixed prefill + decode step against the fp64 oracle."""
import numpy as np
import pytest
import torch

import paged_kv_attention_decode_gb300 as pa
from paged_kv_attention_decode_gb300 import workloads as W
from tests._gpu_util import TOL, gpu_step, max_err, oracle_rows, snapshot

pytestmark = pytest.mark.gpu
DEV = "cuda"

# (q_len, cached prefix) per sequence: chunks shorter and longer than a tile,
# ragged block and tile tails, empty and long prefixes, decode rows mixed in,
# and a sequence with no new rows this step (q_len 0).
CASES = [(2, 0), (17, 0), (64, 0), (65, 3), (100, 200), (1, 50), (0, 40), (130, 1000), (33, 15), (1, 1),
         (300, 17)]


@pytest.mark.parametrize("Hq,Hkv,D,dtype", [
    (8, 2, 128, "bf16"), (4, 4, 64, "f16"), (32, 8, 128, "bf16"), (8, 1, 64, "bf16"), (6, 2, 128, "f16"),
    (16, 2, 128, "f16"),
    # groupings that do not divide 128 rows: tiles of 42, 25, 21 and 18 queries
    (28, 4, 128, "bf16"), (10, 2, 64, "f16"), (12, 2, 128, "bf16"), (7, 1, 128, "f16"),
    # 16, 32 and 64 heads per kv head: tiles of 8, 4 and 2 queries
    (32, 2, 128, "bf16"), (32, 1, 128, "f16"), (64, 1, 64, "bf16"),
])
def test_prefill_parity(Hq, Hkv, D, dtype):
    q_lens = [c[0] for c in CASES]
    seq_lens = [c[0] + c[1] for c in CASES]
    w = W.build_workload(name="pre", seq_lens=seq_lens, q_lens=q_lens, num_q_heads=Hq, num_kv_heads=Hkv,
                         head_dim=D, dtype=dtype, seed=Hq + 17 * D, device=DEV, poison=True, pool_slack=0.2)
    seqs = np.arange(w.batch)
    snap = snapshot(w, seqs)
    _, out = gpu_step(w, prefill=True)
    rows, ref = oracle_rows(w, seqs, snap)
    err = max_err(out[torch.from_numpy(rows).to(DEV)], ref)
    assert err <= TOL[dtype], err
    assert pa.device_error() == 0


@pytest.mark.parametrize("scale", [-0.09, 0.0, 3.0])
def test_prefill_any_scale(scale):
    """Scale is any finite number: negative (the softmax favours the smallest
    scores), zero (uniform weights over the visible keys) and large; the
    tensor-core kernel takes a different softmax path for non-positive scales."""
    q_lens = [c[0] for c in CASES]
    seq_lens = [c[0] + c[1] for c in CASES]
    w = W.build_workload(name="pre_scale", seq_lens=seq_lens, q_lens=q_lens, num_q_heads=8, num_kv_heads=2,
                         head_dim=128, dtype="bf16", seed=91, device=DEV, poison=True, pool_slack=0.2, scale=scale)
    assert w.scale == scale
    seqs = np.arange(w.batch)
    snap = snapshot(w, seqs)
    _, out = gpu_step(w, prefill=True)
    rows, ref = oracle_rows(w, seqs, snap)
    err = max_err(out[torch.from_numpy(rows).to(DEV)], ref)
    assert err <= TOL["bf16"], err
    assert pa.device_error() == 0


@pytest.mark.parametrize("D,dtype", [(128, "bf16"), (128, "f16"), (64, "bf16")])
def test_prefill_reference_moves_in_a_later_key_tile(D, dtype):
    """Keys grow key tile by key tile (K of tile i scaled by 2^i, exact in
    16-bit), so a later tile's scores pass the running reference by more than
    2^8: the kernel must notice it from the tile's sum of P, take the row
    maximum and rescale O and l.  The precondition is checked on the inputs."""
    Hq, Hkv, prefix, q_len = 8, 2, 440, 200
    w = W.build_workload(name="pre_grow", seq_lens=[prefix + q_len], q_lens=[q_len], num_q_heads=Hq,
                         num_kv_heads=Hkv, head_dim=D, dtype=dtype, seed=123, device=DEV, poison=True,
                         pool_slack=0.2)
    n = prefix + q_len
    factor = torch.tensor([2.0 ** (t // 128) for t in range(n)], dtype=torch.float32)
    for t in range(prefix):
        blk = int(w.block_tables[0, t // 16])
        w.k_cache[blk, t % 16] *= float(factor[t])
    w.key[:q_len] *= factor[prefix:].to(DEV, w.key.dtype).view(q_len, 1, 1)
    # precondition: some query row sees a key tile whose maximum passes the
    # running maximum of the earlier tiles by more than 8 (log2 units)
    k_all = torch.empty(n, Hkv, D, dtype=torch.float64)
    for t in range(prefix):
        k_all[t] = w.k_cache[int(w.block_tables[0, t // 16]), t % 16].double().cpu()
    k_all[prefix:] = w.key[:q_len].double().cpu()
    q = w.q[:q_len].double().cpu()
    G = Hq // Hkv
    jump = 0.0
    for i in range(0, q_len, 37):
        pos = prefix + i
        for h in range(Hq):
            s = (k_all[: pos + 1, h // G] @ q[i, h]).numpy() * w.scale * np.log2(np.e)
            run = -np.inf
            for k0 in range(0, pos + 1, 128):
                mx = s[k0:k0 + 128].max()
                if np.isfinite(run):
                    jump = max(jump, mx - run)
                run = max(run, mx)
    assert jump > 8.0, jump
    seqs = np.arange(w.batch)
    snap = snapshot(w, seqs)
    _, out = gpu_step(w, prefill=True)
    rows, ref = oracle_rows(w, seqs, snap)
    err = max_err(out[torch.from_numpy(rows).to(DEV)], ref)
    assert err <= TOL[dtype], err
    assert pa.device_error() == 0


@pytest.mark.parametrize("last_q,past", [(100, 50), (3, 1)])
def test_chunk_outside_the_rows_is_flagged(last_q, past):
    """The last chunk's rows run past the call's num_tokens rows (cu_q_lens
    inconsistent with q): no row of it is read or written, PA_DEVERR_SEQ_LEN
    is set, and the other chunks are computed as usual.  A long last chunk
    goes to the tensor-core kernel, a 3-query one to the decode kernel."""
    q_lens = [40, 1, 5, last_q]
    seq_lens = [90, 21, 35, last_q + 10]
    w = W.build_workload(name="rows", seq_lens=seq_lens, q_lens=q_lens, num_q_heads=8, num_kv_heads=2,
                         head_dim=128, dtype="bf16", seed=77, device=DEV)
    seqs = np.arange(w.batch - 1)
    snap = snapshot(w, seqs)
    bt = torch.from_numpy(w.block_tables).to(DEV)
    sl = torch.from_numpy(w.seq_lens).to(DEV)
    cu = torch.from_numpy(w.cu_q_lens).to(DEV)
    T = w.num_tokens
    slots = pa.slot_mapping(bt, sl, cu, T, w.num_blocks)
    pa.paged_kv_write(w.key, w.value, w.k_cache, w.v_cache, slots)
    cu_bad = cu.clone()
    cu_bad[-1] = T + past
    sentinel = 3.0
    out_full = torch.full((T + 64, 8, 128), sentinel, dtype=torch.bfloat16, device=DEV)
    out = out_full[:T]
    pa.device_error()
    pa.paged_attention_prefill(w.q, w.k_cache, w.v_cache, bt, sl, cu_bad, w.scale, max(q_lens) + past,
                               w.max_seq_len, out=out)
    torch.cuda.synchronize()
    assert pa.device_error() == 1 << 2          # PA_DEVERR_SEQ_LEN
    assert bool((out_full[T:] == sentinel).all())          # nothing past the rows
    assert bool((out[int(w.cu_q_lens[-2]):] == sentinel).all())   # the rejected chunk's rows untouched
    rows, ref = oracle_rows(w, seqs, snap)
    assert max_err(out[torch.from_numpy(rows).to(DEV)], ref) <= TOL["bf16"]


def test_bad_block_id_in_a_chunk_is_masked_and_flagged():
    """A live table entry outside the pool in a long chunk's cached prefix:
    the tensor-core kernel neither loads nor reads that block (its keys are
    masked, its V rows cleared), sets PA_DEVERR_BLOCK_ID and keeps the chunk's
    rows finite; the other sequences' rows match the oracle."""
    q_lens, seq_lens = [40, 1, 130, 9], [90, 21, 400, 35]
    w = W.build_workload(name="badpre", seq_lens=seq_lens, q_lens=q_lens, num_q_heads=8, num_kv_heads=2,
                         head_dim=128, dtype="bf16", seed=29, device=DEV, poison=True, pool_slack=0.2)
    seqs = np.array([0, 1, 3])
    snap = snapshot(w, seqs)
    bt = torch.from_numpy(w.block_tables).to(DEV)
    sl = torch.from_numpy(w.seq_lens).to(DEV)
    cu = torch.from_numpy(w.cu_q_lens).to(DEV)
    slots = pa.slot_mapping(bt, sl, cu, w.num_tokens, w.num_blocks)
    pa.paged_kv_write(w.key, w.value, w.k_cache, w.v_cache, slots)
    tables = w.block_tables.copy()
    tables[2, 3] = w.num_blocks + 7                 # tokens 48-63 of the 400-token sequence (its prefix)
    pa.device_error()
    out = pa.paged_attention_prefill(w.q, w.k_cache, w.v_cache, torch.from_numpy(tables).to(DEV), sl, cu,
                                     w.scale, w.max_q_len, w.max_seq_len)
    torch.cuda.synchronize()
    assert pa.device_error() == 1                   # PA_DEVERR_BLOCK_ID
    bad_rows = out[int(w.cu_q_lens[2]):int(w.cu_q_lens[3])]
    assert bool(torch.isfinite(bad_rows.float()).all())
    rows, ref = oracle_rows(w, seqs, snap)
    assert max_err(out[torch.from_numpy(rows).to(DEV)], ref) <= TOL["bf16"]


def test_mixed_step_small():
    w = W.make("mixed", device=DEV, poison=True, n_prefill=3, chunk=150, n_decode=40, prefix_hi=700,
               dec_lo=1, dec_hi=900)
    seqs = np.arange(w.batch)
    snap = snapshot(w, seqs)
    _, out = gpu_step(w)
    rows, ref = oracle_rows(w, seqs, snap)
    err = max_err(out[torch.from_numpy(rows).to(DEV)], ref)
    assert err <= TOL["bf16"], err
    assert pa.device_error() == 0


def test_pure_prefill_without_prefix_matches_decode_of_last_row():
    w = W.build_workload(name="pp", seq_lens=[77, 200], q_lens=[77, 200], num_q_heads=8, num_kv_heads=8,
                         head_dim=128, dtype="f16", seed=21, device=DEV)
    _, out = gpu_step(w, prefill=True)
    last = torch.tensor([76, 276], device=DEV)
    bt = torch.from_numpy(w.block_tables).to(DEV)
    sl = torch.from_numpy(w.seq_lens).to(DEV)
    dec = pa.paged_attention_decode(w.q[last].contiguous(), w.k_cache, w.v_cache, bt, sl, w.scale, 200)
    torch.cuda.synchronize()
    assert float((out[last].float() - dec.float()).abs().max()) <= 2e-3


def test_long_chunks_many_tiles_per_cta():
    # more (tile, kv head) work items than resident CTAs, long key ranges:
    # every persistent CTA runs several items back to back
    w = W.build_workload(name="long_chunks", seq_lens=[1536 + 4000, 1536 + 3100, 1536 + 2500, 1536, 300],
                         q_lens=[1536, 1536, 1536, 1536, 1], num_q_heads=32, num_kv_heads=8, head_dim=128,
                         dtype="bf16", seed=31, device=DEV, poison=True)
    seqs = np.arange(w.batch)
    snap = snapshot(w, seqs)
    _, out = gpu_step(w, prefill=True)
    assert pa.device_error() == 0
    assert torch.isfinite(out.float()).all()

    def pick(b, ql):
        if ql == 1:
            return [0]
        return sorted(set([0, 31, 32, 127, 128, ql // 2, ql - 33, ql - 1] +
                          np.random.default_rng(b).choice(ql, 8, replace=False).tolist()))

    rows, ref = oracle_rows(w, seqs, snap, q_rows_per_seq=pick)
    err = max_err(out[torch.from_numpy(rows).to(DEV)], ref)
    assert err <= TOL["bf16"], err


def test_call_completes_in_stream_order():
    """The prefill kernel and the decode kernel run side by side inside one
    call; work queued after the call on the same stream, with no device
    synchronisation, must see every row of both."""
    w = W.make("mixed", device=DEV, n_prefill=3, chunk=1536, n_decode=64, prefix_hi=3000)
    bt = torch.from_numpy(w.block_tables).to(DEV)
    sl = torch.from_numpy(w.seq_lens).to(DEV)
    cu = torch.from_numpy(w.cu_q_lens).to(DEV)
    seqs = np.arange(w.batch)
    snap = snapshot(w, seqs)
    slots = pa.slot_mapping(bt, sl, cu, w.num_tokens, w.num_blocks)
    pa.paged_kv_write(w.key, w.value, w.k_cache, w.v_cache, slots)
    out = torch.full_like(w.q, float("nan"))
    pa.paged_attention_prefill(w.q, w.k_cache, w.v_cache, bt, sl, cu, w.scale, w.max_q_len, w.max_seq_len, out=out)
    copy = out.clone()          # same stream, queued right behind the call
    torch.cuda.synchronize()
    assert pa.device_error() == 0
    assert torch.equal(copy.view(torch.int16), out.view(torch.int16))

    def pick(b, ql):
        return [0] if ql == 1 else [0, 1, ql // 2, ql - 1]

    rows, ref = oracle_rows(w, seqs, snap, q_rows_per_seq=pick)
    assert max_err(copy[torch.from_numpy(rows).to(DEV)], ref) <= TOL["bf16"]
