"""Pins for the CPU oracle: each test ties it to something other than itself.

The pages print no numeric example for paged attention, so the oracle is
pinned by library routines it does not call (numpy float16 and torch bfloat16
decoding, numpy fancy-index assignment, torch scaled_dot_product_attention),
by closed forms (contiguous tables, one-token context, uniform scores, one
dominant key), by invariants the pages fix (physical placement is invisible,
shared prefix blocks equal private copies, causality) and by a pure-Python
brute force on the tiny workload.
"""
import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
from paged_kv_attention_decode_gb300 import workloads as W
from tests._util import bits, from_bits

TD = {"f16": torch.float16, "bf16": torch.bfloat16}


# --------------------------------------------------------------------------
# storage decoding
# --------------------------------------------------------------------------

def test_decode_f16_every_pattern_matches_numpy():
    pat = np.arange(65536, dtype=np.uint16)
    got = oracle.decode_values(pat, "f16")
    ref = pat.view(np.float16).astype(np.float64)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])
    # signed zeros survive
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(ref[~nan]))


def test_decode_bf16_every_pattern_matches_torch():
    pat = np.arange(65536, dtype=np.uint16)
    got = oracle.decode_values(pat, "bf16")
    ref = from_bits(pat, torch.bfloat16).to(torch.float64).numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(ref[~nan]))


# --------------------------------------------------------------------------
# slot address translation and the cache write
# --------------------------------------------------------------------------

def test_slot_mapping_contiguous_tables_closed_form():
    # With table[b][j] = b * maxb + j the pool is a plain contiguous
    # [B, maxb * bs] cache, so the slot of position p of sequence b is
    # b * maxb * bs + p.
    rng = np.random.default_rng(1)
    bs, B = 16, 7
    lens = rng.integers(1, 200, size=B).astype(np.int32)
    qlens = np.minimum(lens, rng.integers(1, 40, size=B)).astype(np.int32)
    maxb = int(-(-lens.max() // bs))
    tables = (np.arange(B)[:, None] * maxb + np.arange(maxb)[None, :]).astype(np.int32)
    got = oracle.slot_mapping(tables, lens, qlens, bs, B * maxb)
    want = np.concatenate([b * maxb * bs + np.arange(lens[b] - qlens[b], lens[b]) for b in range(B)])
    assert np.array_equal(got, want)


def test_slot_mapping_follows_block_permutation():
    w = W.make("tiny")
    lens, ql = w.seq_lens, np.minimum(w.seq_lens, 5).astype(np.int32)
    base = oracle.slot_mapping(w.block_tables, lens, ql, 16, w.num_blocks)
    pi = np.random.default_rng(3).permutation(w.num_blocks).astype(np.int32)
    moved = oracle.slot_mapping(pi[w.block_tables], lens, ql, 16, w.num_blocks)
    assert np.array_equal(moved, pi[base // 16].astype(np.int64) * 16 + base % 16)
    assert np.unique(base).size == base.size


def test_slot_mapping_rejects_out_of_range_table():
    tables = np.array([[0, 99]], dtype=np.int32)
    with pytest.raises(ValueError):
        oracle.slot_mapping(tables, np.array([20], np.int32), np.array([20], np.int32), 16, 4)


def test_kv_write_matches_numpy_fancy_index_assignment():
    rng = np.random.default_rng(5)
    NB, bs, H, D, T = 9, 16, 3, 8, 40
    kc = rng.integers(0, 65536, size=(NB, bs, H, D), dtype=np.uint16)
    vc = rng.integers(0, 65536, size=(NB, bs, H, D), dtype=np.uint16)
    key = rng.integers(0, 65536, size=(T, H, D), dtype=np.uint16)
    val = rng.integers(0, 65536, size=(T, H, D), dtype=np.uint16)
    slots = rng.permutation(NB * bs)[:T].astype(np.int64)
    slots[::7] = -1                                  # padding tokens: no write
    k_ref, v_ref = kc.copy(), vc.copy()
    keep = slots >= 0
    k_ref.reshape(NB * bs, H, D)[slots[keep]] = key[keep]
    v_ref.reshape(NB * bs, H, D)[slots[keep]] = val[keep]
    oracle.kv_write(key, val, kc, vc, slots)
    assert np.array_equal(kc, k_ref) and np.array_equal(vc, v_ref)


def test_kv_write_rejects_slot_past_pool():
    kc = np.zeros((2, 16, 1, 8), np.uint16)
    with pytest.raises(ValueError):
        oracle.kv_write(np.zeros((1, 1, 8), np.uint16), np.zeros((1, 1, 8), np.uint16), kc,
                        kc.copy(), np.array([32], np.int64))


# --------------------------------------------------------------------------
# paged attention == contiguous attention
# --------------------------------------------------------------------------

def _scatter_contiguous(lens, Hq, Hkv, D, dtype, seed, q_lens=None):
    """Random contiguous per-sequence K/V, written into a scattered pool through
    the oracle's own slot mapping and write (every token treated as new)."""
    w = W.build_workload(name="pin", seq_lens=lens, q_lens=1, num_q_heads=Hq, num_kv_heads=Hkv,
                         head_dim=D, dtype=dtype, seed=seed, pool_slack=0.5, poison=True)
    g = torch.Generator().manual_seed(seed + 1)
    Ks = [torch.randn(int(n), Hkv, D, generator=g).to(TD[dtype]) for n in lens]
    Vs = [torch.randn(int(n), Hkv, D, generator=g).to(TD[dtype]) for n in lens]
    slots = oracle.slot_mapping(w.block_tables, w.seq_lens, w.seq_lens, 16, w.num_blocks)
    kc, vc = bits(w.k_cache), bits(w.v_cache)
    oracle.kv_write(bits(torch.cat(Ks)), bits(torch.cat(Vs)), kc, vc, slots)
    return w, Ks, Vs, kc, vc


def _sdpa(q, k, v, scale, mask=None):
    """q [Hq, L, D], k/v [Hkv, N, D] in float64 through torch's SDPA (GQA by
    repeating each kv head for its contiguous group of q heads)."""
    G = q.shape[0] // k.shape[0]
    k = k.repeat_interleave(G, dim=0)
    v = v.repeat_interleave(G, dim=0)
    return F.scaled_dot_product_attention(q[None], k[None], v[None], attn_mask=mask, scale=scale)[0]


@pytest.mark.parametrize("Hq,Hkv,D,dtype", [(4, 4, 64, "f16"), (8, 2, 128, "bf16"), (6, 1, 32, "f16")])
def test_decode_equals_sdpa_on_contiguous_kv(Hq, Hkv, D, dtype):
    lens = np.array([1, 16, 17, 31, 64, 100, 257], dtype=np.int32)
    w, Ks, Vs, kc, vc = _scatter_contiguous(lens, Hq, Hkv, D, dtype, seed=11)
    scale = 1.0 / math.sqrt(D)
    out = oracle.paged_attention_decode(bits(w.q), kc, vc, w.block_tables, w.seq_lens, scale, dtype)
    for b, n in enumerate(lens):
        q = w.q[b].to(torch.float64)[:, None, :]                      # [Hq, 1, D]
        ref = _sdpa(q, Ks[b].to(torch.float64).transpose(0, 1), Vs[b].to(torch.float64).transpose(0, 1),
                    scale)[:, 0, :].numpy()
        np.testing.assert_allclose(out[b], ref, rtol=1e-11, atol=1e-12)


def test_prefill_equals_sdpa_with_causal_mask():
    Hq, Hkv, D, dtype = 8, 2, 64, "bf16"
    lens = np.array([5, 40, 77, 130], dtype=np.int32)
    qls = np.array([5, 17, 1, 33], dtype=np.int32)
    w, Ks, Vs, kc, vc = _scatter_contiguous(lens, Hq, Hkv, D, dtype, seed=12)
    g = torch.Generator().manual_seed(99)
    q = torch.randn(int(qls.sum()), Hq, D, generator=g).to(torch.bfloat16)
    scale = 0.11
    out = oracle.paged_attention_prefill(bits(q), kc, vc, w.block_tables, lens, qls, scale, dtype)
    r0 = 0
    for b, (n, ql) in enumerate(zip(lens, qls)):
        qb = q[r0:r0 + ql].to(torch.float64).transpose(0, 1)          # [Hq, ql, D]
        k = Ks[b].to(torch.float64).transpose(0, 1)
        v = Vs[b].to(torch.float64).transpose(0, 1)
        if ql == n:
            G = Hq // Hkv
            ref = F.scaled_dot_product_attention(qb[None], k.repeat_interleave(G, 0)[None],
                                                 v.repeat_interleave(G, 0)[None], is_causal=True,
                                                 scale=scale)[0]
        else:
            # query i sits at position n - ql + i and sees positions 0..n - ql + i
            mask = torch.from_numpy(np.arange(n)[None, :] <= (n - ql + np.arange(ql))[:, None])
            ref = _sdpa(qb, k, v, scale, mask)
        np.testing.assert_allclose(out[r0:r0 + ql], ref.transpose(0, 1).numpy(), rtol=1e-11, atol=1e-12)
        r0 += ql


# --------------------------------------------------------------------------
# closed forms and special cases
# --------------------------------------------------------------------------

def test_seq_len_one_returns_v_exactly():
    w = W.make("tiny")
    kc, vc = bits(w.k_cache), bits(w.v_cache)
    out = oracle.paged_attention_decode(bits(w.q), kc, vc, w.block_tables, w.seq_lens, w.scale, "f16")
    assert w.seq_lens[0] == 1
    v0 = oracle.decode_values(vc[w.block_tables[0, 0], 0], "f16")     # [H, D]
    assert np.array_equal(out[0], v0)


def test_zero_query_gives_mean_of_values():
    w = W.make("tiny")
    q = np.zeros_like(bits(w.q))
    kc, vc = bits(w.k_cache), bits(w.v_cache)
    out = oracle.paged_attention_decode(q, kc, vc, w.block_tables, w.seq_lens, w.scale, "f16")
    b = 3
    n = int(w.seq_lens[b])
    for h in range(4):
        for d in range(0, 64, 7):
            vals = [oracle.decode_values(vc[w.block_tables[b, t // 16], t % 16, h, d:d + 1], "f16")[0]
                    for t in range(n)]
            assert out[b, h, d] == pytest.approx(math.fsum(vals) / n, rel=1e-14, abs=1e-15)


def test_one_dominant_key_selects_its_value():
    w = W.make("tiny")
    kc, vc = bits(w.k_cache), bits(w.v_cache)
    b, t_star, h = 3, 41, 2
    q = torch.zeros_like(w.q)
    q[b, h, 0] = 1.0
    kcf = w.k_cache.clone()
    kcf[..., 0] = 0.0
    blk, off = w.block_tables[b, t_star // 16], t_star % 16
    kcf[blk, off, h, 0] = 2048.0                       # score 256 above every other key
    out = oracle.paged_attention_decode(bits(q), bits(kcf), vc, w.block_tables, w.seq_lens, w.scale, "f16")
    want = oracle.decode_values(vc[blk, off, h], "f16")
    np.testing.assert_allclose(out[b, h], want, rtol=0, atol=1e-90)


def test_tiny_against_pure_python_brute_force():
    w = W.make("tiny")
    kc, vc = bits(w.k_cache), bits(w.v_cache)
    out = oracle.paged_attention_decode(bits(w.q), kc, vc, w.block_tables, w.seq_lens, w.scale, "f16")
    qf = w.q.to(torch.float64).tolist()
    kf = w.k_cache.to(torch.float64).tolist()
    vf = w.v_cache.to(torch.float64).tolist()
    for b in range(w.batch):
        n = int(w.seq_lens[b])
        keys = [kf[int(w.block_tables[b][t // 16])][t % 16] for t in range(n)]
        vals = [vf[int(w.block_tables[b][t // 16])][t % 16] for t in range(n)]
        for h in range(4):
            s = [w.scale * sum(a * c for a, c in zip(qf[b][h], keys[t][h])) for t in range(n)]
            mx = max(s)
            e = [math.exp(x - mx) for x in s]
            tot = sum(e)
            for d in range(64):
                ref = sum(e[t] * vals[t][h][d] for t in range(n)) / tot
                assert out[b, h, d] == pytest.approx(ref, rel=1e-12, abs=1e-13)


# --------------------------------------------------------------------------
# invariants
# --------------------------------------------------------------------------

def test_physical_block_permutation_is_invisible():
    w = W.make("gqa_prefix", batch=32)
    kc, vc = bits(w.k_cache), bits(w.v_cache)
    base = oracle.paged_attention_decode(bits(w.q), kc, vc, w.block_tables, w.seq_lens, w.scale, "bf16")
    pi = np.random.default_rng(7).permutation(w.num_blocks)
    kc2, vc2 = np.empty_like(kc), np.empty_like(vc)
    kc2[pi] = kc                                       # block x moves to pi[x]
    vc2[pi] = vc
    tables2 = pi[w.block_tables].astype(np.int32)
    moved = oracle.paged_attention_decode(bits(w.q), kc2, vc2, tables2, w.seq_lens, w.scale, "bf16")
    assert np.array_equal(base, moved)


def test_shared_prefix_blocks_equal_private_copies():
    w = W.make("gqa_prefix", batch=32)
    assert (w.meta["shared_blocks"] > 0).sum() > 8
    kc, vc = bits(w.k_cache), bits(w.v_cache)
    base = oracle.paged_attention_decode(bits(w.q), kc, vc, w.block_tables, w.seq_lens, w.scale, "bf16")
    # give every sequence private copies of its shared blocks
    tables = w.block_tables.copy()
    extra_k, extra_v = [], []
    nxt = w.num_blocks
    for b in range(w.batch):
        for j in range(int(w.meta["shared_blocks"][b])):
            src = tables[b, j]
            extra_k.append(kc[src])
            extra_v.append(vc[src])
            tables[b, j] = nxt
            nxt += 1
    kc2 = np.concatenate([kc, np.stack(extra_k)])
    vc2 = np.concatenate([vc, np.stack(extra_v)])
    priv = oracle.paged_attention_decode(bits(w.q), kc2, vc2, tables, w.seq_lens, w.scale, "bf16")
    assert np.array_equal(base, priv)


def test_prefill_is_causal_and_last_row_is_decode():
    Hq, Hkv, D = 4, 2, 32
    lens = np.array([50, 90], dtype=np.int32)
    qls = np.array([20, 35], dtype=np.int32)
    w = W.build_workload(name="c", seq_lens=lens, q_lens=qls, num_q_heads=Hq, num_kv_heads=Hkv,
                         head_dim=D, dtype="f16", seed=3)
    kc, vc = bits(w.k_cache), bits(w.v_cache)
    q = bits(w.q)
    base = oracle.paged_attention_prefill(q, kc, vc, w.block_tables, lens, qls, 0.2, "f16")
    # perturb every position after the first query of sequence 1 (position 55)
    kc2, vc2 = kc.copy(), vc.copy()
    for t in range(56, 90):
        blk, off = w.block_tables[1, t // 16], t % 16
        kc2[blk, off] ^= 0x1234
        vc2[blk, off] ^= 0x0321
    pert = oracle.paged_attention_prefill(q, kc2, vc2, w.block_tables, lens, qls, 0.2, "f16")
    r1 = 20                                            # first row of sequence 1
    assert np.array_equal(base[:r1 + 1], pert[:r1 + 1])   # sequence 0 + the row at position 55
    assert not np.array_equal(base[r1 + 1:], pert[r1 + 1:])
    # the last row of each sequence is the decode query at seq_len - 1
    last = np.cumsum(qls) - 1
    dec = oracle.paged_attention_decode(q[last], kc, vc, w.block_tables, lens, 0.2, "f16")
    assert np.array_equal(dec, base[last])


def test_decode_empty_sequence_gives_zeros():
    w = W.make("tiny")
    lens = w.seq_lens.copy()
    lens[2] = 0
    out = oracle.paged_attention_decode(bits(w.q), bits(w.k_cache), bits(w.v_cache), w.block_tables,
                                        lens, w.scale, "f16")
    assert np.array_equal(out[2], np.zeros((4, 64)))
    assert np.all(np.isfinite(out))


def test_selected_rows_match_full_run():
    w = W.make("gqa_prefix", batch=24)
    kc, vc = bits(w.k_cache), bits(w.v_cache)
    full = oracle.paged_attention_decode(bits(w.q), kc, vc, w.block_tables, w.seq_lens, w.scale, "bf16")
    sel = np.array([3, 0, 17, 17, 23])
    part = oracle.paged_attention_decode(bits(w.q), kc, vc, w.block_tables, w.seq_lens, w.scale, "bf16",
                                         select=sel, threads=3)
    assert np.array_equal(part, full[sel])
