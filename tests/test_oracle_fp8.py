"""Pins for the oracle's FP8 (E4M3) KV-cache functions.

The pages name the quantised cache ("vLLM-Ascend 原理", section 4 "量化": k and
v quantised to FP8/INT8 as they are written, dequantised after the block-table
read); they fix no format details, so the oracle follows the OCP E4M3 ("FN")
format, round to nearest even with saturation at +-448, and one fp32 scale per
cache.  Pinned against torch's float8_e4m3fn conversions (a library routine
the oracle does not call), closed forms, and SDPA on the dequantised values.
"""
import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
from paged_kv_attention_decode_gb300 import workloads as W
from tests._util import bits

F8 = torch.float8_e4m3fn


def test_decode_every_code_matches_torch():
    codes = np.arange(256, dtype=np.uint8)
    got = oracle.decode_e4m3(codes)
    ref = torch.from_numpy(codes).view(F8).to(torch.float64).numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan) and nan.sum() == 2
    assert np.array_equal(got[~nan], ref[~nan])
    assert got[0x7e] == 448.0 and got[0x01] == 2.0 ** -9


def test_encode_matches_torch_rounding_including_ties():
    finite = np.arange(0, 0x7f, dtype=np.uint8)
    vals = oracle.decode_e4m3(finite)
    mids = (vals[:-1] + vals[1:]) / 2                     # exact ties
    rng = np.random.default_rng(0)
    x = np.concatenate([vals, mids, mids + 1e-7, mids - 1e-7, rng.normal(0, 40, 20000),
                        rng.uniform(-448, 448, 20000), rng.normal(0, 0.01, 5000)]).astype(np.float32)
    x = np.concatenate([x, -x])
    x = x[np.abs(x) < 448]
    got = oracle.encode_e4m3(x)
    ref = torch.from_numpy(x).to(F8).view(torch.uint8).numpy()
    assert np.array_equal(got, ref)


def test_encode_saturates_and_keeps_nan():
    x = np.array([448.0, 449.0, 1e6, np.inf, -448.0, -5000.0, -np.inf, np.nan], dtype=np.float32)
    got = oracle.encode_e4m3(x)
    assert list(got[:4]) == [0x7e] * 4 and list(got[4:7]) == [0xfe] * 3 and got[7] == 0x7f


@pytest.mark.parametrize("src", ["f16", "bf16"])
def test_fp8_write_matches_torch_quantisation(src):
    rng = np.random.default_rng(3)
    NB, bs, H, D, T = 6, 16, 2, 128, 30
    g = torch.Generator().manual_seed(4)
    key = (torch.randn(T, H, D, generator=g) * 3).to(W.torch_dtype(src))
    val = (torch.randn(T, H, D, generator=g) * 200).to(W.torch_dtype(src))
    kc = rng.integers(0, 256, size=(NB, H, bs, D), dtype=np.uint8)   # head-major E4M3 pools
    vc = kc.copy()
    slots = rng.permutation(NB * bs)[:T].astype(np.int64)
    slots[::5] = -1
    k_scale, v_scale = 1 / 16, 0.37
    kref, vref = kc.copy(), vc.copy()
    keep = slots >= 0

    def quant(x, scale):
        inv = np.float32(1) / np.float32(scale)
        y = (x.to(torch.float32) * torch.tensor(inv)).clamp(-448, 448)
        return y.to(F8).view(torch.uint8).numpy()

    # slot s, head h lives at [s // bs, h, s % bs]: index the pools block by block
    blk, off = slots[keep] // bs, slots[keep] % bs
    kref.transpose(0, 2, 1, 3)[blk, off] = quant(key, k_scale)[keep]
    vref.transpose(0, 2, 1, 3)[blk, off] = quant(val, v_scale)[keep]
    oracle.kv_write_fp8(bits(key), bits(val), kc, vc, slots, src, k_scale, v_scale)
    assert np.array_equal(kc, kref) and np.array_equal(vc, vref)


def test_fp8_decode_equals_sdpa_on_dequantised_values():
    Hq, Hkv, D = 8, 2, 128
    lens = np.array([1, 17, 100, 300], dtype=np.int32)
    w = W.build_workload(name="f8", seq_lens=lens, q_lens=1, num_q_heads=Hq, num_kv_heads=Hkv, head_dim=D,
                         dtype="bf16", seed=9, pool_slack=0.5, materialize=False)
    g = torch.Generator().manual_seed(10)
    q = torch.randn(len(lens), Hq, D, generator=g).to(torch.bfloat16)
    Kc = [(torch.randn(int(n), Hkv, D, generator=g) * 8).to(F8) for n in lens]
    Vc = [(torch.randn(int(n), Hkv, D, generator=g) * 8).to(F8) for n in lens]
    kpool = np.zeros((w.num_blocks, Hkv, 16, D), np.uint8)     # head-major E4M3 pools
    vpool = np.zeros_like(kpool)
    slots = oracle.slot_mapping(w.block_tables, lens, lens, 16, w.num_blocks)
    kpool.transpose(0, 2, 1, 3)[slots // 16, slots % 16] = torch.cat(Kc).view(torch.uint8).numpy()
    vpool.transpose(0, 2, 1, 3)[slots // 16, slots % 16] = torch.cat(Vc).view(torch.uint8).numpy()
    k_scale, v_scale, scale = 1 / 8, 1 / 4, 1 / math.sqrt(D)
    out = oracle.paged_attention_decode_fp8(bits(q), kpool, vpool, w.block_tables, lens, scale, "bf16",
                                            k_scale, v_scale)
    for b in range(len(lens)):
        k = (Kc[b].to(torch.float64) * k_scale).transpose(0, 1).repeat_interleave(Hq // Hkv, 0)
        v = (Vc[b].to(torch.float64) * v_scale).transpose(0, 1).repeat_interleave(Hq // Hkv, 0)
        ref = F.scaled_dot_product_attention(q[b].to(torch.float64)[:, None][None], k[None], v[None],
                                             scale=scale)[0, :, 0]
        np.testing.assert_allclose(out[b], ref.numpy(), rtol=1e-11, atol=1e-12)


def test_fp8_decode_against_pure_python_brute_force():
    """A third implementation on a tiny case: E4M3 codes decoded from their
    bit fields (sign, 4-bit exponent with bias 7, 3-bit mantissa, subnormals
    below exponent 1; no infinities), the head-major pool walked token by
    token, and the softmax with math.exp."""
    def e4m3(code):
        sgn = -1.0 if code & 0x80 else 1.0
        e, m = (code >> 3) & 0xF, code & 0x7
        if e == 0xF and m == 0x7:
            return math.nan
        return sgn * (m / 8.0) * 2.0 ** -6 if e == 0 else sgn * (1.0 + m / 8.0) * 2.0 ** (e - 7)

    Hq, Hkv, D = 4, 2, 128
    lens = np.array([1, 19, 40], dtype=np.int32)
    w = W.build_workload(name="f8bf", seq_lens=lens, q_lens=1, num_q_heads=Hq, num_kv_heads=Hkv, head_dim=D,
                         dtype="f16", seed=21, pool_slack=0.5, materialize=False)
    rng = np.random.default_rng(22)
    kpool = rng.integers(0, 256, size=(w.num_blocks, Hkv, 16, D), dtype=np.uint8)
    kpool[(kpool & 0x7F) == 0x7F] = 0x3C          # no NaN codes
    vpool = rng.integers(0, 256, size=(w.num_blocks, Hkv, 16, D), dtype=np.uint8)
    vpool[(vpool & 0x7F) == 0x7F] = 0x2A
    q = (torch.randn(len(lens), Hq, D, generator=torch.Generator().manual_seed(23)) * 0.1).to(torch.float16)
    k_scale, v_scale, scale = 1 / 64, 1 / 32, 1 / math.sqrt(D)
    out = oracle.paged_attention_decode_fp8(bits(q), kpool, vpool, w.block_tables, lens, scale, "f16",
                                            k_scale, v_scale)
    qf = q.to(torch.float64).tolist()
    for b, n in enumerate(lens):
        for h in range(Hq):
            g = h // (Hq // Hkv)
            rows = [(int(w.block_tables[b][t // 16]), t % 16) for t in range(n)]
            s = [scale * sum(qf[b][h][d] * e4m3(int(kpool[blk, g, off, d])) * k_scale for d in range(D))
                 for blk, off in rows]
            mx = max(s)
            e = [math.exp(x - mx) for x in s]
            tot = sum(e)
            for d in range(0, D, 7):
                ref = sum(e[t] * e4m3(int(vpool[blk, g, off, d])) * v_scale for t, (blk, off) in enumerate(rows)) / tot
                assert out[b, h, d] == pytest.approx(ref, rel=1e-11, abs=1e-12)


# --- FP8 prefill (varlen causal rows over the E4M3 cache) --------------------

def _e4m3_bits(code):
    """E4M3 (FN) from its bit fields: sign, 4-bit exponent (bias 7), 3-bit
    mantissa, subnormals at exponent 0, NaN at S.1111.111, no infinities."""
    sgn = -1.0 if code & 0x80 else 1.0
    e, m = (code >> 3) & 0xF, code & 0x7
    if e == 0xF and m == 0x7:
        return math.nan
    return sgn * (m / 8.0) * 2.0 ** -6 if e == 0 else sgn * (1.0 + m / 8.0) * 2.0 ** (e - 7)


def _fp8_case(lens, qlens, Hq, Hkv, D, dtype, seed):
    lens = np.asarray(lens, dtype=np.int32)
    qlens = np.asarray(qlens, dtype=np.int32)
    w = W.build_workload(name="f8p", seq_lens=lens, q_lens=qlens, num_q_heads=Hq, num_kv_heads=Hkv, head_dim=D,
                         dtype=dtype, seed=seed, pool_slack=0.5, materialize=False)
    g = torch.Generator().manual_seed(seed + 1)
    q = torch.randn(int(qlens.sum()), Hq, D, generator=g).to(W.torch_dtype(dtype))
    Kc = [(torch.randn(int(n), Hkv, D, generator=g) * 8).to(F8) for n in lens]
    Vc = [(torch.randn(int(n), Hkv, D, generator=g) * 8).to(F8) for n in lens]
    # every position of each sequence (its whole context), NaN codes elsewhere
    kpool = np.full((w.num_blocks, Hkv, 16, D), 0x7F, np.uint8)
    vpool = kpool.copy()
    slots = oracle.slot_mapping(w.block_tables, lens, lens, 16, w.num_blocks)
    kpool.transpose(0, 2, 1, 3)[slots // 16, slots % 16] = torch.cat(Kc).view(torch.uint8).numpy()
    vpool.transpose(0, 2, 1, 3)[slots // 16, slots % 16] = torch.cat(Vc).view(torch.uint8).numpy()
    return w, lens, qlens, q, Kc, Vc, kpool, vpool, slots


def test_fp8_prefill_equals_causal_sdpa_on_dequantised_values():
    Hq, Hkv, D = 8, 2, 128
    w, lens, qlens, q, Kc, Vc, kpool, vpool, _ = _fp8_case([40, 130, 17, 300], [40, 33, 1, 4], Hq, Hkv, D,
                                                           "bf16", 31)
    k_scale, v_scale, scale = 1 / 8, 1 / 4, 1 / math.sqrt(D)
    out = oracle.paged_attention_prefill_fp8(bits(q), kpool, vpool, w.block_tables, lens, qlens, scale, "bf16",
                                             k_scale, v_scale)
    row = 0
    for b, (n, c) in enumerate(zip(lens.tolist(), qlens.tolist())):
        k = (Kc[b].to(torch.float64) * k_scale).transpose(0, 1).repeat_interleave(Hq // Hkv, 0)
        v = (Vc[b].to(torch.float64) * v_scale).transpose(0, 1).repeat_interleave(Hq // Hkv, 0)
        qb = q[row:row + c].to(torch.float64).transpose(0, 1)           # [Hq, c, D]
        mask = torch.arange(n)[None, :] <= (n - c + torch.arange(c))[:, None]   # bottom-right causal
        ref = F.scaled_dot_product_attention(qb[None], k[None], v[None], attn_mask=mask, scale=scale)[0]
        np.testing.assert_allclose(out[row:row + c], ref.transpose(0, 1).numpy(), rtol=1e-11, atol=1e-12)
        row += c


def test_fp8_prefill_is_the_16_bit_prefill_on_the_dequantised_values():
    # power-of-two scales and E4M3 values are exact in fp16, so the 16-bit
    # oracle reading an fp16 cache of code * scale computes the same doubles
    Hq, Hkv, D = 4, 4, 64
    w, lens, qlens, q, Kc, Vc, kpool, vpool, slots = _fp8_case([50, 90], [20, 9], Hq, Hkv, D, "f16", 41)
    k_scale, v_scale, scale = 1 / 16, 2.0, 0.125
    out8 = oracle.paged_attention_prefill_fp8(bits(q), kpool, vpool, w.block_tables, lens, qlens, scale, "f16",
                                              k_scale, v_scale)
    k16 = np.zeros((w.num_blocks, 16, Hkv, D), np.uint16)
    v16 = np.zeros_like(k16)
    k16.reshape(-1, Hkv, D)[slots] = bits((torch.cat(Kc).to(torch.float32) * k_scale).to(torch.float16))
    v16.reshape(-1, Hkv, D)[slots] = bits((torch.cat(Vc).to(torch.float32) * v_scale).to(torch.float16))
    out16 = oracle.paged_attention_prefill(bits(q), k16, v16, w.block_tables, lens, qlens, scale, "f16")
    assert np.array_equal(out8, out16)


def test_fp8_prefill_last_rows_are_the_decode_rows_and_causality_holds():
    Hq, Hkv, D = 8, 4, 128
    w, lens, qlens, q, Kc, Vc, kpool, vpool, slots = _fp8_case([64, 100, 7], [30, 8, 7], Hq, Hkv, D, "f16", 51)
    k_scale, v_scale, scale = 1 / 32, 1 / 8, 1 / math.sqrt(D)
    out = oracle.paged_attention_prefill_fp8(bits(q), kpool, vpool, w.block_tables, lens, qlens, scale, "f16",
                                             k_scale, v_scale)
    last = np.cumsum(qlens) - 1
    dec = oracle.paged_attention_decode_fp8(bits(q)[last], kpool, vpool, w.block_tables, lens, scale, "f16",
                                            k_scale, v_scale)
    assert np.array_equal(out[last], dec)
    # perturb the codes at and after position 70 of sequence 1 (its rows sit at
    # positions 92..99): rows of sequences 0 and 2 keep their bits, all of
    # sequence 1's rows change
    k2, v2 = kpool.copy(), vpool.copy()
    n1 = int(lens[1])
    s1 = slots[int(lens[0]):int(lens[0]) + n1]
    for t in range(70, n1):
        k2[s1[t] // 16, :, s1[t] % 16] ^= 0x01
        v2[s1[t] // 16, :, s1[t] % 16] ^= 0x08
    out2 = oracle.paged_attention_prefill_fp8(bits(q), k2, v2, w.block_tables, lens, qlens, scale, "f16",
                                              k_scale, v_scale)
    r0, r1 = int(qlens[0]), int(qlens[0] + qlens[1])
    assert np.array_equal(out2[:r0], out[:r0]) and np.array_equal(out2[r1:], out[r1:])
    assert np.all(np.any(out2[r0:r1] != out[r0:r1], axis=(1, 2)))


def test_fp8_prefill_against_pure_python_brute_force():
    Hq, Hkv, D = 2, 1, 128
    lens, qlens = np.array([21, 5], np.int32), np.array([4, 5], np.int32)
    w = W.build_workload(name="f8pb", seq_lens=lens, q_lens=qlens, num_q_heads=Hq, num_kv_heads=Hkv, head_dim=D,
                         dtype="bf16", seed=61, pool_slack=0.5, materialize=False)
    rng = np.random.default_rng(62)
    kpool = rng.integers(0, 256, size=(w.num_blocks, Hkv, 16, D), dtype=np.uint8)
    kpool[(kpool & 0x7F) == 0x7F] = 0x33
    vpool = rng.integers(0, 256, size=(w.num_blocks, Hkv, 16, D), dtype=np.uint8)
    vpool[(vpool & 0x7F) == 0x7F] = 0x21
    q = (torch.randn(int(qlens.sum()), Hq, D, generator=torch.Generator().manual_seed(63)) * 0.05).to(torch.bfloat16)
    k_scale, v_scale, scale = 1 / 64, 1 / 16, 1 / math.sqrt(D)
    out = oracle.paged_attention_prefill_fp8(bits(q), kpool, vpool, w.block_tables, lens, qlens, scale, "bf16",
                                             k_scale, v_scale)
    qf = q.to(torch.float64).tolist()
    row = 0
    for b, (n, c) in enumerate(zip(lens.tolist(), qlens.tolist())):
        for i in range(c):
            pos = n - c + i
            for h in range(Hq):
                cells = [(int(w.block_tables[b][t // 16]), t % 16) for t in range(pos + 1)]
                s = [scale * sum(qf[row][h][d] * _e4m3_bits(int(kpool[blk, 0, off, d])) * k_scale for d in range(D))
                     for blk, off in cells]
                mx = max(s)
                e = [math.exp(x - mx) for x in s]
                for d in range(0, D, 11):
                    ref = sum(e[t] * _e4m3_bits(int(vpool[blk, 0, off, d])) * v_scale
                              for t, (blk, off) in enumerate(cells)) / sum(e)
                    assert out[row, h, d] == pytest.approx(ref, rel=1e-11, abs=1e-12)
            row += 1
