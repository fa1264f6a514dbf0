"""GPU parity of the FP8 (E4M3) KV cache path: the quantising write is
bit-exact against the oracle; decode attention over the FP8 pools is within
the tolerance of the query dtype against the fp64 oracle on the same codes."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_attention_decode_gb300 as pa
from paged_kv_attention_decode_gb300 import workloads as W
from tests._gpu_util import TOL, bits

pytestmark = pytest.mark.gpu
DEV = "cuda"
LENS = [1, 2, 15, 16, 17, 31, 33, 100, 511, 512, 513, 1000, 2049]


def u8(t):
    return t.detach().contiguous().cpu().numpy().view(np.uint8)


@pytest.mark.parametrize("src", ["f16", "bf16"])
def test_fp8_write_is_bit_exact(src):
    NB, H, D, T = 300, 8, 128, 2000
    g = torch.Generator(device=DEV).manual_seed(5)
    key = (torch.randn(T, H, D, device=DEV, generator=g) * 5).to(W.torch_dtype(src))
    val = (torch.randn(T, H, D, device=DEV, generator=g) * 700).to(W.torch_dtype(src))  # saturates
    key[0, 0, :4] = float("nan")
    kc = torch.randint(0, 256, (NB, H, 16, D), device=DEV, dtype=torch.uint8, generator=g)   # head-major
    vc = kc.clone()
    rng = np.random.default_rng(6)
    slots = rng.permutation(NB * 16)[:T].astype(np.int64)
    slots[rng.random(T) < 0.1] = -1
    k_ref, v_ref = u8(kc), u8(vc)
    oracle.kv_write_fp8(bits(key), bits(val), k_ref, v_ref, slots, src, 0.3, 1.7)
    pa.paged_kv_write_fp8(key, val, kc, vc, torch.from_numpy(slots).to(DEV), 0.3, 1.7)
    torch.cuda.synchronize()
    assert np.array_equal(u8(kc), k_ref) and np.array_equal(u8(vc), v_ref)


@pytest.mark.parametrize("Hq,Hkv,dtype", [(8, 8, "f16"), (8, 8, "bf16"), (5, 5, "bf16"), (16, 4, "bf16"), (16, 2, "f16"),
                                          (12, 4, "bf16"), (32, 2, "bf16"), (32, 1, "f16")])
@pytest.mark.parametrize("partition", [0, 48])
def test_fp8_decode_step_parity(Hq, Hkv, dtype, partition):
    w = W.build_workload(name="f8", seq_lens=LENS, q_lens=1, num_q_heads=Hq, num_kv_heads=Hkv, head_dim=128,
                         dtype=dtype, seed=Hq * 7 + Hkv, device=DEV, poison=True, pool_slack=0.3,
                         cache_dtype="fp8")
    sc = w.meta["kv_scale"]
    bt = torch.from_numpy(w.block_tables).to(DEV)
    sl = torch.from_numpy(w.seq_lens).to(DEV)
    k_ref, v_ref = u8(w.k_cache), u8(w.v_cache)
    slots = pa.slot_mapping(bt, sl, None, w.batch, w.num_blocks)
    pa.paged_kv_write_fp8(w.key, w.value, w.k_cache, w.v_cache, slots, sc, sc)
    out = pa.paged_attention_decode_fp8(w.q, w.k_cache, w.v_cache, bt, sl, w.scale, sc, sc, w.max_seq_len,
                                        partition_size=partition)
    torch.cuda.synchronize()
    ref_slots = oracle.slot_mapping(w.block_tables, w.seq_lens, w.q_lens, 16, w.num_blocks)
    oracle.kv_write_fp8(bits(w.key), bits(w.value), k_ref, v_ref, ref_slots, dtype, sc, sc)
    assert np.array_equal(u8(w.k_cache), k_ref) and np.array_equal(u8(w.v_cache), v_ref)
    ref = oracle.paged_attention_decode_fp8(bits(w.q), k_ref, v_ref, w.block_tables, w.seq_lens, w.scale,
                                            dtype, sc, sc)
    got = out.double().cpu().numpy()
    assert np.all(np.isfinite(got))
    err = float(np.max(np.abs(got - ref)))
    assert err <= TOL[dtype], err
    assert pa.device_error() == 0


@pytest.mark.slow
def test_fp8_full_size_sampled():
    w = W.make("llama7b_decode_fp8", device=DEV)
    sc = w.meta["kv_scale"]
    seqs = np.sort(np.random.default_rng(2).choice(w.batch, 12, replace=False))
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
    slots = pa.slot_mapping(bt, sl, None, w.batch, w.num_blocks)
    pa.paged_kv_write_fp8(w.key, w.value, w.k_cache, w.v_cache, slots, sc, sc)
    out = pa.paged_attention_decode_fp8(w.q, w.k_cache, w.v_cache, bt, sl, w.scale, sc, sc, w.max_seq_len)
    torch.cuda.synchronize()
    rows = torch.from_numpy(seqs).to(DEV)
    s2 = oracle.slot_mapping(tables, w.seq_lens[seqs], np.ones(len(seqs), np.int32), 16, len(used))
    oracle.kv_write_fp8(bits(w.key[rows]), bits(w.value[rows]), k_snap, v_snap, s2, "f16", sc, sc)
    ref = oracle.paged_attention_decode_fp8(bits(w.q[rows]), k_snap, v_snap, tables, w.seq_lens[seqs], w.scale,
                                            "f16", sc, sc)
    err = float(np.max(np.abs(out[rows].double().cpu().numpy() - ref)))
    assert err <= TOL["f16"], err
