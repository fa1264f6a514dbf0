"""GPU parity of the slot address step and the KV write: bit-exact vs the oracle."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_attention_decode_gb300 as pa
from paged_kv_attention_decode_gb300 import workloads as W
from tests._gpu_util import bits

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _tables(w):
    return (torch.from_numpy(w.block_tables).to(DEV), torch.from_numpy(w.seq_lens).to(DEV),
            torch.from_numpy(w.cu_q_lens).to(DEV))


@pytest.mark.parametrize("name,kw", [
    ("tiny", {}),
    ("mixed", dict(n_prefill=3, chunk=37, n_decode=50, prefix_hi=300, dec_lo=1, dec_hi=200)),
    ("gqa_prefix", dict(batch=48)),
])
def test_slot_mapping_and_write_are_bit_exact(name, kw):
    w = W.make(name, device=DEV, poison=True, **kw)
    bt, sl, cu = _tables(w)
    pre_k, pre_v = bits(w.k_cache), bits(w.v_cache)
    decode_form = w.is_decode
    slots = pa.slot_mapping(bt, sl, None if decode_form else cu, w.num_tokens, w.num_blocks)
    pa.paged_kv_write(w.key, w.value, w.k_cache, w.v_cache, slots)
    torch.cuda.synchronize()
    ref = oracle.slot_mapping(w.block_tables, w.seq_lens, w.q_lens, 16, w.num_blocks)
    assert np.array_equal(slots.cpu().numpy(), ref)
    oracle.kv_write(bits(w.key), bits(w.value), pre_k, pre_v, ref)
    assert np.array_equal(bits(w.k_cache), pre_k)
    assert np.array_equal(bits(w.v_cache), pre_v)
    assert pa.device_error() == 0


def test_write_skips_negative_slots_and_handles_many_tokens():
    NB, H, D, T = 700, 8, 128, 9000
    g = torch.Generator(device=DEV).manual_seed(1)
    kc = torch.randn(NB, 16, H, D, device=DEV, generator=g).to(torch.bfloat16)
    vc = torch.randn(NB, 16, H, D, device=DEV, generator=g).to(torch.bfloat16)
    key = torch.randn(T, H, D, device=DEV, generator=g).to(torch.bfloat16)
    val = torch.randn(T, H, D, device=DEV, generator=g).to(torch.bfloat16)
    rng = np.random.default_rng(2)
    slots = rng.permutation(NB * 16)[:T].astype(np.int64)
    slots[rng.random(T) < 0.2] = -1
    k_ref, v_ref = bits(kc), bits(vc)
    oracle.kv_write(bits(key), bits(val), k_ref, v_ref, slots)
    pa.paged_kv_write(key, val, kc, vc, torch.from_numpy(slots).to(DEV))
    torch.cuda.synchronize()
    assert np.array_equal(bits(kc), k_ref) and np.array_equal(bits(vc), v_ref)


def test_slot_past_pool_is_dropped_and_flagged():
    NB, H, D = 4, 2, 64
    kc = torch.zeros(NB, 16, H, D, device=DEV, dtype=torch.float16)
    vc = torch.zeros_like(kc)
    key = torch.ones(2, H, D, device=DEV, dtype=torch.float16)
    slots = torch.tensor([NB * 16 + 3, 5], device=DEV, dtype=torch.int64)
    pa.device_error()
    pa.paged_kv_write(key, key, kc, vc, slots)
    assert pa.device_error() == 2
    assert float(kc.float().sum()) == H * D  # only slot 5 written


def test_out_of_range_table_entry_gives_slot_minus_one_and_flag():
    bt = torch.tensor([[0, 1], [2, 99]], device=DEV, dtype=torch.int32)
    sl = torch.tensor([20, 30], device=DEV, dtype=torch.int32)
    pa.device_error()
    slots = pa.slot_mapping(bt, sl, None, 2, 4)
    assert slots.cpu().tolist() == [1 * 16 + 3, -1]
    assert pa.device_error() == 1


@pytest.mark.parametrize("name,fp8", [("gqa_prefix", False), ("llama7b_decode_fp8", True), ("tiny", False)])
def test_gather_matches_numpy_fancy_index(name, fp8):
    """pa_paged_kv_gather returns, byte for byte, the rows a NumPy fancy-index
    gather of the pool through the block tables returns."""
    kw = {"batch": 24} if name != "tiny" else {}
    w = W.make(name, device=DEV, **kw)
    bt = torch.from_numpy(w.block_tables).to(DEV)
    sl = torch.from_numpy(w.seq_lens).to(DEV)
    k, v = pa.paged_kv_gather(w.k_cache, w.v_cache, bt, sl, w.max_seq_len)
    torch.cuda.synchronize()
    assert pa.device_error() == 0
    rows = []
    for b in range(w.batch):
        t = np.arange(int(w.seq_lens[b]))
        rows.append(w.block_tables[b, t // 16].astype(np.int64) * 16 + t % 16)
    idx = np.concatenate(rows)
    H, D = w.num_kv_heads, w.head_dim
    view = torch.uint8 if fp8 else torch.int16
    kc = w.k_cache.view(view).cpu().numpy()
    vc = w.v_cache.view(view).cpu().numpy()
    if fp8:   # head-major [NB, H, 16, D] -> token-major rows
        kc, vc = kc.transpose(0, 2, 1, 3), vc.transpose(0, 2, 1, 3)
    kc, vc = kc.reshape(-1, H, D), vc.reshape(-1, H, D)
    assert np.array_equal(k.view(view).cpu().numpy(), kc[idx])
    assert np.array_equal(v.view(view).cpu().numpy(), vc[idx])


def test_gather_out_of_pool_entry_zero_fills_and_flags():
    w = W.make("tiny", device=DEV)
    tables = w.block_tables.copy()
    tables[3, 2] = w.num_blocks + 5            # a live entry of the 100-token sequence
    bt = torch.from_numpy(tables).to(DEV)
    sl = torch.from_numpy(w.seq_lens).to(DEV)
    pa.device_error()
    k, v = pa.paged_kv_gather(w.k_cache, w.v_cache, bt, sl, w.max_seq_len)
    torch.cuda.synchronize()
    assert pa.device_error() == 1
    start = int(w.seq_lens[:3].sum())
    assert float(k[start + 32: start + 48].float().abs().max()) == 0.0
    assert float(k[start: start + 32].float().abs().max()) > 0.0
