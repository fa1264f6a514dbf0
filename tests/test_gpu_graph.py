"""A decode step captured once in a CUDA graph and replayed, as a serving
engine does ("vLLM-Ascend 原理", section 4 "图模式": capture a decode step,
then replay it with new contents written into fixed-address inputs; block
tables are inputs whose contents change every step).  The library's calls
only enqueue work on the caller's stream, so the whole step (slot mapping,
KV write, work-list, decode, reduce) is capturable; max_seq_len is the
capture-time bound and the batch size is fixed (a bucket)."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_attention_decode_gb300 as pa
from paged_kv_attention_decode_gb300 import workloads as W
from tests._gpu_util import TOL, bits

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _step_inputs(seed, lens, nb, Hq=8, Hkv=2, D=128):
    return W.build_workload(name=f"g{seed}", seq_lens=lens, q_lens=1, num_q_heads=Hq, num_kv_heads=Hkv,
                            head_dim=D, dtype="bf16", seed=seed, num_blocks=nb, device=DEV)


def test_captured_decode_step_replays_with_new_inputs():
    max_len, nb = 2048, 2000
    w0 = _step_inputs(1, [100, 2048, 700, 33], nb)
    # fixed-address buffers
    q, key, value = w0.q.clone(), w0.key.clone(), w0.value.clone()
    kc, vc = w0.k_cache.clone(), w0.v_cache.clone()
    bt = torch.zeros(4, max_len // 16, dtype=torch.int32, device=DEV)
    sl = torch.zeros(4, dtype=torch.int32, device=DEV)
    slots = torch.empty(4, dtype=torch.int64, device=DEV)
    out = torch.empty_like(q)
    ws = torch.empty(pa.decode_workspace_bytes(4, 8, 128, max_len, 0), dtype=torch.uint8, device=DEV)

    def load(w):
        q.copy_(w.q); key.copy_(w.key); value.copy_(w.value)
        bt.zero_(); bt[:, : w.block_tables.shape[1]].copy_(torch.from_numpy(w.block_tables))
        sl.copy_(torch.from_numpy(w.seq_lens))

    def step():
        pa.slot_mapping(bt, sl, None, 4, nb, out=slots)
        pa.paged_kv_write(key, value, kc, vc, slots)
        pa.paged_attention_decode(q, kc, vc, bt, sl, w0.scale, max_len, out=out, workspace=ws)

    load(w0)
    step()                      # first call on the device does its one-time set-up
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()

    for seed, lens in ((2, [1, 1500, 2047, 16]), (3, [512, 513, 2, 900])):
        w = _step_inputs(seed, lens, nb)
        kc.copy_(w.k_cache); vc.copy_(w.v_cache)
        load(w)
        graph.replay()
        torch.cuda.synchronize()
        replayed = out.clone()
        # eager on the same inputs (the cache already holds this step's tokens)
        kc.copy_(w.k_cache); vc.copy_(w.v_cache)
        step()
        torch.cuda.synchronize()
        assert torch.equal(replayed.view(torch.int16), out.view(torch.int16))
        # and the oracle
        okc, ovc = bits(w.k_cache), bits(w.v_cache)
        oracle.kv_write(bits(w.key), bits(w.value), okc, ovc,
                        oracle.slot_mapping(w.block_tables, w.seq_lens, w.q_lens, 16, nb))
        ref = oracle.paged_attention_decode(bits(w.q), okc, ovc, w.block_tables, w.seq_lens, w.scale, "bf16")
        err = float(np.max(np.abs(replayed.double().cpu().numpy() - ref)))
        assert err <= TOL["bf16"], err
    assert pa.device_error() == 0


def test_captured_decode_bucket_with_padding_rows():
    """A batch smaller than the captured bucket: the unused rows are padding
    (seq_len 0).  They place no token, read nothing and come out as zero rows;
    the real rows match eager calls and the oracle, and nothing is flagged."""
    max_len, nb, B = 1024, 600, 6
    w0 = _step_inputs(11, [300, 1024, 17, 512, 64, 900], nb)
    q, key, value = w0.q.clone(), w0.key.clone(), w0.value.clone()
    kc, vc = w0.k_cache.clone(), w0.v_cache.clone()
    bt = torch.zeros(B, max_len // 16, dtype=torch.int32, device=DEV)
    sl = torch.zeros(B, dtype=torch.int32, device=DEV)
    slots = torch.empty(B, dtype=torch.int64, device=DEV)
    out = torch.empty_like(q)
    ws = torch.empty(pa.decode_workspace_bytes(B, 8, 128, max_len, 0), dtype=torch.uint8, device=DEV)

    def step():
        pa.slot_mapping(bt, sl, None, B, nb, out=slots)
        pa.paged_kv_write(key, value, kc, vc, slots)
        pa.paged_attention_decode(q, kc, vc, bt, sl, w0.scale, max_len, out=out, workspace=ws)

    bt[:, : w0.block_tables.shape[1]].copy_(torch.from_numpy(w0.block_tables))
    sl.copy_(torch.from_numpy(w0.seq_lens))
    step()
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()

    real = [0, 2, 3]                     # rows 1, 4 and 5 are padding in this step
    w = _step_inputs(12, [700, 1, 1000, 250, 1, 1], nb)
    lens = w.seq_lens.copy()
    lens[[1, 4, 5]] = 0
    kc.copy_(w.k_cache); vc.copy_(w.v_cache)
    q.copy_(w.q); key.copy_(w.key); value.copy_(w.value)
    bt.zero_(); bt[:, : w.block_tables.shape[1]].copy_(torch.from_numpy(w.block_tables))
    sl.copy_(torch.from_numpy(lens))
    pa.device_error()
    graph.replay()
    torch.cuda.synchronize()
    assert pa.device_error() == 0
    assert torch.all(slots[[1, 4, 5]] == -1)
    assert torch.count_nonzero(out[[1, 4, 5]]) == 0
    replayed = out.clone()
    okc, ovc = bits(w.k_cache), bits(w.v_cache)
    sel = np.array(real)
    oracle.kv_write(bits(w.key[real]), bits(w.value[real]), okc, ovc,
                    oracle.slot_mapping(w.block_tables[sel], lens[sel], np.ones(len(real), np.int32), 16, nb))
    ref = oracle.paged_attention_decode(bits(w.q[real]), okc, ovc, w.block_tables[sel], lens[sel], w.scale, "bf16")
    err = float(np.max(np.abs(replayed[real].double().cpu().numpy() - ref)))
    assert err <= TOL["bf16"], err


def test_captured_mixed_step_replays_with_new_inputs():
    """A continuous-batching step (a prefill chunk, a speculative-verify chunk
    and decodes in one varlen call) captured once and replayed with other
    splits of the same token budget: the chunk tile plan, the decode plan and
    the side-by-side prefill and decode kernels all run from device data, so
    only num_tokens, num_seqs and the host bounds (max_q_len, max_seq_len)
    are fixed at capture."""
    B, T, max_q, max_len, nb = 4, 64, 64, 2048, 2000
    Hq, Hkv, D = 8, 2, 128

    def inputs(seed, q_lens, prefix):
        return W.build_workload(name=f"m{seed}", seq_lens=[q + p for q, p in zip(q_lens, prefix)], q_lens=q_lens,
                                num_q_heads=Hq, num_kv_heads=Hkv, head_dim=D, dtype="bf16", seed=seed,
                                num_blocks=nb, device=DEV)

    w0 = inputs(11, [40, 1, 3, 20], [100, 700, 50, 1000])
    q, key, value = w0.q.clone(), w0.key.clone(), w0.value.clone()
    kc, vc = w0.k_cache.clone(), w0.v_cache.clone()
    bt = torch.zeros(B, max_len // 16, dtype=torch.int32, device=DEV)
    sl = torch.zeros(B, dtype=torch.int32, device=DEV)
    cu = torch.zeros(B + 1, dtype=torch.int32, device=DEV)
    slots = torch.empty(T, dtype=torch.int64, device=DEV)
    out = torch.empty_like(q)
    ws = torch.empty(pa.prefill_workspace_bytes(B, T, Hq, D, max_len), dtype=torch.uint8, device=DEV)

    def load(w):
        q.copy_(w.q); key.copy_(w.key); value.copy_(w.value)
        bt.zero_(); bt[:, : w.block_tables.shape[1]].copy_(torch.from_numpy(w.block_tables))
        sl.copy_(torch.from_numpy(w.seq_lens))
        cu.copy_(torch.from_numpy(w.cu_q_lens))

    def step():
        pa.slot_mapping(bt, sl, cu, T, nb, out=slots)
        pa.paged_kv_write(key, value, kc, vc, slots)
        pa.paged_attention_prefill(q, kc, vc, bt, sl, cu, w0.scale, max_q, max_len, out=out, workspace=ws)

    load(w0)
    step()
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()

    for seed, q_lens, prefix in ((12, [8, 1, 1, 54], [2000, 5, 300, 0]),      # verify-size chunk + a long one
                                 (13, [1, 1, 1, 61], [1, 1500, 900, 1987]),    # decodes + one long chunk
                                 (14, [16, 16, 16, 16], [16, 0, 700, 33])):    # four prefill chunks
        w = inputs(seed, q_lens, prefix)
        kc.copy_(w.k_cache); vc.copy_(w.v_cache)
        load(w)
        graph.replay()
        torch.cuda.synchronize()
        replayed = out.clone()
        kc.copy_(w.k_cache); vc.copy_(w.v_cache)
        step()
        torch.cuda.synchronize()
        assert torch.equal(replayed.view(torch.int16), out.view(torch.int16)), q_lens
        okc, ovc = bits(w.k_cache), bits(w.v_cache)
        oracle.kv_write(bits(w.key), bits(w.value), okc, ovc,
                        oracle.slot_mapping(w.block_tables, w.seq_lens, w.q_lens, 16, nb))
        ref = oracle.paged_attention_prefill(bits(w.q), okc, ovc, w.block_tables, w.seq_lens, w.q_lens, w.scale,
                                             "bf16")
        err = float(np.max(np.abs(replayed.double().cpu().numpy() - ref)))
        assert err <= TOL["bf16"], (q_lens, err)
    assert pa.device_error() == 0
