"""Failure detection without a GPU fault: a bounded wait runs out on a
barrier phase that nothing completes, the kernel records PA_DEVERR_TIMEOUT
and returns, the host reads the status, and the context stays usable for the
attention path afterwards."""
import time

import numpy as np
import pytest
import torch

import oracle
import paged_kv_attention_decode_gb300 as pa
from paged_kv_attention_decode_gb300 import workloads as W
from tests._gpu_util import bits

pytestmark = pytest.mark.gpu
DEV = "cuda"


def test_bounded_wait_gives_up_and_the_context_stays_usable():
    pa.device_error()                      # start from a clear error word
    t0 = time.perf_counter()
    pa.selftest_wait_timeout()
    code = pa.device_error()               # waits for the stream, reads and clears
    elapsed = time.perf_counter() - t0
    assert code == 8, code                 # PA_DEVERR_TIMEOUT
    assert 0.5 < elapsed < 30.0, elapsed   # the wait's limit is about one second
    assert pa.device_error() == 0

    # the same context still runs slot mapping, KV write and decode correctly
    w = W.make("tiny")
    bt = torch.from_numpy(w.block_tables).to(DEV)
    sl = torch.from_numpy(w.seq_lens).to(DEV)
    kc, vc = w.k_cache.to(DEV), w.v_cache.to(DEV)
    slots = pa.slot_mapping(bt, sl, None, w.batch, w.num_blocks)
    pa.paged_kv_write(w.key.to(DEV), w.value.to(DEV), kc, vc, slots)
    out = pa.paged_attention_decode(w.q.to(DEV), kc, vc, bt, sl, w.scale, max_seq_len=w.max_seq_len)
    torch.cuda.synchronize()
    okc, ovc = bits(w.k_cache), bits(w.v_cache)
    oracle.kv_write(bits(w.key), bits(w.value), okc, ovc,
                    oracle.slot_mapping(w.block_tables, w.seq_lens, w.q_lens, 16, w.num_blocks))
    ref = oracle.paged_attention_decode(bits(w.q), okc, ovc, w.block_tables, w.seq_lens, w.scale, "f16")
    assert float(np.max(np.abs(out.cpu().double().numpy() - ref))) <= 2e-3
    assert pa.device_error() == 0
