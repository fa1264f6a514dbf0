"""Host-side checks of the seeded workload builder and of the byte accounting."""
import json
import os

import numpy as np
import pytest
import torch

from paged_kv_attention_decode_gb300 import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def test_kv_byte_accounting_matches_the_pages_sizing_example():
    g = json.load(open(os.path.join(GOLDEN, "kv_sizing.json")))
    for n, want in ((1, g["kv_bytes_per_token"]), (g["seq_tokens"], g["kv_bytes_per_seq"])):
        w = W.build_workload(name="s", seq_lens=[n], q_lens=1, num_q_heads=g["kv_heads"],
                             num_kv_heads=g["kv_heads"], head_dim=g["head_dim"], dtype="f16",
                             seed=0, num_blocks=-(-n // 16))
        assert w.kv_bytes_logical() * g["layers"] == want


def test_tiny_matches_its_description():
    w = W.make("tiny")
    assert list(w.seq_lens) == [1, 17, 33, 100]
    assert w.num_blocks == 64 and w.head_dim == 64 and w.num_q_heads == w.num_kv_heads == 4
    live = np.concatenate([w.block_tables[b, : -(-int(n) // 16)] for b, n in enumerate(w.seq_lens)])
    assert live.size == 13 and np.unique(live).size == 13
    assert w.k_cache.dtype == torch.float16


def test_builds_are_deterministic():
    a = W.make("gqa_prefix", batch=32)
    b = W.make("gqa_prefix", batch=32)
    assert np.array_equal(a.block_tables, b.block_tables)
    assert torch.equal(a.k_cache.view(torch.int16), b.k_cache.view(torch.int16))
    assert torch.equal(a.q.view(torch.int16), b.q.view(torch.int16))


def test_live_blocks_are_private_except_shared_prefix():
    w = W.make("gqa_prefix", batch=64)
    shared = w.meta["shared_blocks"]
    owners = {}
    for b in range(w.batch):
        nb = -(-int(w.seq_lens[b]) // 16)
        for j in range(nb):
            owners.setdefault(int(w.block_tables[b, j]), set()).add((b, j))
    for blk, who in owners.items():
        if len(who) > 1:
            # only the same logical block index of one group may share
            js = {j for _, j in who}
            groups = {b // 16 for b, _ in who}
            assert len(js) == 1 and len(groups) == 1
            assert all(j < shared[b] for b, j in who)
    # every new token's block is private
    for b in range(w.batch):
        j = (int(w.seq_lens[b]) - 1) // 16
        assert len(owners[int(w.block_tables[b, j])]) == 1


def test_mixed_step_shape():
    w = W.make("mixed", n_decode=64)
    assert int((w.q_lens == 1536).sum()) == 4
    assert w.num_tokens == 4 * 1536 + 64
    pre = w.q_lens > 1
    assert np.all(w.seq_lens[pre] >= 1536) and np.all(w.seq_lens[pre] <= 1536 + 4096)


def test_poison_marks_only_dead_positions():
    w = W.build_workload(name="p", seq_lens=[5, 20, 33], q_lens=[1, 4, 1], num_q_heads=2,
                         num_kv_heads=2, head_dim=8, dtype="f16", seed=1, pool_slack=1.0,
                         poison=True)
    kc = w.k_cache.float()
    for b, (n, ql) in enumerate(zip(w.seq_lens, w.q_lens)):
        for t in range(-(-int(n) // 16) * 16):
            blk, off = w.block_tables[b, t // 16], t % 16
            assert bool(torch.isnan(kc[blk, off]).all()) == (t >= n - ql)


@pytest.mark.parametrize("name", ["llama7b_decode", "long_context", "mixed", "gqa_prefix"])
def test_large_config_tables(name):
    w = W.make(name, materialize=False)
    nb = -(-w.seq_lens.astype(np.int64) // 16)
    assert w.num_blocks >= nb.sum() - (w.meta["shared_blocks"].sum())
    live = np.concatenate([w.block_tables[b, : nb[b]] for b in range(w.batch)])
    assert live.min() >= 0 and live.max() < w.num_blocks
    if name != "gqa_prefix":
        assert np.unique(live).size == live.size
