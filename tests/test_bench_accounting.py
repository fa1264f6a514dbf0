"""The benchmark's roofline numerators, pinned on the CPU.

`bench._algorithmic_bytes` is what the HBM roofline divides by time and
`bench._prefill_flops` what the tensor roofline divides by time.  They are
pinned to the pages' own sizing example ("vLLM-Ascend 原理", section 2.1
PagedAttention: about 512 KB of K/V per token and 2 GB per 4096-token sequence
for LLaMA-2-7B in fp16), to totals counted by hand for small workloads
(private blocks, a shared prefix, an FP8 cache, varlen rows), and, for the
FLOPs, to a brute-force count of the (query, key) pairs causal attention
visits.
"""
import json
import os

import numpy as np
import pytest

import bench
from paged_kv_attention_decode_gb300 import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def test_kv_bytes_match_the_pages_sizing_example():
    g = json.load(open(os.path.join(GOLDEN, "kv_sizing.json")))
    for n, want in ((1, g["kv_bytes_per_token"]), (g["seq_tokens"], g["kv_bytes_per_seq"])):
        w = W.build_workload(name="s", seq_lens=[n], q_lens=1, num_q_heads=g["kv_heads"],
                             num_kv_heads=g["kv_heads"], head_dim=g["head_dim"], dtype="f16",
                             seed=0, num_blocks=-(-n // 16))
        ab = bench._algorithmic_bytes(w)
        assert ab["kv"] * g["layers"] == want
        assert ab["kv_unique"] == ab["kv"]


def test_tiny_workload_hand_count():
    # lengths 1, 17, 33, 100 (151 tokens, 1 + 2 + 3 + 7 = 13 live blocks);
    # 4 kv heads x 64 dims x 2 bytes x (K and V) = 1024 bytes per token
    ab = bench._algorithmic_bytes(W.make("tiny"))
    assert ab["kv"] == ab["kv_unique"] == 151 * 1024
    assert ab["q"] == ab["out"] == 4 * 4 * 64 * 2          # 4 rows x 4 q heads x 64 dims x 2 bytes
    assert ab["meta"] == 13 * 4 + 4 * 4                      # live table entries + lengths
    assert ab["total"] == 151 * 1024 + 2 * 2048 + 68 == 158_788


def test_shared_prefix_counts_shared_blocks_once():
    # three sequences share the physical blocks of their first 32 tokens
    # (two full blocks); 2 kv heads x 64 dims x 2 bytes x 2 = 512 bytes per token
    w = W.build_workload(name="share", seq_lens=[40, 50, 70], q_lens=1, num_q_heads=8, num_kv_heads=2,
                         head_dim=64, dtype="bf16", seed=3, share_groups=3, share_tokens=32)
    assert np.array_equal(w.block_tables[:, :2], np.repeat(w.block_tables[:1, :2], 3, axis=0))
    ab = bench._algorithmic_bytes(w)
    assert ab["kv"] == 160 * 512
    assert ab["kv_unique"] == (32 + 8 + 18 + 38) * 512      # the shared 32 rows once, then each private tail
    assert ab["meta"] == (3 + 4 + 5) * 4 + 3 * 4
    assert ab["total"] == 96 * 512 + 2 * (3 * 8 * 64 * 2) + 60
    assert ab["total_logical"] == 160 * 512 + 2 * (3 * 8 * 64 * 2) + 60


def test_fp8_cache_moves_one_byte_per_element():
    w = W.build_workload(name="fp8", seq_lens=[20, 33], q_lens=1, num_q_heads=4, num_kv_heads=4,
                         head_dim=128, dtype="f16", seed=4, cache_dtype="fp8")
    ab = bench._algorithmic_bytes(w)
    assert ab["kv"] == 53 * 4 * 128 * 2                     # K and V codes, one byte each
    assert ab["q"] == 2 * 4 * 128 * 2                       # queries stay 16-bit


def test_varlen_rows_count_queries_and_both_length_arrays():
    # a 3-query verify row and a 20-token chunk: 23 query rows; seq_lens and
    # cu_q_lens are both read
    w = W.build_workload(name="var", seq_lens=[5, 40], q_lens=[3, 20], num_q_heads=4, num_kv_heads=2,
                         head_dim=64, dtype="bf16", seed=5)
    ab = bench._algorithmic_bytes(w)
    assert ab["q"] == 23 * 4 * 64 * 2
    assert ab["meta"] == (1 + 3) * 4 + 2 * 4 * 2
    assert ab["kv"] == 45 * 2 * 64 * 2 * 2


def _visited_pairs_flops(w):
    """Brute force: every query row of a chunk longer than one token, at
    position n - c + i, attends to positions 0..n - c + i; each visited
    (query, key) pair costs 2 D flops for q.k and 2 D for p.v, per q head."""
    f = 0
    for n, c in zip(w.seq_lens.tolist(), w.q_lens.tolist()):
        if c <= 1:
            continue
        for i in range(c):
            f += (n - c + i + 1) * 4 * w.head_dim * w.num_q_heads
    return f


def test_prefill_flops_hand_count():
    # one chunk of 3 on a 2-token prefix: its queries see 3, 4 and 5 keys
    w = W.build_workload(name="pf", seq_lens=[5], q_lens=[3], num_q_heads=2, num_kv_heads=1,
                         head_dim=64, dtype="bf16", seed=6)
    assert bench._prefill_flops(w) == (3 + 4 + 5) * 4 * 64 * 2 == 6144


@pytest.mark.parametrize("lens,qlens", [
    ([100, 1, 37, 300], [100, 1, 9, 17]),        # a whole-sequence chunk, a decode row, chunks on prefixes
    ([1600, 4000, 1536], [1536, 1536, 1536]),    # the mixed step's chunk length
])
def test_prefill_flops_match_a_brute_force_count(lens, qlens):
    w = W.build_workload(name="pf", seq_lens=lens, q_lens=qlens, num_q_heads=4, num_kv_heads=2,
                         head_dim=128, dtype="bf16", seed=7)
    assert bench._prefill_flops(w) == _visited_pairs_flops(w)
