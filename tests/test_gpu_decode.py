"""GPU parity of decode attention against the fp64 oracle, plus its edge cases.

Tolerance: max |err| <= 2e-3 (fp16) and <= 1.6e-2 (bf16) against the fp64
oracle on the same inputs.  Every case writes the step's new token through
the library first, then attends; unused pool memory is NaN-poisoned, so a
kernel that reads a slot it must not read fails the finiteness check.
"""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_attention_decode_gb300 as pa
from paged_kv_attention_decode_gb300 import workloads as W
from tests._gpu_util import TOL, bits, gpu_step, max_err, oracle_rows, snapshot

pytestmark = pytest.mark.gpu
DEV = "cuda"
LENS = [1, 2, 15, 16, 17, 31, 33, 100, 511, 512, 513, 1000, 2049]


def _check(w, partition=0):
    seqs = np.arange(w.batch)
    snap = snapshot(w, seqs)
    _, out = gpu_step(w, partition_size=partition, prefill=False)
    rows, ref = oracle_rows(w, seqs, snap)
    err = max_err(out[torch.from_numpy(rows).to(DEV)], ref)
    assert err <= TOL[w.dtype], err
    assert pa.device_error() == 0
    return out


def test_tiny_workload():
    _check(W.make("tiny", device=DEV, poison=True))


@pytest.mark.parametrize("Hq,Hkv,D,dtype", [
    (4, 4, 64, "f16"), (8, 8, 128, "f16"), (8, 8, 128, "bf16"), (8, 4, 128, "bf16"),
    (16, 4, 128, "bf16"), (16, 2, 64, "f16"), (24, 3, 128, "bf16"), (8, 1, 128, "f16"),
    (12, 4, 64, "bf16"), (7, 7, 128, "f16"),
    # large groups: 16 and 32 (multi-query) heads per kv head, and the limit
    (32, 2, 128, "bf16"), (32, 1, 128, "f16"), (64, 1, 64, "bf16"),
])
@pytest.mark.parametrize("partition", [0, 16, 48, 4096])
def test_decode_parity(Hq, Hkv, D, dtype, partition):
    w = W.build_workload(name="case", seq_lens=LENS, q_lens=1, num_q_heads=Hq, num_kv_heads=Hkv,
                         head_dim=D, dtype=dtype, seed=Hq * 131 + Hkv * 7 + D, device=DEV, poison=True,
                         pool_slack=0.3)
    _check(w, partition)


def test_prefix_sharing_gqa():
    _check(W.make("gqa_prefix", batch=48, device=DEV, poison=True))


# Prefix sharing (sequences whose leading block ids are the same physical
# blocks): share groups of several sizes over an odd batch, shared prefixes
# shorter than a partition, and partition lengths that put the shared blocks
# in one or many partitions.
@pytest.mark.parametrize("Hq,Hkv,dtype", [(16, 4, "bf16"), (16, 8, "f16"), (8, 4, "f16")])
@pytest.mark.parametrize("share_groups,share_tokens", [(2, 1024), (3, 512), (5, 1536), (16, 48)])
@pytest.mark.parametrize("partition", [0, 16, 64])
def test_shared_prefix_groups(Hq, Hkv, dtype, share_groups, share_tokens, partition):
    lens = np.random.default_rng(share_groups * 31 + share_tokens).integers(1, 3000, size=23)
    w = W.build_workload(name="share", seq_lens=lens, q_lens=1, num_q_heads=Hq, num_kv_heads=Hkv,
                         head_dim=128, dtype=dtype, seed=Hq + share_groups, device=DEV, poison=True,
                         pool_slack=0.3, share_groups=share_groups, share_tokens=share_tokens)
    _check(w, partition)


def test_output_is_independent_of_physical_placement():
    w = W.build_workload(name="perm", seq_lens=LENS, q_lens=1, num_q_heads=16, num_kv_heads=4,
                         head_dim=128, dtype="bf16", seed=3, device=DEV)
    bt = torch.from_numpy(w.block_tables).to(DEV)
    sl = torch.from_numpy(w.seq_lens).to(DEV)
    out = pa.paged_attention_decode(w.q, w.k_cache, w.v_cache, bt, sl, w.scale, w.max_seq_len)
    pi = torch.from_numpy(np.random.default_rng(4).permutation(w.num_blocks)).to(DEV)
    kc2 = torch.empty_like(w.k_cache)
    vc2 = torch.empty_like(w.v_cache)
    kc2[pi] = w.k_cache
    vc2[pi] = w.v_cache
    bt2 = pi[bt.long()].to(torch.int32)
    out2 = pa.paged_attention_decode(w.q, kc2, vc2, bt2, sl, w.scale, w.max_seq_len)
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int16), out2.view(torch.int16))


def test_seq_len_one_returns_v_and_zero_len_returns_zeros():
    w = W.build_workload(name="edge", seq_lens=[1, 5, 1], q_lens=1, num_q_heads=8, num_kv_heads=2,
                         head_dim=128, dtype="f16", seed=8, device=DEV, poison=True)
    gpu_step(w)  # writes the new tokens; seq 0 and 2 have only that token
    bt = torch.from_numpy(w.block_tables).to(DEV)
    sl = torch.tensor([1, 0, 1], dtype=torch.int32, device=DEV)
    out = pa.paged_attention_decode(w.q, w.k_cache, w.v_cache, bt, sl, w.scale, max_seq_len=5)
    torch.cuda.synchronize()
    assert torch.count_nonzero(out[1]) == 0
    for b in (0, 2):
        v = w.value[b].repeat_interleave(4, dim=0)          # q head h reads kv head h // 4
        assert torch.equal(out[b].view(torch.int16), v.view(torch.int16))
    assert pa.device_error() == 0


def test_seq_len_above_bound_is_flagged_with_zero_row():
    w = W.build_workload(name="over", seq_lens=[40, 50], q_lens=1, num_q_heads=4, num_kv_heads=4,
                         head_dim=64, dtype="f16", seed=9, device=DEV)
    bt = torch.from_numpy(w.block_tables).to(DEV)
    sl = torch.from_numpy(w.seq_lens).to(DEV)
    pa.device_error()
    out = pa.paged_attention_decode(w.q, w.k_cache, w.v_cache, bt, sl, w.scale, max_seq_len=45)
    assert pa.device_error() == 4
    assert torch.count_nonzero(out[1]) == 0


def test_bad_block_id_is_skipped_and_flagged():
    w = W.build_workload(name="bad", seq_lens=[64, 64], q_lens=1, num_q_heads=8, num_kv_heads=2,
                         head_dim=128, dtype="bf16", seed=10, device=DEV)
    tables = w.block_tables.copy()
    tables[1, 1] = w.num_blocks + 5          # a live entry outside the pool
    bt = torch.from_numpy(tables).to(DEV)
    sl = torch.from_numpy(w.seq_lens).to(DEV)
    pa.device_error()
    out = pa.paged_attention_decode(w.q, w.k_cache, w.v_cache, bt, sl, w.scale, max_seq_len=64,
                                    partition_size=32)
    assert pa.device_error() == 1
    assert torch.isfinite(out.float()).all()


def test_unsupported_shapes_are_rejected_before_launch():
    q = torch.zeros(2, 4, 96, device=DEV, dtype=torch.float16)
    kc = torch.zeros(4, 16, 4, 96, device=DEV, dtype=torch.float16)
    bt = torch.zeros(2, 1, device=DEV, dtype=torch.int32)
    sl = torch.ones(2, device=DEV, dtype=torch.int32)
    with pytest.raises(pa.PagedAttnError):
        pa.paged_attention_decode(q, kc, kc, bt, sl, 0.1, max_seq_len=1)


@pytest.mark.parametrize("empty_row", [False, True])
def test_calls_back_to_back_on_one_workspace(empty_row):
    """Decode calls queued with no other kernel between them, on one workspace,
    each of one partition (so no reduce kernel separates them).  A call's
    plan rewrites the work list, the work counter and the zero rows of empty
    sequences; it must not do so while the previous call's kernel still
    claims items.  The second call has fewer sequences, and optionally an
    empty one whose zero row lands on a row the first call writes."""
    rng = np.random.default_rng(21)
    wa = W.build_workload(name="b2b_a", seq_lens=rng.integers(300, 513, 120), q_lens=1, num_q_heads=32,
                          num_kv_heads=32, head_dim=128, dtype="f16", seed=31, device=DEV)
    wb = W.build_workload(name="b2b_b", seq_lens=rng.integers(1, 513, 13), q_lens=1, num_q_heads=32,
                          num_kv_heads=8, head_dim=128, dtype="f16", seed=32, device=DEV)
    bta, sla = (torch.from_numpy(x).to(DEV) for x in (wa.block_tables, wa.seq_lens))
    btb = torch.from_numpy(wb.block_tables).to(DEV)
    lens_b = wb.seq_lens.copy()
    if empty_row:
        lens_b[4] = 0
    slb = torch.from_numpy(lens_b).to(DEV)
    assert pa.decode_partition(512) == 512
    need = max(pa.decode_workspace_bytes(wa.batch, 32, 128, 512), pa.decode_workspace_bytes(wb.batch, 32, 128, 512))
    ws = torch.empty(need, dtype=torch.uint8, device=DEV)
    snap_a = snapshot(wa, np.arange(wa.batch))
    snap_b = snapshot(wb, np.arange(wb.batch))
    out_a = torch.full_like(wa.q, float("nan"))
    out_b = torch.full_like(wb.q, float("nan"))
    # the second call writes into the first call's output rows as well
    shared_out = out_a[: wb.batch]
    torch.cuda.synchronize()
    for _ in range(3):
        pa.paged_attention_decode(wa.q, wa.k_cache, wa.v_cache, bta, sla, wa.scale, max_seq_len=512, out=out_a,
                                  workspace=ws)
        pa.paged_attention_decode(wb.q, wb.k_cache, wb.v_cache, btb, slb, wb.scale, max_seq_len=512, out=out_b,
                                  workspace=ws)
    pa.paged_attention_decode(wb.q, wb.k_cache, wb.v_cache, btb, slb, wb.scale, max_seq_len=512,
                              out=shared_out, workspace=ws)
    torch.cuda.synchronize()
    kc, vc, tables = snap_a
    ref_a = oracle.paged_attention_decode(bits(wa.q), kc, vc, tables, wa.seq_lens, wa.scale, "f16")
    kc, vc, tables = snap_b
    ref_b = oracle.paged_attention_decode(bits(wb.q), kc, vc, tables, lens_b, wb.scale, "f16")
    assert max_err(out_a[wb.batch:], ref_a[wb.batch:]) <= TOL["f16"]
    assert max_err(out_b, ref_b) <= TOL["f16"]
    assert torch.equal(shared_out.view(torch.int16), out_b.view(torch.int16))
    if empty_row:
        assert torch.count_nonzero(out_b[4]) == 0
    assert pa.device_error() == 0
