"""The host block manager driving real device steps: the copy-on-write block
copy kernel (bit-exact), and continuous-batching steps whose tables, lengths
and slots come from the manager (slot mapping bit-exact against the
manager's; attention identical with and without prefix sharing, and within
tolerance of the fp64 oracle)."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_attention_decode_gb300 as pa
from tests._gpu_util import TOL, bits, max_err

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.mark.parametrize("H,D,dtype", [(8, 128, torch.float16), (4, 64, torch.bfloat16), (8, 128, torch.uint8)])
def test_copy_blocks_bit_exact(H, D, dtype):
    g = torch.Generator(device=DEV)
    g.manual_seed(3)
    NB = 300
    if dtype == torch.uint8:
        kc = torch.randint(0, 256, (NB, 16, H, D), generator=g, device=DEV, dtype=torch.uint8)
        vc = torch.randint(0, 256, (NB, 16, H, D), generator=g, device=DEV, dtype=torch.uint8)
    else:
        kc = torch.randn(NB, 16, H, D, generator=g, device=DEV).to(dtype)
        vc = torch.randn(NB, 16, H, D, generator=g, device=DEV).to(dtype)
    rng = np.random.default_rng(4)
    perm = rng.permutation(NB)
    pairs = np.stack([perm[:40], perm[40:80]], axis=1).astype(np.int32)   # distinct sources and destinations
    k_ref, v_ref = kc.cpu().clone(), vc.cpu().clone()
    k_ref[torch.from_numpy(pairs[:, 1]).long()] = k_ref[torch.from_numpy(pairs[:, 0]).long()]
    v_ref[torch.from_numpy(pairs[:, 1]).long()] = v_ref[torch.from_numpy(pairs[:, 0]).long()]
    pa.device_error()
    pa.copy_blocks(kc, vc, torch.from_numpy(pairs).to(DEV))
    torch.cuda.synchronize()
    assert pa.device_error() == 0
    assert torch.equal(kc.cpu(), k_ref) and torch.equal(vc.cpu(), v_ref)
    # a pair outside the pool is skipped and flagged; the others still land
    bad = torch.tensor([[NB, 1], [2, 3]], dtype=torch.int32, device=DEV)
    before = kc[1].clone()
    pa.copy_blocks(kc, vc, bad)
    torch.cuda.synchronize()
    assert pa.device_error() == 1
    assert torch.equal(kc[1], before) and torch.equal(kc[3], kc[2])


def _kv(tokens, positions, H, D, which):
    g = np.random.default_rng(1000 + which)
    emb = g.standard_normal((64, H, D), dtype=np.float32)
    pos = g.standard_normal((8192, H, D), dtype=np.float32) * 0.5
    x = emb[np.asarray(tokens) % 64] + pos[np.asarray(positions)]
    return torch.from_numpy(x).to(torch.bfloat16)


def _serve_gpu(caching, steps=7, Hq=16, H=4, D=128):
    """Continuous batching on the device, driven by the manager: shared system
    prompts, prefill chunks, decodes, a 4-token verify chunk with rollback and
    a fork.  Returns {(step, seq, position): output row} and the last step's
    inputs for an oracle check."""
    rng = np.random.default_rng(11)
    NB = 512
    m = pa.BlockManager(NB, 16, caching)
    kc = torch.zeros(NB, 16, H, D, dtype=torch.bfloat16, device=DEV)
    vc = torch.zeros_like(kc)
    qtab = torch.from_numpy(rng.standard_normal((64, Hq, D), dtype=np.float32)).to(torch.bfloat16)
    system = [int(x) for x in rng.integers(0, 64, size=300)]
    prompts = {s: system + [int(x) for x in rng.integers(0, 64, size=int(rng.integers(5, 200)))] for s in range(1, 5)}
    prompts[5] = [int(x) for x in rng.integers(0, 64, size=700)]
    tokens, rows, last = {}, {}, None
    for step in range(steps):
        batch, qlens = [], []
        for sid in ([1, 5] if step == 0 else [2, 3] if step == 1 else [4] if step == 2 else []):
            tokens[sid] = list(prompts[sid])
            cached = m.add_sequence(sid, prompts[sid])
            assert m.allocate_slots(sid, len(prompts[sid]) - cached) is None
            batch.append(sid)
            qlens.append(len(prompts[sid]) - cached)
        if step == 4:
            m.fork(2, 6)
            tokens[6] = list(tokens[2])
        if step == 5:
            m.truncate(5, m.seq_len(5) - 3)                        # 3 of 4 drafts rejected
            del tokens[5][-3:]
        pairs = []
        for sid in sorted(t for t in tokens if t not in batch):
            k = 4 if sid == 5 else 1
            new = [int(x) for x in rng.integers(0, 64, size=k)]
            tokens[sid] += new
            m.append_tokens(sid, new)
            pr = m.allocate_slots(sid, k)
            if pr:
                pairs.append(pr)
            batch.append(sid)
            qlens.append(k)
        if pairs:
            pa.copy_blocks(kc, vc, torch.tensor(pairs, dtype=torch.int32, device=DEV))
        tables, lens, cu, slots = m.build_step(batch, qlens, 64)
        toks, poss, keys = [], [], []
        for i, sid in enumerate(batch):
            for pos in range(lens[i] - qlens[i], lens[i]):
                toks.append(tokens[sid][pos])
                poss.append(pos)
                keys.append((step, sid, pos))
        bt, sl, cq = (torch.from_numpy(x).to(DEV) for x in (tables, lens, cu))
        T = len(toks)
        dslots = pa.slot_mapping(bt, sl, cq, T, NB)
        assert np.array_equal(dslots.cpu().numpy(), slots)
        key = _kv(toks, poss, H, D, 0).to(DEV)
        val = _kv(toks, poss, H, D, 1).to(DEV)
        q = qtab[torch.from_numpy(np.asarray(toks) % 64)].contiguous().to(DEV)
        snap = (bits(kc), bits(vc))
        pa.paged_kv_write(key, val, kc, vc, dslots)
        out = pa.paged_attention_prefill(q, kc, vc, bt, sl, cq, 0.088, int(max(qlens)), int(lens.max()))
        torch.cuda.synchronize()
        assert pa.device_error() == 0
        rows.update(zip(keys, out.cpu()))
        last = (snap, tables, lens, np.asarray(qlens, np.int32), slots, key, val, q, out)
    return rows, m.num_free_blocks, last


def test_manager_driven_steps():
    shared, free_shared, last = _serve_gpu(True)
    private, free_private, _ = _serve_gpu(False)
    assert free_shared > free_private
    assert set(shared) < set(private)
    for k, row in shared.items():
        assert torch.equal(row, private[k]), k
    # the last step of the shared run against the fp64 oracle
    (kcb, vcb), tables, lens, qlens, slots, key, val, q, out = last
    oracle.kv_write(bits(key), bits(val), kcb, vcb, slots)
    ref = oracle.paged_attention_prefill(bits(q), kcb, vcb, tables, lens, qlens, 0.088, "bf16")
    assert max_err(out, ref) <= TOL["bf16"]
