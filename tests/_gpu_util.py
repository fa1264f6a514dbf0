"""GPU-test plumbing: run the library's step on a workload and build the
oracle's view of the same inputs (no attention arithmetic here)."""
import numpy as np
import torch

import oracle
import paged_kv_attention_decode_gb300 as pa

TOL = {"f16": 2e-3, "bf16": 1.6e-2}   # max |err| vs the fp64 oracle


def bits(t: torch.Tensor) -> np.ndarray:
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


def live_blocks(w, b: int) -> np.ndarray:
    return w.block_tables[b, : -(-int(w.seq_lens[b]) // 16)]


def snapshot(w, seqs):
    """CPU copy of the pool blocks the given sequences use, with their tables
    renumbered onto the compact copy (a physical-block permutation)."""
    seqs = np.asarray(seqs, dtype=np.int64)
    used = np.unique(np.concatenate([live_blocks(w, b) for b in seqs])).astype(np.int64)
    idx = torch.from_numpy(used).to(w.k_cache.device)
    kc = bits(w.k_cache.index_select(0, idx))
    vc = bits(w.v_cache.index_select(0, idx))
    remap = {int(x): i for i, x in enumerate(used)}
    tables = np.zeros((len(seqs), w.max_blocks_per_seq), dtype=np.int32)
    for r, b in enumerate(seqs):
        lb = live_blocks(w, b)
        tables[r, : lb.size] = [remap[int(x)] for x in lb]
    return kc, vc, tables


def gpu_step(w, partition_size=0, prefill=None):
    """slot mapping -> KV write -> attention, all through the library.
    Returns (slots, out) as torch tensors; the caches are updated in place."""
    dev = w.k_cache.device
    bt = torch.from_numpy(w.block_tables).to(dev)
    sl = torch.from_numpy(w.seq_lens).to(dev)
    if prefill is None:
        prefill = not w.is_decode
    cu = torch.from_numpy(w.cu_q_lens).to(dev) if prefill else None
    slots = pa.slot_mapping(bt, sl, cu, w.num_tokens, w.num_blocks)
    pa.paged_kv_write(w.key, w.value, w.k_cache, w.v_cache, slots)
    if prefill:
        out = pa.paged_attention_prefill(w.q, w.k_cache, w.v_cache, bt, sl, cu, w.scale, w.max_q_len,
                                         w.max_seq_len)
    else:
        out = pa.paged_attention_decode(w.q, w.k_cache, w.v_cache, bt, sl, w.scale,
                                        max_seq_len=w.max_seq_len, partition_size=partition_size)
    torch.cuda.synchronize()
    return slots, out


def oracle_rows(w, seqs, snap, q_rows_per_seq=None):
    """fp64 oracle for the given sequences on a pre-write snapshot: the oracle
    writes the new tokens itself, then attends.  Returns (rows, out[rows])."""
    kc, vc, tables = snap
    seqs = np.asarray(seqs, dtype=np.int64)
    cu = w.cu_q_lens
    sl = w.seq_lens[seqs]
    ql = w.q_lens[seqs]
    rows = np.concatenate([np.arange(cu[b], cu[b + 1]) for b in seqs]).astype(np.int64)
    slots = oracle.slot_mapping(tables, sl, ql, 16, kc.shape[0])
    rows_t = torch.from_numpy(rows).to(w.key.device)
    oracle.kv_write(bits(w.key.index_select(0, rows_t)), bits(w.value.index_select(0, rows_t)), kc, vc, slots)
    q = bits(w.q.index_select(0, rows_t))
    if q_rows_per_seq is None:
        out = oracle.paged_attention_prefill(q, kc, vc, tables, sl, ql, w.scale, w.dtype)
        return rows, out
    # a subset of each sequence's rows (local indices into the packed q of seqs)
    sel, keep = [], []
    base = 0
    for r, b in enumerate(seqs):
        for i in q_rows_per_seq(int(b), int(ql[r])):
            sel.append(base + i)
            keep.append(rows[base + i])
        base += int(ql[r])
    out = oracle.paged_attention_prefill(q, kc, vc, tables, sl, ql, w.scale, w.dtype, select=np.array(sel))
    return np.array(keep, dtype=np.int64), out


def max_err(gpu_rows: torch.Tensor, ref: np.ndarray) -> float:
    g = gpu_rows.detach().cpu().to(torch.float64).numpy()
    assert g.shape == ref.shape
    assert np.all(np.isfinite(g)), "non-finite GPU output"
    return float(np.max(np.abs(g - ref))) if g.size else 0.0
