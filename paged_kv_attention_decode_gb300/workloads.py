"""Seeded synthetic workloads for paged KV attention.

This module only *builds inputs*: per-sequence context lengths, block tables
(a scheduler's job: which physical block holds each logical 16-token block),
the query rows and the new key/value rows of one step, and a pre-filled block
pool.  It holds none of the attention arithmetic and none of the slot-address
translation; both the CUDA path and the CPU oracle consume what it returns.

The layout follows the pages' description of vLLM's paged cache ("vLLM 在
CANN 上的推理优化", section "vLLM 的 PagedAttention 数据结构": a pool
``[num_blocks, block_size, num_heads, head_dim]`` with K and V kept as two
tensors, as in the Model Runner V2 notes, section 4.1), 16 tokens per block
("vLLM-Ascend 原理", section 2.1).

Shapes and distributions of the five named workloads:

* ``tiny``            B=4, lens {1,17,33,100}, 4/4 heads, D=64, fp16, pool of 64
                      blocks, tables = first 13 entries of a seeded permutation.
* ``llama7b_decode``  B=64, lens U[512,4096], 32/32 heads, D=128, fp16, pool
                      = ceil(1.1 x blocks in use), blocks scattered at random.
* ``llama7b_ctx4096`` same, every length 4096 (the B=64, 4K-context point).
* ``gqa_prefix``      B=256, lens lognormal(mu=ln 1024, sigma=1) clipped to
                      [128, 8192], 32/8 heads, bf16; groups of 16 sequences
                      share the physical blocks of their first 1024 tokens
                      (full blocks strictly before the newest token's block).
* ``long_context``    B=8, lens U[32768,131072], 64/8 heads, bf16.
* ``mixed``           token budget 8192: 4 chunks of 1536 new tokens on cached
                      prefixes U[0,4096] + 2048 decodes at ctx U[256,4096];
                      32/8 heads, bf16; prefill sequences placed at seeded
                      random batch positions.
* ``spec_verify``     B=64 speculative-decoding verify rows: the last accepted
                      token + 3 drafts (q_len 4) on cached contexts
                      U[512,4096]; 32/8 heads, bf16.

q, k and v are N(0,1) in fp32 rounded to the storage dtype.  Seeds are
``20261202 + config index``.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np
import torch

BLOCK_SIZE = 16
BASE_SEED = 20261202

_TORCH_DTYPES = {"f16": torch.float16, "bf16": torch.bfloat16}


def torch_dtype(name: str) -> torch.dtype:
    return _TORCH_DTYPES[name]


@dataclass
class Workload:
    """One step of paged attention over a block pool.

    ``seq_lens[b]`` counts every token of sequence ``b`` including the
    ``q_lens[b]`` tokens that arrive this step (their k/v are in ``key`` and
    ``value`` and still have to be written into the pool).  Query and new-token
    rows are packed sequence after sequence: sequence ``b`` owns rows
    ``cu_q_lens[b] : cu_q_lens[b+1]``.
    """

    name: str
    dtype: str
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    block_size: int
    seq_lens: np.ndarray          # int32 [B]
    q_lens: np.ndarray            # int32 [B]
    block_tables: np.ndarray      # int32 [B, max_blocks_per_seq]
    num_blocks: int
    scale: float
    q: torch.Tensor               # [T, Hq, D]
    key: torch.Tensor             # [T, Hkv, D]
    value: torch.Tensor           # [T, Hkv, D]
    k_cache: torch.Tensor         # [NB, bs, Hkv, D]
    v_cache: torch.Tensor         # [NB, bs, Hkv, D]
    seed: int = 0
    meta: dict = field(default_factory=dict)

    @property
    def batch(self) -> int:
        return int(self.seq_lens.shape[0])

    @property
    def num_tokens(self) -> int:
        return int(self.q_lens.sum())

    @property
    def cu_q_lens(self) -> np.ndarray:
        cu = np.zeros(self.batch + 1, dtype=np.int32)
        np.cumsum(self.q_lens, out=cu[1:])
        return cu

    @property
    def max_blocks_per_seq(self) -> int:
        return int(self.block_tables.shape[1])

    @property
    def max_seq_len(self) -> int:
        return int(self.seq_lens.max()) if self.batch else 0

    @property
    def max_q_len(self) -> int:
        return int(self.q_lens.max()) if self.batch else 0

    @property
    def is_decode(self) -> bool:
        return bool(np.all(self.q_lens == 1))

    @property
    def cache_elem_bytes(self) -> int:
        return 1 if self.meta.get("cache_dtype") == "fp8" else 2

    def kv_bytes_logical(self) -> int:
        """K+V bytes that attention reads if every sequence's blocks are distinct."""
        return (int(self.seq_lens.astype(np.int64).sum()) * 2 * self.num_kv_heads * self.head_dim
                * self.cache_elem_bytes)

    def used_blocks(self) -> np.ndarray:
        """Sorted distinct physical block ids referenced by the live part of the tables."""
        nb = -(-self.seq_lens.astype(np.int64) // self.block_size)
        ids = [self.block_tables[b, : nb[b]] for b in range(self.batch)]
        return np.unique(np.concatenate(ids)) if ids else np.zeros(0, np.int32)


def _blocks_for(n: np.ndarray, bs: int) -> np.ndarray:
    return (-(-n.astype(np.int64) // bs)).astype(np.int64)


def _fill_normal(t: torch.Tensor, gen: torch.Generator, chunk_elems: int = 1 << 26, scale: float = 1.0) -> None:
    """Fill ``t`` (any float dtype) with N(0, scale^2) drawn in fp32, in chunks of dim-0 rows."""
    flat = t.view(t.shape[0], -1)
    chunk_rows = max(1, chunk_elems // max(1, flat.shape[1]))
    for r0 in range(0, flat.shape[0], chunk_rows):
        r1 = min(flat.shape[0], r0 + chunk_rows)
        tmp = torch.randn((r1 - r0, flat.shape[1]), generator=gen, device=t.device, dtype=torch.float32)
        if scale != 1.0:
            tmp.mul_(scale)
        flat[r0:r1].copy_(tmp)


def build_workload(
    *,
    name: str,
    seq_lens,
    q_lens,
    num_q_heads: int,
    num_kv_heads: int,
    head_dim: int,
    dtype: str,
    seed: int,
    num_blocks: int | None = None,
    pool_slack: float = 0.10,
    share_groups: int = 0,
    share_tokens: int = 0,
    device: str | torch.device = "cpu",
    poison: bool = False,
    table_pad: str = "random",
    scale: float | None = None,
    block_size: int = BLOCK_SIZE,
    materialize: bool = True,
    cache_dtype: str = "same",
    kv_scale: float = 1.0 / 16,
) -> Workload:
    """Build a seeded workload.

    share_groups / share_tokens: consecutive groups of ``share_groups``
    sequences point their first full blocks (up to ``share_tokens`` tokens, and
    only blocks strictly before the block that holds each sequence's first new
    token) at one common set of physical blocks, as a prefix cache would.

    poison: fill every pool position that no live table entry covers, and every
    position at or after a sequence's first new token, with NaN before the
    step's write.  A correct write fills the new-token slots; a correct
    attention never reads the rest.

    table_pad: what the unused tail of each block-table row holds:
    ``"random"`` (valid but wrong block ids), ``"zero"`` or ``"garbage"``
    (ids outside the pool, including negative ones).

    materialize: False builds the integer tables only (tensors are None).

    cache_dtype: "same" (the pools hold ``dtype``) or "fp8": the pools are
    head-major [NB, Hkv, bs, D] and hold
    E4M3 codes (uint8) of N(0, 1) / kv_scale values drawn in fp32 and
    converted by torch, so that code * kv_scale is about N(0, 1); the new
    key/value rows stay in ``dtype`` (they are quantised by the write).
    """
    rng = np.random.Generator(np.random.PCG64(seed))
    seq_lens = np.asarray(seq_lens, dtype=np.int32).reshape(-1)
    q_lens = np.asarray(q_lens, dtype=np.int32).reshape(-1)
    if q_lens.size == 1 and seq_lens.size != 1:
        q_lens = np.full_like(seq_lens, int(q_lens[0]))
    B = seq_lens.size
    assert q_lens.size == B
    assert np.all(q_lens >= 0) and np.all(q_lens <= seq_lens)
    assert num_q_heads % num_kv_heads == 0
    bs = block_size
    nblk = _blocks_for(seq_lens, bs)

    # prefix sharing: number of shared leading blocks per sequence
    shared = np.zeros(B, dtype=np.int64)
    if share_groups > 1 and share_tokens > 0:
        cap = share_tokens // bs
        first_new = (seq_lens.astype(np.int64) - q_lens.astype(np.int64))
        # blocks strictly before the block holding the first new token are full
        before = np.where(first_new > 0, first_new // bs, 0)
        shared = np.minimum(cap, before)
    n_groups = (B + share_groups - 1) // share_groups if share_groups > 1 else 0
    group_blocks = int(share_tokens // bs) if n_groups else 0
    private = nblk - shared
    needed = int(private.sum()) + n_groups * group_blocks
    if num_blocks is None:
        num_blocks = max(1, int(math.ceil(needed * (1.0 + pool_slack))))
    assert num_blocks >= needed, (num_blocks, needed)

    perm = rng.permutation(num_blocks).astype(np.int32)
    cursor = 0
    group_ids = []
    for _ in range(n_groups):
        group_ids.append(perm[cursor: cursor + group_blocks])
        cursor += group_blocks
    max_blocks = int(max(1, nblk.max() if B else 1))
    tables = np.zeros((B, max_blocks), dtype=np.int32)
    for b in range(B):
        row = []
        if shared[b]:
            row.extend(group_ids[b // share_groups][: shared[b]].tolist())
        k = int(private[b])
        row.extend(perm[cursor: cursor + k].tolist())
        cursor += k
        tables[b, : len(row)] = row
        pad = max_blocks - len(row)
        if pad:
            if table_pad == "random":
                tables[b, len(row):] = rng.integers(0, num_blocks, size=pad, dtype=np.int32)
            elif table_pad == "garbage":
                tables[b, len(row):] = rng.integers(-(1 << 30), 1 << 30, size=pad, dtype=np.int32)
            else:
                tables[b, len(row):] = 0

    if scale is None:
        scale = 1.0 / math.sqrt(head_dim)
    meta = {"shared_blocks": shared.astype(np.int32)}
    if not materialize:
        return Workload(
            name=name, dtype=dtype, num_q_heads=num_q_heads, num_kv_heads=num_kv_heads,
            head_dim=head_dim, block_size=bs, seq_lens=seq_lens, q_lens=q_lens,
            block_tables=tables, num_blocks=int(num_blocks), scale=float(scale),
            q=None, key=None, value=None, k_cache=None, v_cache=None, seed=seed, meta=meta)
    tdt = torch_dtype(dtype)
    dev = torch.device(device)
    gen = torch.Generator(device=dev)
    gen.manual_seed(seed)
    T = int(q_lens.sum())
    q = torch.empty((T, num_q_heads, head_dim), dtype=tdt, device=dev)
    key = torch.empty((T, num_kv_heads, head_dim), dtype=tdt, device=dev)
    value = torch.empty((T, num_kv_heads, head_dim), dtype=tdt, device=dev)
    fp8 = cache_dtype == "fp8"
    cdt = torch.float8_e4m3fn if fp8 else tdt
    # FP8 pools are head-major [NB, Hkv, bs, D]; 16-bit pools [NB, bs, Hkv, D]
    shape = (num_blocks, num_kv_heads, bs, head_dim) if fp8 else (num_blocks, bs, num_kv_heads, head_dim)
    k_cache = torch.empty(shape, dtype=cdt, device=dev)
    v_cache = torch.empty(shape, dtype=cdt, device=dev)
    for t in (q, key, value):
        if t.numel():
            _fill_normal(t, gen)
    for t in (k_cache, v_cache):
        if t.numel():
            _fill_normal(t, gen, scale=1.0 / kv_scale if fp8 else 1.0)
    if fp8:
        k_cache = k_cache.view(torch.uint8)
        v_cache = v_cache.view(torch.uint8)

    if poison:
        live = np.zeros((num_blocks, bs), dtype=bool)
        for b in range(B):
            first_new = int(seq_lens[b] - q_lens[b])
            for j in range(int(nblk[b])):
                lo = j * bs
                n_ok = max(0, min(bs, first_new - lo))
                live[tables[b, j], :n_ok] = True
        dead = torch.from_numpy(~live).to(dev)
        nan = torch.tensor(0x7F if fp8 else float("nan"), dtype=k_cache.dtype, device=dev)
        mask = dead[:, None, :, None] if fp8 else dead[:, :, None, None]
        k_cache.masked_fill_(mask, nan)
        v_cache.masked_fill_(mask, nan)
    if fp8:
        meta["kv_scale"] = float(kv_scale)
        meta["cache_dtype"] = "fp8"

    return Workload(
        name=name, dtype=dtype, num_q_heads=num_q_heads, num_kv_heads=num_kv_heads,
        head_dim=head_dim, block_size=bs, seq_lens=seq_lens, q_lens=q_lens,
        block_tables=tables, num_blocks=int(num_blocks), scale=float(scale),
        q=q, key=key, value=value, k_cache=k_cache, v_cache=v_cache, seed=seed, meta=meta,
    )


# ---------------------------------------------------------------------------
# the named workloads
# ---------------------------------------------------------------------------

CONFIG_NAMES = ("tiny", "llama7b_decode", "gqa_prefix", "long_context", "mixed", "llama7b_ctx4096",
                "llama7b_decode_fp8", "spec_verify")


def _seed(idx: int) -> int:
    return BASE_SEED + idx


def config_tiny(device="cpu", poison=False, **kw) -> Workload:
    seed = _seed(0)
    rng = np.random.Generator(np.random.PCG64(seed))
    lens = np.array([1, 17, 33, 100], dtype=np.int32)
    nb = _blocks_for(lens, BLOCK_SIZE)                     # 1, 2, 3, 7 -> 13 blocks
    perm = rng.permutation(64).astype(np.int32)[: int(nb.sum())]
    w = build_workload(name="tiny", seq_lens=lens, q_lens=1, num_q_heads=4, num_kv_heads=4,
                       head_dim=64, dtype="f16", seed=seed, num_blocks=64, device=device,
                       poison=poison, **kw)
    # the tiny case fixes its tables as consecutive entries of one permutation
    tables = np.zeros_like(w.block_tables)
    c = 0
    for b in range(4):
        tables[b, : nb[b]] = perm[c: c + nb[b]]
        c += int(nb[b])
    w.block_tables = tables
    if poison:   # re-poison against the fixed tables
        return _repoison(w)
    return w


def _repoison(w: Workload) -> Workload:
    bs = w.block_size
    live = np.zeros((w.num_blocks, bs), dtype=bool)
    nblk = _blocks_for(w.seq_lens, bs)
    for b in range(w.batch):
        first_new = int(w.seq_lens[b] - w.q_lens[b])
        for j in range(int(nblk[b])):
            n_ok = max(0, min(bs, first_new - j * bs))
            live[w.block_tables[b, j], :n_ok] = True
    dev = w.k_cache.device
    gen = torch.Generator(device=dev)
    gen.manual_seed(w.seed + 7)
    _fill_normal(w.k_cache, gen)
    _fill_normal(w.v_cache, gen)
    dead = torch.from_numpy(~live).to(dev)
    nan = torch.tensor(float("nan"), dtype=w.k_cache.dtype, device=dev)
    w.k_cache.masked_fill_(dead[:, :, None, None], nan)
    w.v_cache.masked_fill_(dead[:, :, None, None], nan)
    return w


def config_llama7b_decode(device="cpu", batch=64, lo=512, hi=4096, **kw) -> Workload:
    seed = _seed(1)
    rng = np.random.Generator(np.random.PCG64(seed))
    lens = rng.integers(lo, hi + 1, size=batch).astype(np.int32)
    return build_workload(name="llama7b_decode", seq_lens=lens, q_lens=1, num_q_heads=32,
                          num_kv_heads=32, head_dim=128, dtype="f16", seed=seed + 1000,
                          device=device, **kw)


def config_llama7b_ctx4096(device="cpu", batch=64, **kw) -> Workload:
    seed = _seed(5)
    lens = np.full(batch, 4096, dtype=np.int32)
    return build_workload(name="llama7b_ctx4096", seq_lens=lens, q_lens=1, num_q_heads=32,
                          num_kv_heads=32, head_dim=128, dtype="f16", seed=seed + 1000,
                          device=device, **kw)


def config_gqa_prefix(device="cpu", batch=256, **kw) -> Workload:
    seed = _seed(2)
    rng = np.random.Generator(np.random.PCG64(seed))
    raw = rng.lognormal(mean=math.log(1024.0), sigma=1.0, size=batch)
    lens = np.clip(np.rint(raw), 128, 8192).astype(np.int32)
    return build_workload(name="gqa_prefix", seq_lens=lens, q_lens=1, num_q_heads=32,
                          num_kv_heads=8, head_dim=128, dtype="bf16", seed=seed + 1000,
                          share_groups=16, share_tokens=1024, device=device, **kw)


def config_long_context(device="cpu", batch=8, lo=32768, hi=131072, **kw) -> Workload:
    seed = _seed(3)
    rng = np.random.Generator(np.random.PCG64(seed))
    lens = rng.integers(lo, hi + 1, size=batch).astype(np.int32)
    return build_workload(name="long_context", seq_lens=lens, q_lens=1, num_q_heads=64,
                          num_kv_heads=8, head_dim=128, dtype="bf16", seed=seed + 1000,
                          device=device, **kw)


def config_mixed(device="cpu", n_prefill=4, chunk=1536, n_decode=2048,
                 prefix_hi=4096, dec_lo=256, dec_hi=4096, **kw) -> Workload:
    seed = _seed(4)
    rng = np.random.Generator(np.random.PCG64(seed))
    prefixes = rng.integers(0, prefix_hi + 1, size=n_prefill)
    dec_lens = rng.integers(dec_lo, dec_hi + 1, size=n_decode)
    B = n_prefill + n_decode
    where = np.sort(rng.choice(B, size=n_prefill, replace=False))
    seq_lens = np.empty(B, dtype=np.int32)
    q_lens = np.ones(B, dtype=np.int32)
    is_pre = np.zeros(B, dtype=bool)
    is_pre[where] = True
    seq_lens[is_pre] = prefixes + chunk
    q_lens[is_pre] = chunk
    seq_lens[~is_pre] = dec_lens
    return build_workload(name="mixed", seq_lens=seq_lens, q_lens=q_lens, num_q_heads=32,
                          num_kv_heads=8, head_dim=128, dtype="bf16", seed=seed + 1000,
                          device=device, **kw)


def config_prefill(device="cpu", n_prefill=16, chunk=1536, prefix_hi=4096, **kw) -> Workload:
    """Chunked prefill on its own: ``n_prefill`` chunks of ``chunk`` tokens on
    cached prefixes U[0, prefix_hi] (the mixed step's chunk length and prefix
    distribution; its first four prefixes are the mixed step's), no decode
    rows.  16 chunks read about 0.24 GB of cache per step, more than L2."""
    w = config_mixed(device=device, n_prefill=n_prefill, chunk=chunk, n_decode=0, prefix_hi=prefix_hi, **kw)
    w.name = "prefill"
    return w


def config_llama7b_decode_fp8(device="cpu", batch=64, lo=512, hi=4096, **kw) -> Workload:
    """The LLaMA-2-7B-shaped decode workload with an FP8 (E4M3) cache."""
    seed = _seed(1)
    rng = np.random.Generator(np.random.PCG64(seed))
    lens = rng.integers(lo, hi + 1, size=batch).astype(np.int32)
    return build_workload(name="llama7b_decode_fp8", seq_lens=lens, q_lens=1, num_q_heads=32,
                          num_kv_heads=32, head_dim=128, dtype="f16", seed=seed + 1000,
                          device=device, cache_dtype="fp8", **kw)


def config_mixed_fp8(device="cpu", **kw) -> Workload:
    """The continuous-batching step (``mixed``) with an FP8 (E4M3) cache: the
    same lengths and chunks, pools of E4M3 codes of N(0, 1) values (scale 1/16)."""
    w = config_mixed(device=device, cache_dtype="fp8", **kw)
    w.name = "mixed_fp8"
    return w


def config_prefill_fp8(device="cpu", **kw) -> Workload:
    """Chunked prefill on its own (``prefill``) over an FP8 (E4M3) cache."""
    w = config_prefill(device=device, cache_dtype="fp8", **kw)
    w.name = "prefill_fp8"
    return w


def config_spec_verify(device="cpu", batch=64, drafts=3, lo=512, hi=4096, **kw) -> Workload:
    """Speculative-decoding verify step: each sequence appends its last
    accepted token and `drafts` draft tokens (q_len = drafts + 1) onto a cached
    context of U[lo, hi] tokens; 32/8 heads, bf16."""
    seed = _seed(6)
    rng = np.random.Generator(np.random.PCG64(seed))
    ctx = rng.integers(lo, hi + 1, size=batch).astype(np.int32)
    q = drafts + 1
    return build_workload(name="spec_verify", seq_lens=ctx + q, q_lens=q, num_q_heads=32,
                          num_kv_heads=8, head_dim=128, dtype="bf16", seed=seed + 1000,
                          device=device, **kw)


CONFIGS = {
    "tiny": config_tiny,
    "llama7b_decode": config_llama7b_decode,
    "gqa_prefix": config_gqa_prefix,
    "long_context": config_long_context,
    "mixed": config_mixed,
    "llama7b_ctx4096": config_llama7b_ctx4096,
    "llama7b_decode_fp8": config_llama7b_decode_fp8,
    "spec_verify": config_spec_verify,
    "prefill": config_prefill,
    "mixed_fp8": config_mixed_fp8,
    "prefill_fp8": config_prefill_fp8,
}


def make(name: str, **kw) -> Workload:
    return CONFIGS[name](**kw)
