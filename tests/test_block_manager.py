"""Host block manager (C++, in libpagedattn.so) against a worked example
derived by hand from the pages' rules, against the plain reference model in
oracle/block_model.py on random operation sequences, and end to end through
the fp64 attention oracle (prefix sharing must not change any output)."""
import numpy as np
import pytest

import oracle
from oracle import block_model as M
import paged_kv_attention_decode_gb300 as pa

bm_mod = pytest.importorskip("paged_kv_attention_decode_gb300.block_manager")


class Lib:
    """The C++ manager behind the model's call convention (status, value)."""

    def __init__(self, num_blocks, bs, caching=True):
        self.m = pa.BlockManager(num_blocks, bs, caching)

    def _run(self, fn, *a):
        try:
            return M.OK, fn(*a)
        except pa.BlockManagerError as e:
            return e.status, None

    def add_sequence(self, sid, prompt, extra=0):
        return self._run(self.m.add_sequence, sid, prompt, extra)

    def append_tokens(self, sid, toks):
        return self._run(self.m.append_tokens, sid, toks)[0]

    def allocate_slots(self, sid, n):
        return self._run(self.m.allocate_slots, sid, n)

    def truncate(self, sid, n):
        return self._run(self.m.truncate, sid, n)[0]

    def fork(self, a, b):
        return self._run(self.m.fork, a, b)[0]

    def free_sequence(self, sid):
        return self._run(self.m.free_sequence, sid)[0]

    def num_free_blocks(self):
        return self.m.num_free_blocks

    def seq_len(self, sid):
        return self.m.seq_len(sid)

    def block_table(self, sid):
        return self.m.block_table(sid).tolist()

    def block_ref(self, b):
        return self.m.block_ref(b)

    def block_cached(self, b):
        return self.m.block_cached(b)


IMPLS = {"library": Lib, "model": M.BlockModel}


@pytest.mark.parametrize("impl", sorted(IMPLS))
def test_worked_example(impl):
    """Pool of 8 blocks of 4 tokens.  Each expectation follows from the rules
    by hand: head-out / tail-in free list, keys on full blocks chained through
    the previous block, counts, copy-on-write of a shared partial block,
    truncation, and freed blocks keeping their keys until handed out."""
    m = IMPLS[impl](8, 4)
    P = list(range(10))
    assert m.add_sequence(1, P) == (M.OK, 0)                      # empty cache
    assert m.allocate_slots(1, 10) == (M.OK, None)                # blocks 0,1,2; keys on 0 and 1
    assert m.block_table(1) == [0, 1, 2] and m.num_free_blocks() == 5
    assert [m.block_cached(b) for b in range(3)] == [True, True, False]
    # same first 8 tokens: both full blocks are shared
    assert m.add_sequence(2, list(range(8)) + [50, 51, 52]) == (M.OK, 8)
    assert [m.block_ref(b) for b in (0, 1)] == [2, 2]
    assert m.allocate_slots(2, 3) == (M.OK, None)                 # block 3
    assert m.block_table(2) == [0, 1, 3]
    # another extra key (model, adapter or salt): no sharing
    assert m.add_sequence(3, P, 7) == (M.OK, 0)
    assert m.allocate_slots(3, 10) == (M.OK, None)                # blocks 4,5,6
    assert m.block_table(3) == [4, 5, 6] and m.num_free_blocks() == 1
    # a pool too short: nothing changes
    assert m.add_sequence(4, list(range(100, 108))) == (M.OK, 0)
    assert m.allocate_slots(4, 8)[0] == M.NO_SPACE
    assert m.num_free_blocks() == 1 and m.seq_len(4) == 0
    # free sequence 1 (last block first): block 2 returns; 0 and 1 stay with 2
    assert m.free_sequence(1) == M.OK
    assert m.num_free_blocks() == 2 and [m.block_ref(b) for b in (0, 1, 2)] == [1, 1, 0]
    assert m.allocate_slots(4, 8) == (M.OK, None)                 # blocks 7, then 2
    assert m.block_table(4) == [7, 2]
    # free sequence 3: blocks 6, 5, 4 return; 5 and 4 keep their keys
    assert m.free_sequence(3) == M.OK
    assert [m.block_cached(b) for b in (4, 5, 6)] == [True, True, False]
    # the same prompt and extra key as sequence 3 revives blocks 4 and 5
    assert m.add_sequence(5, P, 7) == (M.OK, 8)
    assert m.block_table(5) == [4, 5] and m.num_free_blocks() == 1
    assert m.allocate_slots(5, 2) == (M.OK, None)                 # block 6
    assert m.num_free_blocks() == 0
    # fork shares every block, the partial last one too
    assert m.fork(2, 6) == M.OK
    assert [m.block_ref(b) for b in (0, 1, 3)] == [2, 2, 2]
    assert m.append_tokens(6, [60]) == M.OK
    assert m.allocate_slots(6, 1)[0] == M.NO_SPACE                # the copy needs a block
    assert m.free_sequence(4) == M.OK                             # blocks 2, 7 return (cached)
    # copy-on-write: block 2 (its key evicted) receives block 3's bytes
    assert m.allocate_slots(6, 1) == (M.OK, (3, 2))
    assert m.block_table(6) == [0, 1, 2] and m.block_ref(3) == 1 and m.block_cached(2)
    # rollback of a draft: the partial block is written again, so its key goes
    assert m.truncate(6, 9) == M.OK
    assert m.seq_len(6) == 9 and m.block_table(6) == [0, 1, 2] and not m.block_cached(2)
    assert m.truncate(2, 4) == M.OK                               # releases blocks 3, then 1
    assert m.block_table(2) == [0] and [m.block_ref(b) for b in (0, 1, 3)] == [2, 1, 0]
    # block 7 still holds the key of tokens 100..103
    assert m.add_sequence(7, [100, 101, 102, 103, 104]) == (M.OK, 4)
    assert m.block_table(7) == [7] and m.num_free_blocks() == 1
    assert [m.block_ref(b) for b in range(8)] == [2, 1, 1, 0, 1, 1, 1, 1]
    assert [m.block_cached(b) for b in range(8)] == [True, True, False, False, True, True, False, True]
    assert [m.seq_len(s) for s in (2, 5, 6, 7)] == [4, 10, 9, 4]


def test_without_prefix_caching_nothing_is_shared():
    for m in (Lib(8, 4, caching=False), M.BlockModel(8, 4, prefix_caching=False)):
        assert m.add_sequence(1, list(range(10))) == (M.OK, 0)
        assert m.allocate_slots(1, 10) == (M.OK, None)
        assert m.add_sequence(2, list(range(10))) == (M.OK, 0)
        assert m.allocate_slots(2, 10) == (M.OK, None)
        assert m.block_table(2) == [3, 4, 5]
        assert not any(m.block_cached(b) for b in range(8))


def _check_invariants(m, live, nblocks):
    held = [0] * nblocks
    for s in live:
        t = m.block_table(s)
        assert len(t) == -(-m.seq_len(s) // m_bs(m))
        for b in t:
            held[b] += 1
    assert [m.block_ref(b) for b in range(nblocks)] == held
    assert m.num_free_blocks() == held.count(0)


def m_bs(m):
    return m.m.block_size if isinstance(m, Lib) else m.bs


@pytest.mark.parametrize("seed,nblocks,bs", [(1, 24, 4), (2, 64, 16), (3, 12, 2), (4, 40, 4), (5, 200, 16)])
def test_random_operations_match_the_model(seed, nblocks, bs):
    rng = np.random.default_rng(seed)
    lib, ref = Lib(nblocks, bs), M.BlockModel(nblocks, bs)
    systems = [list(rng.integers(0, 50, size=int(rng.integers(1, 4 * bs)))) for _ in range(3)]
    live, next_id = [], 1
    for step in range(1500):
        op = rng.choice(["add", "grow", "grow", "grow", "truncate", "fork", "free"])
        if op == "add" or not live:
            prompt = list(systems[rng.integers(0, 3)]) + list(rng.integers(0, 50, size=int(rng.integers(0, 3 * bs))))
            extra = int(rng.integers(0, 2))
            a, b = lib.add_sequence(next_id, prompt, extra), ref.add_sequence(next_id, prompt, extra)
            assert a == b, (step, a, b)
            # the prompt's uncached part gets its slots now (or the sequence waits)
            rest = len(prompt) - a[1]
            ra, rb = lib.allocate_slots(next_id, rest), ref.allocate_slots(next_id, rest)
            assert ra == rb, (step, ra, rb)
            if ra[0] == M.NO_SPACE:
                # not admitted: its shared prefix blocks are released again
                assert lib.free_sequence(next_id) == ref.free_sequence(next_id) == M.OK
            else:
                live.append(next_id)
            next_id += 1
        else:
            s = live[int(rng.integers(0, len(live)))]
            if op == "grow":
                k = int(rng.integers(1, 7))
                toks = list(rng.integers(0, 50, size=k))
                known = len(ref.seqs[s]["tokens"]) - ref.seq_len(s)
                if known == 0:
                    assert lib.append_tokens(s, toks) == ref.append_tokens(s, toks) == M.OK
                    known = k
                n = min(known, k)
                ra, rb = lib.allocate_slots(s, n), ref.allocate_slots(s, n)
                assert ra == rb, (step, ra, rb)
                if ra[0] == M.NO_SPACE:
                    # preempt (recompute): the most recent other sequence gives its blocks back
                    victim = live[-1] if live[-1] != s else live[0]
                    if victim != s:
                        assert lib.free_sequence(victim) == ref.free_sequence(victim) == M.OK
                        live.remove(victim)
            elif op == "truncate":
                n = int(rng.integers(0, ref.seq_len(s) + 1))
                assert lib.truncate(s, n) == ref.truncate(s, n) == M.OK
            elif op == "fork":
                assert lib.fork(s, next_id) == ref.fork(s, next_id) == M.OK
                live.append(next_id)
                next_id += 1
            else:
                assert lib.free_sequence(s) == ref.free_sequence(s) == M.OK
                live.remove(s)
        assert lib.num_free_blocks() == ref.num_free_blocks()
        for s in live:
            assert lib.seq_len(s) == ref.seq_len(s)
            assert lib.block_table(s) == ref.block_table(s), (step, s)
        if step % 50 == 0:
            assert [lib.block_cached(b) for b in range(nblocks)] == [ref.block_cached(b) for b in range(nblocks)]
            _check_invariants(lib, live, nblocks)
            _check_invariants(ref, live, nblocks)


def test_bad_arguments_change_nothing():
    m = pa.BlockManager(4, 16)
    m.add_sequence(1, [1, 2, 3])
    for call in (lambda: m.add_sequence(1, [5]),           # duplicate id
                 lambda: m.allocate_slots(2, 1),           # unknown id
                 lambda: m.allocate_slots(1, 4),           # more tokens than known
                 lambda: m.truncate(1, 1),                 # longer than the length (0)
                 lambda: m.fork(1, 1),
                 lambda: m.fork(9, 3),
                 lambda: m.free_sequence(9)):
        with pytest.raises(pa.BlockManagerError) as e:
            call()
        assert e.value.status == M.INVALID_ARG
    assert m.num_free_blocks == 4 and m.seq_len(1) == 0
    with pytest.raises(pa.BlockManagerError):
        pa.BlockManager(0, 16)
    with pytest.raises(pa.BlockManagerError):
        pa.BlockManager(8, 0)
    m.allocate_slots(1, 3)
    with pytest.raises(pa.BlockManagerError) as e:
        m.build_step([1], [4], 4)                          # q_len above the length
    assert e.value.status == M.INVALID_ARG
    with pytest.raises(pa.BlockManagerError) as e:
        m.build_step([1], [1], 0)
    assert e.value.status == M.INVALID_ARG


def test_build_step_matches_the_oracle_slot_mapping():
    rng = np.random.default_rng(9)
    m = pa.BlockManager(300, 16)
    ids, qlens = [], []
    for s in range(12):
        prompt = list(rng.integers(0, 1000, size=int(rng.integers(1, 200))))
        cached = m.add_sequence(s, prompt)
        m.allocate_slots(s, len(prompt) - cached)
        ids.append(s)
        qlens.append(int(rng.integers(1, len(prompt) - cached + 1)))
    tables, lens, cu, slots = m.build_step(ids, qlens, 16)
    assert np.array_equal(cu, np.concatenate([[0], np.cumsum(qlens)]))
    assert np.array_equal(lens, [m.seq_len(s) for s in ids])
    ref = oracle.slot_mapping(tables, lens, np.asarray(qlens, np.int32), 16, 300)
    assert np.array_equal(slots, ref)
    for i, s in enumerate(ids):
        t = m.block_table(s)
        assert np.array_equal(tables[i, : len(t)], t) and np.all(tables[i, len(t):] == -1)
    with pytest.raises(pa.BlockManagerError) as e:
        m.build_step(ids, qlens, 2)                         # tables wider than 2 blocks
    assert e.value.status == M.CAPACITY


# ---------------------------------------------------------------------------
# end to end on the CPU: KV content is a function of (token, position), as a
# model's would be, so a shared prefix block must hold exactly what the
# sequence would have written itself
# ---------------------------------------------------------------------------

def _kv_rows(tokens, positions, H, D, which):
    g = np.random.default_rng(1000 + which)
    emb = g.standard_normal((64, H, D), dtype=np.float32)
    pos = g.standard_normal((4096, H, D), dtype=np.float32) * 0.5
    x = emb[np.asarray(tokens) % 64] + pos[np.asarray(positions)]
    return x.astype(np.float16).view(np.uint16)


def _serve(caching, steps=6, H=2, D=64):
    """A few continuous-batching steps driven by the manager: prompts (two
    share a 40-token system prompt), decodes, a 3-token verify chunk, a fork
    (copy-on-write of its partial block) and a rollback.  Returns
    {(step, seq, position): fp64 attention row} and the free block count."""
    rng = np.random.default_rng(4)
    nb = 64
    m = pa.BlockManager(nb, 16, caching)
    kc = np.zeros((nb, 16, H, D), np.uint16)
    vc = np.zeros_like(kc)
    qtab = rng.standard_normal((64, 2 * H, D), dtype=np.float32).astype(np.float16).view(np.uint16)
    system = [int(x) for x in rng.integers(0, 64, size=40)]
    prompts = {1: system + [5, 6, 7], 2: system + [9] * 20, 3: [int(x) for x in rng.integers(0, 64, size=30)]}
    tokens = {}          # the test's own record of every sequence's tokens
    rows = {}
    for step in range(steps):
        batch, qlens = [], []

        def admit(sid):
            tokens[sid] = list(prompts[sid])
            cached = m.add_sequence(sid, prompts[sid])
            n = len(prompts[sid]) - cached
            assert m.allocate_slots(sid, n) is None
            batch.append(sid)
            qlens.append(n)

        if step == 0:
            admit(1)
            admit(3)
        if step == 1:
            admit(2)
        if step == 3:
            m.fork(1, 4)
            tokens[4] = list(tokens[1])
        if step == 4:
            m.truncate(3, m.seq_len(3) - 2)                 # two rejected drafts
            del tokens[3][-2:]
        if step > 0:
            for sid in sorted(t for t in tokens if t not in batch):
                k = 3 if sid == 3 else 1                     # a 3-token verify chunk for sequence 3
                new = [int(x) for x in rng.integers(0, 64, size=k)]
                tokens[sid] += new
                m.append_tokens(sid, new)
                pair = m.allocate_slots(sid, k)
                if pair:
                    kc[pair[1]] = kc[pair[0]]
                    vc[pair[1]] = vc[pair[0]]
                batch.append(sid)
                qlens.append(k)
        tables, lens, cu, slots = m.build_step(batch, qlens, 16)
        toks, poss, keys = [], [], []
        for i, sid in enumerate(batch):
            assert lens[i] == len(tokens[sid])
            for pos in range(lens[i] - qlens[i], lens[i]):
                toks.append(tokens[sid][pos])
                poss.append(pos)
                keys.append((step, sid, pos))
        oracle.kv_write(_kv_rows(toks, poss, H, D, 0), _kv_rows(toks, poss, H, D, 1), kc, vc, slots)
        q = np.ascontiguousarray(qtab[np.asarray(toks) % 64])
        out = oracle.paged_attention_prefill(q, kc, vc, tables, lens, np.asarray(qlens, np.int32), 0.125, "f16")
        rows.update(zip(keys, out))
    return rows, m.num_free_blocks


def test_prefix_sharing_and_copy_on_write_do_not_change_any_output():
    shared, free_shared = _serve(True)
    private, free_private = _serve(False)
    assert free_shared > free_private                      # the system prompt's blocks are shared
    assert set(shared) < set(private)                      # cached prompt tokens are not recomputed
    for k, row in shared.items():
        assert np.array_equal(row, private[k]), k
