"""Plain reference model of the host block manager (test infrastructure:
only tests/ use it; it shares nothing with the C++ in the package).

It restates, with Python lists and dicts, what the pages describe:

* a pool of blocks handed out from a free list and returned when a sequence
  ends ("vLLM 在 CANN 上的推理优化", "vLLM 的 PagedAttention 数据结构":
  free_blocks, allocate_slots; "vLLM-Ascend 原理", section 2.1);
* prefix caching ("vLLM学习整理", section 三 "Prefix Caching"): a block that
  fills up gets a key from its own tokens and the previous block's key (plus
  extra keys); equal keys share one physical block with a reference count;
  a block is released when its count reaches 0;
* copy-on-write before a shared block diverges ("vLLM-Ascend 原理", 2.1);
* truncation of a sequence by length for speculative-decoding rollback
  ("vLLM-Ascend 原理", section 4 "推测解码").

and the readings the library states where the pages leave a choice open:
a block's key is (registration id of the previous block's key, own tokens)
with the extra key on the first block, compared exactly, registration ids
never reused; blocks leave the free list at its head and return at its tail,
a sequence's blocks last block first; a freed block keeps its key until the
free list hands it out again; a prompt never matches the block that holds
its last token.
"""
from __future__ import annotations

OK, INVALID_ARG, NO_SPACE, CAPACITY = 0, 1, 5, 6


class BlockModel:
    def __init__(self, num_blocks: int, block_size: int, prefix_caching: bool = True):
        self.bs = block_size
        self.caching = prefix_caching
        self.free = list(range(num_blocks))     # index 0 is the head
        self.ref = [0] * num_blocks
        self.key = {}                            # block -> key it holds
        self.reg = {}                            # block -> registration id of that key
        self.holder = {}                         # key -> block
        self.next_reg = 1
        self.seqs = {}                           # seq id -> dict

    # -- helpers ------------------------------------------------------------
    def _key(self, s, j):
        parent = 0 if j == 0 else s["chain"][j - 1]
        extra = s["extra"] if j == 0 else 0
        return (parent, extra, tuple(s["tokens"][j * self.bs:(j + 1) * self.bs]))

    def _forget_key(self, b):
        if b in self.key:
            k = self.key.pop(b)
            self.reg.pop(b)
            if self.holder.get(k) == b:
                del self.holder[k]

    def _take_free(self):
        b = self.free.pop(0)
        self._forget_key(b)          # its old content is evicted
        self.ref[b] = 1
        return b

    def _release(self, b):
        self.ref[b] -= 1
        if self.ref[b] == 0:
            self.free.append(b)      # keeps its key until handed out again

    def _register_full(self, s):
        if not self.caching:
            return
        while len(s["chain"]) < s["len"] // self.bs:
            j = len(s["chain"])
            k = self._key(s, j)
            if k in self.holder:
                s["chain"].append(self.reg[self.holder[k]])
                continue
            b = s["blocks"][j]
            if b in self.key:
                s["chain"].append(self.next_reg)
                self.next_reg += 1
                continue
            self.key[b] = k
            self.reg[b] = self.next_reg
            self.holder[k] = b
            self.next_reg += 1
            s["chain"].append(self.reg[b])

    # -- operations (same names and results as the C ABI) --------------------
    def num_free_blocks(self):
        return len(self.free)

    def add_sequence(self, seq_id, prompt, extra_key=0):
        if seq_id in self.seqs:
            return INVALID_ARG, None
        s = {"extra": extra_key, "tokens": list(prompt), "blocks": [], "chain": [], "len": 0}
        if self.caching and len(prompt) > 0:
            for j in range((len(prompt) - 1) // self.bs):
                k = self._key(s, j)
                if k not in self.holder:
                    break
                b = self.holder[k]
                s["blocks"].append(b)
                s["chain"].append(self.reg[b])
        for b in s["blocks"]:
            if self.ref[b] == 0:
                self.free.remove(b)
            self.ref[b] += 1
        s["len"] = len(s["blocks"]) * self.bs
        self.seqs[seq_id] = s
        return OK, s["len"]

    def append_tokens(self, seq_id, tokens):
        if seq_id not in self.seqs:
            return INVALID_ARG
        self.seqs[seq_id]["tokens"].extend(tokens)
        return OK

    def allocate_slots(self, seq_id, num_new):
        if seq_id not in self.seqs or num_new < 0:
            return INVALID_ARG, None
        s = self.seqs[seq_id]
        new_len = s["len"] + num_new
        if new_len > len(s["tokens"]):
            return INVALID_ARG, None
        if num_new == 0:
            return OK, None
        want = -(-new_len // self.bs)
        cow = s["len"] % self.bs != 0 and self.ref[s["blocks"][-1]] > 1
        if want - len(s["blocks"]) + (1 if cow else 0) > len(self.free):
            return NO_SPACE, None
        pair = None
        if cow:
            old = s["blocks"][-1]
            fresh = self._take_free()
            self.ref[old] -= 1
            s["blocks"][-1] = fresh
            pair = (old, fresh)
        while len(s["blocks"]) < want:
            s["blocks"].append(self._take_free())
        s["len"] = new_len
        self._register_full(s)
        return OK, pair

    def truncate(self, seq_id, new_len):
        if seq_id not in self.seqs:
            return INVALID_ARG
        s = self.seqs[seq_id]
        if new_len < 0 or new_len > s["len"]:
            return INVALID_ARG
        keep = -(-new_len // self.bs)
        while len(s["blocks"]) > keep:
            self._release(s["blocks"].pop())
        if new_len % self.bs != 0 and self.ref[s["blocks"][-1]] == 1:
            self._forget_key(s["blocks"][-1])
        del s["chain"][new_len // self.bs:]
        del s["tokens"][new_len:]
        s["len"] = new_len
        return OK

    def fork(self, parent_id, child_id):
        if parent_id not in self.seqs or child_id in self.seqs or parent_id == child_id:
            return INVALID_ARG
        p = self.seqs[parent_id]
        c = {"extra": p["extra"], "tokens": list(p["tokens"]), "blocks": list(p["blocks"]),
             "chain": list(p["chain"]), "len": p["len"]}
        for b in c["blocks"]:
            self.ref[b] += 1
        self.seqs[child_id] = c
        return OK

    def free_sequence(self, seq_id):
        if seq_id not in self.seqs:
            return INVALID_ARG
        s = self.seqs.pop(seq_id)
        for b in reversed(s["blocks"]):
            self._release(b)
        return OK

    def seq_len(self, seq_id):
        return self.seqs[seq_id]["len"] if seq_id in self.seqs else -1

    def block_table(self, seq_id):
        return list(self.seqs[seq_id]["blocks"])

    def block_ref(self, b):
        return self.ref[b]

    def block_cached(self, b):
        return b in self.key
