"""Plain Python model of the block manager (allocation, reference counts,
copy-on-write, radix prefix reuse).

TEST INFRASTRUCTURE ONLY: the tests use it to check the library's C++ block
manager; the product path never does.  It shares no code with the library.

What it models: the engine side of paged KV on the pages -- the inferd
README's block allocator and per-sequence page table (its "Paged KV" phase,
and "prefix-sharing via copy-on-write KV blocks" in its backlog) and the
lfm25-inference README's engine-managed KV pages with radix-tree prefix
caching, page size 16.  The pages name these parts but fix no policy; the
policies restated here, in the same order of steps as the library's header
states them, are:

* free blocks form a stack (initially 0 on top, then 1, 2, ...; a freed
  block goes on top);
* a block's reference count = the sequences whose table holds it + 1 if the
  radix tree holds it; count 0 = free;
* the tree maps a full block's 16 token ids, under the chain of blocks
  before it, to a block; a new sequence reuses the longest chain matching
  its prompt, leaving at least one prompt token to compute;
* with no free block, the least recently used tree leaf that only the tree
  holds is evicted (ties: lowest block id); matching or inserting an entry
  uses it;
* writing into a partially filled block another sequence also holds copies
  it first (copy-on-write);
* an operation that runs out of blocks gives back what it allocated and
  leaves the sequence as it was (evictions it made stay made).

Everything is a linear scan or a dict lookup: slow and plain on purpose.
"""

from __future__ import annotations

BS = 16
OK, INVALID, NO_BLOCKS, UNKNOWN_SEQ = 0, 1, 7, 8


class _Node:
    def __init__(self, parent, block, tick):
        self.parent = parent
        self.block = block
        self.last_access = tick
        self.children = {}          # tuple of 16 token ids -> _Node


class BlockManagerModel:
    def __init__(self, num_blocks: int):
        self.num_blocks = num_blocks
        self.free = list(range(num_blocks - 1, -1, -1))      # top of the stack = end of the list
        self.ref = [0] * num_blocks
        self.root = _Node(None, -1, 0)
        self.seqs = {}              # id -> {"tokens": [...], "blocks": [...]}
        self.tick = 0

    # ---------------------------------------------------------------- tree

    def _tree_nodes(self):
        out, todo = [], [self.root]
        while todo:
            n = todo.pop()
            for c in n.children.values():
                out.append(c)
                todo.append(c)
        return out

    def tree_blocks(self):
        return {n.block for n in self._tree_nodes()}

    def _evict_one(self) -> bool:
        cands = [n for n in self._tree_nodes() if not n.children and self.ref[n.block] == 1]
        if not cands:
            return False
        victim = min(cands, key=lambda n: (n.last_access, n.block))
        parent = victim.parent
        for k, v in list(parent.children.items()):
            if v is victim:
                del parent.children[k]
        self._decref(victim.block)
        return True

    # ---------------------------------------------------------------- blocks

    def _decref(self, b):
        self.ref[b] -= 1
        if self.ref[b] == 0:
            self.free.append(b)

    def _alloc(self):
        if not self.free and not self._evict_one():
            return -1
        b = self.free.pop()
        self.ref[b] = 1
        return b

    def _append(self, s, tokens):
        """-> (status, slots, copy pair or None)."""
        length, nb = len(s["tokens"]), len(s["blocks"])
        cow_src = cow_dst = -1
        if length % BS != 0 and self.ref[s["blocks"][-1]] > 1:
            cow_dst = self._alloc()
            if cow_dst < 0:
                return NO_BLOCKS, None, None
            cow_src = s["blocks"][-1]
        need = -(-(length + len(tokens)) // BS) - nb
        fresh = []
        for _ in range(need):
            b = self._alloc()
            if b < 0:
                for f in fresh:
                    self._decref(f)
                if cow_dst >= 0:
                    self._decref(cow_dst)
                return NO_BLOCKS, None, None
            fresh.append(b)
        copy = None
        if cow_dst >= 0:
            s["blocks"][-1] = cow_dst
            self._decref(cow_src)
            copy = (cow_src, cow_dst)
        s["blocks"].extend(fresh)
        slots = []
        for t in tokens:
            pos = len(s["tokens"])
            slots.append(s["blocks"][pos // BS] * BS + pos % BS)
            s["tokens"].append(int(t))
        return OK, slots, copy

    # ---------------------------------------------------------------- operations

    def add_sequence(self, seq, tokens):
        """-> (status, cached_tokens, slots)."""
        tokens = [int(t) for t in tokens]
        if not tokens:
            return INVALID, None, None
        if seq in self.seqs:
            return UNKNOWN_SEQ, None, None
        self.tick += 1
        s = {"tokens": [], "blocks": []}
        node = self.root
        for i in range((len(tokens) - 1) // BS):
            child = node.children.get(tuple(tokens[i * BS:(i + 1) * BS]))
            if child is None:
                break
            node = child
            node.last_access = self.tick
            self.ref[node.block] += 1
            s["blocks"].append(node.block)
            s["tokens"].extend(tokens[i * BS:(i + 1) * BS])
        cached = len(s["tokens"])
        st, slots, _ = self._append(s, tokens[cached:])
        if st != OK:
            for b in s["blocks"]:
                self._decref(b)
            return st, None, None
        self.seqs[seq] = s
        return OK, cached, slots

    def append(self, seq, tokens):
        """-> (status, slots, copy pair or None)."""
        if seq not in self.seqs:
            return UNKNOWN_SEQ, None, None
        self.tick += 1
        return self._append(self.seqs[seq], [int(t) for t in tokens])

    def commit(self, seq):
        if seq not in self.seqs:
            return UNKNOWN_SEQ
        self.tick += 1
        s = self.seqs[seq]
        in_tree = self.tree_blocks()
        node = self.root
        for i in range(len(s["tokens"]) // BS):
            key = tuple(s["tokens"][i * BS:(i + 1) * BS])
            child = node.children.get(key)
            if child is not None:
                if child.block != s["blocks"][i]:
                    break
                node = child
                node.last_access = self.tick
                continue
            if s["blocks"][i] in in_tree:
                break
            child = _Node(node, s["blocks"][i], self.tick)
            node.children[key] = child
            self.ref[child.block] += 1
            in_tree.add(child.block)
            node = child
        return OK

    def fork(self, parent, child):
        if parent not in self.seqs or child in self.seqs:
            return UNKNOWN_SEQ
        self.tick += 1
        p = self.seqs[parent]
        self.seqs[child] = {"tokens": list(p["tokens"]), "blocks": list(p["blocks"])}
        for b in p["blocks"]:
            self.ref[b] += 1
        return OK

    def release(self, seq):
        if seq not in self.seqs:
            return UNKNOWN_SEQ
        self.tick += 1
        for b in self.seqs.pop(seq)["blocks"]:
            self._decref(b)
        return OK

    def tables(self, seqs, max_blocks):
        rows, lens = [], []
        for q in seqs:
            s = self.seqs[q]
            rows.append(s["blocks"] + [-1] * (max_blocks - len(s["blocks"])))
            lens.append(len(s["tokens"]))
        return rows, lens

    def num_free(self):
        return len(self.free)

    def num_cached(self):
        return len(self._tree_nodes())
