"""Block manager of a paged KV cache: free pool, per-sequence block tables,
reference counts, copy-on-write, exhaustion.

TEST INFRASTRUCTURE ONLY (see the package docstring).

What the pages say, and what this model does with it:

* Physical blocks of a fixed number of token slots, each with a reference
  count starting at zero; a free pool of unused blocks; per sequence a table
  from logical block index to physical block id, grown by taking a block from
  the free pool, whose reference count goes up by one.  An empty pool is an
  error that the caller answers by preempting a request.  [FN] "Paged KV-Cache
  with Radix Tree Prefix Cache" (the paged scheduler: physical block, block
  table, slot allocation) and [SC] "9. Failure modes and limitations", item 2
  (preemption when memory is exhausted).
* Memory is taken on demand, one block at a time, so a sequence never holds
  more than ceil(tokens / block_size) blocks.  [SC] "PagedAttention & Memory
  Management (vLLM)".
* Requests that share a prompt reference the same physical blocks through
  copy-on-write pointers.  [FN] "Paged KV-Cache with Radix Tree Prefix
  Cache"; [SC] "14. ... GPU VRAM & PagedAttention KV Cache Simulator"
  (copy-on-write prefix caching).

Readings where the pages leave a step open (also listed in the design notes):

1. The free pool is a stack: the block taken is the one on top, i.e. the last
   one pushed; the pool starts as blocks 0, 1, ..., N-1 pushed in that order
   (so block N-1 is taken first).  The allocation listing of [FN] takes the
   last element of a Python list, which is this order.
2. Freeing a sequence drops one reference from each block of its table in
   table order; a block whose count reaches zero is pushed back on the pool
   at that moment.
3. Sharing is by forking: the child gets the parent's table and length, and
   every block of it gains one reference.
4. Appending n tokens to a sequence of length L writes positions L..L+n-1.
   A position that starts a block takes a new block.  A position inside the
   last block writes into it only if that block has a single reference;
   otherwise the block is first copied (copy-on-write): a new block is taken,
   the pair (old, new) is reported for the device copy, the old block loses a
   reference and the table points at the new one.  Slot = block * block_size
   + position % block_size, as in the decode path.
5. One append call over several sequences is all or nothing: if the pool
   runs out anywhere in it, the call fails with nothing changed.

The model mutates plain Python lists and dicts; it is the specification the
native block manager is compared against operation by operation.
"""

import copy


class OutOfBlocks(Exception):
    """The free pool ran out (the pages raise MemoryError and preempt)."""


class BlockManagerModel:
    def __init__(self, num_blocks, block_size):
        if num_blocks < 1 or block_size < 1:
            raise ValueError("num_blocks and block_size must be positive")
        self.block_size = block_size
        self.ref = [0] * num_blocks
        self.free = list(range(num_blocks))   # top of the stack = end of list
        self.tables = {}                      # seq_id -> [physical block ids]
        self.lens = {}                        # seq_id -> tokens held

    # -------------------------------------------------------------- queries
    @property
    def num_blocks(self):
        return len(self.ref)

    def num_free(self):
        return len(self.free)

    def ref_count(self, block):
        return self.ref[block]

    def seq_len(self, seq_id):
        return self.lens[seq_id]

    def table(self, seq_id):
        return list(self.tables[seq_id])

    # ----------------------------------------------------------- operations
    def _take(self):
        if not self.free:
            raise OutOfBlocks("free pool exhausted")
        b = self.free.pop()
        self.ref[b] += 1
        return b

    def add_sequence(self, seq_id):
        if seq_id in self.tables:
            raise KeyError(f"sequence {seq_id} exists")
        self.tables[seq_id] = []
        self.lens[seq_id] = 0

    def fork(self, parent, child):
        if parent not in self.tables or child in self.tables:
            raise KeyError("fork needs an existing parent and a new child")
        self.tables[child] = list(self.tables[parent])
        self.lens[child] = self.lens[parent]
        for b in self.tables[child]:
            self.ref[b] += 1

    def free_sequence(self, seq_id):
        for b in self.tables.pop(seq_id):
            self.ref[b] -= 1
            if self.ref[b] == 0:
                self.free.append(b)
        del self.lens[seq_id]

    def _append_one(self, seq_id, n_new, slots, cows):
        bs = self.block_size
        tbl = self.tables[seq_id]
        for j in range(n_new):
            pos = self.lens[seq_id] + j
            if pos % bs == 0:
                tbl.append(self._take())
            else:
                last = tbl[pos // bs]
                if self.ref[last] > 1:
                    nb = self._take()
                    cows.append((last, nb))
                    self.ref[last] -= 1
                    tbl[pos // bs] = nb
            slots.append(tbl[pos // bs] * bs + pos % bs)
        self.lens[seq_id] += n_new

    def append(self, seq_ids, n_new):
        """Reserve slots for n_new[i] tokens of seq_ids[i], in order.

        Returns (slots, cow_pairs); on exhaustion raises OutOfBlocks and the
        state is exactly as before the call.
        """
        if len(set(seq_ids)) != len(seq_ids):
            raise KeyError("a sequence appears twice in one append")
        for s in seq_ids:
            if s not in self.tables:
                raise KeyError(f"unknown sequence {s}")
        saved = (copy.deepcopy(self.ref), list(self.free), copy.deepcopy(self.tables),
                 dict(self.lens))
        slots, cows = [], []
        try:
            for s, n in zip(seq_ids, n_new):
                self._append_one(s, int(n), slots, cows)
        except OutOfBlocks:
            self.ref, self.free, self.tables, self.lens = saved
            raise
        return slots, cows

    def block_tables(self, seq_ids, max_blocks):
        """[n, max_blocks] table rows (-1 past each sequence's blocks) and lengths."""
        rows, lens = [], []
        for s in seq_ids:
            t = self.tables[s]
            if len(t) > max_blocks:
                raise ValueError("table longer than max_blocks")
            rows.append(t + [-1] * (max_blocks - len(t)))
            lens.append(self.lens[s])
        return rows, lens

    def snapshot(self):
        """Everything observable, for comparisons."""
        return {"ref": list(self.ref), "free": list(self.free),
                "tables": {k: list(v) for k, v in self.tables.items()},
                "lens": dict(self.lens)}


def copy_blocks(cache, pairs):
    """Device copy-on-write step on a numpy cache [NB, ...]: block dst := block src,
    all pairs read from the cache as it was before the call."""
    out = cache.copy()
    for src, dst in pairs:
        out[dst] = cache[src]
    return out
