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

Host tier (swap / stage / evict), from [UI] "Architecting Multi-Tier
Disaggregated KV-Cache Hierarchies...", "C++ Block Scheduler and Asynchronous
Fetch Kernel" (promote a block from host memory to HBM, demote it back; an
already resident block is left alone) and
"Predictive Prefetching and Attention-Salience Eviction Policy" (evicted
blocks predicted to be needed soon are staged ahead of the step that reads
them), and [SC] "9. Failure modes and limitations", item 2
(swap a preempted request's blocks to host memory):

6. A second pool of host blocks with its own free stack (same order rule).
   Every table entry is (tier, id).  Evicting entry j of a sequence takes a
   host block, reports (device id, host id) for the copy and drops the
   sequence's reference to the device block (freed when it was the last).
   Staging takes a device block, reports (host id, device id) and frees the
   host block.  Both are all or nothing over the entries of one call;
   entries already in the target tier are skipped.
7. A sequence with any host entry cannot be appended to, forked or attended
   (its block table is not handed out) until it is staged back.
8. Prefetch candidates: the host entries whose predicted activation is
   above the threshold, most probable first (ties by logical index), no
   more than the caller's capacity nor the free device blocks.  Which
   entries to evict is the caller's choice (a salience statistic needs a
   real model's attention weights).
"""

import copy


class OutOfBlocks(Exception):
    """The free pool ran out (the pages raise MemoryError and preempt)."""


class BlockManagerModel:
    def __init__(self, num_blocks, block_size, num_host_blocks=0):
        if num_blocks < 1 or block_size < 1:
            raise ValueError("num_blocks and block_size must be positive")
        self.block_size = block_size
        self.ref = [0] * num_blocks
        self.free = list(range(num_blocks))   # top of the stack = end of list
        self.tables = {}                      # seq_id -> [physical block ids]
        self.lens = {}                        # seq_id -> tokens held
        self.host_free = list(range(num_host_blocks))
        self.on_host = {}                     # seq_id -> set of logical indices held on the host

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
        self.on_host[seq_id] = set()

    def _resident(self, seq_id):
        if self.on_host[seq_id]:
            raise KeyError(f"sequence {seq_id} has blocks on the host")

    def fork(self, parent, child):
        if parent not in self.tables or child in self.tables:
            raise KeyError("fork needs an existing parent and a new child")
        self._resident(parent)
        self.tables[child] = list(self.tables[parent])
        self.lens[child] = self.lens[parent]
        self.on_host[child] = set()
        for b in self.tables[child]:
            self.ref[b] += 1

    def free_sequence(self, seq_id):
        host = self.on_host.pop(seq_id)
        for j, b in enumerate(self.tables.pop(seq_id)):
            if j in host:
                self.host_free.append(b)
                continue
            self.ref[b] -= 1
            if self.ref[b] == 0:
                self.free.append(b)
        del self.lens[seq_id]

    # ------------------------------------------------------------ host tier
    def evict(self, seq_id, logical):
        """Demote entries `logical` of a sequence; returns [(device, host)]."""
        tbl, host = self.tables[seq_id], self.on_host[seq_id]
        logical = list(logical)
        if len(set(logical)) != len(logical) or any(not 0 <= j < len(tbl) for j in logical):
            raise KeyError("bad logical block list")
        todo = [j for j in logical if j not in host]
        if len(todo) > len(self.host_free):
            raise OutOfBlocks("host pool exhausted")
        pairs = []
        for j in todo:
            hb = self.host_free.pop()
            d = tbl[j]
            pairs.append((d, hb))
            self.ref[d] -= 1
            if self.ref[d] == 0:
                self.free.append(d)
            tbl[j] = hb
            host.add(j)
        return pairs

    def stage(self, seq_id, logical):
        """Promote entries `logical` of a sequence; returns [(host, device)]."""
        tbl, host = self.tables[seq_id], self.on_host[seq_id]
        logical = list(logical)
        if len(set(logical)) != len(logical) or any(not 0 <= j < len(tbl) for j in logical):
            raise KeyError("bad logical block list")
        todo = [j for j in logical if j in host]
        if len(todo) > len(self.free):
            raise OutOfBlocks("device pool exhausted")
        pairs = []
        for j in todo:
            d = self._take()
            hb = tbl[j]
            pairs.append((hb, d))
            self.host_free.append(hb)
            tbl[j] = d
            host.discard(j)
        return pairs

    def swap_out(self, seq_id):
        return self.evict(seq_id, range(len(self.tables[seq_id])))

    def swap_in(self, seq_id):
        return self.stage(seq_id, range(len(self.tables[seq_id])))

    def prefetch_candidates(self, seq_id, activation, threshold, capacity=None):
        """Host entries with activation above the threshold, most probable
        first (ties by index), no more than `capacity` nor the free device
        blocks ([UI] "Predictive Prefetching and Attention-Salience Eviction
        Policy": evicted blocks predicted to be needed are staged ahead)."""
        host = self.on_host[seq_id]
        c = sorted((j for j in host if activation[j] > threshold), key=lambda j: (-activation[j], j))
        cap = len(c) if capacity is None else capacity
        return c[:min(cap, len(self.free))]

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
            self._resident(s)
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
            self._resident(s)
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
                "lens": dict(self.lens), "host_free": list(self.host_free),
                "on_host": {k: sorted(v) for k, v in self.on_host.items()}}


def copy_blocks(cache, pairs):
    """Device copy-on-write step on a numpy cache [NB, ...]: block dst := block src,
    all pairs read from the cache as it was before the call."""
    out = cache.copy()
    for src, dst in pairs:
        out[dst] = cache[src]
    return out
