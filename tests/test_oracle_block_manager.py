"""Pins of the block-manager model (oracle/block_manager.py) against what the
pages state and against properties any correct paged allocator has."""

import random

import numpy as np
import pytest

from oracle.block_manager import BlockManagerModel, OutOfBlocks, copy_blocks


def test_simulator_pool_holds_exactly_sixty_four_tokens():
    # [SC] "14. ... GPU VRAM & PagedAttention KV Cache Simulator": a physical
    # pool of 16 blocks x 4 tokens = 64 tokens at most.
    m = BlockManagerModel(16, 4)
    m.add_sequence(0)
    slots, cows = m.append([0], [64])
    assert sorted(slots) == list(range(64)) and cows == []
    assert m.num_free() == 0
    before = m.snapshot()
    with pytest.raises(OutOfBlocks):
        m.append([0], [1])
    assert m.snapshot() == before


def test_simulator_pool_sixteen_short_requests():
    m = BlockManagerModel(16, 4)
    for s in range(16):
        m.add_sequence(s)
        m.append([s], [3])
    m.add_sequence(99)
    with pytest.raises(OutOfBlocks):
        m.append([99], [1])
    # the partly filled blocks still take tokens without new blocks
    slots, _ = m.append(list(range(16)), [1] * 16)
    assert len(set(slots)) == 16 and m.num_free() == 0


def test_allocation_takes_top_of_free_stack_and_counts_references():
    # [FN] "Paged KV-Cache with Radix Tree Prefix Cache": a block is taken from
    # the free pool (the last element), its reference count goes up by one and
    # the block id is appended to the sequence's table; an empty pool raises.
    m = BlockManagerModel(5, 16)
    m.add_sequence(7)
    m.append([7], [40])
    assert m.table(7) == [4, 3, 2]
    assert [m.ref_count(b) for b in range(5)] == [0, 0, 1, 1, 1]
    m.add_sequence(8)
    with pytest.raises(OutOfBlocks):
        m.append([8], [33])


def test_slots_follow_the_block_table():
    # [SC] "PagedAttention & Memory Management (vLLM)": logical block j of a
    # sequence maps to a physical block; token t sits at offset t % bs of
    # logical block t // bs.
    m = BlockManagerModel(32, 16)
    m.add_sequence(1)
    slots, _ = m.append([1], [50])
    tbl = m.table(1)
    assert slots == [tbl[t // 16] * 16 + t % 16 for t in range(50)]


def test_fork_shares_blocks_and_copy_on_write_splits_the_last_block():
    m = BlockManagerModel(10, 4)
    m.add_sequence(0)
    m.append([0], [6])           # blocks 9 (full), 8 (2 of 4)
    m.fork(0, 1)
    assert [m.ref_count(b) for b in (9, 8)] == [2, 2]
    slots, cows = m.append([0, 1], [1, 1])
    # seq 0 copies block 8 to a fresh block 7; seq 1 is then the sole owner of 8
    assert cows == [(8, 7)]
    assert slots == [7 * 4 + 2, 8 * 4 + 2]
    assert m.table(0) == [9, 7] and m.table(1) == [9, 8]
    assert [m.ref_count(b) for b in (9, 8, 7)] == [2, 1, 1]


def test_fork_at_block_boundary_needs_no_copy():
    m = BlockManagerModel(10, 4)
    m.add_sequence(0)
    m.append([0], [8])
    m.fork(0, 1)
    slots, cows = m.append([0, 1], [1, 1])
    assert cows == [] and m.num_free() == 6


def test_free_returns_blocks_when_last_reference_goes():
    m = BlockManagerModel(6, 4)
    m.add_sequence(0)
    m.append([0], [8])
    m.fork(0, 1)
    m.free_sequence(0)
    assert m.num_free() == 4
    m.free_sequence(1)
    assert m.num_free() == 6
    # pushed back in table order: the last block of the table is on top
    assert m.free[-2:] == [5, 4]


def test_failed_batch_changes_nothing():
    m = BlockManagerModel(4, 4)
    for s in range(3):
        m.add_sequence(s)
    m.append([0], [4])
    before = m.snapshot()
    with pytest.raises(OutOfBlocks):
        m.append([1, 2], [8, 5])      # 2 + 2 blocks, 3 free
    assert m.snapshot() == before


def _check_invariants(m):
    used = {}
    for s, t in m.tables.items():
        assert len(t) == -(-m.lens[s] // m.block_size)
        for b in t:
            used[b] = used.get(b, 0) + 1
    for b in range(m.num_blocks):
        assert m.ref_count(b) == used.get(b, 0)
    assert sorted(m.free) == [b for b in range(m.num_blocks) if used.get(b, 0) == 0]
    # paged allocation wastes less than one block per sequence
    for s in m.tables:
        assert len(m.tables[s]) * m.block_size - m.lens[s] < m.block_size


@pytest.mark.parametrize("seed", range(6))
def test_random_operations_keep_every_sequence_view(seed):
    """Brute force: track the token id held by every slot; after any mix of
    adds, forks, appends (with copy-on-write applied to the slot contents) and
    frees, each sequence must read back exactly the tokens it was given, and
    no append may write a slot of a block that another sequence references."""
    rng = random.Random(seed)
    bs = rng.choice([2, 4, 16])
    m = BlockManagerModel(rng.choice([6, 12, 40]), bs)
    content = {}                 # slot -> token id
    expect = {}                  # seq -> list of token ids
    next_seq, next_tok = 0, 0
    for _ in range(300):
        op = rng.random()
        live = list(m.tables)
        if op < 0.2 or not live:
            m.add_sequence(next_seq)
            expect[next_seq] = []
            next_seq += 1
        elif op < 0.35:
            p = rng.choice(live)
            m.fork(p, next_seq)
            expect[next_seq] = list(expect[p])
            next_seq += 1
        elif op < 0.5:
            s = rng.choice(live)
            m.free_sequence(s)
            del expect[s]
        else:
            k = rng.randint(1, min(4, len(live)))
            ids = rng.sample(live, k)
            n = [rng.randint(0, 2 * bs) for _ in ids]
            before = m.snapshot()
            try:
                slots, cows = m.append(ids, n)
            except OutOfBlocks:
                assert m.snapshot() == before
                continue
            for src, dst in cows:
                for o in range(bs):
                    if src * bs + o in content:
                        content[dst * bs + o] = content[src * bs + o]
            assert len(set(slots)) == len(slots)
            for sl in slots:
                assert m.ref_count(sl // bs) == 1
            it = iter(slots)
            for s, c in zip(ids, n):
                for _ in range(c):
                    content[next(it)] = next_tok
                    expect[s].append(next_tok)
                    next_tok += 1
        _check_invariants(m)
        for s, toks in expect.items():
            t = m.table(s)
            got = [content[t[i // bs] * bs + i % bs] for i in range(m.seq_len(s))]
            assert got == toks


def test_copy_blocks_reads_the_cache_before_the_call():
    rng = np.random.default_rng(3)
    cache = rng.integers(0, 2**16, size=(6, 2, 4, 8), dtype=np.uint16)
    out = copy_blocks(cache, [(1, 4), (2, 5)])
    assert np.array_equal(out[4], cache[1]) and np.array_equal(out[5], cache[2])
    assert np.array_equal(out[:4], cache[:4])


# ------------------------------------------------------------ host tier

def test_swap_out_frees_device_blocks_and_swap_in_restores_the_view():
    m = BlockManagerModel(6, 4, num_host_blocks=5)
    m.add_sequence(0)
    m.append([0], [10])                       # device 5, 4, 3
    pairs = m.swap_out(0)
    assert pairs == [(5, 4), (4, 3), (3, 2)]  # host stack top first
    assert m.num_free() == 6 and m.on_host[0] == {0, 1, 2}
    with pytest.raises(KeyError):
        m.append([0], [1])                    # not resident
    with pytest.raises(KeyError):
        m.block_tables([0], 4)
    back = m.swap_in(0)
    assert back == [(4, 3), (3, 4), (2, 5)]   # device stack: 3, 4, 5 were pushed in that order
    assert m.on_host[0] == set() and m.num_free() == 3


def test_evicting_a_shared_block_gives_a_private_host_copy():
    m = BlockManagerModel(6, 4, num_host_blocks=4)
    m.add_sequence(0)
    m.append([0], [8])
    m.fork(0, 1)
    pairs = m.evict(1, [0])
    assert pairs == [(5, 3)] and m.ref_count(5) == 1 and m.table(0) == [5, 4]
    m.free_sequence(1)
    assert m.num_free() == 4 and len(m.host_free) == 4


def test_tier_moves_are_all_or_nothing():
    m = BlockManagerModel(4, 4, num_host_blocks=2)
    m.add_sequence(0)
    m.append([0], [12])
    before = m.snapshot()
    with pytest.raises(OutOfBlocks):
        m.swap_out(0)                         # 3 blocks, 2 host blocks
    assert m.snapshot() == before
    m.evict(0, [1, 2])
    m.add_sequence(1)
    m.append([1], [12])                       # takes the 3 freed device blocks
    with pytest.raises(OutOfBlocks):
        m.stage(0, [1, 2])
    assert m.on_host[0] == {1, 2}


def test_prefetch_candidates_most_probable_first_within_the_free_blocks():
    # [UI] "Predictive Prefetching and Attention-Salience Eviction Policy":
    # an evicted block whose predicted activation is above the prefetch
    # threshold is staged ahead of need; most probable first, and no more
    # than the device can take.
    m = BlockManagerModel(10, 4, num_host_blocks=8)
    m.add_sequence(0)
    m.append([0], [8 * 4])                    # 8 device blocks, 2 free
    m.evict(0, [1, 3, 4, 6, 7])               # 7 free
    act = [0.9, 0.5, 0.99, 0.05, 0.5, 0.7, 0.8, 0.31]
    # host entries 1, 3, 4, 6, 7 with activation 0.5, 0.05, 0.5, 0.8, 0.31
    assert m.prefetch_candidates(0, act, 0.3) == [6, 1, 4, 7]
    assert m.prefetch_candidates(0, act, 0.3, capacity=2) == [6, 1]
    assert m.prefetch_candidates(0, act, 0.9) == []
    m.add_sequence(1)
    m.append([1], [6 * 4])                    # leaves one free device block
    assert len(m.free) == 1
    assert m.prefetch_candidates(0, act, 0.3) == [6]
    m.stage(0, [6])
    assert m.prefetch_candidates(0, act, 0.3) == []


@pytest.mark.parametrize("seed", range(4))
def test_random_tier_moves_keep_every_sequence_view(seed):
    rng = random.Random(100 + seed)
    bs = rng.choice([2, 4])
    m = BlockManagerModel(rng.choice([8, 20]), bs, num_host_blocks=rng.choice([4, 16]))
    dev, host = {}, {}                        # slot -> token id, per tier
    expect = {}
    nxt, tok = 0, 0

    def read(s):
        t = m.table(s)
        out = []
        for i in range(m.seq_len(s)):
            j = i // bs
            src = host if j in m.on_host[s] else dev
            out.append(src[t[j] * bs + i % bs])
        return out

    for _ in range(300):
        live = list(m.tables)
        op = rng.random()
        if op < 0.15 or not live:
            m.add_sequence(nxt)
            expect[nxt] = []
            nxt += 1
        elif op < 0.25:
            s = rng.choice(live)
            m.free_sequence(s)
            del expect[s]
        elif op < 0.45:
            s = rng.choice(live)
            n = len(m.table(s))
            lg = rng.sample(range(n), rng.randint(0, n)) if n else []
            to_host = rng.random() < 0.5
            try:
                pairs = m.evict(s, lg) if to_host else m.stage(s, lg)
            except OutOfBlocks:
                continue
            src, dst = (dev, host) if to_host else (host, dev)
            for a, b in pairs:
                for o in range(bs):
                    if a * bs + o in src:
                        dst[b * bs + o] = src[a * bs + o]
        else:
            res = [s for s in live if not m.on_host[s]]
            if not res:
                continue
            s = rng.choice(res)
            try:
                slots, cows = m.append([s], [rng.randint(1, 2 * bs)])
            except OutOfBlocks:
                continue
            for a, b in cows:
                for o in range(bs):
                    if a * bs + o in dev:
                        dev[b * bs + o] = dev[a * bs + o]
            for sl in slots:
                dev[sl] = tok
                expect[s].append(tok)
                tok += 1
        # invariants: device refs count device entries; host ids distinct
        used, hused = {}, []
        for s, t in m.tables.items():
            for j, b in enumerate(t):
                if j in m.on_host[s]:
                    hused.append(b)
                else:
                    used[b] = used.get(b, 0) + 1
        assert all(m.ref_count(b) == used.get(b, 0) for b in range(m.num_blocks))
        assert sorted(hused + m.host_free) == sorted(set(hused + m.host_free))
        for s in expect:
            assert read(s) == expect[s]
