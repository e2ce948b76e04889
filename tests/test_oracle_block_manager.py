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
