"""Native block manager (libpkv.so, include/pkv_blocks.h) against the oracle
model, operation by operation, bit for bit.  Host code only: runs without a
GPU."""

import random

import numpy as np
import pytest

import paged_kv_cache_222_gb300 as pkv
from oracle.block_manager import BlockManagerModel, OutOfBlocks


def _same_state(native, model):
    assert native.num_free() == model.num_free()
    assert native.num_sequences() == len(model.tables)
    for b in range(model.num_blocks):
        assert native.ref_count(b) == model.ref_count(b)
    ids = sorted(model.tables)
    if ids:
        mb = max(1, max(len(t) for t in model.tables.values()))
        tbl, lens = native.block_tables(ids, mb)
        rows, mlens = model.block_tables(ids, mb)
        assert tbl.tolist() == rows
        assert lens.tolist() == mlens


@pytest.mark.parametrize("seed", range(8))
def test_native_manager_matches_the_model(seed):
    rng = random.Random(1000 + seed)
    nb = rng.choice([5, 16, 64, 300])
    bs = rng.choice([1, 4, 16, 32])
    native = pkv.BlockManager(nb, bs)
    model = BlockManagerModel(nb, bs)
    nxt = 0
    for _ in range(400):
        live = sorted(model.tables)
        op = rng.random()
        if op < 0.2 or not live:
            native.add_sequence(nxt)
            model.add_sequence(nxt)
            nxt += 1
        elif op < 0.3:
            p = rng.choice(live)
            native.fork(p, nxt)
            model.fork(p, nxt)
            nxt += 1
        elif op < 0.42:
            s = rng.choice(live)
            native.free_sequence(s)
            model.free_sequence(s)
        else:
            k = rng.randint(1, min(6, len(live)))
            ids = rng.sample(live, k)
            n = [rng.randint(0, 3 * bs + 2) for _ in ids]
            try:
                want = model.append(ids, n)
            except OutOfBlocks:
                want = None
            if want is None:
                with pytest.raises(pkv.OutOfBlocks):
                    native.append(ids, n)
            else:
                slots, cows = native.append(ids, n)
                assert slots.tolist() == want[0]
                assert [tuple(c) for c in cows.tolist()] == want[1]
        _same_state(native, model)
    native.close()


def test_blocks_needed_predicts_append():
    rng = random.Random(7)
    bm = pkv.BlockManager(400, 16)
    for s in range(20):
        bm.add_sequence(s)
        bm.append([s], [rng.randint(0, 40)])
    for s in range(20, 30):
        bm.fork(s - 20, s)
    for _ in range(20):
        ids = rng.sample(range(30), 8)
        n = [rng.randint(0, 20) for _ in ids]
        need = bm.blocks_needed(ids, n)
        before = bm.num_free()
        bm.append(ids, n)
        assert before - bm.num_free() == need


def test_rejections_change_nothing():
    bm = pkv.BlockManager(8, 4)
    bm.add_sequence(1)
    bm.append([1], [5])
    free = bm.num_free()
    with pytest.raises(pkv.PkvError):
        bm.add_sequence(1)                     # taken id
    with pytest.raises(pkv.PkvError):
        bm.append([1, 1], [1, 1])              # repeated id
    with pytest.raises(pkv.PkvError):
        bm.append([2], [1])                    # unknown id
    with pytest.raises(pkv.PkvError):
        bm.append([1], [-1])                   # negative count
    with pytest.raises(pkv.PkvError):
        bm.fork(3, 4)                          # unknown parent
    with pytest.raises(pkv.PkvError):
        bm.block_tables([1], 1)                # table longer than the row
    with pytest.raises(pkv.OutOfBlocks):
        bm.append([1], [100])
    assert bm.num_free() == free and bm.seq_len(1) == 5
    assert bm.seq_len(2) == -1 and bm.ref_count(8) == -1 and bm.ref_count(-1) == -1
    tbl, lens = bm.block_tables([1], 4)
    assert tbl.tolist() == [[7, 6, -1, -1]] and lens.tolist() == [5]


def test_create_rejects_bad_sizes():
    with pytest.raises(pkv.PkvError):
        pkv.BlockManager(0, 16)
    with pytest.raises(pkv.PkvError):
        pkv.BlockManager(16, 0)
    with pytest.raises(pkv.PkvError):
        pkv.BlockManager(2**31, 16)


def test_large_pool_serving_churn_is_fast():
    """A pool of 1M blocks, 2048 live sequences, 200 decode steps of one token
    each with retirements and admissions: host bookkeeping stays far below a
    decode step's time per sequence."""
    import time
    bm = pkv.BlockManager(1 << 20, 16)
    rng = np.random.default_rng(0)
    live = list(range(2048))
    for s in live:
        bm.add_sequence(s)
    bm.append(live, rng.integers(1, 4000, size=len(live)).tolist())
    nxt = len(live)
    t0 = time.perf_counter()
    for step in range(200):
        bm.append(live, [1] * len(live))
        if step % 10 == 0:
            for s in live[:8]:
                bm.free_sequence(s)
            live = live[8:] + list(range(nxt, nxt + 8))
            for s in live[-8:]:
                bm.add_sequence(s)
            nxt += 8
    dt = (time.perf_counter() - t0) / 200
    assert dt < 0.05, f"{dt * 1e3:.2f} ms per step"


def _same_tier_state(native, model):
    assert native.num_free() == model.num_free()
    assert native.num_free_host() == len(model.host_free)
    for b in range(model.num_blocks):
        assert native.ref_count(b) == model.ref_count(b)
    for s in model.tables:
        ids, host = native.table_entries(s)
        assert ids.tolist() == model.table(s)
        assert [j for j in range(len(host)) if host[j]] == sorted(model.on_host[s])
        assert native.host_entries(s) == len(model.on_host[s])


@pytest.mark.parametrize("seed", range(6))
def test_native_host_tier_matches_the_model(seed):
    rng = random.Random(2000 + seed)
    nb, nh, bs = rng.choice([8, 32]), rng.choice([4, 24]), rng.choice([4, 16])
    native = pkv.BlockManager(nb, bs)
    native.set_host_blocks(nh)
    model = BlockManagerModel(nb, bs, num_host_blocks=nh)
    nxt = 0
    for _ in range(300):
        live = sorted(model.tables)
        op = rng.random()
        if op < 0.15 or not live:
            native.add_sequence(nxt)
            model.add_sequence(nxt)
            nxt += 1
        elif op < 0.22:
            s = rng.choice(live)
            native.free_sequence(s)
            model.free_sequence(s)
        elif op < 0.3:
            s, c = rng.choice(live), nxt
            if model.on_host[s]:
                with pytest.raises(pkv.PkvError):
                    native.fork(s, c)
                continue
            native.fork(s, c)
            model.fork(s, c)
            nxt += 1
        elif op < 0.55:
            s = rng.choice(live)
            n = len(model.table(s))
            lg = rng.sample(range(n), rng.randint(0, n)) if n else []
            evict = rng.random() < 0.5
            try:
                want = model.evict(s, lg) if evict else model.stage(s, lg)
            except OutOfBlocks:
                want = None
            fn = native.evict if evict else native.stage
            if want is None:
                with pytest.raises(pkv.OutOfBlocks):
                    fn(s, lg)
            else:
                assert [tuple(p) for p in fn(s, lg).tolist()] == want
        elif op < 0.62:
            s = rng.choice(live)
            n = len(model.table(s))
            act = [rng.choice([0.0, 0.2, 0.35, 0.6, 0.9]) for _ in range(n)]
            cap = rng.randint(0, n + 1)
            assert native.prefetch_candidates(s, act, 0.3, cap).tolist() == \
                model.prefetch_candidates(s, act, 0.3, cap)
        else:
            s = rng.choice(live)
            k = rng.randint(1, 2 * bs)
            if model.on_host[s]:
                with pytest.raises(pkv.PkvError):
                    native.append([s], [k])
                continue
            try:
                want = model.append([s], [k])
            except OutOfBlocks:
                want = None
            if want is None:
                with pytest.raises(pkv.OutOfBlocks):
                    native.append([s], [k])
            else:
                slots, cows = native.append([s], [k])
                assert slots.tolist() == want[0] and [tuple(c) for c in cows.tolist()] == want[1]
        _same_tier_state(native, model)


def test_host_tier_rejections():
    bm = pkv.BlockManager(8, 4)
    bm.add_sequence(0)
    bm.append([0], [6])
    with pytest.raises(pkv.PkvError):
        bm.evict(0, [0])                      # no host tier yet
    bm.set_host_blocks(4)
    with pytest.raises(pkv.PkvError):
        bm.set_host_blocks(4)                 # once
    with pytest.raises(pkv.PkvError):
        bm.evict(0, [2])                      # outside the table
    with pytest.raises(pkv.PkvError):
        bm.evict(0, [1, 1])                   # repeated
    bm.evict(0, [1])
    with pytest.raises(pkv.PkvError):
        bm.block_tables([0], 4)               # not resident
    with pytest.raises(pkv.PkvError):
        bm.blocks_needed([0], [1])
    assert bm.stage(0, [0]).shape == (0, 2)   # already on the device: nothing to do
    bm.stage(0, [1])
    tbl, lens = bm.block_tables([0], 4)
    assert lens.tolist() == [6] and bm.num_free_host() == 4
