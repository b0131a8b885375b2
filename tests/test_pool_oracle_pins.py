"""Pins for the session store/restore oracle (oracle/kvo_pool_oracle.py).

Each check ties the oracle to something other than itself: the tier sizes
printed on "A 60k-token context comes back off disk in 17 seconds instead of
65 seconds of prefill" (vllm-bounded-fs-kv-tier README), hand-worked FIFO
block tables that follow its free-queue rule, the all-or-nothing invariant of
"Making KV offload correct" ("A grouped allocation is a transaction"), the
copy-completion rule of its section "Response completion is not copy
completion", and conservation / byte-identity invariants over random
operation sequences.
"""
from __future__ import annotations

import pathlib
import random

import numpy as np
import pytest

from oracle import kvo_pool_oracle as po

GOLDEN = pathlib.Path(__file__).parent / "golden" / "tier_sizing.txt"
ROW = 656


def golden_rows():
    out = []
    for line in GOLDEN.read_text().splitlines():
        if line.startswith("#") or not line.strip():
            continue
        tb, rb, nb, rps, mt = line.split()
        out.append((int(tb), int(rb), int(nb), int(rps), mt))
    return out


@pytest.mark.parametrize("row", golden_rows())
def test_tier_blocks_printed_sizes(row):
    tier_bytes, row_bytes, nblocks, rps, mtok = row
    assert po.tier_blocks(tier_bytes, row_bytes) == nblocks
    if rps:
        assert f"{nblocks * 3584 / rps / 1e6:.2f}" == mtok


def rows_for(seed, n):
    return np.random.default_rng(seed).integers(0, 256, (n, ROW), dtype=np.uint8)


def test_fifo_block_tables_worked_example():
    # 8 blocks of 4 tokens, 2 layers.  The free queue starts 0..7, allocation
    # pops from the front and freed blocks go to the back.
    o = po.PoolOracle(layers=2, pool_blocks=8, block_tokens=4, row_bytes=ROW, tier_blocks_n=8)
    assert o.alloc(1, 5) == po.KVO_OK                 # ceil(5/4) = 2 blocks per layer
    assert o.sessions[1].pool == [[0, 1], [2, 3]]
    assert o.alloc(2, 4) == po.KVO_OK
    assert o.sessions[2].pool == [[4], [5]]
    assert o.release(1) == po.KVO_OK
    assert list(o.pool_alloc.free) == [6, 7, 0, 1, 2, 3]
    assert o.alloc(3, 9) == po.KVO_OK                 # 3 blocks per layer
    assert o.sessions[3].pool == [[6, 7, 0], [1, 2, 3]]
    assert o.alloc(4, 1) == po.KVO_ECAPACITY          # nothing left
    assert list(o.pool_alloc.free) == []


def test_restore_admission_worked_example():
    o = po.PoolOracle(layers=2, pool_blocks=6, block_tokens=4, row_bytes=ROW, tier_blocks_n=8)
    assert o.alloc(1, 8) == po.KVO_OK                 # 2 blocks x 2 layers
    assert o.alloc(2, 4) == po.KVO_OK                 # 1 block x 2 layers: the pool is full
    assert o.sessions[1].pool == [[0, 1], [2, 3]] and o.sessions[2].pool == [[4], [5]]
    assert o.store(1) == po.KVO_OK and o.store(2) == po.KVO_OK
    assert o.sessions[1].tier == [[0, 1], [2, 3]] and o.sessions[2].tier == [[4], [5]]
    o.complete_copies()
    assert o.release(1) == po.KVO_OK and o.release(2) == po.KVO_OK
    assert list(o.pool_alloc.free) == [0, 1, 2, 3, 4, 5]
    assert o.alloc(9, 4) == po.KVO_OK                 # takes 0 and 1
    # 6 groups' worth (2+2+1+1) needed, 4 free: refused, nothing moves
    snap = o.snapshot()
    assert o.restore([1, 2]) == po.KVO_ECAPACITY
    assert o.snapshot() == snap
    assert o.restore([2]) == po.KVO_OK
    assert o.sessions[2].pool == [[2], [3]]
    # tier blocks come back only once the copy has completed
    assert list(o.tier_alloc.free) == [6, 7]
    o.complete_copies()
    assert list(o.tier_alloc.free) == [6, 7, 4, 5]


def test_release_waits_for_copy_completion():
    o = po.PoolOracle(layers=3, pool_blocks=16, block_tokens=4, row_bytes=ROW, tier_blocks_n=16)
    assert o.alloc(7, 10) == po.KVO_OK
    assert o.store(7) == po.KVO_OK
    assert o.release(7) == po.KVO_EBUSY               # transfer still pending
    assert o.sessions[7].pool is not None
    o.complete_copies()
    assert o.release(7) == po.KVO_OK
    assert o.restore([7]) == po.KVO_OK
    assert o.release(7) == po.KVO_EBUSY
    o.complete_copies()
    assert o.release(7) == po.KVO_OK
    assert 7 not in o.sessions                        # neither in pool nor in tier


@pytest.mark.parametrize("fail_at", range(0, 12))
def test_failed_transaction_leaves_state_unchanged(fail_at):
    def build():
        o = po.PoolOracle(layers=4, pool_blocks=40, block_tokens=4, row_bytes=ROW, tier_blocks_n=40)
        assert o.alloc(1, 7) == po.KVO_OK             # 2 per layer: 8 blocks
        assert o.alloc(2, 3) == po.KVO_OK             # 1 per layer
        assert o.release(2) == po.KVO_OK
        return o

    o = build()
    snap = o.snapshot()
    o.pool_alloc.fail_after = fail_at                 # 12 blocks asked for; one of them fails
    assert o.alloc(3, 12) == po.KVO_ECAPACITY
    assert o.snapshot() == snap
    assert o.stats["rollbacks"] == 1
    # and what succeeds afterwards is exactly what a run without the fault gets
    assert o.alloc(3, 12) == po.KVO_OK
    ref = build()
    assert ref.alloc(3, 12) == po.KVO_OK
    assert o.sessions[3].pool == ref.sessions[3].pool
    assert list(o.pool_alloc.free) == list(ref.pool_alloc.free)

    # the same for the tier side of a store and the pool side of a restore
    o = build()
    assert o.store(1) == po.KVO_OK
    o.complete_copies()
    assert o.release(1) == po.KVO_OK
    snap = o.snapshot()
    o.pool_alloc.fail_after = fail_at % 8
    assert o.restore([1]) == po.KVO_ECAPACITY
    assert o.snapshot() == snap
    o2 = build()
    snap2 = o2.snapshot()
    o2.tier_alloc.fail_after = fail_at % 8
    assert o2.store(1) == po.KVO_ECAPACITY
    assert o2.snapshot() == snap2


def test_planted_rollback_mistake_is_caught():
    """A rollback that returns blocks to the back of the queue (instead of
    where they were) must fail the snapshot check."""
    class Leaky(po.BlockAllocator):
        def give_front(self, blocks):
            self.free.extend(blocks)

    o = po.PoolOracle(layers=2, pool_blocks=10, block_tokens=4, row_bytes=ROW, tier_blocks_n=4)
    o.pool_alloc = Leaky(10)
    snap = o.snapshot()
    o.pool_alloc.fail_after = 3
    assert o.alloc(1, 8) == po.KVO_ECAPACITY
    assert o.snapshot() != snap


def test_store_fill_restore_is_byte_identity():
    o = po.PoolOracle(layers=3, pool_blocks=64, block_tokens=16, row_bytes=ROW, tier_blocks_n=64)
    data = {}
    for sid, tokens in ((1, 37), (2, 16), (3, 100)):
        assert o.alloc(sid, tokens) == po.KVO_OK
        for layer in range(3):
            data[sid, layer] = rows_for(sid * 10 + layer, tokens)
            assert o.write(sid, layer, 0, data[sid, layer]) == po.KVO_OK
    for sid in (1, 2, 3):
        assert o.store(sid) == po.KVO_OK
    o.complete_copies()
    for sid in (1, 2, 3):
        assert o.release(sid) == po.KVO_OK
    o.fill(0xA5)
    assert o.alloc(4, 200) == po.KVO_OK               # a newcomer reuses the freed blocks
    for layer in range(3):
        assert (o.read(4, layer, 0, 200) == 0xA5).all()
    assert o.restore([3, 1]) == po.KVO_ECAPACITY      # 13 blocks per layer held by session 4
    assert o.release(4) == po.KVO_OK
    assert o.restore([3, 1]) == po.KVO_OK
    assert o.restore([2]) == po.KVO_OK
    for (sid, layer), rows in data.items():
        np.testing.assert_array_equal(o.read(sid, layer, 0, rows.shape[0]), rows)


def test_partial_writes_land_at_their_token():
    o = po.PoolOracle(layers=1, pool_blocks=8, block_tokens=4, row_bytes=ROW, tier_blocks_n=0)
    assert o.alloc(1, 11) == po.KVO_OK
    a, b = rows_for(1, 6), rows_for(2, 5)
    assert o.write(1, 0, 0, a) == po.KVO_OK
    assert o.write(1, 0, 6, b) == po.KVO_OK
    assert o.write(1, 0, 7, b) == po.KVO_EINVAL       # past the session's tokens
    np.testing.assert_array_equal(o.read(1, 0, 0, 11), np.concatenate([a, b]))
    # token 5 is row 1 of the second block (blocks 0, 1, 2)
    np.testing.assert_array_equal(o.pool[1, ROW:2 * ROW], a[5])


def test_random_operation_sequences_conserve_blocks_and_bytes():
    rng = random.Random(1234)
    layers, bt = 3, 4
    o = po.PoolOracle(layers=layers, pool_blocks=60, block_tokens=bt, row_bytes=ROW, tier_blocks_n=50)
    truth = {}
    next_sid = 0
    for step in range(400):
        op = rng.choice(["alloc", "alloc", "store", "release", "restore", "complete"])
        if op == "alloc":
            tokens = rng.randint(1, 30)
            if o.alloc(next_sid, tokens) == po.KVO_OK:
                for layer in range(layers):
                    truth[next_sid, layer] = rows_for(step * 7 + layer, tokens)
                    o.write(next_sid, layer, 0, truth[next_sid, layer])
            next_sid += 1
        elif op == "store":
            c = [i for i, s in o.sessions.items() if s.pool is not None and s.tier is None]
            if c:
                o.store(rng.choice(c))
        elif op == "release":
            c = [i for i, s in o.sessions.items() if s.pool is not None]
            if c:
                sid = rng.choice(c)
                had_tier = o.sessions[sid].tier is not None
                if o.release(sid) == po.KVO_OK and not had_tier:
                    for layer in range(layers):
                        truth.pop((sid, layer))
        elif op == "restore":
            c = [i for i, s in o.sessions.items() if s.tier is not None and s.pool is None]
            if c:
                o.restore(rng.sample(c, min(len(c), rng.randint(1, 3))))
        else:
            o.complete_copies()
        # conservation: every block is free or owned, never both, never twice
        owned = [b for s in o.sessions.values() if s.pool for g in s.pool for b in g]
        assert sorted(owned + list(o.pool_alloc.free)) == list(range(60))
        pend_tier = [b for _, frees in o.pending for _, g in frees for b in g]
        tier_owned = [b for s in o.sessions.values() if s.tier for g in s.tier for b in g]
        assert sorted(tier_owned + pend_tier + list(o.tier_alloc.free)) == list(range(50))
        for s in o.sessions.values():
            assert s.pool is not None or s.tier is not None
            for g in (s.pool or s.tier):
                assert len(g) == -(-s.tokens // bt)
    o.complete_copies()
    for (sid, layer), rows in truth.items():
        s = o.sessions[sid]
        if s.pool is None:
            assert o.restore([sid]) in (po.KVO_OK, po.KVO_ECAPACITY)
        if o.sessions[sid].pool is not None:
            np.testing.assert_array_equal(o.read(sid, layer, 0, rows.shape[0]), rows)
