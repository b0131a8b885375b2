"""Session block store/restore on the GPU vs the oracle, through the C ABI.

Bar: identical status codes, block tables (pool and tier), free-queue order
and counters after every call; byte-identical rows.
"""
import random

import numpy as np
import pytest

from oracle import kvo_pool_oracle as PO
from synth import workloads as W
from tests.gpu_harness import cuda_ok

pytestmark = [pytest.mark.gpu, pytest.mark.skipif(not cuda_ok(), reason="needs a CUDA GPU")]

ROW = 656


@pytest.fixture(scope="module")
def kvo():
    from gather_radix_top_gb300 import build, kvo as K
    build.build()
    return K


class Mirror:
    """One oracle pool and one GPU pool driven with the same calls."""

    def __init__(self, kvo, layers, pool_blocks, bt, tier_blocks, seed=7):
        self.K = kvo
        self.o = PO.PoolOracle(layers, pool_blocks, bt, ROW, tier_blocks)
        self.g = kvo.Pool(layers, pool_blocks, bt, tier_blocks)
        self.layers, self.bt = layers, bt
        self.sw = W.SESSIONS.scaled(seed=seed, layers=layers, block_tokens=bt, tokens=256)
        self.ids = set()

    def alloc(self, sid, tokens):
        self.ids.add(sid)
        a, b = self.o.alloc(sid, tokens), self.g.alloc(sid, tokens)
        assert a == b
        return a

    def write(self, sid, layer, first, n):
        import torch
        rows = W.session_rows(self.sw, sid, layer, first, n)
        assert self.o.write(sid, layer, first, rows) == PO.KVO_OK
        self.g.write(sid, layer, first, torch.from_numpy(rows).cuda())

    def write_all(self, sid):
        for layer in range(self.layers):
            self.write(sid, layer, 0, self.o.sessions[sid].tokens)

    def store(self, sid):
        a, b = self.o.store(sid), self.g.store(sid)
        assert a == b
        return a

    def release(self, sid):
        a, b = self.o.release(sid), self.g.release(sid)
        assert a == b
        return a

    def restore(self, sids):
        a, b = self.o.restore(list(sids)), self.g.restore(list(sids))
        assert a == b
        return a

    def sync(self):
        self.o.complete_copies()
        self.g.sync()

    def check(self, rows=True):
        import torch
        o, g = self.o, self.g
        assert g.free_queue(0) == list(o.pool_alloc.free)
        assert g.free_queue(1) == list(o.tier_alloc.free)
        for sid in self.ids:
            s = o.sessions.get(sid)
            for layer in range(self.layers):
                want_p = s.pool[layer] if s is not None and s.pool else None
                want_t = s.tier[layer] if s is not None and s.tier else None
                assert g.block_table(sid, layer, 0) == want_p, (sid, layer)
                assert g.block_table(sid, layer, 1) == want_t, (sid, layer)
                if rows and want_p is not None:
                    out = torch.empty((s.tokens, ROW), dtype=torch.uint8, device="cuda")
                    g.read(sid, layer, 0, out)
                    np.testing.assert_array_equal(out.cpu().numpy(), o.read(sid, layer, 0, s.tokens))
        st = g.stats()
        for k in ("stores", "restores", "rollbacks", "bytes_stored", "bytes_restored"):
            assert st[k] == o.stats[k], k
        assert st["free_blocks"] == len(o.pool_alloc.free)
        assert st["tier_free_blocks"] == len(o.tier_alloc.free)


def test_worked_cycle(kvo):
    m = Mirror(kvo, layers=2, pool_blocks=6, bt=4, tier_blocks=8)
    assert m.alloc(1, 8) == PO.KVO_OK
    assert m.alloc(2, 4) == PO.KVO_OK
    m.write_all(1)
    m.write_all(2)
    m.check()
    assert m.store(1) == PO.KVO_OK and m.store(2) == PO.KVO_OK
    m.sync()
    assert m.release(1) == PO.KVO_OK and m.release(2) == PO.KVO_OK
    m.o.fill(0x5A)
    m.g.fill(0x5A)
    assert m.alloc(9, 4) == PO.KVO_OK
    m.check()
    assert m.restore([1, 2]) == PO.KVO_ECAPACITY
    m.check()
    assert m.restore([2]) == PO.KVO_OK
    m.sync()
    m.check()


def test_partial_writes_and_reads(kvo):
    import torch
    m = Mirror(kvo, layers=1, pool_blocks=16, bt=16, tier_blocks=0)
    assert m.alloc(3, 100) == PO.KVO_OK
    m.write(3, 0, 0, 37)
    m.write(3, 0, 37, 1)
    m.write(3, 0, 38, 62)
    m.write(3, 0, 15, 2)        # across a block edge, over earlier rows
    m.check()
    out = torch.empty((21, ROW), dtype=torch.uint8, device="cuda")
    m.g.read(3, 0, 30, out)
    np.testing.assert_array_equal(out.cpu().numpy(), m.o.read(3, 0, 30, 21))
    with pytest.raises(kvo.KvoError):
        m.g.read(3, 0, 90, out)  # past the session's tokens
    import ctypes
    host = np.zeros(2 * ROW + 16, np.uint8)                     # pageable host memory is refused
    ptr = host.ctypes.data + (-host.ctypes.data) % 16
    assert kvo.lib().kvo_pool_write(m.g.handle, 3, 0, 0, ctypes.c_void_p(ptr), 2, None) == kvo.KVO_EINVAL


@pytest.mark.parametrize("fail_at", [0, 1, 2, 5, 7, 11])
def test_forced_failures_roll_back(kvo, fail_at):
    m = Mirror(kvo, layers=4, pool_blocks=40, bt=4, tier_blocks=40)
    assert m.alloc(1, 7) == PO.KVO_OK
    m.write_all(1)
    assert m.alloc(2, 3) == PO.KVO_OK
    assert m.release(2) == PO.KVO_OK
    m.check()
    m.o.pool_alloc.fail_after = fail_at
    m.g.fail_after(0, fail_at)
    assert m.alloc(3, 12) == PO.KVO_ECAPACITY
    m.check()
    assert m.alloc(3, 12) == PO.KVO_OK
    m.check()
    m.o.tier_alloc.fail_after = fail_at % 8
    m.g.fail_after(1, fail_at % 8)
    assert m.store(1) == PO.KVO_ECAPACITY
    m.check()
    assert m.store(1) == PO.KVO_OK
    m.sync()
    assert m.release(1) == PO.KVO_OK
    m.o.pool_alloc.fail_after = fail_at % 8
    m.g.fail_after(0, fail_at % 8)
    assert m.restore([1]) == PO.KVO_ECAPACITY
    m.check()
    assert m.restore([1]) == PO.KVO_OK
    m.sync()
    m.check()


def test_release_waits_for_copy_completion(kvo):
    """The copy is held back behind a spin kernel on the same stream, so it
    is certainly pending when release is called."""
    import torch
    m = Mirror(kvo, layers=3, pool_blocks=32, bt=8, tier_blocks=32)
    assert m.alloc(5, 40) == PO.KVO_OK
    m.write_all(5)
    torch.cuda._sleep(200_000_000)           # ~0.1 s of device time before the copy
    assert m.store(5) == PO.KVO_OK
    assert m.release(5) == PO.KVO_EBUSY      # both: the copy has not completed
    assert m.g.stats()["pending_copies"] == 1
    m.sync()
    assert m.g.stats()["pending_copies"] == 0
    assert m.release(5) == PO.KVO_OK
    m.o.fill(0)
    m.g.fill(0)
    torch.cuda._sleep(200_000_000)
    assert m.restore([5]) == PO.KVO_OK
    # the tier blocks of a restore are freed only once its copy is done
    assert m.g.free_queue(1) == list(m.o.tier_alloc.free)
    assert m.release(5) == PO.KVO_EBUSY
    m.sync()
    m.check()
    assert m.release(5) == PO.KVO_OK
    m.check(rows=False)


def test_random_operation_sequences(kvo):
    rng = random.Random(99)
    m = Mirror(kvo, layers=3, pool_blocks=48, bt=16, tier_blocks=40, seed=11)
    sid = 0
    for step in range(160):
        op = rng.choice(["alloc", "alloc", "store", "release", "restore", "write"])
        o = m.o
        if op == "alloc":
            if m.alloc(sid, rng.randint(1, 60)) == PO.KVO_OK:
                m.write_all(sid)
            sid += 1
        elif op == "write":
            c = [i for i, s in o.sessions.items() if s.pool is not None]
            if c:
                i = rng.choice(c)
                t = o.sessions[i].tokens
                first = rng.randrange(t)
                m.write(i, rng.randrange(3), first, rng.randint(1, t - first))
        elif op == "store":
            c = [i for i, s in o.sessions.items() if s.pool is not None and s.tier is None]
            if c:
                m.store(rng.choice(c))
                m.sync()
        elif op == "release":
            c = [i for i, s in o.sessions.items() if s.pool is not None]
            if c:
                m.release(rng.choice(c))
        else:
            c = [i for i, s in o.sessions.items() if s.tier is not None and s.pool is None]
            if c:
                m.restore(rng.sample(c, min(len(c), rng.randint(1, 3))))
                m.sync()
        m.check(rows=(step % 10 == 0))
    m.check()


def test_eight_sessions_store_fill_restore(kvo):
    """Eight sessions, 78 layers, 16-token blocks (the evict/restore cycle at
    a tenth of the 60,000-token length): bytewise identity, restored as one
    admission."""
    import torch
    sw = W.SESSIONS.scaled(tokens=6_000)
    per = sw.blocks_per_session
    pool = kvo.Pool(sw.layers, sw.sessions * per, sw.block_tokens, sw.sessions * per)
    dev = torch.device("cuda")
    for s in range(sw.sessions):
        assert pool.alloc(s, sw.tokens) == PO.KVO_OK
        for layer in range(sw.layers):
            pool.write(s, layer, 0, W.session_rows_device(sw, s, layer, dev))
    for s in range(sw.sessions):
        assert pool.store(s) == PO.KVO_OK
    pool.sync()
    for s in range(sw.sessions):
        assert pool.release(s) == PO.KVO_OK
    pool.fill(0xA5)
    out = torch.empty((sw.tokens, ROW), dtype=torch.uint8, device=dev)
    assert pool.alloc(100, sw.tokens) == PO.KVO_OK       # the filler session takes blocks from the front
    pool.read(100, 7, 0, out)
    assert bool((out == 0xA5).all())
    assert pool.restore(list(range(sw.sessions))) == PO.KVO_ECAPACITY
    assert pool.release(100) == PO.KVO_OK
    order = [3, 0, 7, 1, 6, 2, 5, 4]
    # a forced failure 60% of the way through the admission leaves everything as it was
    before = (pool.free_queue(0), pool.free_queue(1),
              [pool.block_table(s, l, w) for s in order for l in (0, sw.layers - 1) for w in (0, 1)])
    pool.fail_after(0, int(0.6 * sw.sessions * per))
    assert pool.restore(order) == PO.KVO_ECAPACITY
    after = (pool.free_queue(0), pool.free_queue(1),
             [pool.block_table(s, l, w) for s in order for l in (0, sw.layers - 1) for w in (0, 1)])
    assert after == before
    assert pool.restore(order) == PO.KVO_OK
    pool.sync()
    for s in range(sw.sessions):
        for layer in range(sw.layers):
            pool.read(s, layer, 0, out)
            assert torch.equal(out, W.session_rows_device(sw, s, layer, dev)), (s, layer)
    st = pool.stats()
    assert st["stores"] == 8 and st["restores"] == 1 and st["rollbacks"] == 2
    assert st["bytes_stored"] == st["bytes_restored"] == sw.sessions * per * sw.block_bytes
    assert st["tier_free_blocks"] == sw.sessions * per and st["free_blocks"] == 0
    pool.close()


def test_full_length_session_identity(kvo):
    """One 60,000-token, 78-layer session (3.07 GB of blocks) through store,
    filler overwrite and restore."""
    import torch
    sw = W.SESSIONS.scaled(sessions=1)
    per = sw.blocks_per_session
    pool = kvo.Pool(sw.layers, per, sw.block_tokens, per)
    dev = torch.device("cuda")
    assert pool.alloc(0, sw.tokens) == PO.KVO_OK
    for layer in range(sw.layers):
        pool.write(0, layer, 0, W.session_rows_device(sw, 0, layer, dev))
    assert pool.store(0) == PO.KVO_OK
    pool.sync()
    assert pool.release(0) == PO.KVO_OK
    pool.fill(0x00)
    assert pool.restore([0]) == PO.KVO_OK
    pool.sync()
    out = torch.empty((sw.tokens, ROW), dtype=torch.uint8, device=dev)
    for layer in range(sw.layers):
        pool.read(0, layer, 0, out)
        assert torch.equal(out, W.session_rows_device(sw, 0, layer, dev)), layer
    # tier ids after a full cycle: the session's first store took tier blocks 0..per-1 in order
    assert pool.free_queue(1)[:4] == [0, 1, 2, 3]
    pool.close()


def test_argument_errors(kvo):
    import torch
    pool = kvo.Pool(2, 8, 4, 8)
    assert pool.alloc(1, 4) == PO.KVO_OK
    with pytest.raises(kvo.KvoError):
        pool.alloc(1, 4)                                 # id in use
    with pytest.raises(kvo.KvoError):
        pool.alloc(2, 0)
    with pytest.raises(kvo.KvoError):
        pool.restore([1])                                # not stored
    with pytest.raises(kvo.KvoError):
        pool.store(42)                                   # unknown session
    with pytest.raises(kvo.KvoError):
        pool.write(1, 2, 0, torch.zeros((1, ROW), dtype=torch.uint8, device="cuda"))   # layer out of range
    assert pool.store(1) == PO.KVO_OK
    with pytest.raises(kvo.KvoError):
        pool.store(1)                                    # already stored
    pool.sync()
    assert pool.release(1) == PO.KVO_OK
    with pytest.raises(kvo.KvoError):
        pool.restore([1, 1])                             # duplicate ids
    pool.close()
