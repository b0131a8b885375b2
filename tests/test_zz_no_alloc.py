"""kvo_copy_blocks_noalloc against kvo_store_blocks / kvo_restore_blocks.

The no-alloc call runs the same block-copy kernel with its pair list staged
in a static device array.  Here it repeats, on caller-owned buffers, the two
copies of a store -> restore cycle of a kvo_pool (two calls in a row, the
second with a different pair list), and each result is compared with what
the pool's own calls produced.  The file is named to be collected last, so
it also runs after every other test in the same process.
"""
import numpy as np
import pytest

from synth import workloads as W
from tests.gpu_harness import cuda_ok

pytestmark = [pytest.mark.gpu, pytest.mark.skipif(not cuda_ok(), reason="needs a CUDA GPU")]

ROW = 656


@pytest.fixture(scope="module")
def kvo():
    from gather_radix_top_gb300 import build, kvo as K
    build.build()
    return K


def test_matches_store_and_restore(kvo):
    import torch
    sw = W.SESSIONS.scaled(tokens=1000, layers=5, sessions=3)
    bt, bb = sw.block_tokens, sw.block_bytes
    nb = sw.sessions * sw.blocks_per_session + 30
    pool = kvo.Pool(sw.layers, nb, bt, nb)
    dev = torch.device("cuda")
    rows = {}
    for s in range(sw.sessions):
        assert pool.alloc(s, sw.tokens) == kvo.KVO_OK
        for layer in range(sw.layers):
            rows[s, layer] = W.session_rows_device(sw, s, layer, dev)
            pool.write(s, layer, 0, rows[s, layer])
    # the caller's own block pool: same block ids, same bytes
    mine = torch.zeros((nb, bb), dtype=torch.uint8, device=dev)
    pad = sw.blocks_per_layer * bt - sw.tokens
    for (s, layer), r in rows.items():
        ids = torch.tensor(pool.block_table(s, layer, 0), device=dev, dtype=torch.long)
        mine[ids] = torch.cat([r, torch.zeros((pad, ROW), dtype=torch.uint8, device=dev)]).view(-1, bb)
    first_pool = {(s, l): pool.block_table(s, l, 0) for s in range(sw.sessions) for l in range(sw.layers)}

    kvo.kvo_copy_blocks_noalloc(mine, mine, bb, np.zeros((0, 2)))    # n = 0: first-call setup only
    for s in range(sw.sessions):
        assert pool.store(s) == kvo.KVO_OK
    pool.sync()
    tier = {(s, l): pool.block_table(s, l, 1) for s in range(sw.sessions) for l in range(sw.layers)}
    for s in range(sw.sessions):
        assert pool.release(s) == kvo.KVO_OK
    pool.fill(0x3C)
    assert pool.alloc(99, 5 * bt) == kvo.KVO_OK                       # shift the restore's block ids
    assert pool.restore([2, 0, 1]) == kvo.KVO_OK
    pool.sync()
    second_pool = {(s, l): pool.block_table(s, l, 0) for s in range(sw.sessions) for l in range(sw.layers)}
    assert second_pool != first_pool

    # call 1: pool -> pinned tier, with the store's pairs
    my_tier = torch.zeros((nb, bb), dtype=torch.uint8).pin_memory()
    back = torch.full((nb, bb), 0x3C, dtype=torch.uint8, device=dev)
    p1 = np.array([(a, b) for key in first_pool for a, b in zip(first_pool[key], tier[key])], np.int32)
    p2 = np.array([(a, b) for key in tier for a, b in zip(tier[key], second_pool[key])], np.int32)
    torch.cuda.synchronize()
    free_before = torch.cuda.mem_get_info()[0]
    kvo.kvo_copy_blocks_noalloc(mine, my_tier, bb, p1)
    # call 2, right after: tier -> a fresh pool, with the restore's pairs
    kvo.kvo_copy_blocks_noalloc(my_tier, back, bb, p2)
    torch.cuda.synchronize()
    assert torch.cuda.mem_get_info()[0] == free_before            # the two calls took no device memory

    out = torch.empty((sw.tokens, ROW), dtype=torch.uint8, device=dev)
    for (s, layer), r in rows.items():
        t_ids = torch.tensor(tier[s, layer], dtype=torch.long)
        got_tier = my_tier[t_ids].view(-1, ROW)[:sw.tokens].to(dev)
        assert torch.equal(got_tier, r), (s, layer)
        pool.read(s, layer, 0, out)                                    # what kvo_restore_blocks produced
        ids = torch.tensor(second_pool[s, layer], device=dev, dtype=torch.long)
        assert torch.equal(back[ids].view(-1, ROW)[:sw.tokens], out), (s, layer)
    # blocks no pair wrote keep their bytes
    used = {b for v in second_pool.values() for b in v}
    untouched = torch.tensor([b for b in range(nb) if b not in used], device=dev, dtype=torch.long)
    assert bool((back[untouched] == 0x3C).all())
    pool.close()


def test_limits(kvo):
    import ctypes

    import torch
    a = torch.zeros((4, 32), dtype=torch.uint8, device="cuda")
    b = torch.zeros((4, 32), dtype=torch.uint8, device="cuda")
    big = np.zeros((kvo.NOALLOC_MAX_PAIRS + 1, 2), np.int32)
    with pytest.raises(kvo.KvoError):
        kvo.kvo_copy_blocks_noalloc(a, b, 32, big)                   # beyond the static scratch
    L = kvo.lib()
    pr = np.zeros(2, np.int32)
    p = ctypes.c_void_p(pr.ctypes.data)
    assert L.kvo_copy_blocks_noalloc(ctypes.c_void_p(a.data_ptr()), ctypes.c_void_p(b.data_ptr()), 24, p, 1,
                                     None) == kvo.KVO_EINVAL          # block_bytes not a multiple of 16
    assert L.kvo_copy_blocks_noalloc(ctypes.c_void_p(a.data_ptr() + 8), ctypes.c_void_p(b.data_ptr()), 32, p,
                                     1, None) == kvo.KVO_EINVAL       # misaligned source
    host = np.zeros(96, np.uint8)
    hp = host.ctypes.data + (-host.ctypes.data) % 16
    assert L.kvo_copy_blocks_noalloc(ctypes.c_void_p(hp), ctypes.c_void_p(b.data_ptr()), 32, p,
                                     1, None) == kvo.KVO_EINVAL       # pageable host memory
    pr[:] = (-1, 0)
    assert L.kvo_copy_blocks_noalloc(ctypes.c_void_p(a.data_ptr()), ctypes.c_void_p(b.data_ptr()), 32, p, 1,
                                     None) == kvo.KVO_EINVAL          # negative block id
    with pytest.raises(ValueError):
        kvo.kvo_copy_blocks_noalloc(a, b, 32, np.array([[4, 0]], np.int32))    # past the end of src
    with pytest.raises(ValueError):
        kvo.kvo_copy_blocks_noalloc(a, b, 32, np.array([[0, 4]], np.int32))    # past the end of dst
    with pytest.raises(ValueError):
        kvo.kvo_copy_blocks_noalloc(a, b, 48, np.array([[0, 0]], np.int32))    # does not divide the buffers
    pr[:] = (0, 0)
    assert L.kvo_copy_blocks_noalloc(ctypes.c_void_p(a.data_ptr()), ctypes.c_void_p(b.data_ptr()), 16 << 32, p, 1,
                                     None) == kvo.KVO_EINVAL          # block_bytes / 16 beyond 32 bits
    a.fill_(7)
    kvo.kvo_copy_blocks_noalloc(a, b, 32, np.array([[3, 0], [0, 2]], np.int32))
    torch.cuda.synchronize()
    assert b[0].eq(7).all() and b[2].eq(7).all() and b[1].eq(0).all() and b[3].eq(0).all()
