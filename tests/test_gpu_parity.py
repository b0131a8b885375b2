"""CUDA path vs oracle, element by element, through the C ABI.

Bar: bit-exact for positions, maps, eviction order and raw rows; 0 bf16 ULP
for the dequant (both sides round the same exact float32 product once).
"""
import numpy as np
import pytest

from oracle import kvo_oracle as O
from synth import workloads as W
from tests.gpu_harness import GpuLayerRun, OracleLayerRun, compare_state, cuda_ok

pytestmark = [pytest.mark.gpu, pytest.mark.skipif(not cuda_ok(), reason="needs a CUDA GPU")]


@pytest.fixture(scope="module")
def kvo():
    from gather_radix_top_gb300 import build, kvo as K
    build.build()
    return K


@pytest.fixture(scope="module")
def ctx(kvo):
    c = kvo.Context(1, 64, 16)
    yield c
    c.close()


def _bits(x):
    return np.asarray(x).view(np.uint16)


def assert_bf16_equal(got, want):
    """Bit-equal bf16, except that a NaN matches any NaN: IEEE-754 leaves the
    sign and payload of a NaN result open, and CPUs and GPUs differ there."""
    got, want = _bits(got), _bits(want)
    nan_g = (got & 0x7F80) == 0x7F80
    nan_g &= (got & 0x7F) != 0
    nan_w = (want & 0x7F80) == 0x7F80
    nan_w &= (want & 0x7F) != 0
    np.testing.assert_array_equal(nan_g, nan_w)
    np.testing.assert_array_equal(np.where(nan_g, 0, got), np.where(nan_w, 0, want))


# ------------------------------------------------------------------ top-K
TOPK_CASES = [
    (1, 1, "normal"), (5, 3, "normal"), (31, 31, "normal"), (64, 32, "normal"), (100, 33, "ties"),
    (1000, 256, "special"), (4096, 256, "normal"), (4096, 256, "ties"), (4099, 1000, "special"),
    (50_023, 2048, "normal"), (50_023, 2048, "ties"), (51_047, 2048, "special"),
    (65_537, 4096, "normal"), (200_000, 2048, "ties"), (1_048_576, 2048, "normal"),
    (1_048_576, 2048, "ties"), (1_048_583, 4093, "special"),
    # beyond the shared-memory-resident size: the filtered route and its fallback
    (786_433, 2048, "normal"), (1_048_576, 1, "normal"), (1_048_576, 2048, "coarse"),
    (1_048_576, 4096, "coarse"), (1_048_576, 2048, "recent"), (1_048_577, 4096, "recent"),
    (2_000_003, 2048, "lognormal"), (3_000_017, 4096, "coarse"), (1_048_576, 2048, "sprinkled"),
    (1_048_576, 2048, "negative"), (1_048_576, 2048, "negzero"), (1_048_576, 4096, "negzero"),
    (1_048_576, 2048, "nan_inf"),
    (1_048_579, 1000, "nan_inf"),
]


@pytest.mark.parametrize("n,k,kind", TOPK_CASES)
def test_topk_matches_oracle(ctx, n, k, kind):
    import torch
    s = W.random_scores(n * 7 + k, n, kind)
    idx = ctx.select_topk(torch.from_numpy(s).cuda(), k)
    np.testing.assert_array_equal(idx.cpu().numpy(), O.select_topk(s, k))


@pytest.mark.parametrize("n,k", [(4096, 256), (50_023, 2048), (1_048_576, 2048)])
def test_topk_degenerate_orders(ctx, n, k):
    import torch
    for s in (np.zeros(n, np.float32), np.arange(n, dtype=np.float32),
              -np.arange(n, dtype=np.float32), np.full(n, np.nan, np.float32)):
        idx = ctx.select_topk(torch.from_numpy(s).cuda(), k).cpu().numpy()
        np.testing.assert_array_equal(idx, O.select_topk(s, k))


@pytest.mark.parametrize("nq,n,ld,k", [(1, 1000, 1000, 100), (4, 50_024, 51_200, 2048), (3, 4099, 4101, 1000),
                                        (5, 1_048_576, 1_048_576, 2048), (2, 200_000, 200_003, 4093),
                                        (3, 1_048_583, 1_048_591, 2048)])
def test_topk_batch_matches_oracle_per_row(ctx, nq, n, ld, k):
    """One launch, one cluster per row; rows at any stride (unaligned too)."""
    import torch
    rows = np.zeros((nq, ld), np.float32)
    for q in range(nq):
        kinds = ["normal", "ties", "special"] if n < 1_048_583 else ["normal", "coarse", "recent"]
        rows[q, :n] = W.random_scores(nq * 1000 + q + n, n, kinds[q % 3])
        rows[q, n:] = np.inf                          # beyond n: must never be selected
    idx = ctx.select_topk_batch(torch.from_numpy(rows).cuda(), k, n)
    got = idx.cpu().numpy()
    for q in range(nq):
        np.testing.assert_array_equal(got[q], O.select_topk(rows[q, :n], k))


def test_topk_k_equals_n_and_unaligned_scores(ctx):
    import torch
    s = W.random_scores(11, 3001, "special")
    idx = ctx.select_topk(torch.from_numpy(s).cuda(), 3001).cpu().numpy()
    np.testing.assert_array_equal(idx, np.arange(3001))
    big = torch.from_numpy(W.random_scores(12, 9001)).cuda()
    view = big[1:]                                   # 4-byte aligned, not 16
    idx = ctx.select_topk(view, 777).cpu().numpy()
    np.testing.assert_array_equal(idx, O.select_topk(big.cpu().numpy()[1:], 777))


# ---------------------------------------------------------------- resolve
def test_tiny_workload_full_parity(kvo):
    w = W.TINY
    g = GpuLayerRun(w, 0, want_bf16=True)
    o = OracleLayerRun(w, 0, want_bf16=True)
    g.ctx.record_evictions(True)
    for step in range(w.steps):
        gi = g.step(step)
        oi = o.step(step)
        np.testing.assert_array_equal(gi, oi)
        np.testing.assert_array_equal(g.rows(), o.last.rows)
        np.testing.assert_array_equal(g.bf16(), o.last.bf16)
        assert g.ctx.evictions(0) == o.last.evictions
        compare_state(g.ctx, 0, o.st)
    assert g.ctx.sync() == 0
    st = g.ctx.stats(0)
    assert st["steps"] == w.steps and st["rows_out"] == w.steps * w.k
    g.ctx.close()


@pytest.mark.parametrize("seed,H,n,k,dup,bad", [
    (1, 16, 40, 16, 0.3, 2), (2, 64, 300, 33, 0.5, 0), (3, 1024, 5000, 256, 0.2, 5),
    (4, 1024, 5000, 1024, 0.0, 0), (5, 4096, 70_000, 2048, 0.4, 3), (6, 32_768, 60_000, 4096, 0.1, 1), (7, 131_072, 300_000, 4096, 0.0, 0),
])
def test_resolve_random_selections(kvo, seed, H, n, k, dup, bad):
    """Arbitrary order, duplicates and out-of-range entries; many steps so the
    cache fills, then evicts."""
    import torch
    g = np.random.default_rng(seed)
    hist = g.integers(0, 256, size=(n, O.ROW_BYTES), dtype=np.uint8)
    ctx = kvo.Context(1, n, H)
    ctx.append_rows(0, hist)
    ctx.record_evictions(True)
    st = O.LayerState(n, H)
    st.append(hist)
    out = torch.empty((k, O.ROW_BYTES), dtype=torch.uint8, device="cuda")
    outb = torch.empty((k, O.DEQUANT_VALUES), dtype=torch.int16, device="cuda")
    for step in range(12):
        idx = W.random_idx(seed * 100 + step, n if step % 3 else min(n, 2 * H), k, dup, bad if step % 2 else 0)
        ctx.resolve_gather(0, torch.from_numpy(idx).cuda(), out, outb)
        res = O.resolve_gather(st, idx, want_bf16=True)
        np.testing.assert_array_equal(out.cpu().numpy(), res.rows)
        assert_bf16_equal(outb.cpu().numpy(), res.bf16)
        assert ctx.evictions(0) == res.evictions
        status = ctx.sync()
        assert status == (kvo.KVO_ERANGE if res.invalid else 0)
    compare_state(ctx, 0, st)
    s = ctx.stats(0)
    ctx.close()


@pytest.mark.parametrize("H,k,sub,dup", [(64, 64, 100, 0.0), (64, 40, 90, 0.0), (64, 8, 70, 0.0), (64, 40, 90, 0.3)])
def test_lru_queue_compaction_over_many_steps(kvo, H, k, sub, dup):
    """Selections drawn from a small range of positions, so most entries hit
    and few slots are evicted: the LRU queue fills with stale entries and is
    compacted many times over 120 steps.  Evictions compared every step."""
    import torch
    n = 400
    hist = np.random.default_rng(H + k).integers(0, 256, size=(n, O.ROW_BYTES), dtype=np.uint8)
    ctx = kvo.Context(1, n, H)
    ctx.append_rows(0, hist)
    ctx.record_evictions(True)
    st = O.LayerState(n, H)
    st.append(hist)
    out = torch.empty((k, O.ROW_BYTES), dtype=torch.uint8, device="cuda")
    for step in range(120):
        idx = W.random_idx(7000 + step, sub if step % 10 else n, k, dup, 0)
        if dup == 0.0:
            idx = np.sort(idx)
        ctx.resolve_gather(0, torch.from_numpy(idx).cuda(), out)
        res = O.resolve_gather(st, idx)
        np.testing.assert_array_equal(out.cpu().numpy(), res.rows)
        assert ctx.evictions(0) == res.evictions, step
    assert ctx.sync() == 0
    compare_state(ctx, 0, st)
    ctx.close()


def test_hot_cache_exactly_k_rows(kvo):
    """k = hot_rows: every slot may be needed in one step."""
    import torch
    n, H = 4000, 512
    hist = np.random.default_rng(9).integers(0, 256, size=(n, O.ROW_BYTES), dtype=np.uint8)
    ctx = kvo.Context(1, n, H)
    ctx.append_rows(0, hist)
    st = O.LayerState(n, H)
    st.append(hist)
    out = torch.empty((H, O.ROW_BYTES), dtype=torch.uint8, device="cuda")
    for step in range(6):
        idx = np.sort(np.random.default_rng(step).choice(n, H, replace=False)).astype(np.int32)
        ctx.resolve_gather(0, torch.from_numpy(idx).cuda(), out)
        res = O.resolve_gather(st, idx)
        np.testing.assert_array_equal(out.cpu().numpy(), res.rows)
    compare_state(ctx, 0, st)
    ctx.close()


def test_append_host_and_device_rows(kvo):
    import torch
    w = W.TINY.scaled(appends_per_step=3, steps=6)
    g = GpuLayerRun(w, 0)
    o = OracleLayerRun(w, 0)
    for step in range(w.steps):
        np.testing.assert_array_equal(g.step(step), o.step(step))
        np.testing.assert_array_equal(g.rows(), o.last.rows)
    assert g.ctx.history_length(0) == o.st.length
    compare_state(g.ctx, 0, o.st)
    g.ctx.close()


# -------------------------------------------------- full-size workloads
def test_50k_single_layer_all_steps(kvo):
    """The 50K single-layer workload, all 1,024 steps, in the launch shape the
    benchmark times: selections compared every step, rows every 64th step,
    full state at the end."""
    w = W.K50
    g = GpuLayerRun(w, 0)
    o = OracleLayerRun(w, 0)
    for step in range(w.steps):
        np.testing.assert_array_equal(g.step(step), o.step(step))
        if step % 64 == 0 or step == w.steps - 1:
            np.testing.assert_array_equal(g.rows(), o.last.rows)
    compare_state(g.ctx, 0, o.st)
    s = g.ctx.stats(0)
    assert s["hits"] + s["misses"] == w.steps * w.k
    g.ctx.close()


def test_1m_cold_stress_sampled(kvo):
    """1M positions, bf16 output on: one layer's first 6 steps, every output."""
    w = W.M1.scaled(steps=6)
    g = GpuLayerRun(w, 3)
    o = OracleLayerRun(w, 3)
    for step in range(w.steps):
        np.testing.assert_array_equal(g.step(step), o.step(step))
        np.testing.assert_array_equal(g.rows(), o.last.rows)
        np.testing.assert_array_equal(g.bf16(), o.last.bf16)
    compare_state(g.ctx, 0, o.st, check_hot=False)
    g.ctx.close()


def test_stack_layers_share_selection(kvo):
    """Full-stack layout in one context: layers 0-3 share layer 0's selection,
    each keeps its own history and hot cache."""
    import torch
    w = W.STACK.scaled(layers=4, steps=24)
    ctx = kvo.Context(4, w.history_cap, w.hot_rows)
    gs = [GpuLayerRun(w, l, ctx=ctx, ctx_layer=l) for l in range(4)]
    os_ = [OracleLayerRun(w, l) for l in range(4)]
    for step in range(w.steps):
        idx = gs[0].step(step)                       # layer 0 selects
        oidx = os_[0].step(step)
        np.testing.assert_array_equal(idx, oidx)
        idx_d = torch.from_numpy(idx).cuda()
        for l in range(1, 4):
            for a in range(w.appends_per_step):
                pos = w.n0 + step
                ctx.append_rows(l, gs[l].new_rows[pos - w.n0:pos - w.n0 + 1])
            ctx.resolve_gather(l, idx_d, gs[l].out_rows)
            os_[l].step(step, idx_override=oidx)
            if step % 8 == 7:
                np.testing.assert_array_equal(gs[l].rows(), os_[l].last.rows)
    for l in range(4):
        compare_state(ctx, l, os_[l].st)
    ctx.close()


# ------------------------------------------------------------ arguments
def test_argument_errors_change_nothing(kvo):
    import torch
    ctx = kvo.Context(2, 100, 8)
    ctx.append_rows(0, np.zeros((10, O.ROW_BYTES), np.uint8))
    idx = torch.arange(9, dtype=torch.int32, device="cuda")
    out = torch.empty((9, O.ROW_BYTES), dtype=torch.uint8, device="cuda")
    with pytest.raises(kvo.KvoError):
        ctx.resolve_gather(0, idx, out)                  # k > hot_rows
    with pytest.raises(kvo.KvoError):
        ctx.resolve_gather(2, idx[:4], out[:4])          # bad layer
    with pytest.raises(kvo.KvoError):
        ctx.select_topk(torch.zeros(5, device="cuda"), 6)
    with pytest.raises(kvo.KvoError):
        ctx.append_rows(1, np.zeros((101, O.ROW_BYTES), np.uint8))
    assert ctx.history_length(1) == 0
    d = ctx.dump_layer(0)
    assert d["step"] == 0 and (d["slot2pos"] == -1).all()
    ctx.close()


def test_timed_out_copy_makes_the_context_refuse_launches(kvo):
    """A bounded wait that gave up is reported once by kvo_sync; when its
    second wait gave up too (a bulk copy may still land), the context
    refuses every later launch.  The status bits are raised by the test hook,
    as the kernel would raise them: no wait is made to run out."""
    import torch
    ctx = kvo.Context(1, 100, 16)
    ctx.append_rows(0, np.zeros((50, O.ROW_BYTES), np.uint8))
    idx = torch.arange(8, dtype=torch.int32, device="cuda")
    out = torch.empty((8, O.ROW_BYTES), dtype=torch.uint8, device="cuda")
    ctx.raise_status(4)                                  # a wait gave up, its second wait did not
    assert ctx.sync() == kvo.KVO_ETIMEDOUT
    assert ctx.sync() == 0                               # reported once
    ctx.resolve_gather(0, idx, out)                      # still usable
    assert ctx.sync() == 0
    ctx.raise_status(4 | 8)                              # the second wait gave up too
    assert ctx.sync() == kvo.KVO_ETIMEDOUT
    with pytest.raises(kvo.KvoError):
        ctx.resolve_gather(0, idx, out)
    with pytest.raises(kvo.KvoError):
        ctx.append_rows(0, np.zeros((1, O.ROW_BYTES), np.uint8))
    ctx.close()


def test_touch_history_changes_nothing(kvo):
    """kvo_touch_history reads one piece per 4 KiB of every layer's history
    and changes no state: the maps before and after are equal, and the next
    step still equals the oracle's."""
    w = W.TINY.scaled(steps=3)
    ctx = kvo.Context(2, w.history_cap, w.hot_rows)
    g = GpuLayerRun(w, 0, ctx=ctx, ctx_layer=0)
    o = OracleLayerRun(w, 0)
    for step in range(2):
        np.testing.assert_array_equal(g.step(step), o.step(step))
    before = ctx.dump_layer(0)
    ctx.touch_history()                                  # every layer (layer 1 is empty)
    ctx.touch_history(0)
    assert ctx.sync() == 0
    after = ctx.dump_layer(0)
    for key in ("pos2slot", "slot2pos", "last_use", "hot"):
        np.testing.assert_array_equal(before[key], after[key])
    np.testing.assert_array_equal(g.step(2), o.step(2))
    np.testing.assert_array_equal(g.rows(), o.last.rows)
    with pytest.raises(kvo.KvoError):
        ctx.touch_history(2)
    ctx.close()


# ------------------------------------------------ fused decode step
@pytest.mark.parametrize("appends", [0, 2])
def test_decode_step_tiny_full_parity(kvo, appends):
    """One launch per step (append + select + resolve) equals the oracle
    step by step: selections, rows, bf16, eviction order, maps."""
    w = W.TINY.scaled(appends_per_step=appends)
    g = GpuLayerRun(w, 0, want_bf16=True, fused=True)
    o = OracleLayerRun(w, 0, want_bf16=True)
    g.ctx.record_evictions(True)
    for step in range(w.steps):
        np.testing.assert_array_equal(g.step(step), o.step(step))
        np.testing.assert_array_equal(g.rows(), o.last.rows)
        np.testing.assert_array_equal(g.bf16(), o.last.bf16)
        assert g.ctx.evictions(0) == o.last.evictions
        compare_state(g.ctx, 0, o.st)
    assert g.ctx.history_length(0) == o.st.length
    assert g.ctx.sync() == 0
    g.ctx.close()


@pytest.mark.parametrize("cluster", [2, 4, 8])
@pytest.mark.parametrize("fused", [False, True])
def test_smaller_clusters_full_parity(kvo, monkeypatch, cluster, fused):
    """Every cluster size the launcher may pick (KVO_MAX_CLUSTER caps it):
    one CTA keeps the LRU order, the others split the selection."""
    monkeypatch.setenv("KVO_MAX_CLUSTER", str(cluster))
    w = W.TINY.scaled(appends_per_step=1, steps=12)
    g = GpuLayerRun(w, 0, want_bf16=True, fused=fused)
    o = OracleLayerRun(w, 0, want_bf16=True)
    g.ctx.record_evictions(True)
    for step in range(w.steps):
        np.testing.assert_array_equal(g.step(step), o.step(step))
        np.testing.assert_array_equal(g.rows(), o.last.rows)
        np.testing.assert_array_equal(g.bf16(), o.last.bf16)
        assert g.ctx.evictions(0) == o.last.evictions
        compare_state(g.ctx, 0, o.st)
    assert g.ctx.sync() == 0
    g.ctx.close()


def test_decode_step_50k_all_steps(kvo):
    """The benchmark's configuration: 50K single layer, 1,024 fused steps."""
    w = W.K50
    g = GpuLayerRun(w, 0, fused=True)
    o = OracleLayerRun(w, 0)
    for step in range(w.steps):
        np.testing.assert_array_equal(g.step(step), o.step(step))
        if step % 64 == 0 or step == w.steps - 1:
            np.testing.assert_array_equal(g.rows(), o.last.rows)
    compare_state(g.ctx, 0, o.st)
    g.ctx.close()


def test_decode_step_1m_sampled(kvo):
    """1M positions (scores streamed, not resident), bf16 on, fused steps."""
    w = W.M1.scaled(steps=4)
    g = GpuLayerRun(w, 5, fused=True)
    o = OracleLayerRun(w, 5)
    for step in range(w.steps):
        np.testing.assert_array_equal(g.step(step), o.step(step))
        np.testing.assert_array_equal(g.rows(), o.last.rows)
        np.testing.assert_array_equal(g.bf16(), o.last.bf16)
    compare_state(g.ctx, 0, o.st, check_hot=False)
    g.ctx.close()


def test_decode_step_selects_rows_appended_in_the_same_step(kvo):
    """Increasing scores put the rows appended by this very call into the
    selection: they are misses read from the device copy, and equal the
    oracle's history rows."""
    import torch
    n0, r, k, H = 3000, 40, 64, 128
    hist = np.random.default_rng(3).integers(0, 256, size=(n0 + 5 * r, O.ROW_BYTES), dtype=np.uint8)
    ctx = kvo.Context(1, n0 + 5 * r, H)
    ctx.append_rows(0, hist[:n0])
    st = O.LayerState(n0 + 5 * r, H)
    st.append(hist[:n0])
    out = torch.empty((k, O.ROW_BYTES), dtype=torch.uint8, device="cuda")
    for step in range(5):
        lo = n0 + step * r
        new = torch.from_numpy(hist[lo:lo + r]).cuda()
        scores = np.arange(lo + r, dtype=np.float32)
        idx = ctx.decode_step(0, new, torch.from_numpy(scores).cuda(), k, out_rows=out).cpu().numpy()
        st.append(hist[lo:lo + r])
        oidx = O.select_topk(scores, k)
        res = O.resolve_gather(st, oidx)
        np.testing.assert_array_equal(idx, oidx)
        np.testing.assert_array_equal(out.cpu().numpy(), res.rows)
    compare_state(ctx, 0, st)
    ctx.close()


def test_decode_step_rejects_host_rows_and_bad_sizes(kvo):
    import torch
    ctx = kvo.Context(1, 100, 16)
    ctx.append_rows(0, np.zeros((50, O.ROW_BYTES), np.uint8))
    scores = torch.zeros(50, device="cuda")
    out = torch.empty((8, O.ROW_BYTES), dtype=torch.uint8, device="cuda")
    host_rows = torch.zeros((1, O.ROW_BYTES), dtype=torch.uint8)
    with pytest.raises(ValueError):
        ctx.decode_step(0, host_rows, scores, 8, out_rows=out)      # binding refuses CPU tensors
    with pytest.raises(kvo.KvoError):
        ctx.decode_step(0, None, scores, 17, out_rows=out)          # k > hot_rows
    with pytest.raises(kvo.KvoError):
        ctx.decode_step(0, torch.zeros((51, O.ROW_BYTES), dtype=torch.uint8, device="cuda"), scores, 8,
                        out_rows=out)                               # past history_cap
    assert ctx.history_length(0) == 50
    ctx.close()


@pytest.mark.parametrize("pinned", [True, False])
def test_decode_step_host_matches_device_buffers(kvo, pinned):
    """kvo_decode_step_host gives the same selections, rows, bf16 rows and
    layer state as kvo_decode_step on device tensors, step for step (appends,
    carry-over, bf16 on): pinned CPU tensors are read and written in place by
    the kernel, pageable ones go through the context's staging."""
    import torch
    pin = (lambda t: t.pin_memory()) if pinned else (lambda t: t)
    w = W.K50.scaled(steps=12)
    ctxs = [kvo.Context(1, w.history_cap, w.hot_rows) for _ in range(2)]
    for c in ctxs:
        c.append_rows(0, W.rows(w, 0, 0, w.n0))
    extra = W.rows(w, 0, w.n0, w.history_cap - w.n0)
    k = w.k
    d_idx = torch.empty(k, dtype=torch.int32, device="cuda")
    d_out = torch.empty((k, O.ROW_BYTES), dtype=torch.uint8, device="cuda")
    d_bf = torch.empty((k, O.DEQUANT_VALUES), dtype=torch.int16, device="cuda")
    h_idx = pin(torch.empty(k, dtype=torch.int32))
    h_out = pin(torch.empty((k, O.ROW_BYTES), dtype=torch.uint8))
    h_bf = pin(torch.empty((k, O.DEQUANT_VALUES), dtype=torch.int16))
    prev = None
    for step in range(w.steps):
        n = w.n_at(step)
        sc = W.apply_carry(W.base_scores(w, 0, step, n), prev, W.carry_draw(w, 0, step), w.carry_boost)
        row = extra[step:step + 1]
        ctxs[0].decode_step(0, torch.from_numpy(row).cuda(), torch.from_numpy(sc).cuda(), k, d_idx, d_out, d_bf)
        ctxs[1].decode_step_host(0, pin(torch.from_numpy(row)), pin(torch.from_numpy(sc)), k, h_idx, h_out, h_bf)
        assert ctxs[0].sync() == kvo.KVO_OK and ctxs[1].sync() == kvo.KVO_OK
        np.testing.assert_array_equal(h_idx.numpy(), d_idx.cpu().numpy())
        np.testing.assert_array_equal(h_out.numpy(), d_out.cpu().numpy())
        np.testing.assert_array_equal(h_bf.numpy(), d_bf.cpu().numpy())
        np.testing.assert_array_equal(h_idx.numpy(), O.select_topk(sc, k))
        prev = h_idx.numpy().copy()
    a, b = (c.dump_layer(0) for c in ctxs)
    for key in ("pos2slot", "slot2pos", "last_use", "hot"):
        np.testing.assert_array_equal(a[key], b[key])
    assert ctxs[0].stats(0) == ctxs[1].stats(0)
    assert ctxs[1].history_length(0) == w.n0 + w.steps
    np.testing.assert_array_equal(ctxs[1].read_history(0, w.n0, w.steps), extra[:w.steps])
    for c in ctxs:
        c.close()


def test_decode_step_host_rejects_device_buffers_and_bad_sizes(kvo):
    import ctypes
    import torch
    ctx = kvo.Context(1, 100, 16)
    ctx.append_rows(0, np.zeros((50, O.ROW_BYTES), np.uint8))
    sc = torch.zeros(50).pin_memory()
    idx = torch.empty(8, dtype=torch.int32).pin_memory()
    out = torch.empty((8, O.ROW_BYTES), dtype=torch.uint8).pin_memory()
    with pytest.raises(ValueError):
        ctx.decode_step_host(0, None, sc.cuda(), 8, idx, out)       # binding refuses CUDA tensors
    lib = kvo.lib()
    d_sc = sc.cuda()
    rc = lib.kvo_decode_step_host(ctypes.c_void_p(ctx.handle), 0, None, 0, ctypes.c_void_p(d_sc.data_ptr()), 50, 8,
                                  ctypes.c_void_p(idx.data_ptr()), ctypes.c_void_p(out.data_ptr()), None, None)
    assert rc == kvo.KVO_EINVAL                                       # device scores refused by the library too
    with pytest.raises(kvo.KvoError):
        ctx.decode_step_host(0, None, sc, 17, torch.empty(17, dtype=torch.int32), out)   # k > hot_rows
    with pytest.raises(kvo.KvoError):
        ctx.decode_step_host(0, torch.zeros((51, O.ROW_BYTES), dtype=torch.uint8), sc, 8, idx, out)  # past cap
    with pytest.raises(kvo.KvoError):
        ctx.decode_step_host(0, None, sc, 8, idx, None, None)        # no output
    assert ctx.history_length(0) == 50
    assert ctx.stats(0)["steps"] == 0
    ctx.close()


def test_misaligned_scores_and_idx_are_refused(kvo):
    """fp32 scores and int32 positions must be 4-byte aligned: every call
    that takes them returns KVO_EINVAL for a misaligned pointer and changes
    nothing."""
    import ctypes
    import torch
    ctx = kvo.Context(1, 100, 16)
    ctx.append_rows(0, np.zeros((50, O.ROW_BYTES), np.uint8))
    buf = torch.zeros(4096, dtype=torch.uint8, device="cuda")
    base = buf.data_ptr()                              # 256-byte aligned
    out = torch.empty((8, O.ROW_BYTES), dtype=torch.uint8, device="cuda")
    lib = kvo.lib()
    h = ctypes.c_void_p(ctx.handle)
    vp = lambda a: ctypes.c_void_p(a)
    scores_ok, scores_bad = vp(base), vp(base + 2)
    idx_ok, idx_bad = vp(base + 2048), vp(base + 2048 + 1)
    assert lib.kvo_select_topk(h, scores_bad, 50, 8, idx_ok, None) == kvo.KVO_EINVAL
    assert lib.kvo_select_topk(h, scores_ok, 50, 8, idx_bad, None) == kvo.KVO_EINVAL
    assert lib.kvo_select_topk_batch(h, scores_bad, 50, 50, 1, 8, idx_ok, None) == kvo.KVO_EINVAL
    assert lib.kvo_resolve_gather(h, 0, idx_bad, 8, vp(out.data_ptr()), None, None) == kvo.KVO_EINVAL
    assert lib.kvo_resolve_gather_multi(h, 0, idx_bad, 1, 8, vp(out.data_ptr()), None, None) == kvo.KVO_EINVAL
    assert lib.kvo_decode_step(h, 0, None, 0, scores_bad, 50, 8, idx_ok, vp(out.data_ptr()), None,
                               None) == kvo.KVO_EINVAL
    assert lib.kvo_decode_step(h, 0, None, 0, scores_ok, 50, 8, idx_bad, vp(out.data_ptr()), None,
                               None) == kvo.KVO_EINVAL
    bad = kvo.make_layer_tasks([{"layer": 0, "idx": torch.empty(8, dtype=torch.int32, device="cuda"),
                                 "out_rows": out}])
    bad[0].idx = idx_bad
    with pytest.raises(kvo.KvoError):
        ctx.decode_layers_prepared(bad, 8)
    assert ctx.sync() == kvo.KVO_OK
    assert ctx.history_length(0) == 50 and ctx.stats(0)["steps"] == 0
    ctx.close()


# ------------------------------------------------ multi-query rounds (MTP)
def _mtp_run(kvo, w, steps, check_every=1, want_bf16=False):
    """Each step: append, nq top-K selections (row 0 from the score model,
    rows 1.. = row 0 + noise), one multi-query round; GPU vs oracle."""
    import torch
    nq, k = w.queries, w.k
    ctx = kvo.Context(1, w.history_cap, w.hot_rows)
    ctx.append_rows(0, W.rows(w, 0, 0, w.n0))
    ctx.record_evictions(True)
    st = O.LayerState(w.history_cap, w.hot_rows)
    st.append(W.rows(w, 0, 0, w.n0))
    extra = W.rows(w, 0, w.n0, w.history_cap - w.n0) if w.history_cap > w.n0 else None
    out = torch.empty((nq * k, O.ROW_BYTES), dtype=torch.uint8, device="cuda")
    outb = torch.empty((nq * k, O.DEQUANT_VALUES), dtype=torch.int16, device="cuda") if want_bf16 else None
    idx = torch.empty((nq, k), dtype=torch.int32, device="cuda")
    prev = None
    for step in range(steps):
        for a in range(w.appends_per_step):
            pos = w.n0 + step * w.appends_per_step + a
            row = extra[pos - w.n0:pos - w.n0 + 1]
            ctx.append_rows(0, torch.from_numpy(row).cuda())
            st.append(row)
        row0 = W.apply_carry(W.base_scores(w, 0, step), prev, W.carry_draw(w, 0, step), w.carry_boost)
        rows = [row0] + [W.query_scores(w, 0, step, q, row0) for q in range(1, nq)]
        ctx.select_topk_batch(torch.from_numpy(np.stack(rows)).cuda(), k, idx=idx)
        ctx.resolve_gather_multi(0, idx, out, outb)
        want = np.stack([O.select_topk(r, k) for r in rows])
        res = O.resolve_gather_multi(st, want, want_bf16=want_bf16)
        np.testing.assert_array_equal(idx.cpu().numpy(), want)
        assert ctx.evictions(0) == res.evictions, step
        if step % check_every == 0 or step == steps - 1:
            np.testing.assert_array_equal(out.cpu().numpy(), res.rows)
            if want_bf16:
                assert_bf16_equal(outb.cpu().numpy(), res.bf16)
        prev = want[0]
    assert ctx.sync() == 0
    compare_state(ctx, 0, st)
    s = ctx.stats(0)
    assert s["rows_out"] == steps * nq * k and s["misses"] >= s["unique_misses"]
    ctx.close()


def test_multi_query_rounds_tiny(kvo):
    _mtp_run(kvo, W.TINY.scaled(queries=4, appends_per_step=1), 16, want_bf16=True)


def test_multi_query_rounds_50k(kvo):
    """The MTP bench workload: 4 query rows of 2,048 per round, 120 rounds."""
    _mtp_run(kvo, W.K50_MTP.scaled(steps=120), 120, check_every=10)


def test_multi_query_argument_errors(kvo):
    import torch
    ctx = kvo.Context(1, 20_000, 8192)
    ctx.append_rows(0, np.zeros((20_000, O.ROW_BYTES), np.uint8))
    out = torch.empty((8193, O.ROW_BYTES), dtype=torch.uint8, device="cuda")
    with pytest.raises(kvo.KvoError):                  # nq * k > KVO_MAX_ROUND
        ctx.resolve_gather_multi(0, torch.zeros((3, 2731), dtype=torch.int32, device="cuda"), out)
    with pytest.raises(kvo.KvoError):                  # k > KVO_MAX_K
        ctx.resolve_gather_multi(0, torch.zeros((1, 4097), dtype=torch.int32, device="cuda"), out)
    ctx.resolve_gather_multi(0, torch.arange(8192, dtype=torch.int32, device="cuda").view(4, 2048), out[:8192])
    assert ctx.sync() == 0
    assert ctx.stats(0)["unique_misses"] == 8192
    small = kvo.Context(1, 100, 16)
    small.append_rows(0, np.zeros((100, O.ROW_BYTES), np.uint8))
    with pytest.raises(kvo.KvoError):                  # nq * k > hot_rows
        small.resolve_gather_multi(0, torch.zeros((2, 9), dtype=torch.int32, device="cuda"), out[:18])
    ctx.close()
    small.close()


# ------------------------------------------------ circular replacement
@pytest.mark.parametrize("fused", [False, True])
def test_circular_policy_tiny_full_parity(kvo, fused):
    w = W.TINY.scaled(appends_per_step=1)
    g = GpuLayerRun(w, 0, want_bf16=True, fused=fused, policy=kvo.POLICY_CIRCULAR)
    o = OracleLayerRun(w, 0, want_bf16=True, policy="circular")
    g.ctx.record_evictions(True)
    for step in range(w.steps):
        np.testing.assert_array_equal(g.step(step), o.step(step))
        np.testing.assert_array_equal(g.rows(), o.last.rows)
        np.testing.assert_array_equal(g.bf16(), o.last.bf16)
        assert g.ctx.evictions(0) == o.last.evictions
        compare_state(g.ctx, 0, o.st)
        assert g.ctx.counters(0)["hand"] == o.st.hand
    assert g.ctx.sync() == 0
    g.ctx.close()


@pytest.mark.parametrize("seed,H,n,k,dup", [(1, 16, 40, 16, 0.3), (3, 1024, 5000, 256, 0.2),
                                           (6, 32_768, 60_000, 4096, 0.1), (8, 4096, 9000, 3000, 0.0)])
def test_circular_policy_random_selections(kvo, seed, H, n, k, dup):
    """The hand wraps many times; duplicates and arbitrary order."""
    import torch
    g = np.random.default_rng(seed)
    hist = g.integers(0, 256, size=(n, O.ROW_BYTES), dtype=np.uint8)
    ctx = kvo.Context(1, n, H)
    ctx.set_policy(kvo.POLICY_CIRCULAR)
    ctx.append_rows(0, hist)
    ctx.record_evictions(True)
    st = O.LayerState(n, H, policy="circular")
    st.append(hist)
    out = torch.empty((k, O.ROW_BYTES), dtype=torch.uint8, device="cuda")
    for step in range(20):
        idx = W.random_idx(seed * 100 + step, n if step % 3 else min(n, 2 * H), k, dup, 0)
        ctx.resolve_gather(0, torch.from_numpy(idx).cuda(), out)
        res = O.resolve_gather(st, idx)
        np.testing.assert_array_equal(out.cpu().numpy(), res.rows)
        assert ctx.evictions(0) == res.evictions, step
        assert ctx.counters(0)["hand"] == st.hand
    assert ctx.sync() == 0
    compare_state(ctx, 0, st)
    with pytest.raises(kvo.KvoError):                  # the policy is fixed once resolves ran
        ctx.set_policy(kvo.POLICY_LRU)
    ctx.close()


def test_circular_policy_50k_all_steps(kvo):
    w = W.K50
    g = GpuLayerRun(w, 0, fused=True, policy=kvo.POLICY_CIRCULAR)
    o = OracleLayerRun(w, 0, policy="circular")
    for step in range(w.steps):
        np.testing.assert_array_equal(g.step(step), o.step(step))
        if step % 64 == 0 or step == w.steps - 1:
            np.testing.assert_array_equal(g.rows(), o.last.rows)
    compare_state(g.ctx, 0, o.st)
    assert g.ctx.counters(0)["hand"] == o.st.hand
    g.ctx.close()


# ------------------------------------------------------- recent ring
@pytest.mark.parametrize("fused", [False, True])
@pytest.mark.parametrize("appends", [1, 5])
def test_recent_ring_parity(kvo, fused, appends):
    """Device appends wait in a 128-row ring; 64-row batches reach RAM.
    Rows, evictions and maps equal the oracle's; RAM holds exactly the
    oracle's first ram_len rows; host_bytes counts only RAM reads."""
    w = W.TINY.scaled(appends_per_step=appends, steps=40)
    g = GpuLayerRun(w, 0, want_bf16=True, fused=fused, ring=128)
    o = OracleLayerRun(w, 0, want_bf16=True, ring=128)
    g.ctx.record_evictions(True)
    host_reads = 0
    for step in range(w.steps):
        np.testing.assert_array_equal(g.step(step), o.step(step))
        np.testing.assert_array_equal(g.rows(), o.last.rows)
        np.testing.assert_array_equal(g.bf16(), o.last.bf16)
        assert g.ctx.evictions(0) == o.last.evictions
        assert g.ctx.ram_length(0) == o.st.ram_len
        host_reads += o.last.host_reads
        if step % 8 == 7:
            compare_state(g.ctx, 0, o.st)
            ram = o.st.ram_len
            np.testing.assert_array_equal(g.ctx.read_history(0, 0, ram), o.st.history[:ram])
    assert g.ctx.stats(0)["host_bytes"] == host_reads * O.ROW_BYTES
    assert host_reads < g.ctx.stats(0)["misses"]     # recent rows came from the ring
    g.ctx.flush_ring(0)
    n = o.st.length
    assert g.ctx.ram_length(0) == n
    np.testing.assert_array_equal(g.ctx.read_history(0, 0, n), o.st.history[:n])
    assert g.ctx.sync() == 0
    g.ctx.close()


def test_recent_ring_host_rows_flush_first(kvo):
    import torch
    ctx = kvo.Context(1, 2000, 64)
    ctx.set_recent_ring(128)
    st = O.LayerState(2000, 64, ring_rows=128)
    rng = np.random.default_rng(3)
    base = rng.integers(0, 256, size=(500, O.ROW_BYTES), dtype=np.uint8)
    ctx.append_rows(0, base)
    st.append(base)
    for chunk in (10, 30, 50, 7):                       # device rows
        rows = rng.integers(0, 256, size=(chunk, O.ROW_BYTES), dtype=np.uint8)
        ctx.append_rows(0, torch.from_numpy(rows).cuda())
        st.append(rows, from_device=True)
        assert ctx.ram_length(0) == st.ram_len
    host = rng.integers(0, 256, size=(5, O.ROW_BYTES), dtype=np.uint8)
    ctx.append_rows(0, host)                            # host rows: the ring goes first
    st.append(host)
    assert ctx.ram_length(0) == st.ram_len == st.length
    np.testing.assert_array_equal(ctx.read_history(0, 0, st.length), st.history[:st.length])
    idx = torch.arange(st.length - 64, st.length, dtype=torch.int32, device="cuda")
    out = torch.empty((64, O.ROW_BYTES), dtype=torch.uint8, device="cuda")
    ctx.resolve_gather(0, idx, out)
    np.testing.assert_array_equal(out.cpu().numpy(), st.history[st.length - 64:st.length])
    with pytest.raises(kvo.KvoError):                   # more than ring - batch rows in one call
        ctx.append_rows(0, torch.zeros((65, O.ROW_BYTES), dtype=torch.uint8, device="cuda"))
    with pytest.raises(kvo.KvoError):                   # the ring is fixed once rows exist
        ctx.set_recent_ring(256)
    assert ctx.sync() == 0
    ctx.close()


def test_recent_ring_50k_fused(kvo):
    """The benchmark's fused path with a 1,024-row ring, 300 steps: the same
    oracle as the separate calls, RAM length and RAM reads included."""
    w = W.K50.scaled(steps=300)
    g = GpuLayerRun(w, 0, fused=True, ring=1024)
    o = OracleLayerRun(w, 0, ring=1024)
    host_reads = 0
    for step in range(w.steps):
        np.testing.assert_array_equal(g.step(step), o.step(step))
        assert g.ctx.ram_length(0) == o.st.ram_len
        host_reads += o.last.host_reads
        if step % 50 == 0 or step == w.steps - 1:
            np.testing.assert_array_equal(g.rows(), o.last.rows)
            assert g.ctx.stats(0)["host_bytes"] == host_reads * O.ROW_BYTES, step
    compare_state(g.ctx, 0, o.st)
    ram = o.st.ram_len
    np.testing.assert_array_equal(g.ctx.read_history(0, ram - 3000, 3000), o.st.history[ram - 3000:ram])
    g.ctx.close()


# ------------------------------------------------ staged (TMA) gather
GATHERS = [(0, 0), (1, 0), (2, 10)]   # loads; staged always; staged for CTAs with at least 10 % misses


@pytest.mark.parametrize("gather", GATHERS)
@pytest.mark.parametrize("fused", [False, True])
def test_staged_gather_tiny_full_parity(kvo, gather, fused):
    w = W.TINY.scaled(appends_per_step=2)
    g = GpuLayerRun(w, 0, want_bf16=True, fused=fused, gather=gather)
    o = OracleLayerRun(w, 0, want_bf16=True)
    g.ctx.record_evictions(True)
    for step in range(w.steps):
        np.testing.assert_array_equal(g.step(step), o.step(step))
        np.testing.assert_array_equal(g.rows(), o.last.rows)
        np.testing.assert_array_equal(g.bf16(), o.last.bf16)
        assert g.ctx.evictions(0) == o.last.evictions
        compare_state(g.ctx, 0, o.st)
    assert g.ctx.sync() == 0
    g.ctx.close()


@pytest.mark.parametrize("gather", GATHERS)
@pytest.mark.parametrize("seed,H,n,k,dup,bad", [(1, 16, 40, 16, 0.3, 2), (3, 1024, 5000, 256, 0.2, 5),
                                               (5, 4096, 70_000, 2048, 0.4, 3), (6, 32_768, 60_000, 4096, 0.1, 1)])
def test_staged_gather_random_selections(kvo, gather, seed, H, n, k, dup, bad):
    """Duplicates, invalid entries (zero rows), host misses by TMA; bf16 only
    on odd steps (the fills then come from shared memory, not the output)."""
    import torch
    g = np.random.default_rng(seed)
    hist = g.integers(0, 256, size=(n, O.ROW_BYTES), dtype=np.uint8)
    ctx = kvo.Context(1, n, H)
    ctx.set_gather_mode(*gather)
    ctx.append_rows(0, hist)
    ctx.record_evictions(True)
    st = O.LayerState(n, H)
    st.append(hist)
    out = torch.empty((k, O.ROW_BYTES), dtype=torch.uint8, device="cuda")
    outb = torch.empty((k, O.DEQUANT_VALUES), dtype=torch.int16, device="cuda")
    for step in range(10):
        idx = W.random_idx(seed * 100 + step, n if step % 3 else min(n, 2 * H), k, dup, bad if step % 2 else 0)
        rows_out = None if step % 2 else out
        ctx.resolve_gather(0, torch.from_numpy(idx).cuda(), rows_out, outb)
        res = O.resolve_gather(st, idx, want_bf16=True)
        if rows_out is not None:
            np.testing.assert_array_equal(out.cpu().numpy(), res.rows)
        assert_bf16_equal(outb.cpu().numpy(), res.bf16)
        assert ctx.evictions(0) == res.evictions
        assert ctx.sync() == (kvo.KVO_ERANGE if res.invalid else 0)
    compare_state(ctx, 0, st)
    ctx.close()


@pytest.mark.parametrize("gather", GATHERS)
def test_staged_gather_50k_fused_with_ring(kvo, gather):
    w = W.K50.scaled(steps=200)
    g = GpuLayerRun(w, 0, fused=True, ring=1024, gather=gather)
    o = OracleLayerRun(w, 0, ring=1024)
    host_reads = 0
    for step in range(w.steps):
        np.testing.assert_array_equal(g.step(step), o.step(step))
        assert g.ctx.ram_length(0) == o.st.ram_len
        host_reads += o.last.host_reads
        if step % 25 == 0 or step == w.steps - 1:
            np.testing.assert_array_equal(g.rows(), o.last.rows)
    assert g.ctx.stats(0)["host_bytes"] == host_reads * O.ROW_BYTES
    compare_state(g.ctx, 0, o.st)
    assert g.ctx.sync() == 0
    g.ctx.close()


# ------------------------------------------------ batched layers (one launch)
def _run_layers(kvo, w, steps, *, policy=0, ring=0, gather=None, full_check=lambda step: True, one_call=True,
                miss=None):
    """Drives a workload through kvo_decode_layers: per step one call with
    every layer, a reusing layer naming its source layer's idx (the way the
    benchmark does), or with one_call=False a call with the selecting layers
    and then one with the reusing layers, each on its own copy of the
    selection.  Every layer's selection is
    compared every step; rows, bf16 rows and eviction order of every layer
    on the steps `full_check` accepts; the maps and hot rows of every layer,
    the RAM length and the RAM reads at the end."""
    import torch
    L = w.layers
    ctx = kvo.Context(L, w.history_cap, w.hot_rows)
    if policy:
        ctx.set_policy(policy)
    if ring:
        ctx.set_recent_ring(ring)
    if gather:
        ctx.set_gather_mode(*gather)
    if miss:
        ctx.set_miss_fetch(*miss)
    ctx.record_evictions(True)
    pol = "circular" if policy else "lru"
    orc = [OracleLayerRun(w, l, policy=pol, ring=ring) for l in range(L)]
    a = w.appends_per_step
    new = [torch.from_numpy(W.rows(w, l, w.n0, w.history_cap - w.n0)).cuda() if a else None for l in range(L)]
    for l in range(L):
        ctx.append_rows(l, W.rows(w, l, 0, w.n0))
    idx = [torch.empty(w.k, dtype=torch.int32, device="cuda") for _ in range(L)]
    out = [torch.empty((w.k, O.ROW_BYTES), dtype=torch.uint8, device="cuda") for _ in range(L)]
    outb = [torch.empty((w.k, O.DEQUANT_VALUES), dtype=torch.int16, device="cuda") for _ in range(L)] if w.bf16 else None
    prev = {}
    host_reads = [0] * L
    for step in range(steps):
        sel_tasks, reuse_tasks = [], []
        for l in range(L):
            t = {"layer": l, "idx": idx[w.source_layer(l) if one_call else l], "out_rows": out[l]}
            if outb is not None:
                t["out_bf16"] = outb[l]
            if a:
                t["new_rows"] = new[l][step * a:(step + 1) * a]
            if l in w.selecting_layers():
                s = W.apply_carry(W.base_scores(w, l, step), prev.get(l), W.carry_draw(w, l, step), w.carry_boost)
                t["scores"] = torch.from_numpy(s).cuda()
                sel_tasks.append(t)
            else:
                reuse_tasks.append(t)
        if one_call:
            ctx.decode_layers(sel_tasks + reuse_tasks, w.k)
        else:
            ctx.decode_layers(sel_tasks, w.k)
            for t in reuse_tasks:                       # the source layer's selection, copied in stream order
                t["idx"].copy_(idx[w.source_layer(t["layer"])])
            if reuse_tasks:
                ctx.decode_layers(reuse_tasks, w.k)
        full = full_check(step)
        for l in range(L):
            src = w.source_layer(l)
            if l == src:
                want = orc[l].step(step)
                np.testing.assert_array_equal(idx[l].cpu().numpy(), want)
                prev[l] = want
            elif not one_call:
                orc[l].step(step, idx_override=prev[src])
                np.testing.assert_array_equal(idx[l].cpu().numpy(), prev[src])
            else:
                orc[l].step(step, idx_override=prev[src])
            host_reads[l] += orc[l].last.host_reads
            if full:
                np.testing.assert_array_equal(out[l].cpu().numpy(), orc[l].last.rows)
                if outb is not None:
                    assert_bf16_equal(outb[l].cpu().numpy(), orc[l].last.bf16)
                assert ctx.evictions(l) == orc[l].last.evictions, (step, l)
    for l in range(L):
        compare_state(ctx, l, orc[l].st)
        assert ctx.history_length(l) == orc[l].st.length
        assert ctx.ram_length(l) == orc[l].st.ram_len
        assert ctx.stats(l)["host_bytes"] == host_reads[l] * O.ROW_BYTES, l
    assert ctx.sync() == 0
    ctx.close()
    return orc


@pytest.mark.parametrize("one_call", [True, False])
@pytest.mark.parametrize("policy,ring,gather", [(0, 0, None), (1, 128, (1, 0)), (0, 128, None)])
def test_decode_layers_stack_parity(kvo, policy, ring, gather, one_call):
    """Eight layers, selection on layers 0 and 4, reused by the others;
    appends every step; in one call per step or in two.  Every layer equals
    its own oracle: selections, rows, evictions, maps, RAM reads."""
    w = W.STACK.scaled(layers=8, n0=6000, hot_rows=1024, k=256, steps=40, carry=150)
    _run_layers(kvo, w, w.steps, policy=policy, ring=ring, gather=gather, one_call=one_call)


@pytest.mark.parametrize("miss", [(1, 100), (2, 0), (2, 30)])
@pytest.mark.parametrize("policy,ring", [(0, 0), (1, 128), (0, 128)])
def test_decode_layers_batched_miss_fetch(kvo, miss, policy, ring):
    """The misses of the host history fetched by batched copies (always, or
    chosen by the measured miss share): the same oracle as zero-copy loads,
    rows, bf16 rows, evictions, maps and RAM reads included (the recent ring
    and this step's rows still come from device memory)."""
    w = W.STACK.scaled(layers=8, n0=6000, hot_rows=1024, k=256, steps=40, carry=150, bf16=True)
    _run_layers(kvo, w, w.steps, policy=policy, ring=ring, miss=miss)


def test_decode_layers_batched_miss_fetch_1m(kvo):
    """Batched copies on 8 layers of 1M positions with bf16 output: about
    2,000 scattered missing rows per layer and step, one copy each."""
    w = W.M1.scaled(steps=2)
    _run_layers(kvo, w, w.steps, miss=(1, 100))


def test_decode_layers_full_stack_parity(kvo):
    """The 78-layer stack at full size, in the launch shapes the benchmark
    times (20 selecting tasks, then 58 reusing ones; K = 2,048, 32,768 hot
    rows per layer, 50,023-row histories), for 126 steps: the hot caches
    fill up at step 121, so the last steps evict mapped positions.
    Selections of every layer every step; rows, evictions and maps of every
    layer every 16th step and on each of the last six."""
    w = W.STACK.scaled(steps=126)
    orc = _run_layers(kvo, w, w.steps, full_check=lambda step: step % 16 == 15 or step >= 120)
    assert all(any(e[1] >= 0 for e in o.last.evictions) for o in orc)   # real LRU victims on every layer


def test_decode_layers_1m_one_wave_parity(kvo):
    """Eight layers of 1M positions in one launch with bf16 output (the
    1M benchmark's shape): every output, both formats, every step."""
    w = W.M1.scaled(steps=3)
    _run_layers(kvo, w, w.steps)


@pytest.mark.parametrize("seed,H,n,k,dup,bad", [(1, 16, 40, 16, 0.3, 2), (3, 1024, 5000, 256, 0.2, 5),
                                               (5, 4096, 70_000, 2048, 0.4, 3), (7, 4096, 70_000, 2048, 0.0, 0)])
def test_decode_layers_random_idx(kvo, seed, H, n, k, dup, bad):
    """kvo_decode_layers with resolve-only tasks on three layers whose idx is
    in any order, with duplicates (the first occurrence claims the slot,
    later ones read the source) and out-of-range entries (zero rows,
    counted), and one layer whose idx increases (no claims needed); bf16
    rows on odd steps.  Rows, evictions, maps and status equal the oracle's
    on every step."""
    import torch
    L = 4
    g = np.random.default_rng(seed)
    hist = [g.integers(0, 256, size=(n, O.ROW_BYTES), dtype=np.uint8) for _ in range(L)]
    ctx = kvo.Context(L, n, H)
    ctx.record_evictions(True)
    st = []
    for l in range(L):
        ctx.append_rows(l, hist[l])
        st.append(O.LayerState(n, H))
        st[l].append(hist[l])
    out = [torch.empty((k, O.ROW_BYTES), dtype=torch.uint8, device="cuda") for _ in range(L)]
    outb = [torch.empty((k, O.DEQUANT_VALUES), dtype=torch.int16, device="cuda") for _ in range(L)]
    for step in range(10):
        span = n if step % 3 else min(n, 2 * H)
        idx = [W.random_idx(seed * 100 + 10 * step + l, span, k, dup, bad if step % 2 else 0) for l in range(L - 1)]
        idx.append(np.sort(np.random.default_rng(seed + step).choice(span, size=k, replace=False)).astype(np.int32))
        dev = [torch.from_numpy(i).cuda() for i in idx]
        tasks = [{"layer": l, "idx": dev[l], "out_rows": out[l]} for l in range(L)]
        if step % 2:
            for l in range(L):
                tasks[l]["out_bf16"] = outb[l]
        ctx.decode_layers(tasks, k)
        invalid = False
        for l in range(L):
            res = O.resolve_gather(st[l], idx[l], want_bf16=bool(step % 2))
            np.testing.assert_array_equal(out[l].cpu().numpy(), res.rows, err_msg=f"step {step} layer {l}")
            if step % 2:
                assert_bf16_equal(outb[l].cpu().numpy(), res.bf16)
            assert ctx.evictions(l) == res.evictions, (step, l)
            invalid = invalid or bool(res.invalid)
        assert ctx.sync() == (kvo.KVO_ERANGE if invalid else 0)
    for l in range(L):
        compare_state(ctx, l, st[l])
    ctx.close()


def test_decode_layers_more_tasks_than_one_launch_holds(kvo):
    """140 layers in one kvo_decode_layers call: more than the 128 tasks one
    launch takes, so every phase runs as two launches (130 selecting layers:
    two histogram and two selection launches; 140 tasks: two resolve and two
    gather launches).  The last 10 layers reuse the selections of layers
    0-9, made in the other launch.  Selections, rows, evictions and maps
    equal the oracle's over three steps."""
    import torch
    L, n, H, k = 140, 3000, 256, 64
    ctx = kvo.Context(L, n + 8, H)
    ctx.record_evictions(True)
    g = np.random.default_rng(140)
    st = []
    for l in range(L):
        hist = g.integers(0, 256, size=(n, O.ROW_BYTES), dtype=np.uint8)
        ctx.append_rows(l, hist)
        st.append(O.LayerState(n + 8, H))
        st[-1].append(hist)
    sel = list(range(130))                              # layers 130..139 reuse layers 0..9
    src = {l: l if l < 130 else l - 130 for l in range(L)}
    idx = {l: torch.empty(k, dtype=torch.int32, device="cuda") for l in sel}
    out = [torch.empty((k, O.ROW_BYTES), dtype=torch.uint8, device="cuda") for _ in range(L)]
    for step in range(3):
        scores = {l: g.standard_normal(n, dtype=np.float32) for l in sel}
        dev = {l: torch.from_numpy(scores[l]).cuda() for l in sel}
        tasks = []
        for l in range(L):
            t = {"layer": l, "idx": idx[src[l]], "out_rows": out[l]}
            if l in idx:
                t["scores"] = dev[l]
            tasks.append(t)
        ctx.decode_layers(tasks, k)
        want = {l: O.select_topk(scores[l], k) for l in sel}
        for l in sel:
            np.testing.assert_array_equal(idx[l].cpu().numpy(), want[l], err_msg=f"step {step} layer {l}")
        for l in range(L):
            res = O.resolve_gather(st[l], want[src[l]])
            np.testing.assert_array_equal(out[l].cpu().numpy(), res.rows, err_msg=f"step {step} layer {l}")
            assert ctx.evictions(l) == res.evictions, (step, l)
    assert ctx.sync() == 0
    for l in range(L):
        compare_state(ctx, l, st[l])
    ctx.close()


def _selection_kinds(n_scale):
    k = 2048
    crowded = W.random_scores(31, 40_000 * n_scale, "normal")
    crowded[5_000 * n_scale:35_000 * n_scale] = np.float32(1.0)
    return [crowded, W.random_scores(32, 33_001 * n_scale, "special"), W.random_scores(33, 20_000 * n_scale, "coarse"),
            W.random_scores(34, 45_000 * n_scale, "recent"), W.random_scores(35, 12_289 * n_scale, "negzero"),
            W.random_scores(36, k, "normal")]


@pytest.mark.parametrize("n_scale", [1, 16])
def test_decode_layers_selection_score_kinds(kvo, n_scale):
    """One kvo_decode_layers call whose selecting layers hold different
    history lengths and score shapes: a crowded cut bucket (equal scores on
    three quarters of the positions: more keys in and above it than a
    selecting CTA can list, so the selection streams the scores), specials
    (NaN, +-0, +-inf, denormals), a coarse grid, raised recent positions,
    all-negative scores with -0, and k = n.  The lengths differ, so the
    histogram launch has CTAs past some layers' scores; 16x the lengths
    reach 720,000 scores.  Four calls in a row take every way through the
    candidate lists the histogram launch makes from the previous call's cut
    (none yet; used; a cut below them; a cut far above them).  Every
    selection equals the oracle's."""
    import torch
    k = 2048
    cases = _selection_kinds(n_scale)
    L = len(cases)
    ctx = kvo.Context(L, max(sc.size for sc in cases), 4096)
    for l, sc in enumerate(cases):
        ctx.append_rows(l, np.zeros((sc.size, O.ROW_BYTES), np.uint8))
    idx = [torch.empty(k, dtype=torch.int32, device="cuda") for _ in range(L)]
    out = [torch.empty((k, O.ROW_BYTES), dtype=torch.uint8, device="cuda") for _ in range(L)]
    dev = [torch.from_numpy(sc).cuda() for sc in cases]
    lower = [(sc - np.float32(4.0)).astype(np.float32) for sc in cases]
    dev_lower = [torch.from_numpy(sc).cuda() for sc in lower]
    want = [O.select_topk(sc, k) for sc in cases]
    want_lower = [O.select_topk(sc, k) for sc in lower]
    # the second call lists candidates from one bucket below the first's cut
    # and uses them; the third (every score 4 lower) cuts below the listing
    # bucket and filters the scores itself; the fourth lists from far below
    # its cut (more candidates than fit, or many extra ones)
    for rep, (d, wnt) in enumerate([(dev, want), (dev, want), (dev_lower, want_lower), (dev, want)]):
        ctx.decode_layers([{"layer": l, "idx": idx[l], "out_rows": out[l], "scores": d[l]} for l in range(L)], k)
        for l in range(L):
            np.testing.assert_array_equal(idx[l].cpu().numpy(), wnt[l], err_msg=f"call {rep} layer {l}")
    assert ctx.sync() == 0
    ctx.close()


def test_decode_layers_argument_errors(kvo):
    import torch
    ctx = kvo.Context(2, 1000, 64)
    for l in range(2):
        ctx.append_rows(l, np.zeros((500, O.ROW_BYTES), np.uint8))
    i0, i1 = (torch.zeros(16, dtype=torch.int32, device="cuda") for _ in range(2))
    o = torch.empty((16, O.ROW_BYTES), dtype=torch.uint8, device="cuda")
    sc = torch.zeros(500, device="cuda")
    with pytest.raises(kvo.KvoError):                   # the same layer twice
        ctx.decode_layers([{"layer": 0, "idx": i0, "out_rows": o}, {"layer": 0, "idx": i1, "out_rows": o}], 16)
    with pytest.raises(kvo.KvoError):                   # n beyond the history
        ctx.decode_layers([{"layer": 1, "idx": i0, "out_rows": o, "scores": torch.zeros(600, device="cuda")}], 16)
    with pytest.raises(kvo.KvoError):                   # no output
        ctx.decode_layers([{"layer": 1, "idx": i0}], 16)
    ctx.decode_layers([{"layer": 0, "idx": i0, "out_rows": o, "scores": sc},
                       {"layer": 1, "idx": i1, "out_rows": torch.empty_like(o)}], 16)
    assert ctx.sync() == 0
    assert ctx.stats(0)["steps"] == 1 and ctx.stats(1)["steps"] == 1
    ctx.close()
