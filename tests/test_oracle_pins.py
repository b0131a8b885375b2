"""Pins of the CPU oracle against what the pages and the mathematics fix.

None of these checks re-types the oracle's own formula: each compares it with a
value the pages print, a brute-force definition, a library routine, a closed
form or an invariant.
"""
import itertools
import os

import numpy as np
import pytest

from oracle import kvo_oracle as O
from synth import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
UNITS = {"MiB": 1 << 20, "GiB": 1 << 30, "TiB": 1 << 40}


# --------------------------------------------------------------------- sizes
def _golden(name):
    rows = []
    for line in open(os.path.join(GOLDEN, name)):
        line = line.split("|")[0].strip()
        if line and not line.startswith("#"):
            rows.append(line.split())
    return rows


def test_row_is_656_bytes():
    # "512 B of latent data, 16 B of scales, and 128 B of RoPE data: 656 B in total"
    assert (O.LATENT_BYTES, O.SCALE_BYTES, O.ROPE_BYTES, O.ROW_BYTES) == (512, 16, 128, 656)
    assert O.N_GROUPS * O.GROUP == O.LATENT_BYTES and O.SCALE_BYTES == 2 * O.N_GROUPS
    assert O.ROPE_VALUES == 64 and O.DEQUANT_VALUES == 576


@pytest.mark.parametrize("row", _golden("payload_sizes.txt"))
def test_payload_sizes_match_pages(row):
    tokens, layers, replicas, unit, printed, decimals = row
    b = O.mla_payload_bytes(int(tokens), int(layers), int(replicas))
    assert round(b / UNITS[unit], int(decimals)) == float(printed)


def test_payload_sizes_catch_a_wrong_row_size():
    # A row size off by one 16-byte field would miss the printed table.
    b = 50000 * (O.ROW_BYTES - 16)
    assert round(b / UNITS["MiB"], 3) != 31.281


# -------------------------------------------------------------------- top-K
def _brute_topk(scores, k):
    """Rank counting: position p is chosen iff fewer than k positions beat it.

    q beats p when q's score is greater, or equal with q < p.  NaN is below
    everything and equal to NaN; -0 equals +0.
    """
    n = len(scores)

    def beats(q, p):
        a, b = scores[q], scores[p]
        an, bn = np.isnan(a), np.isnan(b)
        if an and bn:
            return q < p
        if an:
            return False
        if bn:
            return True
        if a != b:
            return a > b
        return q < p

    chosen = [p for p in range(n) if sum(beats(q, p) for q in range(n) if q != p) < k]
    return np.array(chosen, np.int32)


@pytest.mark.parametrize("kind", ["normal", "ties", "special"])
@pytest.mark.parametrize("n,k", [(1, 1), (7, 3), (33, 32), (64, 1), (97, 50), (128, 128)])
def test_topk_equals_brute_force(kind, n, k):
    s = W.random_scores(n * 31 + k, n, kind)
    np.testing.assert_array_equal(O.select_topk(s, k), _brute_topk(s, k))


def test_topk_special_cases():
    n = 1000
    assert np.array_equal(O.select_topk(np.full(n, 0.5, np.float32), 10), np.arange(10))
    inc = np.arange(n, dtype=np.float32)
    assert np.array_equal(O.select_topk(inc, 10), np.arange(n - 10, n))
    assert np.array_equal(O.select_topk(W.random_scores(3, n), n), np.arange(n))
    s = np.zeros(8, np.float32)
    s[5] = -0.0
    assert np.array_equal(O.select_topk(s, 3), [0, 1, 2])          # -0 ties with +0
    s = np.array([np.nan, -np.inf, np.nan, 1.0], np.float32)
    assert np.array_equal(O.select_topk(s, 2), [1, 3])               # NaN below -inf
    assert np.array_equal(O.select_topk(s, 3), [0, 1, 3])            # lowest-position NaN next
    with pytest.raises(ValueError):
        O.select_topk(s, 0)
    with pytest.raises(ValueError):
        O.select_topk(s, 5)


def test_topk_threshold_invariant_at_50k_size():
    w = W.K50
    s = W.base_scores(w, 0, 3)
    sel = O.select_topk(s, w.k)
    assert len(sel) == w.k and np.all(np.diff(sel) > 0)
    mask = np.zeros(len(s), bool)
    mask[sel] = True
    lo = s[mask].min()
    assert s[~mask].max() <= lo
    # ties at the threshold go to the lowest positions
    tied_out = np.nonzero((~mask) & (s == lo))[0]
    tied_in = np.nonzero(mask & (s == lo))[0]
    if len(tied_out) and len(tied_in):
        assert tied_in.max() < tied_out.min()


# ------------------------------------------------------------ residency/LRU
def _brute_step(hist, length, H, pairs, slot2pos, last_use, t, idx):
    """Sequential LRU written from the definition, on plain lists.

    pairs: list of [pos, slot] (the position->slot map).  Each unique miss,
    in selection order, evicts the slot with the smallest (last_use, slot)
    among the slots not referenced in this step (last_use < t), found by a
    fresh O(H) scan.
    """
    out = []
    touched = set()
    misses_in_order = []
    for p in idx:
        p = int(p)
        if p < 0 or p >= length:
            out.append(bytes(O.ROW_BYTES))
            continue
        s = next((sl for (q, sl) in pairs if q == p), None)
        if s is not None:
            last_use[s] = t
        elif p not in misses_in_order:
            misses_in_order.append(p)
        out.append(bytes(hist[p]))
    evictions = []
    for p in misses_in_order:
        best = None
        for s in range(H):
            if last_use[s] < t and (best is None or (last_use[s], s) < (last_use[best], best)):
                best = s
        old = slot2pos[best]
        if old >= 0:
            pairs[:] = [pr for pr in pairs if pr[0] != old]
        pairs.append([p, best])
        slot2pos[best] = p
        last_use[best] = t
        evictions.append((best, old, p))
    return out, evictions


@pytest.mark.parametrize("seed", range(6))
def test_resolve_equals_brute_force_lru(seed):
    g = np.random.default_rng(seed)
    H = int(g.integers(4, 65))
    n = int(g.integers(H, 4 * H + 8))
    cap = n + 40
    st = O.LayerState(cap, H)
    hist = g.integers(0, 256, size=(cap, O.ROW_BYTES), dtype=np.uint8)
    st.append(hist[:n])
    pairs, slot2pos, last_use = [], [-1] * H, [0] * H
    length = n
    for t in range(1, 30):
        if g.random() < 0.3:                       # occasional append
            st.append(hist[length:length + 1])
            length += 1
        k = int(g.integers(1, min(16, H) + 1))
        idx = g.integers(0, length, size=k)
        if g.random() < 0.5:                       # duplicates
            idx[g.integers(0, k)] = idx[0]
        if g.random() < 0.2:                       # an invalid entry
            idx[g.integers(0, k)] = length + 3
        res = O.resolve_gather(st, idx)
        out, ev = _brute_step(hist, length, H, pairs, slot2pos, last_use, t, idx)
        assert res.evictions == ev
        assert [bytes(r) for r in res.rows] == out
        assert np.array_equal(st.slot2pos, slot2pos)
        assert np.array_equal(st.last_use, last_use)
        assert st.pos2slot == {p: s for p, s in pairs}


def _check_invariants(st, res, idx, t, seen):
    k = len(idx)
    assert res.hits + res.misses + res.invalid == k
    for p, s in st.pos2slot.items():
        assert st.slot2pos[s] == p
    filled = np.nonzero(st.slot2pos >= 0)[0]
    assert len(filled) == len(st.pos2slot)
    for s in filled:                                # every hot slot holds its position's row
        assert np.array_equal(st.hot[s], st.history[st.slot2pos[s]])
    for j, p in enumerate(idx):                     # every gathered row equals history[idx]
        if 0 <= p < st.length:
            assert np.array_equal(res.rows[j], st.history[p])
        else:
            assert not res.rows[j].any()
    hit_slots = {int(s) for s in res.slot_of if s >= 0}
    for v, _old, _p in res.evictions:               # no slot referenced at t is evicted at t
        assert v not in hit_slots
    assert len(st.pos2slot) == min(st.hot_rows, len(seen))


def test_residency_invariants_tiny_workload():
    w = W.TINY
    st = O.LayerState(w.history_cap, w.hot_rows)
    st.append(W.rows(w, 0, 0, w.n0))
    prev, seen = None, set()
    for step in range(w.steps):
        s = W.apply_carry(W.base_scores(w, 0, step), prev, W.carry_draw(w, 0, step), w.carry_boost)
        idx = O.select_topk(s, w.k)
        seen.update(int(p) for p in idx)
        res = O.resolve_gather(st, idx)
        _check_invariants(st, res, idx, step + 1, seen)
        if step > 0:   # the carried half is always selected again
            carried = set(prev[W.carry_draw(w, 0, step)].tolist())
            assert carried <= set(idx.tolist())
        prev = idx


def test_repeated_working_set_hits_after_first_step():
    st = O.LayerState(512, 64)
    st.append(np.arange(512 * O.ROW_BYTES, dtype=np.uint64).astype(np.uint8).reshape(512, -1))
    idx = np.array([5, 17, 400, 3, 99, 17], np.int32)
    r1 = O.resolve_gather(st, idx)
    assert (r1.hits, r1.misses, r1.unique_misses) == (0, 6, 5)
    for _ in range(5):
        r = O.resolve_gather(st, idx)
        assert (r.hits, r.misses) == (6, 0) and r.evictions == []


def test_empty_slots_fill_in_slot_order_then_lru():
    st = O.LayerState(100, 4)
    st.append(np.zeros((100, O.ROW_BYTES), np.uint8))
    r = O.resolve_gather(st, [10, 11])
    assert r.evictions == [(0, -1, 10), (1, -1, 11)]
    r = O.resolve_gather(st, [12, 10, 13])                 # 10 hits and is pinned
    assert r.evictions == [(2, -1, 12), (3, -1, 13)]
    r = O.resolve_gather(st, [14, 15])                      # LRU: slot 1 (t=1), then 0 (t=2)
    assert r.evictions == [(1, 11, 14), (0, 10, 15)]


# ------------------------------------------------------- recent ring
def test_ring_copyback_schedule_closed_form():
    """Device rows wait in the ring; whole 64-row batches reach RAM."""
    st = O.LayerState(1000, 16, ring_rows=256)
    st.append(np.zeros((300, O.ROW_BYTES), np.uint8))          # host rows: straight to RAM
    assert st.ram_len == 300
    for i in range(1, 200):
        st.append(np.full((1, O.ROW_BYTES), i % 251, np.uint8), from_device=True)
        assert st.ram_len == 300 + 64 * (i // 64)
        assert 0 <= st.length - st.ram_len < 64
    st.append(np.zeros((7, O.ROW_BYTES), np.uint8), from_device=True)
    assert st.ram_len == 300 + 64 * ((199 + 7) // 64)
    st.append(np.zeros((5, O.ROW_BYTES), np.uint8))            # host rows flush the ring first
    assert st.ram_len == st.length == 511
    st.append(np.zeros((3, O.ROW_BYTES), np.uint8), from_device=True)
    st.flush_ring()
    assert st.ram_len == st.length == 514


def test_ring_changes_no_output_only_where_rows_come_from():
    """The same run with and without the ring: identical rows, evictions and
    maps; host reads are the misses below ram_len (all misses without ring)."""
    w = W.TINY.scaled(appends_per_step=3, steps=16)
    runs = {}
    for ring in (0, 256):
        st = O.LayerState(w.history_cap, w.hot_rows, ring_rows=ring)
        st.append(W.rows(w, 0, 0, w.n0))
        extra = W.rows(w, 0, w.n0, w.history_cap - w.n0)
        prev, log = None, []
        for step in range(w.steps):
            st.append(extra[step * 3:step * 3 + 3], from_device=True)
            ram = st.ram_len
            s = W.apply_carry(W.base_scores(w, 0, step), prev, W.carry_draw(w, 0, step), w.carry_boost)
            idx = O.select_topk(s, w.k)
            res = O.resolve_gather(st, idx)
            missed = [int(p) for p, sl in zip(idx, res.slot_of) if sl == -1]
            assert res.host_reads == sum(p < ram for p in missed)
            log.append((idx.tobytes(), res.rows.tobytes(), tuple(res.evictions), res.host_reads, res.misses))
            prev = idx
        runs[ring] = (log, st)
    for a, b in zip(runs[0][0], runs[256][0]):
        assert a[:3] == b[:3]
        assert a[3] == a[4]                       # without the ring every miss reads RAM
        assert b[3] <= b[4]
    assert any(b[3] < b[4] for b in runs[256][0])   # recent rows were selected and read from the ring
    assert runs[0][1].pos2slot == runs[256][1].pos2slot


# ------------------------------------------------- circular replacement
def _brute_step_circular(H, pairs, slot2pos, last_use, hand, t, idx, length):
    """The circular rule one miss at a time: from the hand, step over every
    slot referenced in this step (hits and slots already filled in it) and
    evict the first other one; the hand then points past it."""
    touched = set()
    unique = []
    for p in idx:
        p = int(p)
        if p < 0 or p >= length:
            continue
        s = next((sl for (q, sl) in pairs if q == p), None)
        if s is not None:
            touched.add(s)
        elif p not in unique:
            unique.append(p)
    ev = []
    for p in unique:
        while hand in touched:
            hand = (hand + 1) % H
        v = hand
        hand = (hand + 1) % H
        touched.add(v)
        old = slot2pos[v]
        if old >= 0:
            pairs[:] = [pr for pr in pairs if pr[0] != old]
        pairs.append([p, v])
        slot2pos[v] = p
        ev.append((v, old, p))
    for s in touched:
        last_use[s] = t
    return ev, hand


@pytest.mark.parametrize("seed", range(6))
def test_circular_equals_sequential_definition(seed):
    g = np.random.default_rng(500 + seed)
    H = int(g.integers(4, 40))
    n = int(g.integers(H, 4 * H + 8))
    st = O.LayerState(n, H, policy="circular")
    st.append(g.integers(0, 256, size=(n, O.ROW_BYTES), dtype=np.uint8))
    pairs, slot2pos, last_use, hand = [], [-1] * H, [0] * H, 0
    for t in range(1, 40):
        k = int(g.integers(1, min(12, H) + 1))
        idx = g.integers(0, n, size=k)
        if g.random() < 0.5:
            idx[g.integers(0, k)] = idx[0]
        res = O.resolve_gather(st, idx)
        ev, hand = _brute_step_circular(H, pairs, slot2pos, last_use, hand, t, idx, n)
        assert res.evictions == ev
        assert st.hand == hand
        assert np.array_equal(st.slot2pos, slot2pos)
        assert np.array_equal(st.last_use, last_use)


def test_circular_worked_example():
    st = O.LayerState(100, 4, policy="circular")
    st.append(np.zeros((100, O.ROW_BYTES), np.uint8))
    assert O.resolve_gather(st, [10, 11, 12]).evictions == [(0, -1, 10), (1, -1, 11), (2, -1, 12)]
    assert st.hand == 3
    # 10 and 12 pinned by hits; the hand takes 3, wraps, skips 0 (pinned), takes 1
    assert O.resolve_gather(st, [10, 12, 13, 14]).evictions == [(3, -1, 13), (1, 11, 14)]
    assert st.hand == 2
    # LRU takes the same two here: slot 3 (never used) before slot 1 (used at t=1)
    lru = O.LayerState(100, 4)
    lru.append(np.zeros((100, O.ROW_BYTES), np.uint8))
    O.resolve_gather(lru, [10, 11, 12])
    assert O.resolve_gather(lru, [10, 12, 13, 14]).evictions == [(3, -1, 13), (1, 11, 14)]
    # the policies part ways when a recently used slot lies under the hand
    assert O.resolve_gather(st, [15]).evictions == [(2, 12, 15)]      # circular: next after the hand
    assert O.resolve_gather(lru, [15]).evictions == [(0, 10, 15)]     # LRU: the oldest (slot 0, t=2)


# ------------------------------------------------- multi-query rounds
def test_multi_query_round_worked_example():
    """Two query rows select the same missing position in one round: only
    its first occurrence takes a slot, the second reads host memory, and the
    slot becomes a hit source in the next round."""
    st = O.LayerState(100, 4)
    st.append(np.arange(100 * O.ROW_BYTES, dtype=np.uint64).astype(np.uint8).reshape(100, -1))
    r = O.resolve_gather_multi(st, [[10, 20], [20, 30]])
    assert (r.hits, r.misses, r.unique_misses) == (0, 4, 3)
    assert r.evictions == [(0, -1, 10), (1, -1, 20), (2, -1, 30)]
    assert list(r.slot_of) == [-1, -1, -1, -1]       # the repeat of 20 is not served from slot 1
    np.testing.assert_array_equal(r.rows[2], st.history[20])
    r = O.resolve_gather_multi(st, [[20, 40], [40, 10]])
    assert (r.hits, r.misses, r.unique_misses) == (2, 2, 1)
    assert r.evictions == [(3, -1, 40)]
    # rows taken as separate rounds would differ: row 1 would hit the slot row 0 filled
    st2 = O.LayerState(100, 4)
    st2.append(st.history[:100])
    O.resolve_gather(st2, [10, 20])
    assert O.resolve_gather(st2, [20, 30]).hits == 1


@pytest.mark.parametrize("seed", range(4))
def test_multi_query_round_equals_brute_force(seed):
    """Rows of overlapping selections (as MTP draft rows are) resolved as one
    round equal the sequential-LRU definition applied to the whole round."""
    g = np.random.default_rng(100 + seed)
    H, n, nq, k = 48, 160, 4, 10
    st = O.LayerState(n, H)
    hist = g.integers(0, 256, size=(n, O.ROW_BYTES), dtype=np.uint8)
    st.append(hist)
    pairs, slot2pos, last_use = [], [-1] * H, [0] * H
    for t in range(1, 25):
        base = g.choice(n, size=k, replace=False)
        rows = np.stack([np.where(g.random(k) < 0.3, g.integers(0, n, size=k), base) for _ in range(nq)])
        res = O.resolve_gather_multi(st, rows)
        out, ev = _brute_step(hist, n, H, pairs, slot2pos, last_use, t, rows.reshape(-1))
        assert res.evictions == ev
        assert [bytes(x) for x in res.rows] == out
        assert st.pos2slot == {p: s for p, s in pairs}


# ------------------------------------------------------------------ dequant
def _all_finite_fp16():
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    h = bits.view(np.float16)
    return h[np.isfinite(h)]


def test_all_finite_fp16_count():
    assert _all_finite_fp16().size == 63488


def test_bf16_rounding_matches_torch_exhaustively():
    torch = pytest.importorskip("torch")
    scales = _all_finite_fp16().astype(np.float64)
    q = np.arange(-128, 128, dtype=np.float64)
    prod = (q[:, None] * scales[None, :]).astype(np.float32).ravel()   # exact products
    ours = O.bf16_round_nearest_even(prod)
    ref = torch.from_numpy(prod).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)


def _rne_by_neighbours(x):
    """Nearest bf16 by comparing the two neighbours in float64, ties to even."""
    out = np.empty(x.shape, np.uint16)
    for i, v in enumerate(x.astype(np.float64)):
        b = np.float32(v).view(np.uint32) >> 16          # truncation toward zero
        lo = np.uint32(b) << 16
        hi = np.uint32(b + 1) << 16
        vlo = float(np.uint32(lo).view(np.float32))
        vhi = float(np.uint32(hi).view(np.float32))
        dlo, dhi = abs(v - vlo), abs(vhi - v)
        if dlo < dhi or (dlo == dhi and b % 2 == 0):
            out[i] = b
        else:
            out[i] = b + 1
    return out


def test_bf16_rounding_matches_neighbour_definition():
    g = np.random.default_rng(7)
    q = g.integers(-128, 128, size=4000).astype(np.float64)
    sc = g.choice(_all_finite_fp16(), size=4000).astype(np.float64)
    x = (q * sc).astype(np.float32)
    # include exact ties: values whose low 16 bits are exactly 0x8000
    ties = (g.integers(1, 1 << 15, size=200).astype(np.uint32) << 16 | 0x8000).view(np.float32)
    x = np.concatenate([x, ties])
    assert np.array_equal(O.bf16_round_nearest_even(x), _rne_by_neighbours(x))


def test_dequant_worked_row():
    # latent byte i = 1, scale g = g + 1 -> value i is exactly (i // 64) + 1;
    # a wrong group map (e.g. byte // 8) or field order fails this.
    row = np.zeros(O.ROW_BYTES, np.uint8)
    row[:512] = 1
    row[512:528] = (np.arange(8) + 1).astype("<f2").view(np.uint8)
    rope = (np.arange(64, dtype=np.float32) - 3.5).view(np.uint32) >> 16
    row[528:] = rope.astype("<u2").view(np.uint8)
    latent, scales, rope_bits = O.split_row(row)
    assert np.array_equal(scales.astype(np.float64), np.arange(8) + 1)
    out = O.dequant_rows(row[None])[0]
    vals = (out[:512].astype(np.uint32) << 16).view(np.float32)
    assert np.array_equal(vals, (np.arange(512) // 64 + 1).astype(np.float32))
    assert np.array_equal(out[512:], rope)
    row[:512] = np.uint8(0xFF)                        # int8 -1, sign handled
    vals = (O.dequant_rows(row[None])[0][:512].astype(np.uint32) << 16).view(np.float32)
    assert np.array_equal(vals, -(np.arange(512) // 64 + 1).astype(np.float32))


def test_generator_rows_have_the_stated_distributions():
    r = W.rows(W.TINY, 0, 0, 4096)
    lat = r[:, :512].view(np.int8)
    assert lat.min() >= -127 and lat.max() <= 127
    sc = r[:, 512:528].copy().view("<f2").astype(np.float64)
    assert sc.min() >= 1e-3 * 0.999 and sc.max() <= 1e-2 * 1.001
    # position-deterministic: the same rows come back when drawn in pieces
    assert np.array_equal(W.rows(W.TINY, 0, 100, 50), r[100:150])
