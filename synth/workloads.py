"""Seeded synthetic workloads for the sparse KV residency path.

This module is the one piece shared by the CUDA path's tests/benchmark and the
CPU oracle.  It only draws random numbers and lays out bytes; it holds none of
the method's arithmetic (no selection, no lookup, no eviction, no dequant).

Row bytes follow the Q8G64 MLA record described in "From 1M Total to 15+ x 1M
Contexts: GLM-5.3 KV Cache Offloading", section "Separate historical capacity
from the current working set": 512 B int8 latent, 16 B of scales (8 fp16, one
per 64 latent bytes) and 128 B of RoPE data (64 bf16), 656 B in total, in that
order.

Recipes (every draw comes from ``numpy.random.default_rng`` keyed by a tuple
that starts with the workload's seed and id):
  * latent int8 uniform on [-127, 127];
  * scales fp16(uniform[1e-3, 1e-2]);
  * RoPE bf16 bit patterns: the upper 16 bits of float32 N(0, 1) draws;
  * scores float32 N(0, 1), plus an optional recency term
    ``amp * exp(-age / tau)`` (age = n - 1 - pos, computed in float64 and
    added before the single cast to float32);
  * carry-over: from step 1 on, ``carry`` entries of the previous step's
    selection, drawn uniformly without replacement, get ``+carry_boost``
    (a float32 add).  The draw is an index set into the previous selection,
    so each side applies it to its own previous selection.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

ROW_BYTES = 656
LATENT_BYTES = 512
SCALE_BYTES = 16
ROPE_BYTES = 128
ROW_CHUNK = 1 << 16          # rows are drawn in chunks of this many positions

# stream tags, so that the different draws of one workload never share a key
_TAG_ROWS = 0x524F5753
_TAG_SCORES = 0x53434F52
_TAG_CARRY = 0x43415259
_TAG_SESSION = 0x53455353
_TAG_QUERY = 0x51524F57
_TAG_PROBE = 0x50524F42


def _rng(*key: int) -> np.random.Generator:
    return np.random.default_rng([int(k) & 0xFFFFFFFF for k in key])


@dataclass(frozen=True)
class Workload:
    """Shape of one synthetic decode workload.

    ``select_every`` = 4 means only layers 0, 4, 8, ... compute a selection and
    the next three layers reuse it (selection reuse by subsequent layers).
    """
    name: str
    cfg_id: int
    seed: int
    layers: int
    n0: int                  # history rows present before step 0
    hot_rows: int
    k: int
    steps: int
    appends_per_step: int
    select_every: int = 1
    carry: int = 0
    carry_boost: float = 16.0
    recency_amp: float = 0.0
    recency_tau: float = 4096.0
    bf16: bool = False
    queries: int = 1                     # query rows per step (MTP verification rounds)
    query_noise: float = 0.25            # rows 1.. = row 0's scores + N(0, query_noise)
    extra: dict = field(default_factory=dict, compare=False, hash=False)

    @property
    def history_cap(self) -> int:
        return self.n0 + self.steps * self.appends_per_step

    def n_at(self, step: int) -> int:
        """History length seen by the selection of ``step`` (appends come first)."""
        return self.n0 + (step + 1) * self.appends_per_step

    def selecting_layers(self) -> list[int]:
        return [l for l in range(self.layers) if l % self.select_every == 0]

    def source_layer(self, layer: int) -> int:
        return layer - layer % self.select_every

    def scaled(self, **kw) -> "Workload":
        d = dict(self.__dict__)
        d.update(kw)
        return Workload(**d)


TINY = Workload("tiny", 0, 1, layers=1, n0=4096, hot_rows=1024, k=256, steps=16,
                appends_per_step=0, carry=128)
K50 = Workload("50k_single_layer", 1, 2, layers=1, n0=50_023, hot_rows=32_768, k=2048,
               steps=1024, appends_per_step=1, carry=1229, recency_amp=2.0)
# the 78 layers' first steps after loading 2.5 GB of host history are slow
# (18.7 ms, 16.7 ms, then ~8 steps down to the steady ~0.25 ms): "settle"
STACK = Workload("50k_full_stack", 2, 3, layers=78, n0=50_023, hot_rows=32_768, k=2048,
                 steps=256, appends_per_step=1, select_every=4, carry=1229, recency_amp=2.0,
                 extra={"settle": 16})
# "settle": untimed steps before a timed run's warm-up (the 32,768-slot hot
# cache fills in 16 steps of 2,048 misses; the GPU's view of the 5.5 GB host
# history settles in about as many more)
M1 = Workload("1m_cold_stress", 3, 4, layers=8, n0=1_048_576, hot_rows=32_768, k=2048,
              steps=80, appends_per_step=0, bf16=True, extra={"settle": 24})

# MTP verification: four query rows per step (the token and three drafts),
# row 0 exactly the 50K single-layer scores, rows 1-3 close to it
K50_MTP = K50.scaled(name="50k_mtp4", queries=4)

# Replacement-policy probe ("GPU cache management has hazards too": a full
# hot cache, every slot recently used, 1% misses per 2,048-row gather).
# Rounds 0..15 fill the 32,768 slots with positions 0..32,767; from then on
# every round keeps 2,028 positions of the previous round (all hits) and
# adds 20 never-seen positions (the misses).
PROBE = Workload("eviction_probe_1pct", 6, 7, layers=1, n0=32_768 + 20 * 1024, hot_rows=32_768, k=2048,
                 steps=1024, appends_per_step=0, extra={"warm_rounds": 16, "fresh": 20})

WORKLOADS = {w.name: w for w in (TINY, K50, STACK, M1, K50_MTP, PROBE)}


def rows(w: Workload, layer: int, start: int, count: int) -> np.ndarray:
    """Rows for history positions [start, start+count) of ``layer`` (uint8 [count, 656]).

    A position's bytes depend only on (workload, layer, position).
    """
    out = np.empty((count, ROW_BYTES), np.uint8)
    pos = start
    end = start + count
    while pos < end:
        chunk = pos // ROW_CHUNK
        c0 = chunk * ROW_CHUNK
        block = _row_chunk(w, layer, chunk)
        lo = pos - c0
        hi = min(end - c0, ROW_CHUNK)
        out[pos - start:pos - start + (hi - lo)] = block[lo:hi]
        pos = c0 + hi
    return out


def _row_chunk(w: Workload, layer: int, chunk: int) -> np.ndarray:
    g = _rng(w.seed, w.cfg_id, layer, _TAG_ROWS, chunk)
    m = ROW_CHUNK
    block = np.empty((m, ROW_BYTES), np.uint8)
    block[:, :LATENT_BYTES] = g.integers(-127, 128, size=(m, LATENT_BYTES), dtype=np.int8).view(np.uint8)
    sc = g.uniform(1e-3, 1e-2, size=(m, 8)).astype("<f2")
    block[:, LATENT_BYTES:LATENT_BYTES + SCALE_BYTES] = sc.view(np.uint8)
    rope = (g.standard_normal((m, 64), dtype=np.float32).view(np.uint32) >> 16).astype("<u2")
    block[:, LATENT_BYTES + SCALE_BYTES:] = rope.view(np.uint8)
    return block


def base_scores(w: Workload, layer: int, step: int, n: int | None = None) -> np.ndarray:
    """Indexer-score stand-in for ``layer`` at ``step`` before the carry boost (float32 [n])."""
    if n is None:
        n = w.n_at(step)
    g = _rng(w.seed, w.cfg_id, layer, _TAG_SCORES, step)
    z = g.standard_normal(n, dtype=np.float64)
    if w.recency_amp:
        age = (n - 1 - np.arange(n, dtype=np.float64))
        z = z + w.recency_amp * np.exp(-age / w.recency_tau)
    return z.astype(np.float32)


def carry_draw(w: Workload, layer: int, step: int) -> np.ndarray:
    """Indices into the previous step's selection that get the carry boost (int64)."""
    if step == 0 or w.carry == 0:
        return np.zeros(0, np.int64)
    g = _rng(w.seed, w.cfg_id, layer, _TAG_CARRY, step)
    return np.sort(g.choice(w.k, size=w.carry, replace=False)).astype(np.int64)


def apply_carry(scores: np.ndarray, prev_sel: np.ndarray | None, draw: np.ndarray,
                boost: float) -> np.ndarray:
    """scores with ``+boost`` (float32 add) at ``prev_sel[draw]``."""
    s = np.array(scores, dtype=np.float32, copy=True)
    if prev_sel is not None and len(draw):
        s[np.asarray(prev_sel, np.int64)[draw]] += np.float32(boost)
    return s


def query_noise32(w: Workload, layer: int, step: int, q: int, n: int) -> np.ndarray:
    """The float32 noise of query row q (q >= 1) of a step: N(0, query_noise)."""
    g = _rng(w.seed, w.cfg_id, layer, step, q, _TAG_QUERY)
    return (g.standard_normal(n) * w.query_noise).astype(np.float32)


def query_scores(w: Workload, layer: int, step: int, q: int, row0: np.ndarray) -> np.ndarray:
    """Scores of query row q (q >= 1) of a step: row 0's scores (after the
    carry-over) plus the row's float32 noise, added in float64 and cast once
    to float32 (exact on any IEEE device)."""
    noise = query_noise32(w, layer, step, q, row0.shape[0])
    return (row0.astype(np.float64) + noise.astype(np.float64)).astype(np.float32)


def probe_idx(w: Workload, step: int, prev) -> np.ndarray:
    """The probe's selection for round `step` (ascending), given the previous
    round's selection `prev` (None for round 0)."""
    warm, fresh = w.extra["warm_rounds"], w.extra["fresh"]
    if step < warm:
        return np.arange(step * w.k, (step + 1) * w.k, dtype=np.int32)
    g = _rng(w.seed, w.cfg_id, step, _TAG_PROBE)
    keep = g.choice(np.asarray(prev), size=w.k - fresh, replace=False)
    base = warm * w.k + (step - warm) * fresh
    new = np.arange(base, base + fresh)
    return np.sort(np.concatenate([keep, new])).astype(np.int32)


def random_scores(seed: int, n: int, kind: str = "normal") -> np.ndarray:
    """Small-case score vectors for edge-case tests."""
    g = _rng(seed, n, 0x45444745)
    if kind == "normal":
        return g.standard_normal(n, dtype=np.float32)
    if kind == "ties":          # few distinct values, many equal keys
        return g.integers(-3, 4, size=n).astype(np.float32)
    if kind == "special":       # +-0, +-inf, NaN, denormals mixed in
        s = g.standard_normal(n, dtype=np.float32)
        pick = g.integers(0, 7, size=n)
        specials = np.array([0.0, -0.0, np.inf, -np.inf, np.nan, 1e-45, -1e-45], np.float32)
        mask = g.random(n) < 0.3
        s[mask] = specials[pick[mask]]
        return s
    if kind == "coarse":        # N(0, 1) on a 1/64 grid: dozens of equal keys at any cut
        return (np.round(g.standard_normal(n) * 64.0) / 64.0).astype(np.float32)
    if kind == "recent":        # N(0, 1) with the last 4,096 positions raised by 6
        s = g.standard_normal(n, dtype=np.float32)
        s[max(0, n - 4096):] += np.float32(6.0)
        return s
    if kind == "lognormal":     # exp(N(0, 2)): positive, spread over many binades
        return np.exp(2.0 * g.standard_normal(n)).astype(np.float32)
    if kind == "sprinkled":     # N(0, 1) with 1% specials (+-0, +-inf, NaN, denormals)
        s = g.standard_normal(n, dtype=np.float32)
        specials = np.array([0.0, -0.0, np.inf, -np.inf, np.nan, 1e-45, -1e-45], np.float32)
        where = g.choice(n, size=n // 100, replace=False)
        s[where] = specials[g.integers(0, 7, size=where.size)]
        return s
    if kind == "negative":      # every score negative: -(|N(0, 1)| + 1e-3)
        return (-(np.abs(g.standard_normal(n)) + 1e-3)).astype(np.float32)
    if kind == "negzero":       # "negative" with 0.25% -0.0 and 0.25% -1e-45 (above every other score)
        s = (-(np.abs(g.standard_normal(n)) + 1e-3)).astype(np.float32)
        where = g.choice(n, size=n // 200, replace=False)
        s[where] = np.array([-0.0, -1e-45], np.float32)[g.integers(0, 2, size=where.size)]
        return s
    if kind == "nan_inf":       # NaN everywhere but 3,000 -inf and 1,000 -1e30
        s = np.full(n, np.nan, np.float32)
        where = g.choice(n, size=4000, replace=False)
        s[where[:3000]] = -np.inf
        s[where[3000:]] = np.float32(-1e30)
        return s
    raise ValueError(kind)


def random_idx(seed: int, n: int, k: int, dup_frac: float = 0.0, invalid: int = 0) -> np.ndarray:
    """Selection vectors for resolve tests: arbitrary order, optional duplicates and bad entries."""
    g = _rng(seed, n, k, 0x49445820)
    base = g.choice(n, size=k, replace=False) if k <= n else g.integers(0, n, size=k)
    base = base.astype(np.int32)
    ndup = int(round(dup_frac * k))
    if ndup:
        where = g.choice(k, size=ndup, replace=False)
        base[where] = base[g.integers(0, k, size=ndup)]
    if invalid:
        where = g.choice(k, size=invalid, replace=False)
        bad = np.array([-1, n, n + 7, -(2 ** 31), 2 ** 31 - 1], np.int64)
        base[where] = bad[g.integers(0, len(bad), size=invalid)].astype(np.int32)
    return base


# ------------------------------------------------------- session store/restore
@dataclass(frozen=True)
class SessionWorkload:
    """Sessions whose KV lives in fixed-size blocks of an HBM pool and is
    stored to / restored from a pinned host tier (the bounded-FS tier page's
    evict/restore cycle: ~60k-token sessions, 16-token blocks)."""
    name: str
    cfg_id: int
    seed: int
    sessions: int
    tokens: int
    layers: int
    block_tokens: int = 16

    @property
    def blocks_per_layer(self) -> int:
        return -(-self.tokens // self.block_tokens)

    @property
    def blocks_per_session(self) -> int:
        return self.blocks_per_layer * self.layers

    @property
    def block_bytes(self) -> int:
        return self.block_tokens * ROW_BYTES

    def scaled(self, **kw) -> "SessionWorkload":
        d = dict(self.__dict__)
        d.update(kw)
        return SessionWorkload(**d)


SESSIONS = SessionWorkload("session_evict_restore", 4, 5, sessions=8, tokens=60_000, layers=78)


def session_rows(sw: SessionWorkload, session: int, layer: int, start: int, count: int) -> np.ndarray:
    """Uniform random bytes for tokens [start, start+count) of one (session,
    layer) group, uint8 [count, 656]; a token's bytes depend only on
    (workload, session, layer, token)."""
    out = np.empty((count, ROW_BYTES), np.uint8)
    t = start
    while t < start + count:
        c = t // ROW_CHUNK
        lo, hi = c * ROW_CHUNK, (c + 1) * ROW_CHUNK
        g = _rng(sw.seed, sw.cfg_id, _TAG_SESSION, session, layer, c)
        block = g.integers(0, 256, size=(min(hi, sw.tokens) - lo, ROW_BYTES), dtype=np.uint8)
        e = min(hi, start + count)
        out[t - start:e - start] = block[t - lo:e - lo]
        t = e
    return out


def session_rows_device(sw: SessionWorkload, session: int, layer: int, device):
    """All of one group's rows drawn on the GPU (torch, seeded by (workload,
    session, layer)): uint8 [tokens, 656].  For sizes where a CPU draw is too
    slow; not bytewise equal to ``session_rows``."""
    import torch
    g = torch.Generator(device=device)
    g.manual_seed((sw.seed * 1_000_003 + sw.cfg_id * 10_007 + session * 101 + layer) & 0x7FFFFFFFFFFFFFFF)
    return torch.randint(0, 256, (sw.tokens, ROW_BYTES), dtype=torch.uint8, device=device, generator=g)
