"""Plain CPU oracle for the sparse KV residency path.

TEST INFRASTRUCTURE.  Only the tests, the package's ``smoke()`` check and the
benchmark's CPU-baseline leg may import this module.  The product path (the
CUDA library and its binding) never calls it and never falls back to it.

Everything here is written for a reader to check by eye against the pages; it
is deliberately slow.  It shares no code with the CUDA path.

Sources (page title, section):
  [KVO]  "From 1M Total to 15+ x 1M Contexts: GLM-5.3 KV Cache Offloading"
         (zhuai.tech blog).
  [TIER] "A 60k-token context comes back off disk in 17 seconds instead of 65
         seconds of prefill" (vllm-bounded-fs-kv-tier README).
  [CORR] "Making KV offload correct" (Running large language models on dual
         GH200, post 4).

What the method computes (the plain definitions, in the pages' order):
  * Row: [KVO] "Separate historical capacity from the current working set":
    a Q8G64 MLA row is 512 B latent + 16 B scales + 128 B RoPE = 656 B.
  * Selection: [KVO] same section: the indexer keeps the top 2,048 history
    positions.  Ties go to the lower position.
  * Residency: [KVO] "Decision three: let the GPU manage the hot cache
    directly": selected positions are checked against hot slots; hits read
    the HBM slot, misses read host memory; the gather emits a compact
    selection.  [KVO] "GPU cache management has hazards too": slots filled
    this round become hit sources only next round, duplicate misses read host
    memory, slots used by the current round are pinned.
  * Victims: least-recently-used order on (last_use_step, slot) among slots
    not referenced this step, taken one miss at a time in selection order.
  * Dequant: bf16 = round-to-nearest-even(float32(q) * float32(scale)).

Where the pages leave a point open, the function that meets it states the
reading it uses.
"""
from __future__ import annotations

import numpy as np

# ---------------------------------------------------------------------------
# Row format  ([KVO] "Separate historical capacity from the current working set")
# ---------------------------------------------------------------------------
LATENT_BYTES = 512            # int8 latent
SCALE_BYTES = 16              # 8 x fp16 scales
ROPE_BYTES = 128              # 64 x bf16 RoPE
ROW_BYTES = LATENT_BYTES + SCALE_BYTES + ROPE_BYTES
GROUP = 64                    # "G64": one scale per 64 latent bytes
N_GROUPS = LATENT_BYTES // GROUP
ROPE_VALUES = ROPE_BYTES // 2
DEQUANT_VALUES = LATENT_BYTES + ROPE_VALUES   # 576 bf16 per dequantised row
COPYBACK_BATCH = 64       # rows per recent-ring copyback

MiB = 1 << 20
GiB = 1 << 30


def split_row(row: np.ndarray):
    """Fields of one 656-byte row, in the order the section lists them.

    Reading: fields are stored latent, scales, RoPE; scale g covers latent
    bytes [64g, 64g+64); all multi-byte values little-endian.
    """
    row = np.asarray(row, np.uint8)
    assert row.shape == (ROW_BYTES,)
    latent = row[:LATENT_BYTES].view(np.int8)
    scales = row[LATENT_BYTES:LATENT_BYTES + SCALE_BYTES].view("<f2")
    rope_bits = row[LATENT_BYTES + SCALE_BYTES:].view("<u2")
    return latent, scales, rope_bits


def mla_payload_bytes(tokens: int, layers: int = 1, replicas: int = 1) -> int:
    """MLA payload of ``tokens`` rows ([KVO] payload table; "Does RAM fit
    fifteen million-token histories?": tokens x 656 B x layers x replicas)."""
    return tokens * ROW_BYTES * layers * replicas


# ---------------------------------------------------------------------------
# Top-K selection  ([KVO] "Separate historical capacity ...": the DSA indexer
# selects the top 2,048 historical positions)
# ---------------------------------------------------------------------------
def select_topk(scores: np.ndarray, k: int) -> np.ndarray:
    """The k highest-scoring positions, returned in ascending position order.

    Order used: higher score first; equal scores -> lower position first.
    Readings: -0.0 equals +0.0 (IEEE comparison); NaN ranks below every other
    value, -inf included, and NaNs tie among themselves by position.
    Raises ValueError unless 0 < k <= n.
    """
    scores = np.asarray(scores, np.float32)
    n = scores.shape[0]
    if not (0 < k <= n):
        raise ValueError("need 0 < k <= n")
    value = scores.astype(np.float64)
    is_nan = np.isnan(value)
    value[is_nan] = 0.0
    value = value + 0.0                       # -0.0 + 0.0 == +0.0
    pos = np.arange(n, dtype=np.int64)
    # np.lexsort sorts by the LAST key first: non-NaN before NaN, then by
    # score descending, then by position ascending.
    order = np.lexsort((pos, -value, is_nan))
    return np.sort(order[:k]).astype(np.int32)


# ---------------------------------------------------------------------------
# Hot-cache residency  ([KVO] "Decision three", "GPU cache management has
# hazards too")
# ---------------------------------------------------------------------------
class LayerState:
    """One layer's history (host RAM) and hot cache (HBM) with its maps.

    pos2slot is a plain dict (position -> slot); slot2pos uses -1 for an
    empty slot; last_use uses 0 for "never referenced"; ``step`` counts this
    layer's resolve calls (the first call runs at step 1).

    ``ring_rows`` > 0 turns on the recent ring ("From 1M Total to 15+ x 1M
    Contexts", pipeline "New KV -> GPU recent ring -> batched copyback -> RAM
    history"; "GPU cache management has hazards too": the ring protects new
    tokens that have not yet reached RAM): rows appended from device memory
    wait in the ring and reach RAM in batches of COPYBACK_BATCH rows;
    ``ram_len`` is how many rows RAM holds (a miss below it reads RAM, at or
    above it the ring).  Rows appended from host memory go straight to RAM
    after the pending ring rows.  Without the ring, ram_len == length.

    ``policy`` picks the replacement rule: "lru" (least recently used
    unpinned slot first, keyed (last_use, slot)) or "circular" (the pages'
    final rule, "GPU cache management has hazards too": a hand walks the
    slots in circular order and the next unpinned slot is evicted; ``hand``
    is where the next walk starts).
    """

    def __init__(self, history_cap: int, hot_rows: int, policy: str = "lru", ring_rows: int = 0):
        if policy not in ("lru", "circular"):
            raise ValueError("policy must be 'lru' or 'circular'")
        self.policy = policy
        self.hand = 0
        self.ring_rows = int(ring_rows)
        self.ram_len = 0
        self.history_cap = int(history_cap)
        self.hot_rows = int(hot_rows)
        self.history = np.zeros((self.history_cap, ROW_BYTES), np.uint8)
        self.length = 0
        self.hot = np.zeros((self.hot_rows, ROW_BYTES), np.uint8)
        self.pos2slot: dict[int, int] = {}
        self.slot2pos = np.full(self.hot_rows, -1, np.int64)
        self.last_use = np.zeros(self.hot_rows, np.int64)
        self.step = 0

    def append(self, new_rows: np.ndarray, from_device: bool = False) -> None:
        """Rows for history positions [length, length + r); length grows.

        Reading: append never touches the hot cache; an appended row becomes
        a miss the first time it is selected.  With the ring, the pipeline
        "New KV -> GPU recent ring -> batched copyback -> RAM history" runs
        as one step: device rows enter the ring, and every whole batch of
        COPYBACK_BATCH pending rows then moves to RAM before the append
        returns (a batch is copied back as soon as it is complete).  Host rows
        first flush the ring, then go to RAM.  Without the ring, every
        appended row is in RAM at once.
        """
        new_rows = np.asarray(new_rows, np.uint8).reshape(-1, ROW_BYTES)
        r = new_rows.shape[0]
        if self.length + r > self.history_cap:
            raise ValueError("history capacity exceeded")
        self.history[self.length:self.length + r] = new_rows
        self.length += r
        if self.ring_rows and from_device:
            pending = self.length - self.ram_len
            self.ram_len += pending // COPYBACK_BATCH * COPYBACK_BATCH
        else:
            self.ram_len = self.length

    def flush_ring(self) -> None:
        """Every pending ring row to RAM (the export consistency boundary)."""
        self.ram_len = self.length

    def pos2slot_array(self) -> np.ndarray:
        """pos2slot as a dense int32 array over [0, history_cap) (-1 = absent)."""
        a = np.full(self.history_cap, -1, np.int32)
        for p, s in self.pos2slot.items():
            a[p] = s
        return a


class ResolveResult:
    def __init__(self):
        self.rows = None            # uint8 [k, 656]
        self.bf16 = None            # uint16 [k, 576]
        self.hits = 0               # occurrences found in the hot cache
        self.misses = 0             # occurrences read from host memory
        self.unique_misses = 0
        self.invalid = 0            # entries outside [0, length)
        self.host_reads = 0         # miss occurrences served from RAM (position < ram_len)
        self.evictions = []         # (victim slot, evicted position or -1, new position)
        self.slot_of = None         # int32 [k]: hot slot read for a hit, -1 miss, -2 invalid


def resolve_gather(state: LayerState, idx, want_bf16: bool = False) -> ResolveResult:
    """One resolve + gather call on one layer.

    1. The layer's step counter advances: t = step + 1.
    2. Classify every idx[j] in order.  A position outside [0, length) is
       invalid: its output row is zero and it changes no state.  A position
       with a hot slot is a hit; the slot is stamped last_use = t (pinned for
       this step).  Any other position is a miss; its first occurrence makes
       it a unique miss.
    3. Victims: one linear scan collects (last_use, slot) for every slot with
       last_use < t; sorted ascending, the i-th unique miss (in idx order)
       takes the i-th entry.  This equals taking the misses one at a time and
       evicting the least recently used unpinned slot each time.
    4. Map update per unique miss p with victim v: the position v held is
       unmapped, then pos2slot[p] = v, slot2pos[v] = p, last_use[v] = t.
    5. Gather: out[j] = history[idx[j]] for every valid j (hits and misses give
       the same bytes: a hot slot holds a copy of its position's row); each
       victim slot receives its new position's row.
    A filled slot is never read as a hit in the step that fills it, because
    victims come only from slots with last_use < t and every hit is stamped t.
    """
    idx = np.asarray(idx, np.int64)
    k = idx.shape[0]
    if k == 0:
        raise ValueError("k must be > 0")
    res = ResolveResult()
    t = state.step + 1
    state.step = t

    slot_of = np.full(k, -1, np.int32)
    unique: list[int] = []
    seen_missing: set[int] = set()
    for j in range(k):
        p = int(idx[j])
        if p < 0 or p >= state.length:
            slot_of[j] = -2
            res.invalid += 1
            continue
        s = state.pos2slot.get(p)
        if s is not None:
            slot_of[j] = s
            state.last_use[s] = t
            res.hits += 1
        else:
            res.misses += 1
            res.host_reads += p < state.ram_len
            if p not in seen_missing:
                seen_missing.add(p)
                unique.append(p)
    res.unique_misses = len(unique)

    if state.policy == "lru":
        free = np.nonzero(state.last_use < t)[0]
        order = np.lexsort((free, state.last_use[free]))    # by last_use, then slot
        victims = free[order][:len(unique)]
    else:
        # circular: the unpinned slots in the order hand, hand+1, ... (mod H);
        # the hand moves past the last victim
        H = state.hot_rows
        walk = (state.hand + np.arange(H)) % H
        victims = walk[state.last_use[walk] < t][:len(unique)]
        if len(victims):
            state.hand = (int(victims[-1]) + 1) % H
    assert len(victims) == len(unique)

    for p, v in zip(unique, victims):
        v = int(v)
        old = int(state.slot2pos[v])
        if old >= 0:
            del state.pos2slot[old]
        state.pos2slot[p] = v
        state.slot2pos[v] = p
        state.last_use[v] = t
        res.evictions.append((v, old, p))

    out = np.zeros((k, ROW_BYTES), np.uint8)
    for j in range(k):
        if slot_of[j] != -2:
            out[j] = state.history[idx[j]]
    for v, _old, p in res.evictions:
        state.hot[v] = state.history[p]
    res.rows = out
    res.slot_of = slot_of
    if want_bf16:
        res.bf16 = dequant_rows(out)
    return res


# ---------------------------------------------------------------------------
# Dequantisation to bf16: bf16 = RNE(float32(q) * float32(scale[g])), RoPE
# copied bit for bit.
# ---------------------------------------------------------------------------
def resolve_gather_multi(state: LayerState, idx_rows, want_bf16: bool = False) -> ResolveResult:
    """One round of several query rows ("GPU cache management has hazards
    too": MTP verification processes several rows, and several queries can
    select the same missing position).  The round is one resolve over the
    rows' selections taken one row after another: the step advances once,
    the first occurrence of a missing position takes the slot, every later
    occurrence (in any row) reads host memory, a slot filled in the round is
    a hit source only from the next round, and every slot the round uses is
    pinned.  Output entry q * k + j belongs to row q, entry j."""
    rows = np.asarray(idx_rows, np.int64)
    if rows.ndim != 2 or rows.shape[0] < 1:
        raise ValueError("idx_rows must be [nq, k]")
    return resolve_gather(state, rows.reshape(-1), want_bf16)


def bf16_round_nearest_even(x: np.ndarray) -> np.ndarray:
    """IEEE-754 round-to-nearest, ties-to-even, of float32 values to bf16 bits.

    bf16 keeps the upper 16 bits of a float32.  The discarded lower 16 bits are
    compared with half an ulp (0x8000): above rounds up, below rounds down, at
    exactly half the kept part is made even.  NaN stays NaN (quiet bit set).
    """
    bits = np.asarray(x, np.float32).view(np.uint32).astype(np.uint64)
    upper = bits >> 16
    lower = bits & 0xFFFF
    round_up = (lower > 0x8000) | ((lower == 0x8000) & ((upper & 1) == 1))
    out = upper + round_up.astype(np.uint64)
    nan = np.isnan(np.asarray(x, np.float32))
    out = np.where(nan, upper | 0x40, out)
    return out.astype(np.uint16)


def dequant_rows(rows: np.ndarray) -> np.ndarray:
    """uint16 [k, 576]: 512 dequantised latent values, then the 64 RoPE values.

    The product of an int8 (8 significant bits) and an fp16 (11) fits a
    float32 exactly, so it is formed in float64 (also exact) and rounded once.
    """
    rows = np.asarray(rows, np.uint8).reshape(-1, ROW_BYTES)
    k = rows.shape[0]
    out = np.zeros((k, DEQUANT_VALUES), np.uint16)
    for j in range(k):
        latent, scales, rope_bits = split_row(rows[j])
        scale_per_byte = np.repeat(scales.astype(np.float64), GROUP)
        product = latent.astype(np.float64) * scale_per_byte
        out[j, :LATENT_BYTES] = bf16_round_nearest_even(product.astype(np.float32))
        out[j, LATENT_BYTES:] = rope_bits
    return out
