"""Plain CPU oracle for session block store/restore.

TEST INFRASTRUCTURE.  Only the tests, the package's ``smoke()`` check and the
benchmark's CPU-baseline leg may import this module.

Sources (page title, section):
  [TIER] "A 60k-token context comes back off disk in 17 seconds instead of 65
         seconds of prefill" (vllm-bounded-fs-kv-tier README): KV lives in
         fixed-size blocks of a GPU pool; whole sessions are stored to a tier
         and restored; a restore is admitted only when every group's blocks
         can be placed; the tier holds num_blocks = bytes // block_bytes; the
         pool's free queue hands out blocks from its front and takes freed
         blocks at its back.
  [CORR] "Making KV offload correct", section "A grouped allocation is a
         transaction" (Figure 1): reserve all groups, then commit ownership;
         if a later group fails, every earlier mutation is undone (request
         tables, free-list membership, counters); section "Response
         completion is not copy completion": a block may be released only
         after the transfers that depend on it have finished.

Model: blocks hold block_tokens consecutive rows of one (session, layer)
group; a session owns ceil(tokens / block_tokens) blocks in every layer.
Copies complete when the caller says so (``complete_copies``), standing in
for a CUDA event.
"""
from __future__ import annotations

import collections

import numpy as np

KVO_OK, KVO_EINVAL, KVO_EBUSY, KVO_ECAPACITY = 0, -1, -5, -7


def tier_blocks(tier_bytes: int, block_bytes: int) -> int:
    """[TIER]: num_blocks = bytes // aligned block bytes (floor division)."""
    return tier_bytes // block_bytes


class BlockAllocator:
    """A FIFO free queue of block ids with a fault hook (the n-th allocation
    from arming fails)."""

    def __init__(self, nblocks: int):
        self.free = collections.deque(range(nblocks))
        self.fail_after = -1

    def take(self, n: int):
        """n blocks from the front, or None (and nothing taken) if any single
        allocation fails."""
        got = []
        for _ in range(n):
            if self.fail_after == 0 or not self.free:
                if self.fail_after == 0:
                    self.fail_after = -1
                self.give_front(got)
                return None
            if self.fail_after > 0:
                self.fail_after -= 1
            got.append(self.free.popleft())
        return got

    def give_front(self, blocks):
        """Undo a take: the blocks go back to the front in their order."""
        for b in reversed(blocks):
            self.free.appendleft(b)

    def give_back(self, blocks):
        self.free.extend(blocks)


class Session:
    def __init__(self, tokens: int):
        self.tokens = tokens
        self.pool = None       # per layer: list of pool block ids, or None
        self.tier = None       # per layer: list of tier block ids, or None
        self.busy = 0          # copies in flight that read or write its blocks


class PoolOracle:
    def __init__(self, layers: int, pool_blocks: int, block_tokens: int, row_bytes: int, tier_blocks_n: int):
        self.layers, self.block_tokens, self.row_bytes = layers, block_tokens, row_bytes
        self.block_bytes = block_tokens * row_bytes
        self.pool_alloc = BlockAllocator(pool_blocks)
        self.tier_alloc = BlockAllocator(tier_blocks_n)
        self.pool = np.zeros((pool_blocks, self.block_bytes), np.uint8)
        self.tier = np.zeros((tier_blocks_n, self.block_bytes), np.uint8)
        self.sessions: dict[int, Session] = {}
        self.pending = []      # (session ids, blocks to free afterwards: (allocator, blocks))
        self.stats = collections.Counter()

    # ---------------------------------------------------------------- sizes
    def blocks_per_layer(self, tokens: int) -> int:
        return -(-tokens // self.block_tokens)

    # ------------------------------------------------------------- allocate
    def _take_groups(self, alloc: BlockAllocator, groups):
        """Transaction: every group's blocks, or none (each earlier group is
        given back, front first, exactly as it was)."""
        taken = []
        for n in groups:
            got = alloc.take(n)
            if got is None:
                for g in reversed(taken):
                    alloc.give_front(g)
                return None
            taken.append(got)
        return taken

    def alloc(self, sid: int, tokens: int) -> int:
        if sid in self.sessions or tokens <= 0:
            return KVO_EINVAL
        nb = self.blocks_per_layer(tokens)
        got = self._take_groups(self.pool_alloc, [nb] * self.layers)
        if got is None:
            self.stats["rollbacks"] += 1
            return KVO_ECAPACITY
        s = Session(tokens)
        s.pool = got
        self.sessions[sid] = s
        return KVO_OK

    # ----------------------------------------------------------------- data
    def write(self, sid: int, layer: int, first: int, rows: np.ndarray) -> int:
        s = self.sessions.get(sid)
        rows = np.asarray(rows, np.uint8).reshape(-1, self.row_bytes)
        if s is None or s.pool is None or first < 0 or first + len(rows) > s.tokens:
            return KVO_EINVAL
        for i, row in enumerate(rows):
            t = first + i
            b = s.pool[layer][t // self.block_tokens]
            o = (t % self.block_tokens) * self.row_bytes
            self.pool[b, o:o + self.row_bytes] = row
        return KVO_OK

    def read(self, sid: int, layer: int, first: int, n: int):
        s = self.sessions[sid]
        out = np.zeros((n, self.row_bytes), np.uint8)
        for i in range(n):
            t = first + i
            b = s.pool[layer][t // self.block_tokens]
            o = (t % self.block_tokens) * self.row_bytes
            out[i] = self.pool[b, o:o + self.row_bytes]
        return out

    def fill(self, byte: int):
        self.pool[:] = byte

    # ---------------------------------------------------- store and restore
    def store(self, sid: int) -> int:
        """Copy every pool block of the session to newly taken tier blocks."""
        s = self.sessions.get(sid)
        if s is None or s.pool is None or s.tier is not None:
            return KVO_EINVAL
        got = self._take_groups(self.tier_alloc, [len(g) for g in s.pool])
        if got is None:
            self.stats["rollbacks"] += 1
            return KVO_ECAPACITY
        for layer in range(self.layers):
            for pb, tb in zip(s.pool[layer], got[layer]):
                self.tier[tb] = self.pool[pb]
        s.tier = got
        s.busy += 1
        self.pending.append(([sid], []))
        self.stats["stores"] += 1
        self.stats["bytes_stored"] += sum(len(g) for g in got) * self.block_bytes
        return KVO_OK

    def release(self, sid: int) -> int:
        """Give the session's pool blocks back, unless a copy still depends
        on them ([CORR] "Response completion is not copy completion")."""
        s = self.sessions.get(sid)
        if s is None or s.pool is None:
            return KVO_EINVAL
        if s.busy:
            return KVO_EBUSY
        for g in s.pool:
            self.pool_alloc.give_back(g)
        s.pool = None
        if s.tier is None:
            del self.sessions[sid]
        return KVO_OK

    def restore(self, sids) -> int:
        """Every listed session's groups get pool blocks, all or none; then the
        tier copies come back and their tier blocks are freed once the copy
        has completed."""
        ss = [self.sessions.get(i) for i in sids]
        if not sids or len(set(sids)) != len(sids) or any(s is None or s.tier is None or s.pool is not None
                                                          for s in ss):
            return KVO_EINVAL
        groups = [len(g) for s in ss for g in s.tier]
        got = self._take_groups(self.pool_alloc, groups)
        if got is None:
            self.stats["rollbacks"] += 1
            return KVO_ECAPACITY
        it = iter(got)
        freed = []
        for s in ss:
            s.pool = [next(it) for _ in range(self.layers)]
            for layer in range(self.layers):
                for pb, tb in zip(s.pool[layer], s.tier[layer]):
                    self.pool[pb] = self.tier[tb]
                freed.append(s.tier[layer])
            s.tier = None
            s.busy += 1
        self.pending.append((list(sids), [(self.tier_alloc, b) for b in freed]))
        self.stats["restores"] += 1
        self.stats["bytes_restored"] += sum(groups) * self.block_bytes
        return KVO_OK

    def complete_copies(self):
        """Every copy issued so far has finished (a CUDA stream synchronise)."""
        for sids, frees in self.pending:
            for i in sids:
                self.sessions[i].busy -= 1
            for alloc, blocks in frees:
                alloc.give_back(blocks)
        self.pending = []

    # --------------------------------------------------------------- state
    def snapshot(self):
        """Everything a failed transaction must leave unchanged."""
        return (list(self.pool_alloc.free), list(self.tier_alloc.free),
                {i: ([list(g) for g in s.pool] if s.pool else None,
                     [list(g) for g in s.tier] if s.tier else None) for i, s in self.sessions.items()},
                {k: v for k, v in self.stats.items() if k != "rollbacks"})
