"""Shared drivers for the GPU parity tests: run a workload through the CUDA
path (via the C ABI binding) and through the oracle on the same seeded
inputs, one step at a time.  Each side applies the carry-over boost to its
own previous selection."""
from __future__ import annotations

import numpy as np

from oracle import kvo_oracle as O
from synth import workloads as W


def cuda_ok() -> bool:
    try:
        import torch
        return torch.cuda.is_available()
    except Exception:
        return False


class GpuLayerRun:
    """One layer of a workload on the GPU, driven step by step."""

    def __init__(self, w: W.Workload, layer: int, ctx=None, ctx_layer: int = 0, want_rows=True,
                 want_bf16=None, fused: bool = False, policy: int = 0, ring: int = 0, gather=None):
        import torch
        from gather_radix_top_gb300 import kvo
        self.torch = torch
        self.w, self.layer = w, layer
        self.own = ctx is None
        self.ctx = ctx or kvo.Context(1, w.history_cap, w.hot_rows)
        if policy:
            self.ctx.set_policy(policy)
        if ring:
            self.ctx.set_recent_ring(ring)
        if gather is not None:
            self.ctx.set_gather_mode(*gather)
        self.cl = ctx_layer
        self.ctx.append_rows(self.cl, W.rows(w, layer, 0, w.n0))          # host rows
        extra = w.history_cap - w.n0
        self.new_rows = (torch.from_numpy(W.rows(w, layer, w.n0, extra)).cuda()
                         if extra else None)
        bf = w.bf16 if want_bf16 is None else want_bf16
        self.out_rows = torch.empty((w.k, O.ROW_BYTES), dtype=torch.uint8, device="cuda") if want_rows else None
        self.out_bf16 = torch.empty((w.k, O.DEQUANT_VALUES), dtype=torch.bfloat16, device="cuda") if bf else None
        self.prev = None
        self.fused = fused

    def step(self, step: int):
        torch = self.torch
        w = self.w
        a = w.appends_per_step
        s = W.apply_carry(W.base_scores(w, self.layer, step), self.prev,
                          W.carry_draw(w, self.layer, step), w.carry_boost)
        scores = torch.from_numpy(s).cuda()
        if self.fused:
            new = self.new_rows[step * a:(step + 1) * a] if a else None
            idx = self.ctx.decode_step(self.cl, new, scores, w.k, out_rows=self.out_rows, out_bf16=self.out_bf16)
        else:
            for i in range(a):
                pos = w.n0 + step * a + i
                self.ctx.append_rows(self.cl, self.new_rows[pos - w.n0:pos - w.n0 + 1])   # device rows
            idx = self.ctx.select_topk(scores, w.k)
            self.ctx.resolve_gather(self.cl, idx, self.out_rows, self.out_bf16)
        idx_h = idx.cpu().numpy()
        self.prev = idx_h
        return idx_h

    def rows(self):
        return None if self.out_rows is None else self.out_rows.cpu().numpy()

    def bf16(self):
        if self.out_bf16 is None:
            return None
        return self.out_bf16.view(self.torch.int16).cpu().numpy().view(np.uint16)


class OracleLayerRun:
    """One layer of a workload through the oracle: append, select, resolve.
    Every GPU entry point (separate calls, the one-launch decode step, the
    batched layers) is checked against this one sequence."""

    def __init__(self, w: W.Workload, layer: int, want_bf16=None, policy: str = "lru", ring: int = 0):
        self.w, self.layer = w, layer
        self.st = O.LayerState(w.history_cap, w.hot_rows, policy=policy, ring_rows=ring)
        self.st.append(W.rows(w, layer, 0, w.n0))
        self.extra = W.rows(w, layer, w.n0, w.history_cap - w.n0) if w.history_cap > w.n0 else None
        self.bf = w.bf16 if want_bf16 is None else want_bf16
        self.prev = None
        self.last = None

    def step(self, step: int, idx_override=None):
        w = self.w
        for a in range(w.appends_per_step):
            pos = w.n0 + step * w.appends_per_step + a
            self.st.append(self.extra[pos - w.n0:pos - w.n0 + 1], from_device=True)
        if idx_override is None:
            s = W.apply_carry(W.base_scores(w, self.layer, step), self.prev,
                              W.carry_draw(w, self.layer, step), w.carry_boost)
            idx = O.select_topk(s, w.k)
        else:
            idx = idx_override
        self.last = O.resolve_gather(self.st, idx, want_bf16=self.bf)
        self.prev = idx
        return idx


def compare_state(ctx, ctx_layer: int, st: O.LayerState, check_hot=True):
    """GPU layer state == oracle state (maps exactly; hot rows of filled slots)."""
    d = ctx.dump_layer(ctx_layer, hot=check_hot)
    np.testing.assert_array_equal(d["slot2pos"], st.slot2pos.astype(np.int32))
    np.testing.assert_array_equal(d["last_use"], st.last_use.astype(np.uint32))
    np.testing.assert_array_equal(d["pos2slot"], st.pos2slot_array())
    assert d["step"] == st.step
    if check_hot:
        filled = np.nonzero(st.slot2pos >= 0)[0]
        np.testing.assert_array_equal(d["hot"][filled], st.hot[filled])
