#!/usr/bin/env python
"""Throughput of the sparse KV residency hot path on GB300.

A step is one decode step of the workload: for every layer, append the new
row to the host history, select the top-K positions from the indexer scores
(on selecting layers), then resolve + gather the K rows (hits from the HBM
hot cache, misses from pinned host memory, LRU fills) into the contiguous
attention input.  Metric: selected rows resolved+gathered per second.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl kvo|reference]
                    [--workload 50k_single_layer|50k_full_stack|1m_cold_stress|tiny|
                                session_evict_restore]

With --workload session_evict_restore a step is one evict/restore cycle of
the secondary path instead: store every session's blocks from the HBM pool
to the pinned host tier, release them, overwrite the pool with filler, and
restore all sessions in one admission.

Timing: inputs (history, scores, new rows) are resident before the timed
region; a 1 GiB memset flushes L2 between steps; each step is bracketed by
CUDA events on the launching stream and every kernel of the path by its own
event pair.  Under torchrun each rank runs an independent replica (the path
shards by layer/session with no exchange) and rank 0 prints one JSON line
with the max step time over ranks.
"""
from __future__ import annotations

import argparse
import ctypes
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

from synth import workloads as W  # noqa: E402

METRIC = "selected KV rows resolved+gathered/s; GB/s vs HBM and host-link roofline"
ROW = 656
FALLBACK_HBM_GBS = 6800.0


# ----------------------------------------------------------------- helpers
def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        d = json.load(open(p))
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled during the timed region."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                 "-lms", "20"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.05)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.t.join(timeout=2)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
            except ValueError:
                continue
            for nm, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def algorithmic_bytes(w: W.Workload, n_avg: float, stats_delta: dict, resolve_launches: int,
                      select_launches: int):
    """Bytes the method must move per launch (reads + writes), from the
    counters of the timed launches.

    select:  4n (scores) + 4k (positions).
    resolve: 4K (positions) + 4K (pos2slot lookups) + 4*hits (last_use stamps)
             + 656*hits (hot rows) + R_out*K (output) + 656*fills (victim rows)
             + 16*fills (map and stamp updates) + 12*4096 (the LRU-queue window
             and its slots' last_use) + 8*(hits + fills) (queue appends);
             host link: 656 per miss occurrence.  K = k x query rows.
    """
    k = w.k * w.queries
    r_out = ROW + (2 * 576 if w.bf16 else 0)
    L = max(resolve_launches, 1)
    hits = stats_delta["hits"] / L
    fills = stats_delta["unique_misses"] / L
    misses = stats_delta["misses"] / L
    window = min(4096, 8 * w.hot_rows)
    resolve_hbm = (8 * k + 4 * hits + ROW * hits + r_out * k + (ROW + 16) * fills + 12 * window
                   + 8 * (hits + fills))
    select_hbm = 4 * n_avg + 4 * k
    host = stats_delta.get("host_bytes", ROW * stats_delta["misses"]) / L   # misses served from the ring excluded
    return {"resolve_hbm": resolve_hbm, "resolve_host": host, "select_hbm": select_hbm,
            "append_host": ROW * w.appends_per_step, "hits": hits, "misses": misses, "fills": fills}


def gather_bytes(w: W.Workload, ab: dict) -> float:
    """HBM bytes of one layer in the gather launch of kvo_decode_layers: its
    entry codes and positions (4k + 4k), the hit rows (656 per hit), the
    output (R_out per entry) and the fills (656 written to each victim slot
    from the same registers); misses cross the host link instead."""
    k = w.k * w.queries
    r_out = ROW + (2 * 576 if w.bf16 else 0)
    return 8 * k + ROW * ab["hits"] + r_out * k + ROW * ab["fills"]


def resolve_bytes(w: W.Workload, ab: dict) -> float:
    """HBM bytes of one layer in the resolve launch: the positions and their
    pos2slot entries (8k), the hit stamps (4 per hit), the misses' claims
    and their re-read (8 per miss), the LRU queue window and its slots'
    last_use (12 per entry; up to 4,096), the map updates (16 per fill), the
    entry codes (4k), the used slots' queue entries (8 per used slot), and
    the new rows read from their device copy (656 per row)."""
    k = w.k * w.queries
    window = min(4096, 8 * w.hot_rows)
    return (12 * k + 4 * ab["hits"] + 8 * ab["misses"] + 12 * window + 16 * ab["fills"]
            + 8 * (ab["hits"] + ab["fills"]) + ROW * w.appends_per_step)


def max_over_ranks(x: float, device: str = "cuda") -> float:
    """The largest x over the ranks of the default process group (x itself
    without one): a multi-GPU run reports the slowest replica's time."""
    import torch
    import torch.distributed as tdist
    if not (tdist.is_available() and tdist.is_initialized()) or tdist.get_world_size() == 1:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    tdist.all_reduce(t, op=tdist.ReduceOp.MAX)
    return float(t.item())


def dram_traffic(workload: str, kernel: str):
    """DRAM bytes per launch from the committed ncu capture, or None when the
    kernel's source has changed since the counters were taken."""
    import hashlib
    try:
        prof = json.load(open(os.path.join(ROOT, "profiles", "dram_traffic.json")))
        ent = prof[workload][kernel]
        for name, want in ent["source_sha256_16"].items():
            path = os.path.join(ROOT, "gather_radix_top_gb300", "csrc", name)
            if hashlib.sha256(open(path, "rb").read()).hexdigest()[:16] != want:
                return None
        return ent["bytes"]
    except (OSError, KeyError, ValueError):
        return None


# ------------------------------------------------------------- GPU arm
class GpuWorkload:
    """Device-resident inputs and a context for one replica of a workload."""

    def __init__(self, w: W.Workload, layer_base: int, steps: int, host_inputs: bool = False,
                 fused: bool = True, policy: str = "lru", ring: int = 0, gather: str = "auto",
                 auto_miss_pct: int = 5, layer_calls: int = 1):
        import torch
        from gather_radix_top_gb300 import kvo
        self.torch, self.kvo, self.w = torch, kvo, w
        self.steps = steps
        self.layer_calls = layer_calls
        self.host_inputs = host_inputs
        self.ctx = kvo.Context(w.layers, w.history_cap, w.hot_rows)
        if policy == "circular":
            self.ctx.set_policy(kvo.POLICY_CIRCULAR)
        if ring:
            self.ctx.set_recent_ring(ring)
        self.ctx.set_gather_mode({"loads": kvo.GATHER_LOADS, "staged": kvo.GATHER_STAGED,
                                  "auto": kvo.GATHER_AUTO}[gather], auto_miss_pct)
        self.sel = w.selecting_layers()
        for l in range(w.layers):
            self.ctx.append_rows(l, W.rows(w, layer_base + l, 0, w.n0))
        dev = "cuda"
        a = w.appends_per_step
        if a:
            new = np.stack([W.rows(w, layer_base + l, w.n0, steps * a) for l in range(w.layers)])
            self.new_rows_host = torch.from_numpy(new).pin_memory() if host_inputs else None
            self.new_rows = None if host_inputs else torch.from_numpy(new).to(dev)
        nmax = w.n_at(steps - 1)
        self.nmax = nmax
        # every selecting layer's scores in one array [steps, selecting layers,
        # nmax] (layer j's are a view), so that the carry boost of a step is a
        # few whole-array ops rather than a few per layer
        nsel = len(self.sel)
        stride = (nmax + 3) // 4 * 4                   # each layer's scores start 16-byte aligned
        base = np.zeros((steps, nsel, stride), np.float32)
        for j, l in enumerate(self.sel):
            for s in range(steps):
                n = w.n_at(s)
                base[s, j, :n] = W.base_scores(w, layer_base + l, s, n)
        t = torch.from_numpy(base)
        self.scores_all = t.pin_memory() if host_inputs else t.to(dev)
        self.scores = {l: self.scores_all[:, j] for j, l in enumerate(self.sel)}
        self.draws = {}
        if w.carry:
            d = np.stack([np.stack([W.carry_draw(w, layer_base + l, s) if s else np.zeros(w.carry, np.int64)
                                    for s in range(steps)]) for l in self.sel], axis=1)
            self.draws_all = torch.from_numpy(d).to(dev)           # [steps, nsel, carry]
            self.draws = {l: self.draws_all[:, j] for j, l in enumerate(self.sel)}
            self.row_off = (torch.arange(nsel, dtype=torch.int64, device=dev) * stride).unsqueeze(1)
            self.boost = torch.full((w.carry,), w.carry_boost, dtype=torch.float32, device=dev)
            self.boost_all = torch.full((nsel * w.carry,), w.carry_boost, dtype=torch.float32, device=dev)
        # query rows 1.. of an MTP round: row 0 plus float32 noise, added in float64
        self.nq = w.queries
        self.noise = {}
        if self.nq > 1:
            for l in self.sel:
                z = np.zeros((steps, self.nq - 1, nmax), np.float32)
                for s in range(steps):
                    for q in range(1, self.nq):
                        z[s, q - 1, :w.n_at(s)] = W.query_noise32(w, layer_base + l, s, q, w.n_at(s))
                t = torch.from_numpy(z)
                self.noise[l] = t.pin_memory() if host_inputs else t.to(dev)
        self.noise_stage = {l: torch.empty((self.nq - 1, nmax), dtype=torch.float32, device=dev)
                            for l in self.sel} if self.nq > 1 and host_inputs else None
        self.qrows = {l: torch.empty((self.nq, nmax), dtype=torch.float32, device=dev) for l in self.sel}
        self.stage = {l: torch.empty(nmax, dtype=torch.float32, device=dev) for l in self.sel}
        self.idx_all = torch.zeros((2, nsel, self.nq, w.k), dtype=torch.int32, device=dev)
        self.idx = {l: [self.idx_all[0, j], self.idx_all[1, j]] for j, l in enumerate(self.sel)}
        self.prepared = {}                    # step -> task arrays (device addresses only)
        kq = self.nq * w.k
        self.out_rows = torch.empty((kq, ROW), dtype=torch.uint8, device=dev)
        # batched layers run concurrently: one output buffer per layer
        self.batched = fused and self.nq == 1 and w.layers > 1
        self.out_layers = (torch.empty((w.layers, w.k, ROW), dtype=torch.uint8, device=dev)
                           if self.batched else None)
        self.out_layers_bf16 = (torch.empty((w.layers, w.k, 576), dtype=torch.bfloat16, device=dev)
                                if self.batched and w.bf16 else None)
        self.out_bf16 = torch.empty((kq, 576), dtype=torch.bfloat16, device=dev) if w.bf16 else None
        self.out_host = torch.empty((kq, ROW), dtype=torch.uint8).pin_memory() if host_inputs else None
        self.idx_hist = torch.zeros((steps, w.k), dtype=torch.int32, device=dev)
        self.launches = 0
        self.api_host_s = 0.0                 # host time spent inside the kvo_decode_layers calls
        self.stream = torch.cuda.current_stream()
        self.stream_ptr = ctypes.c_void_p(self.stream.cuda_stream)
        self.check = kvo._check
        self.fused = fused
        # host-input runs stage each step's new rows on the device (H2D inside the step)
        self.new_stage = (torch.empty((w.layers, max(a, 1), ROW), dtype=torch.uint8, device=dev)
                          if host_inputs and a else None)

    def scores_for(self, l, s):
        """The step's scores on the device with the carry boost applied (not timed)."""
        torch, w = self.torch, self.w
        n = w.n_at(s)
        if self.host_inputs:
            sc = self.stage[l][:n]
            sc.copy_(self.scores[l][s, :n], non_blocking=True)
        else:
            sc = self.scores[l][s, :n]
        if w.carry and s > 0:
            prev = self.idx[l][(s - 1) & 1][0]
            pos = prev.index_select(0, self.draws[l][s]).long()
            sc.index_add_(0, pos, self.boost)
        return sc

    def all_scores(self, s):
        """Every selecting layer's scores of step s on the device, the carry
        boost applied to all of them at once (device inputs; not timed): the
        same one float32 add per boosted position as scores_for."""
        w = self.w
        n = w.n_at(s)
        if w.carry and s > 0:
            prev = self.idx_all[(s - 1) & 1, :, 0]                   # [nsel, k]
            pos = prev.gather(1, self.draws_all[s]).long() + self.row_off
            self.scores_all[s].view(-1).index_add_(0, pos.view(-1), self.boost_all)
        return {l: self.scores[l][s, :n] for l in self.sel}

    def query_rows(self, l, s, row0):
        """Rows 1.. of an MTP round (row 0 + noise in float64, cast once)."""
        n = row0.shape[0]
        if self.host_inputs:
            z = self.noise_stage[l][:, :n]
            z.copy_(self.noise[l][s, :, :n], non_blocking=True)
        else:
            z = self.noise[l][s, :, :n]
        out = self.qrows[l]
        out[0, :n].copy_(row0)
        out[1:, :n].copy_((row0.double().unsqueeze(0) + z.double()).float())
        return out, n

    def prepare_layers(self, s, sc):
        """The kvo_layer_task arrays of step s (device addresses only): one
        array with every layer (a reusing layer names its source layer's
        idx, which the call's selections fill first), or with
        layer_calls = 2 the selecting layers and then the reusing ones."""
        w = self.w
        a = w.appends_per_step
        groups = {True: [], False: []}
        for l in range(w.layers):
            t = {"layer": l, "out_rows": self.out_layers[l], "idx": self.idx[w.source_layer(l)][s & 1][0]}
            if self.out_layers_bf16 is not None:
                t["out_bf16"] = self.out_layers_bf16[l]
            if a:
                t["new_rows"] = self.new_stage[l, :a] if self.host_inputs else self.new_rows[l, s * a:(s + 1) * a]
            if l in self.sel:
                t["scores"] = sc[l]
            groups[l in self.sel].append(t)
        if self.layer_calls == 1:
            return (self.kvo.make_layer_tasks(groups[True] + groups[False]), None)
        return (self.kvo.make_layer_tasks(groups[True]),
                self.kvo.make_layer_tasks(groups[False]) if groups[False] else None)

    def prepare_all(self):
        """The task arrays of every step, built before the first (device
        inputs: the addresses they hold do not change), so that the host's
        work per step is the boost, the call and the events, and the GPU's
        queue stays ahead of it."""
        if self.batched and not self.host_inputs and self.nq == 1:
            for s in range(self.steps):
                n = self.w.n_at(s)
                self.prepared[s] = self.prepare_layers(s, {l: self.scores[l][s, :n] for l in self.sel})

    def step(self, s, ev=None, kev=None):
        """One decode step over all layers.  ev: (start, end) events; kev: dict
        kind -> list of (start, end) event pairs appended per launch."""
        torch, w, ctx = self.torch, self.w, self.ctx
        if self.batched and not self.host_inputs and self.nq == 1:
            sc = self.all_scores(s)
        else:
            sc = {l: self.scores_for(l, s) for l in self.sel}
        qr = {l: self.query_rows(l, s, sc[l]) for l in self.sel} if self.nq > 1 and not self.host_inputs else None

        # per-launch event pairs, made before the step's first event so that
        # the host work between the step's events is the calls themselves
        nrec = 2 if self.batched else 2 + 3 * w.layers
        spare = [torch.cuda.Event(enable_timing=True) for _ in range(2 * nrec)] if kev is not None else []

        def rec(kind, fn):
            if kev is None:
                fn()
            else:
                a, b = spare.pop(), spare.pop()
                a.record()
                fn()
                b.record()
                kev.setdefault(kind, []).append((a, b))
            self.launches += 1

        prepared = None
        if self.batched:                    # host work, before the events; device inputs: once per step
            prepared = self.prepared.get(s) if not self.host_inputs else None
            if prepared is None:
                prepared = self.prepare_layers(s, sc)
                if not self.host_inputs:
                    self.prepared[s] = prepared
        if ev:
            ev[0].record()
        if self.nq > 1 and self.host_inputs:                # the rows' noise is a step input too
            qr = {l: self.query_rows(l, s, sc[l]) for l in self.sel}
        a = w.appends_per_step
        if self.batched:
            # two launches per step: the selecting layers, then the layers
            # that reuse their selection (kvo_decode_layers; the task arrays
            # hold device addresses and are built once per step parity)
            sel_arr, reuse_arr = prepared
            if a and self.host_inputs:
                for l in range(w.layers):
                    self.new_stage[l, :a].copy_(self.new_rows_host[l, s * a:(s + 1) * a], non_blocking=True)
            # the C function itself, its arguments made beforehand: the host
            # work between the step's events is the call
            fn = self.kvo.lib().kvo_decode_layers
            calls = [(ctx.handle, arr, len(arr), w.k, self.stream_ptr) for arr in (sel_arr, reuse_arr)
                     if arr is not None]
            h0 = time.perf_counter()
            for args in calls:
                self.check(fn(*args), "kvo_decode_layers")
                self.launches += 1
            self.api_host_s += time.perf_counter() - h0
            if self.host_inputs:
                self.out_host.copy_(self.out_layers[w.layers - 1], non_blocking=True)
            if ev:
                ev[1].record()
            self.idx_hist[s].copy_(self.idx[self.sel[0]][s & 1][0])
            return
        for l in range(w.layers):
            src = None
            if a:
                if self.host_inputs:
                    src = self.new_stage[l, :a]
                    src.copy_(self.new_rows_host[l, s * a:(s + 1) * a], non_blocking=True)
                else:
                    src = self.new_rows[l, s * a:(s + 1) * a]
            src_l = w.source_layer(l)
            if self.fused and self.nq == 1 and l in self.sel:
                rec("step", lambda: ctx.decode_step(l, src, sc[l], w.k, self.idx[l][s & 1][0], self.out_rows,
                                                    self.out_bf16))
                continue
            if a:
                rec("append", lambda: ctx.append_rows(l, src))
            if self.nq > 1:
                if l in self.sel:
                    rows, n = qr[l]
                    rec("select", lambda: ctx.select_topk_batch(rows, w.k, n, self.idx[l][s & 1]))
                rec("resolve", lambda: ctx.resolve_gather_multi(l, self.idx[src_l][s & 1], self.out_rows,
                                                                 self.out_bf16))
                continue
            if l in self.sel:
                rec("select", lambda: ctx.select_topk(sc[l], w.k, self.idx[l][s & 1][0]))
            rec("resolve", lambda: ctx.resolve_gather(l, self.idx[src_l][s & 1][0], self.out_rows,
                                                      self.out_bf16))
        if self.host_inputs:
            self.out_host.copy_(self.out_rows, non_blocking=True)
        if ev:
            ev[1].record()
        self.idx_hist[s].copy_(self.idx[self.sel[0]][s & 1][0])

    def close(self):
        self.ctx.close()


def measure_host_link(torch, kvo):
    """Best of pinned H2D memcpy and zero-copy 16-byte loads over 1 GiB."""
    nbytes = 1 << 30
    host = torch.empty(nbytes, dtype=torch.uint8).pin_memory()
    host.fill_(1)
    dev = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    sink = torch.zeros(16, dtype=torch.uint8, device="cuda")
    res = {}
    for name, fn in (("memcpy_h2d", lambda: dev.copy_(host, non_blocking=True)),
                     ("memcpy_d2h", lambda: host.copy_(dev, non_blocking=True)),
                     ("zero_copy_loads", lambda: kvo.kvo_probe_host_read(host, sink))):
        best = 0.0
        for _ in range(4):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            fn()
            b.record()
            b.synchronize()
            best = max(best, nbytes / (a.elapsed_time(b) * 1e-3) / 1e9)
        res[name] = round(best, 1)
    del host, dev
    res["peak_gbs"] = max(res["memcpy_h2d"], res["zero_copy_loads"])
    res["peak_d2h_gbs"] = res["memcpy_d2h"]
    return res


def run_gpu_arm(args, w, rank, world):
    import torch
    from gather_radix_top_gb300 import build, kvo
    build.build()
    torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", "0")))
    steps = args.warmup + args.steps
    batched = not args.separate and w.queries == 1 and w.layers > 1
    phase_steps = args.phase_steps if batched else 0
    wl = GpuWorkload(w, layer_base=rank * w.layers, steps=steps + phase_steps, fused=not args.separate,
                     policy=args.policy, ring=args.ring, gather=args.gather, auto_miss_pct=args.auto_miss_pct,
                     layer_calls=args.layer_calls)
    wl.prepare_all()
    flush = torch.empty(1 << 30, dtype=torch.uint8, device="cuda")
    dist = world > 1
    if dist:
        import torch.distributed as tdist

    def barrier():
        if dist:
            tdist.barrier()

    # settle phase and warm-up (not part of the timed region; each step's
    # own events are kept, so that the cold start can be reported)
    settle_ev = []
    for s in range(args.warmup):
        flush.zero_()
        ev = (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
        wl.step(s, ev)
        settle_ev.append(ev)
    torch.cuda.synchronize()
    settle_ms = [a.elapsed_time(b) for a, b in settle_ev]
    st0 = {l: wl.ctx.stats(l) for l in range(w.layers)}
    clocks = ClockSampler(torch.cuda.current_device())
    evs, kev = [], {}
    barrier()
    torch.cuda.synchronize()
    clocks.start()
    t0 = time.perf_counter()
    launches0 = wl.launches
    klaunch0, khost0 = wl.ctx.layers_counters() if wl.batched else (0, 0.0)
    wl.api_host_s = 0.0
    for s in range(args.warmup, steps):
        flush.zero_()                      # L2 flush between timed steps (not timed)
        ev = (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
        wl.step(s, ev, kev)
        evs.append(ev)
    torch.cuda.synchronize()
    barrier()
    wall = time.perf_counter() - t0
    clk = clocks.stop()
    launches = wl.launches - launches0
    api_host_us = 1e6 * wl.api_host_s / max(1, steps - args.warmup)
    lib_host_us = None
    if wl.batched:                         # the kernels kvo_decode_layers launched in the timed steps
        klaunch1, khost1 = wl.ctx.layers_counters()
        launches = klaunch1 - klaunch0
        lib_host_us = 1e6 * (khost1 - khost0) / max(1, steps - args.warmup)
    st1 = {l: wl.ctx.stats(l) for l in range(w.layers)}
    status = wl.ctx.sync()
    phases = None
    if phase_steps:
        # A pass after the timed region, for the kernels' own durations:
        # events between the three launches of every kvo_decode_layers call,
        # which then run in order on one stream (no overlap of the call's
        # parts, no early scheduling).
        wl.ctx.set_phase_timing(True)
        pst0 = {l: wl.ctx.stats(l) for l in range(w.layers)}
        pev = []
        for s in range(steps, steps + phase_steps):
            flush.zero_()
            ev = (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
            wl.step(s, ev)
            pev.append(ev)
        torch.cuda.synchronize()
        (t_sel, t_res, t_gat), calls = wl.ctx.layers_phase_times()
        wl.ctx.set_phase_timing(False)
        pst1 = {l: wl.ctx.stats(l) for l in range(w.layers)}
        phases = {"calls": calls, "steps": phase_steps, "layers_select": t_sel, "layers_resolve": t_res,
                  "layers_gather": t_gat, "step_ms": [a.elapsed_time(b) for a, b in pev],
                  "delta": {f: sum(pst1[l][f] - pst0[l][f] for l in range(w.layers)) for f in pst0[0]}}
    step_ms = [a.elapsed_time(b) for a, b in evs]
    total_s = sum(step_ms) * 1e-3
    total_s = max_over_ranks(total_s)
    kern = {kind: [a.elapsed_time(b) for a, b in pairs] for kind, pairs in kev.items()}
    delta = {f: sum(st1[l][f] - st0[l][f] for l in range(w.layers)) for f in st0[0]}
    idx_hist = wl.idx_hist.cpu().numpy()
    wl.close()
    del flush
    torch.cuda.empty_cache()
    return {"total_s": total_s, "step_ms": step_ms, "kern_ms": kern, "delta": delta, "wall": wall,
            "clocks": clk, "launches": launches, "status": status, "idx_hist": idx_hist, "settle_ms": settle_ms,
            "phases": phases, "api_host_us": api_host_us, "lib_host_us": lib_host_us}


def run_e2e_host_step(args, w, steps):
    """One layer, one query row: every step is one kvo_decode_step_host call
    on pinned host buffers (scores and the new row in; idx and the gathered
    rows out), which the step kernel reads and writes in place: every byte
    crosses the host link inside the step's events.  The indexer stand-in
    (the carry boost from the previous step's selection) builds the step's
    scores in pinned memory before the events, as an indexer would hand them
    over; its arithmetic is the float32 add of the device path."""
    import torch
    from gather_radix_top_gb300 import kvo
    ctx = kvo.Context(1, w.history_cap, w.hot_rows)
    if args.policy == "circular":
        ctx.set_policy(kvo.POLICY_CIRCULAR)
    if args.ring:
        ctx.set_recent_ring(args.ring)
    ctx.set_gather_mode({"loads": kvo.GATHER_LOADS, "staged": kvo.GATHER_STAGED,
                         "auto": kvo.GATHER_AUTO}[args.gather], args.auto_miss_pct)
    ctx.append_rows(0, W.rows(w, 0, 0, w.n0))
    a = w.appends_per_step
    new = torch.from_numpy(W.rows(w, 0, w.n0, steps * a)).pin_memory() if a else None
    nmax = w.n_at(steps - 1)
    sc_host = torch.empty(nmax, dtype=torch.float32).pin_memory()
    idx_h = torch.empty(w.k, dtype=torch.int32).pin_memory()
    out_h = torch.empty((w.k, ROW), dtype=torch.uint8).pin_memory()
    bf_h = torch.empty((w.k, 576), dtype=torch.int16).pin_memory() if w.bf16 else None
    flush = torch.empty(1 << 30, dtype=torch.uint8, device="cuda")
    prev, evs = None, []
    for s in range(steps):
        n = w.n_at(s)
        sc_host[:n].numpy()[:] = W.apply_carry(W.base_scores(w, 0, s, n), prev, W.carry_draw(w, 0, s),
                                               w.carry_boost)
        flush.zero_()
        ev = (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
        ev[0].record()
        ctx.decode_step_host(0, new[s * a:(s + 1) * a] if a else None, sc_host[:n], w.k, idx_h, out_h, bf_h)
        ev[1].record()
        torch.cuda.synchronize()                       # the host reads idx and rewrites the scores next
        prev = idx_h.numpy().copy()
        if s >= args.warmup:
            evs.append(ev)
    total = sum(x.elapsed_time(y) for x, y in evs) * 1e-3
    nmean = float(np.mean([w.n_at(s) for s in range(args.warmup, steps)]))
    ctx.close()
    del flush
    return {"value": round(args.steps * w.k / total, 1), "unit": "rows/s",
            "h2d_bytes_per_step": int(nmean * 4 + a * ROW),
            "d2h_bytes_per_step": int(w.k * 4 + w.k * ROW + (w.k * 576 * 2 if w.bf16 else 0)),
            "call": "kvo_decode_step_host",
            "transfer": "pinned host buffers read and written in place by the step kernel over the host link"}


def run_e2e_layers(args, w, steps):
    """Several layers, one query row: every step is the kvo_decode_layers
    call(s) of the device path on device buffers; inside the step's events the scores
    of all selecting layers and every layer's new rows come in from pinned
    host memory (one contiguous copy each) and every selecting layer's idx and
    the last layer's rows go back.  The indexer stand-in builds the scores in
    pinned memory before the events, from the selections the previous step
    returned, and the task arrays are built there too."""
    import torch
    from gather_radix_top_gb300 import kvo
    ctx = kvo.Context(w.layers, w.history_cap, w.hot_rows)
    if args.policy == "circular":
        ctx.set_policy(kvo.POLICY_CIRCULAR)
    if args.ring:
        ctx.set_recent_ring(args.ring)
    ctx.set_gather_mode({"loads": kvo.GATHER_LOADS, "staged": kvo.GATHER_STAGED,
                         "auto": kvo.GATHER_AUTO}[args.gather], args.auto_miss_pct)
    for l in range(w.layers):
        ctx.append_rows(l, W.rows(w, l, 0, w.n0))
    sel = w.selecting_layers()
    nsel, a, k = len(sel), w.appends_per_step, w.k
    nmax = w.n_at(steps - 1)
    sc_host = torch.empty(nsel * nmax, dtype=torch.float32).pin_memory()
    sc_dev = torch.empty(nsel * nmax, dtype=torch.float32, device="cuda")
    new_host = new_dev = None
    if a:                                             # [step, layer, row]: one contiguous block per step
        rows = np.stack([W.rows(w, l, w.n0, steps * a) for l in range(w.layers)])   # [layer, step*a + j]
        new_host = torch.from_numpy(np.ascontiguousarray(
            rows.reshape(w.layers, steps, a, ROW).transpose(1, 0, 2, 3)).reshape(steps, w.layers * a, ROW)).pin_memory()
        new_dev = torch.empty((w.layers * a, ROW), dtype=torch.uint8, device="cuda")
    idx_dev = torch.empty((2, nsel, k), dtype=torch.int32, device="cuda")
    idx_host = torch.empty((nsel, k), dtype=torch.int32).pin_memory()
    out_dev = torch.empty((w.layers, k, ROW), dtype=torch.uint8, device="cuda")
    bf_dev = torch.empty((w.layers, k, 576), dtype=torch.int16, device="cuda") if w.bf16 else None
    out_host = torch.empty((k, ROW), dtype=torch.uint8).pin_memory()
    flush = torch.empty(1 << 30, dtype=torch.uint8, device="cuda")
    prev, evs = [None] * nsel, []
    for s in range(steps):
        n, par = w.n_at(s), s & 1
        sch = sc_host[:nsel * n].view(nsel, n).numpy()
        for i, l in enumerate(sel):
            sch[i] = W.apply_carry(W.base_scores(w, l, s, n), prev[i], W.carry_draw(w, l, s), w.carry_boost)
        groups = {True: [], False: []}
        for l in range(w.layers):
            i = sel.index(w.source_layer(l))
            t = {"layer": l, "idx": idx_dev[par, i], "out_rows": out_dev[l]}
            if bf_dev is not None:
                t["out_bf16"] = bf_dev[l]
            if a:
                t["new_rows"] = new_dev[l * a:(l + 1) * a]
            if l in sel:
                t["scores"] = sc_dev[i * n:(i + 1) * n]
            groups[l in sel].append(t)
        if args.layer_calls == 1:                      # every layer in one call
            arr_sel, arr_reuse = kvo.make_layer_tasks(groups[True] + groups[False]), None
        else:
            arr_sel = kvo.make_layer_tasks(groups[True])
            arr_reuse = kvo.make_layer_tasks(groups[False]) if groups[False] else None
        flush.zero_()
        ev = (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
        ev[0].record()
        sc_dev[:nsel * n].copy_(sc_host[:nsel * n], non_blocking=True)
        if a:
            new_dev.copy_(new_host[s], non_blocking=True)
        ctx.decode_layers_prepared(arr_sel, k)
        if arr_reuse is not None:
            ctx.decode_layers_prepared(arr_reuse, k)
        idx_host.copy_(idx_dev[par], non_blocking=True)
        out_host.copy_(out_dev[w.layers - 1], non_blocking=True)
        ev[1].record()
        torch.cuda.synchronize()                       # the host reads idx and rewrites the scores next
        prev = [idx_host[i].numpy().copy() for i in range(nsel)]
        if s >= args.warmup:
            evs.append(ev)
    total = sum(x.elapsed_time(y) for x, y in evs) * 1e-3
    nmean = float(np.mean([w.n_at(s) for s in range(args.warmup, steps)]))
    ctx.close()
    del flush
    return {"value": round(args.steps * w.layers * k / total, 1), "unit": "rows/s",
            "h2d_bytes_per_step": int(nsel * nmean * 4 + w.layers * a * ROW),
            "d2h_bytes_per_step": int(nsel * k * 4 + k * ROW),
            "call": "kvo_decode_layers x%d, contiguous host copies in and out" % args.layer_calls,
            "to_host": "every selecting layer's idx (the indexer stand-in's next input) and the last layer's "
                       "rows; the other layers' rows stay in HBM, where attention reads them",
            "from_host": "the selecting layers' scores and every layer's new rows"}


def run_e2e_mtp(args, w, steps):
    """One layer, several query rows (MTP verification rounds): per round the
    device path's append, batched top-K of every row and multi-query resolve;
    inside the round's events the new row and all query rows come in from
    pinned host memory (one contiguous copy each) and every row's selection
    and the round's rows go back.  The rows are built on the host before the
    events: row 0 by the indexer stand-in (the carry boost from the previous
    round's row-0 selection), rows 1.. as row 0 plus their float32 noise
    added in float64 (the device path's arithmetic)."""
    import torch
    from gather_radix_top_gb300 import kvo
    ctx = kvo.Context(1, w.history_cap, w.hot_rows)
    if args.policy == "circular":
        ctx.set_policy(kvo.POLICY_CIRCULAR)
    if args.ring:
        ctx.set_recent_ring(args.ring)
    ctx.set_gather_mode({"loads": kvo.GATHER_LOADS, "staged": kvo.GATHER_STAGED,
                         "auto": kvo.GATHER_AUTO}[args.gather], args.auto_miss_pct)
    ctx.append_rows(0, W.rows(w, 0, 0, w.n0))
    a, k, nq = w.appends_per_step, w.k, w.queries
    nmax = w.n_at(steps - 1)
    new_host = torch.from_numpy(W.rows(w, 0, w.n0, steps * a)).pin_memory() if a else None
    new_dev = torch.empty((max(a, 1), ROW), dtype=torch.uint8, device="cuda")
    q_host = torch.empty(nq * nmax, dtype=torch.float32).pin_memory()
    q_dev = torch.empty(nq * nmax, dtype=torch.float32, device="cuda")
    idx_dev = torch.empty((nq, k), dtype=torch.int32, device="cuda")
    idx_host = torch.empty((nq, k), dtype=torch.int32).pin_memory()
    out_dev = torch.empty((nq * k, ROW), dtype=torch.uint8, device="cuda")
    out_host = torch.empty((nq * k, ROW), dtype=torch.uint8).pin_memory()
    bf_dev = torch.empty((nq * k, 576), dtype=torch.int16, device="cuda") if w.bf16 else None
    bf_host = torch.empty((nq * k, 576), dtype=torch.int16).pin_memory() if w.bf16 else None
    flush = torch.empty(1 << 30, dtype=torch.uint8, device="cuda")
    prev, evs = None, []
    for s in range(steps):
        n = w.n_at(s)
        qh = q_host[:nq * n].view(nq, n).numpy()
        qh[0] = W.apply_carry(W.base_scores(w, 0, s, n), prev, W.carry_draw(w, 0, s), w.carry_boost)
        for q in range(1, nq):
            qh[q] = W.query_scores(w, 0, s, q, qh[0])
        flush.zero_()
        ev = (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
        ev[0].record()
        q_dev[:nq * n].copy_(q_host[:nq * n], non_blocking=True)
        if a:
            new_dev[:a].copy_(new_host[s * a:(s + 1) * a], non_blocking=True)
            ctx.append_rows(0, new_dev[:a])
        ctx.select_topk_batch(q_dev[:nq * n].view(nq, n), k, n, idx_dev)
        ctx.resolve_gather_multi(0, idx_dev, out_dev, bf_dev)
        idx_host.copy_(idx_dev, non_blocking=True)
        out_host.copy_(out_dev, non_blocking=True)
        if bf_dev is not None:
            bf_host.copy_(bf_dev, non_blocking=True)
        ev[1].record()
        torch.cuda.synchronize()                       # the host reads idx and rewrites the rows next
        prev = idx_host[0].numpy().copy()
        if s >= args.warmup:
            evs.append(ev)
    total = sum(x.elapsed_time(y) for x, y in evs) * 1e-3
    nmean = float(np.mean([w.n_at(s) for s in range(args.warmup, steps)]))
    ctx.close()
    del flush
    return {"value": round(args.steps * nq * k / total, 1), "unit": "rows/s",
            "h2d_bytes_per_step": int(nq * nmean * 4 + a * ROW),
            "d2h_bytes_per_step": int(nq * k * 4 + nq * k * ROW + (nq * k * 576 * 2 if w.bf16 else 0)),
            "call": "kvo_append_rows + kvo_select_topk_batch + kvo_resolve_gather_multi, contiguous host copies"}


def run_e2e(args, w):
    """Same steps through the public API with host inputs/outputs: scores and
    new rows from pinned host memory, gathered rows back to pinned host memory,
    copies inside each step's events."""
    import torch
    steps = args.warmup + args.steps
    if w.layers == 1 and w.queries == 1 and not args.separate:
        return run_e2e_host_step(args, w, steps)
    if w.layers > 1 and w.queries == 1 and not args.separate:
        return run_e2e_layers(args, w, steps)
    if w.layers == 1 and w.queries > 1 and not args.separate:
        return run_e2e_mtp(args, w, steps)
    wl = GpuWorkload(w, layer_base=0, steps=steps, host_inputs=True, fused=not args.separate, policy=args.policy,
                     ring=args.ring, gather=args.gather, auto_miss_pct=args.auto_miss_pct)
    flush = torch.empty(1 << 30, dtype=torch.uint8, device="cuda")
    evs = []
    for s in range(steps):
        flush.zero_()
        ev = (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
        # the H2D copy of this step's scores sits inside the events
        ev[0].record()
        sc = {l: wl.scores_for(l, s) for l in wl.sel}
        wl.scores_for = (lambda cached: (lambda l, s_: cached[l]))(sc)
        wl.step(s)
        del wl.scores_for
        ev[1].record()
        if s >= args.warmup:
            evs.append(ev)
    torch.cuda.synchronize()
    total = sum(a.elapsed_time(b) for a, b in evs) * 1e-3
    nmean = float(np.mean([w.n_at(s) for s in range(args.warmup, steps)]))
    h2d = int(len(wl.sel) * nmean * 4 * w.queries + w.layers * w.appends_per_step * ROW)
    d2h = int(w.queries * w.k * ROW)
    wl.close()
    del flush
    return {"value": round(args.steps * w.layers * w.k * w.queries / total, 1), "unit": "rows/s",
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h}


# ----------------------------------------------------------- oracle arm
def run_oracle(w, max_steps, budget_s, layers=None, policy="lru", ring=0):
    """The oracle as it stands, on the host cores: the first steps of the
    workload (every layer, or the first `layers`) until `budget_s` of oracle
    time.  Returns rows/s, the steps done and the selections."""
    from oracle import kvo_oracle as O
    L = w.layers if layers is None else min(layers, w.layers)
    states = []
    extra = {}
    for l in range(L):
        st = O.LayerState(w.history_cap, w.hot_rows, policy=policy, ring_rows=ring)
        st.append(W.rows(w, l, 0, w.n0))
        states.append(st)
        if w.appends_per_step:
            extra[l] = W.rows(w, l, w.n0, max_steps * w.appends_per_step)
    prev = {}
    sels = []
    spent = 0.0
    cpu0 = time.process_time()
    done = 0
    for s in range(max_steps):
        scores = {l: W.apply_carry(W.base_scores(w, l, s), prev.get(l), W.carry_draw(w, l, s), w.carry_boost)
                  for l in range(L) if l % w.select_every == 0}
        t = time.perf_counter()
        idx = {}
        for l in range(L):
            for a in range(w.appends_per_step):
                states[l].append(extra[l][s * w.appends_per_step + a][None], from_device=True)
            if l % w.select_every == 0:
                rows = [scores[l]] + [W.query_scores(w, l, s, q, scores[l]) for q in range(1, w.queries)]
                idx[l] = np.stack([O.select_topk(row, w.k) for row in rows])
            O.resolve_gather_multi(states[l], idx[w.source_layer(l)], want_bf16=w.bf16)
        spent += time.perf_counter() - t
        prev = {l: v[0] for l, v in idx.items()}
        sels.append(idx[0][0])
        done += 1
        if spent >= budget_s:
            break
    cpu = time.process_time() - cpu0
    return {"rows_per_s": done * L * w.k * w.queries / spent, "steps": done, "layers": L, "seconds": spent,
            "cores": max(1, round(cpu / max(spent, 1e-9))), "sels": sels}


# ------------------------------------------------- session evict/restore
SESSION_METRIC = ("session KV rows stored+restored/s (HBM block pool <-> pinned host tier); "
                  "GB/s vs host-link roofline")


def session_config(sw, world):
    return {"workload": sw.name, "sessions": sw.sessions, "tokens": sw.tokens, "layers": sw.layers,
            "block_tokens": sw.block_tokens, "block_bytes": sw.block_bytes, "parallelism": f"replicas{world}",
            "calls": "kvo_store_blocks x sessions, kvo_pool_release, kvo_pool_fill, kvo_restore_blocks(all)",
            "l2": "inputs (%.1f GB per direction) far larger than L2" % (
                sw.sessions * sw.blocks_per_session * sw.block_bytes / 1e9)}


def run_sessions_oracle(sw, budget_s):
    """The pool oracle as it stands: one session of the workload's length on
    the first 8 layers, store -> complete -> release -> fill -> restore ->
    complete, repeated until `budget_s` of oracle time."""
    from oracle import kvo_pool_oracle as PO
    L = min(8, sw.layers)
    nb = sw.blocks_per_layer * L
    o = PO.PoolOracle(L, nb, sw.block_tokens, ROW, nb)
    assert o.alloc(0, sw.tokens) == PO.KVO_OK
    cpu0, spent, cycles = time.process_time(), 0.0, 0
    while spent < budget_s or cycles == 0:
        t = time.perf_counter()
        assert o.store(0) == PO.KVO_OK
        o.complete_copies()
        assert o.release(0) == PO.KVO_OK
        o.fill(0xA5)
        assert o.restore([0]) == PO.KVO_OK
        o.complete_copies()
        spent += time.perf_counter() - t
        cycles += 1
    cpu = time.process_time() - cpu0
    rows = 2 * cycles * L * sw.tokens
    return {"rows_per_s": rows / spent, "cycles": cycles, "layers": L, "seconds": spent,
            "cores": max(1, round(cpu / max(spent, 1e-9)))}


def run_sessions(args, rank, world):
    import torch
    from gather_radix_top_gb300 import build, kvo
    build.build()
    torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", "0")))
    sw = session_workload(args)
    S, per = sw.sessions, sw.blocks_per_session
    nb = S * per
    pool = kvo.Pool(sw.layers, nb, sw.block_tokens, nb)
    dev = torch.device("cuda")
    for s in range(S):
        assert pool.alloc(s, sw.tokens) == kvo.KVO_OK
        for layer in range(sw.layers):
            pool.write(s, layer, 0, W.session_rows_device(sw, s, layer, dev))
    torch.cuda.synchronize()
    order = list(range(S))
    ev = lambda: torch.cuda.Event(enable_timing=True)  # noqa: E731

    def cycle(timed):
        e = [ev() for _ in range(4)]
        w0 = time.perf_counter()
        e[0].record()
        for s in order:
            assert pool.store(s) == kvo.KVO_OK
        e[1].record()
        pool.sync()
        w1 = time.perf_counter()
        for s in order:
            assert pool.release(s) == kvo.KVO_OK
        pool.fill(0xA5)                              # filler overwrites the whole pool
        torch.cuda.synchronize()
        w2 = time.perf_counter()
        e[2].record()
        assert pool.restore(order) == kvo.KVO_OK
        e[3].record()
        pool.sync()
        w3 = time.perf_counter()
        return e, (w1 - w0) + (w3 - w2)

    for _ in range(args.warmup):
        cycle(False)
    clocks = ClockSampler(torch.cuda.current_device())
    clocks.start()
    evs, walls = [], []
    for _ in range(args.steps):
        e, wall = cycle(True)
        evs.append(e)
        walls.append(wall)
    torch.cuda.synchronize()
    clk = clocks.stop()
    store_ms = [e[0].elapsed_time(e[1]) for e in evs]
    restore_ms = [e[2].elapsed_time(e[3]) for e in evs]
    # bytewise check of a sample of groups after the last restore
    out = torch.empty((sw.tokens, ROW), dtype=torch.uint8, device=dev)
    checked = 0
    for s in range(S):
        for layer in (0, sw.layers // 2, sw.layers - 1):
            pool.read(s, layer, 0, out)
            assert torch.equal(out, W.session_rows_device(sw, s, layer, dev)), (s, layer)
            checked += 1
    st = pool.stats()
    pool.close()
    return {"store_ms": store_ms, "restore_ms": restore_ms, "walls": walls, "clocks": clk, "stats": st,
            "checked_groups": checked, "launches_per_cycle": S + 1}


def session_workload(args):
    sw = W.SESSIONS
    if args.sessions:
        sw = sw.scaled(sessions=args.sessions)
    if args.session_tokens:
        sw = sw.scaled(tokens=args.session_tokens)
    return sw


def sessions_main(args, rank, world):
    sw = session_workload(args)
    config = session_config(sw, world)
    rows_cycle = 2 * sw.sessions * sw.tokens * sw.layers
    bytes_dir = sw.sessions * sw.blocks_per_session * sw.block_bytes
    if args.impl == "reference":
        if rank != 0:
            return
        o = run_sessions_oracle(sw, max(10.0, args.cpu_seconds))
        line = {"impl": "reference", "metric": SESSION_METRIC, "value": round(o["rows_per_s"], 1),
                "unit": "rows/s", "n_gpus": world, "steps": o["cycles"], "warmup": 0,
                "ms_per_step": round(1e3 * o["seconds"] / o["cycles"], 3), "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": "u8", "data": "synthetic", "config": config,
                "cpu_baseline": {"value": round(o["rows_per_s"], 1), "unit": "rows/s", "cores": o["cores"],
                                 "kind": "oracle",
                                 "sample": f"1 session x {o['layers']} layers x {sw.tokens} tokens, "
                                           f"{o['cycles']} store/restore cycles"},
                "e2e": {"value": round(o["rows_per_s"], 1), "unit": "rows/s", "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}}
        print(json.dumps(line))
        return
    if world > 1:
        import torch
        import torch.distributed as tdist
        torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", "0")))
        tdist.init_process_group("nccl")
    cpu = run_sessions_oracle(sw, args.cpu_seconds) if rank == 0 and world == 1 else None
    g = run_sessions(args, rank, world)
    total_s = (sum(g["store_ms"]) + sum(g["restore_ms"])) * 1e-3
    total_s = max_over_ranks(total_s)
    if world > 1:
        import torch.distributed as tdist
        if rank != 0:
            tdist.destroy_process_group()
            return
    import torch
    from gather_radix_top_gb300 import kvo
    link = measure_host_link(torch, kvo)
    st_avg, rs_avg = float(np.mean(g["store_ms"])), float(np.mean(g["restore_ms"]))
    store_gbs = bytes_dir / (st_avg * 1e-3) / 1e9
    restore_gbs = bytes_dir / (rs_avg * 1e-3) / 1e9
    value = args.steps * rows_cycle * world / total_s
    line = {
        "metric": SESSION_METRIC, "value": round(value, 1), "unit": "rows/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(1e3 * total_s / args.steps, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "u8", "data": "synthetic",
        "config": config,
        "roofline": {"bound": "host_link", "kernel": "restore", "achieved": round(restore_gbs, 1),
                     "peak": link["peak_gbs"], "unit": "GB/s", "frac": round(restore_gbs / link["peak_gbs"], 4),
                     "traffic": None, "peak_source": "measured in this run: best of pinned H2D memcpy and "
                                                     "zero-copy loads over 1 GiB",
                     "algorithmic_bytes_per_launch": bytes_dir},
        "store": {"ms": round(st_avg, 3), "gbs": round(store_gbs, 1), "peak_d2h_gbs": link["peak_d2h_gbs"],
                  "frac": round(store_gbs / link["peak_d2h_gbs"], 4)},
        "restore": {"ms": round(rs_avg, 3), "gbs": round(restore_gbs, 1)},
        "host_link": link, "pool_stats": g["stats"], "checked_groups": g["checked_groups"],
        "gpu_launches": args.steps * g["launches_per_cycle"], "clocks": g["clocks"],
        "e2e": {"value": round(args.steps * rows_cycle / sum(g["walls"]), 1), "unit": "rows/s",
                "h2d_bytes_per_step": bytes_dir, "d2h_bytes_per_step": bytes_dir,
                "note": "host wall clock from the first kvo_store_blocks call to kvo_pool_sync, plus from "
                        "kvo_restore_blocks to kvo_pool_sync (release and filler excluded)"},
    }
    if cpu is not None:
        line["cpu_baseline"] = {"value": round(cpu["rows_per_s"], 1), "unit": "rows/s", "cores": cpu["cores"],
                                "kind": "oracle",
                                "sample": f"1 session x {cpu['layers']} layers x {sw.tokens} tokens, "
                                          f"{cpu['cycles']} store/restore cycles ({cpu['seconds']:.1f} s)"}
    print(json.dumps(line))


# ----------------------------------------------- replacement-policy probe
def probe_rounds(w, steps):
    idxs, prev = [], None
    for s in range(steps):
        prev = W.probe_idx(w, s, prev)
        idxs.append(prev)
    return np.stack(idxs)


def run_probe_oracle(w, idxs, first, budget_s, policy):
    """The oracle on the probe's rounds; rounds before `first` are the untimed fill."""
    from oracle import kvo_oracle as O
    st = O.LayerState(w.n0, w.hot_rows, policy=policy)
    st.append(W.rows(w, 0, 0, w.n0))
    spent, done, cpu = 0.0, 0, 0.0
    for s in range(idxs.shape[0]):
        t, c = time.perf_counter(), time.process_time()
        O.resolve_gather(st, idxs[s])
        if s >= first:
            spent += time.perf_counter() - t
            cpu += time.process_time() - c
            done += 1
            if spent >= budget_s:
                break
    return {"rows_per_s": done * w.k / max(spent, 1e-9), "rounds": done, "seconds": spent,
            "cores": max(1, round(cpu / max(spent, 1e-9)))}


def probe_main(args, rank, world):
    """Per-gather latency of the resolve on a full hot cache with 1% misses,
    for the chosen replacement policy (the pages' clock pathology probe)."""
    w = W.PROBE
    warm = w.extra["warm_rounds"]
    if args.steps is None:
        args.steps = 512
    steps = warm + args.warmup + args.steps
    idxs = probe_rounds(w, steps)
    config = {"workload": w.name, "policy": args.policy, "hot_rows": w.hot_rows, "k": w.k,
              "misses_per_round": w.extra["fresh"], "history": w.n0, "fill_rounds": warm,
              "calls": "kvo_resolve_gather", "parallelism": f"replicas{world}",
              "l2": "flushed between rounds (1 GiB memset, outside the events)"}
    if args.impl == "reference":
        if rank != 0:
            return
        o = run_probe_oracle(w, idxs, warm + args.warmup, max(10.0, args.cpu_seconds), args.policy)
        print(json.dumps({"impl": "reference", "metric": METRIC, "value": round(o["rows_per_s"], 1),
                          "unit": "rows/s", "n_gpus": world, "steps": o["rounds"], "warmup": 0,
                          "ms_per_step": round(1e3 * o["seconds"] / max(o["rounds"], 1), 3),
                          "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "u8",
                          "data": "synthetic", "config": config,
                          "cpu_baseline": {"value": round(o["rows_per_s"], 1), "unit": "rows/s",
                                           "cores": o["cores"], "kind": "oracle",
                                           "sample": f"{o['rounds']} probe rounds"},
                          "e2e": {"value": round(o["rows_per_s"], 1), "unit": "rows/s", "h2d_bytes_per_step": 0,
                                  "d2h_bytes_per_step": 0}}))
        return
    import torch
    from gather_radix_top_gb300 import build, kvo
    build.build()
    torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", "0")))
    cpu = (run_probe_oracle(w, idxs, warm + args.warmup, args.cpu_seconds, args.policy)
           if rank == 0 and world == 1 else None)
    ctx = kvo.Context(1, w.n0, w.hot_rows)
    if args.policy == "circular":
        ctx.set_policy(kvo.POLICY_CIRCULAR)
    ctx.append_rows(0, W.rows(w, 0, 0, w.n0))
    idx_dev = torch.from_numpy(idxs).cuda()
    out = torch.empty((w.k, ROW), dtype=torch.uint8, device="cuda")
    flush = torch.empty(1 << 30, dtype=torch.uint8, device="cuda")
    for s in range(warm + args.warmup):
        flush.zero_()
        ctx.resolve_gather(0, idx_dev[s], out)
    torch.cuda.synchronize()
    st0 = ctx.stats(0)
    clocks = ClockSampler(torch.cuda.current_device())
    clocks.start()
    evs = []
    for s in range(warm + args.warmup, steps):
        flush.zero_()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        ctx.resolve_gather(0, idx_dev[s], out)
        b.record()
        evs.append((a, b))
    torch.cuda.synchronize()
    clk = clocks.stop()
    status = ctx.sync()
    st1 = ctx.stats(0)
    ms = [a.elapsed_time(b) for a, b in evs]
    total_s = sum(ms) * 1e-3
    delta = {f: st1[f] - st0[f] for f in st0}
    ctx.close()
    total_s = max_over_ranks(total_s)
    if world > 1 and rank != 0:
        return
    hbm_peak, peak_src = load_peaks()
    ab = algorithmic_bytes(w, 0.0, delta, args.steps, 1)
    us = float(np.mean(ms)) * 1e3
    achieved = ab["resolve_hbm"] / (us * 1e-6) / 1e9
    line = {"metric": METRIC, "value": round(args.steps * w.k * world / total_s, 1), "unit": "rows/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(1e3 * total_s / args.steps, 4), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "u8", "data": "synthetic", "config": config,
            "roofline": {"bound": "hbm", "kernel": "resolve", "achieved": round(achieved, 1), "peak": hbm_peak,
                         "unit": "GB/s", "frac": round(achieved / hbm_peak, 4), "traffic": None,
                         "peak_source": f"{peak_src} (MEASURED_PEAKS.json hbm_gbs)",
                         "algorithmic_bytes_per_launch": round(ab["resolve_hbm"])},
            "per_call": {"us_p50": round(1e3 * float(np.percentile(ms, 50)), 2),
                         "us_p99": round(1e3 * float(np.percentile(ms, 99)), 2),
                         "us_max": round(1e3 * float(np.max(ms)), 2),
                         "hits": round(ab["hits"], 1), "misses": round(ab["misses"], 1)},
            "gpu_launches": args.steps, "clocks": clk, "device_status": status}
    if cpu is not None:
        line["cpu_baseline"] = {"value": round(cpu["rows_per_s"], 1), "unit": "rows/s", "cores": cpu["cores"],
                                "kind": "oracle", "sample": f"{cpu['rounds']} probe rounds ({cpu['seconds']:.1f} s)"}
    print(json.dumps(line))


# ------------------------------------------------------- miss-rate sweep
SWEEP_PCTS = [0, 1, 5, 10, 25, 50, 75, 100]


def sweep_rounds(m, rounds, warm, k, spread, seed):
    """A full 32,768-row hot cache, then rounds that keep k - m positions of
    the previous round (hits) and add m never-seen ones (misses): one run of
    consecutive positions (spread 1), or one position every `spread` (runs
    of length 1)."""
    g = np.random.default_rng([seed, m, spread])
    idxs, prev = [], None
    base = warm * k
    for s in range(warm + rounds):
        if s < warm:
            cur = np.arange(s * k, (s + 1) * k)
        else:
            keep = g.choice(prev, size=k - m, replace=False) if m < k else np.zeros(0, np.int64)
            new = base + spread * np.arange(m)
            base += spread * max(m, 1)
            cur = np.sort(np.concatenate([keep, new]))
        idxs.append(cur.astype(np.int32))
        prev = cur
    return np.stack(idxs), base


def sweep_main(args):
    """Against the miss rate, on a full 32,768-row hot cache with 2,048-row
    calls: (1) the single-layer resolve's two gather modes (register loads,
    TMA-staged); (2) kvo_decode_layers' two ways of fetching the misses from
    the host history, zero-copy loads and batched copies (one
    cudaMemcpyAsync per run of consecutive positions), with the misses in one
    run per call and with every miss its own run."""
    import torch
    from gather_radix_top_gb300 import build, kvo
    build.build()
    rounds = args.steps or 64
    warm = 16
    k, H = 2048, 32_768
    flush = torch.empty(1 << 30, dtype=torch.uint8, device="cuda")
    nmax = max(sweep_rounds(k * p // 100, args.warmup + rounds, warm, k, sp, 11)[1]
               for p in SWEEP_PCTS for sp in (1, 8))
    all_rows = W.rows(W.PROBE.scaled(name="miss_rate_sweep", n0=nmax), 0, 0, nmax)   # a row depends on its position only

    def history(n):
        return all_rows[:n]

    def timed(ctx, call, idxs):
        ms = []
        for s in range(idxs.shape[0]):
            flush.zero_()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            call(idxs[s])
            b.record()
            if s >= warm + args.warmup:
                ms.append((a, b))
        torch.cuda.synchronize()
        assert ctx.sync() == 0
        # CUDA event stamps tick in ~2 us steps here: the mean of many calls is the estimate
        return round(float(np.mean([x.elapsed_time(y) * 1e3 for x, y in ms])), 2)

    gather_rows, fetch_rows = [], []
    for pct in SWEEP_PCTS:
        m = k * pct // 100
        for spread in (1, 8):
            idx_np, n = sweep_rounds(m, args.warmup + rounds, warm, k, spread, 11)
            idxs = torch.from_numpy(idx_np).cuda()
            hist = history(n)
            out = torch.empty((k, ROW), dtype=torch.uint8, device="cuda")
            res = {"miss_pct": pct, "misses_per_call": m, "runs_per_call": (1 if spread == 1 else m) if m else 0}
            if spread == 1:                            # (1) gather modes of the single-layer resolve
                gres = {"miss_pct": pct}
                for mode, code in (("loads", kvo.GATHER_LOADS), ("staged", kvo.GATHER_STAGED)):
                    ctx = kvo.Context(1, n, H)
                    ctx.set_gather_mode(code, 0)
                    ctx.append_rows(0, hist)
                    gres[mode + "_us_mean"] = timed(ctx, lambda i: ctx.resolve_gather(0, i, out), idxs)
                    ctx.close()
                gres["faster"] = "staged" if gres["staged_us_mean"] < gres["loads_us_mean"] else "loads"
                gather_rows.append(gres)
            for mode, code in (("zerocopy", kvo.MISS_ZEROCOPY), ("batched", kvo.MISS_BATCHED)):   # (2)
                ctx = kvo.Context(1, n, H)
                ctx.set_miss_fetch(code)
                ctx.append_rows(0, hist)
                holder = {}

                def call(i, ctx=ctx, holder=holder):
                    holder["arr"] = kvo.make_layer_tasks([{"layer": 0, "idx": i, "out_rows": out}])
                    ctx.decode_layers_prepared(holder["arr"], k)
                res[mode + "_us_mean"] = timed(ctx, call, idxs)
                ctx.close()
            res["faster"] = "batched" if res["batched_us_mean"] < res["zerocopy_us_mean"] else "zerocopy"
            fetch_rows.append(res)
    staged_up_to = max([r["miss_pct"] for r in gather_rows if r["faster"] == "staged"], default=None)
    batched_wins = [(r["miss_pct"], r["runs_per_call"]) for r in fetch_rows if r["faster"] == "batched"]
    best = min(min(r["loads_us_mean"], r["staged_us_mean"]) for r in gather_rows)
    line = {"metric": METRIC, "value": round(k / (best * 1e-6), 1), "unit": "rows/s", "n_gpus": 1,
            "steps": rounds, "warmup": args.warmup, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "u8", "data": "synthetic",
            "config": {"workload": "miss_rate_sweep", "hot_rows": H, "k": k,
                       "calls": "kvo_resolve_gather (gather modes); kvo_decode_layers (miss fetch modes)",
                       "l2": "flushed between calls"},
            "gather_modes": gather_rows, "staged_faster_up_to_miss_pct": staged_up_to,
            "miss_fetch": fetch_rows, "batched_faster_at": batched_wins}
    print(json.dumps(line))


# -------------------------------------------------------------- cold start
def _read_text(path):
    try:
        return open(path).read().strip()
    except OSError:
        return None


def cold_start_main(args):
    """The first decode steps of a fresh stack after its host history was
    written, under several conditions, each on a fresh context: nothing
    before step 0; every byte of the history read once from the GPU; one
    16-byte GPU load per 4 KiB and per 64 KiB page; every byte read once by
    the CPU.  Then step 0 alone with the selection confined to few or to many
    distinct host pages (every layer resolving one given selection).  The
    host's memory settings are recorded beside the numbers.  Nothing here is
    timed for the headline: this locates where a cold start goes."""
    import torch
    from gather_radix_top_gb300 import build, kvo
    build.build()
    w = W.STACK.scaled(layers=args.layers or W.STACK.layers, steps=8)
    L, k = w.layers, w.k
    nsteps = 4
    rows = [W.rows(w, l, 0, w.n0) for l in range(L)]
    new = torch.from_numpy(np.stack([W.rows(w, l, w.n0, nsteps) for l in range(L)])).cuda()
    sel = w.selecting_layers()
    sink = torch.zeros(16, dtype=torch.uint8, device="cuda")
    hist_bytes = w.history_cap * ROW

    def fresh():
        ctx = kvo.Context(L, w.history_cap, w.hot_rows)
        for l in range(L):
            ctx.append_rows(l, rows[l])
        torch.cuda.synchronize()
        return ctx

    def run_steps(ctx):
        idx = {l: torch.empty(k, dtype=torch.int32, device="cuda") for l in sel}
        out = torch.empty((L, k, ROW), dtype=torch.uint8, device="cuda")
        prev, times = {}, []
        for s in range(nsteps):
            n = w.n_at(s)
            sc = {l: torch.from_numpy(W.apply_carry(W.base_scores(w, l, s, n), prev.get(l), W.carry_draw(w, l, s),
                                                    w.carry_boost)).cuda() for l in sel}
            tasks = [{"layer": l, "idx": idx[w.source_layer(l)], "out_rows": out[l], "new_rows": new[l, s:s + 1],
                      **({"scores": sc[l]} if l in sel else {})} for l in range(L)]
            arr = kvo.make_layer_tasks(tasks)
            torch.cuda.synchronize()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            ctx.decode_layers_prepared(arr, k)
            b.record()
            b.synchronize()
            times.append(round(a.elapsed_time(b), 3))
            prev = {l: idx[l].cpu().numpy() for l in sel}
        assert ctx.sync() == 0
        return times

    res = {}
    for name, pre in (("plain", None), ("gpu_read_every_byte", 16), ("gpu_touch_4k", 4096),
                      ("gpu_touch_64k", 65536), ("cpu_read_every_byte", "cpu")):
        ctx = fresh()
        t0 = time.perf_counter()
        if pre == "cpu":
            acc = 0
            for l in range(L):
                buf = (ctypes.c_uint8 * hist_bytes).from_address(ctx.history_host(l))
                acc ^= int(np.frombuffer(buf, dtype=np.uint64).sum() & 0xffff)
        elif pre:
            for l in range(L):
                kvo.kvo_probe_host_touch(ctx.history_host(l), hist_bytes, pre, sink)
            torch.cuda.synchronize()
        pre_ms = round(1e3 * (time.perf_counter() - t0), 1)
        res[name] = {"pass_ms": pre_ms if pre else 0.0, "step_ms": run_steps(ctx)}
        ctx.close()
    # step 0 with one given selection on every layer: contiguous rows (few
    # pages) against rows one every 24 positions (a different 4 KiB page each)
    for name, pos in (("pages_contiguous", np.arange(k)), ("pages_spread", np.arange(k) * 24)):
        ctx = fresh()
        idx = torch.from_numpy(pos.astype(np.int32)).cuda()
        out = torch.empty((L, k, ROW), dtype=torch.uint8, device="cuda")
        arr = kvo.make_layer_tasks([{"layer": l, "idx": idx, "out_rows": out[l]} for l in range(L)])
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        ctx.decode_layers_prepared(arr, k)
        b.record()
        b.synchronize()
        assert ctx.sync() == 0
        span = int(pos[-1]) * ROW + ROW
        res[name] = {"step0_ms": round(a.elapsed_time(b), 3), "pages_4k_per_layer": len({int(p) * ROW // 4096 for p in pos}),
                     "span_bytes_per_layer": span}
        ctx.close()
    line = {"workload": "cold_start", "layers": L, "history_bytes_per_layer": hist_bytes,
            "page_size": os.sysconf("SC_PAGE_SIZE"),
            "numa_balancing": _read_text("/proc/sys/kernel/numa_balancing"),
            "compaction_proactiveness": _read_text("/proc/sys/vm/compaction_proactiveness"),
            "thp": _read_text("/sys/kernel/mm/transparent_hugepage/enabled"), "results": res}
    print(json.dumps(line))


# -------------------------------------------------------------------- main
def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["kvo", "reference"], default="kvo")
    ap.add_argument("--workload", choices=sorted(W.WORKLOADS) + [W.SESSIONS.name, "miss_rate_sweep", "cold_start"],
                    default="50k_full_stack")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--policy", choices=["lru", "circular"], default="lru", help="hot-cache replacement policy")
    ap.add_argument("--ring", type=int, default=0, help="recent-ring rows per layer (0: appends go straight to RAM)")
    ap.add_argument("--gather", choices=["loads", "staged", "auto"], default="auto", help="row gather mode")
    ap.add_argument("--auto-miss-pct", type=int, default=5, help="--gather auto: staged from this miss share on")
    ap.add_argument("--sessions", type=int, default=None, help="session_evict_restore: number of sessions")
    ap.add_argument("--session-tokens", type=int, default=None, help="session_evict_restore: tokens per session")
    ap.add_argument("--layers", type=int, default=None,
                    help="run the workload with this many layers (a smaller case of the same shape, for profiling)")
    ap.add_argument("--settle", type=int, default=None, help="untimed settle steps (default: the workload's own)")
    ap.add_argument("--phase-steps", type=int, default=30,
                    help="multi-layer workloads: steps after the timed region run with CUDA events between the "
                         "launches of every kvo_decode_layers call, for the kernels' own durations (roofline)")
    ap.add_argument("--layer-calls", type=int, choices=[1, 2], default=1,
                    help="multi-layer workloads: kvo_decode_layers calls per step (2: selecting layers, then "
                         "the layers reusing their selection)")
    ap.add_argument("--separate", action="store_true",
                    help="time kvo_append_rows + kvo_select_topk + kvo_resolve_gather instead of kvo_decode_step")
    args = ap.parse_args()

    if args.workload == "miss_rate_sweep":
        sweep_main(args)
        return
    if args.workload == "cold_start":
        cold_start_main(args)
        return
    if args.workload == W.PROBE.name:
        probe_main(args, int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")))
        return
    if args.workload == W.SESSIONS.name:
        if args.steps is None:
            args.steps = 5
        sessions_main(args, int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")))
        return
    w = W.WORKLOADS[args.workload]
    if args.layers:                        # a smaller stack of the same layers (profiling captures)
        w = w.scaled(layers=args.layers)
    settle = int(w.extra.get("settle", 0)) if args.settle is None else args.settle
    args.warmup += settle                  # untimed steps: the workload's settle phase, then the warm-up
    if args.steps is None:
        args.steps = max(1, w.steps - args.warmup)
    extra = args.phase_steps if (not args.separate and w.queries == 1 and w.layers > 1) else 0
    if args.warmup + args.steps + extra > w.steps:
        w = w.scaled(steps=args.warmup + args.steps + extra)
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    config = {"workload": w.name, "layers": w.layers, "history": w.n0, "hot_rows": w.hot_rows, "k": w.k,
              "appends_per_step": w.appends_per_step, "select_every": w.select_every,
              "bf16_output": w.bf16, "queries": w.queries, "policy": args.policy, "recent_ring": args.ring,
              "gather": args.gather if args.gather != "auto" else f"auto>={args.auto_miss_pct}%", "parallelism": f"replicas{world}",
              "calls": ("kvo_append_rows+kvo_select_topk_batch(%d rows)+kvo_resolve_gather_multi" % w.queries if w.queries > 1
                        else "kvo_append_rows+kvo_select_topk+kvo_resolve_gather" if args.separate
                        else ("kvo_decode_layers (every layer; reusing layers name their source's idx)"
                              if args.layer_calls == 1 else
                              "kvo_decode_layers x2 (selecting layers, then reusing layers)") if w.layers > 1
                        else "kvo_decode_step"),
              "l2": "flushed between steps (1 GiB memset, outside the step events)"}
    if settle:
        config["settle_steps"] = settle

    if args.impl == "reference":
        if rank != 0:
            return
        o = run_oracle(w, args.warmup + args.steps, budget_s=max(30.0, 0.5 * args.cpu_seconds * 8), policy=args.policy,
                       ring=args.ring)
        line = {"impl": "reference", "metric": METRIC, "value": round(o["rows_per_s"], 1), "unit": "rows/s",
                "n_gpus": world, "steps": o["steps"], "warmup": 0,
                "ms_per_step": round(1e3 * o["seconds"] / o["steps"], 3), "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": "u8", "data": "synthetic", "config": config,
                "cpu_baseline": {"value": round(o["rows_per_s"], 1), "unit": "rows/s", "cores": o["cores"],
                                 "kind": "oracle",
                                 "sample": f"first {o['steps']} steps x {o['layers']} layers of {w.name}"},
                "e2e": {"value": round(o["rows_per_s"], 1), "unit": "rows/s", "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}}
        print(json.dumps(line))
        return

    if world > 1:
        import torch
        import torch.distributed as tdist
        torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", "0")))
        tdist.init_process_group("nccl")

    cpu = None
    if rank == 0 and world == 1:
        cpu = run_oracle(w, args.warmup + args.steps, budget_s=args.cpu_seconds, policy=args.policy, ring=args.ring)

    g = run_gpu_arm(args, w, rank, world)
    if rank != 0:
        if world > 1:
            import torch.distributed as tdist
            tdist.destroy_process_group()
        return

    import torch
    from gather_radix_top_gb300 import kvo
    hbm_peak, peak_src = load_peaks()
    link = measure_host_link(torch, kvo)
    total_rows = args.steps * w.layers * w.k * w.queries * world
    value = total_rows / g["total_s"]
    nmean = float(np.mean([w.n_at(s) for s in range(args.warmup, args.warmup + args.steps)]))
    nres = args.steps * w.layers                          # layer resolves in the timed steps
    nsel = args.steps * len(w.selecting_layers())
    ab = algorithmic_bytes(w, nmean, g["delta"], nres, nsel)
    kern_ms = dict(g["kern_ms"])
    if not kern_ms:                        # batched layers without a phase pass: the whole call
        kern_ms["layers"] = g["step_ms"]
    kern_avg = {kind: float(np.mean(v)) for kind, v in kern_ms.items()}
    kern_tot = {kind: float(np.sum(v)) for kind, v in kern_ms.items()}
    step_bytes = (w.layers * (ab["resolve_hbm"] + ROW * w.appends_per_step)
                  + len(w.selecting_layers()) * ab["select_hbm"])
    gpu_launches = g["launches"]
    ph = g.get("phases")
    kern_note = None
    if ph and ph["calls"]:
        kern_note = (f"kernel durations from {ph['steps']} steps after the timed region, with CUDA events between "
                     "the launches of each kvo_decode_layers call (launches serialised on one stream); step "
                     f"p50 there {1e3 * float(np.percentile(ph['step_ms'], 50)):.1f} us")
        # kvo_decode_layers by its launches, from the pass after the timed
        # region: the selections, the resolves and the gathers (one launch
        # over every layer of the call), with their own counters
        pst = ph["steps"]
        calls_per_step = ph["calls"] / pst
        nmean_p = float(np.mean([w.n_at(s) for s in range(args.warmup + args.steps,
                                                              args.warmup + args.steps + pst)]))
        abp = algorithmic_bytes(w, nmean_p, ph["delta"], pst * w.layers, pst * len(w.selecting_layers()))
        kern_tot = {"layers_select": ph["layers_select"], "layers_resolve": ph["layers_resolve"],
                    "layers_gather": ph["layers_gather"]}
        kern_avg = {"layers_select": ph["layers_select"] / pst,
                    "layers_resolve": ph["layers_resolve"] / ph["calls"],
                    "layers_gather": ph["layers_gather"] / ph["calls"], "layers": kern_avg.get("layers")}
        gb = gather_bytes(w, abp)
        per_launch = {"layers_select": len(w.selecting_layers()) * abp["select_hbm"],
                      "layers_resolve": w.layers * resolve_bytes(w, abp) / calls_per_step,
                      "layers_gather": w.layers * gb / calls_per_step}
    else:
        per_launch = {"resolve": ab["resolve_hbm"], "select": ab["select_hbm"],
                      "append": 2 * ROW * w.appends_per_step,
                      "step": ab["resolve_hbm"] + ab["select_hbm"] + ROW * w.appends_per_step,
                      "layers": step_bytes / max(1, len(kern_ms.get("layers", [])) / args.steps)}
    dominant = max((kd for kd in kern_tot), key=kern_tot.get)
    per_launch_bytes = per_launch[dominant]
    achieved = per_launch_bytes / (kern_avg[dominant] * 1e-3) / 1e9
    traffic = dram_traffic(w.name, dominant)
    # miss traffic over the host link: the resolving launches' host bytes over
    # their time (per resolve launch, per gather launch of the batched layers)
    if ph and ph["calls"]:
        host_gbs = w.layers * abp["resolve_host"] / (kern_tot["layers_gather"] / ph["steps"] * 1e-3) / 1e9
    elif "layers" in kern_tot:
        host_gbs = w.layers * ab["resolve_host"] / (kern_tot["layers"] / args.steps * 1e-3) / 1e9
    else:
        t_resolve = kern_avg.get("resolve", kern_avg.get("step", 1e9))
        host_gbs = ab["resolve_host"] / (t_resolve * 1e-3) / 1e9
    line = {
        "metric": METRIC, "value": round(value, 1), "unit": "rows/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(1e3 * g["total_s"] / args.steps, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "u8",
        "data": "synthetic", "config": config,
        "roofline": {"bound": "hbm", "kernel": dominant, "achieved": round(achieved, 1),
                     "peak": hbm_peak, "unit": "GB/s", "frac": round(achieved / hbm_peak, 4),
                     "traffic": traffic, "peak_source": f"{peak_src} (MEASURED_PEAKS.json hbm_gbs)"
                     if peak_src == "measured" else "fallback 6.8 TB/s",
                     "algorithmic_bytes_per_launch": round(per_launch_bytes)},
        "host_link": {"achieved_miss_gbs": round(host_gbs, 2), "peak_gbs": link["peak_gbs"],
                      "frac": round(host_gbs / link["peak_gbs"], 4) if link["peak_gbs"] else None,
                      "probe": link, "miss_bytes_per_launch": round(ab["resolve_host"]),
                      # the whole timed step: every layer's miss bytes over the step time
                      "step_miss_gbs": round(w.layers * ab["resolve_host"] * args.steps / g["total_s"] / 1e9, 2),
                      "step_frac": round(w.layers * ab["resolve_host"] * args.steps / g["total_s"] / 1e9
                                         / link["peak_gbs"], 4) if link["peak_gbs"] else None},
        "kernels_us": {k: round(1e3 * v, 3) for k, v in kern_avg.items() if v is not None},
        "kernels_note": kern_note,
        "per_step": {"hits": round(ab["hits"], 1), "misses": round(ab["misses"], 1),
                     "fills": round(ab["fills"], 1),
                     "step_us_p50": round(1e3 * float(np.percentile(g["step_ms"], 50)), 2),
                     "step_us_p99": round(1e3 * float(np.percentile(g["step_ms"], 99)), 2),
                     "step_us_max": round(1e3 * float(np.max(g["step_ms"])), 2),
                     # the untimed steps before the timed region: the workload's
                     # settle phase, then the warm-up (the cold start)
                     "untimed_steps": len(g["settle_ms"]),
                     "untimed_first_us": [round(1e3 * x, 1) for x in g["settle_ms"][:4]],
                     "untimed_us_p50": round(1e3 * float(np.percentile(g["settle_ms"], 50)), 2)
                     if g["settle_ms"] else None,
                     "untimed_us_max": round(1e3 * float(np.max(g["settle_ms"])), 2) if g["settle_ms"] else None},
        "gpu_launches": gpu_launches, "clocks": g["clocks"],
        "wall_s": round(g["wall"], 3), "device_status": g["status"],
        "api_host_us_per_step": round(g["api_host_us"], 1),
        "lib_host_us_per_step": round(g["lib_host_us"], 1) if g.get("lib_host_us") is not None else None,
    }
    if cpu is not None:
        line["cpu_baseline"] = {"value": round(cpu["rows_per_s"], 1), "unit": "rows/s", "cores": cpu["cores"],
                                "kind": "oracle",
                                "sample": f"first {cpu['steps']} steps x {cpu['layers']} layers of {w.name} "
                                          f"({cpu['seconds']:.1f} s of oracle time)"}
        m = min(len(cpu["sels"]), g["idx_hist"].shape[0])
        same = all(np.array_equal(cpu["sels"][s], g["idx_hist"][s]) for s in range(m))
        line["parity"] = {"steps_compared": m, "selections_equal": bool(same)}
    if not args.no_e2e and world == 1:
        line["e2e"] = run_e2e(args, w)
    print(json.dumps(line))


if __name__ == "__main__":
    main()
