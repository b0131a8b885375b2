"""ctypes binding of libkvo (include/kvo.h): argument marshalling only.

Each ``kvo_*`` function here calls the C function of the same name.  Device
buffers are passed as torch CUDA tensors (PyTorch supplies device memory and
streams; all the work runs in libkvo's kernels).  A missing library raises
ImportError: there is no fallback implementation.
"""
from __future__ import annotations

import ctypes
import os

from . import build as _build

ROW_BYTES = 656
DEQUANT_VALUES = 576
MAX_K = 4096
MAX_ROUND = 8192
POLICY_LRU, POLICY_CIRCULAR = 0, 1
COPYBACK_BATCH = 64
GATHER_LOADS, GATHER_STAGED, GATHER_AUTO = 0, 1, 2
MISS_ZEROCOPY, MISS_BATCHED, MISS_AUTO = 0, 1, 2
MAX_HOT_ROWS = 131072
NOALLOC_MAX_PAIRS = 65536

KVO_OK, KVO_EINVAL, KVO_ENOMEM, KVO_ECUDA, KVO_ERANGE, KVO_EBUSY, KVO_ETIMEDOUT, KVO_ECAPACITY = (
    0, -1, -2, -3, -4, -5, -6, -7)

EXPORTED = [
    "kvo_status_string", "kvo_create", "kvo_destroy", "kvo_append_rows", "kvo_select_topk",
    "kvo_select_topk_batch",
    "kvo_resolve_gather", "kvo_resolve_gather_multi", "kvo_decode_step", "kvo_decode_step_host", "kvo_decode_layers", "kvo_sync", "kvo_get_stats", "kvo_history_length",
    "kvo_debug_dump_layer", "kvo_debug_record_evictions", "kvo_debug_evictions", "kvo_set_policy",
    "kvo_debug_layer_counters", "kvo_debug_raise_status", "kvo_set_recent_ring", "kvo_flush_ring", "kvo_ram_length",
    "kvo_debug_read_history", "kvo_set_gather_mode",
    "kvo_probe_host_read",
    "kvo_tier_blocks", "kvo_pool_create", "kvo_pool_destroy", "kvo_pool_alloc", "kvo_pool_write",
    "kvo_pool_read", "kvo_pool_fill", "kvo_store_blocks", "kvo_pool_release", "kvo_restore_blocks",
    "kvo_pool_sync", "kvo_pool_block_table", "kvo_pool_get_stats", "kvo_pool_debug_fail_after",
    "kvo_pool_debug_free_queue", "kvo_copy_blocks_noalloc", "kvo_set_phase_timing", "kvo_layers_phase_times",
    "kvo_layers_counters", "kvo_probe_host_touch", "kvo_debug_history_host", "kvo_set_miss_fetch",
    "kvo_touch_history",
]


class KvoError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {status_string(status)} ({status})")


class kvo_stats(ctypes.Structure):
    _fields_ = [(n, ctypes.c_uint64) for n in (
        "steps", "hits", "misses", "unique_misses", "evictions", "invalid", "host_bytes", "rows_out")]

    def as_dict(self) -> dict:
        return {n: int(getattr(self, n)) for n, _ in self._fields_}


class kvo_layer_task(ctypes.Structure):
    _fields_ = [("layer", ctypes.c_int32), ("reserved", ctypes.c_int32), ("new_rows", ctypes.c_void_p),
                ("r", ctypes.c_int64), ("scores", ctypes.c_void_p), ("n", ctypes.c_int64),
                ("idx", ctypes.c_void_p), ("out_rows", ctypes.c_void_p), ("out_bf16", ctypes.c_void_p)]


class kvo_pool_stats(ctypes.Structure):
    _fields_ = [(n, ctypes.c_uint64) for n in (
        "stores", "restores", "rollbacks", "bytes_stored", "bytes_restored", "free_blocks",
        "tier_free_blocks", "pending_copies")]

    def as_dict(self) -> dict:
        return {n: int(getattr(self, n)) for n, _ in self._fields_}


_lib = None
_vp, _i32, _i64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64


def library_path() -> str:
    return _build.LIB


def lib() -> ctypes.CDLL:
    """Load libkvo.so (built in-tree by gather_radix_top_gb300.build)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(_build.LIB):
        raise ImportError(f"{_build.LIB} is missing: build it with gather_radix_top_gb300.build.build()")
    L = ctypes.CDLL(_build.LIB)
    sig = {
        "kvo_status_string": (ctypes.c_char_p, [ctypes.c_int]),
        "kvo_create": (ctypes.c_int, [_i32, _i64, _i32, _i32, ctypes.POINTER(_vp)]),
        "kvo_destroy": (ctypes.c_int, [_vp]),
        "kvo_append_rows": (ctypes.c_int, [_vp, _i32, _vp, _i64, _vp]),
        "kvo_select_topk": (ctypes.c_int, [_vp, _vp, _i64, _i32, _vp, _vp]),
        "kvo_select_topk_batch": (ctypes.c_int, [_vp, _vp, _i64, _i64, _i32, _i32, _vp, _vp]),
        "kvo_resolve_gather": (ctypes.c_int, [_vp, _i32, _vp, _i32, _vp, _vp, _vp]),
        "kvo_resolve_gather_multi": (ctypes.c_int, [_vp, _i32, _vp, _i32, _i32, _vp, _vp, _vp]),
        "kvo_decode_step": (ctypes.c_int, [_vp, _i32, _vp, _i64, _vp, _i64, _i32, _vp, _vp, _vp, _vp]),
        "kvo_decode_step_host": (ctypes.c_int, [_vp, _i32, _vp, _i64, _vp, _i64, _i32, _vp, _vp, _vp, _vp]),
        "kvo_decode_layers": (ctypes.c_int, [_vp, ctypes.POINTER(kvo_layer_task), _i32, _i32, _vp]),
        "kvo_sync": (ctypes.c_int, [_vp, _vp]),
        "kvo_get_stats": (ctypes.c_int, [_vp, _i32, ctypes.POINTER(kvo_stats)]),
        "kvo_history_length": (ctypes.c_int, [_vp, _i32, ctypes.POINTER(_i64)]),
        "kvo_debug_dump_layer": (ctypes.c_int, [_vp, _i32, _vp, _vp, _vp, _vp, _vp]),
        "kvo_debug_record_evictions": (ctypes.c_int, [_vp, _i32]),
        "kvo_debug_evictions": (ctypes.c_int, [_vp, _i32, _vp, _i32, ctypes.POINTER(_i32)]),
        "kvo_probe_host_read": (ctypes.c_int, [_vp, _i64, _vp, _vp]),
        "kvo_set_policy": (ctypes.c_int, [_vp, _i32]),
        "kvo_set_recent_ring": (ctypes.c_int, [_vp, _i32]),
        "kvo_set_gather_mode": (ctypes.c_int, [_vp, _i32, _i32]),
        "kvo_flush_ring": (ctypes.c_int, [_vp, _i32, _vp]),
        "kvo_ram_length": (ctypes.c_int, [_vp, _i32, ctypes.POINTER(_i64)]),
        "kvo_debug_read_history": (ctypes.c_int, [_vp, _i32, _i64, _i64, _vp]),
        "kvo_debug_layer_counters": (ctypes.c_int, [_vp, _i32, _vp]),
        "kvo_debug_raise_status": (ctypes.c_int, [_vp, ctypes.c_uint32]),
        "kvo_tier_blocks": (_i64, [_i64, _i64]),
        "kvo_pool_create": (ctypes.c_int, [_i32, _i64, _i32, _i32, _i64, ctypes.POINTER(_vp)]),
        "kvo_pool_destroy": (ctypes.c_int, [_vp]),
        "kvo_pool_alloc": (ctypes.c_int, [_vp, _i32, _i64]),
        "kvo_pool_write": (ctypes.c_int, [_vp, _i32, _i32, _i64, _vp, _i64, _vp]),
        "kvo_pool_read": (ctypes.c_int, [_vp, _i32, _i32, _i64, _i64, _vp, _vp]),
        "kvo_pool_fill": (ctypes.c_int, [_vp, ctypes.c_uint8, _vp]),
        "kvo_store_blocks": (ctypes.c_int, [_vp, _i32, _vp]),
        "kvo_pool_release": (ctypes.c_int, [_vp, _i32]),
        "kvo_restore_blocks": (ctypes.c_int, [_vp, _vp, _i32, _vp]),
        "kvo_pool_sync": (ctypes.c_int, [_vp, _vp]),
        "kvo_pool_block_table": (ctypes.c_int, [_vp, _i32, _i32, _i32, _vp, _i64, ctypes.POINTER(_i64)]),
        "kvo_pool_get_stats": (ctypes.c_int, [_vp, ctypes.POINTER(kvo_pool_stats)]),
        "kvo_pool_debug_fail_after": (ctypes.c_int, [_vp, _i32, _i64]),
        "kvo_pool_debug_free_queue": (ctypes.c_int, [_vp, _i32, _vp, _i64, ctypes.POINTER(_i64)]),
        "kvo_copy_blocks_noalloc": (ctypes.c_int, [_vp, _vp, _i64, _vp, _i64, _vp]),
        "kvo_set_phase_timing": (ctypes.c_int, [_vp, _i32]),
        "kvo_layers_phase_times": (ctypes.c_int, [_vp, _vp, _vp]),
        "kvo_layers_counters": (ctypes.c_int, [_vp, _vp, _vp]),
        "kvo_probe_host_touch": (ctypes.c_int, [_vp, _i64, _i64, _vp, _vp]),
        "kvo_debug_history_host": (ctypes.c_int, [_vp, _i32, _vp]),
        "kvo_set_miss_fetch": (ctypes.c_int, [_vp, _i32, _i32]),
        "kvo_touch_history": (ctypes.c_int, [_vp, _i32, _vp]),
    }
    for name, (res, args) in sig.items():
        f = getattr(L, name)
        f.restype = res
        f.argtypes = args
    _lib = L
    return L


def status_string(status: int) -> str:
    return lib().kvo_status_string(int(status)).decode()


def _check(status: int, what: str) -> int:
    if status != KVO_OK:
        raise KvoError(status, what)
    return status


def _host_ptr(t, dtype_name: str | None = None):
    """data_ptr of a contiguous CPU tensor (None -> NULL); pinned memory gives
    the host link's full rate."""
    if t is None:
        return None
    if t.is_cuda:
        raise ValueError("expected a CPU tensor")
    if not t.is_contiguous():
        raise ValueError("expected a contiguous tensor")
    if dtype_name is not None and str(t.dtype) != dtype_name:
        raise ValueError(f"expected {dtype_name}, got {t.dtype}")
    return ctypes.c_void_p(t.data_ptr())


def _dev_ptr(t, dtype_name: str | None = None):
    """data_ptr of a contiguous CUDA tensor (None -> NULL)."""
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("expected a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError("expected a contiguous tensor")
    if dtype_name is not None and str(t.dtype) != dtype_name:
        raise ValueError(f"expected {dtype_name}, got {t.dtype}")
    return ctypes.c_void_p(t.data_ptr())


def _stream_ptr(stream):
    if stream is None:
        import torch
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


# ----------------------------------------------------------------- calls
def kvo_create(layers: int, history_cap: int, hot_rows: int, row_bytes: int = ROW_BYTES) -> int:
    h = _vp()
    _check(lib().kvo_create(layers, history_cap, hot_rows, row_bytes, ctypes.byref(h)), "kvo_create")
    return h.value


def kvo_destroy(ctx: int) -> None:
    _check(lib().kvo_destroy(ctx), "kvo_destroy")


def kvo_append_rows(ctx: int, layer: int, rows, stream=None) -> None:
    """rows: uint8 tensor [r, 656] on the GPU, or a CPU tensor / numpy array."""
    import numpy as np
    if hasattr(rows, "is_cuda") and rows.is_cuda:
        ptr, r, keep = _dev_ptr(rows, "torch.uint8"), rows.numel() // ROW_BYTES, rows
    else:
        keep = np.ascontiguousarray(np.asarray(rows, dtype=np.uint8))
        if keep.ctypes.data % 16:                 # the C call wants 16-byte aligned rows
            buf = np.empty(keep.nbytes + 16, np.uint8)
            off = (-buf.ctypes.data) % 16
            buf[off:off + keep.nbytes] = keep.ravel()
            keep = buf[off:off + keep.nbytes]
        ptr, r = ctypes.c_void_p(keep.ctypes.data), keep.size // ROW_BYTES
    _check(lib().kvo_append_rows(ctx, layer, ptr, r, _stream_ptr(stream)), "kvo_append_rows")
    del keep


def kvo_select_topk(ctx: int, scores, k: int, idx=None, stream=None):
    import torch
    if idx is None:
        idx = torch.empty(k, dtype=torch.int32, device=scores.device)
    _check(lib().kvo_select_topk(ctx, _dev_ptr(scores, "torch.float32"), scores.numel(), k,
                                 _dev_ptr(idx, "torch.int32"), _stream_ptr(stream)), "kvo_select_topk")
    return idx


def kvo_select_topk_batch(ctx: int, scores, k: int, n: int | None = None, idx=None, stream=None):
    """scores: float32 CUDA tensor [nq, ld] (row-contiguous); the first n
    (default ld) of each row are selected from.  Returns idx int32 [nq, k]."""
    import torch
    if scores.dim() != 2 or scores.stride(1) != 1:
        raise ValueError("scores must be [nq, ld] with contiguous rows")
    nq, ld = scores.shape[0], scores.stride(0)
    n = scores.shape[1] if n is None else n
    if idx is None:
        idx = torch.empty((nq, k), dtype=torch.int32, device=scores.device)
    _check(lib().kvo_select_topk_batch(ctx, ctypes.c_void_p(scores.data_ptr()), n, ld, nq, k,
                                       _dev_ptr(idx, "torch.int32"), _stream_ptr(stream)), "kvo_select_topk_batch")
    return idx


def kvo_resolve_gather(ctx: int, layer: int, idx, out_rows=None, out_bf16=None, stream=None) -> None:
    """out_rows: uint8 [k, 656]; out_bf16: bfloat16 (or int16 bit buffer) [k, 576]."""
    if out_bf16 is not None and str(out_bf16.dtype) not in ("torch.bfloat16", "torch.int16"):
        raise ValueError("out_bf16 must be bfloat16 or int16")
    _check(lib().kvo_resolve_gather(ctx, layer, _dev_ptr(idx, "torch.int32"), idx.numel(),
                                    _dev_ptr(out_rows, "torch.uint8"), _dev_ptr(out_bf16),
                                    _stream_ptr(stream)), "kvo_resolve_gather")


def kvo_resolve_gather_multi(ctx: int, layer: int, idx, out_rows=None, out_bf16=None, stream=None) -> None:
    """idx: int32 CUDA tensor [nq, k] (one query row's selection per row);
    out_rows: uint8 [nq*k, 656]; out_bf16: bfloat16 (or int16) [nq*k, 576]."""
    if idx.dim() != 2:
        raise ValueError("idx must be [nq, k]")
    if out_bf16 is not None and str(out_bf16.dtype) not in ("torch.bfloat16", "torch.int16"):
        raise ValueError("out_bf16 must be bfloat16 or int16")
    _check(lib().kvo_resolve_gather_multi(ctx, layer, _dev_ptr(idx, "torch.int32"), idx.shape[0], idx.shape[1],
                                          _dev_ptr(out_rows, "torch.uint8"), _dev_ptr(out_bf16),
                                          _stream_ptr(stream)), "kvo_resolve_gather_multi")


def kvo_decode_step_host(ctx: int, layer: int, new_rows, scores, k: int, idx, out_rows=None, out_bf16=None,
                         stream=None):
    """kvo_decode_step on CPU tensors (pinned for full speed): new_rows uint8
    [r, 656] or None, scores fp32[n], idx int32[k] (output), out_rows uint8
    [k, 656] and/or out_bf16 [k, 576].  Enqueued on `stream`: synchronise
    before reading the outputs."""
    if out_bf16 is not None and str(out_bf16.dtype) not in ("torch.bfloat16", "torch.int16"):
        raise ValueError("out_bf16 must be bfloat16 or int16")
    r = 0 if new_rows is None else new_rows.numel() // ROW_BYTES
    _check(lib().kvo_decode_step_host(ctx, layer, _host_ptr(new_rows, "torch.uint8"), r,
                                      _host_ptr(scores, "torch.float32"), scores.numel(), k,
                                      _host_ptr(idx, "torch.int32"), _host_ptr(out_rows, "torch.uint8"),
                                      _host_ptr(out_bf16), _stream_ptr(stream)), "kvo_decode_step_host")
    return idx


def kvo_decode_step(ctx: int, layer: int, new_rows, scores, k: int, idx=None, out_rows=None, out_bf16=None,
                    stream=None):
    """Append (new_rows: uint8 CUDA tensor [r, 656] or None), select and
    resolve one layer's decode step in one launch; returns idx."""
    import torch
    if idx is None:
        idx = torch.empty(k, dtype=torch.int32, device=scores.device)
    if out_bf16 is not None and str(out_bf16.dtype) not in ("torch.bfloat16", "torch.int16"):
        raise ValueError("out_bf16 must be bfloat16 or int16")
    r = 0 if new_rows is None else new_rows.numel() // ROW_BYTES
    _check(lib().kvo_decode_step(ctx, layer, _dev_ptr(new_rows, "torch.uint8"), r,
                                 _dev_ptr(scores, "torch.float32"), scores.numel(), k,
                                 _dev_ptr(idx, "torch.int32"), _dev_ptr(out_rows, "torch.uint8"),
                                 _dev_ptr(out_bf16), _stream_ptr(stream)), "kvo_decode_step")
    return idx


def make_layer_tasks(tasks):
    """A kvo_layer_task array from dicts with layer, idx (int32 CUDA [k]) and
    out_rows and/or out_bf16, optionally new_rows (uint8 CUDA [r, 656]) and
    scores (float32 CUDA [n]; without scores idx is resolved as given).  The
    array holds raw device addresses: it stays valid while the tensors do."""
    arr = (kvo_layer_task * len(tasks))()
    for i, t in enumerate(tasks):
        nr = t.get("new_rows")
        sc = t.get("scores")
        ob = t.get("out_bf16")
        if ob is not None and str(ob.dtype) not in ("torch.bfloat16", "torch.int16"):
            raise ValueError("out_bf16 must be bfloat16 or int16")
        arr[i].layer = t["layer"]
        arr[i].new_rows = None if nr is None else _dev_ptr(nr, "torch.uint8")
        arr[i].r = 0 if nr is None else nr.numel() // ROW_BYTES
        arr[i].scores = None if sc is None else _dev_ptr(sc, "torch.float32")
        arr[i].n = 0 if sc is None else sc.numel()
        arr[i].idx = _dev_ptr(t["idx"], "torch.int32")
        arr[i].out_rows = _dev_ptr(t.get("out_rows"), "torch.uint8")
        arr[i].out_bf16 = _dev_ptr(ob)
    return arr


def kvo_decode_layers_prepared(ctx: int, arr, k: int, stream=None) -> None:
    """kvo_decode_layers with an array from make_layer_tasks (no marshalling)."""
    _check(lib().kvo_decode_layers(ctx, arr, len(arr), k, _stream_ptr(stream)), "kvo_decode_layers")


def kvo_decode_layers(ctx: int, tasks, k: int, stream=None) -> None:
    """One decode step of several layers in one launch; tasks as in make_layer_tasks."""
    kvo_decode_layers_prepared(ctx, make_layer_tasks(tasks), k, stream)


def kvo_sync(ctx: int, stream=None) -> int:
    """Synchronise and return the latched device status (KVO_OK, KVO_ERANGE, ...)."""
    return lib().kvo_sync(ctx, _stream_ptr(stream))


def kvo_get_stats(ctx: int, layer: int) -> dict:
    s = kvo_stats()
    _check(lib().kvo_get_stats(ctx, layer, ctypes.byref(s)), "kvo_get_stats")
    return s.as_dict()


def kvo_history_length(ctx: int, layer: int) -> int:
    n = _i64()
    _check(lib().kvo_history_length(ctx, layer, ctypes.byref(n)), "kvo_history_length")
    return n.value


def kvo_debug_dump_layer(ctx: int, layer: int, history_cap: int, hot_rows: int, hot: bool = True) -> dict:
    import numpy as np
    d = {
        "pos2slot": np.empty(history_cap, np.int32),
        "slot2pos": np.empty(hot_rows, np.int32),
        "last_use": np.empty(hot_rows, np.uint32),
        "hot": np.empty((hot_rows, ROW_BYTES), np.uint8) if hot else None,
        "step": np.zeros(1, np.uint32),
    }
    p = lambda a: None if a is None else ctypes.c_void_p(a.ctypes.data)
    _check(lib().kvo_debug_dump_layer(ctx, layer, p(d["pos2slot"]), p(d["slot2pos"]), p(d["last_use"]),
                                      p(d["hot"]), p(d["step"])), "kvo_debug_dump_layer")
    d["step"] = int(d["step"][0])
    return d


def kvo_set_policy(ctx: int, policy: int) -> None:
    """POLICY_LRU or POLICY_CIRCULAR; only before the context's first resolve."""
    _check(lib().kvo_set_policy(ctx, policy), "kvo_set_policy")


def kvo_set_gather_mode(ctx: int, mode: int, auto_miss_pct: int = 0) -> None:
    """GATHER_LOADS, GATHER_STAGED or GATHER_AUTO (staged for CTAs whose
    misses are at least auto_miss_pct percent of their entries)."""
    _check(lib().kvo_set_gather_mode(ctx, mode, auto_miss_pct), "kvo_set_gather_mode")


def kvo_set_recent_ring(ctx: int, rows: int) -> None:
    """0 (no ring) or a power of two in [128, 65536]; before the first append."""
    _check(lib().kvo_set_recent_ring(ctx, rows), "kvo_set_recent_ring")


def kvo_flush_ring(ctx: int, layer: int, stream=None) -> None:
    _check(lib().kvo_flush_ring(ctx, layer, _stream_ptr(stream)), "kvo_flush_ring")


def kvo_ram_length(ctx: int, layer: int) -> int:
    n = _i64()
    _check(lib().kvo_ram_length(ctx, layer, ctypes.byref(n)), "kvo_ram_length")
    return n.value


def kvo_debug_read_history(ctx: int, layer: int, start: int, count: int):
    import numpy as np
    out = np.empty((count, ROW_BYTES), np.uint8)
    _check(lib().kvo_debug_read_history(ctx, layer, start, count, ctypes.c_void_p(out.ctypes.data)),
           "kvo_debug_read_history")
    return out


def kvo_debug_layer_counters(ctx: int, layer: int) -> dict:
    import numpy as np
    c = np.zeros(8, np.uint32)
    _check(lib().kvo_debug_layer_counters(ctx, layer, ctypes.c_void_p(c.ctypes.data)), "kvo_debug_layer_counters")
    return {"step": int(c[0]), "length": int(c[1]), "queue_head": int(c[2]), "queue_tail": int(c[3]),
            "queue_buffer": int(c[4]), "hand": int(c[5])}


def kvo_debug_record_evictions(ctx: int, on: bool) -> None:
    _check(lib().kvo_debug_record_evictions(ctx, 1 if on else 0), "kvo_debug_record_evictions")


def kvo_debug_evictions(ctx: int, layer: int) -> list:
    import numpy as np
    buf = np.zeros(3 * MAX_ROUND, np.int32)
    n = _i32()
    _check(lib().kvo_debug_evictions(ctx, layer, ctypes.c_void_p(buf.ctypes.data), MAX_ROUND, ctypes.byref(n)),
           "kvo_debug_evictions")
    return [tuple(int(x) for x in buf[3 * i:3 * i + 3]) for i in range(n.value)]


def kvo_probe_host_read(src_pinned, sink, stream=None) -> None:
    """src_pinned: pinned CPU tensor (multiple of 16 bytes); sink: 16-byte CUDA tensor."""
    _check(lib().kvo_probe_host_read(ctypes.c_void_p(src_pinned.data_ptr()),
                                     src_pinned.numel() * src_pinned.element_size(),
                                     _dev_ptr(sink), _stream_ptr(stream)), "kvo_probe_host_read")


def kvo_probe_host_touch(addr: int, nbytes: int, stride: int, sink, stream=None) -> None:
    """One 16-byte zero-copy load every `stride` bytes of pinned host memory
    at `addr` (an address, e.g. Context.history_host); sink: 16-byte CUDA tensor."""
    _check(lib().kvo_probe_host_touch(ctypes.c_void_p(addr), nbytes, stride, _dev_ptr(sink), _stream_ptr(stream)),
           "kvo_probe_host_touch")


class Context:
    """Owns one kvo context; methods forward to the kvo_* calls above."""

    def __init__(self, layers: int, history_cap: int, hot_rows: int, row_bytes: int = ROW_BYTES):
        self.layers, self.history_cap, self.hot_rows = layers, history_cap, hot_rows
        self.handle = kvo_create(layers, history_cap, hot_rows, row_bytes)

    def close(self):
        if self.handle:
            kvo_destroy(self.handle)
            self.handle = None

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def append_rows(self, layer, rows, stream=None):
        kvo_append_rows(self.handle, layer, rows, stream)

    def select_topk(self, scores, k, idx=None, stream=None):
        return kvo_select_topk(self.handle, scores, k, idx, stream)

    def select_topk_batch(self, scores, k, n=None, idx=None, stream=None):
        return kvo_select_topk_batch(self.handle, scores, k, n, idx, stream)

    def resolve_gather(self, layer, idx, out_rows=None, out_bf16=None, stream=None):
        kvo_resolve_gather(self.handle, layer, idx, out_rows, out_bf16, stream)

    def resolve_gather_multi(self, layer, idx, out_rows=None, out_bf16=None, stream=None):
        kvo_resolve_gather_multi(self.handle, layer, idx, out_rows, out_bf16, stream)

    def decode_step(self, layer, new_rows, scores, k, idx=None, out_rows=None, out_bf16=None, stream=None):
        return kvo_decode_step(self.handle, layer, new_rows, scores, k, idx, out_rows, out_bf16, stream)

    def decode_step_host(self, layer, new_rows, scores, k, idx, out_rows=None, out_bf16=None, stream=None):
        return kvo_decode_step_host(self.handle, layer, new_rows, scores, k, idx, out_rows, out_bf16, stream)

    def decode_layers(self, tasks, k, stream=None):
        kvo_decode_layers(self.handle, tasks, k, stream)

    def decode_layers_prepared(self, arr, k, stream=None):
        kvo_decode_layers_prepared(self.handle, arr, k, stream)

    def set_phase_timing(self, on=True):
        _check(lib().kvo_set_phase_timing(self.handle, 1 if on else 0), "kvo_set_phase_timing")

    def touch_history(self, layer=-1, stream=None):
        _check(lib().kvo_touch_history(self.handle, layer, _stream_ptr(stream)), "kvo_touch_history")

    def history_host(self, layer) -> int:
        """Host address of the layer's pinned history (read-only use)."""
        p = ctypes.c_void_p()
        _check(lib().kvo_debug_history_host(self.handle, layer, ctypes.byref(p)), "kvo_debug_history_host")
        return p.value

    def layers_counters(self):
        """(kernels launched by kvo_decode_layers, host seconds spent in its calls)."""
        n, t = ctypes.c_int64(), ctypes.c_double()
        _check(lib().kvo_layers_counters(self.handle, ctypes.byref(n), ctypes.byref(t)), "kvo_layers_counters")
        return n.value, t.value

    def layers_phase_times(self):
        """(select, resolve, gather) milliseconds summed over the recorded
        kvo_decode_layers calls, and the number of calls."""
        ms = (ctypes.c_double * 3)()
        calls = ctypes.c_int64()
        _check(lib().kvo_layers_phase_times(self.handle, ms, ctypes.byref(calls)), "kvo_layers_phase_times")
        return (ms[0], ms[1], ms[2]), calls.value

    def sync(self, stream=None) -> int:
        return kvo_sync(self.handle, stream)

    def stats(self, layer) -> dict:
        return kvo_get_stats(self.handle, layer)

    def history_length(self, layer) -> int:
        return kvo_history_length(self.handle, layer)

    def dump_layer(self, layer, hot=True) -> dict:
        return kvo_debug_dump_layer(self.handle, layer, self.history_cap, self.hot_rows, hot)

    def set_policy(self, policy):
        kvo_set_policy(self.handle, policy)

    def set_gather_mode(self, mode, auto_miss_pct=0):
        kvo_set_gather_mode(self.handle, mode, auto_miss_pct)

    def set_miss_fetch(self, mode, auto_miss_pct=100):
        _check(lib().kvo_set_miss_fetch(self.handle, mode, auto_miss_pct), "kvo_set_miss_fetch")

    def set_recent_ring(self, rows):
        kvo_set_recent_ring(self.handle, rows)

    def flush_ring(self, layer, stream=None):
        kvo_flush_ring(self.handle, layer, stream)

    def ram_length(self, layer) -> int:
        return kvo_ram_length(self.handle, layer)

    def read_history(self, layer, start, count):
        return kvo_debug_read_history(self.handle, layer, start, count)

    def counters(self, layer) -> dict:
        return kvo_debug_layer_counters(self.handle, layer)

    def raise_status(self, bits):
        _check(lib().kvo_debug_raise_status(self.handle, bits), "kvo_debug_raise_status")

    def record_evictions(self, on=True):
        kvo_debug_record_evictions(self.handle, on)

    def evictions(self, layer) -> list:
        return kvo_debug_evictions(self.handle, layer)


# ------------------------------------------------------ session block pool
def kvo_tier_blocks(tier_bytes: int, block_bytes: int) -> int:
    return int(lib().kvo_tier_blocks(tier_bytes, block_bytes))


def kvo_pool_create(layers: int, pool_blocks: int, block_tokens: int, tier_blocks: int,
                    row_bytes: int = ROW_BYTES) -> int:
    h = _vp()
    _check(lib().kvo_pool_create(layers, pool_blocks, block_tokens, row_bytes, tier_blocks, ctypes.byref(h)),
           "kvo_pool_create")
    return h.value


def kvo_pool_destroy(pool: int) -> None:
    _check(lib().kvo_pool_destroy(pool), "kvo_pool_destroy")


def kvo_pool_alloc(pool: int, session: int, tokens: int) -> int:
    """Returns KVO_OK or KVO_ECAPACITY (a refused, rolled-back allocation);
    raises on other errors."""
    st = lib().kvo_pool_alloc(pool, session, tokens)
    if st not in (KVO_OK, KVO_ECAPACITY):
        raise KvoError(st, "kvo_pool_alloc")
    return st


def kvo_pool_write(pool: int, session: int, layer: int, first_token: int, rows, stream=None) -> None:
    """rows: uint8 CUDA tensor [n, 656]."""
    _check(lib().kvo_pool_write(pool, session, layer, first_token, _dev_ptr(rows, "torch.uint8"),
                                rows.numel() // ROW_BYTES, _stream_ptr(stream)), "kvo_pool_write")


def kvo_pool_read(pool: int, session: int, layer: int, first_token: int, out, stream=None) -> None:
    """out: uint8 CUDA tensor [n, 656]."""
    _check(lib().kvo_pool_read(pool, session, layer, first_token, out.numel() // ROW_BYTES,
                               _dev_ptr(out, "torch.uint8"), _stream_ptr(stream)), "kvo_pool_read")


def kvo_pool_fill(pool: int, byte: int, stream=None) -> None:
    _check(lib().kvo_pool_fill(pool, byte, _stream_ptr(stream)), "kvo_pool_fill")


def kvo_store_blocks(pool: int, session: int, stream=None) -> int:
    st = lib().kvo_store_blocks(pool, session, _stream_ptr(stream))
    if st not in (KVO_OK, KVO_ECAPACITY):
        raise KvoError(st, "kvo_store_blocks")
    return st


def kvo_pool_release(pool: int, session: int) -> int:
    """Returns KVO_OK or KVO_EBUSY (a copy that depends on the blocks is pending)."""
    st = lib().kvo_pool_release(pool, session)
    if st not in (KVO_OK, KVO_EBUSY):
        raise KvoError(st, "kvo_pool_release")
    return st


def kvo_restore_blocks(pool: int, sessions, stream=None) -> int:
    ids = (_i32 * len(sessions))(*sessions)
    st = lib().kvo_restore_blocks(pool, ids, len(sessions), _stream_ptr(stream))
    if st not in (KVO_OK, KVO_ECAPACITY):
        raise KvoError(st, "kvo_restore_blocks")
    return st


def kvo_pool_sync(pool: int, stream=None) -> None:
    _check(lib().kvo_pool_sync(pool, _stream_ptr(stream)), "kvo_pool_sync")


def kvo_pool_block_table(pool: int, session: int, layer: int, which: int = 0):
    """Block ids of the session's layer group (which 0: pool, 1: tier), or None."""
    n = _i64()
    _check(lib().kvo_pool_block_table(pool, session, layer, which, None, 0, ctypes.byref(n)),
           "kvo_pool_block_table")
    if n.value == 0:
        return None
    buf = (_i32 * n.value)()
    _check(lib().kvo_pool_block_table(pool, session, layer, which, buf, n.value, ctypes.byref(n)),
           "kvo_pool_block_table")
    return list(buf)


def kvo_pool_get_stats(pool: int) -> dict:
    s = kvo_pool_stats()
    _check(lib().kvo_pool_get_stats(pool, ctypes.byref(s)), "kvo_pool_get_stats")
    return s.as_dict()


def kvo_pool_debug_fail_after(pool: int, which: int, n: int) -> None:
    _check(lib().kvo_pool_debug_fail_after(pool, which, n), "kvo_pool_debug_fail_after")


def kvo_pool_debug_free_queue(pool: int, which: int) -> list:
    n = _i64()
    _check(lib().kvo_pool_debug_free_queue(pool, which, None, 0, ctypes.byref(n)), "kvo_pool_debug_free_queue")
    buf = (_i32 * max(n.value, 1))()
    _check(lib().kvo_pool_debug_free_queue(pool, which, buf, n.value, ctypes.byref(n)),
           "kvo_pool_debug_free_queue")
    return list(buf)[:n.value]


def kvo_copy_blocks_noalloc(src, dst, block_bytes: int, pairs, stream=None) -> None:
    """Copy blocks pairs[i, 0] of `src` to blocks pairs[i, 1] of `dst`
    without allocating (the pair list goes through the library's fixed
    static device array).  src, dst: CUDA tensors or pinned CPU tensors;
    pairs: int32 array-like of shape [n, 2] (host)."""
    import numpy as np
    pr = np.ascontiguousarray(np.asarray(pairs, dtype=np.int32).reshape(-1, 2))

    def ptr(t):
        if not t.is_contiguous():
            raise ValueError("expected a contiguous tensor")
        if not t.is_cuda and not t.is_pinned():
            raise ValueError("expected a CUDA tensor or pinned host memory")
        return ctypes.c_void_p(t.data_ptr())

    # the library cannot see the buffers' sizes: every block id must lie
    # inside its tensor, or the kernel would address past it
    if block_bytes <= 0:
        raise ValueError("block_bytes must be positive")
    nbytes = [t.numel() * t.element_size() for t in (src, dst)]
    if any(b % block_bytes for b in nbytes):
        raise ValueError("block_bytes must divide the byte size of src and dst")
    if pr.shape[0]:
        if int(pr.min()) < 0:
            raise ValueError("block ids must be non-negative")
        if int(pr[:, 0].max()) >= nbytes[0] // block_bytes or int(pr[:, 1].max()) >= nbytes[1] // block_bytes:
            raise ValueError("a block id lies past the end of src or dst")
    _check(lib().kvo_copy_blocks_noalloc(ptr(src), ptr(dst), block_bytes, ctypes.c_void_p(pr.ctypes.data),
                                         pr.shape[0], _stream_ptr(stream)), "kvo_copy_blocks_noalloc")


class Pool:
    """Owns one session block pool; methods forward to the kvo_pool_* calls."""

    def __init__(self, layers: int, pool_blocks: int, block_tokens: int, tier_blocks: int,
                 row_bytes: int = ROW_BYTES):
        self.layers, self.pool_blocks, self.block_tokens, self.tier_blocks = (
            layers, pool_blocks, block_tokens, tier_blocks)
        self.handle = kvo_pool_create(layers, pool_blocks, block_tokens, tier_blocks, row_bytes)

    def close(self):
        if self.handle:
            kvo_pool_destroy(self.handle)
            self.handle = None

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def alloc(self, session, tokens):
        return kvo_pool_alloc(self.handle, session, tokens)

    def write(self, session, layer, first_token, rows, stream=None):
        kvo_pool_write(self.handle, session, layer, first_token, rows, stream)

    def read(self, session, layer, first_token, out, stream=None):
        kvo_pool_read(self.handle, session, layer, first_token, out, stream)

    def fill(self, byte, stream=None):
        kvo_pool_fill(self.handle, byte, stream)

    def store(self, session, stream=None):
        return kvo_store_blocks(self.handle, session, stream)

    def release(self, session):
        return kvo_pool_release(self.handle, session)

    def restore(self, sessions, stream=None):
        return kvo_restore_blocks(self.handle, list(sessions), stream)

    def sync(self, stream=None):
        kvo_pool_sync(self.handle, stream)

    def block_table(self, session, layer, which=0):
        return kvo_pool_block_table(self.handle, session, layer, which)

    def stats(self) -> dict:
        return kvo_pool_get_stats(self.handle)

    def fail_after(self, which, n):
        kvo_pool_debug_fail_after(self.handle, which, n)

    def free_queue(self, which=0) -> list:
        return kvo_pool_debug_free_queue(self.handle, which)
