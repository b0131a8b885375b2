"""Host-side checks of the C ABI that need no GPU: the library builds for
sm_103a, exports every function include/kvo.h declares, and rejects bad
arguments before touching the device."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def kvo():
    from gather_radix_top_gb300 import build, kvo as K
    build.build()
    return K


def _declared():
    text = open(os.path.join(ROOT, "include", "kvo.h")).read()
    return sorted(set(re.findall(r"\b(kvo_[a-z_]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = _declared()
    for n in ("kvo_create", "kvo_destroy", "kvo_append_rows", "kvo_select_topk", "kvo_resolve_gather",
              "kvo_sync", "kvo_get_stats", "kvo_debug_dump_layer"):
        assert n in names


def test_library_exports_every_declared_symbol(kvo):
    L = kvo.lib()
    for n in _declared():
        assert hasattr(L, n), n
    assert sorted(kvo.EXPORTED) == _declared()


def test_bad_arguments_rejected_without_a_device(kvo):
    L = kvo.lib()
    h = ctypes.c_void_p()
    assert L.kvo_create(0, 10, 4, 656, ctypes.byref(h)) == kvo.KVO_EINVAL
    assert L.kvo_create(1, 10, 4, 640, ctypes.byref(h)) == kvo.KVO_EINVAL
    assert L.kvo_create(1, 10, kvo.MAX_HOT_ROWS + 1, 656, ctypes.byref(h)) == kvo.KVO_EINVAL
    assert L.kvo_create(1, 2 ** 31, 4, 656, ctypes.byref(h)) == kvo.KVO_EINVAL
    assert h.value is None
    assert L.kvo_sync(None, None) == kvo.KVO_EINVAL
    assert L.kvo_select_topk(None, None, 10, 5, None, None) == kvo.KVO_EINVAL
    assert L.kvo_resolve_gather(None, 0, None, 5, None, None, None) == kvo.KVO_EINVAL
    assert L.kvo_append_rows(None, 0, None, 1, None) == kvo.KVO_EINVAL
    assert L.kvo_destroy(None) == kvo.KVO_EINVAL
    assert L.kvo_set_policy(None, 0) == kvo.KVO_EINVAL
    assert L.kvo_decode_layers(None, None, 1, 16, None) == kvo.KVO_EINVAL
    assert L.kvo_set_miss_fetch(None, 0, 0) == kvo.KVO_EINVAL
    assert L.kvo_set_phase_timing(None, 1) == kvo.KVO_EINVAL
    assert L.kvo_layers_phase_times(None, None, None) == kvo.KVO_EINVAL
    assert L.kvo_layers_counters(None, None, None) == kvo.KVO_EINVAL
    assert L.kvo_touch_history(None, -1, None) == kvo.KVO_EINVAL
    assert L.kvo_debug_raise_status(None, 4) == kvo.KVO_EINVAL
    assert L.kvo_probe_host_touch(None, 16, 16, None, None) == kvo.KVO_EINVAL
    assert kvo.status_string(kvo.KVO_ERANGE) == "selected position outside the history"


def test_pool_bad_arguments_rejected_without_a_device(kvo):
    L = kvo.lib()
    h = ctypes.c_void_p()
    assert L.kvo_pool_create(0, 8, 16, 656, 8, ctypes.byref(h)) == kvo.KVO_EINVAL
    assert L.kvo_pool_create(1, 0, 16, 656, 8, ctypes.byref(h)) == kvo.KVO_EINVAL
    assert L.kvo_pool_create(1, 8, 0, 656, 8, ctypes.byref(h)) == kvo.KVO_EINVAL
    assert L.kvo_pool_create(1, 8, 16, 640, 8, ctypes.byref(h)) == kvo.KVO_EINVAL
    assert L.kvo_pool_create(1, 8, 16, 656, -1, ctypes.byref(h)) == kvo.KVO_EINVAL
    assert L.kvo_pool_create(1, 2 ** 31, 16, 656, 8, ctypes.byref(h)) == kvo.KVO_EINVAL
    assert h.value is None
    assert L.kvo_pool_alloc(None, 0, 10) == kvo.KVO_EINVAL
    assert L.kvo_store_blocks(None, 0, None) == kvo.KVO_EINVAL
    assert L.kvo_restore_blocks(None, None, 1, None) == kvo.KVO_EINVAL
    assert L.kvo_pool_release(None, 0) == kvo.KVO_EINVAL
    assert L.kvo_pool_destroy(None) == kvo.KVO_EINVAL


def test_tier_blocks_matches_the_printed_sizes(kvo):
    # "A 60k-token context comes back off disk ..." README: 32 GiB -> 632 and
    # 260 GB -> 4785 blocks of 54,329,344 bytes
    assert kvo.kvo_tier_blocks(32 * 2 ** 30, 54_329_344) == 632
    assert kvo.kvo_tier_blocks(260_000_000_000, 54_329_344) == 4785
    assert kvo.kvo_tier_blocks(-1, 10) == -1 and kvo.kvo_tier_blocks(10, 0) == -1


def test_binding_has_no_fallback(tmp_path, monkeypatch):
    from gather_radix_top_gb300 import build, kvo as K
    monkeypatch.setattr(build, "LIB", str(tmp_path / "missing.so"))
    monkeypatch.setattr(K, "_lib", None)
    with pytest.raises(ImportError):
        K.lib()
