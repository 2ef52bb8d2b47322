"""The C-ABI library loads and exports every entry point include/kvmm.h declares.

Runs without a GPU: only host-side code paths are exercised (symbol lookup,
status strings, workspace sizing, argument validation that fails before any
launch).
"""
import ctypes
import os
import re

import pytest

from paged_kv_cache_minmax_gb300 import build, kvmm

HEADER = os.path.join(build.INCLUDE, "kvmm.h")


@pytest.fixture(scope="module")
def lib():
    build.build_library()
    return kvmm.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:kvmm_status|size_t|int32_t|const char\*)\s+(\w+)\s*\(", text, flags=re.M)))


def test_header_declares_the_four_calls_and_helpers():
    names = declared_functions()
    for n in ("kv_minmax_update", "page_score_topk", "sparse_paged_decode_attn", "topk_promotion_diff",
              "kvmm_workspace_size", "kvmm_auto_splits", "kvmm_status_string", "kvmm_last_cuda_error"):
        assert n in names


def test_every_declared_function_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), f"{name} declared in kvmm.h but not exported"


def test_status_strings(lib):
    for code in range(5):
        assert kvmm.status_string(code)
    assert kvmm.status_string(0) == "ok"
    assert "unknown" in kvmm.status_string(99)


def test_workspace_size_and_shape_checks(lib):
    s = kvmm.make_shape(8, 32, 32, 8, 128, 16, 2048, 128, 8 * 32 * 8 * 2048)
    n = kvmm.workspace_size(s, 4)
    units = 8 * 8
    assert n >= units * 2048 * 4  # the score buffer
    assert n >= units * 4 * 4 * 128 * 4  # split partials
    assert kvmm.workspace_size(kvmm.make_shape(1, 1, 4, 1, 96, 16, 8, 4, 8), 1) == 0  # D=96 unsupported
    assert kvmm.workspace_size(kvmm.make_shape(1, 1, 4, 1, 64, 8, 8, 4, 8), 1) == 0  # T=8 unsupported
    assert kvmm.workspace_size(kvmm.make_shape(1, 1, 36, 4, 64, 16, 8, 4, 8), 1) == 0  # G=9 unsupported
    assert kvmm.workspace_size(kvmm.make_shape(1, 1, 4, 1, 64, 16, 8, 40000, 8), 1) == 0  # Kmax too large


def test_validation_rejects_before_any_launch(lib):
    s = kvmm.make_shape(1, 1, 4, 1, 64, 16, 64, 8, 64)
    P = ctypes.c_void_p
    fake = P(0x10000)  # aligned, never dereferenced: validation fails first
    bad_align = P(0x10002)
    # null pointers
    assert lib.page_score_topk(ctypes.byref(s), 0, None, None, None, None, 8, 0, None, None, None, None, 0, 0,
                               None, None) == kvmm.INVALID_ARG
    # K out of range, layer out of range, bad group flag
    args = [fake, fake, fake, None, 8, 0, fake, fake, None, fake, 1 << 20, 0, None, None]
    assert lib.page_score_topk(ctypes.byref(s), 0, *args[:4], 9, *args[5:]) == kvmm.INVALID_ARG
    assert lib.page_score_topk(ctypes.byref(s), 1, *args) == kvmm.INVALID_ARG
    assert lib.page_score_topk(ctypes.byref(s), 0, *args[:5], 2, *args[6:]) == kvmm.INVALID_ARG
    # misaligned bf16 array
    assert lib.page_score_topk(ctypes.byref(s), 0, bad_align, *args[1:]) == kvmm.INVALID_ARG
    # workspace too small
    assert lib.page_score_topk(ctypes.byref(s), 0, *args[:9], fake, 16, 0, None, None) == kvmm.WORKSPACE_TOO_SMALL
    # an unknown flag bit
    assert lib.page_score_topk(ctypes.byref(s), 0, *args[:11], 2, None, None) == kvmm.INVALID_ARG
    # unsupported shape
    s2 = kvmm.make_shape(1, 1, 4, 1, 80, 16, 64, 8, 64)
    assert lib.page_score_topk(ctypes.byref(s2), 0, *args) == kvmm.UNSUPPORTED_SHAPE
    # update: only one of new_k / new_v
    assert lib.kv_minmax_update(ctypes.byref(s), 0, fake, None, 1, fake, fake, fake, fake, fake, fake, None,
                                None) == kvmm.INVALID_ARG
    # attention: non-finite scale
    assert lib.sparse_paged_decode_attn(ctypes.byref(s), 0, fake, fake, fake, fake, fake, fake, fake,
                                        float("nan"), 1, fake, None, None, 0, 0, None, None) == kvmm.INVALID_ARG
    assert lib.sparse_paged_decode_attn(ctypes.byref(s), 0, fake, fake, fake, fake, fake, fake, fake,
                                        0.0, 0, fake, None, None, 0, 8, None, None) == kvmm.INVALID_ARG
    # fused select + attend: null pointers, bad K, non-finite scale, small workspace
    fa = [fake, fake, fake, fake, fake, fake, None, 8, 0, 0.0, fake, fake, None, fake, None, fake, 1 << 20, None,
          None]
    assert lib.page_score_topk_attn(ctypes.byref(s), 0, None, *fa[1:]) == kvmm.INVALID_ARG
    assert lib.page_score_topk_attn(ctypes.byref(s), 0, *fa[:7], 9, *fa[8:]) == kvmm.INVALID_ARG
    assert lib.page_score_topk_attn(ctypes.byref(s), 0, *fa[:9], float("inf"), *fa[10:]) == kvmm.INVALID_ARG
    assert lib.page_score_topk_attn(ctypes.byref(s), 0, *fa[:16], 64, None, None) == kvmm.WORKSPACE_TOO_SMALL
    # decode_layer: null query, an unknown flag bit
    da = [fake, None, None, 0, None, None, fake, fake, fake, fake, fake, None, 8, 0, 0.0, fake, fake, None, fake,
          None, None, 0]
    assert lib.decode_layer(ctypes.byref(s), 0, None, *da[1:], 0, None, None) == kvmm.INVALID_ARG
    assert lib.decode_layer(ctypes.byref(s), 0, *da, 2, None, None) == kvmm.INVALID_ARG
    assert lib.decode_layer(ctypes.byref(s), 0, *da, kvmm.DECODE_EARLY_READS | 4, None, None) == kvmm.INVALID_ARG
    # diff: missing promoted list
    assert lib.topk_promotion_diff(ctypes.byref(s), 0, None, fake, fake, fake, fake, 1, None, fake, None, None,
                                   None, None, None) == kvmm.INVALID_ARG
    # promotion: missing host store, negative grid bound
    pa = (None, fake, fake, fake, fake, fake, fake, fake, fake, fake, None, None, None)
    assert lib.promote_pages(ctypes.byref(s), 0, *pa, 0, None, None) == kvmm.INVALID_ARG
    assert lib.promote_pages(ctypes.byref(s), 0, None, fake, fake, fake, fake, None, fake, fake, fake, fake, None,
                             None, None, 0, None, None) == kvmm.INVALID_ARG
    assert lib.promote_pages(ctypes.byref(s), 0, None, fake, fake, fake, fake, fake, fake, fake, fake, fake, None,
                             None, None, -1, None, None) == kvmm.INVALID_ARG
    # history record: slot outside the ring, missing history
    assert lib.topk_history_record(ctypes.byref(s), 0, fake, fake, fake, 4, 4, fake, fake, fake, None,
                                   None) == kvmm.INVALID_ARG
    assert lib.topk_history_record(ctypes.byref(s), 0, fake, fake, fake, 4, 0, None, fake, fake, None,
                                   None) == kvmm.INVALID_ARG
    # stability: lag must be below the window, the window inside the ring, the fraction in [0, 1]
    ok = (fake, fake, fake, 8, 8, 7, 1)
    assert lib.topk_stability_rco(ctypes.byref(s), *ok[:6], 8, 0.25, fake, None, None, None,
                                  None) == kvmm.INVALID_ARG
    assert lib.topk_stability_rco(ctypes.byref(s), *ok[:4], 9, 7, 1, 0.25, fake, None, None, None,
                                  None) == kvmm.INVALID_ARG
    assert lib.topk_stability_rco(ctypes.byref(s), *ok, 1.5, fake, None, None, None, None) == kvmm.INVALID_ARG
    assert lib.topk_stability_rco(ctypes.byref(s), *ok, 0.25, None, None, None, None, None) == kvmm.INVALID_ARG


def test_binding_fails_loudly_without_library(tmp_path):
    with pytest.raises(RuntimeError, match="not found"):
        kvmm.load(str(tmp_path / "missing.so"))
