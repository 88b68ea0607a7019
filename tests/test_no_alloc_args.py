"""Host-side argument checks of nvfp4_sparse_mla_decode_no_alloc (no GPU needed): a call with
a bad argument returns the same status as nvfp4_sparse_mla_decode, before the library asks
the CUDA runtime for anything, also for split counts that would use its scratch array."""
import ctypes

import pytest

import nvfp4_kv_cache_sparse_gb300 as lib


def _call(cdll, fn, q, cache, idx, out, lse, splits, extra):
    args = [q, cache, 100, 352, idx, 2, 1, 128, 512, ctypes.c_float(0.1), None, out, lse, splits]
    return getattr(cdll, fn)(*(args + extra))


@pytest.mark.parametrize("splits", [2, 4, 0])
@pytest.mark.parametrize("null", ["q", "cache", "idx", "out", "lse"])
def test_null_pointers_are_rejected_before_any_device_query(splits, null):
    cdll = lib.load(build_if_missing=True)
    good = ctypes.c_void_p(1 << 20)   # 16-byte aligned, never dereferenced
    ptrs = {k: good for k in ("q", "cache", "idx", "out", "lse")}
    ptrs[null] = None
    st = _call(cdll, "nvfp4_sparse_mla_decode_no_alloc", ptrs["q"], ptrs["cache"], ptrs["idx"], ptrs["out"],
               ptrs["lse"], splits, [None, None])
    st_ws = _call(cdll, "nvfp4_sparse_mla_decode", ptrs["q"], ptrs["cache"], ptrs["idx"], ptrs["out"],
                  ptrs["lse"], splits, [None, 0, None, None])
    assert st == lib.ERR_INVALID_ARG
    assert st == st_ws


def test_misaligned_and_unsupported_arguments_match_the_workspace_entry_point():
    cdll = lib.load(build_if_missing=True)
    good = ctypes.c_void_p(1 << 20)
    odd = ctypes.c_void_p((1 << 20) + 8)   # not 16-byte aligned
    st = _call(cdll, "nvfp4_sparse_mla_decode_no_alloc", odd, good, good, good, good, 4, [None, None])
    assert st == lib.ERR_INVALID_ARG
    args = [good, good, 100, 352, good, 2, 1, 96, 512, ctypes.c_float(0.1), None, good, good, 4]   # h_q 96
    assert cdll.nvfp4_sparse_mla_decode_no_alloc(*(args + [None, None])) == lib.ERR_UNSUPPORTED
    assert cdll.nvfp4_sparse_mla_decode(*(args + [None, 0, None, None])) == lib.ERR_UNSUPPORTED


def test_decode_plan_checks_its_arguments_without_a_device():
    cdll = lib.load(build_if_missing=True)
    sp, k = ctypes.c_int32(0), ctypes.c_int32(0)
    assert cdll.nvfp4_sparse_mla_decode_plan(1, 1, 128, 64, 352, 1, None, ctypes.byref(k)) == lib.ERR_INVALID_ARG
    assert cdll.nvfp4_sparse_mla_decode_plan(1, 1, 96, 64, 352, 1, ctypes.byref(sp), ctypes.byref(k)) == lib.ERR_UNSUPPORTED
    assert cdll.nvfp4_sparse_mla_decode_plan(1, 1, 128, 0, 352, 1, ctypes.byref(sp), ctypes.byref(k)) == lib.ERR_INVALID_ARG
