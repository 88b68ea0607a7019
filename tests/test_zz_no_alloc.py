"""nvfp4_sparse_mla_decode_no_alloc, called through the C ABI, against nvfp4_sparse_mla_decode.

The no-allocation variant exists for callers that cannot give the library device scratch
memory (a device-memory budget fixed at start-up, or code that must not call cudaMalloc /
cudaFree because they can synchronize the device). It keeps its scratch in a library-owned
fixed array shared by all calls, so this test makes two calls in a row with different inputs
on the same stream and checks each against the workspace-taking entry point with the same
split count. The file is named to be collected last, and it builds everything it needs
itself, so it also passes alone in a fresh process."""
import ctypes

import numpy as np
import pytest
import torch

import nvfp4_kv_cache_sparse_gb300 as lib
from synth.pool import fill_pool

pytestmark = pytest.mark.gpu
DEV = "cuda"
ATOL, RTOL, LSE_TOL = 1e-2, 1e-2, 1e-3


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _no_alloc(cdll, q, cache, idx, sm_scale, sink, out, lse, splits, status):
    B, s_q, h_q, _ = q.shape
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return cdll.nvfp4_sparse_mla_decode_no_alloc(
        _ptr(q), _ptr(cache), cache.shape[0], cache.shape[1], _ptr(idx), B, s_q, h_q, idx.shape[2],
        ctypes.c_float(sm_scale), _ptr(sink), _ptr(out), _ptr(lse), splits, _ptr(status), stream)


def test_no_alloc_matches_the_workspace_entry_point_on_two_calls_in_a_row():
    cdll = lib.load(build_if_missing=True)
    rng = np.random.default_rng(2024)
    B, s_q, h_q, topk, n_slots, splits = 3, 2, 128, 700, 5000, 4
    cache = fill_pool(lib.quantize_append, n_slots, 352, 99, DEV)
    sink = torch.from_numpy(rng.standard_normal(h_q).astype(np.float32)).to(DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    assert lib.workspace_size(B, s_q, h_q, topk, 352, splits) > 0          # this problem uses scratch
    for call in range(2):
        q = torch.from_numpy(rng.standard_normal((B, s_q, h_q, 576)).astype(np.float32)).to(torch.bfloat16).to(DEV)
        idx = np.stack([rng.choice(n_slots, topk, replace=False) for _ in range(B * s_q)]).astype(np.int32)
        idx[rng.random(idx.shape) < 0.1] = -1
        idx = torch.from_numpy(idx.reshape(B, s_q, topk)).to(DEV)
        out = torch.full((B, s_q, h_q, 512), float("nan"), dtype=torch.bfloat16, device=DEV)
        lse = torch.full((B, s_q, h_q), float("nan"), dtype=torch.float32, device=DEV)
        st = _no_alloc(cdll, q, cache, idx, 1 / 24, sink, out, lse, splits, status)
        assert st == lib.OK, lib.status_string(st)
        ref_out, ref_lse = lib.sparse_mla_decode(q, cache, idx, 1 / 24, attn_sink=sink, num_splits=splits)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        o, r = out.float(), ref_out.float()
        assert torch.all((o - r).abs() <= ATOL + RTOL * r.abs()), f"call {call}: out differs"
        assert torch.all((lse - ref_lse).abs() <= LSE_TOL), f"call {call}: lse differs"


def test_no_alloc_rejects_problems_beyond_its_scratch_limit():
    cdll = lib.load(build_if_missing=True)
    limit = 32 << 20
    # 64 splits x 128 heads x 512 f16 per row is 8 MiB: five rows need more than the limit
    assert lib.workspace_size(5, 1, 128, 4096, 352, 64) > limit
    q = torch.zeros((5, 1, 128, 576), dtype=torch.bfloat16, device=DEV)
    idx = torch.zeros((5, 1, 4096), dtype=torch.int32, device=DEV)
    cache = torch.zeros((16, 352), dtype=torch.uint8, device=DEV)
    out = torch.zeros((5, 1, 128, 512), dtype=torch.bfloat16, device=DEV)
    lse = torch.zeros((5, 1, 128), dtype=torch.float32, device=DEV)
    st = _no_alloc(cdll, q, cache, idx, 0.1, None, out, lse, 64, None)
    assert st == lib.ERR_WORKSPACE


@pytest.mark.parametrize("record_bytes,splits", [(352, 0), (432, 2), (352, 3)])
def test_no_alloc_is_bit_identical_to_the_workspace_entry_point(record_bytes, splits):
    """Both entry points run the same kernels with the same split count (num_splits = 0: the
    library's own choice, which both must make alike), so out and lse agree bit for bit."""
    cdll = lib.load(build_if_missing=True)
    rng = np.random.default_rng(7 + record_bytes + splits)
    B, s_q, h_q, topk, n_slots = 2, 1, 128, 900, 3000
    cache = fill_pool(lib.quantize_append, n_slots, record_bytes, 5, DEV)
    sink = torch.from_numpy(rng.standard_normal(h_q).astype(np.float32)).to(DEV)
    q = torch.from_numpy(rng.standard_normal((B, s_q, h_q, 576)).astype(np.float32)).to(torch.bfloat16).to(DEV)
    idx = np.stack([rng.choice(n_slots, topk, replace=False) for _ in range(B * s_q)]).astype(np.int32)
    idx[rng.random(idx.shape) < 0.05] = -1
    idx = torch.from_numpy(idx.reshape(B, s_q, topk)).to(DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    out = torch.full((B, s_q, h_q, 512), float("nan"), dtype=torch.bfloat16, device=DEV)
    lse = torch.full((B, s_q, h_q), float("nan"), dtype=torch.float32, device=DEV)
    st = _no_alloc(cdll, q, cache, idx, 1 / 24, sink, out, lse, splits, status)
    assert st == lib.OK, lib.status_string(st)
    ref_out, ref_lse = lib.sparse_mla_decode(q, cache, idx, 1 / 24, attn_sink=sink, num_splits=splits)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert torch.equal(out, ref_out)
    assert torch.equal(lse, ref_lse)


def test_decode_plan_matches_the_launch_structure():
    """One kernel per call when the splits merge inside the decode grid (2-4 splits, one wave of
    clusters) or there is one split; two (decode + merge grid) otherwise."""
    assert lib.decode_plan(32, 1, 128, 2048, 352, 1) == (1, 1)
    assert lib.decode_plan(32, 1, 128, 2048, 352, 2) == (2, 1)
    assert lib.decode_plan(32, 1, 128, 2048, 352, 8) == (8, 2)
    assert lib.decode_plan(32, 1, 128, 2048, 352, 0)[0] >= 1
    assert lib.decode_plan(4, 1, 64, 2048, 352, 2) == (2, 2)       # h_q 64: the merge grid follows
    assert lib.decode_plan(0, 1, 128, 2048, 352, 2)[1] == 0
