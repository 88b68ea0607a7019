"""Sparse MLA decode on the GPU against the CPU oracle.

Tolerances: |out - ref| <= 1e-2 + 1e-2 |ref| element by element and |lse - ref| <= 1e-3
(-inf must match exactly). The dequantized keys are exact, so the 16-bit rounding of P, the
fp32 accumulation order in the tensor core and the final bf16 rounding of `out` are the only
differences from the fp64 oracle.

Small problems are compared in full; the benchmark-sized workloads are compared on sampled
query rows (the oracle recomputes those rows from records it quantizes itself)."""
import math

import numpy as np
import pytest
import torch

import nvfp4_kv_cache_sparse_gb300 as lib
import oracle
import synth
from synth.pool import fill_pool

pytestmark = pytest.mark.gpu
DEV = "cuda"
ATOL, RTOL, LSE_TOL = 1e-2, 1e-2, 1e-3


def assert_close(out_gpu: torch.Tensor, lse_gpu: torch.Tensor, out_ref: np.ndarray, lse_ref: np.ndarray):
    o = out_gpu.float().cpu().numpy().reshape(out_ref.shape).astype(np.float64)
    l = lse_gpu.cpu().numpy().reshape(lse_ref.shape).astype(np.float64)
    err = np.abs(o - out_ref)
    bad = err > ATOL + RTOL * np.abs(out_ref)
    assert not bad.any(), f"{bad.sum()} of {bad.size} out values off; worst {err.max():.3g}"
    inf_ref = np.isneginf(lse_ref)
    assert np.array_equal(np.isneginf(l), inf_ref), "empty rows disagree"
    if (~inf_ref).any():
        lerr = np.abs(l[~inf_ref] - lse_ref[~inf_ref])
        assert lerr.max() <= LSE_TOL, f"lse off by {lerr.max():.3g}"


def oracle_pool(seed: int, n: int, R: int) -> np.ndarray:
    lat, rope = synth.pool_rows(seed, torch.arange(n))
    return oracle.quantize_records(synth.bf16_bits(lat), synth.bf16_bits(rope), R)


def run_small(q_f32: np.ndarray, idx: np.ndarray, R: int, pool_n: int, pool_seed: int, sm_scale: float,
              sink=None, splits=0):
    """q_f32 [B, s_q, H, 576]; idx [B, s_q, topk]. Pool built by the GPU quantizer; the oracle
    uses its own records of the same contents."""
    B, s_q, H, _ = q_f32.shape
    q = torch.from_numpy(q_f32.astype(np.float32)).to(torch.bfloat16)
    cache = fill_pool(lib.quantize_append, pool_n, R, pool_seed, DEV)
    recs = oracle_pool(pool_seed, pool_n, R)
    assert np.array_equal(cache.cpu().numpy(), recs)
    sink_t = None if sink is None else torch.from_numpy(np.asarray(sink, dtype=np.float32)).to(DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    out, lse = lib.sparse_mla_decode(q.to(DEV), cache, torch.from_numpy(idx.astype(np.int32)).to(DEV), sm_scale,
                                     attn_sink=sink_t, num_splits=splits, dev_status=status)
    torch.cuda.synchronize()
    ref_out, ref_lse = oracle.sparse_mla_decode(synth.bf16_bits(q), recs, idx.reshape(B * s_q, -1), sm_scale,
                                                attn_sink=None if sink is None else np.asarray(sink, np.float32))
    return out, lse, ref_out.reshape(B, s_q, H, 512), ref_lse.reshape(B, s_q, H), int(status.item())


@pytest.mark.parametrize("splits", [0, 1, 2])
def test_tiny_workload(splits):
    w = synth.tiny_decode(seed=0)
    cache = fill_pool(lib.quantize_append, w.num_slots, w.record_bytes, w.pool_seed, DEV)
    recs = oracle_pool(w.pool_seed, w.num_slots, w.record_bytes)
    assert np.array_equal(cache.cpu().numpy(), recs)
    out, lse = lib.sparse_mla_decode(w.q.to(DEV), cache, w.indices.to(DEV), w.sm_scale, num_splits=splits)
    torch.cuda.synchronize()
    ref_out, ref_lse = oracle.sparse_mla_decode(synth.bf16_bits(w.q), recs, w.indices.numpy().reshape(1, -1),
                                                w.sm_scale)
    assert_close(out, lse, ref_out, ref_lse)


CASES = [
    # (B, s_q, H, topk, R, sink, splits)
    (1, 1, 128, 64, 352, False, 1),
    (2, 1, 128, 96, 352, True, 2),
    (3, 2, 64, 50, 352, True, 0),
    (2, 1, 64, 1, 352, False, 1),
    (1, 1, 128, 33, 432, False, 3),
    (4, 1, 128, 256, 432, True, 0),
    (2, 2, 64, 200, 432, False, 4),
    (1, 1, 64, 2048, 352, True, 5),
]


@pytest.mark.parametrize("B,s_q,H,topk,R,sink,splits", CASES)
def test_small_problems(B, s_q, H, topk, R, sink, splits):
    rng = np.random.default_rng(B * 1000 + topk + R + splits)
    n_slots = max(300, topk + 10)
    q = rng.standard_normal((B, s_q, H, 576)).astype(np.float32)
    idx = np.stack([rng.choice(n_slots, size=topk, replace=topk > n_slots) for _ in range(B * s_q)])
    idx = idx.reshape(B, s_q, topk).astype(np.int32)
    idx[rng.random(idx.shape) < 0.15] = -1
    sk = rng.standard_normal(H).astype(np.float32) if sink else None
    out, lse, ref_out, ref_lse, st = run_small(q, idx, R, n_slots, 31 + topk, 1 / math.sqrt(576), sk, splits)
    assert st == 0
    assert_close(out, lse, ref_out, ref_lse)


def test_edge_rows_empty_single_duplicate_out_of_range():
    rng = np.random.default_rng(9)
    n_slots, topk, H = 128, 40, 64
    q = rng.standard_normal((5, 1, H, 576)).astype(np.float32)
    idx = np.full((5, 1, topk), -1, dtype=np.int32)             # row 0: every entry masked
    idx[1, 0, 17] = 5                                           # row 1: a single used entry
    idx[2, 0, :] = 7                                            # row 2: one slot 40 times
    idx[3, 0, :] = rng.choice(n_slots, topk, replace=False)     # row 3: normal, plus entries >= num_slots
    idx[3, 0, ::9] = n_slots + 3
    idx[4, 0, :20] = rng.choice(n_slots, 20, replace=False)     # row 4: all used entries in the first tile
    for splits in (1, 2):
        out, lse, ref_out, ref_lse, st = run_small(q, idx, 352, n_slots, 77, 0.05, rng.standard_normal(H), splits)
        assert st == lib.DEV_INDEX_OUT_OF_RANGE
        assert_close(out, lse, ref_out, ref_lse)
        o = out.float().cpu().numpy()
        assert np.all(o[0] == 0) and np.all(np.isneginf(lse[0].cpu().numpy()))


@pytest.mark.parametrize("H", [64, 128])
@pytest.mark.parametrize("e", [-30, -12, 0, 20])
def test_query_magnitudes_outside_the_f16_range(e, H):
    """Queries of magnitude 2^e with sm_scale 2^-e / 24 give ordinary logits: q enters the
    tensor core unchanged at any magnitude (tiny rows, rows above the f16 maximum, a zero head,
    and a head whose odd dims are 2^-20 of the rest)."""
    rng = np.random.default_rng(40 + e + H)
    B, topk, n_slots = 2, 150, 400
    q = rng.standard_normal((B, 1, H, 576)).astype(np.float32)
    q[:, :, 5] = 0.0
    q[:, :, 7, 1::2] *= 2.0 ** -20
    q *= 2.0 ** e
    idx = np.stack([rng.choice(n_slots, size=topk, replace=False) for _ in range(B)]).reshape(B, 1, topk)
    idx = idx.astype(np.int32)
    for splits in (1, 2):
        out, lse, ref_out, ref_lse, st = run_small(q, idx, 352, n_slots, 13, 2.0 ** -e / 24.0, None, splits)
        assert st == 0
        assert_close(out, lse, ref_out, ref_lse)
        assert np.allclose(lse.cpu().numpy()[:, :, 5], math.log(topk), atol=1e-4)


@pytest.mark.parametrize("H", [64, 128])
def test_zero_query_is_mean_of_values_and_splits_agree(H):
    rng = np.random.default_rng(10)
    q = np.zeros((2, 1, H, 576), dtype=np.float32)
    idx = np.stack([rng.choice(1000, size=512, replace=False) for _ in range(2)]).reshape(2, 1, 512).astype(np.int32)
    outs = []
    for splits in (1, 2, 4, 8):
        out, lse, ref_out, ref_lse, st = run_small(q, idx, 352, 1000, 5, 0.04, None, splits)
        assert_close(out, lse, ref_out, ref_lse)
        assert np.allclose(lse.cpu().numpy(), math.log(512), atol=1e-4)
        outs.append(out.float().cpu())
    for o in outs[1:]:
        assert torch.allclose(o, outs[0], atol=1e-2, rtol=1e-2)


@pytest.mark.parametrize("H,R,sm_scale", [(64, 352, 0.6), (64, 432, -0.45), (64, 352, 1.5), (128, 352, 0.6),
                                           (128, 432, -0.45)])
def test_reference_maximum_moves_on_later_tiles(H, R, sm_scale):
    """|sm_scale| of order one spreads each head's logits over tens of log2 units, so its running
    maximum keeps moving after the first tile (the rescale of O and of the row sums runs on later
    tiles too, with both signs of sm_scale), over several tiles and a ragged last one."""
    rng = np.random.default_rng(int(abs(sm_scale) * 100) + H + R)
    B, topk, n_slots = 2, 900, 1200
    q = rng.standard_normal((B, 1, H, 576)).astype(np.float32)
    idx = np.stack([rng.choice(n_slots, size=topk, replace=False) for _ in range(B)]).reshape(B, 1, topk)
    idx = idx.astype(np.int32)
    idx[rng.random(idx.shape) < 0.05] = -1
    for splits in (1, 3):
        out, lse, ref_out, ref_lse, st = run_small(q, idx, R, n_slots, 21, sm_scale, rng.standard_normal(H), splits)
        assert st == 0
        assert_close(out, lse, ref_out, ref_lse)


@pytest.mark.parametrize("R", [352, 432])
def test_more_rows_than_sms_two_parts(R):
    """64 heads, 200 query rows (between one and two per SM on a 152-SM GB300, so the grid runs in
    two waves), by the library's choice of parts and with two parts per row; every row is compared
    with the oracle."""
    rng = np.random.default_rng(200 + R)
    B, s_q, H, topk, n_slots = 100, 2, 64, 600, 2000
    q = rng.standard_normal((B, s_q, H, 576)).astype(np.float32)
    idx = np.stack([rng.choice(n_slots, size=topk, replace=False) for _ in range(B * s_q)]).reshape(B, s_q, topk)
    idx = idx.astype(np.int32)
    idx[rng.random(idx.shape) < 0.1] = -1
    sink = rng.standard_normal(H).astype(np.float32)
    for splits in (0, 2):
        out, lse, ref_out, ref_lse, st = run_small(q, idx, R, n_slots, 41, 1 / math.sqrt(576), sink, splits)
        assert st == 0
        assert_close(out, lse, ref_out, ref_lse)


def test_many_splits_reused_dirty_workspace_is_deterministic():
    """Five splits with a sink: the partials and their merge depend on nothing left in the
    workspace, so a reused workspace and one filled with junk give the same bits, and those
    match the oracle."""
    rng = np.random.default_rng(4242)
    B, H, topk, n_slots, splits, R = 3, 128, 640, 1000, 5, 352
    q = rng.standard_normal((B, 1, H, 576)).astype(np.float32)
    idx = np.stack([rng.choice(n_slots, size=topk, replace=False) for _ in range(B)]).reshape(B, 1, topk)
    idx = idx.astype(np.int32)
    idx[rng.random(idx.shape) < 0.1] = -1
    sink = rng.standard_normal(H).astype(np.float32)
    cache = fill_pool(lib.quantize_append, n_slots, R, 9, DEV)
    qd = torch.from_numpy(q).to(torch.bfloat16).to(DEV)
    idd = torch.from_numpy(idx).to(DEV)
    sink_d = torch.from_numpy(sink).to(DEV)
    ws = torch.zeros(lib.workspace_size(B, 1, H, topk, R, splits), dtype=torch.uint8, device=DEV)

    def call():
        out, lse = lib.sparse_mla_decode(qd, cache, idd, 0.05, attn_sink=sink_d, num_splits=splits, workspace=ws)
        torch.cuda.synchronize()
        return out.clone(), lse.clone()

    first = call()
    again = call()
    ws.fill_(0x7F)
    dirty = call()
    for o, l in (again, dirty):
        assert torch.equal(o, first[0]) and torch.equal(l, first[1])
    recs = oracle_pool(9, n_slots, R)
    ref_out, ref_lse = oracle.sparse_mla_decode(synth.bf16_bits(qd.cpu()), recs, idx.reshape(B, -1), 0.05,
                                                attn_sink=sink)
    assert_close(first[0], first[1], ref_out.reshape(B, 1, H, 512), ref_lse.reshape(B, 1, H))


# ---- benchmark-sized workloads, sampled rows ---------------------------------------------

def _sampled_parity(w: synth.DecodeWorkload, n_rows: int):
    cache = fill_pool(lib.quantize_append, w.num_slots, w.record_bytes, w.pool_seed, DEV)
    sink = None if w.attn_sink is None else w.attn_sink.to(DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    out, lse = lib.sparse_mla_decode(w.q.to(DEV), cache, w.indices.to(DEV), w.sm_scale, attn_sink=sink,
                                     dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    rows = synth.sample_rows(w, n_rows)
    slots, q_rows, idx = synth.compact_for_rows(w, rows)
    lat, rope = synth.pool_rows(w.pool_seed, torch.from_numpy(slots))
    recs = oracle.quantize_records(synth.bf16_bits(lat), synth.bf16_bits(rope), w.record_bytes)
    # the device pool holds exactly the oracle's records for every sampled slot
    assert np.array_equal(cache[torch.from_numpy(slots).to(DEV)].cpu().numpy(), recs)
    ref_out, ref_lse = oracle.sparse_mla_decode(synth.bf16_bits(q_rows), recs, idx, w.sm_scale,
                                                attn_sink=None if w.attn_sink is None else w.attn_sink.numpy())
    o = out.reshape(w.n_rows, w.h_q, 512)[torch.from_numpy(rows).to(DEV)]
    l = lse.reshape(w.n_rows, w.h_q)[torch.from_numpy(rows).to(DEV)]
    assert_close(o, l, ref_out, ref_lse)
    del cache
    torch.cuda.empty_cache()


def test_batch_decode_b32_h128_sampled():
    _sampled_parity(synth.batch_decode(seed=0), 8)


def test_varlen_mtp_sink_sampled():
    _sampled_parity(synth.varlen_decode(seed=0), 8)


def test_sparse_prefill_sampled():
    """Sparse prefill / extend: 2 requests x 256 new tokens, causal top-k over a 16K prefix."""
    _sampled_parity(synth.sparse_prefill(seed=0), 8)


def test_long_context_432_sampled():
    _sampled_parity(synth.long_context(seed=0), 8)


def test_a_wait_that_runs_out_reports_a_timeout_and_leaves_the_context_usable():
    """The decode's pipeline waits are bounded in time: one that nothing completes gives up after
    about a second, sets DEV_TIMEOUT and lets the kernel return; the next decode runs normally."""
    st, ns = lib.selftest_wait_timeout()
    assert st & lib.DEV_TIMEOUT
    assert 0.9e9 <= ns <= 10e9, ns
    w = synth.tiny_decode(seed=3)
    cache = fill_pool(lib.quantize_append, w.num_slots, w.record_bytes, w.pool_seed, DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    out, lse = lib.sparse_mla_decode(w.q.to(DEV), cache, w.indices.to(DEV), w.sm_scale, dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    ref_out, ref_lse = oracle.sparse_mla_decode(synth.bf16_bits(w.q), oracle_pool(w.pool_seed, w.num_slots,
                                                                                  w.record_bytes),
                                                w.indices.numpy().reshape(1, -1), w.sm_scale)
    assert_close(out, lse, ref_out, ref_lse)
