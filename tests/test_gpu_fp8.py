"""The 656-byte fp8 record (vLLM PR 82 "kv: nvfp4_ds_mla - 4-bit NVFP4 KV cache for B12X sparse
MLA (SM120)", Problem section: 512 B fp8 NoPE + 16 B fp32 tile scales + 128 B BF16 RoPE) on the
GPU: the append kernel is bit-exact against the oracle, and the decode over such records
matches the oracle within the decode tolerances (|out - ref| <= 1e-2 + 1e-2 |ref|, lse within
1e-3), on small problems compared in full and on the B=32 / h_q=128 / top-k 2048 batch decode
compared on sampled rows."""
import dataclasses
import math

import numpy as np
import pytest
import torch

import nvfp4_kv_cache_sparse_gb300 as lib
import oracle
import synth
from test_gpu_decode import DEV, _sampled_parity, assert_close, run_small
from test_gpu_quantize import finite_bf16_bits

pytestmark = pytest.mark.gpu


def gpu_append(lat: np.ndarray, rope: np.ndarray, slots: np.ndarray, num_slots: int):
    cache = torch.full((num_slots, 656), 0xAB, dtype=torch.uint8, device=DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    lib.quantize_append(torch.from_numpy(lat.view(np.int16)).view(torch.bfloat16).to(DEV),
                        torch.from_numpy(rope.view(np.int16)).view(torch.bfloat16).to(DEV),
                        torch.from_numpy(slots).to(DEV), cache, dev_status=status)
    torch.cuda.synchronize()
    return cache.cpu().numpy(), int(status.item())


def check_append(lat: np.ndarray, rope: np.ndarray, num_slots: int):
    T = lat.shape[0]
    slots = np.random.default_rng(T).permutation(num_slots)[:T].astype(np.int64)
    got, st = gpu_append(lat, rope, slots, num_slots)
    exp = np.full((num_slots, 656), 0xAB, dtype=np.uint8)
    assert oracle.quantize_append(lat, rope, slots, exp) == 0
    mism = np.argwhere(got != exp)
    assert mism.size == 0, f"{len(mism)} bytes differ, first at {mism[:5].tolist()}"
    x = (lat.astype(np.uint32) << 16).view(np.float32).reshape(T, 4, 128)
    big = bool((np.abs(x).max(axis=2) >= 65536).any())
    assert st == (lib.DEV_FP8_RANGE if big else 0)


def test_append_every_finite_bf16_value_bit_exact():
    vals = finite_bf16_bits()
    vals = vals[np.random.default_rng(1).permutation(vals.size)]
    T = (vals.size + 511) // 512
    lat = np.zeros(T * 512, dtype=np.uint16)
    lat[:vals.size] = vals
    check_append(lat.reshape(T, 512), np.resize(vals, T * 64).reshape(T, 64), T + 5)


def test_append_small_ranges_and_zero_tiles_bit_exact():
    """Tiles whose maxima span the bf16 range below 65536: subnormal fp32 scales, exact powers
    of two, all-zero tiles with signed zeros, and values far below their tile's maximum."""
    rng = np.random.default_rng(2)
    T = 512
    x = rng.standard_normal((T, 4, 128)).astype(np.float32)
    x *= np.float32(2.0) ** rng.integers(-133, 14, size=(T, 4, 1)).astype(np.float32)
    x[::7, 1] = 0.0
    x[::7, 1, ::3] = -0.0
    x[3::11, 2] *= np.float32(2.0) ** rng.integers(-30, 0, size=(x[3::11, 2].shape)).astype(np.float32)
    lat = synth.bf16_bits(torch.from_numpy(x.reshape(T, 512)).to(torch.bfloat16))
    rope = synth.bf16_bits(torch.from_numpy(rng.standard_normal((T, 64)).astype(np.float32)).to(torch.bfloat16))
    check_append(lat, rope, 2 * T)


FP8_CASES = [
    # (B, s_q, H, topk, sink, splits)
    (1, 1, 128, 64, False, 1),
    (2, 1, 128, 96, True, 2),
    (3, 2, 64, 50, True, 0),
    (2, 2, 64, 200, False, 4),
    (1, 1, 128, 2048, True, 5),
]


@pytest.mark.parametrize("B,s_q,H,topk,sink,splits", FP8_CASES)
def test_small_problems(B, s_q, H, topk, sink, splits):
    rng = np.random.default_rng(B * 1000 + topk + splits + 656)
    n_slots = max(300, topk + 10)
    q = rng.standard_normal((B, s_q, H, 576)).astype(np.float32)
    idx = np.stack([rng.choice(n_slots, size=topk, replace=topk > n_slots) for _ in range(B * s_q)])
    idx = idx.reshape(B, s_q, topk).astype(np.int32)
    idx[rng.random(idx.shape) < 0.15] = -1
    if B > 1:
        idx[1, 0] = -1                                  # an empty row
    sk = rng.standard_normal(H).astype(np.float32) if sink else None
    out, lse, ref_out, ref_lse, st = run_small(q, idx, 656, n_slots, 17 + topk, 1 / math.sqrt(576), sk, splits)
    assert st == 0
    assert_close(out, lse, ref_out, ref_lse)


def test_batch_decode_b32_h128_656_sampled():
    w = synth.batch_decode(seed=0)
    w = dataclasses.replace(w, name="decode_b32_sq1_h128_topk2048_R656", record_bytes=656)
    _sampled_parity(w, 8)
