"""The 352-byte record with its scales in block order (the unpermuted side of the scale-layout
comparison in the FlashMLA PR 18 format block) on the GPU: the quantizer is bit-exact against
the oracle, the decode matches the oracle within the decode tolerances, and on the same pool
contents the decode returns exactly what it returns for the permuted record (the two kernels
differ only in where they load the scales from)."""
import functools
import math

import numpy as np
import pytest
import torch

import nvfp4_kv_cache_sparse_gb300 as lib
import oracle
import synth
from synth.pool import fill_pool
from test_gpu_decode import DEV, assert_close
from test_gpu_quantize import finite_bf16_bits

pytestmark = pytest.mark.gpu
append_blk = functools.partial(lib.quantize_append, block_scales=True)


def test_every_finite_bf16_value_bit_exact():
    vals = finite_bf16_bits()
    vals = vals[np.random.default_rng(4).permutation(vals.size)]
    T = (vals.size + 511) // 512
    lat = np.zeros(T * 512, dtype=np.uint16)
    lat[:vals.size] = vals
    lat = lat.reshape(T, 512)
    rope = np.resize(vals, T * 64).reshape(T, 64)
    slots = np.arange(T, dtype=np.int64)[::-1].copy()
    lat_d = torch.from_numpy(lat.view(np.int16)).view(torch.bfloat16).to(DEV)
    rope_d = torch.from_numpy(rope.view(np.int16)).view(torch.bfloat16).to(DEV)
    slots_d = torch.from_numpy(slots).to(DEV)
    blk = torch.full((T + 3, 352), 0xAB, dtype=torch.uint8, device=DEV)
    perm = blk.clone()
    append_blk(lat_d, rope_d, slots_d, blk)
    lib.quantize_append(lat_d, rope_d, slots_d, perm)
    torch.cuda.synchronize()
    exp = np.full((T + 3, 352), 0xAB, dtype=np.uint8)
    assert oracle.quantize_append(lat, rope, slots, exp, block_scales=True) == 0
    got = blk.cpu().numpy()
    mism = np.argwhere(got != exp)
    assert mism.size == 0, f"{len(mism)} bytes differ, first at {mism[:5].tolist()}"
    p = perm.cpu().numpy()
    assert np.array_equal(got[:, :320], p[:, :320])


@pytest.mark.parametrize("B,s_q,H,topk,sink,splits", [
    (1, 1, 128, 64, False, 1),
    (2, 2, 64, 150, True, 0),
    (3, 1, 128, 700, True, 3),
])
def test_small_problems_against_the_oracle(B, s_q, H, topk, sink, splits):
    rng = np.random.default_rng(77 + topk)
    n_slots = max(300, topk + 10)
    q = torch.from_numpy(rng.standard_normal((B, s_q, H, 576)).astype(np.float32)).to(torch.bfloat16)
    idx = np.stack([rng.choice(n_slots, size=topk, replace=False) for _ in range(B * s_q)])
    idx = idx.reshape(B, s_q, topk).astype(np.int32)
    idx[rng.random(idx.shape) < 0.15] = -1
    sk = rng.standard_normal(H).astype(np.float32) if sink else None
    cache = fill_pool(append_blk, n_slots, 352, 5 + topk, DEV)
    lat, rope = synth.pool_rows(5 + topk, torch.arange(n_slots))
    recs = oracle.quantize_records(synth.bf16_bits(lat), synth.bf16_bits(rope), 352, block_scales=True)
    assert np.array_equal(cache.cpu().numpy(), recs)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    out, lse = lib.sparse_mla_decode(q.to(DEV), cache, torch.from_numpy(idx).to(DEV), 1 / math.sqrt(576),
                                     attn_sink=None if sk is None else torch.from_numpy(sk).to(DEV),
                                     num_splits=splits, dev_status=status, block_scales=True)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    ref_out, ref_lse = oracle.sparse_mla_decode(synth.bf16_bits(q), recs, idx.reshape(B * s_q, -1),
                                                1 / math.sqrt(576), attn_sink=sk, block_scales=True)
    assert_close(out, lse, ref_out.reshape(B, s_q, H, 512), ref_lse.reshape(B, s_q, H))


def test_batch_decode_b32_h128_identical_to_the_permuted_record():
    """Full-size batch decode (B=32, h_q=128, top-k 2048, 2M-slot pool), launched as the
    benchmark launches it: the block-order pool gives bit-identical out and lse."""
    w = synth.batch_decode(seed=0)
    q, idx = w.q.to(DEV), w.indices.to(DEV)
    perm = fill_pool(lib.quantize_append, w.num_slots, 352, w.pool_seed, DEV)
    o_p, l_p = lib.sparse_mla_decode(q, perm, idx, w.sm_scale)
    torch.cuda.synchronize()
    o_p, l_p = o_p.clone(), l_p.clone()
    del perm
    blk = fill_pool(append_blk, w.num_slots, 352, w.pool_seed, DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    o_b, l_b = lib.sparse_mla_decode(q, blk, idx, w.sm_scale, dev_status=status, block_scales=True)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert torch.equal(o_b, o_p) and torch.equal(l_b, l_p)
    del blk
    torch.cuda.empty_cache()
