"""Pins for the oracle's block-order variant of the 352-byte record, the unpermuted side of the
scale-layout comparison.

FlashMLA PR 18 "W4A16 DSA: NVFP4 KV cache format for SM100 sparse decode" (format block
"nvfp4.fp8rope (352 B/token)") stores the 32 scales of a record permuted (block s at byte
320 + 8*(s&3) + (s>>2)) and credits that placement with 10-12% of decode latency. The record
it is compared with keeps every other byte and stores block s at 320 + s, the order the
432-byte record of vLLM PR 82 "kv: nvfp4_ds_mla - 4-bit NVFP4 KV cache for B12X sparse MLA
(SM120)" (Problem) uses for its own scale field. These tests tie the variant to the hand-worked
record, to the 432-byte record's scale field, and to a dequantization that does not use the
oracle.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from test_oracle_codec import _hand_expected_nope_and_scales, _hand_token, f32_to_bf16_bits
from test_oracle_decode import _independent_keys, rand_q


def test_block_order_offsets_and_the_432_record_refuses_the_flag():
    assert [oracle.scale_offset(352, s, block_scales=True) for s in range(32)] == list(range(320, 352))
    with pytest.raises(AssertionError):
        oracle.scale_offset(432, 0, block_scales=True)


def test_hand_record_352_block_scales():
    lat, rope = _hand_token()
    lb, rb = f32_to_bf16_bits(lat)[None], f32_to_bf16_bits(rope)[None]
    blk = oracle.quantize_records(lb, rb, 352, block_scales=True)[0]
    perm = oracle.quantize_records(lb, rb, 352)[0]
    nope, scales = _hand_expected_nope_and_scales()
    assert np.array_equal(blk[:256], nope)
    assert np.array_equal(blk[256:320], perm[256:320])     # RoPE field unchanged
    assert np.array_equal(blk[320:352], scales)            # block order


@pytest.fixture(scope="module")
def tokens():
    w = synth.write_path(seed=11, T=1024, num_slots=2048)
    return synth.bf16_bits(w.latent), synth.bf16_bits(w.rope)


def test_block_scales_equal_the_432_scale_field_and_the_unpermuted_352_field(tokens):
    lat, rope = tokens
    blk = oracle.quantize_records(lat, rope, 352, block_scales=True)
    perm = oracle.quantize_records(lat, rope, 352)
    r432 = oracle.quantize_records(lat, rope, 432)
    assert np.array_equal(blk[:, :320], perm[:, :320])
    assert np.array_equal(blk[:, 320:352], r432[:, 256:288])
    # the permuted field, read as an 8 x 4 matrix (row = s >> 2), is the 4 x 8 transpose
    assert np.array_equal(perm[:, 320:352].reshape(-1, 4, 8).transpose(0, 2, 1).reshape(-1, 32), blk[:, 320:352])


def test_dequant_of_either_layout_gives_the_same_keys(tokens):
    lat, rope = tokens
    blk = oracle.quantize_records(lat, rope, 352, block_scales=True)
    perm = oracle.quantize_records(lat, rope, 352)
    k_blk = oracle.dequant_records(blk, block_scales=True)
    assert np.array_equal(k_blk, oracle.dequant_records(perm))
    assert np.array_equal(k_blk, _independent_keys(perm, 352))
    # read with the wrong layout, the scales land on the wrong blocks
    assert not np.array_equal(oracle.dequant_records(blk), k_blk)


def test_append_and_decode_agree_across_layouts():
    rng = np.random.default_rng(21)
    T, N, n_tok, H, K = 96, 128, 6, 8, 40
    lat, rope = synth.pool_rows(3, torch.arange(T))
    lb, rb = synth.bf16_bits(lat), synth.bf16_bits(rope)
    slots = rng.permutation(N)[:T].astype(np.int64)
    c_perm = np.full((N, 352), 0xAB, dtype=np.uint8)
    c_blk = c_perm.copy()
    assert oracle.quantize_append(lb, rb, slots, c_perm) == 0
    assert oracle.quantize_append(lb, rb, slots, c_blk, block_scales=True) == 0
    untouched = np.setdiff1d(np.arange(N), slots)
    assert np.all(c_blk[untouched] == 0xAB)
    assert np.array_equal(c_blk[slots, :320], c_perm[slots, :320])
    idx = slots[rng.integers(0, T, size=(n_tok, K))].astype(np.int32)
    idx[0, ::5] = -1
    q = rand_q(rng, n_tok, H)
    o_p, l_p = oracle.sparse_mla_decode(q, c_perm, idx, 0.04)
    o_b, l_b = oracle.sparse_mla_decode(q, c_blk, idx, 0.04, block_scales=True)
    assert np.array_equal(o_p, o_b) and np.array_equal(l_p, l_b)
