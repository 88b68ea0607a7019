"""Pins for the oracle's sparse MLA decode (read side): closed forms, special cases, a
two-key example worked by hand, invariances, and brute force against scipy's softmax on tiny
inputs.

Sources: FlashMLA PR 18 "W4A16 DSA: NVFP4 KV cache format for SM100 sparse decode" ("Kernel:"
paragraph: keys dequantized to bf16, QK over 576 and PV over the 512 NoPE dims, fp32
accumulation; the validation list: invalid indices, attention sink); the split/merge of
partial results follows the same softmax definition.
"""
import math

import numpy as np
import pytest
import scipy.special
import torch

import oracle
import synth


def bits(a) -> np.ndarray:
    return synth.bf16_bits(torch.tensor(np.asarray(a, dtype=np.float32)).to(torch.bfloat16))


def pool(seed, n, R=352):
    lat, rope = synth.pool_rows(seed, torch.arange(n))
    return oracle.quantize_records(synth.bf16_bits(lat), synth.bf16_bits(rope), R)


def rand_q(rng, n, h):
    return bits(rng.standard_normal((n, h, 576)).astype(np.float32))


def test_two_key_decode_by_hand():
    # key A: element 0 = 1.0 (nibble 0x2, scale of block 0 = e4m3 1.0 = 0x38), all else 0
    # key B: element 0 = 2.0 (nibble 0x4)
    A = np.zeros(352, dtype=np.uint8)
    B = np.zeros(352, dtype=np.uint8)
    A[0], B[0] = 0x02, 0x04
    A[320] = B[320] = 0x38                       # block 0 scale sits at byte 320 + 8*0 + 0
    cache = np.stack([A, B])
    q = np.zeros((1, 1, 576), dtype=np.float32)
    q[0, 0, 0] = 1.0
    idx = np.array([[1, -1, 0]], dtype=np.int32)
    # z_A = ln 3, z_B = 2 ln 3 -> weights 3/12 and 9/12 -> out[0] = 1/4 + 3/2 = 1.75, lse = ln 12
    out, lse = oracle.sparse_mla_decode(bits(q), cache, idx, math.log(3.0))
    assert out[0, 0, 0] == pytest.approx(1.75, abs=1e-15)
    assert np.all(out[0, 0, 1:] == 0)
    assert lse[0, 0] == pytest.approx(math.log(12.0), abs=1e-15)
    # a sink of ln 4 adds 4 to the denominator only: out[0] = (3 + 18) / 16; lse unchanged
    out_s, lse_s = oracle.sparse_mla_decode(bits(q), cache, idx, math.log(3.0), attn_sink=np.float32([math.log(4.0)]))
    assert out_s[0, 0, 0] == pytest.approx(21.0 / 16.0, rel=1e-7)   # sink passes through fp32
    assert lse_s[0, 0] == pytest.approx(math.log(12.0), abs=1e-15)


@pytest.mark.parametrize("R", [352, 432])
def test_single_index_returns_its_value_row_exactly(R):
    rng = np.random.default_rng(1)
    cache = pool(5, 64, R)
    q = rand_q(rng, 3, 4)
    idx = np.full((3, 16), -1, dtype=np.int32)
    idx[:, 7] = [3, 40, 63]
    out, lse = oracle.sparse_mla_decode(q, cache, idx, 0.05)
    k = oracle.dequant_records(cache[[3, 40, 63]])
    qf = (q.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    for t in range(3):
        for h in range(4):
            assert np.array_equal(out[t, h], k[t, :512])
            assert lse[t, h] == pytest.approx(0.05 * float(qf[t, h] @ k[t]), rel=1e-13, abs=1e-13)


def test_zero_query_gives_mean_of_used_value_rows():
    cache = pool(6, 100)
    idx = np.array([[5, -1, 17, 99, 250, 3, -7]], dtype=np.int32)   # 250 >= num_slots: unused
    q = np.zeros((1, 2, 576), dtype=np.uint16)
    out, lse = oracle.sparse_mla_decode(q, cache, idx, 0.1)
    k = oracle.dequant_records(cache[[5, 17, 99, 3]])
    for h in range(2):
        assert np.allclose(out[0, h], k[:, :512].mean(axis=0), rtol=1e-14, atol=1e-14)
        assert lse[0, h] == pytest.approx(math.log(4.0), abs=1e-14)


def test_no_used_index_gives_zero_and_minus_infinity():
    cache = pool(7, 32)
    idx = np.array([[-1] * 8, [32, 40, -1, -5, 1000, -1, -1, -1]], dtype=np.int32)
    q = rand_q(np.random.default_rng(2), 2, 3)
    for sink in (None, np.float32([0.5, -1.0, 3.0])):
        out, lse = oracle.sparse_mla_decode(q, cache, idx, 0.04, attn_sink=sink)
        assert np.all(out == 0) and np.all(np.isneginf(lse))


def test_sink_closed_form_and_minus_infinity_limit():
    rng = np.random.default_rng(3)
    cache = pool(8, 200)
    idx = rng.choice(200, size=(4, 32), replace=True).astype(np.int32)
    q = rand_q(rng, 4, 8)
    sink = rng.standard_normal(8).astype(np.float32)
    out0, lse0 = oracle.sparse_mla_decode(q, cache, idx, 1 / 24)
    out1, lse1 = oracle.sparse_mla_decode(q, cache, idx, 1 / 24, attn_sink=sink)
    outn, lsen = oracle.sparse_mla_decode(q, cache, idx, 1 / 24, attn_sink=np.full(8, -np.inf, dtype=np.float32))
    assert np.array_equal(lse1, lse0) and np.array_equal(lsen, lse0)
    assert np.array_equal(outn, out0)
    factor = 1.0 / (1.0 + np.exp(sink.astype(np.float64)[None, :] - lse0))
    assert np.allclose(out1, out0 * factor[..., None], rtol=1e-12, atol=1e-14)


def test_index_order_does_not_matter_and_duplicates_count_twice():
    rng = np.random.default_rng(4)
    cache = pool(9, 300)
    idx = rng.choice(300, size=(2, 24), replace=False).astype(np.int32)
    q = rand_q(rng, 2, 4)
    out, lse = oracle.sparse_mla_decode(q, cache, idx, 0.05)
    perm = idx[:, rng.permutation(24)]
    out_p, lse_p = oracle.sparse_mla_decode(q, cache, perm, 0.05)
    assert np.allclose(out_p, out, rtol=1e-12, atol=1e-14) and np.allclose(lse_p, lse, atol=1e-12)
    dup = np.concatenate([idx, idx], axis=1)
    out_d, lse_d = oracle.sparse_mla_decode(q, cache, dup, 0.05)
    assert np.allclose(out_d, out, rtol=1e-12, atol=1e-14)
    assert np.allclose(lse_d, lse + math.log(2.0), atol=1e-12)


def _independent_keys(records: np.ndarray, R: int) -> np.ndarray:
    """Dequantize with library fp8 decoding and an explicit grid, without the oracle."""
    grid = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6], dtype=np.float64)
    nib = np.stack([records[:, :256] & 15, records[:, :256] >> 4], axis=2).reshape(-1, 512)
    vals = grid[nib & 7] * np.where(nib & 8, -1.0, 1.0)
    if R == 352:
        sbytes = records[:, 320:352].reshape(-1, 4, 8).transpose(0, 2, 1).reshape(-1, 32)   # 4x8 -> 8x4
        rope = torch.from_numpy(np.ascontiguousarray(records[:, 256:320])).view(torch.float8_e4m3fn).double().numpy()
    else:
        sbytes = records[:, 256:288]
        rope = torch.from_numpy(np.ascontiguousarray(records[:, 304:432])).view(torch.bfloat16).double().numpy()
    s = torch.from_numpy(np.ascontiguousarray(sbytes)).view(torch.float8_e4m3fn).double().numpy()
    return np.concatenate([vals * np.repeat(s, 16, axis=1), rope], axis=1)


@pytest.mark.parametrize("R", [352, 432])
@pytest.mark.parametrize("with_sink", [False, True])
def test_brute_force_against_scipy_softmax(R, with_sink):
    rng = np.random.default_rng(10 + R + with_sink)
    n_slots, n_tok, H, K = 12, 5, 4, 8
    recs = rng.integers(0, 256, size=(n_slots, R)).astype(np.uint8)   # hand-built random records
    if R == 352:
        for lo, hi in ((256, 352),):
            seg = recs[:, lo:hi]
            seg[(seg & 0x7F) == 0x7F] = 0x00                             # no NaN codes
    else:
        seg = recs[:, 256:288]
        seg[(seg & 0x7F) == 0x7F] = 0x00
        r16 = recs[:, 304:432].view(np.uint16)
        r16[((r16 >> 7) & 0xFF) == 0xFF] &= 0xBFFF
    keys = _independent_keys(recs, R)
    assert np.array_equal(keys, oracle.dequant_records(recs))
    idx = rng.integers(-2, n_slots + 2, size=(n_tok, K)).astype(np.int32)
    q = rand_q(rng, n_tok, H)
    sink = rng.standard_normal(H).astype(np.float32) if with_sink else None
    scale = 0.01
    out, lse = oracle.sparse_mla_decode(q, recs, idx, scale, attn_sink=sink)
    qf = (q.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    for t in range(n_tok):
        used = [int(i) for i in idx[t] if 0 <= i < n_slots]
        for h in range(H):
            if not used:
                assert np.isneginf(lse[t, h]) and np.all(out[t, h] == 0)
                continue
            z = scale * (keys[used] @ qf[t, h])
            ref_lse = scipy.special.logsumexp(z)
            if with_sink:
                w = scipy.special.softmax(np.append(z, float(sink[h])))[:-1]
            else:
                w = scipy.special.softmax(z)
            ref = w @ keys[used, :512]
            assert lse[t, h] == pytest.approx(ref_lse, rel=1e-12, abs=1e-12)
            assert np.allclose(out[t, h], ref, rtol=1e-10, atol=1e-10 * np.abs(keys).max())


@pytest.mark.parametrize("with_sink", [False, True])
def test_merging_partials_over_any_partition_equals_the_whole(with_sink):
    rng = np.random.default_rng(20 + with_sink)
    cache = pool(11, 500)
    K = 64
    idx = rng.choice(500, size=(1, K), replace=False).astype(np.int32)
    idx[0, rng.choice(K, 6, replace=False)] = -1
    q = rand_q(rng, 1, 2)
    sink = np.float32([0.7, -0.3]) if with_sink else None
    whole_out, whole_lse = oracle.sparse_mla_decode(q, cache, idx, 1 / 24, attn_sink=sink)
    for parts in ([0, 64], [0, 10, 11, 40, 64], [0, 1, 2, 3, 64], [0, 32, 33, 64]):
        lse_p, out_p = [], []
        for a, b in zip(parts[:-1], parts[1:]):
            sub = np.full((1, K), -1, dtype=np.int32)
            sub[0, a:b] = idx[0, a:b]
            o, l = oracle.sparse_mla_decode(q, cache, sub, 1 / 24)
            lse_p.append(l[0])
            out_p.append(o[0])
        for h in range(2):
            o, l = oracle.merge_partials(np.array([x[h] for x in lse_p]), np.stack([x[h] for x in out_p]),
                                         None if sink is None else float(sink[h]))
            assert l == pytest.approx(whole_lse[0, h], abs=1e-12)
            assert np.allclose(o, whole_out[0, h], rtol=1e-11, atol=1e-12)


def test_merging_only_empty_partials_is_empty():
    o, l = oracle.merge_partials(np.array([-np.inf, -np.inf]), np.zeros((2, 512)), 1.0)
    assert np.isneginf(l) and np.all(o == 0)
