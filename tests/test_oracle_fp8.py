"""Pins for the oracle's 656-byte fp8 record (the V3.2 "fp8_ds_mla" record the NVFP4 records are
measured against) and for the decode over it.

Source: vLLM PR 82 "kv: nvfp4_ds_mla - 4-bit NVFP4 KV cache for B12X sparse MLA (SM120)",
Problem section (656 B = 512 B fp8 NoPE + 16 B fp32 tile scales + 128 B BF16 RoPE); FlashMLA
PR 18 "W4A16 DSA: NVFP4 KV cache format for SM100 sparse decode" (dispatch list: 656 = V32
fp8 for d_qk 576 / d_v 512; keys dequantized to bf16). The pages give no fp8 scale rule; the
oracle reads it as scale = amax / 448 per 128-value tile, code = e4m3(x / scale), key =
bf16(e4m3(code) * scale). These tests check that reading against library conversions (numpy
fp32 division, torch float8_e4m3fn and bfloat16 casts), a record worked by hand, and brute
force.
"""
import json
import os

import numpy as np
import pytest
import scipy.special
import torch

import oracle
import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def bits(a) -> np.ndarray:
    return synth.bf16_bits(torch.tensor(np.asarray(a, dtype=np.float32)).to(torch.bfloat16))


def torch_e4m3(values: np.ndarray) -> np.ndarray:
    return torch.from_numpy(np.ascontiguousarray(values, dtype=np.float32)).to(torch.float8_e4m3fn) \
        .view(torch.uint8).numpy()


def e4m3_value(codes: np.ndarray) -> np.ndarray:
    return torch.from_numpy(np.ascontiguousarray(codes, dtype=np.uint8)).view(torch.float8_e4m3fn).double().numpy()


def round_bf16_numpy(x: np.ndarray) -> np.ndarray:
    """bf16 round-to-nearest-even of doubles by frexp and numpy's half-to-even rounding."""
    x = np.asarray(x, dtype=np.float64)
    _, e = np.frexp(x)
    lsb = np.maximum(e - 8, -133)
    return np.ldexp(np.round(np.ldexp(x, -lsb)), lsb)


def independent_keys(recs: np.ndarray) -> np.ndarray:
    codes = recs[:, :512]
    scales = np.ascontiguousarray(recs[:, 512:528]).view("<f4").astype(np.float64)   # [n, 4]
    nope = round_bf16_numpy(e4m3_value(codes) * np.repeat(scales, 128, axis=1))
    rope = torch.from_numpy(np.ascontiguousarray(recs[:, 528:656])).view(torch.bfloat16).double().numpy()
    return np.concatenate([nope, rope], axis=1)


def test_layout_arithmetic_matches_the_page():
    lay = json.load(open(os.path.join(GOLDEN, "layout.json")))["fp8_ds_mla"]
    assert sum(f["bytes"] for f in lay["fields"]) == lay["record_bytes"] == 656
    assert lay["fields"][0]["bytes"] == lay["d_v"]                 # one byte per NoPE value
    assert lay["fields"][1]["bytes"] // 4 == lay["d_v"] // 128      # one fp32 scale per 128 values
    assert lay["fields"][2]["bytes"] == 2 * (lay["d_qk"] - lay["d_v"])


def test_round_to_bf16_matches_torch_on_float32_inputs():
    rng = np.random.default_rng(3)
    f = np.concatenate([rng.standard_normal(20000).astype(np.float32) * np.float32(1e3),
                        (rng.integers(0, 1 << 31, size=20000, dtype=np.uint32) & 0x7F7FFFFF).view(np.float32),
                        np.array([1 + 2.0 ** -8, 1 + 3 * 2.0 ** -8, 2.0 ** -134, 3 * 2.0 ** -134, 2.0 ** -126,
                                  -(1 + 2.0 ** -8)], dtype=np.float32)])
    expect = torch.from_numpy(f).to(torch.bfloat16).double().numpy()
    got = np.array([oracle.round_to_bf16(float(v)) for v in f])
    assert np.array_equal(got, expect)


def _hand_token():
    lat = np.zeros(512, dtype=np.float32)
    # tile 0: amax 448 -> scale 1.0; codes by RNE, ties to the even code
    lat[0:12] = [448, -448, 1, 0.5, 17, 19, -240, 2.0 ** -9, 2.0 ** -10, 3 * 2.0 ** -10, 0.0, -0.0]
    # tile 1: all zero with one -0 -> scale 0, codes carry only signs
    lat[130] = -0.0
    # tile 2: amax 7 -> scale 7/448 = 2^-6 exactly; bf16(0.1) = 0.10009765625 -> x/s = 6.40625 -> 6.5
    lat[256:259] = [7, -3.5, 0.1]
    # tile 3: amax 1 -> scale fl32(1/448); 1/s and 0.5/s round to 448 and 224
    lat[384:386] = [1.0, -0.5]
    rope = np.linspace(-3, 3, 64).astype(np.float32)
    return lat, rope


def test_hand_record_656():
    lat, rope = _hand_token()
    rope_bits = bits(rope)
    rec = oracle.quantize_records(bits(lat)[None], rope_bits[None], 656)[0]
    codes = np.zeros(512, dtype=np.uint8)
    codes[0:12] = [0x7E, 0xFE, 0x38, 0x30, 0x58, 0x5A, 0xF7, 0x01, 0x00, 0x02, 0x00, 0x80]
    codes[130] = 0x80
    codes[256:259] = [0x7E, 0xF6, 0x4D]
    codes[384:386] = [0x7E, 0xF6]
    assert np.array_equal(rec[:512], codes)
    scales = rec[512:528].view("<f4")
    assert scales[0] == 1.0 and scales[1] == 0.0 and not np.signbit(scales[1]) and scales[2] == 2.0 ** -6
    assert scales[3] == np.float32(1.0) / np.float32(448.0)
    assert list(rec[512:516]) == [0x00, 0x00, 0x80, 0x3F] and list(rec[520:524]) == [0x00, 0x00, 0x80, 0x3C]
    assert np.array_equal(rec[528:656].view(np.uint16), rope_bits)   # little-endian bf16 copy
    k = oracle.dequant_records(rec[None])[0]
    assert list(k[0:12]) == [448, -448, 1, 0.5, 16, 20, -240, 2.0 ** -9, 0, 2.0 ** -8, 0, 0]
    assert list(k[256:259]) == [7, -3.5, 0.1015625] and list(k[384:386]) == [1.0, -0.5]


@pytest.fixture(scope="module")
def tokens():
    w = synth.write_path(seed=13, T=1024, num_slots=2048)
    return synth.bf16_bits(w.latent), synth.bf16_bits(w.rope)


def test_scale_is_fp32_amax_over_448_and_codes_are_e4m3_of_the_fp32_quotient(tokens):
    lat, rope = tokens
    recs = oracle.quantize_records(lat, rope, 656)
    x = (lat.astype(np.uint32) << 16).view(np.float32).reshape(-1, 4, 128)
    amax = np.abs(x).max(axis=2)
    s = np.ascontiguousarray(recs[:, 512:528]).view("<f4")
    assert np.array_equal(s, amax / np.float32(448.0))
    q = np.where(s[:, :, None] != 0, x / np.where(s == 0, np.float32(1), s)[:, :, None], np.float32(0))
    expect = torch_e4m3(q.astype(np.float32)).reshape(-1, 512)
    assert np.array_equal(recs[:, :512], expect)
    assert np.array_equal(np.ascontiguousarray(recs[:, 528:]).view(np.uint16), rope)


def test_error_within_half_an_e4m3_step_of_the_scaled_value(tokens):
    lat, rope = tokens
    recs = oracle.quantize_records(lat, rope, 656)
    x = (lat.astype(np.uint32) << 16).view(np.float32).astype(np.float64).reshape(-1, 4, 128)
    s = np.ascontiguousarray(recs[:, 512:528]).view("<f4").astype(np.float64)[:, :, None]
    xhat = e4m3_value(recs[:, :512]).reshape(-1, 4, 128) * s
    r = np.abs(x) / s
    step = np.where(r >= 2.0 ** -6, 2.0 ** (np.floor(np.log2(np.maximum(r, 2.0 ** -6))) - 3), 2.0 ** -9)
    assert np.all(np.abs(x - xhat) <= step / 2 * s * (1 + 2.0 ** -20))


def test_dequant_matches_an_independent_dequantizer(tokens):
    lat, rope = tokens
    recs = oracle.quantize_records(lat, rope, 656)
    assert np.array_equal(oracle.dequant_records(recs), independent_keys(recs))


@pytest.mark.parametrize("with_sink", [False, True])
def test_decode_brute_force_against_scipy_softmax(with_sink):
    rng = np.random.default_rng(40 + with_sink)
    n_slots, n_tok, H, K = 16, 5, 4, 9
    lat, rope = synth.pool_rows(8, torch.arange(n_slots))
    recs = oracle.quantize_records(synth.bf16_bits(lat), synth.bf16_bits(rope), 656)
    keys = independent_keys(recs)
    idx = rng.integers(-2, n_slots + 2, size=(n_tok, K)).astype(np.int32)
    q = bits(rng.standard_normal((n_tok, H, 576)).astype(np.float32))
    sink = rng.standard_normal(H).astype(np.float32) if with_sink else None
    scale = 0.03
    out, lse = oracle.sparse_mla_decode(q, recs, idx, scale, attn_sink=sink)
    qf = (q.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    for t in range(n_tok):
        used = [int(i) for i in idx[t] if 0 <= i < n_slots]
        for h in range(H):
            if not used:
                assert np.isneginf(lse[t, h]) and np.all(out[t, h] == 0)
                continue
            z = scale * (keys[used] @ qf[t, h])
            w = scipy.special.softmax(np.append(z, float(sink[h])))[:-1] if with_sink else scipy.special.softmax(z)
            assert lse[t, h] == pytest.approx(scipy.special.logsumexp(z), rel=1e-12, abs=1e-12)
            assert np.allclose(out[t, h], w @ keys[used, :512], rtol=1e-10, atol=1e-10 * np.abs(keys).max())


def test_e4m3_encode_of_arbitrary_fp32_quotients_matches_torch():
    # the fp8 record encodes fp32 quotients with up to 24 significant bits (not only bf16 values):
    # random magnitudes over the whole e4m3 range, exact ties between neighbouring codes, and
    # values one fp32 ulp either side of those ties
    rng = np.random.default_rng(17)
    mag = np.ldexp(rng.uniform(1.0, 2.0, 200_000), rng.integers(-12, 9, 200_000)).astype(np.float32)
    mag = mag[mag <= 448.0]
    codes = np.arange(0x00, 0x7E, dtype=np.uint8)
    lo, hi = e4m3_value(codes), e4m3_value(codes + 1)
    ties = ((lo + hi) / 2).astype(np.float32)
    near = np.concatenate([ties, np.nextafter(ties, np.float32(0)), np.nextafter(ties, np.float32(1e9))])
    x = np.concatenate([mag, near])
    x = np.concatenate([x, -x]).astype(np.float32)
    assert np.array_equal(oracle.e4m3_encode(x), torch_e4m3(x))
