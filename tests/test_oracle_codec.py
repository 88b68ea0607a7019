"""Pins for the oracle's record codec (write side), checked against what the pages fix and
against library conversions the oracle does not use.

Sources: FlashMLA PR 18 "W4A16 DSA: NVFP4 KV cache format for SM100 sparse decode" (format
block "nvfp4.fp8rope (352 B/token)", the scale permutation, the unscaled-RoPE paragraph);
vLLM PR 82 "kv: nvfp4_ds_mla - 4-bit NVFP4 KV cache for B12X sparse MLA (SM120)" (Problem:
432-B field list; Fix / Write side; Tests: scale = E4M3(group_amax/6), error bound by the
E2M1 grid half-gap, zero pad, verbatim RoPE, untouched slots).
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def f32_to_bf16_bits(values) -> np.ndarray:
    t = torch.tensor(np.asarray(values, dtype=np.float32)).to(torch.bfloat16)
    return synth.bf16_bits(t)


def torch_e4m3(values: np.ndarray) -> np.ndarray:
    """Library e4m3fn conversion (round-to-nearest-even; NaN beyond the overflow threshold)."""
    return torch.from_numpy(np.ascontiguousarray(values, dtype=np.float32)).to(torch.float8_e4m3fn) \
        .view(torch.uint8).numpy()


def all_finite_bf16() -> np.ndarray:
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    f = (bits.astype(np.uint32) << 16).view(np.float32)
    return f[np.isfinite(f)]


# ---- layout arithmetic the pages print ------------------------------------------------

def test_layout_arithmetic_matches_pages():
    lay = json.load(open(os.path.join(GOLDEN, "layout.json")))
    r352 = lay["nvfp4.fp8rope"]
    fields = r352["fields"]
    assert [f["begin"] for f in fields] == [0, 256, 320] and fields[-1]["end"] == r352["record_bytes"] == 352
    assert fields[0]["count"] // fields[0]["per_byte"] == 256
    assert fields[2]["count"] * fields[2]["block"] == 512
    assert round(352 * 8 / 576, 2) == r352["effective_bits_per_value"]
    assert round(r352["capacity_vs_fp8_record"]["fp8_record_bytes"] / 352, 1) == r352["capacity_vs_fp8_record"]["ratio"]
    r432 = lay["nvfp4_ds_mla"]
    assert sum(f["bytes"] for f in r432["fields"]) == r432["record_bytes"] == 432


def test_scale_permutation_is_the_stated_transpose():
    # "the scale for element block s lives at byte 8*(s & 3) + (s >> 2), an 8x4 -> 4x8
    # transpose ... blocks {4c+q : c=0..7} for fixed q ... one contiguous 8-byte load"
    pos = [oracle.scale_offset(352, s) - 320 for s in range(32)]
    assert sorted(pos) == list(range(32))
    for q in range(4):
        run = [oracle.scale_offset(352, 4 * c + q) - 320 for c in range(8)]
        assert run == list(range(8 * q, 8 * q + 8))
    # viewed as an 8x4 matrix (row = s >> 2, col = s & 3) the bytes are its 4x8 transpose
    m = np.arange(32).reshape(8, 4)
    assert [pos[s] for s in m.T.reshape(-1)] == list(range(32))
    # the 432-B record keeps element order
    assert [oracle.scale_offset(432, s) for s in range(32)] == list(range(256, 288))


# ---- e4m3 / e2m1 primitives ------------------------------------------------------------

def test_e4m3_decode_matches_library_on_all_codes():
    codes = np.arange(256, dtype=np.uint8)
    ours = oracle.e4m3_decode(codes)
    lib = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    nan = np.isnan(lib)
    assert np.array_equal(np.isnan(ours), nan) and set(np.flatnonzero(nan)) == {0x7F, 0xFF}
    assert np.array_equal(ours[~nan], lib[~nan])
    assert ours[0x7E] == 448.0 and ours[0x01] == 2.0 ** -9 and ours[0x08] == 2.0 ** -6 and ours[0x38] == 1.0


def test_e4m3_decode_matches_fp16_bit_placement():
    # FreeToken PR 408 "feat(kvcache): add nvfp4 kv quantization": (v + (v & 0x80)) << 7 read
    # as fp16 bits is the e4m3 value divided by 2^8 -- an independent decoder.
    codes = np.arange(256, dtype=np.uint32)
    bits = (((codes + (codes & 0x80)) << 7) & 0xFFFF).astype(np.uint16)
    alt = bits.view(np.float16).astype(np.float64) * 256.0
    ours = oracle.e4m3_decode(codes.astype(np.uint8))
    ok = ~np.isnan(ours)
    assert np.array_equal(alt[ok], ours[ok])


def test_e4m3_encode_matches_library_rne_on_every_bf16_input():
    f = all_finite_bf16()
    inside = np.abs(f) <= 464.0            # beyond 464 the library gives NaN; the oracle saturates
    ours = oracle.e4m3_encode(f[inside])
    lib = torch_e4m3(f[inside])
    assert np.array_equal(ours, lib)
    sat = oracle.e4m3_encode(f[~inside])
    assert np.all((sat & 0x7F) == 0x7E) and np.array_equal(sat >> 7, np.signbit(f[~inside]).astype(np.uint8))


def test_e4m3_encode_hand_cases():
    cases = [(1.0, 0x38), (-1.0, 0xB8), (448.0, 0x7E), (500.0, 0x7E), (-1000.0, 0xFE), (0.0, 0x00),
             (-0.0, 0x80), (2.0 ** -9, 0x01), (2.0 ** -10, 0x00), (3 * 2.0 ** -11, 0x01), (1.0625, 0x38),
             (1.1875, 0x3A), (240.0, 0x77), (232.0, 0x76), (464.0, 0x7E), (-(2.0 ** -12), 0x80)]
    for x, code in cases:
        assert oracle.e4m3_encode(np.float32(x)) == code, (x, hex(code))


E2M1_GRID = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]


def test_e2m1_encode_ties_saturation_and_sign():
    # round-to-nearest-even onto the e2m1 grid: a tie goes to the even code
    cases = {0.0: 0, 0.25: 0, 0.5: 1, 0.75: 2, 1.0: 2, 1.25: 2, 1.5: 3, 1.75: 4, 2.0: 4, 2.5: 4,
             3.0: 5, 3.5: 6, 4.0: 6, 5.0: 6, 6.0: 7, 6.5: 7, 1e30: 7, 0.2499: 0, 0.2501: 1,
             4.999: 6, 5.001: 7}
    for x, code in cases.items():
        assert oracle.e2m1_encode(np.float32(x)) == code, x
        assert oracle.e2m1_encode(np.float32(-x)) == code | 8, -x
    assert oracle.e2m1_encode(np.float32(-0.0)) == 8
    for c in range(16):
        assert oracle.e2m1_decode(c) == (-1 if c & 8 else 1) * E2M1_GRID[c & 7]


def test_e2m1_encode_matches_threshold_form_on_a_dense_sweep():
    # Closed form of the same rounding written as interval bounds (open at odd-code ties).
    x = np.concatenate([np.linspace(0, 8, 400_001, dtype=np.float32), np.float32([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0])])
    code = ((x > 0.25).astype(int) + (x >= 0.75) + (x > 1.25) + (x >= 1.75) + (x > 2.5) + (x >= 3.5) + (x > 5.0))
    assert np.array_equal(oracle.e2m1_encode(x), code.astype(np.uint8))


# ---- one record worked out by hand -----------------------------------------------------

def _hand_token():
    """A token chosen so every byte of its record can be derived by hand (see comments)."""
    lat = np.zeros(512, dtype=np.float32)
    # group 0: amax 6 -> amax/6 = 1 -> scale 0x38 (s = 1); codes by RNE with ties to even
    lat[0:16] = [6, -3, 1.5, 0.75, 0.25, -0.25, 5, -5, 2.5, 3.5, 1.75, 1.25, 0.5, -0.0, 0.0, 4]
    # group 1: all zero (one -0) -> scale 0x00, nibbles carry only signs
    lat[16 + 3] = -0.0
    # group 2: amax 3 -> 0.5 -> scale 0x30; x/s = 6, 2, -4, 1
    lat[32:36] = [3, 1, -2, 0.5]
    # group 3: amax 6.375 -> 1.0625, a tie between e4m3 1.0 and 1.125 -> even -> 0x38;
    # 6.375/1 and 5.5/1 round to 6 (6.375 saturates)
    lat[48:51] = [6.375, -6.375, 5.5]
    # group 4: amax 6.75 -> 1.125 -> 0x39; quotients 6, 1.5, 0.75 (a tie -> 1.0)
    lat[64:67] = [6.75, 1.6875, 0.84375]
    # group 5: amax 6*2^-9 -> 2^-9 -> subnormal scale 0x01; quotients 6, 1, -3
    lat[80:83] = [6 * 2.0 ** -9, 2.0 ** -9, -3 * 2.0 ** -9]
    # group 6: amax 6*2^-10 -> 2^-10, a tie between 0 and 2^-9 -> 0x00; signs only
    lat[96:98] = [6 * 2.0 ** -10, -(2.0 ** -10)]
    # group 7: amax 3072 -> 512 saturates to 448 (0x7E); quotients 6.86 (-> 6), 0.5, -3
    lat[112:115] = [3072, 224, -1344]
    # groups 8..31: a single 6*2^(g-20) at the group start -> distinct scales
    for g in range(8, 32):
        lat[16 * g] = 6 * 2.0 ** (g - 20)
    rope = np.zeros(64, dtype=np.float32)
    rope[:16] = [1.0, -1.0, 448, 500, -1000, 0.0, -0.0, 2.0 ** -9, 2.0 ** -10, 3 * 2.0 ** -11,
                 1.0625, 1.1875, 240, 232, 464, -(2.0 ** -12)]
    return lat, rope


def _hand_expected_nope_and_scales():
    nope = np.zeros(256, dtype=np.uint8)
    scales = np.zeros(32, dtype=np.uint8)
    # nibble pairs (low = even element, high = odd element)
    nope[0:8] = [0xD7, 0x23, 0x80, 0xE6, 0x64, 0x24, 0x81, 0x60]
    nope[8:16] = [0x00, 0x80, 0, 0, 0, 0, 0, 0]
    nope[16:18] = [0x47, 0x2E]
    nope[24:26] = [0xF7, 0x07]
    nope[32:34] = [0x37, 0x02]
    nope[40:42] = [0x27, 0x0D]
    nope[48] = 0x80
    nope[56:58] = [0x17, 0x0D]
    scales[0:8] = [0x38, 0x00, 0x30, 0x38, 0x39, 0x01, 0x00, 0x7E]
    for g in range(8, 32):
        e = g - 20
        if e <= -10:
            s = 0x00                       # amax/6 <= 2^-10 rounds to zero
        elif e <= -7:
            s = {-9: 0x01, -8: 0x02, -7: 0x04}[e]   # e4m3 subnormals m * 2^-9
        elif e <= 8:
            s = (e + 7) << 3               # exact powers of two
        else:
            s = 0x7E                       # saturated at 448
        scales[g] = s
        nope[8 * g] = 0x00 if s == 0 else 0x07
    return nope, scales


def test_hand_record_352():
    lat, rope = _hand_token()
    rec = oracle.quantize_records(f32_to_bf16_bits(lat)[None], f32_to_bf16_bits(rope)[None], 352)[0]
    nope, scales = _hand_expected_nope_and_scales()
    assert np.array_equal(rec[:256], nope)
    exp_rope = np.zeros(64, dtype=np.uint8)
    exp_rope[:16] = [0x38, 0xB8, 0x7E, 0x7E, 0xFE, 0x00, 0x80, 0x01, 0x00, 0x01, 0x38, 0x3A, 0x77, 0x76, 0x7E, 0x80]
    assert np.array_equal(rec[256:320], exp_rope)
    # permuted placement: byte 8q + c holds block 4c + q
    for q in range(4):
        for c in range(8):
            assert rec[320 + 8 * q + c] == scales[4 * c + q]


def test_hand_record_432():
    lat, rope = _hand_token()
    rope_bits = f32_to_bf16_bits(rope)
    rec = oracle.quantize_records(f32_to_bf16_bits(lat)[None], rope_bits[None], 432)[0]
    nope, scales = _hand_expected_nope_and_scales()
    assert np.array_equal(rec[:256], nope)
    assert np.array_equal(rec[256:288], scales)
    assert np.all(rec[288:304] == 0)
    assert np.array_equal(rec[304:432].view(np.uint16), rope_bits)   # little-endian bf16 copy


# ---- properties the Tests section of vLLM PR 82 states, on random data --------------------

@pytest.fixture(scope="module")
def random_tokens():
    w = synth.write_path(seed=7, T=2048, num_slots=4096)
    return synth.bf16_bits(w.latent), synth.bf16_bits(w.rope)


@pytest.mark.parametrize("R", [352, 432])
def test_stored_scale_is_e4m3_of_amax_over_6(random_tokens, R):
    lat, rope = random_tokens
    recs = oracle.quantize_records(lat, rope, R)
    x = (lat.astype(np.uint32) << 16).view(np.float32).reshape(-1, 32, 16)
    amax = np.abs(x).max(axis=2)
    expect = torch_e4m3((amax / np.float32(6.0)).astype(np.float32))
    got = np.stack([recs[:, oracle.scale_offset(R, g)] for g in range(32)], axis=1)
    assert np.array_equal(got, expect)
    # "within half a mantissa step" of amax/6 (normal range)
    s = oracle.e4m3_decode(got)
    t = amax.astype(np.float64) / 6.0
    normal = t >= 2.0 ** -6
    step = 2.0 ** (np.floor(np.log2(t[normal])) - 3)
    assert np.all(np.abs(s[normal] - t[normal]) <= step / 2)


@pytest.mark.parametrize("R", [352, 432])
def test_nope_error_within_grid_half_gap(random_tokens, R):
    lat, rope = random_tokens
    recs = oracle.quantize_records(lat, rope, R)
    k = oracle.dequant_records(recs)
    x = (lat.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    s = np.stack([oracle.e4m3_decode(recs[:, oracle.scale_offset(R, g)]) for g in range(32)], axis=1)
    s = np.repeat(s, 16, axis=1)
    err = np.abs(x - k[:, :512])
    normal = s >= 2.0 ** -6
    assert np.all(err[normal] <= 1.0 * s[normal])        # largest e2m1 half-gap (4 -> 6) is 1
    assert np.all(err[normal] <= 1.25 * s[normal])       # the looser bound the page tests use
    assert np.mean(normal) > 0.99


def test_rope_lanes(random_tokens):
    lat, rope = random_tokens
    r352 = oracle.quantize_records(lat, rope, 352)
    rf = (rope.astype(np.uint32) << 16).view(np.float32)
    assert np.array_equal(r352[:, 256:320], torch_e4m3(rf))          # unscaled e4m3 RoPE
    r432 = oracle.quantize_records(lat, rope, 432)
    assert np.array_equal(r432[:, 304:432].view(np.uint16), rope)      # verbatim 16-bit RoPE
    assert np.all(r432[:, 288:304] == 0)                               # zeroed pad


@pytest.mark.parametrize("R", [352, 432])
def test_requantizing_a_dequantized_record_is_a_fixed_point(R):
    # A record in which every group holds a +-6 code: its dequantized values have amax = 6s,
    # so amax/6 = s exactly and every value/s is already on the grid.
    rng = np.random.default_rng(11)
    n = 512
    recs = np.zeros((n, R), dtype=np.uint8)
    nib = rng.integers(0, 16, size=(n, 512)).astype(np.uint8)
    nib[:, ::16] = np.where(rng.random((n, 32)) < 0.5, 0x7, 0xF)
    recs[:, :256] = nib[:, 0::2] | (nib[:, 1::2] << 4)
    sbytes = rng.integers(0x08, 0x7F, size=(n, 32)).astype(np.uint8)          # normal scales
    for g in range(32):
        recs[:, oracle.scale_offset(R, g)] = sbytes[:, g]
    if R == 352:
        rc = rng.integers(0, 256, size=(n, 64)).astype(np.uint8)
        rc[(rc & 0x7F) == 0x7F] = 0x00
        recs[:, 256:320] = rc
    else:
        recs[:, 304:432] = rng.integers(0, 256, size=(n, 128)).astype(np.uint8)
        r16 = recs[:, 304:432].view(np.uint16)
        bad = ((r16 >> 7) & 0xFF) == 0xFF          # keep RoPE finite
        r16[bad] &= 0xBFFF
    k = oracle.dequant_records(recs)
    lat = f32_to_bf16_bits(k[:, :512].astype(np.float32))
    if R == 352:
        rope = f32_to_bf16_bits(k[:, 512:].astype(np.float32))
    else:
        rope = recs[:, 304:432].view(np.uint16).copy()
    # dequantized values are exact in bf16 (<= 5 significant bits)
    assert np.array_equal((lat.astype(np.uint32) << 16).view(np.float32).astype(np.float64), k[:, :512])
    again = oracle.quantize_records(lat, rope, R)
    # -0 nibbles come back as +0 or -0 with the sign of the stored value: compare values first
    assert np.array_equal(oracle.dequant_records(again), k)
    # and bytes exactly, except the 0x8 (negative zero) nibbles whose bf16 value is -0.0
    assert np.array_equal(again, recs)


def test_append_skips_negative_and_out_of_range_slots_and_leaves_others_untouched():
    w = synth.write_path(seed=3, T=64, num_slots=128)
    slots = w.slot_mapping.numpy().copy()
    slots[5] = -1
    slots[9] = 10_000
    cache = np.full((128, 352), 0xAB, dtype=np.uint8)
    lat, rope = synth.bf16_bits(w.latent), synth.bf16_bits(w.rope)
    bad = oracle.quantize_append(lat, rope, slots, cache)
    assert bad == 1
    recs = oracle.quantize_records(lat, rope, 352)
    written = set()
    for t, s in enumerate(slots):
        if 0 <= s < 128:
            assert np.array_equal(cache[s], recs[t])
            written.add(int(s))
    untouched = [s for s in range(128) if s not in written]
    assert np.all(cache[untouched] == 0xAB)


def test_append_honours_row_strides():
    w = synth.write_path(seed=4, T=32, num_slots=64)
    lat = synth.bf16_bits(w.latent)
    rope = synth.bf16_bits(w.rope)
    wide = np.zeros((32, 1200), dtype=np.uint16)
    wide[:, 100:612] = lat
    wide[:, 700:764] = rope
    a = np.full((64, 352), 0xAB, dtype=np.uint8)
    b = np.full((64, 352), 0xAB, dtype=np.uint8)
    oracle.quantize_append(lat, rope, w.slot_mapping.numpy(), a)
    oracle.quantize_append(wide[:, 100:612], wide[:, 700:764], w.slot_mapping.numpy(), b)
    assert np.array_equal(a, b)
