"""Pins for the oracle's producer stage (oracle_norm_rope): RMSNorm of the latent and rotary
embedding of k_pe, each in fp64 and rounded once to bf16, with the values near a bf16 rounding
midpoint flagged. Source of the stage: SGLang PR 38646 "[SM120] Add opt-in NVFP4 sparse-MLA KV
cache format for DeepSeek-V4", "Limitations" (no fused NVFP4 norm+rope+quantize+store kernel)
and "Stores"; the readings of its open parameters are listed in nvfp4_oracle.c.

Each pin checks the oracle against something other than its own formula: torch's rms_norm, numpy
complex multiplication, exact special angles, invariances (power-of-two scaling, the permutation
between the two pair layouts) and hand-built rounding midpoints."""
import numpy as np
import pytest
import torch

import oracle


def bf16_bits(x):
    return (np.asarray(x, np.float32).view(np.uint32) >> 16).astype(np.uint16)


def bits_to_f64(b):
    return (np.asarray(b, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def rand_bf16(rng, shape, scale=1.0):
    # round-to-nearest bf16 of normal draws (truncation would also do: any bf16 is an input)
    f = (rng.standard_normal(shape) * scale).astype(np.float32)
    u = f.view(np.uint32)
    u = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return u.astype(np.uint16)


def tables(n_pos, base=10000.0):
    ang = np.arange(n_pos)[:, None] * (base ** (-np.arange(32) / 32.0))[None, :]
    return np.cos(ang).astype(np.float32), np.sin(ang).astype(np.float32)


def test_rmsnorm_matches_torch_rms_norm_in_float64():
    rng = np.random.default_rng(1)
    T = 16
    lat = rand_bf16(rng, (T, 512), 3.0)
    w = rand_bf16(rng, 512)
    cos, sin = tables(4)
    eps = 1e-6
    r = oracle.norm_rope(lat, rand_bf16(rng, (T, 64)), np.zeros(T, np.int64), w, eps, cos, sin, True)
    ref = torch.nn.functional.rms_norm(torch.from_numpy(bits_to_f64(lat)), (512,),
                                       weight=torch.from_numpy(bits_to_f64(w)), eps=eps).numpy()
    np.testing.assert_allclose(r["exact"][:, :512], ref, rtol=1e-13, atol=0)
    # the stored values are the bf16 roundings of the exact ones
    got = bits_to_f64(r["latent"])
    np.testing.assert_allclose(got, ref, rtol=2.0 ** -8, atol=0)


def test_rmsnorm_unit_rms_and_power_of_two_invariance():
    rng = np.random.default_rng(2)
    T = 8
    lat = rand_bf16(rng, (T, 512), 0.01)
    ones = bf16_bits(np.ones(512))
    cos, sin = tables(2)
    kpe = rand_bf16(rng, (T, 64))
    r = oracle.norm_rope(lat, kpe, np.zeros(T, np.int64), ones, 0.0, cos, sin, True)
    np.testing.assert_allclose((r["exact"][:, :512] ** 2).mean(axis=1), 1.0, rtol=1e-13)
    # x -> 2^k x (exact in bf16 and fp64) leaves the normalized values unchanged when eps = 0
    scaled = (lat.astype(np.int32) + (7 << 7)).astype(np.uint16)   # exponent + 7: x * 128
    assert np.array_equal(bits_to_f64(scaled), bits_to_f64(lat) * 128.0)
    r2 = oracle.norm_rope(scaled, kpe, np.zeros(T, np.int64), ones, 0.0, cos, sin, True)
    assert np.array_equal(r["exact"][:, :512], r2["exact"][:, :512])
    assert np.array_equal(r["latent"], r2["latent"])


@pytest.mark.parametrize("rotate_half", [True, False])
def test_rotation_matches_complex_multiplication(rotate_half):
    rng = np.random.default_rng(3)
    T, n_pos = 12, 50
    kpe = rand_bf16(rng, (T, 64), 2.0)
    pos = rng.integers(0, n_pos, T)
    cos, sin = tables(n_pos)
    r = oracle.norm_rope(rand_bf16(rng, (T, 512)), kpe, pos, bf16_bits(np.ones(512)), 1e-6, cos, sin, rotate_half)
    x = bits_to_f64(kpe)
    ia = np.arange(32) if rotate_half else 2 * np.arange(32)
    ib = ia + 32 if rotate_half else ia + 1
    z = (x[:, ia] + 1j * x[:, ib]) * (cos[pos].astype(np.float64) + 1j * sin[pos].astype(np.float64))
    np.testing.assert_allclose(r["exact"][:, 512 + ia], z.real, rtol=1e-15, atol=1e-300)
    np.testing.assert_allclose(r["exact"][:, 512 + ib], z.imag, rtol=1e-15, atol=1e-300)


@pytest.mark.parametrize("rotate_half", [True, False])
def test_special_angles_are_exact(rotate_half):
    rng = np.random.default_rng(4)
    T = 3
    kpe = rand_bf16(rng, (T, 64))
    x = bits_to_f64(kpe)
    # angle 0 (identity), 90 degrees ((a, b) -> (-b, a)) and 180 degrees (negation)
    cos = np.array([[1.0] * 32, [0.0] * 32, [-1.0] * 32], np.float32)
    sin = np.array([[0.0] * 32, [1.0] * 32, [0.0] * 32], np.float32)
    r = oracle.norm_rope(rand_bf16(rng, (T, 512)), kpe, np.array([0, 1, 2]), bf16_bits(np.ones(512)), 0.0, cos,
                         sin, rotate_half)
    ia = np.arange(32) if rotate_half else 2 * np.arange(32)
    ib = ia + 32 if rotate_half else ia + 1
    assert np.array_equal(r["rope"][0], kpe[0])
    assert np.array_equal(bits_to_f64(r["rope"][1][ia]), -x[1][ib])
    assert np.array_equal(bits_to_f64(r["rope"][1][ib]), x[1][ia])
    assert np.array_equal(bits_to_f64(r["rope"][2]), -x[2])
    assert not r["flag"][:, 512:].any()


def test_the_two_pair_layouts_are_one_permutation_apart():
    rng = np.random.default_rng(5)
    T, n_pos = 10, 40
    kpe = rand_bf16(rng, (T, 64))
    pos = rng.integers(0, n_pos, T)
    cos, sin = tables(n_pos)
    lat = rand_bf16(rng, (T, 512))
    w = bf16_bits(np.ones(512))
    half = oracle.norm_rope(lat, kpe, pos, w, 1e-6, cos, sin, True)
    perm = np.empty(64, np.int64)        # interleaved position 2f <- f, 2f + 1 <- f + 32
    perm[0::2] = np.arange(32)
    perm[1::2] = np.arange(32) + 32
    inter = oracle.norm_rope(lat, np.ascontiguousarray(kpe[:, perm]), pos, w, 1e-6, cos, sin, False)
    assert np.array_equal(inter["rope"], half["rope"][:, perm])
    assert np.array_equal(inter["latent"], half["latent"])


def test_midpoints_are_flagged_with_the_other_rounding():
    T = 4
    lat = bf16_bits(np.ones((T, 512)))
    kpe = np.zeros((T, 64), np.uint16)
    kpe[:, 0] = bf16_bits(1.0)               # pair (0, 32) in rotate-half: a = 1, b = 0 -> (c, s)
    cos = np.ones((T, 32), np.float32)
    sin = np.zeros((T, 32), np.float32)
    cos[0, 0] = 1 + 2.0 ** -8                # exactly the midpoint between 1 and 1 + 2^-7
    cos[1, 0] = 1 + 2.0 ** -8 + 2.0 ** -20   # within 2^-16 of it: flagged, rounds up
    cos[2, 0] = 1 + 2.0 ** -8 + 2.0 ** -14   # farther: not flagged
    cos[3, 0] = 1 + 3 * 2.0 ** -8            # midpoint between 1 + 2^-7 and 1 + 2^-6 (odd below)
    r = oracle.norm_rope(lat, kpe, np.arange(T), bf16_bits(np.ones(512)), 0.0, cos, sin, True)
    v = bits_to_f64(r["rope"][:, 0])
    o = bits_to_f64(r["other"][:, 512])
    assert list(r["flag"][:, 512]) == [1, 1, 0, 1]
    assert v[0] == 1.0 and o[0] == 1 + 2.0 ** -7                 # ties to even
    assert v[1] == 1 + 2.0 ** -7 and o[1] == 1.0
    assert v[2] == 1 + 2.0 ** -7 and o[2] == v[2]
    assert v[3] == 1 + 2.0 ** -6 and o[3] == 1 + 2.0 ** -7       # ties to even: the even one above
    # the latent of all ones normalizes to exactly 1: nothing flagged there
    assert not r["flag"][:, :512].any() and np.all(bits_to_f64(r["latent"]) == 1.0)


def test_positions_out_of_range_are_not_written():
    rng = np.random.default_rng(6)
    cos, sin = tables(8)
    r = oracle.norm_rope(rand_bf16(rng, (4, 512)), rand_bf16(rng, (4, 64)), np.array([0, -1, 8, 7]),
                         bf16_bits(np.ones(512)), 1e-6, cos, sin, True)
    assert list(r["valid"]) == [1, 0, 0, 1]
    assert not r["latent"][1:3].any() and not r["rope"][1:3].any()
