"""Quantize-and-append on the GPU, bit-exact against the CPU oracle.

Covers every finite bf16 input value, every e4m3 scale with all the bf16 values that can
share a group with it, both record widths, the write workload at full size, untouched and
skipped slots, out-of-range slots, and strided inputs."""
import numpy as np
import pytest
import torch

import nvfp4_kv_cache_sparse_gb300 as lib
import oracle
import synth

pytestmark = pytest.mark.gpu
DEV = "cuda"


def gpu_quantize(lat_bits: np.ndarray, rope_bits: np.ndarray, slots: np.ndarray, num_slots: int, R: int,
                 fill: int = 0xAB):
    lat = torch.from_numpy(lat_bits.view(np.int16)).view(torch.bfloat16).to(DEV)
    rope = torch.from_numpy(rope_bits.view(np.int16)).view(torch.bfloat16).to(DEV)
    cache = torch.full((num_slots, R), fill, dtype=torch.uint8, device=DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    lib.quantize_append(lat, rope, torch.from_numpy(slots).to(DEV), cache, dev_status=status)
    torch.cuda.synchronize()
    return cache.cpu().numpy(), int(status.item())


def oracle_quantize(lat_bits, rope_bits, slots, num_slots, R, fill=0xAB):
    cache = np.full((num_slots, R), fill, dtype=np.uint8)
    bad = oracle.quantize_append(lat_bits, rope_bits, slots, cache)
    return cache, bad


def finite_bf16_bits() -> np.ndarray:
    b = np.arange(65536, dtype=np.uint32)
    f = (b << 16).view(np.float32)
    return b[np.isfinite(f)].astype(np.uint16)


@pytest.mark.parametrize("R", [352, 432])
def test_every_finite_bf16_value(R):
    vals = finite_bf16_bits()
    rng = np.random.default_rng(0)
    vals = vals[rng.permutation(vals.size)]
    T = (vals.size + 511) // 512
    lat = np.zeros(T * 512, dtype=np.uint16)
    lat[:vals.size] = vals
    lat = lat.reshape(T, 512)
    rope = np.resize(vals, T * 64).reshape(T, 64)
    slots = np.arange(T, dtype=np.int64)
    got, st = gpu_quantize(lat, rope, slots, T, R)
    exp, _ = oracle_quantize(lat, rope, slots, T, R)
    assert st == 0
    mism = np.argwhere(got != exp)
    assert mism.size == 0, f"{len(mism)} bytes differ, first at {mism[:5].tolist()}"


@pytest.mark.parametrize("R", [352, 432])
def test_every_scale_with_every_value_it_can_divide(R):
    # Group = [6s, x_1 .. x_15]: amax = 6s gives amax/6 = s exactly, so the stored scale is s
    # and every x with |x| <= 6s is divided by it. For each of the 126 non-zero finite
    # scales, all bf16 x in [s/8, 6s] (both signs) are placed in such groups.
    all_bits = finite_bf16_bits()
    mags = (all_bits.astype(np.uint32) << 16).view(np.float32)
    groups = []
    for code in range(1, 0x7F):
        s = float(oracle.e4m3_decode(np.uint8(code)))
        sel = all_bits[(mags >= s / 8) & (mags <= 6 * s)]           # includes negatives (mags < 0 excluded)
        sel = np.concatenate([sel, sel | 0x8000])
        head = synth.bf16_bits(torch.tensor([6 * s], dtype=torch.float32).to(torch.bfloat16))[0]
        for i in range(0, sel.size, 15):
            g = np.zeros(16, dtype=np.uint16)
            chunk = sel[i:i + 15]
            g[0] = head
            g[1:1 + chunk.size] = chunk
            groups.append(g)
    groups = np.stack(groups)
    T = (len(groups) + 31) // 32
    lat = np.zeros((T * 32, 16), dtype=np.uint16)
    lat[:len(groups)] = groups
    lat = lat.reshape(T, 512)
    rope = np.zeros((T, 64), dtype=np.uint16)
    slots = np.arange(T, dtype=np.int64)
    got, _ = gpu_quantize(lat, rope, slots, T, R)
    exp, _ = oracle_quantize(lat, rope, slots, T, R)
    assert np.array_equal(got, exp)


@pytest.mark.parametrize("R", [352, 432])
def test_tiny_pool(R):
    slots = torch.arange(256)
    lat, rope = synth.pool_rows(0, slots)
    lb, rb = synth.bf16_bits(lat), synth.bf16_bits(rope)
    got, _ = gpu_quantize(lb, rb, slots.numpy(), 256, R)
    exp, _ = oracle_quantize(lb, rb, slots.numpy(), 256, R)
    assert np.array_equal(got, exp)


@pytest.mark.parametrize("R", [352, 432])
def test_write_workload_full_size(R):
    w = synth.write_path(seed=0, record_bytes=R)
    lb, rb = synth.bf16_bits(w.latent), synth.bf16_bits(w.rope)
    slots = w.slot_mapping.numpy()
    got, st = gpu_quantize(lb, rb, slots, w.num_slots, R)
    exp, _ = oracle_quantize(lb, rb, slots, w.num_slots, R)
    assert st == 0
    assert np.array_equal(got, exp)
    untouched = np.setdiff1d(np.arange(w.num_slots), slots)
    assert np.all(got[untouched] == 0xAB)


def test_skipped_and_out_of_range_slots():
    w = synth.write_path(seed=5, T=1000, num_slots=2000)
    lb, rb = synth.bf16_bits(w.latent), synth.bf16_bits(w.rope)
    slots = w.slot_mapping.numpy().copy()
    slots[::7] = -1
    slots[3] = 2000
    slots[11] = 1 << 40
    got, st = gpu_quantize(lb, rb, slots, 2000, 352)
    exp, bad = oracle_quantize(lb, rb, slots, 2000, 352)
    assert bad == 2 and st == lib.DEV_SLOT_OUT_OF_RANGE
    assert np.array_equal(got, exp)


def test_strided_inputs_and_empty_call():
    w = synth.write_path(seed=6, T=300, num_slots=512)
    wide = torch.zeros((300, 1024), dtype=torch.bfloat16)
    wide[:, 64:576] = w.latent
    wide[:, 704:768] = w.rope
    wide = wide.to(DEV)
    cache = torch.full((512, 352), 0xAB, dtype=torch.uint8, device=DEV)
    slots = w.slot_mapping.to(DEV)
    lib.quantize_append(wide[:, 64:576], wide[:, 704:768], slots, cache)
    ref = torch.full((512, 352), 0xAB, dtype=torch.uint8, device=DEV)
    lib.quantize_append(w.latent.to(DEV).contiguous(), w.rope.to(DEV).contiguous(), slots, ref)
    empty = torch.empty((0, 512), dtype=torch.bfloat16, device=DEV)
    lib.quantize_append(empty, torch.empty((0, 64), dtype=torch.bfloat16, device=DEV),
                        torch.empty(0, dtype=torch.int64, device=DEV), cache)
    torch.cuda.synchronize()
    assert torch.equal(cache, ref)


def test_pool_contents_are_identical_on_cpu_and_gpu():
    slots = torch.arange(0, 5_000_000, 997)
    a = synth.pool_rows(17, slots)
    b = synth.pool_rows(17, slots.to(DEV))
    assert torch.equal(a[0], b[0].cpu()) and torch.equal(a[1], b[1].cpu())
