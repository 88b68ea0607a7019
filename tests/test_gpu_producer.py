"""The fused producer (RMSNorm + rotary embedding + quantize + append) on the GPU against the
oracle: SGLang PR 38646 "[SM120] Add opt-in NVFP4 sparse-MLA KV cache format for DeepSeek-V4",
"Limitations" / "Stores".

The oracle computes both stages in fp64 and rounds once to bf16, flagging values whose exact
result lies within 2^-16 (relative to its terms) of a bf16 rounding midpoint, with the other
admissible rounding. The kernel computes in fp32, so:
  * every record field built only from unflagged values must equal the oracle's bit for bit;
  * a field with flagged values (a 16-value group with its scale, a 128-value fp8 tile with its
    scale, one RoPE value) must equal the oracle's field for one of the combinations of the
    admissible roundings of its flagged values.
The count of flagged fields is reported."""
import itertools

import numpy as np
import pytest
import torch

import nvfp4_kv_cache_sparse_gb300 as lib
import oracle
import synth

pytestmark = pytest.mark.gpu
DEV = "cuda"


def field_bytes(R, blk):
    """Byte positions of each field of a record: NoPE units (groups, or fp8 tiles) and RoPE values.
    Returns (units: list of (value indices, byte indices)), rope: list of (value index, bytes))."""
    units, rope = [], []
    if R == 656:
        for t in range(4):
            units.append((np.arange(128 * t, 128 * t + 128), np.r_[np.arange(128 * t, 128 * t + 128),
                                                                   np.arange(512 + 4 * t, 516 + 4 * t)]))
        rope = [(512 + e, np.array([528 + 2 * e, 529 + 2 * e])) for e in range(64)]
    else:
        for g in range(32):
            units.append((np.arange(16 * g, 16 * g + 16),
                          np.r_[np.arange(8 * g, 8 * g + 8), [oracle.scale_offset(R, g, blk)]]))
        if R == 352:
            rope = [(512 + e, np.array([256 + e])) for e in range(64)]
        else:
            rope = [(512 + e, np.array([304 + 2 * e, 305 + 2 * e])) for e in range(64)]
    return units, rope


def check_records(got, lat_in, rope_in, res, slots, R, blk, max_combo_bits=10):
    """Compare the GPU records of the written tokens with the oracle's, field by field."""
    units, rope = field_bytes(R, blk)
    near = np.concatenate([res["latent"], res["rope"]], axis=1)       # [T,576] bf16 bits
    exp = oracle.quantize_records(res["latent"], res["rope"], R, blk)
    flagged_fields = 0
    for t in np.nonzero(res["valid"])[0]:
        rec = got[slots[t]]
        fl = res["flag"][t]
        if not fl.any():
            assert np.array_equal(rec, exp[t]), f"token {t}: record differs with nothing flagged"
            continue
        for vals, byts in units + [(np.array([v]), b) for v, b in rope]:
            f = vals[fl[vals] != 0]
            if f.size == 0:
                assert np.array_equal(rec[byts], exp[t][byts]), f"token {t}: unflagged field differs"
                continue
            flagged_fields += 1
            assert f.size <= max_combo_bits
            ok = False
            for choice in itertools.product((0, 1), repeat=f.size):
                alt = near[t].copy()
                for v, c in zip(f, choice):
                    if c:
                        alt[v] = res["other"][t][v]
                r2 = oracle.quantize_records(alt[None, :512].copy(), alt[None, 512:].copy(), R, blk)[0]
                if np.array_equal(rec[byts], r2[byts]):
                    ok = True
                    break
            assert ok, f"token {t}: flagged field (values {f.tolist()}) matches no admissible rounding"
    return flagged_fields


def run_gpu(pw: synth.ProducerWorkload, R, blk, slots=None):
    w = pw.write
    slots = w.slot_mapping if slots is None else slots
    cache = torch.full((w.num_slots, R), 0xAB, dtype=torch.uint8, device=DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    lib.norm_rope_quantize_append(w.latent.to(DEV), pw.norm_weight.to(DEV), pw.eps, w.rope.to(DEV),
                                  pw.positions.to(DEV), pw.cos_table.to(DEV), pw.sin_table.to(DEV), pw.rotate_half,
                                  slots.to(DEV), cache, dev_status=status, block_scales=blk)
    torch.cuda.synchronize()
    return cache.cpu().numpy(), int(status.item())


def run_oracle(pw: synth.ProducerWorkload, rows=None):
    w = pw.write
    lb, rb = synth.bf16_bits(w.latent), synth.bf16_bits(w.rope)
    pos = pw.positions.numpy()
    if rows is not None:
        lb, rb, pos = lb[rows], rb[rows], pos[rows]
    return oracle.norm_rope(lb, rb, pos, synth.bf16_bits(pw.norm_weight), pw.eps, pw.cos_table.numpy(),
                            pw.sin_table.numpy(), pw.rotate_half)


@pytest.mark.parametrize("R,blk", [(352, False), (432, False), (352, True), (656, False)])
@pytest.mark.parametrize("rotate_half", [True, False])
def test_small_batch_against_the_oracle(R, blk, rotate_half):
    pw = synth.producer_inputs(seed=3 + R, T=300, num_slots=700, record_bytes=R, num_positions=4096,
                               rotate_half=rotate_half)
    pos = pw.positions.numpy().copy()
    pos[[7, 100]] = [-1, 4096]                          # out of range: skipped, status bit
    pw.positions = torch.from_numpy(pos)
    got, st = run_gpu(pw, R, blk)
    assert st == lib.DEV_POSITION_OUT_OF_RANGE
    res = run_oracle(pw)
    slots = pw.write.slot_mapping.numpy()
    n = check_records(got, None, None, res, slots, R, blk)
    print(f"R={R} blk={blk} rotate_half={rotate_half}: {n} flagged fields of {300 * (64 + (4 if R == 656 else 32))}")
    assert np.all(got[slots[[7, 100]]] == 0xAB)
    untouched = np.setdiff1d(np.arange(700), slots)
    assert np.all(got[untouched] == 0xAB)


@pytest.mark.parametrize("R", [352, 432])
def test_write_workload_full_size_sampled(R):
    """The write workload's 65,536 tokens at full size; the oracle checks 1,024 sampled tokens
    and every other slot must stay untouched."""
    pw = synth.producer_inputs(seed=0, record_bytes=R)
    got, st = run_gpu(pw, R, False)
    assert st == 0
    rows = np.random.default_rng(9).choice(pw.write.T, 1024, replace=False)
    res = run_oracle(pw, rows)
    slots = pw.write.slot_mapping.numpy()[rows]
    n = check_records(got, None, None, res, slots, R, False)
    print(f"R={R}: {n} flagged fields among 1024 sampled tokens")
    untouched = np.setdiff1d(np.arange(pw.write.num_slots), pw.write.slot_mapping.numpy())
    assert np.all(got[untouched] == 0xAB)


def test_fused_equals_norm_then_append_where_nothing_is_flagged():
    """The fused call and the unfused path (the oracle's bf16 intermediate, then the GPU append)
    write the same records for every token without a flagged value."""
    pw = synth.producer_inputs(seed=11, T=2000, num_slots=4000, record_bytes=352)
    got, _ = run_gpu(pw, 352, False)
    res = run_oracle(pw)
    lat = torch.from_numpy(res["latent"].view(np.int16)).view(torch.bfloat16).to(DEV)
    rope = torch.from_numpy(res["rope"].view(np.int16)).view(torch.bfloat16).to(DEV)
    cache = torch.full((4000, 352), 0xAB, dtype=torch.uint8, device=DEV)
    lib.quantize_append(lat, rope, pw.write.slot_mapping.to(DEV), cache)
    unfused = cache.cpu().numpy()
    clean = ~res["flag"].any(axis=1)
    slots = pw.write.slot_mapping.numpy()
    assert clean.sum() > 0
    assert np.array_equal(got[slots[clean]], unfused[slots[clean]])


def test_argument_checks():
    dev = torch.device(DEV)
    z = lambda *s, dt=torch.bfloat16: torch.zeros(*s, dtype=dt, device=dev)
    cache = torch.zeros((8, 352), dtype=torch.uint8, device=dev)
    args = dict(kv_latent=z(4, 512), norm_weight=z(512), eps=1e-6, k_pe=z(4, 64),
                positions=z(4, dt=torch.int64), cos_table=z(8, 32, dt=torch.float32),
                sin_table=z(8, 32, dt=torch.float32), rotate_half=True, slot_mapping=z(4, dt=torch.int64), cache=cache)
    lib.norm_rope_quantize_append(**args)
    with pytest.raises(lib.Nvfp4MlaError):
        lib.norm_rope_quantize_append(**dict(args, eps=-1.0))
    with pytest.raises(ValueError):
        lib.norm_rope_quantize_append(**dict(args, cos_table=z(8, 16, dt=torch.float32)))
