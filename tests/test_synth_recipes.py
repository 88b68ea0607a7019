"""The synthetic workloads follow their stated recipes (shapes, sizes, index structure, value
distributions) and are reproducible from their seeds. CPU only."""
import math

import numpy as np
import pytest
import torch

import synth


def _as_f32(t: torch.Tensor) -> np.ndarray:
    return t.float().numpy()


def test_tiny_decode_recipe():
    w = synth.tiny_decode(seed=0)
    assert (w.B, w.s_q, w.h_q, w.topk, w.num_slots, w.record_bytes) == (1, 1, 64, 64, 256, 352)
    assert tuple(w.q.shape) == (1, 1, 64, 576) and w.q.dtype == torch.bfloat16
    idx = w.indices.numpy().reshape(-1)
    assert (idx == -1).sum() == 8
    used = idx[idx >= 0]
    assert len(np.unique(used)) == used.size and used.max() < 256
    assert w.sm_scale == pytest.approx(1 / math.sqrt(576))


def test_write_recipe():
    w = synth.write_path(seed=0)
    assert (w.T, w.num_slots, w.record_bytes) == (65_536, 262_144, 352)
    slots = w.slot_mapping.numpy()
    assert len(np.unique(slots)) == w.T and slots.min() >= 0 and slots.max() < w.num_slots
    x = _as_f32(w.latent)
    assert x.shape == (65_536, 512) and w.rope.shape == (65_536, 64)
    # N(0,1) with 1% of the values scaled by 20: |x| > 6 comes almost only from the scaled ones
    # (P(|20 z| > 6) = P(|z| > 0.3) = 0.764), so about 0.76% of the values
    frac = float((np.abs(x) > 6).mean())
    assert 0.0066 < frac < 0.0087
    assert abs(float(_as_f32(w.rope).std()) - 1.0) < 0.01


def test_batch_decode_recipe():
    w = synth.batch_decode(seed=0)
    assert (w.B, w.s_q, w.h_q, w.topk, w.num_slots) == (32, 1, 128, 2048, 2_097_152)
    idx = w.indices.numpy().reshape(32, 2048)
    assert (idx >= 0).all() and idx.max() < w.num_slots
    pages_of = [set((row // synth.PAGE).tolist()) for row in idx]
    for b, row in enumerate(idx):
        assert len(np.unique(row)) == 2048
        assert len(pages_of[b]) <= 1024                      # each sequence owns 1,024 pages
    for a in range(32):
        for b in range(a + 1, 32):
            assert not (pages_of[a] & pages_of[b])           # no page shared between sequences
    assert abs(float(_as_f32(w.q).std()) - 1.0) < 0.01


def test_varlen_recipe():
    w = synth.varlen_decode(seed=0)
    assert (w.B, w.s_q, w.h_q, w.topk) == (128, 2, 64, 2048) and w.attn_sink.shape == (64,)
    idx = w.indices.numpy()
    lens = w.seq_lens
    assert lens.min() >= 1_024 and lens.max() <= 131_072
    short = lens < 2048
    # rows of short requests hold at most len entries; every row is padded with -1 only
    for b in np.nonzero(short)[0]:
        assert ((idx[b] >= 0).sum(axis=-1) <= lens[b]).all()
    # besides the padding, about 10% of the entries are set to -1
    long_rows = idx[~short]
    frac = float((long_rows < 0).mean())
    assert 0.09 < frac < 0.11
    assert idx.max() < w.num_slots


def test_long_context_recipe():
    w = synth.long_context(seed=0)
    assert (w.B, w.h_q, w.topk, w.record_bytes, w.num_slots) == (64, 128, 2048, 432, 1_048_576)
    assert (w.seq_lens[:2] == 1_048_576).all()
    assert w.seq_lens[2:].min() >= 8_192 and w.seq_lens[2:].max() <= 262_144
    idx = w.indices.numpy().reshape(64, 2048)
    assert (idx >= 0).all() and idx.max() < w.num_slots
    assert all(len(np.unique(row)) == 2048 for row in idx)


def test_workloads_are_reproducible_from_their_seeds():
    a, b = synth.batch_decode(seed=3), synth.batch_decode(seed=3)
    assert torch.equal(a.indices, b.indices) and torch.equal(a.q.view(torch.int16), b.q.view(torch.int16))
    c = synth.batch_decode(seed=4)
    assert not torch.equal(a.indices, c.indices)
    s = torch.arange(1000, 1064)
    l1, r1 = synth.pool_rows(7, s)
    l2, r2 = synth.pool_rows(7, s)
    assert torch.equal(l1.view(torch.int16), l2.view(torch.int16)) and torch.equal(r1.view(torch.int16), r2.view(torch.int16))
    # the pool generator is per slot: a slot's row does not depend on which other slots are drawn
    l3, _ = synth.pool_rows(7, torch.tensor([1000, 5, 1063]))
    assert torch.equal(l3[0].view(torch.int16), l1[0].view(torch.int16))
    assert torch.equal(l3[2].view(torch.int16), l1[63].view(torch.int16))
