"""The end-to-end loop's packed transfer buffers (bench.py pack_layout / pack_views): every part
starts on a 256-byte boundary, parts do not overlap, and a part written through its view reads
back unchanged from the buffer's bytes."""
import numpy as np
import torch

import bench


def test_layout_is_aligned_and_disjoint():
    parts = [((32, 1, 128, 576), torch.bfloat16), ((32, 1, 2048), torch.int32), ((32, 512), torch.bfloat16),
             ((32, 64), torch.bfloat16), ((32,), torch.int64), ((3,), torch.uint8), ((5, 7), torch.float32)]
    offs, n = bench.pack_layout(parts)
    sizes = [int(np.prod(sh)) * torch.empty((), dtype=dt).element_size() for sh, dt in parts]
    assert all(o % 256 == 0 for o in offs)
    for k in range(len(parts) - 1):
        assert offs[k] + sizes[k] <= offs[k + 1]
    assert offs[-1] + sizes[-1] <= n and n % 256 == 0 and n - (offs[-1] + sizes[-1]) < 256


def test_views_round_trip():
    rng = np.random.default_rng(3)
    tensors = [torch.from_numpy(rng.standard_normal((4, 3, 8)).astype(np.float32)).to(torch.bfloat16),
               torch.from_numpy(rng.integers(-5, 2**20, size=(4, 3, 17), dtype=np.int32)),
               torch.from_numpy(rng.integers(0, 2**40, size=(6,), dtype=np.int64)),
               torch.from_numpy(rng.standard_normal((4, 3)).astype(np.float32))]
    parts = [(tuple(t.shape), t.dtype) for t in tensors]
    offs, n = bench.pack_layout(parts)
    buf = torch.zeros(n, dtype=torch.uint8)
    for v, t in zip(bench.pack_views(buf, parts, offs), tensors):
        assert v.is_contiguous() and v.shape == t.shape and v.dtype == t.dtype
        v.copy_(t)
    copy = buf.clone()   # what one byte copy of the buffer carries
    for v, t in zip(bench.pack_views(copy, parts, offs), tensors):
        assert torch.equal(v, t)


def test_valid_only_roofline_counts_used_entries():
    """bench.roofline_numbers_valid_only: only entries >= 0 contribute records and contraction
    work; q and the whole index lists are always read (the tiny workload masks 8 of 64)."""
    import synth
    w = synth.tiny_decode(seed=0)
    used = int((w.indices >= 0).sum())
    assert 0 < used < w.indices.numel()
    flops, bytes_ = bench.roofline_numbers_valid_only(w)
    assert flops == 2.0 * w.h_q * used * (576 + 512)
    assert bytes_ == used * w.record_bytes + w.n_rows * (w.h_q * 576 * 2 + w.topk * 4)
    full_flops, full_bytes = bench.roofline_numbers(w)
    assert flops < full_flops and bytes_ < full_bytes
