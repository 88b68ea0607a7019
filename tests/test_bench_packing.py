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
