"""The Python binding rejects malformed arguments with ValueError before any CUDA call (so
these run on CPU), and its workspace query reaches the C ABI's host-side checks."""
import pytest
import torch

import nvfp4_kv_cache_sparse_gb300 as lib
from nvfp4_kv_cache_sparse_gb300 import build


@pytest.fixture(scope="module", autouse=True)
def built():
    build.build()
    lib.load()


def bf16(*shape):
    return torch.zeros(shape, dtype=torch.bfloat16)


def test_quantize_append_rejects_bad_arguments():
    lat, rope = bf16(4, 512), bf16(4, 64)
    slots = torch.arange(4, dtype=torch.int64)
    cache = torch.zeros(8, 352, dtype=torch.uint8)
    with pytest.raises(ValueError, match="bf16"):
        lib.quantize_append(lat.float(), rope, slots, cache)
    with pytest.raises(ValueError, match="kv_latent"):
        lib.quantize_append(bf16(4, 511), rope, slots, cache)
    with pytest.raises(ValueError, match="token counts"):
        lib.quantize_append(lat, bf16(3, 64), slots, cache)
    with pytest.raises(ValueError, match="slot_mapping"):
        lib.quantize_append(lat, rope, slots.int(), cache)
    with pytest.raises(ValueError, match="record width"):
        lib.quantize_append(lat, rope, slots, torch.zeros(8, 400, dtype=torch.uint8))
    with pytest.raises(ValueError, match="block_scales"):
        lib.quantize_append(lat, rope, slots, torch.zeros(8, 432, dtype=torch.uint8), block_scales=True)
    with pytest.raises(ValueError, match="CUDA device"):
        lib.quantize_append(lat, rope, slots, cache)       # host tensors: refused before any launch


def test_decode_rejects_bad_arguments():
    q = bf16(2, 1, 64, 576)
    idx = torch.zeros(2, 1, 16, dtype=torch.int32)
    cache = torch.zeros(32, 352, dtype=torch.uint8)
    with pytest.raises(ValueError, match="q bf16"):
        lib.sparse_mla_decode(bf16(2, 1, 64, 512), cache, idx, 0.1)
    with pytest.raises(ValueError, match="indices"):
        lib.sparse_mla_decode(q, cache, idx.long(), 0.1)
    with pytest.raises(ValueError, match="cache"):
        lib.sparse_mla_decode(q, torch.zeros(32, 360, dtype=torch.uint8), idx, 0.1)
    with pytest.raises(ValueError, match="attn_sink"):
        lib.sparse_mla_decode(q, cache, idx, 0.1, attn_sink=torch.zeros(63))
    with pytest.raises(ValueError, match="block_scales"):
        lib.sparse_mla_decode(q, torch.zeros(32, 656, dtype=torch.uint8), idx, 0.1, block_scales=True)


def test_workspace_size_for_every_record_layout():
    per_split = 2 * 64 * 512 * 2                  # f16 partials of 2 rows x 64 heads
    for code in (352, 432, 656, 352 | lib.SCALES_BLOCK_ORDER):
        assert lib.workspace_size(2, 1, 64, 64, code, 1) == 0
        assert lib.workspace_size(2, 1, 64, 64, code, 2) == 2 * per_split + 1024
    with pytest.raises(lib.Nvfp4MlaError):
        lib.workspace_size(2, 1, 64, 64, 432 | lib.SCALES_BLOCK_ORDER, 2)
