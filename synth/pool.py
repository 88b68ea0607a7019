"""Fill a device-resident KV pool with the records of ``synth.pool_rows`` contents.

The quantizer is passed in (the library's ``quantize_append``), so this module still holds
none of the method's arithmetic: it only generates slot contents chunk by chunk on the
device and hands them over.
"""
from __future__ import annotations

from typing import Callable

import torch

from . import pool_rows


def fill_pool(quantize_append: Callable, num_slots: int, record_bytes: int, pool_seed: int,
              device, chunk: int = 131_072, fill_byte: int = 0xAB) -> torch.Tensor:
    cache = torch.full((num_slots, record_bytes), fill_byte, dtype=torch.uint8, device=device)
    for start in range(0, num_slots, chunk):
        slots = torch.arange(start, min(num_slots, start + chunk), device=device, dtype=torch.int64)
        lat, rope = pool_rows(pool_seed, slots)
        quantize_append(lat, rope, slots, cache)
    return cache
