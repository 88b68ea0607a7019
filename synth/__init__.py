"""Seeded synthetic inputs shared by the tests, the smoke check and the benchmark.

This module holds no arithmetic of the method (no quantization, no attention): it only draws
numbers. Both the CPU oracle and the CUDA library consume what it produces.

Two generators are used:

* ``numpy.random.default_rng(seed)`` for everything small enough to draw on the host
  (query vectors, index lists, page tables, the write-path batch).
* ``hashed_normal_bf16`` for the contents of large KV pools. It is counter based (value =
  f(seed, slot, column)) and uses only int64 arithmetic, an exact int->fp32 conversion and a
  power-of-two scaling, so the same torch code yields bit-identical bf16 values on the CPU and
  on the GPU. That lets a test rebuild, on the host, exactly the records a pool filled on the
  device holds, for just the slots it samples. Each value is a sum of twelve 16-bit uniforms,
  centred and divided by 2^16 (Irwin-Hall, unit variance, support +-6).

Workloads mirror the five configurations of the benchmark (tiny decode, write path, B=32 decode,
varlen MTP decode with sinks, 432-B long-context pool). ``WORKLOADS`` lists them by name.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import Dict, List, Optional

import numpy as np
import torch

PAGE = 64          # tokens per page of the paged pool
D_NOPE = 512
D_ROPE = 64
D_QK = 576
D_V = 512

_MASK64 = (1 << 64) - 1


def _s64(x: int) -> int:
    """Reinterpret an unsigned 64-bit constant as a signed int64 value (torch int64)."""
    x &= _MASK64
    return x - (1 << 64) if x >= (1 << 63) else x


_GOLDEN = _s64(0x9E3779B97F4A7C15)
_MIX1 = _s64(0xBF58476D1CE4E5B9)
_MIX2 = _s64(0x94D049BB133111EB)


def _lsr(z: torch.Tensor, k: int) -> torch.Tensor:
    """Logical right shift of int64 lanes."""
    return (z >> k) & ((1 << (64 - k)) - 1)


def _splitmix64(z: torch.Tensor) -> torch.Tensor:
    z = z + _GOLDEN
    z = (z ^ _lsr(z, 30)) * _MIX1
    z = (z ^ _lsr(z, 27)) * _MIX2
    return z ^ _lsr(z, 31)


def hashed_normal_bf16(seed: int, rows: torch.Tensor, width: int, salt: int) -> torch.Tensor:
    """bf16 [len(rows), width], approximately N(0,1), a pure function of (seed, salt, row, col).
    Runs on ``rows.device``; CPU and GPU results are bit-identical."""
    rows = rows.to(torch.int64).reshape(-1, 1)
    cols = torch.arange(width, device=rows.device, dtype=torch.int64).reshape(1, -1)
    base = (rows * 4096 + cols) * 4 + _s64((seed * 1_000_003 + salt) << 40)
    total = torch.zeros(rows.shape[0], width, device=rows.device, dtype=torch.int64)
    for k in range(3):
        h = _splitmix64(base + k)
        for j in range(4):
            total += _lsr(h, 16 * j) & 0xFFFF
    centred = (total - 6 * 65535).to(torch.float32)       # exact: |value| < 2^24
    return (centred / 65536.0).to(torch.bfloat16)          # exact scaling, then bf16 RNE


def pool_rows(seed: int, slots: torch.Tensor):
    """KV contents of pool slots: (latent bf16 [n,512], rope bf16 [n,64])."""
    return (hashed_normal_bf16(seed, slots, D_NOPE, salt=1),
            hashed_normal_bf16(seed, slots, D_ROPE, salt=2))


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    """bf16 torch tensor (any device) -> numpy uint16 bit patterns."""
    return t.detach().to("cpu").contiguous().view(torch.int16).numpy().view(np.uint16)


def bf16_from_f32(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16)


# ---------------------------------------------------------------------------------------
# Workloads
# ---------------------------------------------------------------------------------------

@dataclass
class WriteWorkload:
    name: str
    T: int
    num_slots: int
    record_bytes: int
    latent: torch.Tensor            # bf16 [T,512] (CPU)
    rope: torch.Tensor              # bf16 [T,64]  (CPU)
    slot_mapping: torch.Tensor      # int64 [T]    (CPU)
    fill_byte: int = 0xAB


@dataclass
class DecodeWorkload:
    name: str
    B: int
    s_q: int
    h_q: int
    topk: int
    record_bytes: int
    num_slots: int
    sm_scale: float
    q: torch.Tensor                 # bf16 [B, s_q, h_q, 576] (CPU)
    indices: torch.Tensor           # int32 [B, s_q, topk]    (CPU)
    attn_sink: Optional[torch.Tensor]   # fp32 [h_q] or None
    pool_seed: int                  # pool slot s holds pool_rows(pool_seed, s)
    seq_lens: Optional[np.ndarray] = None
    notes: Dict[str, str] = field(default_factory=dict)

    @property
    def n_rows(self) -> int:
        return self.B * self.s_q


def _normal_bf16(rng: np.random.Generator, shape) -> torch.Tensor:
    return bf16_from_f32(rng.standard_normal(shape, dtype=np.float32))


def tiny_decode(seed: int = 0, h_q: int = 64, topk: int = 64, n_invalid: int = 8,
                num_slots: int = 256, record_bytes: int = 352) -> DecodeWorkload:
    """B=1, s_q=1, h_q=64, 256-slot pool, 64 distinct indices with 8 set to -1."""
    rng = np.random.default_rng(seed)
    q = _normal_bf16(rng, (1, 1, h_q, D_QK))
    idx = rng.choice(num_slots, size=topk, replace=False).astype(np.int32)
    idx[rng.choice(topk, size=n_invalid, replace=False)] = -1
    return DecodeWorkload("tiny_decode_b1_h64_topk64", 1, 1, h_q, topk, record_bytes, num_slots,
                          1.0 / math.sqrt(D_QK), q, torch.from_numpy(idx.reshape(1, 1, topk)), None,
                          pool_seed=seed)


def write_path(seed: int = 0, T: int = 65_536, num_slots: int = 262_144,
               record_bytes: int = 352, outlier_p: float = 0.01, outlier_scale: float = 20.0) -> WriteWorkload:
    """Quantize-append of T tokens (latent ~N(0,1) with 1% outliers x20, RoPE ~N(0,1)) into a
    pool of num_slots records via a random unique slot_mapping; other slots hold 0xAB."""
    rng = np.random.default_rng(seed)
    lat = rng.standard_normal((T, D_NOPE), dtype=np.float32)
    lat = np.where(rng.random((T, D_NOPE)) < outlier_p, lat * np.float32(outlier_scale), lat)
    rope = rng.standard_normal((T, D_ROPE), dtype=np.float32)
    slots = rng.permutation(num_slots)[:T].astype(np.int64)
    return WriteWorkload(f"write_T{T}_slots{num_slots}_R{record_bytes}", T, num_slots, record_bytes,
                         bf16_from_f32(lat), bf16_from_f32(rope), torch.from_numpy(slots))


@dataclass
class ProducerWorkload:
    """Inputs of the fused producer (norm + rotary embedding + quantize + append): the write
    workload's latent and k_pe taken as the PRE-norm / PRE-rotation values, plus the stage
    parameters a caller supplies."""
    write: WriteWorkload
    norm_weight: torch.Tensor       # bf16 [512]
    eps: float
    positions: torch.Tensor         # int64 [T]
    cos_table: torch.Tensor         # fp32 [num_positions, 32]
    sin_table: torch.Tensor         # fp32 [num_positions, 32]
    rotate_half: bool


def producer_inputs(seed: int = 0, T: int = 65_536, num_slots: int = 262_144, record_bytes: int = 352,
                    num_positions: int = 65_536, rotate_half: bool = True,
                    rope_base: float = 10_000.0) -> ProducerWorkload:
    """write_path's tokens with per-token magnitudes spread over 2^-8 .. 2^8 (the norm removes
    them), a norm weight ~ 1 + 0.1 N(0,1), eps 1e-6, positions uniform in [0, num_positions),
    and the usual rotary tables: angle p * rope_base^(-f/32) for frequency f."""
    w = write_path(seed=seed, T=T, num_slots=num_slots, record_bytes=record_bytes)
    rng = np.random.default_rng(seed + 1)
    mag = np.exp2(rng.uniform(-8, 8, (T, 1))).astype(np.float32)
    lat = w.latent.float().numpy() * mag
    w.latent = bf16_from_f32(lat)
    weight = bf16_from_f32((1.0 + 0.1 * rng.standard_normal(D_NOPE)).astype(np.float32))
    pos = rng.integers(0, num_positions, T).astype(np.int64)
    ang = np.arange(num_positions, dtype=np.float64)[:, None] * (rope_base ** (-np.arange(32) / 32.0))[None, :]
    return ProducerWorkload(w, weight, 1e-6, torch.from_numpy(pos), torch.from_numpy(np.cos(ang).astype(np.float32)),
                            torch.from_numpy(np.sin(ang).astype(np.float32)), rotate_half)


def _positions_to_slots(page_table: np.ndarray, pos: np.ndarray) -> np.ndarray:
    return page_table[pos // PAGE] * PAGE + pos % PAGE


def batch_decode(seed: int = 0, B: int = 32, h_q: int = 128, topk: int = 2048,
                 seq_len: int = 65_536, num_pages: int = 32_768) -> DecodeWorkload:
    """B sequences of seq_len tokens in a paged pool of num_pages 64-token pages; each sequence
    owns seq_len/64 pages from a seeded permutation; topk distinct positions per query."""
    rng = np.random.default_rng(seed)
    pages_per_seq = seq_len // PAGE
    assert B * pages_per_seq <= num_pages
    perm = rng.permutation(num_pages)
    idx = np.empty((B, 1, topk), dtype=np.int32)
    for b in range(B):
        table = perm[b * pages_per_seq:(b + 1) * pages_per_seq]
        pos = rng.choice(seq_len, size=topk, replace=False)
        idx[b, 0] = _positions_to_slots(table, pos)
    q = _normal_bf16(rng, (B, 1, h_q, D_QK))
    return DecodeWorkload(f"decode_b{B}_sq1_h{h_q}_topk{topk}_R352", B, 1, h_q, topk, 352,
                          num_pages * PAGE, 1.0 / math.sqrt(D_QK), q, torch.from_numpy(idx), None,
                          pool_seed=seed + 1000, seq_lens=np.full(B, seq_len))


def varlen_decode(seed: int = 0, B: int = 128, s_q: int = 2, h_q: int = 64, topk: int = 2048,
                  len_lo: int = 1_024, len_hi: int = 131_072, extra_invalid: float = 0.10) -> DecodeWorkload:
    """MTP decode over per-request cache lengths U[len_lo, len_hi]; short requests pad with -1,
    then 10% of all entries are set to -1; per-head attention sink ~N(0,1)."""
    rng = np.random.default_rng(seed)
    lens = rng.integers(len_lo, len_hi + 1, size=B)
    pages = (lens + PAGE - 1) // PAGE
    num_pages = int(pages.sum())
    perm = rng.permutation(num_pages)
    starts = np.concatenate([[0], np.cumsum(pages)[:-1]])
    idx = np.full((B, s_q, topk), -1, dtype=np.int32)
    for b in range(B):
        table = perm[starts[b]:starts[b] + pages[b]]
        for i in range(s_q):
            n = min(int(lens[b]), topk)
            pos = rng.choice(int(lens[b]), size=n, replace=False)
            idx[b, i, :n] = _positions_to_slots(table, pos)
    idx[rng.random(idx.shape) < extra_invalid] = -1
    q = _normal_bf16(rng, (B, s_q, h_q, D_QK))
    sink = torch.from_numpy(rng.standard_normal(h_q, dtype=np.float32))
    return DecodeWorkload(f"varlen_b{B}_sq{s_q}_h{h_q}_topk{topk}_sink_R352", B, s_q, h_q, topk, 352,
                          num_pages * PAGE, 1.0 / math.sqrt(D_QK), q, torch.from_numpy(idx), sink,
                          pool_seed=seed + 2000, seq_lens=lens)


def long_context(seed: int = 0, B: int = 64, h_q: int = 128, topk: int = 2048, num_slots: int = 1_048_576,
                 n_long: int = 2, len_lo: int = 8_192, len_hi: int = 262_144) -> DecodeWorkload:
    """432-B records in a 1,048,576-slot pool; requests 0..n_long-1 span the whole pool (1M
    tokens), the rest have lengths U[len_lo, len_hi]. Each request's page table is a seeded
    permutation of all pool pages cut to its length, so pages alias across requests (the data
    are read-only)."""
    rng = np.random.default_rng(seed)
    num_pages = num_slots // PAGE
    lens = np.concatenate([np.full(n_long, num_slots), rng.integers(len_lo, len_hi + 1, size=B - n_long)])
    idx = np.empty((B, 1, topk), dtype=np.int32)
    for b in range(B):
        table = rng.permutation(num_pages)[:(lens[b] + PAGE - 1) // PAGE]
        pos = rng.choice(int(lens[b]), size=topk, replace=False)
        idx[b, 0] = _positions_to_slots(table, pos)
    q = _normal_bf16(rng, (B, 1, h_q, D_QK))
    return DecodeWorkload(f"longctx_b{B}_sq1_h{h_q}_topk{topk}_R432", B, 1, h_q, topk, 432, num_slots,
                          1.0 / math.sqrt(D_QK), q, torch.from_numpy(idx), None, pool_seed=seed + 3000,
                          seq_lens=lens)


def sparse_prefill(seed: int = 0, B: int = 2, s_q: int = 256, h_q: int = 128, topk: int = 2048,
                   prefix: int = 16_384) -> DecodeWorkload:
    """Sparse prefill / extend: each of B requests has `prefix` cached tokens plus s_q new ones
    whose records are appended before attention; new token i (position prefix + i) attends to
    topk distinct positions drawn uniformly from 0..prefix + i (causal). Each request owns
    ceil((prefix + s_q) / 64) pages from a seeded permutation of the pool's pages."""
    rng = np.random.default_rng(seed)
    pages_per_req = (prefix + s_q + PAGE - 1) // PAGE
    num_pages = B * pages_per_req
    perm = rng.permutation(num_pages)
    idx = np.full((B, s_q, topk), -1, dtype=np.int32)
    for b in range(B):
        table = perm[b * pages_per_req:(b + 1) * pages_per_req]
        for i in range(s_q):
            visible = prefix + i + 1
            n = min(visible, topk)
            idx[b, i, :n] = _positions_to_slots(table, rng.choice(visible, size=n, replace=False))
    q = _normal_bf16(rng, (B, s_q, h_q, D_QK))
    return DecodeWorkload(f"prefill_b{B}_sq{s_q}_h{h_q}_topk{topk}_prefix{prefix}_R352", B, s_q, h_q, topk, 352,
                          num_pages * PAGE, 1.0 / math.sqrt(D_QK), q, torch.from_numpy(idx), None,
                          pool_seed=seed + 4000, seq_lens=np.full(B, prefix + s_q))


WORKLOADS = {
    "tiny": tiny_decode,
    "write": write_path,
    "decode": batch_decode,
    "varlen": varlen_decode,
    "longctx": long_context,
    "prefill": sparse_prefill,
}


def compact_for_rows(w: DecodeWorkload, rows: np.ndarray):
    """For the listed query rows, gather the distinct valid slots they reference and remap the
    indices to positions in that compact list. Out-of-range and negative entries become -1.
    Returns (slots int64 [n], q_rows bf16 [len(rows), h_q, 576], idx int32 [len(rows), topk])."""
    idx = w.indices.reshape(w.n_rows, w.topk).numpy()[rows]
    valid = (idx >= 0) & (idx < w.num_slots)
    uniq = np.unique(idx[valid]).astype(np.int64)
    remap = np.full(idx.shape, -1, dtype=np.int32)
    remap[valid] = np.searchsorted(uniq, idx[valid]).astype(np.int32)
    q = w.q.reshape(w.n_rows, w.h_q, D_QK)[torch.from_numpy(np.asarray(rows, dtype=np.int64))]
    return uniq, q, remap


def sample_rows(w: DecodeWorkload, n: int, seed: int = 123) -> np.ndarray:
    rng = np.random.default_rng(seed)
    n = min(n, w.n_rows)
    rows = np.sort(rng.choice(w.n_rows, size=n, replace=False))
    return rows
