"""Python binding of the NVFP4 MLA KV-cache library (``include/nvfp4_mla.h``).

Argument marshalling only: every step of the computation runs in the CUDA library
``_build/libnvfp4mla.so`` (built by ``build.py``). PyTorch provides device memory and the
current stream. There is no fallback: if the library is missing or the device is not
sm_103, the calls raise.
"""
from __future__ import annotations

import ctypes
import functools
import os
from typing import Optional, Tuple

import torch

from . import build as _build

RECORD_BYTES = (352, 432, 656)
# OR-ed into record_bytes: a 352-byte record whose scales are stored in block order (the
# unpermuted side of the scale-layout comparison); the cache is still [N, 352]
SCALES_BLOCK_ORDER = 0x10000
# size of the library-owned scratch of nvfp4_sparse_mla_decode_no_alloc
NO_ALLOC_SCRATCH_BYTES = 32 << 20
D_NOPE, D_ROPE, D_QK, D_V = 512, 64, 576, 512

OK = 0
ERR_INVALID_ARG = 1
ERR_UNSUPPORTED = 2
ERR_CUDA = 3
ERR_WORKSPACE = 4
DEV_SLOT_OUT_OF_RANGE = 0x1
DEV_INDEX_OUT_OF_RANGE = 0x2
DEV_TIMEOUT = 0x4
DEV_FP8_RANGE = 0x8
DEV_POSITION_OUT_OF_RANGE = 0x10

EXPORTED = (
    "nvfp4_mla_quantize_append",
    "nvfp4_mla_norm_rope_quantize_append",
    "nvfp4_sparse_mla_decode_workspace_size",
    "nvfp4_sparse_mla_decode_plan",
    "nvfp4_sparse_mla_decode",
    "nvfp4_sparse_mla_decode_no_alloc",
    "nvfp4_mla_status_string",
    "nvfp4_mla_version",
    "nvfp4_mla_selftest_wait_timeout",
)

_lib: Optional[ctypes.CDLL] = None


class Nvfp4MlaError(RuntimeError):
    def __init__(self, call: str, status: int):
        self.status = status
        super().__init__(f"{call} failed with status {status}: {status_string(status)}")


def library_path() -> str:
    return _build.LIB


def load(build_if_missing: bool = False) -> ctypes.CDLL:
    """Load the in-tree library (raises if it is absent and build_if_missing is False)."""
    global _lib
    if _lib is not None:
        return _lib
    path = _build.LIB
    if not os.path.exists(path):
        if not build_if_missing:
            raise ImportError(f"CUDA library not built: {path} (run __graft_entry__.build())")
        _build.build()
    lib = ctypes.CDLL(path)
    P, i64, i32, f32, sz = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_float, ctypes.c_size_t
    lib.nvfp4_mla_quantize_append.restype = ctypes.c_int
    lib.nvfp4_mla_quantize_append.argtypes = [P, i64, P, i64, P, i64, P, i64, i32, P, P]
    lib.nvfp4_mla_norm_rope_quantize_append.restype = ctypes.c_int
    lib.nvfp4_mla_norm_rope_quantize_append.argtypes = [P, i64, P, f32, P, i64, P, P, P, i64, i32, P, i64, P, i64, i32,
                                                        P, P]
    lib.nvfp4_sparse_mla_decode_workspace_size.restype = ctypes.c_int
    lib.nvfp4_sparse_mla_decode_workspace_size.argtypes = [i32, i32, i32, i32, i32, i32, ctypes.POINTER(sz)]
    lib.nvfp4_sparse_mla_decode_plan.restype = ctypes.c_int
    lib.nvfp4_sparse_mla_decode_plan.argtypes = [i32, i32, i32, i32, i32, i32, ctypes.POINTER(i32), ctypes.POINTER(i32)]
    lib.nvfp4_sparse_mla_decode.restype = ctypes.c_int
    lib.nvfp4_sparse_mla_decode.argtypes = [P, P, i64, i32, P, i32, i32, i32, i32, f32, P, P, P, i32, P, sz, P, P]
    lib.nvfp4_sparse_mla_decode_no_alloc.restype = ctypes.c_int
    lib.nvfp4_sparse_mla_decode_no_alloc.argtypes = [P, P, i64, i32, P, i32, i32, i32, i32, f32, P, P, P, i32, P, P]
    lib.nvfp4_mla_status_string.restype = ctypes.c_char_p
    lib.nvfp4_mla_status_string.argtypes = [ctypes.c_int]
    lib.nvfp4_mla_version.restype = ctypes.c_int
    lib.nvfp4_mla_version.argtypes = []
    lib.nvfp4_mla_selftest_wait_timeout.restype = ctypes.c_int
    lib.nvfp4_mla_selftest_wait_timeout.argtypes = [P, P, P]
    _lib = lib
    return lib


def status_string(status: int) -> str:
    return load().nvfp4_mla_status_string(int(status)).decode()


# Pointers and streams go to the C calls as plain integers (their argtypes are c_void_p); None is NULL.
def _ptr(t: Optional[torch.Tensor]) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _stream(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream


def _check(call: str, status: int):
    if status != OK:
        raise Nvfp4MlaError(call, status)


def _need(cond: bool, msg: str):
    if not cond:
        raise ValueError(msg)


def _record_code(cache: torch.Tensor, block_scales: bool) -> int:
    _need(not block_scales or cache.shape[1] == 352, "block_scales applies to 352-byte records")
    return cache.shape[1] | (SCALES_BLOCK_ORDER if block_scales else 0)


def quantize_append(kv_latent: torch.Tensor, k_rope: torch.Tensor, slot_mapping: torch.Tensor,
                    cache: torch.Tensor, dev_status: Optional[torch.Tensor] = None, stream=None,
                    block_scales: bool = False) -> None:
    """Quantize ``kv_latent`` (bf16 [T,512]) and ``k_rope`` (bf16 [T,64]) into records and
    write them to ``cache`` (uint8 [num_slots, 352|432|656]) at ``slot_mapping`` (int64 [T]).
    ``block_scales``: write 352-byte records with their scales in block order."""
    _need(kv_latent.dtype == torch.bfloat16 and k_rope.dtype == torch.bfloat16, "inputs must be bf16")
    _need(kv_latent.dim() == 2 and kv_latent.shape[1] == D_NOPE and kv_latent.stride(1) == 1, "kv_latent [T,512], inner stride 1")
    _need(k_rope.dim() == 2 and k_rope.shape[1] == D_ROPE and k_rope.stride(1) == 1, "k_rope [T,64], inner stride 1")
    T = kv_latent.shape[0]
    _need(k_rope.shape[0] == T and slot_mapping.numel() == T, "token counts differ")
    _need(slot_mapping.dtype == torch.int64 and slot_mapping.is_contiguous(), "slot_mapping int64 contiguous")
    _need(cache.dtype == torch.uint8 and cache.dim() == 2 and cache.is_contiguous(), "cache uint8 [num_slots, R] contiguous")
    _need(cache.shape[1] in RECORD_BYTES, "record width must be 352, 432 or 656")
    code = _record_code(cache, block_scales)
    dev = cache.get_device()   # -1 for a CPU tensor
    _need(dev >= 0 and all(t.get_device() == dev for t in (kv_latent, k_rope, slot_mapping)),
          "all tensors on the same CUDA device")
    st = load().nvfp4_mla_quantize_append(
        _ptr(kv_latent), kv_latent.stride(0), _ptr(k_rope), k_rope.stride(0), _ptr(slot_mapping), T,
        _ptr(cache), cache.shape[0], code, _ptr(dev_status), _stream(stream))
    _check("nvfp4_mla_quantize_append", st)


def norm_rope_quantize_append(kv_latent: torch.Tensor, norm_weight: torch.Tensor, eps: float, k_pe: torch.Tensor,
                              positions: torch.Tensor, cos_table: torch.Tensor, sin_table: torch.Tensor,
                              rotate_half: bool, slot_mapping: torch.Tensor, cache: torch.Tensor,
                              dev_status: Optional[torch.Tensor] = None, stream=None,
                              block_scales: bool = False) -> None:
    """RMSNorm ``kv_latent`` (bf16 [T,512], pre-norm) with ``norm_weight`` (bf16 [512]) and
    ``eps``, rotate ``k_pe`` (bf16 [T,64], pre-rotation) by ``positions`` (int64 [T]) with
    ``cos_table`` / ``sin_table`` (fp32 [P,32]), pairs (f, f+32) when ``rotate_half`` else
    (2f, 2f+1); then quantize and write the records as quantize_append does, in one kernel."""
    _need(kv_latent.dtype == torch.bfloat16 and k_pe.dtype == torch.bfloat16, "inputs must be bf16")
    _need(kv_latent.dim() == 2 and kv_latent.shape[1] == D_NOPE and kv_latent.stride(1) == 1, "kv_latent [T,512], inner stride 1")
    _need(k_pe.dim() == 2 and k_pe.shape[1] == D_ROPE and k_pe.stride(1) == 1, "k_pe [T,64], inner stride 1")
    T = kv_latent.shape[0]
    _need(k_pe.shape[0] == T and slot_mapping.numel() == T and positions.numel() == T, "token counts differ")
    _need(norm_weight.dtype == torch.bfloat16 and norm_weight.numel() == D_NOPE and norm_weight.is_contiguous(),
          "norm_weight bf16 [512] contiguous")
    _need(positions.dtype == torch.int64 and positions.is_contiguous(), "positions int64 contiguous")
    _need(cos_table.dtype == torch.float32 and sin_table.dtype == torch.float32 and cos_table.dim() == 2
          and cos_table.shape[1] == 32 and cos_table.shape == sin_table.shape and cos_table.is_contiguous()
          and sin_table.is_contiguous(), "cos_table / sin_table fp32 [P,32] contiguous")
    _need(slot_mapping.dtype == torch.int64 and slot_mapping.is_contiguous(), "slot_mapping int64 contiguous")
    _need(cache.dtype == torch.uint8 and cache.dim() == 2 and cache.is_contiguous(), "cache uint8 [num_slots, R] contiguous")
    _need(cache.shape[1] in RECORD_BYTES, "record width must be 352, 432 or 656")
    code = _record_code(cache, block_scales)
    for t in (kv_latent, norm_weight, k_pe, positions, cos_table, sin_table, slot_mapping, cache):
        _need(t.is_cuda and t.device == cache.device, "all tensors on the same CUDA device")
    st = load().nvfp4_mla_norm_rope_quantize_append(
        _ptr(kv_latent), kv_latent.stride(0), _ptr(norm_weight), ctypes.c_float(eps), _ptr(k_pe), k_pe.stride(0),
        _ptr(positions), _ptr(cos_table), _ptr(sin_table), cos_table.shape[0], int(bool(rotate_half)),
        _ptr(slot_mapping), T, _ptr(cache), cache.shape[0], code, _ptr(dev_status), _stream(stream))
    _check("nvfp4_mla_norm_rope_quantize_append", st)


@functools.lru_cache(maxsize=256)
def _workspace_size_on(device: int, batch: int, s_q: int, h_q: int, topk: int, record_bytes: int,
                       num_splits: int) -> int:
    """workspace_size for the given device (the automatic split count depends on its SM count)."""
    with torch.cuda.device(device):
        return workspace_size(batch, s_q, h_q, topk, record_bytes, num_splits)


def workspace_size(batch: int, s_q: int, h_q: int, topk: int, record_bytes: int, num_splits: int = 0) -> int:
    n = ctypes.c_size_t(0)
    st = load().nvfp4_sparse_mla_decode_workspace_size(batch, s_q, h_q, topk, record_bytes, num_splits, ctypes.byref(n))
    _check("nvfp4_sparse_mla_decode_workspace_size", st)
    return int(n.value)


def decode_plan(batch: int, s_q: int, h_q: int, topk: int, record_bytes: int, num_splits: int = 0):
    """(splits, kernels per call) of a decode of this shape on the current device."""
    sp, k = ctypes.c_int32(0), ctypes.c_int32(0)
    st = load().nvfp4_sparse_mla_decode_plan(batch, s_q, h_q, topk, record_bytes, num_splits, ctypes.byref(sp),
                                             ctypes.byref(k))
    _check("nvfp4_sparse_mla_decode_plan", st)
    return int(sp.value), int(k.value)


def sparse_mla_decode(q: torch.Tensor, cache: torch.Tensor, indices: torch.Tensor, sm_scale: float,
                      attn_sink: Optional[torch.Tensor] = None, out: Optional[torch.Tensor] = None,
                      lse: Optional[torch.Tensor] = None, num_splits: int = 0,
                      workspace: Optional[torch.Tensor] = None, dev_status: Optional[torch.Tensor] = None,
                      stream=None, block_scales: bool = False) -> Tuple[torch.Tensor, torch.Tensor]:
    """q bf16 [B, s_q, h_q, 576], cache uint8 [N, 352|432|656], indices int32 [B, s_q, topk].
    Returns (out bf16 [B, s_q, h_q, 512], lse fp32 [B, s_q, h_q]). ``block_scales``: the cache
    holds 352-byte records with their scales in block order."""
    _need(q.dtype == torch.bfloat16 and q.dim() == 4 and q.shape[3] == D_QK and q.is_contiguous(), "q bf16 [B,s_q,h_q,576] contiguous")
    B, s_q, h_q, _ = q.shape
    _need(indices.dtype == torch.int32 and indices.dim() == 3 and tuple(indices.shape[:2]) == (B, s_q)
          and indices.is_contiguous(), "indices int32 [B,s_q,topk] contiguous")
    topk = indices.shape[2]
    _need(cache.dtype == torch.uint8 and cache.dim() == 2 and cache.is_contiguous() and cache.shape[1] in RECORD_BYTES,
          "cache uint8 [N, 352|432|656] contiguous")
    code = _record_code(cache, block_scales)
    if attn_sink is not None:
        _need(attn_sink.dtype == torch.float32 and attn_sink.numel() == h_q and attn_sink.is_contiguous(), "attn_sink fp32 [h_q]")
    if out is None:
        out = torch.empty((B, s_q, h_q, D_V), dtype=torch.bfloat16, device=q.device)
    if lse is None:
        lse = torch.empty((B, s_q, h_q), dtype=torch.float32, device=q.device)
    _need(out.dtype == torch.bfloat16 and out.is_contiguous() and tuple(out.shape) == (B, s_q, h_q, D_V), "out bf16 [B,s_q,h_q,512]")
    _need(lse.dtype == torch.float32 and lse.is_contiguous() and tuple(lse.shape) == (B, s_q, h_q), "lse fp32 [B,s_q,h_q]")
    dev = q.get_device()   # -1 for a CPU tensor
    _need(dev >= 0 and all(t.get_device() == dev for t in (cache, indices, out, lse)) and
          (attn_sink is None or attn_sink.get_device() == dev), "all tensors on the same CUDA device")
    need = _workspace_size_on(dev, B, s_q, h_q, topk, code, num_splits)
    if need and (workspace is None or workspace.numel() * workspace.element_size() < need):
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    wbytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    st = load().nvfp4_sparse_mla_decode(
        _ptr(q), _ptr(cache), cache.shape[0], code, _ptr(indices), B, s_q, h_q, topk, float(sm_scale),
        _ptr(attn_sink), _ptr(out), _ptr(lse), int(num_splits), _ptr(workspace), wbytes, _ptr(dev_status),
        _stream(stream))
    _check("nvfp4_sparse_mla_decode", st)
    return out, lse


def selftest_wait_timeout(device=None, stream=None) -> Tuple[int, int]:
    """Runs one of the decode's time-bounded pipeline waits on an mbarrier that nothing arrives
    on. Returns (device status bits, nanoseconds the wait lasted); the status should hold
    DEV_TIMEOUT and the time be about one second."""
    device = torch.device("cuda") if device is None else torch.device(device)
    status = torch.zeros(1, dtype=torch.int32, device=device)
    elapsed = torch.zeros(1, dtype=torch.int64, device=device)
    _check("nvfp4_mla_selftest_wait_timeout",
           load().nvfp4_mla_selftest_wait_timeout(_ptr(status), _ptr(elapsed), _stream(stream)))
    torch.cuda.synchronize(device)
    return int(status.item()), int(elapsed.item())
