"""CPU oracle for the NVFP4 MLA KV-cache codec and sparse MLA decode.

TEST INFRASTRUCTURE ONLY: imported by ``tests/``, by ``__graft_entry__.smoke()`` and by the
CPU-baseline leg of ``bench.py``; never by the library package. The arithmetic lives in
``nvfp4_oracle.c`` (plain C, fp64), compiled with gcc into ``oracle/_build/liboracle.so``;
this module only marshals numpy arrays into it. It shares nothing with the CUDA path.

Every function cites the page section it follows in ``nvfp4_oracle.c``. bf16 values cross
this boundary as their uint16 bit patterns.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from typing import Optional, Tuple

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "nvfp4_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "liboracle.so")
_lib = None

RECORD_BYTES = (352, 432, 656)


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (OpenMP when available). Returns the library path."""
    os.makedirs(_BUILD, exist_ok=True)
    if not force and os.path.exists(_LIB_PATH) and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    base = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fno-fast-math", "-ffp-contract=off"]
    try:
        subprocess.run(base + ["-fopenmp", _SRC, "-o", tmp, "-lm"], check=True, capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base + [_SRC, "-o", tmp, "-lm"], check=True, capture_output=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def lib() -> ctypes.CDLL:
    global _lib
    if _lib is None:
        _lib = ctypes.CDLL(build())
        P = ctypes.c_void_p
        i64 = ctypes.c_int64
        i32 = ctypes.c_int
        d = ctypes.c_double
        _lib.oracle_e4m3_decode.restype = d
        _lib.oracle_e4m3_decode.argtypes = [ctypes.c_uint8]
        _lib.oracle_e2m1_decode.restype = d
        _lib.oracle_e2m1_decode.argtypes = [ctypes.c_uint8]
        _lib.oracle_e4m3_encode.restype = ctypes.c_uint8
        _lib.oracle_e4m3_encode.argtypes = [ctypes.c_float]
        _lib.oracle_e2m1_encode.restype = ctypes.c_uint8
        _lib.oracle_e2m1_encode.argtypes = [ctypes.c_float]
        _lib.oracle_round_to_bf16.restype = d
        _lib.oracle_round_to_bf16.argtypes = [d]
        _lib.oracle_scale_offset.restype = i32
        _lib.oracle_scale_offset.argtypes = [i32, i32, i32]
        _lib.oracle_quantize_record.restype = None
        _lib.oracle_quantize_record.argtypes = [P, P, i32, i32, P]
        _lib.oracle_quantize_append.restype = i64
        _lib.oracle_quantize_append.argtypes = [P, i64, P, i64, P, i64, P, i64, i32, i32]
        _lib.oracle_dequant_records.restype = None
        _lib.oracle_dequant_records.argtypes = [P, i64, i32, i32, P]
        _lib.oracle_sparse_mla_decode.restype = None
        _lib.oracle_sparse_mla_decode.argtypes = [P, P, i64, i32, i32, P, i64, i64, i32, i32, d, P, P, i64, P, P, i32]
        _lib.oracle_merge_partials.restype = None
        _lib.oracle_merge_partials.argtypes = [i32, P, P, P, P, P]
        for name, intype, outtype in (("oracle_e4m3_encode_many", P, P), ("oracle_e2m1_encode_many", P, P),
                                      ("oracle_e4m3_decode_many", P, P)):
            fn = getattr(_lib, name)
            fn.restype = None
            fn.argtypes = [intype, i64, outtype]
        _lib.oracle_norm_rope.restype = None
        _lib.oracle_norm_rope.argtypes = [P, i64, P, i64, P, i64, P, d, P, P, i64, i32, P, P, P, P, P, P]
        _lib.oracle_threads_available.restype = i32
        _lib.oracle_threads_available.argtypes = []
    return _lib


def _ptr(a: Optional[np.ndarray]):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a: np.ndarray, dtype) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=dtype)


def threads_available() -> int:
    return int(lib().oracle_threads_available())


# ---- single-value codec --------------------------------------------------------------

def e4m3_decode(codes) -> np.ndarray:
    c = _c(np.asarray(codes, dtype=np.uint8).reshape(-1), np.uint8)
    out = np.empty(c.size, dtype=np.float64)
    lib().oracle_e4m3_decode_many(_ptr(c), c.size, _ptr(out))
    return out.reshape(np.shape(codes))


def e4m3_encode(values) -> np.ndarray:
    f = _c(np.asarray(values, dtype=np.float32).reshape(-1), np.float32)
    out = np.empty(f.size, dtype=np.uint8)
    lib().oracle_e4m3_encode_many(_ptr(f), f.size, _ptr(out))
    return out.reshape(np.shape(values))


def e2m1_encode(values) -> np.ndarray:
    f = _c(np.asarray(values, dtype=np.float32).reshape(-1), np.float32)
    out = np.empty(f.size, dtype=np.uint8)
    lib().oracle_e2m1_encode_many(_ptr(f), f.size, _ptr(out))
    return out.reshape(np.shape(values))


def e2m1_decode(nibble: int) -> float:
    return float(lib().oracle_e2m1_decode(int(nibble)))


def _block_flag(record_bytes: int, block_scales: bool) -> int:
    # the 432-byte record keeps its scales in block order by definition
    assert not (block_scales and record_bytes != 352), "block_scales applies to the 352-byte record"
    return 1 if block_scales else 0


def round_to_bf16(x: float) -> float:
    """Nearest bf16 value of a finite double, ties to even."""
    return float(lib().oracle_round_to_bf16(float(x)))


def scale_offset(record_bytes: int, g: int, block_scales: bool = False) -> int:
    """Byte offset of 16-value block g's e4m3 scale in an NVFP4 record. ``block_scales``: the
    352-byte record with its scales in block order (the unpermuted side of the scale-layout
    comparison)."""
    assert record_bytes in (352, 432)
    return int(lib().oracle_scale_offset(int(record_bytes), _block_flag(record_bytes, block_scales), int(g)))


# ---- write side -----------------------------------------------------------------------

def quantize_records(latent_bits: np.ndarray, rope_bits: np.ndarray, record_bytes: int,
                     block_scales: bool = False) -> np.ndarray:
    """bf16 bits [T,512] and [T,64] -> records uint8 [T, record_bytes]."""
    assert record_bytes in RECORD_BYTES
    blk = _block_flag(record_bytes, block_scales)
    lat = _c(latent_bits, np.uint16)
    rope = _c(rope_bits, np.uint16)
    T = lat.shape[0]
    assert lat.shape == (T, 512) and rope.shape == (T, 64)
    out = np.zeros((T, record_bytes), dtype=np.uint8)
    L = lib()
    for t in range(T):
        L.oracle_quantize_record(_ptr(lat[t]), _ptr(rope[t]), record_bytes, blk, _ptr(out[t]))
    return out


def quantize_append(latent_bits: np.ndarray, rope_bits: np.ndarray, slot_mapping: np.ndarray,
                    cache: np.ndarray, block_scales: bool = False) -> int:
    """In-place write into ``cache`` (uint8 [num_slots, record_bytes]). Rows of ``latent_bits``
    and ``rope_bits`` may be strided views (element strides, inner stride 1). Returns the
    count of slots >= num_slots (skipped)."""
    assert cache.dtype == np.uint8 and cache.flags.c_contiguous and cache.ndim == 2
    record_bytes = cache.shape[1]
    assert record_bytes in RECORD_BYTES
    assert latent_bits.dtype == np.uint16 and rope_bits.dtype == np.uint16
    assert latent_bits.strides[1] == 2 and rope_bits.strides[1] == 2
    slots = _c(slot_mapping, np.int64)
    T = slots.size
    return int(lib().oracle_quantize_append(
        _ptr(latent_bits), latent_bits.strides[0] // 2, _ptr(rope_bits), rope_bits.strides[0] // 2,
        _ptr(slots), T, _ptr(cache), cache.shape[0], record_bytes, _block_flag(record_bytes, block_scales)))


def norm_rope(latent_bits: np.ndarray, rope_bits: np.ndarray, positions: np.ndarray, weight_bits: np.ndarray,
              eps: float, cos_table: np.ndarray, sin_table: np.ndarray, rotate_half: bool) -> dict:
    """The stage ahead of the append (RMSNorm of the latent, rotary embedding of k_pe), see
    oracle_norm_rope. latent bf16 bits [T,512], k_pe [T,64] (strided rows allowed), positions
    int64 [T], weight bf16 bits [512], cos/sin fp32 [num_positions, 32]. Returns a dict:
    ``latent`` [T,512] and ``rope`` [T,64] bf16 bits, ``exact`` fp64 [T,576], ``flag`` and
    ``other`` [T,576] (the other admissible bf16 rounding where flagged), ``valid`` [T]."""
    assert latent_bits.dtype == np.uint16 and rope_bits.dtype == np.uint16
    assert latent_bits.strides[1] == 2 and rope_bits.strides[1] == 2
    pos = _c(positions, np.int64)
    T = pos.size
    w = _c(weight_bits, np.uint16)
    cs, sn = _c(cos_table, np.float32), _c(sin_table, np.float32)
    assert w.size == 512 and cs.shape == sn.shape and cs.shape[1] == 32
    res = {"latent": np.zeros((T, 512), np.uint16), "rope": np.zeros((T, 64), np.uint16),
           "exact": np.zeros((T, 576), np.float64), "flag": np.zeros((T, 576), np.uint8),
           "other": np.zeros((T, 576), np.uint16), "valid": np.zeros(T, np.uint8)}
    lib().oracle_norm_rope(_ptr(latent_bits), latent_bits.strides[0] // 2, _ptr(rope_bits), rope_bits.strides[0] // 2,
                           _ptr(pos), T, _ptr(w), float(eps), _ptr(cs), _ptr(sn), cs.shape[0], int(bool(rotate_half)),
                           _ptr(res["latent"]), _ptr(res["rope"]), _ptr(res["exact"]), _ptr(res["flag"]),
                           _ptr(res["other"]), _ptr(res["valid"]))
    return res


def dequant_records(records: np.ndarray, block_scales: bool = False) -> np.ndarray:
    """records uint8 [n, R] -> fp64 [n, 576] (K; V is K[:, :512])."""
    recs = _c(records, np.uint8)
    n, R = recs.shape
    out = np.empty((n, 576), dtype=np.float64)
    lib().oracle_dequant_records(_ptr(recs), n, R, _block_flag(R, block_scales), _ptr(out))
    return out


# ---- read side ------------------------------------------------------------------------

def sparse_mla_decode(q_bits: np.ndarray, cache: np.ndarray, indices: np.ndarray, sm_scale: float,
                      attn_sink: Optional[np.ndarray] = None, rows: Optional[np.ndarray] = None,
                      threads: int = 0, block_scales: bool = False) -> Tuple[np.ndarray, np.ndarray]:
    """q bf16 bits [n_tok, h_q, 576] (any leading shape flattened), cache uint8 [N, R],
    indices int32 [n_tok, topk]. Returns fp64 out [n_rows, h_q, 512] and lse [n_rows, h_q]
    for the query rows listed in ``rows`` (all rows when None)."""
    q = _c(q_bits, np.uint16)
    h_q = q.shape[-2]
    q = q.reshape(-1, h_q, 576)
    n_tok = q.shape[0]
    idx = _c(indices, np.int32).reshape(n_tok, -1)
    topk = idx.shape[1]
    cache = _c(cache, np.uint8)
    sink = None if attn_sink is None else _c(attn_sink, np.float32)
    assert sink is None or sink.size == h_q
    tok = None if rows is None else _c(rows, np.int64)
    n_rows = n_tok if tok is None else tok.size
    out = np.empty((n_rows, h_q, 512), dtype=np.float64)
    lse = np.empty((n_rows, h_q), dtype=np.float64)
    lib().oracle_sparse_mla_decode(_ptr(q), _ptr(cache), cache.shape[0], cache.shape[1],
                                   _block_flag(cache.shape[1], block_scales), _ptr(idx), topk,
                                   n_tok, h_q, topk, float(sm_scale), _ptr(sink), _ptr(tok),
                                   0 if tok is None else tok.size, _ptr(out), _ptr(lse), int(threads))
    return out, lse


def merge_partials(lse_p: np.ndarray, out_p: np.ndarray, sink: Optional[float] = None) -> Tuple[np.ndarray, float]:
    """Merge P partials of one (row, head): lse_p [P], out_p [P, 512]."""
    l = _c(lse_p, np.float64)
    o = _c(out_p, np.float64)
    P = l.size
    s = None if sink is None else np.array([sink], dtype=np.float64)
    out = np.empty(512, dtype=np.float64)
    lse = np.empty(1, dtype=np.float64)
    lib().oracle_merge_partials(P, _ptr(l), _ptr(o), _ptr(s), _ptr(out), _ptr(lse))
    return out, float(lse[0])
