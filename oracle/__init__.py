"""fp64 CPU oracle for paged decode attention (test infrastructure only).

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package. It loads ``liboracle.so`` built from
``oracle.c`` (plain C, no code shared with the CUDA library) and exposes numpy
wrappers. The allocator model in ``alloc_model.py`` is the oracle for the host
block allocator.

Passages followed (page title and section):
  * "vLLM 0.5 深度解析" §2.1 block table and ceil(n / block_size) blocks per
    request; §2.2 scale = head_dim ** -0.5; §2.3 block-by-block scaled dot
    product, softmax max/sum, V-weighted sum.
  * "vLLM 0.7.2深度解析" §2.1 shared physical blocks; §2.2 GQA and the FP8 e4m3
    KV cache; §2.3 sliding-window masking.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

from .build import build_oracle, LIB_PATH

F16, BF16, E4M3 = 0, 1, 2
_DT = {"f16": F16, "bf16": BF16, "fp8": E4M3, "e4m3": E4M3}

_lib = None


def lib() -> ctypes.CDLL:
    global _lib
    if _lib is None:
        build_oracle()
        L = ctypes.CDLL(LIB_PATH)
        c_i64, c_i32, c_int, c_dbl, c_flt, vp = (ctypes.c_int64, ctypes.c_int32, ctypes.c_int,
                                                  ctypes.c_double, ctypes.c_float, ctypes.c_void_p)
        L.orc_f16_to_f64.restype = c_dbl
        L.orc_f16_to_f64.argtypes = [ctypes.c_uint16]
        L.orc_bf16_to_f64.restype = c_dbl
        L.orc_bf16_to_f64.argtypes = [ctypes.c_uint16]
        L.orc_e4m3_to_f64.restype = c_dbl
        L.orc_e4m3_to_f64.argtypes = [ctypes.c_uint8]
        L.orc_e4m3_from_f32.restype = ctypes.c_uint8
        L.orc_e4m3_from_f32.argtypes = [c_flt]
        L.orc_decode16_array.argtypes = [vp, c_int, vp, c_i64]
        L.orc_e4m3_decode_array.argtypes = [vp, vp, c_i64]
        L.orc_e4m3_encode_array.argtypes = [vp, vp, c_i64]
        L.orc_reshape_and_cache.restype = c_int
        L.orc_reshape_and_cache.argtypes = [vp, vp, c_i64, c_i64, c_i64, c_int, vp, vp, c_i64,
                                            c_i64, c_int, vp, c_flt, c_flt, c_int]
        L.orc_decode.restype = c_int
        L.orc_decode.argtypes = [vp, vp, c_int, vp, vp, c_int, vp, vp, c_i64, c_i64, c_i64,
                                 c_i64, c_i64, c_i64, c_i64, c_dbl, c_i64, c_dbl, c_dbl, vp,
                                 c_i64, c_int]
        L.orc_decode_multi.restype = c_int
        L.orc_decode_multi.argtypes = [vp, vp, c_int, vp, vp, c_int, vp, vp, c_i64, c_i64, c_i64,
                                       c_i64, c_i64, c_i64, c_i64, c_i64, c_dbl, c_i64, c_dbl,
                                       c_dbl, vp, c_i64, c_int]
        _lib = L
    return _lib


def default_threads() -> int:
    return max(1, len(os.sched_getaffinity(0)))


def _ptr(a: np.ndarray) -> int:
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return a.ctypes.data


def _bits16(a) -> np.ndarray:
    """16-bit payload of a numpy float16/uint16 array or a CPU torch tensor."""
    if hasattr(a, "numpy"):  # torch tensor
        import torch
        a = a.detach().cpu().contiguous().view(torch.int16).numpy()
    a = np.ascontiguousarray(a)
    assert a.dtype.itemsize == 2
    return a.view(np.uint16)


def _bytes8(a) -> np.ndarray:
    if hasattr(a, "numpy"):
        import torch
        a = a.detach().cpu().contiguous().view(torch.uint8).numpy()
    a = np.ascontiguousarray(a)
    assert a.dtype.itemsize == 1
    return a.view(np.uint8)


# ------------------------------------------------------------------ codecs

def f16_to_f64(bits) -> np.ndarray:
    b = _bits16(bits)
    out = np.empty(b.shape, np.float64)
    lib().orc_decode16_array(_ptr(b), F16, _ptr(out), b.size)
    return out


def bf16_to_f64(bits) -> np.ndarray:
    b = _bits16(bits)
    out = np.empty(b.shape, np.float64)
    lib().orc_decode16_array(_ptr(b), BF16, _ptr(out), b.size)
    return out


def decode16(bits, dtype: str) -> np.ndarray:
    return f16_to_f64(bits) if _DT[dtype] == F16 else bf16_to_f64(bits)


def e4m3_to_f64(codes) -> np.ndarray:
    c = _bytes8(codes)
    out = np.empty(c.shape, np.float64)
    lib().orc_e4m3_decode_array(_ptr(c), _ptr(out), c.size)
    return out


def e4m3_from_f32(x) -> np.ndarray:
    x = np.ascontiguousarray(np.asarray(x, dtype=np.float32))
    out = np.empty(x.shape, np.uint8)
    lib().orc_e4m3_encode_array(_ptr(x), _ptr(out), x.size)
    return out


# -------------------------------------------------------------- write path

def reshape_and_cache(k, v, key_cache: np.ndarray, value_cache: np.ndarray,
                      slot_mapping, src_dtype: str, cache_dtype: str,
                      k_scale: float = 1.0, v_scale: float = 1.0, threads: int | None = None) -> None:
    """Scatter k/v [T, H, D] into the caches [NB, H, bs, D] in place.

    The caches are numpy arrays (uint16 for 16-bit caches, uint8 for e4m3).
    """
    kb, vb = _bits16(k), _bits16(v)
    T, H, D = kb.shape
    NB, H2, bs, D2 = key_cache.shape
    assert (H2, D2) == (H, D) and value_cache.shape == key_cache.shape
    slots = np.ascontiguousarray(np.asarray(slot_mapping, dtype=np.int64))
    assert slots.shape == (T,)
    rc = lib().orc_reshape_and_cache(_ptr(kb), _ptr(vb), T, H, D, _DT[src_dtype],
                                     _ptr(key_cache), _ptr(value_cache), NB, bs,
                                     _DT[cache_dtype], _ptr(slots), float(k_scale),
                                     float(v_scale), threads or default_threads())
    if rc != 0:
        raise ValueError(f"oracle reshape_and_cache failed: {rc}")


# ------------------------------------------------------------------ decode

def decode(q, key_cache, value_cache, block_tables, seq_lens, *, num_kv_heads: int,
           scale: float, block_size: int, window: int = 0, q_dtype: str,
           cache_dtype: str, k_scale: float = 1.0, v_scale: float = 1.0,
           pairs=None, threads: int | None = None) -> np.ndarray:
    """fp64 attention output [B, Hq, D]; rows not listed in ``pairs`` stay zero."""
    qb = _bits16(q)
    B, Hq, D = qb.shape
    if _DT[cache_dtype] == E4M3:
        kc, vc = _bytes8(key_cache), _bytes8(value_cache)
    else:
        kc, vc = _bits16(key_cache), _bits16(value_cache)
    NB, Hkv, bs, D2 = kc.shape
    assert Hkv == num_kv_heads and bs == block_size and D2 == D
    bt = np.ascontiguousarray(np.asarray(block_tables, dtype=np.int32))
    lens = np.ascontiguousarray(np.asarray(seq_lens, dtype=np.int32))
    assert bt.shape[0] == B and lens.shape == (B,)
    MB = bt.shape[1]
    out = np.zeros((B, Hq, D), np.float64)
    if pairs is not None:
        # distinct rows only: the C oracle runs listed rows on parallel threads,
        # and two threads must not write one output row
        pr = np.ascontiguousarray(np.unique(np.asarray(pairs, dtype=np.int32).reshape(-1, 2),
                                            axis=0))
        pp, npairs = _ptr(pr), pr.shape[0]
    else:
        pr, pp, npairs = None, None, 0
    rc = lib().orc_decode(_ptr(out), _ptr(qb), _DT[q_dtype], _ptr(kc), _ptr(vc),
                          _DT[cache_dtype], _ptr(bt) if bt.size else None, _ptr(lens), B, Hq,
                          Hkv, D, NB, bs, MB, float(scale), int(window), float(k_scale),
                          float(v_scale), pp, npairs, threads or default_threads())
    if rc != 0:
        raise ValueError(f"oracle decode failed: {rc}")
    return out


def decode_multi(q, key_cache, value_cache, block_tables, seq_lens, *, num_kv_heads: int,
                 scale: float, block_size: int, window: int = 0, q_dtype: str,
                 cache_dtype: str, k_scale: float = 1.0, v_scale: float = 1.0,
                 triples=None, threads: int | None = None) -> np.ndarray:
    """fp64 output [B, T, Hq, D] of T causal queries per sequence at its last T
    positions; rows not listed in ``triples`` (b, t, h) stay zero."""
    qb = _bits16(q)
    B, T, Hq, D = qb.shape
    if _DT[cache_dtype] == E4M3:
        kc, vc = _bytes8(key_cache), _bytes8(value_cache)
    else:
        kc, vc = _bits16(key_cache), _bits16(value_cache)
    NB, Hkv, bs, D2 = kc.shape
    assert Hkv == num_kv_heads and bs == block_size and D2 == D
    bt = np.ascontiguousarray(np.asarray(block_tables, dtype=np.int32))
    lens = np.ascontiguousarray(np.asarray(seq_lens, dtype=np.int32))
    MB = bt.shape[1]
    out = np.zeros((B, T, Hq, D), np.float64)
    if triples is not None:
        tr = np.ascontiguousarray(np.unique(np.asarray(triples, dtype=np.int32).reshape(-1, 3),
                                            axis=0))  # distinct rows, as for pairs
        tp, ntr = _ptr(tr), tr.shape[0]
    else:
        tr, tp, ntr = None, None, 0
    rc = lib().orc_decode_multi(_ptr(out), _ptr(qb), _DT[q_dtype], _ptr(kc), _ptr(vc),
                                _DT[cache_dtype], _ptr(bt) if bt.size else None, _ptr(lens), B,
                                T, Hq, Hkv, D, NB, bs, MB, float(scale), int(window),
                                float(k_scale), float(v_scale), tp, ntr,
                                threads or default_threads())
    if rc != 0:
        raise ValueError(f"oracle decode_multi failed: {rc}")
    return out
