"""GB300 paged-attention decode: Python binding of libpa (include/pa.h).

Argument marshalling only: every step of the path runs in the library's CUDA
kernels. PyTorch supplies device memory and the current stream. If libpa.so
has not been built, every call raises; there is no fallback.
"""
from __future__ import annotations

import ctypes
import os

import torch

from .build import LIB_PATH

PA_F16, PA_BF16, PA_FP8_E4M3, PA_I32, PA_I64 = 0, 1, 2, 3, 4
PA_KV_AUTO, PA_KV_FP8_E4M3 = 0, 2
DEVERR_BLOCK_ID, DEVERR_SEQ_LEN, DEVERR_SLOT, DEVERR_TIMEOUT = 1, 2, 4, 8
_MAX_DIMS = 6

_STATUS = {0: "PA_OK", -1: "PA_ERR_INVALID_ARG", -2: "PA_ERR_UNSUPPORTED", -3: "PA_ERR_LAYOUT",
           -4: "PA_ERR_CUDA", -5: "PA_ERR_OUT_OF_BLOCKS", -6: "PA_ERR_WORKSPACE",
           -7: "PA_ERR_NOT_FOUND", -8: "PA_ERR_HOST_MEMORY"}


class PAError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"{_STATUS.get(status, status)}: {msg}")
        self.status = status


class OutOfBlocks(PAError):
    pass


class PaTensor(ctypes.Structure):
    _fields_ = [("data", ctypes.c_void_p), ("dtype", ctypes.c_int32), ("ndim", ctypes.c_int32),
                ("shape", ctypes.c_int64 * _MAX_DIMS), ("strides", ctypes.c_int64 * _MAX_DIMS)]


_lib_handle = None


def lib() -> ctypes.CDLL:
    """The loaded libpa.so; raises if it was never built."""
    global _lib_handle
    if _lib_handle is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                               "`python -c 'import __graft_entry__ as g; g.build()'`")
        L = ctypes.CDLL(LIB_PATH)
        P = ctypes.POINTER(PaTensor)
        i32, i64, f32, vp, st = (ctypes.c_int32, ctypes.c_int64, ctypes.c_float, ctypes.c_void_p,
                                 ctypes.c_int32)
        sig = {
            "pa_reshape_and_cache": (st, [P, P, P, P, P, i32, f32, f32, vp]),
            "pa_decode": (st, [P, P, P, P, P, P, i32, f32, i32, i32, i32, f32, f32, vp]),
            "pa_decode_noalloc": (st, [P, P, P, P, P, P, i32, f32, i32, i32, i32, f32, f32, vp]),
            "pa_decode_workspace_size": (st, [i64, i32, i32, i32, ctypes.POINTER(ctypes.c_size_t)]),
            "pa_prefill_chunk": (st, [P, P, P, P, P, P, i32, f32, i32, i32, i32, f32, f32, vp]),
            "pa_prefill_chunk_workspace_size": (st, [i64, i32, i32, i32, i32,
                                                     ctypes.POINTER(ctypes.c_size_t)]),
            "pa_set_workspace": (st, [vp, ctypes.c_size_t]),
            "pa_set_decode_tuning": (st, [i32, i32, i32, i32]),
            "pa_set_prefill_path": (st, [i32]),
            "pa_profile_events": (st, [vp, vp]),
            "pa_check_device_error": (st, [ctypes.POINTER(i32), vp]),
            "pa_selftest_bounded_wait": (st, [ctypes.c_uint32, vp, vp]),
            "pa_launch_count": (ctypes.c_uint64, []),
            "pa_last_error": (ctypes.c_char_p, []),
            "pa_version": (i32, []),
            "pa_alloc_create": (st, [i32, i32, ctypes.c_uint64, ctypes.POINTER(vp)]),
            "pa_alloc_destroy": (None, [vp]),
            "pa_alloc_add": (st, [vp, i64, ctypes.POINTER(i32)]),
            "pa_alloc_fork": (st, [vp, i32, ctypes.POINTER(i32)]),
            "pa_alloc_add_cached": (st, [vp, vp, i64, ctypes.POINTER(i32), ctypes.POINTER(i64)]),
            "pa_alloc_append": (st, [vp, i32, i64, ctypes.POINTER(i32), ctypes.POINTER(i32)]),
            "pa_alloc_free": (st, [vp, i32]),
            "pa_alloc_trim_window": (st, [vp, i32, i32, ctypes.POINTER(i32)]),
            "pa_alloc_reclaim": (i32, [vp]),
            "pa_alloc_block_table": (st, [vp, i32, vp, i32, ctypes.POINTER(i32)]),
            "pa_alloc_seq_len": (st, [vp, i32, ctypes.POINTER(i64)]),
            "pa_alloc_fill_tables": (st, [vp, vp, i32, vp, i32, vp]),
            "pa_alloc_refcount": (i32, [vp, i32]),
            "pa_alloc_num_free": (i32, [vp]),
            "pa_alloc_num_pending": (i32, [vp]),
        }
        for name, (res, args) in sig.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib_handle = L
    return _lib_handle


def last_error() -> str:
    return lib().pa_last_error().decode()


def _check(status: int) -> None:
    if status != 0:
        msg = last_error()
        if status == -5:
            raise OutOfBlocks(status, msg)
        raise PAError(status, msg)


_TORCH_TO_PA = {torch.float16: PA_F16, torch.bfloat16: PA_BF16, torch.uint8: PA_FP8_E4M3,
                torch.float8_e4m3fn: PA_FP8_E4M3, torch.int32: PA_I32, torch.int64: PA_I64}


def tensor_desc(t: torch.Tensor) -> PaTensor:
    """pa_tensor describing a torch tensor (no copy)."""
    if t.dtype not in _TORCH_TO_PA:
        raise TypeError(f"unsupported dtype {t.dtype}")
    if t.dim() > _MAX_DIMS:
        raise ValueError("too many dims")
    d = PaTensor()
    d.data = t.data_ptr() if t.numel() > 0 else (t.data_ptr() or None)
    d.dtype = _TORCH_TO_PA[t.dtype]
    d.ndim = t.dim()
    for i, (s, st) in enumerate(zip(t.shape, t.stride())):
        d.shape[i] = s
        d.strides[i] = st
    return d


def _stream(stream) -> int | None:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _kv(kv_dtype) -> int:
    if kv_dtype in ("auto", None, PA_KV_AUTO):
        return PA_KV_AUTO
    if kv_dtype in ("fp8", "fp8_e4m3", "e4m3", PA_KV_FP8_E4M3):
        return PA_KV_FP8_E4M3
    raise ValueError(f"bad kv_dtype {kv_dtype!r}")


# ---------------------------------------------------------------- hot path

def reshape_and_cache(k, v, key_cache, value_cache, slot_mapping, kv_dtype="auto",
                      k_scale: float = 1.0, v_scale: float = 1.0, stream=None) -> None:
    """Scatter k/v [T, Hkv, D] into the caches [NB, Hkv, bs, D] at slot_mapping [T]."""
    descs = [tensor_desc(x) for x in (k, v, key_cache, value_cache, slot_mapping)]
    _check(lib().pa_reshape_and_cache(*[ctypes.byref(d) for d in descs], _kv(kv_dtype),
                                      float(k_scale), float(v_scale), _stream(stream)))


def decode(q, key_cache, value_cache, block_tables, seq_lens, *, num_kv_heads: int,
           scale: float, block_size: int, window: int = 0, kv_dtype="auto",
           k_scale: float = 1.0, v_scale: float = 1.0, out=None, stream=None):
    """One paged decode step; returns out [B, Hq, D] (allocated if not given)."""
    if out is None:
        out = torch.empty_like(q)
    descs = [tensor_desc(x) for x in (out, q, key_cache, value_cache, block_tables, seq_lens)]
    _check(lib().pa_decode(*[ctypes.byref(d) for d in descs], int(num_kv_heads), float(scale),
                           int(block_size), int(window), _kv(kv_dtype), float(k_scale),
                           float(v_scale), _stream(stream)))
    return out


def prefill_chunk(q, key_cache, value_cache, block_tables, seq_lens, *, num_kv_heads: int,
                  scale: float, block_size: int, window: int = 0, kv_dtype="auto",
                  k_scale: float = 1.0, v_scale: float = 1.0, out=None, stream=None):
    """Causal attention of T query tokens per sequence (q [B, T, Hq, D], at
    the last T positions of each sequence) over the paged cache; returns out
    [B, T, Hq, D] (allocated if not given)."""
    if out is None:
        out = torch.empty_like(q)
    descs = [tensor_desc(x) for x in (out, q, key_cache, value_cache, block_tables, seq_lens)]
    _check(lib().pa_prefill_chunk(*[ctypes.byref(d) for d in descs], int(num_kv_heads),
                                  float(scale), int(block_size), int(window), _kv(kv_dtype),
                                  float(k_scale), float(v_scale), _stream(stream)))
    return out


def decode_noalloc(q, key_cache, value_cache, block_tables, seq_lens, *, num_kv_heads: int,
                   scale: float, block_size: int, out, window: int = 0, kv_dtype="auto",
                   k_scale: float = 1.0, v_scale: float = 1.0, stream=None):
    """pa_decode_noalloc: the decode step with the library's built-in scratch
    array instead of a workspace, for callers that cannot allocate device
    memory at decode time. `out` must be given (nothing is allocated)."""
    descs = [tensor_desc(x) for x in (out, q, key_cache, value_cache, block_tables, seq_lens)]
    _check(lib().pa_decode_noalloc(*[ctypes.byref(d) for d in descs], int(num_kv_heads),
                                   float(scale), int(block_size), int(window), _kv(kv_dtype),
                                   float(k_scale), float(v_scale), _stream(stream)))
    return out


def workspace_size(batch: int, num_q_heads: int, num_kv_heads: int, head_dim: int) -> int:
    n = ctypes.c_size_t(0)
    _check(lib().pa_decode_workspace_size(batch, num_q_heads, num_kv_heads, head_dim,
                                          ctypes.byref(n)))
    return n.value


def prefill_chunk_workspace_size(batch: int, num_queries: int, num_q_heads: int,
                                 num_kv_heads: int, head_dim: int) -> int:
    n = ctypes.c_size_t(0)
    _check(lib().pa_prefill_chunk_workspace_size(batch, num_queries, num_q_heads, num_kv_heads,
                                                 head_dim, ctypes.byref(n)))
    return n.value


def set_workspace(buf: torch.Tensor | None) -> None:
    if buf is None:
        _check(lib().pa_set_workspace(None, 0))
    else:
        _check(lib().pa_set_workspace(buf.data_ptr(), buf.numel() * buf.element_size()))


def set_prefill_path(path: int = 0) -> None:
    """pa_prefill_chunk's kernel: 0 auto, 1 persistent split-KV kernel,
    2 tensor-memory kernel wherever it applies."""
    _check(lib().pa_set_prefill_path(path))


def set_decode_tuning(max_ctas: int = 0, min_tiles: int = 0, pool_permille: int = 0,
                      piece_tiles: int = 0) -> None:
    """0 keeps a default; pool_permille < 0 turns the dynamic pool off."""
    _check(lib().pa_set_decode_tuning(max_ctas, min_tiles, pool_permille, piece_tiles))


def profile_events(before=None, after=None) -> None:
    """Record torch.cuda.Event `before`/`after` around the main decode kernel."""
    for ev in (before, after):
        if ev is not None and not ev.cuda_event:
            ev.record()  # torch creates the CUDA event on its first record
    b = before.cuda_event if before is not None else None
    a = after.cuda_event if after is not None else None
    _check(lib().pa_profile_events(b, a))


def check_device_error(stream=None) -> int:
    bits = ctypes.c_int32(0)
    _check(lib().pa_check_device_error(ctypes.byref(bits), _stream(stream)))
    return bits.value


def selftest_bounded_wait(limit_us: int, elapsed=None, stream=None) -> None:
    """pa_selftest_bounded_wait: one CTA whose two waits cannot be satisfied;
    each gives up after `limit_us` and sets PA_DEVERR_TIMEOUT (read it with
    check_device_error). `elapsed`: None, or a contiguous int64 tensor of two
    elements on the device that receives each wait's duration in ns."""
    ptr = None
    if elapsed is not None:
        if elapsed.dtype != torch.int64 or elapsed.numel() != 2 or not elapsed.is_contiguous():
            raise ValueError("elapsed must be a contiguous int64 tensor of 2 elements")
        ptr = elapsed.data_ptr()
    _check(lib().pa_selftest_bounded_wait(limit_us, ptr, _stream(stream)))


def launch_count() -> int:
    return lib().pa_launch_count()


def version() -> int:
    return lib().pa_version()


# ------------------------------------------------------------- allocator

class BlockAllocator:
    """Host block pool (pa_alloc_*): seeded shuffled free list, ref-counted
    sharing, copy-on-write of a shared partial last block, deferred reclaim."""

    def __init__(self, num_blocks: int, block_size: int, seed: int = 0):
        h = ctypes.c_void_p()
        _check(lib().pa_alloc_create(num_blocks, block_size, seed, ctypes.byref(h)))
        self._h = h
        self.num_blocks, self.block_size = num_blocks, block_size

    def __del__(self):
        h = getattr(self, "_h", None)
        if h is not None and _lib_handle is not None:
            _lib_handle.pa_alloc_destroy(h)
            self._h = None

    def add(self, n_tokens: int) -> int:
        s = ctypes.c_int32()
        _check(lib().pa_alloc_add(self._h, n_tokens, ctypes.byref(s)))
        return s.value

    def add_cached(self, tokens) -> tuple[int, int]:
        """New sequence for token ids, reusing cached full blocks of its longest
        cached prefix; returns (sequence id, number of cached tokens)."""
        import numpy as np
        t = np.ascontiguousarray(np.asarray(tokens, dtype=np.int32))
        s, c = ctypes.c_int32(), ctypes.c_int64()
        _check(lib().pa_alloc_add_cached(self._h, t.ctypes.data if t.size else None, t.size,
                                         ctypes.byref(s), ctypes.byref(c)))
        return s.value, c.value

    def fork(self, src: int) -> int:
        s = ctypes.c_int32()
        _check(lib().pa_alloc_fork(self._h, src, ctypes.byref(s)))
        return s.value

    def append(self, seq: int, n_tokens: int) -> tuple[int, int]:
        a, b = ctypes.c_int32(), ctypes.c_int32()
        _check(lib().pa_alloc_append(self._h, seq, n_tokens, ctypes.byref(a), ctypes.byref(b)))
        return a.value, b.value

    def free(self, seq: int) -> None:
        _check(lib().pa_alloc_free(self._h, seq))

    def trim_window(self, seq: int, window: int) -> int:
        """Releases the blocks before the sliding window; returns how many."""
        n = ctypes.c_int32()
        _check(lib().pa_alloc_trim_window(self._h, seq, window, ctypes.byref(n)))
        return n.value

    def reclaim(self) -> int:
        return lib().pa_alloc_reclaim(self._h)

    def table(self, seq: int) -> list[int]:
        n = ctypes.c_int32()
        lib().pa_alloc_block_table(self._h, seq, None, 0, ctypes.byref(n))
        buf = (ctypes.c_int32 * max(n.value, 1))()
        _check(lib().pa_alloc_block_table(self._h, seq, buf, n.value, ctypes.byref(n)))
        return list(buf[:n.value])

    def seq_len(self, seq: int) -> int:
        n = ctypes.c_int64()
        _check(lib().pa_alloc_seq_len(self._h, seq, ctypes.byref(n)))
        return n.value

    def fill_tables(self, seqs, max_blocks: int):
        import numpy as np
        ids = np.ascontiguousarray(np.asarray(seqs, dtype=np.int32))
        tables = np.empty((len(ids), max_blocks), np.int32)
        lens = np.empty(len(ids), np.int32)
        _check(lib().pa_alloc_fill_tables(self._h, ids.ctypes.data, len(ids), tables.ctypes.data,
                                          max_blocks, lens.ctypes.data))
        return tables, lens

    def refcount(self, block: int) -> int:
        return lib().pa_alloc_refcount(self._h, block)

    def num_free(self) -> int:
        return lib().pa_alloc_num_free(self._h)

    def num_pending(self) -> int:
        return lib().pa_alloc_num_pending(self._h)
