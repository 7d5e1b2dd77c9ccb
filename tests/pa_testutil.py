"""Shared helpers for the GPU parity tests.

The product side runs the library's kernels; the oracle side runs the fp64 C
oracle on host copies of the generator's inputs, taken before the product
writes anything, so no oracle input ever comes from the CUDA path.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np
import torch

import oracle
import paged_kv_cache_267_gb300 as pa
from workloads import generate
from workloads.gen import E4M3_NAN

MAX_ABS_TOL = 1e-2   # attention output tolerances (bf16/fp16 outputs vs fp64)
MEAN_ABS_TOL = 1e-3


@dataclass
class Sides:
    w: object
    out: torch.Tensor          # product output (device)
    kc: torch.Tensor           # product caches after the write path (device)
    vc: torch.Tensor
    ref: np.ndarray | None     # oracle output fp64
    kc_ref: np.ndarray         # oracle caches after the write path (host)
    vc_ref: np.ndarray


def host_copy(t: torch.Tensor) -> np.ndarray:
    t = t.detach().cpu().contiguous()
    if t.dtype in (torch.float16, torch.bfloat16):
        return t.view(torch.int16).numpy().view(np.uint16).copy()
    return t.numpy().copy()


def run_both(spec, device="cuda", pairs=None, run_oracle_decode=True, threads=None,
             mutate=None) -> Sides:
    """`mutate(w)`, if given, rewrites the generated inputs (test data
    construction) before either side takes them."""
    w = generate(spec, device=device)
    if mutate is not None:
        mutate(w)
    s = w.spec
    fp8 = s.kv_fp8
    kv = "fp8" if fp8 else "auto"
    # ---- oracle inputs first (host copies of generator output)
    if fp8:
        shape = (w.num_blocks, s.num_kv_heads, s.block_size, s.head_dim)
        kc_ref = np.full(shape, E4M3_NAN, np.uint8)
        vc_ref = np.full(shape, E4M3_NAN, np.uint8)
        oracle.reshape_and_cache(w.k_hist.cpu(), w.v_hist.cpu(), kc_ref, vc_ref,
                                 w.slot_hist.cpu().numpy(), s.dtype, "fp8", w.k_scale,
                                 w.v_scale, threads=threads)
    else:
        kc_ref, vc_ref = host_copy(w.key_cache), host_copy(w.value_cache)
    oracle.reshape_and_cache(w.k_new.cpu(), w.v_new.cpu(), kc_ref, vc_ref,
                             w.slot_new.cpu().numpy(), s.dtype, "fp8" if fp8 else s.dtype,
                             w.k_scale, w.v_scale, threads=threads)
    # ---- product path
    if fp8:
        kc, vc = w.empty_fp8_cache()
        pa.reshape_and_cache(w.k_hist, w.v_hist, kc, vc, w.slot_hist, kv, w.k_scale, w.v_scale)
    else:
        kc, vc = w.key_cache, w.value_cache
    pa.reshape_and_cache(w.k_new, w.v_new, kc, vc, w.slot_new, kv, w.k_scale, w.v_scale)
    bt = torch.from_numpy(w.block_tables).to(device)
    sl = torch.from_numpy(w.seq_lens).to(device)
    out = pa.decode(w.q, kc, vc, bt, sl, num_kv_heads=s.num_kv_heads, scale=s.softmax_scale,
                    block_size=s.block_size, window=s.window, kv_dtype=kv, k_scale=w.k_scale,
                    v_scale=w.v_scale)
    torch.cuda.synchronize()
    ref = None
    if run_oracle_decode:
        ref = oracle.decode(w.q.cpu(), kc_ref, vc_ref, w.block_tables, w.seq_lens,
                            num_kv_heads=s.num_kv_heads, scale=s.softmax_scale,
                            block_size=s.block_size, window=s.window, q_dtype=s.dtype,
                            cache_dtype="fp8" if fp8 else s.dtype, k_scale=w.k_scale,
                            v_scale=w.v_scale, pairs=pairs, threads=threads)
    return Sides(w, out, kc, vc, ref, kc_ref, vc_ref)


def out_f64(out: torch.Tensor) -> np.ndarray:
    return out.detach().float().cpu().double().numpy()


# Chunked queries: rows that attend to a handful of positions have outputs of
# magnitude up to ~4 (nearly one V row), where rounding the output to bf16
# alone costs up to 2^-9 |out| and rounding P to bf16 up to 2^-9 max|v|; the
# bound grows by 2^-8 |ref| on top of the decode tolerance.
CHUNK_REL_TOL = 2.0 ** -8


def assert_close(got: np.ndarray, ref: np.ndarray, pairs=None, what="", rel=0.0):
    if pairs is not None:
        idx = tuple(np.asarray(pairs).T)
        got, ref = got[idx], ref[idx]
    assert np.isfinite(got).all(), f"{what}: non-finite outputs"
    err = np.abs(got - ref)
    excess = err - (MAX_ABS_TOL + rel * np.abs(ref))
    assert excess.max() <= 0, f"{what}: max abs err {err.max():.3e} (bound exceeded by {excess.max():.3e})"
    assert err.mean() <= MEAN_ABS_TOL, f"{what}: mean abs err {err.mean():.3e}"
    return float(err.max()), float(err.mean())


def assert_caches_equal(sides: Sides, what=""):
    kc = host_copy(sides.kc)
    vc = host_copy(sides.vc)
    assert np.array_equal(kc, sides.kc_ref), f"{what}: key cache differs from the oracle"
    assert np.array_equal(vc, sides.vc_ref), f"{what}: value cache differs from the oracle"


def run_chunk(spec, device="cuda", triples=None, threads=None, use_chunk_entry=True,
              mutate=None) -> Sides:
    """The chunked step: the write path stores the B * T new K/V rows, then
    pa_prefill_chunk attends each sequence's T queries causally; the oracle
    runs its reshape and causal multi-query decode on host copies. `mutate`
    as in run_both."""
    w = generate(spec, device=device)
    if mutate is not None:
        mutate(w)
    s = w.spec
    fp8 = s.kv_fp8
    kv = "fp8" if fp8 else "auto"
    if fp8:
        shape = (w.num_blocks, s.num_kv_heads, s.block_size, s.head_dim)
        kc_ref = np.full(shape, E4M3_NAN, np.uint8)
        vc_ref = np.full(shape, E4M3_NAN, np.uint8)
        oracle.reshape_and_cache(w.k_hist.cpu(), w.v_hist.cpu(), kc_ref, vc_ref,
                                 w.slot_hist.cpu().numpy(), s.dtype, "fp8", w.k_scale,
                                 w.v_scale, threads=threads)
    else:
        kc_ref, vc_ref = host_copy(w.key_cache), host_copy(w.value_cache)
    oracle.reshape_and_cache(w.k_new.cpu(), w.v_new.cpu(), kc_ref, vc_ref,
                             w.slot_new.cpu().numpy(), s.dtype, "fp8" if fp8 else s.dtype,
                             w.k_scale, w.v_scale, threads=threads)
    q4 = w.q if w.q.dim() == 4 else w.q.unsqueeze(1)
    if fp8:
        kc, vc = w.empty_fp8_cache()
        pa.reshape_and_cache(w.k_hist, w.v_hist, kc, vc, w.slot_hist, kv, w.k_scale, w.v_scale)
    else:
        kc, vc = w.key_cache, w.value_cache
    pa.reshape_and_cache(w.k_new, w.v_new, kc, vc, w.slot_new, kv, w.k_scale, w.v_scale)
    bt = torch.from_numpy(w.block_tables).to(device)
    sl = torch.from_numpy(w.seq_lens).to(device)
    kw = dict(num_kv_heads=s.num_kv_heads, scale=s.softmax_scale, block_size=s.block_size,
              window=s.window, kv_dtype=kv, k_scale=w.k_scale, v_scale=w.v_scale)
    if use_chunk_entry:
        out = pa.prefill_chunk(q4, kc, vc, bt, sl, **kw)
    else:
        out = pa.decode(w.q, kc, vc, bt, sl, **kw)
    torch.cuda.synchronize()
    ref = oracle.decode_multi(q4.cpu(), kc_ref, vc_ref, w.block_tables, w.seq_lens,
                              num_kv_heads=s.num_kv_heads, scale=s.softmax_scale,
                              block_size=s.block_size, window=s.window, q_dtype=s.dtype,
                              cache_dtype="fp8" if fp8 else s.dtype, k_scale=w.k_scale,
                              v_scale=w.v_scale, triples=triples, threads=threads)
    return Sides(w, out, kc, vc, ref, kc_ref, vc_ref)
