"""Seeded generator for paged decode workloads.

Recipe, in order:
  1. sequence lengths from numpy's PCG64 seeded with ``spec.seed``;
  2. a pool of NB physical blocks and the tables a block allocator gives
     these requests (``layout.py``): a seeded shuffled free list; the shared
     prefix (if any) allocated once and forked by every sequence, then each
     sequence's private blocks, so physical ids are scattered;
  3. one K row and one V row of N(0, 1) values per unique token (shared prefix
     tokens are one row for all sequences), drawn by torch's generator seeded
     with ``spec.seed`` on the target device and rounded to the 16-bit dtype;
  4. q ~ N(0, 1) of shape [B, Hq, D], or [B, T, Hq, D] for a chunk of
     T = ``num_queries`` query tokens per sequence;
  5. the last T positions of each sequence are the new tokens (``k_new``,
     ``v_new`` and their slots, row b * T + t for position L - T + t, slot -1
     where that position is negative); every other position that some
     sequence reads is a history row (``k_hist``, ``v_hist``, ``slot_hist``);
  6. for 16-bit caches, history rows are placed in their slots and every other
     slot of the pool holds NaN, so a read of an unused slot, a tail slot past
     the sequence end, a slot before the window, or a new-token slot that was
     never written shows up in the result. FP8 caches start as all-NaN codes
     (0x7F) and are filled by the write path from the history rows.

The window is read as "a sequence of length L attends to its last min(L, W)
positions" (W <= 0: all positions); query t of a chunk, at position
p = L - T + t, attends to [max(0, p + 1 - W), p], so a chunk reads the
union [max(0, L - T + 1 - W), L).
"""
from __future__ import annotations

import math
from dataclasses import dataclass

import numpy as np
import torch

from .configs import Spec
from .layout import block_tables

TORCH_DTYPES = {"f16": torch.float16, "bf16": torch.bfloat16}
E4M3_NAN = 0x7F


@dataclass
class Workload:
    spec: Spec
    seq_lens: np.ndarray          # int32 [B]
    starts: np.ndarray            # int64 [B], first position read (by the first query)
    block_tables: np.ndarray      # int32 [B, MB], -1 past the used blocks
    num_blocks: int
    max_blocks: int
    q: torch.Tensor               # [B, Hq, D], or [B, T, Hq, D] for a chunk
    key_cache: torch.Tensor | None    # 16-bit [NB, Hkv, bs, D]; None for FP8
    value_cache: torch.Tensor | None
    k_hist: torch.Tensor | None   # [Nh, Hkv, D]
    v_hist: torch.Tensor | None
    slot_hist: torch.Tensor | None  # int64 [Nh]
    k_new: torch.Tensor           # [B * T, Hkv, D] (row b * T + t: position L_b - T + t)
    v_new: torch.Tensor
    slot_new: torch.Tensor        # int64 [B * T]; -1 where the position is negative
    k_scale: float
    v_scale: float

    @property
    def cache_dtype(self) -> str:
        return "fp8" if self.spec.kv_fp8 else self.spec.dtype

    def empty_fp8_cache(self, device=None) -> tuple[torch.Tensor, torch.Tensor]:
        s = self.spec
        shape = (self.num_blocks, s.num_kv_heads, s.block_size, s.head_dim)
        dev = device if device is not None else self.q.device
        return (torch.full(shape, E4M3_NAN, dtype=torch.uint8, device=dev),
                torch.full(shape, E4M3_NAN, dtype=torch.uint8, device=dev))


def draw_seq_lens(spec: Spec, rng: np.random.Generator) -> np.ndarray:
    if spec.seq_lens is not None:
        lens = np.asarray(spec.seq_lens, dtype=np.int64)
        assert lens.shape == (spec.batch,)
        return lens
    n_rand = spec.batch - len(spec.long_seqs)
    kind, lo, hi = spec.len_dist
    if kind == "uniform":
        r = rng.integers(lo, hi + 1, size=n_rand)
    elif kind == "loguniform":
        r = np.floor(np.exp(rng.uniform(math.log(lo), math.log(hi + 1), size=n_rand)))
        r = np.clip(r, lo, hi).astype(np.int64)
    else:
        raise ValueError(kind)
    lens = np.concatenate([np.asarray(spec.long_seqs, dtype=np.int64), r.astype(np.int64)])
    return lens + spec.shared_prefix


def max_len_of(spec: Spec) -> int:
    if spec.max_len is not None:
        return spec.max_len
    if spec.seq_lens is not None:
        return int(max(spec.seq_lens)) if len(spec.seq_lens) else 0
    hi = spec.len_dist[2] + spec.shared_prefix
    return max([hi] + list(spec.long_seqs))


def layout(spec: Spec) -> tuple[np.ndarray, np.ndarray, int, int]:
    """Steps 1 and 2 of the recipe: (seq_lens int64 [B], block tables int32
    [B, MB], pool blocks NB, table width MB), no values."""
    s = spec
    bs = s.block_size
    assert s.shared_prefix % bs == 0
    rng = np.random.default_rng(s.seed)
    lens = draw_seq_lens(s, rng)
    P = s.shared_prefix
    assert (lens >= P).all() and (P == 0 or (lens > P).all())
    MB = -(-max_len_of(s) // bs)
    assert (lens <= MB * bs).all()
    nblk = -(-lens // bs)
    shared_blocks = P // bs
    need = shared_blocks + int((nblk - shared_blocks).clip(min=0).sum())
    NB = s.pool_blocks if s.pool_blocks is not None else int(math.ceil(s.pool_factor * need))
    assert NB >= need, "pool smaller than the layout needs"
    # physical layout: the block allocator's tables for these requests
    return lens, block_tables(lens, bs, P, NB, MB, s.seed), NB, MB


def generate(spec: Spec, device="cpu", keep_hist: bool | None = None) -> Workload:
    s = spec
    dev = torch.device(device)
    bs, Hkv, D = s.block_size, s.num_kv_heads, s.head_dim
    assert s.num_q_heads % Hkv == 0
    lens, tables, NB, MB = layout(s)
    B = s.batch
    P = s.shared_prefix

    # range read per sequence: the union of its queries' ranges
    T = s.num_queries
    assert T >= 1
    W = s.window + T - 1 if s.window > 0 else 0
    starts = np.where((W > 0) & (lens > W), lens - W, 0).astype(np.int64)

    # unique token rows: shared prefix first, then each sequence's private tokens
    priv = lens - P
    priv_off = np.concatenate([[0], np.cumsum(priv)[:-1]]).astype(np.int64)
    R = P + int(priv.sum())

    # every (sequence, position) that is read, mapped to its row and slot
    b_idx = np.repeat(np.arange(B), (lens - starts))
    pos = np.concatenate([np.arange(starts[b], lens[b]) for b in range(B)]) if B else \
        np.zeros(0, np.int64)
    pos = pos.astype(np.int64)
    row = np.where(pos < P, pos, P + priv_off[b_idx] + (pos - P))
    slot = tables[b_idx, pos // bs].astype(np.int64) * bs + pos % bs
    is_new = pos >= (lens[b_idx] - T)
    # rows read by several sequences (shared prefix) appear once
    hist_rows, first = np.unique(row[~is_new], return_index=True)
    hist_slots = slot[~is_new][first]

    # new tokens: position L - T + t of sequence b is row b * T + t
    nb_ = np.repeat(np.arange(B), T)
    npos = np.repeat(lens, T) - T + np.tile(np.arange(T), B)
    live = npos >= 0
    pc = np.maximum(npos, 0)
    new_rows = np.where(pc < P, pc, P + priv_off[nb_] + (pc - P))
    new_rows = np.where(live, new_rows, 0)
    new_slots = np.where(live, tables[nb_, pc // bs].astype(np.int64) * bs + pc % bs, -1)
    if not s.new_tokens:
        # without a write step, the last positions are history rows too
        hist_rows = np.concatenate([hist_rows, new_rows[live]])
        hist_slots = np.concatenate([hist_slots, new_slots[live]])
        new_slots = np.full(B * T, -1, np.int64)

    # values
    tdt = TORCH_DTYPES[s.dtype]
    g = torch.Generator(device=dev)
    g.manual_seed(s.seed)
    Kl = torch.randn((max(R, 1), Hkv, D), generator=g, device=dev, dtype=torch.float32).to(tdt)
    Vl = torch.randn((max(R, 1), Hkv, D), generator=g, device=dev, dtype=torch.float32).to(tdt)
    qshape = (B, s.num_q_heads, D) if T == 1 else (B, T, s.num_q_heads, D)
    q = torch.randn(qshape, generator=g, device=dev, dtype=torch.float32).to(tdt)

    hr = torch.as_tensor(hist_rows, dtype=torch.int64, device=dev)
    k_hist, v_hist = Kl[hr], Vl[hr]
    slot_hist = torch.as_tensor(hist_slots, dtype=torch.int64, device=dev)
    nr = torch.as_tensor(new_rows, dtype=torch.int64, device=dev)
    k_new, v_new = Kl[nr].clone(), Vl[nr].clone()
    slot_new = torch.as_tensor(new_slots, dtype=torch.int64, device=dev)

    if s.kv_fp8:
        k_scale = float((Kl[:R].abs().amax().float() / 448.0).item()) if R else 1.0
        v_scale = float((Vl[:R].abs().amax().float() / 448.0).item()) if R else 1.0
        key_cache = value_cache = None
    else:
        k_scale = v_scale = 1.0
        shape = (NB, Hkv, bs, D)
        key_cache = torch.full(shape, float("nan"), dtype=tdt, device=dev)
        value_cache = torch.full(shape, float("nan"), dtype=tdt, device=dev)
        blk_t = slot_hist // bs
        off_t = slot_hist % bs
        key_cache.permute(0, 2, 1, 3)[blk_t, off_t] = k_hist
        value_cache.permute(0, 2, 1, 3)[blk_t, off_t] = v_hist
    del Kl, Vl
    if keep_hist is None:
        keep_hist = s.kv_fp8
    if not keep_hist:
        k_hist = v_hist = slot_hist = None

    return Workload(spec=s, seq_lens=lens.astype(np.int32), starts=starts, block_tables=tables,
                    num_blocks=NB, max_blocks=MB, q=q, key_cache=key_cache,
                    value_cache=value_cache, k_hist=k_hist, v_hist=v_hist, slot_hist=slot_hist,
                    k_new=k_new, v_new=v_new, slot_new=slot_new, k_scale=k_scale,
                    v_scale=v_scale)
