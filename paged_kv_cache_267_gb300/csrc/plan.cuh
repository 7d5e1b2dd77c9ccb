// The work plan of one decode step, computed from seq_lens alone by the
// decode kernel. Its first CTA stores it in the workspace (plan region, see
// pa_internal.h) before streaming, and the merge kernel reads it there after
// the decode kernel has finished.
//
// Every (sequence b, virtual KV head) pair owns the 16-token tiles covering
// its read range [start, L); all tiles form one flat, pair-major index space.
// Its first part is split into equal static ranges of `ws` tiles, one per
// worker warp (ending at `ts`); the rest is a pool of pieces of `piece`
// tiles claimed dynamically. The pool only covers the trailing run of
// sequences whose tile count is at most four times the mean, so a long
// sequence is never cut into many small pieces. (Ending the pool with
// one-tile pieces, so that a warp holds less work when it runs dry, gave the
// last pairs up to 157 partials and made the step 2 us slower through the
// merge.)
#pragma once

#include "pa_internal.h"

namespace pa {

__device__ __forceinline__ int win_start(int L, int W) { return (W > 0 && L > W) ? L - W : 0; }
__device__ __forceinline__ int tiles_of(int L, int W) {
  return L > 0 ? (L + kTile - 1) / kTile - win_start(L, W) / kTile : 0;
}

struct PlanIn {
  const int32_t* seq_lens;  // [B]
  int32_t* err;             // device error word (null: do not report)
  int B;
  int cap;                  // longest sequence the tables can hold: MB * bs
  int span;                 // window of the pairs' tile ranges (0: none)
  int Hv;                   // pairs per sequence
  int nw;                   // worker warps of the decode kernel
  int pool_permille, min_tiles, np_max, piece_min;
};

struct StepPlan {
  int total;   // tiles of all pairs
  int ws;      // static tiles per warp
  int ts;      // end of the static region
  int piece;   // tiles per pool piece
  int n_pool;  // pool pieces: ceil((total - ts) / piece)
};

// Pool piece holding flat tile f (ts <= f < total).
__device__ __forceinline__ int piece_of(int f, const StepPlan& pl) {
  return (f - pl.ts) / pl.piece;
}

// First flat tile and end of pool piece i (i < n_pool).
__device__ __forceinline__ void piece_range(int i, const StepPlan& pl, int* f0, int* f1) {
  *f0 = pl.ts + i * pl.piece;
  *f1 = min(*f0 + pl.piece, pl.total);
}

// Block-wide: every thread of the block calls it (it synchronises the
// block). Fills s_len[0 .. B) with the lengths clamped to [0, cap] (a length
// outside is reported through `err`) and s_pref[0 .. B] with the exclusive
// prefix of tiles per pair over the sequences. The host bounds B * Hv * tiles
// per pair below 2^31, so the tile counts fit 32-bit integers.
__device__ inline StepPlan plan_step(const PlanIn& p, int* s_len, int* s_pref) {
  constexpr unsigned FULL = 0xffffffffu;
  __shared__ int s_last_long;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  for (int b = tid; b < p.B; b += blockDim.x) {
    int L = p.seq_lens[b];
    if (L < 0 || L > p.cap) {
      if (p.err) atomicOr(p.err, PA_DEVERR_SEQ_LEN);
      L = L < 0 ? 0 : p.cap;
    }
    s_len[b] = L;
  }
  __syncthreads();
  // exclusive prefix of tiles per pair over the sequences (one warp)
  if (warp == 0) {
    int run = 0;
    for (int b0 = 0; b0 < p.B; b0 += 32) {
      const int b = b0 + lane;
      int x = (b < p.B) ? tiles_of(s_len[b], p.span) : 0;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(FULL, x, o);
        if (lane >= o) x += y;
      }
      if (b < p.B) s_pref[b + 1] = run + x;
      run += __shfl_sync(FULL, x, 31);
    }
    if (lane == 0) s_pref[0] = 0;
  }
  __syncthreads();
  // the last sequence longer than four times the mean
  if (warp == 0) {
    const long long thr = 4ll * s_pref[p.B];  // nt_b * B > thr  <=>  nt_b > 4 * mean
    int last = -1;
    for (int b = lane; b < p.B; b += 32)
      if (static_cast<long long>(s_pref[b + 1] - s_pref[b]) * p.B > thr) last = b;
    last = __reduce_max_sync(FULL, last);  // one redux.sync: shuffle chains are slow here
    if (lane == 0) s_last_long = last;
  }
  __syncthreads();
  StepPlan r;
  r.total = p.Hv * s_pref[p.B];
  const int short_tail = r.total - p.Hv * s_pref[s_last_long + 1];
  int pool_want = static_cast<int>(static_cast<long long>(r.total) * p.pool_permille / 1000);
  if (pool_want > short_tail) pool_want = short_tail;
  // rounded up, so that the static ranges never reach into the pool's share
  const unsigned nw = static_cast<unsigned>(p.nw);
  r.ws = static_cast<int>((static_cast<unsigned>(r.total - pool_want) + nw - 1u) / nw);
  if (r.ws < p.min_tiles) r.ws = p.min_tiles;
  r.ts = static_cast<int>(
      min(static_cast<long long>(r.ws) * p.nw, static_cast<long long>(r.total)));
  const int pool_tiles = r.total - r.ts;
  r.piece = static_cast<int>((static_cast<unsigned>(pool_tiles) + p.np_max - 1u) /
                             static_cast<unsigned>(p.np_max));
  if (r.piece < p.piece_min) r.piece = p.piece_min;
  r.n_pool = static_cast<int>((static_cast<unsigned>(pool_tiles) + r.piece - 1u) /
                              static_cast<unsigned>(r.piece));
  return r;
}

__device__ __forceinline__ StepPlan plan_load(const int32_t* src) {
  StepPlan pl;
  pl.total = src[0];
  pl.ws = src[1];
  pl.ts = src[2];
  pl.piece = src[3];
  pl.n_pool = src[4];
  return pl;
}

// Partial results of pair s (tiles [F, F + nt) of the flat space): the
// static slots of the warps whose range meets [F, min(F + nt, ts)), then the
// pool slots of the pieces that meet [max(F, ts), F + nt).
struct Cands {
  int w0, na;  // static warps [w0, w0 + na)
  int i0, np;  // pool pieces [i0, i0 + np)
};

__device__ __forceinline__ Cands pair_cands(int F, int nt, const StepPlan& pl) {
  Cands c = {0, 0, 0, 0};
  if (nt > 0 && F < pl.ts) {
    c.w0 = F / pl.ws;
    c.na = (min(F + nt, pl.ts) - 1) / pl.ws - c.w0 + 1;
  }
  if (nt > 0 && F + nt > pl.ts) {
    c.i0 = piece_of(max(F, pl.ts), pl);
    c.np = piece_of(F + nt - 1, pl) - c.i0 + 1;
  }
  return c;
}

// Upper bound of the partial results of any pair of a sequence whose pairs
// have nt tiles each and span flat tiles [lo, hi) (the merge kernel sizes
// its column groups by it): a run of nt tiles meets at most nt / ws + 2
// static ranges and nt / piece + 2 pool pieces (and no more than its own
// tiles, nor more pieces than the sequence's range meets).
__device__ __forceinline__ int pair_cand_bound(int nt, int lo, int hi, const StepPlan& pl) {
  if (nt <= 0) return 0;
  int ub = 0;
  if (lo < pl.ts) ub += min(nt, nt / pl.ws + 2);
  if (hi > pl.ts) {
    const int first = piece_of(max(lo, pl.ts), pl), last = piece_of(hi - 1, pl);
    ub += min(min(nt, nt / pl.piece + 2), last - first + 1);
  }
  return ub;
}

}  // namespace pa
