// Log-sum-exp merge of decode partials, and the KV write path
// (reshape_and_cache), for sm_103a.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "pa_internal.h"
#include "plan.cuh"
#include "ptx.cuh"

namespace pa {

// Device error word (one per device); kernels of every translation unit get
// its address through their argument structs.
__device__ int32_t g_device_error;

cudaError_t device_error_word(int32_t** ptr) {
  return cudaGetSymbolAddress(reinterpret_cast<void**>(ptr), g_device_error);
}

// ------------------------------------------------------------------ merge
//
// The partial results of a pair (its candidates, see pair_cands) have maxima
// m_p (log2 domain), sums l_p and unnormalised outputs o_p; for an output
// column the result is
//   out = sum_p 2^(m_p - M) o_p / sum_p 2^(m_p - M) l_p,  M = max_p m_p,
// and zero when the denominator is zero (a chunked query placed before the
// start of its sequence attends to nothing). A column is a q head of the pair
// (single-query decode) or a (query, q head) of a chunk; columns that pad the
// last group of a chunk have no output row and are skipped.
//
// The plan of the step (how the decode kernel split the tiles) comes from
// the decode kernel's first CTA through the workspace, so the merge reads
// the tile prefix rather than recomputing it from seq_lens; a CTA that sees
// the plan flag set loads it before its dependency wait (it is launched as
// the decode kernel's programmatic dependent). From the plan each CTA sizes
// the work of each sequence's columns by a bound of the partials of any of
// its pairs (pair_cand_bound): up to 8, one warp per column; up to 32, four
// warps of a CTA (two such columns per CTA); more, all eight warps of a CTA.
// The warps of a group fold equal shares of the column's partials and
// combine their results through shared memory. A warp folds its partials
// online with eight loads in flight per lane (D <= 128; four for D = 256).
constexpr int kMergeThreads = 256;
constexpr int kPlanPolls = 64;       // polls of the plan flag before the wait, at most
constexpr int kPlanPollNs = 500;     // pause between polls
constexpr int kMergeWarps = kMergeThreads / 32;

// Per-lane state of one column: head dims v * 128 + 4 * lane .. + 3 for
// v < VPL (VPL = 1 for D <= 128, 2 for D = 256).
template <int VPL>
struct HeadAcc {
  float M, den;
  float4 acc[VPL];
};

// Folds candidates k0 .. k1 - 1 of column h into `r` (which starts empty),
// U = 8 / VPL candidates' loads in flight per lane. Lane j < U reads
// candidate j's max and sum, which the fold takes by shuffle.
template <int VPL, typename SlotFn>
__device__ __forceinline__ void merge_fold(const MergeArgs& a, SlotFn slot_of, int k0, int k1,
                                           int h, HeadAcc<VPL>& r) {
  constexpr int U = 8 / VPL;
  const int lane = threadIdx.x & 31;
  const int GD = a.CG * a.D;
  const size_t stride = static_cast<size_t>(part_stride(a.CG, a.D));
  r.M = -INFINITY;
  r.den = 0.f;
#pragma unroll
  for (int v = 0; v < VPL; ++v) r.acc[v] = make_float4(0.f, 0.f, 0.f, 0.f);
  const bool on = 4 * lane < a.D;  // D = 64 uses half the lanes
  const uint64_t once = l2_evict_first();  // each partial is read once
  for (int k = k0; k < k1; k += U) {
    float my_m = -INFINITY, my_l = 0.f;
    if (lane < U && k + lane < k1) {
      const float* P = a.part + static_cast<size_t>(slot_of(k + lane)) * stride;
      my_m = ld_f32_hint(P + GD + h, once);
      my_l = ld_f32_hint(P + GD + a.CG + h, once);
    }
    float4 o[U][VPL];
#pragma unroll
    for (int j = 0; j < U; ++j) {
      const int kk = k + j;
#pragma unroll
      for (int v = 0; v < VPL; ++v) o[j][v] = make_float4(0.f, 0.f, 0.f, 0.f);
      if (kk < k1 && on) {
        const float* P = a.part + static_cast<size_t>(slot_of(kk)) * stride;
#pragma unroll
        for (int v = 0; v < VPL; ++v)
          o[j][v] = ld_f32x4_hint(P + h * a.D + v * 128 + 4 * lane, once);
      }
    }
#pragma unroll
    for (int j = 0; j < U; ++j) {
      const float mj = __shfl_sync(0xffffffffu, my_m, j), lj = __shfl_sync(0xffffffffu, my_l, j);
      if (k + j >= k1) break;
      const float Mn = fmaxf(r.M, mj);
      const float sc = fast_exp2(r.M - Mn), f = fast_exp2(mj - Mn);
      r.den = r.den * sc + f * lj;
#pragma unroll
      for (int v = 0; v < VPL; ++v) {
        r.acc[v].x = r.acc[v].x * sc + f * o[j][v].x;
        r.acc[v].y = r.acc[v].y * sc + f * o[j][v].y;
        r.acc[v].z = r.acc[v].z * sc + f * o[j][v].z;
        r.acc[v].w = r.acc[v].w * sc + f * o[j][v].w;
      }
      r.M = Mn;
    }
  }
}

template <int OT>
__device__ __forceinline__ void store_out4(void* out, size_t idx, float4 x, float inv) {
  if constexpr (OT == kBF16) {
    __nv_bfloat162 p0 = __floats2bfloat162_rn(x.x * inv, x.y * inv);
    __nv_bfloat162 p1 = __floats2bfloat162_rn(x.z * inv, x.w * inv);
    uint2 u = make_uint2(*reinterpret_cast<uint32_t*>(&p0), *reinterpret_cast<uint32_t*>(&p1));
    *reinterpret_cast<uint2*>(reinterpret_cast<__nv_bfloat16*>(out) + idx) = u;
  } else {
    __half2 p0 = __floats2half2_rn(x.x * inv, x.y * inv);
    __half2 p1 = __floats2half2_rn(x.z * inv, x.w * inv);
    uint2 u = make_uint2(*reinterpret_cast<uint32_t*>(&p0), *reinterpret_cast<uint32_t*>(&p1));
    *reinterpret_cast<uint2*>(reinterpret_cast<__half*>(out) + idx) = u;
  }
}

template <int OT, int VPL>
__device__ __forceinline__ void store_head(const MergeArgs& a, size_t orow, const HeadAcc<VPL>& r,
                                           bool zero) {
  const int lane = threadIdx.x & 31;
  if (4 * lane >= a.D) return;
  const float inv = (zero || !(r.den > 0.f)) ? 0.f : 1.f / r.den;
  const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
  for (int v = 0; v < VPL; ++v)
    store_out4<OT>(a.out, orow + v * 128 + 4 * lane, zero ? z : r.acc[v], inv);
}

// Half-warp form for D <= 128, used when a step has more output columns than
// the grid has warps: lanes 16 j .. 16 j + 15 of a warp fold one column each,
// lane i of a half holding head dims 64 v + 4 i .. + 3 for v < D / 64, with
// four candidates' loads in flight per lane. Both halves run the same number
// of rounds (the larger of their two columns'), and every lane takes part in
// the shuffles of the round's maxima and sums before any lane skips a
// candidate, so the shuffles never diverge.
struct HalfAcc {
  float M, den;
  float4 acc[2];
};

template <typename SlotFn>
__device__ __forceinline__ void merge_fold_half(const MergeArgs& a, SlotFn slot_of, int n, int h,
                                                HalfAcc& r) {
  constexpr int U = 4;
  const int lane = threadIdx.x & 31, l16 = lane & 15, hb = lane & 16;
  const int GD = a.CG * a.D, nv = a.D >> 6;
  const size_t stride = static_cast<size_t>(part_stride(a.CG, a.D));
  r.M = -INFINITY;
  r.den = 0.f;
  r.acc[0] = r.acc[1] = make_float4(0.f, 0.f, 0.f, 0.f);
  const uint64_t once = l2_evict_first();  // each partial is read once
  int rounds = (n + U - 1) / U;
  rounds = max(rounds, __shfl_xor_sync(0xffffffffu, rounds, 16));
  for (int k = 0; k < rounds * U; k += U) {
    float my_m = -INFINITY, my_l = 0.f;
    if (l16 < U && k + l16 < n) {
      const float* P = a.part + static_cast<size_t>(slot_of(k + l16)) * stride;
      my_m = ld_f32_hint(P + GD + h, once);
      my_l = ld_f32_hint(P + GD + a.CG + h, once);
    }
    float4 o[U][2];
#pragma unroll
    for (int j = 0; j < U; ++j) {
      o[j][0] = o[j][1] = make_float4(0.f, 0.f, 0.f, 0.f);
      if (k + j < n) {
        const float* P = a.part + static_cast<size_t>(slot_of(k + j)) * stride + h * a.D;
#pragma unroll
        for (int v = 0; v < 2; ++v)
          if (v < nv) o[j][v] = ld_f32x4_hint(P + 64 * v + 4 * l16, once);
      }
    }
    float mv[U], lv[U];
#pragma unroll
    for (int j = 0; j < U; ++j) {
      mv[j] = __shfl_sync(0xffffffffu, my_m, hb + j);
      lv[j] = __shfl_sync(0xffffffffu, my_l, hb + j);
    }
#pragma unroll
    for (int j = 0; j < U; ++j) {
      if (k + j >= n) break;
      const float Mn = fmaxf(r.M, mv[j]);
      const float sc = fast_exp2(r.M - Mn), f = fast_exp2(mv[j] - Mn);
      r.den = r.den * sc + f * lv[j];
#pragma unroll
      for (int v = 0; v < 2; ++v) {
        r.acc[v].x = r.acc[v].x * sc + f * o[j][v].x;
        r.acc[v].y = r.acc[v].y * sc + f * o[j][v].y;
        r.acc[v].z = r.acc[v].z * sc + f * o[j][v].z;
        r.acc[v].w = r.acc[v].w * sc + f * o[j][v].w;
      }
      r.M = Mn;
    }
  }
}

template <int OT>
__device__ __forceinline__ void store_half(const MergeArgs& a, size_t orow, const HalfAcc& r,
                                           bool zero) {
  const int l16 = threadIdx.x & 15, nv = a.D >> 6;
  const float inv = (zero || !(r.den > 0.f)) ? 0.f : 1.f / r.den;
  const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
  for (int v = 0; v < 2; ++v)
    if (v < nv) store_out4<OT>(a.out, orow + 64 * v + 4 * l16, zero ? z : r.acc[v], inv);
}

// Where output column `col` of sequence b lives, and its candidates.
struct MergeCol {
  bool pad;     // a column padding the last group of a chunk
  int h;        // column within its pair
  size_t orow;  // first element of its output row
  int s;        // pair index
  Cands cd;
  int ncand;
};

__device__ __forceinline__ MergeCol merge_col(const MergeArgs& a, const StepPlan& pl,
                                              const int* s_pref, int b, int col) {
  MergeCol c;
  const int vh = col / a.CG;
  c.h = col - vh * a.CG;  // pair and column within it
  const int kvh = vh / a.NCG;
  const int gc = (vh - kvh * a.NCG) * a.CG + c.h;  // column among the kv head's T * G
  c.pad = gc >= a.T * a.G;
  const int tq = gc / a.G;
  c.s = b * a.Hv + vh;
  const int nt = s_pref[b + 1] - s_pref[b];
  const int F = a.Hv * s_pref[b] + vh * nt;
  c.cd = pair_cands(F, nt, pl);
  c.ncand = c.cd.na + c.cd.np;
  c.orow = ((static_cast<size_t>(b) * a.T + tq) * a.Hq + kvh * a.G + (gc - tq * a.G)) * a.D;
  return c;
}

// Combines the results of ngrp warps (shared-memory rows s_grp[w0 ..
// w0 + ngrp)) and stores the column (zeros when ngrp == 0).
template <int OT, int VPL>
__device__ __forceinline__ void combine_groups(const MergeArgs& a, const float* s_grp, int w0,
                                               int ngrp, size_t orow) {
  constexpr int ROW = VPL * 128 + 4;
  const int lane = threadIdx.x & 31;
  HeadAcc<VPL> r;
  r.M = -INFINITY;
  r.den = 0.f;
#pragma unroll
  for (int v = 0; v < VPL; ++v) r.acc[v] = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int j = 0; j < ngrp; ++j) {
    const float* g = s_grp + (w0 + j) * ROW;
    const float mj = g[VPL * 128], dj = g[VPL * 128 + 1];
    const float Mn = fmaxf(r.M, mj);
    const float sc = fast_exp2(r.M - Mn), f = fast_exp2(mj - Mn);
    r.den = r.den * sc + f * dj;
    if (4 * lane < a.D) {
#pragma unroll
      for (int v = 0; v < VPL; ++v) {
        const float4 o = *reinterpret_cast<const float4*>(g + v * 128 + 4 * lane);
        r.acc[v].x = r.acc[v].x * sc + f * o.x;
        r.acc[v].y = r.acc[v].y * sc + f * o.y;
        r.acc[v].z = r.acc[v].z * sc + f * o.z;
        r.acc[v].w = r.acc[v].w * sc + f * o.w;
      }
    }
    r.M = Mn;
  }
  store_head<OT, VPL>(a, orow, r, ngrp == 0);
}

template <int OT, int VPL>
__global__ void __launch_bounds__(kMergeThreads, 3) merge_kernel(const MergeArgs a) {
  constexpr int ROW = VPL * 128 + 4;  // floats per group result in shared memory
  extern __shared__ __align__(16) float s_dyn[];
  float* s_grp = s_dyn;                                                 // [8][ROW]
  int* s_plan = reinterpret_cast<int*>(s_dyn + kMergeWarps * ROW);      // plan_words(B)
  int* s_pref = s_plan + kPlanScalars;                                  // B + 1
  int* s_wide = s_plan + plan_words(a.B);                               // B + 1, see below
  __shared__ int s_red[kMergeWarps];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  // The decode kernel's first CTA publishes the plan a few microseconds
  // after it starts, long before the decode kernel ends. A CTA that sees the
  // flag set (it polls a bounded number of times) loads the plan and works
  // out its columns and their partials' slots before the dependency wait;
  // each thread waits right before its first load of a partial, so that
  // after the wait only the partials are a round trip away. A CTA that gives
  // up polling loads the plan after the wait. Each CTA counts itself in
  // pool[2] once it has read the flag; the last one clears flag and count
  // after the wait (the decode kernel has then set the flag, and no CTA of
  // this grid reads it again), so a flag seen set always belongs to this
  // step.
  int32_t* const flag = reinterpret_cast<int32_t*>(a.pool) + 1;
  uint32_t* const checked = a.pool + 2;
  int early = 0;
  bool last = false;
  if (tid == 0) {
    for (int i = 0; i < kPlanPolls; ++i) {
      early = ld_acquire_gpu(flag) == 1;
      if (early) break;
      __nanosleep(kPlanPollNs);
    }
    last = atomicAdd(checked, 1u) == gridDim.x - 1;
  }
  early = __syncthreads_or(early);
  if (early) {
    for (int i = tid; i < plan_words(a.B); i += blockDim.x) s_plan[i] = ld_relaxed_gpu(a.plan + i);
  } else {
    griddep_wait();  // the decode kernel's plan and partials are complete and visible
    for (int i = tid; i < plan_words(a.B); i += blockDim.x) s_plan[i] = a.plan[i];
  }
  __syncthreads();
  const StepPlan pl = plan_load(s_plan);
  const int HC = a.Hv * a.CG;  // columns per sequence
  const int S = a.B * a.Hv;

  // Wide columns, counted in half-CTA units: a column whose pairs may have
  // more than 4 * kMergeNarrow partials takes a whole CTA (two units; its
  // eight warps fold an eighth of the partials each), more than kMergeNarrow
  // a half (one unit; its four warps fold a quarter each), the others one
  // warp in the narrow phase below. Every sequence has an even number of
  // units, so a CTA's two units belong to one sequence. s_wide[b] = (first
  // unit of sequence b) << 2 | its class (0 narrow, 1 half, 2 whole);
  // s_wide[B] = units << 2.
  {
    int carry = 0;
    for (int b0 = 0; b0 < a.B; b0 += blockDim.x) {
      const int b = b0 + tid;
      int cls = 0, x = 0;
      if (b < a.B) {
        const int nt = s_pref[b + 1] - s_pref[b];
        const int ub = pair_cand_bound(nt, a.Hv * s_pref[b], a.Hv * s_pref[b + 1], pl);
        cls = ub > 4 * kMergeNarrow ? 2 : (ub > kMergeNarrow ? 1 : 0);
        x = cls == 2 ? 2 * HC : (cls == 1 ? HC + (HC & 1) : 0);
      }
      int y = x;  // inclusive scan over the warp, then over the CTA
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int t = __shfl_up_sync(0xffffffffu, y, o);
        if (lane >= o) y += t;
      }
      if (lane == 31) s_red[warp] = y;
      __syncthreads();
      int before = 0, all = 0;
#pragma unroll
      for (int w = 0; w < kMergeWarps; ++w) {
        const int t = s_red[w];
        before += w < warp ? t : 0;
        all += t;
      }
      if (b < a.B) s_wide[b] = ((carry + before + y - x) << 2) | cls;
      carry += all;
      __syncthreads();  // s_red is reused
    }
    if (tid == 0) s_wide[a.B] = carry << 2;
    __syncthreads();
  }
  const int n_wide = ((s_wide[a.B] >> 2) + 1) >> 1;  // CTA units
  for (int cu = blockIdx.x; cu < n_wide; cu += gridDim.x) {
    int lo = 0, hi = a.B;  // the sequence of units 2 cu, 2 cu + 1
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if ((s_wide[mid] >> 2) <= 2 * cu) lo = mid; else hi = mid;
    }
    const bool whole = (s_wide[lo] & 3) == 2;
    const int first = s_wide[lo] >> 2;
    const int half = warp >> 2;
    const int col = whole ? (2 * cu - first) >> 1 : 2 * cu + half - first;
    const int w0 = whole ? 0 : 4 * half;  // the group's first warp
    const int nwg = whole ? kMergeWarps : kMergeWarps / 2;
    bool active = col < HC;  // an odd HC pads a half-column sequence by one unit
    MergeCol c;
    if (active) {
      c = merge_col(a, pl, s_pref, lo, col);
      active = !c.pad;
    }
    int ngrp = 0;
    if (active) {
      auto slot = [&](int k) -> int {
        return k < c.cd.na ? c.s + c.cd.w0 + k : S + a.NW + c.s + c.cd.i0 + (k - c.cd.na);
      };
      const int gsz = c.ncand > 0 ? (c.ncand + nwg - 1) / nwg : 1;
      ngrp = c.ncand > 0 ? (c.ncand + gsz - 1) / gsz : 0;
      const int wi = warp - w0;
      griddep_wait();  // the partials are complete and visible
      if (wi < ngrp) {
        HeadAcc<VPL> r;
        merge_fold(a, slot, wi * gsz, min((wi + 1) * gsz, c.ncand), c.h, r);
        float* g = s_grp + warp * ROW;
        if (4 * lane < a.D) {
#pragma unroll
          for (int v = 0; v < VPL; ++v)
            *reinterpret_cast<float4*>(g + v * 128 + 4 * lane) = r.acc[v];
        }
        if (lane == 0) {
          g[VPL * 128] = r.M;
          g[VPL * 128 + 1] = r.den;
        }
      }
    }
    __syncthreads();
    if (active && warp == w0) {
      griddep_wait();
      combine_groups<OT, VPL>(a, s_grp, w0, ngrp, c.orow);
    }
    __syncthreads();  // s_grp is reused by the next wide unit
  }

  // ---- narrow columns: one warp each. The CTAs that took a wide column in
  // the last round come last in the order.
  const int rot = (blockIdx.x + gridDim.x - (n_wide % gridDim.x)) % gridDim.x;
  const int nwarps = gridDim.x * kMergeWarps;
  if (VPL == 1 && a.B * HC > nwarps) {
    // more columns than warps: half a warp per column (warp-uniform loop;
    // a half without a column folds nothing but joins the shuffles)
    for (int u2 = rot * kMergeWarps + warp; 2 * u2 < a.B * HC; u2 += nwarps) {
      const int u = 2 * u2 + (lane >> 4);
      bool act = u < a.B * HC;
      const int b = act ? u / HC : 0;
      act = act && (s_wide[b] & 3) == 0;  // wide columns are taken by the wide phase
      MergeCol c = {};
      if (act) {
        c = merge_col(a, pl, s_pref, b, u - b * HC);
        act = !c.pad;
      }
      auto slot = [&](int k) -> int {
        return k < c.cd.na ? c.s + c.cd.w0 + k : S + a.NW + c.s + c.cd.i0 + (k - c.cd.na);
      };
      HalfAcc r;
      griddep_wait();  // the partials are complete and visible
      merge_fold_half(a, slot, act ? c.ncand : 0, act ? c.h : 0, r);
      if (act) store_half<OT>(a, c.orow, r, c.ncand == 0);
    }
  } else {
    for (int u = rot * kMergeWarps + warp; u < a.B * HC; u += nwarps) {
      const int b = u / HC;
      if (s_wide[b] & 3) continue;  // taken by the wide phase
      const MergeCol c = merge_col(a, pl, s_pref, b, u - b * HC);
      if (c.pad) continue;
      auto slot = [&](int k) -> int {
        return k < c.cd.na ? c.s + c.cd.w0 + k : S + a.NW + c.s + c.cd.i0 + (k - c.cd.na);
      };
      HeadAcc<VPL> r;
      griddep_wait();  // the partials are complete and visible
      merge_fold(a, slot, 0, c.ncand, c.h, r);
      store_head<OT, VPL>(a, c.orow, r, c.ncand == 0);
    }
  }
  // the counters are zero between calls
  if (tid == 0 && (blockIdx.x == 0 || last)) {
    griddep_wait();
    if (blockIdx.x == 0) *a.pool = 0u;
    if (last) {
      st_relaxed_gpu(flag, 0);
      *checked = 0u;
    }
  }
}

cudaError_t merge_launch(int out_type, const MergeArgs& a, int grid, cudaStream_t s, bool pdl) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kMergeThreads);
  const int row = (a.D > 128 ? 2 : 1) * 128 + 4;
  cfg.dynamicSmemBytes = static_cast<size_t>(kMergeWarps) * row * sizeof(float) +
                         static_cast<size_t>(plan_words(a.B) + a.B + 1) * sizeof(int);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  void (*fn)(const MergeArgs);
  if (a.D > 128) fn = out_type == kBF16 ? merge_kernel<kBF16, 2> : merge_kernel<kF16, 2>;
  else fn = out_type == kBF16 ? merge_kernel<kBF16, 1> : merge_kernel<kF16, 1>;
  if (cfg.dynamicSmemBytes > 48 * 1024) {  // large batches: the per-sequence prefixes
    const cudaError_t e = cudaFuncSetAttribute(
        reinterpret_cast<const void*>(fn), cudaFuncAttributeMaxDynamicSharedMemorySize,
        static_cast<int>(cfg.dynamicSmemBytes));
    if (e != cudaSuccess) return e;
  }
  return cudaLaunchKernelEx(&cfg, fn, a);
}

// ------------------------------------------------------------- write path
//
// One thread per 16-byte chunk (8 elements) of a source row; blockIdx.y picks
// K (0) or V (1). 16-bit caches get a 16-byte copy. FP8 caches get
// e4m3 = cvt.rn.satfinite(float(x) / scale), the division in IEEE fp32.
__device__ __forceinline__ uint16_t e4m3x2_from_f32(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

template <int ST, bool FP8>
__global__ void __launch_bounds__(128) reshape_kernel(const ReshapeArgs a) {
  // k/v may come from the previous kernel, and the cache may still be read
  // by it: touch nothing before it completes; then let the next kernel (the
  // decode) start its launch
  griddep_wait();
  griddep_launch_dependents();
  const int chunks = a.D >> 3;
  const long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  const long long n = static_cast<long long>(a.T) * a.H * chunks;
  if (i >= n) return;
  const bool is_v = blockIdx.y == 1;
  const int c = static_cast<int>(i % chunks);
  const long long th = i / chunks;
  const int h = static_cast<int>(th % a.H);
  const int t = static_cast<int>(th / a.H);
  const long long slot = a.slots[t];
  if (slot < 0) return;
  if (slot >= a.NB * a.bs) {
    atomicOr(a.err, 4);
    return;
  }
  const long long blk = slot / a.bs;
  const int off = static_cast<int>(slot - blk * a.bs);
  const uint16_t* src = reinterpret_cast<const uint16_t*>(is_v ? a.v : a.k) +
                        t * (is_v ? a.v_stride_t : a.k_stride_t) +
                        h * (is_v ? a.v_stride_h : a.k_stride_h) + 8 * c;
  const uint4 x = *reinterpret_cast<const uint4*>(src);
  const size_t dst = ((static_cast<size_t>(blk) * a.H + h) * a.bs + off) * a.D + 8 * c;
  void* cache = is_v ? a.vc : a.kc;
  if constexpr (!FP8) {
    *reinterpret_cast<uint4*>(reinterpret_cast<uint16_t*>(cache) + dst) = x;
  } else {
    const float scale = is_v ? a.v_scale : a.k_scale;
    const uint32_t w[4] = {x.x, x.y, x.z, x.w};
    uint32_t packed[2];
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      float f[4];
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const uint32_t word = w[2 * j + e];
        const uint16_t lo = static_cast<uint16_t>(word & 0xffffu);
        const uint16_t hi = static_cast<uint16_t>(word >> 16);
        if constexpr (ST == kBF16) {
          f[2 * e] = __uint_as_float(static_cast<uint32_t>(lo) << 16);
          f[2 * e + 1] = __uint_as_float(static_cast<uint32_t>(hi) << 16);
        } else {
          f[2 * e] = __half2float(__ushort_as_half(lo));
          f[2 * e + 1] = __half2float(__ushort_as_half(hi));
        }
      }
      const uint16_t c01 = e4m3x2_from_f32(f[0] / scale, f[1] / scale);
      const uint16_t c23 = e4m3x2_from_f32(f[2] / scale, f[3] / scale);
      packed[j] = static_cast<uint32_t>(c01) | (static_cast<uint32_t>(c23) << 16);
    }
    *reinterpret_cast<uint2*>(reinterpret_cast<uint8_t*>(cache) + dst) =
        make_uint2(packed[0], packed[1]);
  }
}

cudaError_t reshape_launch(int src_type, bool fp8, const ReshapeArgs& a, cudaStream_t s) {
  const long long n = static_cast<long long>(a.T) * a.H * (a.D / 8);
  if (n == 0) return cudaSuccess;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>((n + 127) / 128), 2);
  cfg.blockDim = dim3(128);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (src_type == kBF16)
    return fp8 ? cudaLaunchKernelEx(&cfg, reshape_kernel<kBF16, true>, a)
               : cudaLaunchKernelEx(&cfg, reshape_kernel<kBF16, false>, a);
  return fp8 ? cudaLaunchKernelEx(&cfg, reshape_kernel<kF16, true>, a)
             : cudaLaunchKernelEx(&cfg, reshape_kernel<kF16, false>, a);
}

}  // namespace pa
