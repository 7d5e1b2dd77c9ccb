// Log-sum-exp merge of decode partials, and the KV write path
// (reshape_and_cache), for sm_103a.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "pa_internal.h"
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
// Partials of pair s (tiles [F, F + nt) of the flat space) are its candidates:
// the static slots s + w of the warps w whose static range meets
// [F, min(F + nt, Ts)), then the pool slots S + NW + s + i of the pieces i
// that meet [max(F, Ts), F + nt). With partial maxima m_p (log2 domain), sums
// l_p and unnormalised outputs o_p the result for an output column is
//   out = sum_p 2^(m_p - M) o_p / sum_p 2^(m_p - M) l_p,  M = max_p m_p,
// and zero when the denominator is zero (a chunked query placed before the
// start of its sequence attends to nothing). A column is a q head of the pair
// (single-query decode) or a (query, q head) of a chunk; columns that pad the
// last group of a chunk have no output row and are skipped.
// Work units are (group g of candidates, column of pair s), one warp each,
// spread over a persistent grid of many warps per SM so that the L2 latency
// of one unit hides behind the others. A unit folds its candidates in online
// (eight loads in flight per lane; groups of max(8, ceil(n / 8)) of a head's
// n candidates, so at most eight groups). A head whose candidates fit one group is
// written out directly; otherwise each unit stores its group result, which
// has the same form as a partial, in place in the slot of the group's first
// candidate, and the unit that completes the head's counter combines the
// group results and resets the counter. Pairs without tiles get zeros.
constexpr int kMergeThreads = 256;
constexpr int kMergeWarps = kMergeThreads / 32;

// Per-lane state of one q head: head dims v * 128 + 4 * lane .. + 3 for
// v < VPL (VPL = 1 for D <= 128, 2 for D = 256).
template <int VPL>
struct HeadAcc {
  float M, den;
  float4 acc[VPL];
};

// Folds candidates k0, k0 + step, ... (< k1) of head h into `r`, with
// U = 8 / VPL candidates' loads in flight per lane (a group of 8 partials is
// one round trip for D <= 128). Lane j < U reads candidate j's max and sum,
// which the fold takes by shuffle.
template <int VPL, typename SlotFn>
__device__ __forceinline__ void merge_fold(const MergeArgs& a, SlotFn slot_of, int k0, int k1,
                                           int step, int h, HeadAcc<VPL>& r) {
  constexpr int U = 8 / VPL;
  const int lane = threadIdx.x & 31;
  const int GD = a.CG * a.D;
  const size_t stride = static_cast<size_t>(part_stride(a.CG, a.D));
  r.M = -INFINITY;
  r.den = 0.f;
#pragma unroll
  for (int v = 0; v < VPL; ++v) r.acc[v] = make_float4(0.f, 0.f, 0.f, 0.f);
  const bool on = 4 * lane < a.D;  // D = 64 uses half the lanes
  for (int k = k0; k < k1; k += U * step) {
    float my_m = -INFINITY, my_l = 0.f;
    if (lane < U && k + lane * step < k1) {
      const float* P = a.part + static_cast<size_t>(slot_of(k + lane * step)) * stride;
      my_m = P[GD + h];
      my_l = P[GD + a.CG + h];
    }
    float4 o[U][VPL];
#pragma unroll
    for (int j = 0; j < U; ++j) {
      const int kk = k + j * step;
#pragma unroll
      for (int v = 0; v < VPL; ++v) o[j][v] = make_float4(0.f, 0.f, 0.f, 0.f);
      if (kk < k1 && on) {
        const float* P = a.part + static_cast<size_t>(slot_of(kk)) * stride;
#pragma unroll
        for (int v = 0; v < VPL; ++v)
          o[j][v] = *reinterpret_cast<const float4*>(P + h * a.D + v * 128 + 4 * lane);
      }
    }
#pragma unroll
    for (int j = 0; j < U; ++j) {
      const float mj = __shfl_sync(0xffffffffu, my_m, j), lj = __shfl_sync(0xffffffffu, my_l, j);
      if (k + j * step >= k1) break;
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

// Candidate range of pair (b, kvh): static warps [w0, w0 + na), pool pieces
// [i0, i0 + np).
struct Cands {
  int w0, na, i0, np;
};

__device__ __forceinline__ Cands pair_cands(int F, int nt, int ws, int ts, int piece) {
  Cands c = {0, 0, 0, 0};
  if (nt > 0 && F < ts) {
    c.w0 = F / ws;
    c.na = (min(F + nt, ts) - 1) / ws - c.w0 + 1;
  }
  if (nt > 0 && F + nt > ts) {
    c.i0 = (max(F, ts) - ts) / piece;
    c.np = (F + nt - 1 - ts) / piece - c.i0 + 1;
  }
  return c;
}

// Units: first group 0 of every column (B * Hv * CG of them), then groups 1..
// of the columns of sequences whose candidate bound needs more than one group; the
// latter are enumerated through a prefix over sequences (written by the
// decode kernel), and a unit whose group turns out empty is skipped.
template <int OT, int VPL>
__global__ void __launch_bounds__(kMergeThreads, 3) merge_kernel(const MergeArgs a) {
  extern __shared__ int s_dyn[];
  int* s_pref = s_dyn;             // B + 1 tile prefix
  int* s_extra = s_dyn + a.B + 1;  // B + 1 prefix of extra units per sequence
  griddep_wait();
  const int tid = threadIdx.x, lane = tid & 31;
  if (blockIdx.x == 0 && tid == 0) *a.pool = 0u;
  const int ws = a.ctrl[0], ts = a.ctrl[2], piece = a.ctrl[3];
  for (int i = tid; i <= a.B; i += blockDim.x) {
    s_pref[i] = a.ctrl[4 + i];
    s_extra[i] = a.ctrl[5 + a.B + i];
  }
  __syncthreads();
  const int S = a.B * a.Hv, GD = a.CG * a.D;
  const int HC = a.Hv * a.CG;  // columns per sequence
  const int heads = a.B * HC;
  const int units = heads + s_extra[a.B];
  const int nwarps = gridDim.x * kMergeWarps;
  for (int u = blockIdx.x * kMergeWarps + (tid >> 5); u < units; u += nwarps) {
    int b, col, g;
    if (u < heads) {
      b = u / HC;
      col = u - b * HC;
      g = 0;
    } else {
      const int e = u - heads;
      int lo = 0, hi = a.B;  // largest b with s_extra[b] <= e
      while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (s_extra[mid] <= e) lo = mid; else hi = mid;
      }
      b = lo;
      const int rem = e - s_extra[b];
      g = 1 + rem / HC;
      col = rem - (g - 1) * HC;
    }
    const int vh = col / a.CG, h = col - vh * a.CG;  // pair and column within it
    const int kvh = vh / a.NCG;
    const int gc = (vh - kvh * a.NCG) * a.CG + h;    // column among the kv head's T * G
    if (gc >= a.T * a.G) continue;                    // padding column
    const int tq = gc / a.G;
    const int s = b * a.Hv + vh;
    const int hr = b * HC + col;
    const int nt = s_pref[b + 1] - s_pref[b];
    const int F = a.Hv * s_pref[b] + vh * nt;
    const Cands cd = pair_cands(F, nt, ws, ts, piece);
    const int ncand = cd.na + cd.np;
    const int gsz = merge_group_size(ncand);
    const int ngroups = ncand > 0 ? (ncand + gsz - 1) / gsz : 1;
    if (g >= ngroups) continue;
    const size_t orow =
        ((static_cast<size_t>(b) * a.T + tq) * a.Hq + kvh * a.G + (gc - tq * a.G)) * a.D;
    HeadAcc<VPL> r;
    r.M = -INFINITY;
    r.den = 1.f;
#pragma unroll
    for (int v = 0; v < VPL; ++v) r.acc[v] = make_float4(0.f, 0.f, 0.f, 0.f);
    if (ncand == 0) {
      store_head<OT, VPL>(a, orow, r, true);
      continue;
    }
    auto slot_of = [&](int k) -> int {
      return k < cd.na ? s + cd.w0 + k : S + a.NW + s + cd.i0 + (k - cd.na);
    };
    const int k0 = g * gsz, k1 = min(k0 + gsz, ncand);
    merge_fold(a, slot_of, k0, k1, 1, h, r);
    if (ngroups == 1) {
      store_head<OT, VPL>(a, orow, r, false);
      continue;
    }
    // group result, in place in the slot of the group's first candidate
    {
      float* P = a.part + static_cast<size_t>(slot_of(k0)) * part_stride(a.CG, a.D);
      if (4 * lane < a.D) {
#pragma unroll
        for (int v = 0; v < VPL; ++v)
          *reinterpret_cast<float4*>(P + h * a.D + v * 128 + 4 * lane) = r.acc[v];
      }
      if (lane == 0) {
        P[GD + h] = r.M;
        P[GD + a.CG + h] = r.den;
      }
    }
    // the warp's stores, then lane 0's release increment; the unit that
    // completes the count reads the group results after its acquire (the
    // warp barriers order the other lanes' stores and loads around lane 0's)
    __syncwarp();
    int last = 0;
    if (lane == 0) {
      uint32_t prev;
      asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], 1;"
                   : "=r"(prev)
                   : "l"(a.counters + hr)
                   : "memory");
      last = (prev + 1 == static_cast<uint32_t>(ngroups));
      if (last) a.counters[hr] = 0u;
    }
    last = __shfl_sync(0xffffffffu, last, 0);
    if (!last) continue;
    __syncwarp();
    // combine the group results (the first candidate of each group)
    merge_fold(a, slot_of, 0, ngroups * gsz, gsz, h, r);
    store_head<OT, VPL>(a, orow, r, false);
  }
}

cudaError_t merge_launch(int out_type, const MergeArgs& a, int grid, cudaStream_t s, bool pdl) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kMergeThreads);
  cfg.dynamicSmemBytes = static_cast<size_t>(2 * (a.B + 1)) * sizeof(int);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (a.D > 128) {
    if (out_type == kBF16) return cudaLaunchKernelEx(&cfg, merge_kernel<kBF16, 2>, a);
    return cudaLaunchKernelEx(&cfg, merge_kernel<kF16, 2>, a);
  }
  if (out_type == kBF16) return cudaLaunchKernelEx(&cfg, merge_kernel<kBF16, 1>, a);
  return cudaLaunchKernelEx(&cfg, merge_kernel<kF16, 1>, a);
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
