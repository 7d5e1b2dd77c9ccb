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
// l_p and unnormalised outputs o_p the result is
//   out = sum_p 2^(m_p - M) o_p / sum_p 2^(m_p - M) l_p,  M = max_p m_p.
// Work units are (group g of candidates, pair s, chunk c of 512 (head, dim)
// elements), spread over a persistent grid. A unit combines its group with all
// eight warps (each warp a strided subset, online in registers, then across
// warps in shared memory). A pair whose candidates fit one group is written
// out directly. Otherwise each unit stores its group result, which has the
// same form as a partial, in place in the slot of the group's first
// candidate; the unit that completes the (pair, chunk) counter combines the
// group results and resets the counter. Pairs without tiles get zeros.
constexpr int kMergeThreads = 256;
constexpr int kMergeWarps = kMergeThreads / 32;

struct __align__(16) MergeSmem {
  float M[kMergeWarps][kMergeChunk / 4];
  float den[kMergeWarps][kMergeChunk / 4];
  float acc[kMergeWarps][kMergeChunk];
  int last;
};

// Combines candidates k0, k0 + step, ... (< k1) of one pair for chunk c; on
// return every thread holds the combined (M, den, acc) of its two elements
// el = 2 * tid, 2 * tid + 1 of the chunk (M, den per element's head).
template <typename SlotFn>
__device__ __forceinline__ void merge_combine(const MergeArgs& a, MergeSmem& sm, SlotFn slot_of,
                                              int k0, int k1, int step, int c, float (&rM)[2],
                                              float (&rden)[2], float (&racc)[2]) {
  const int tid = threadIdx.x, wp = tid >> 5, lane = tid & 31;
  const int GD = a.G * a.D;
  const size_t stride = static_cast<size_t>(part_stride(a.G, a.D));
  float M[4], den[4];
  float4 acc[4];
  int eq[4], hq[4];
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    M[q] = -INFINITY;
    den[q] = 0.f;
    acc[q] = make_float4(0.f, 0.f, 0.f, 0.f);
    eq[q] = c * kMergeChunk + q * 128 + lane * 4;
    hq[q] = eq[q] / a.D;
  }
  for (int k = k0 + wp * step; k < k1; k += kMergeWarps * step) {
    const float* P = a.part + static_cast<size_t>(slot_of(k)) * stride;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      if (eq[q] >= GD || eq[q] >= (c + 1) * kMergeChunk) continue;
      const float mm = P[GD + hq[q]], ll = P[GD + a.G + hq[q]];
      const float4 o = *reinterpret_cast<const float4*>(P + eq[q]);
      const float Mn = fmaxf(M[q], mm);
      const float sc = exp2f(M[q] - Mn), f = exp2f(mm - Mn);
      den[q] = den[q] * sc + f * ll;
      acc[q].x = acc[q].x * sc + f * o.x;
      acc[q].y = acc[q].y * sc + f * o.y;
      acc[q].z = acc[q].z * sc + f * o.z;
      acc[q].w = acc[q].w * sc + f * o.w;
      M[q] = Mn;
    }
  }
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    sm.M[wp][q * 32 + lane] = M[q];
    sm.den[wp][q * 32 + lane] = den[q];
    *reinterpret_cast<float4*>(&sm.acc[wp][q * 128 + lane * 4]) = acc[q];
  }
  __syncthreads();
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    const int el = 2 * tid + j, gi = el >> 2;
    float Ms = -INFINITY;
#pragma unroll
    for (int w = 0; w < kMergeWarps; ++w) Ms = fmaxf(Ms, sm.M[w][gi]);
    float d = 0.f, x = 0.f;
#pragma unroll
    for (int w = 0; w < kMergeWarps; ++w) {
      const float f = exp2f(sm.M[w][gi] - Ms);  // 0 for warps without candidates
      d += f * sm.den[w][gi];
      x += f * sm.acc[w][el];
    }
    rM[j] = Ms;
    rden[j] = d;
    racc[j] = x;
  }
  __syncthreads();
}

template <int OT>
__device__ __forceinline__ void store_out2(void* out, size_t idx, float x0, float x1) {
  if constexpr (OT == kBF16) {
    *reinterpret_cast<__nv_bfloat162*>(reinterpret_cast<__nv_bfloat16*>(out) + idx) =
        __floats2bfloat162_rn(x0, x1);
  } else {
    *reinterpret_cast<__half2*>(reinterpret_cast<__half*>(out) + idx) = __floats2half2_rn(x0, x1);
  }
}

template <int OT>
__global__ void __launch_bounds__(kMergeThreads) merge_kernel(const MergeArgs a) {
  extern __shared__ int s_pref[];  // B + 1
  __shared__ MergeSmem sm;
  griddep_wait();
  const int tid = threadIdx.x;
  if (blockIdx.x == 0 && tid == 0) *a.pool = 0u;
  const int ws = a.ctrl[0], ts = a.ctrl[2], piece = a.ctrl[3];
  for (int i = tid; i <= a.B; i += blockDim.x) s_pref[i] = a.ctrl[4 + i];
  __syncthreads();
  const int S = a.B * a.Hkv, GD = a.G * a.D;
  const int nchunk = (GD + kMergeChunk - 1) / kMergeChunk;
  const long long units = static_cast<long long>(kMergeGroupsMax) * S * nchunk;
  for (long long u = blockIdx.x; u < units; u += gridDim.x) {
    const int g = static_cast<int>(u / (static_cast<long long>(S) * nchunk));
    const int r = static_cast<int>(u % (static_cast<long long>(S) * nchunk));
    const int s = r / nchunk, c = r - (r / nchunk) * nchunk;
    const int b = s / a.Hkv, kvh = s - b * a.Hkv;
    const int nt = s_pref[b + 1] - s_pref[b];
    const int F = a.Hkv * s_pref[b] + kvh * nt;
    int w0 = 0, na = 0, i0 = 0, np = 0;
    if (nt > 0 && F < ts) {
      w0 = F / ws;
      na = (min(F + nt, ts) - 1) / ws - w0 + 1;
    }
    if (nt > 0 && F + nt > ts) {
      i0 = (max(F, ts) - ts) / piece;
      np = (F + nt - 1 - ts) / piece - i0 + 1;
    }
    const int ncand = na + np;
    int gsz = (ncand + kMergeGroupsMax - 1) / kMergeGroupsMax;
    if (gsz < kMergeGroupMin) gsz = kMergeGroupMin;
    const int ngroups = ncand > 0 ? (ncand + gsz - 1) / gsz : 1;
    if (g >= ngroups) continue;
    const size_t obase = (static_cast<size_t>(b) * a.Hq + kvh * a.G) * a.D;
    const int e0 = c * kMergeChunk + 2 * tid;
    if (ncand == 0) {
      if (e0 < GD) store_out2<OT>(a.out, obase + e0, 0.f, 0.f);
      continue;
    }
    auto slot_of = [&](int k) -> int {
      return k < na ? s + w0 + k : S + a.NW + s + i0 + (k - na);
    };
    float rM[2], rden[2], racc[2];
    const int k0 = g * gsz, k1 = min(k0 + gsz, ncand);
    merge_combine(a, sm, slot_of, k0, k1, 1, c, rM, rden, racc);
    if (ngroups == 1) {
      if (e0 < GD) store_out2<OT>(a.out, obase + e0, racc[0] / rden[0], racc[1] / rden[1]);
      continue;
    }
    // group result, in place in the slot of the group's first candidate
    {
      const size_t stride = static_cast<size_t>(part_stride(a.G, a.D));
      float* P = a.part + static_cast<size_t>(slot_of(k0)) * stride;
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const int e = e0 + j;
        if (e < GD) {
          P[e] = racc[j];
          if (e % a.D == 0) {
            P[GD + e / a.D] = rM[j];
            P[GD + a.G + e / a.D] = rden[j];
          }
        }
      }
    }
    __threadfence();
    __syncthreads();
    if (tid == 0) {
      const uint32_t done = atomicAdd(a.counters + static_cast<size_t>(s) * nchunk + c, 1u) + 1;
      sm.last = (done == static_cast<uint32_t>(ngroups));
      if (sm.last) a.counters[static_cast<size_t>(s) * nchunk + c] = 0u;
    }
    __syncthreads();
    if (!sm.last) continue;
    __threadfence();
    // combine the group results (first candidate of each group)
    merge_combine(a, sm, slot_of, 0, ngroups * gsz, gsz, c, rM, rden, racc);
    if (e0 < GD) store_out2<OT>(a.out, obase + e0, racc[0] / rden[0], racc[1] / rden[1]);
  }
}

cudaError_t merge_launch(int out_type, const MergeArgs& a, int grid, cudaStream_t s, bool pdl) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kMergeThreads);
  cfg.dynamicSmemBytes = static_cast<size_t>(a.B + 1) * sizeof(int);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (out_type == kBF16) return cudaLaunchKernelEx(&cfg, merge_kernel<kBF16>, a);
  return cudaLaunchKernelEx(&cfg, merge_kernel<kF16>, a);
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
  const dim3 grid(static_cast<unsigned>((n + 127) / 128), 2);
  if (src_type == kBF16) {
    if (fp8) reshape_kernel<kBF16, true><<<grid, 128, 0, s>>>(a);
    else reshape_kernel<kBF16, false><<<grid, 128, 0, s>>>(a);
  } else {
    if (fp8) reshape_kernel<kF16, true><<<grid, 128, 0, s>>>(a);
    else reshape_kernel<kF16, false><<<grid, 128, 0, s>>>(a);
  }
  return cudaGetLastError();
}

}  // namespace pa
