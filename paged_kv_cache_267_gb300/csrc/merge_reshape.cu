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
// One CTA per (pair, q head of the group); each thread owns two head dims.
// The partials of pair s (tiles [F, F + nt) of the flat space) are the static
// slots s + w of the warps w whose static range meets [F, min(F + nt, Ts)),
// and the pool slots S + NW + s + i of the pieces i that meet [max(F, Ts),
// F + nt). With partial maxima m_p (log2 domain), sums l_p and unnormalised
// outputs o_p:
//   out = sum_p 2^(m_p - M) o_p / sum_p 2^(m_p - M) l_p,  M = max_p m_p,
// evaluated in chunks with a running maximum, so any number of partials
// works. A pair with no tiles (seq_len 0) gets zeros. Block (0, 0) also
// resets the pool counter for the next step.
constexpr int kMergeChunk = 256;

template <int OT>
__global__ void __launch_bounds__(128) merge_kernel(const MergeArgs a) {
  __shared__ uint32_t s_slot[kMergeChunk];
  __shared__ float s_fac[kMergeChunk];
  __shared__ float s_M, s_den, s_scale;
  griddep_wait();
  const int s = blockIdx.x, h = blockIdx.y;
  const int b = s / a.Hkv, kvh = s - b * a.Hkv;
  const int tid = threadIdx.x;
  const int d = 2 * tid;
  if (s == 0 && h == 0 && tid == 0) *a.pool = 0u;
  const size_t orow = (static_cast<size_t>(b) * a.Hq + kvh * a.G + h) * a.D + d;
  const int ws = a.ctrl[0], ts = a.ctrl[2], piece = a.ctrl[3];
  const int pb = a.ctrl[4 + b], nt = a.ctrl[5 + b] - pb;
  const int S = a.B * a.Hkv;
  float n0 = 0.f, n1 = 0.f, r0 = 0.f, r1 = 0.f;
  if (nt > 0) {
    const int F = a.Hkv * pb + kvh * nt;
    // candidate slots: static warps [w0, w1], then pool pieces [i0, i1]
    int w0 = 0, w1 = -1, i0 = 0, i1 = -1;
    if (F < ts) {
      w0 = F / ws;
      w1 = (min(F + nt, ts) - 1) / ws;
    }
    if (F + nt > ts) {
      i0 = (max(F, ts) - ts) / piece;
      i1 = (F + nt - 1 - ts) / piece;
    }
    const int na = w1 - w0 + 1, np = i1 - i0 + 1, ntot = na + np;
    const size_t stride = static_cast<size_t>(a.G) * (a.D + 2);
    const int mo = a.G * a.D + h, lo = a.G * a.D + a.G + h;
    if (tid == 0) {
      s_M = -INFINITY;
      s_den = 0.f;
    }
    for (int c0 = 0; c0 < ntot; c0 += kMergeChunk) {
      const int n = min(kMergeChunk, ntot - c0);
      for (int i = tid; i < n; i += blockDim.x) {
        const int k = c0 + i;
        s_slot[i] = (k < na) ? static_cast<uint32_t>(s + w0 + k)
                             : static_cast<uint32_t>(S + a.NW + s + i0 + (k - na));
      }
      __syncthreads();
      if (tid < 32) {
        float mx = -INFINITY;
        for (int i = tid; i < n; i += 32) mx = fmaxf(mx, a.part[s_slot[i] * stride + mo]);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
        const float Mn = fmaxf(s_M, mx);
        float den = 0.f;
        for (int i = tid; i < n; i += 32) {
          const float* P = a.part + s_slot[i] * stride;
          const float fct = exp2f(P[mo] - Mn);
          s_fac[i] = fct;
          den += fct * P[lo];
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) den += __shfl_xor_sync(0xffffffffu, den, o);
        if (tid == 0) {
          const float sc = exp2f(s_M - Mn);  // 0 on the first chunk
          s_scale = sc;
          s_den = s_den * sc + den;
          s_M = Mn;
        }
      }
      __syncthreads();
      if (d < a.D) {
        const float sc = s_scale;
        n0 *= sc;
        n1 *= sc;
        for (int i = 0; i < n; ++i) {
          const float2 o =
              *reinterpret_cast<const float2*>(a.part + s_slot[i] * stride + h * a.D + d);
          n0 += s_fac[i] * o.x;
          n1 += s_fac[i] * o.y;
        }
      }
      __syncthreads();
    }
    const float den = s_den;
    r0 = n0 / den;
    r1 = n1 / den;
  }
  if (d >= a.D) return;
  if constexpr (OT == kBF16) {
    *reinterpret_cast<__nv_bfloat162*>(reinterpret_cast<__nv_bfloat16*>(a.out) + orow) =
        __floats2bfloat162_rn(r0, r1);
  } else {
    *reinterpret_cast<__half2*>(reinterpret_cast<__half*>(a.out) + orow) =
        __floats2half2_rn(r0, r1);
  }
}

cudaError_t merge_launch(int out_type, const MergeArgs& a, cudaStream_t s, bool pdl) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.B * a.Hkv, a.G);
  cfg.blockDim = dim3((a.D / 2 + 31) / 32 * 32);
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
