// Tensor-memory kernel for chunked causal queries over the paged cache
// (the chunked-prefill step of "vLLM 0.5 深度解析" §5.2; the attention itself
// is the block-wise scaled dot product with a running max/sum of §2.3 of
// the same page), on the 5th-generation tensor cores of sm_103a.
//
// Work unit: one (sequence b, KV head, tile of 128 (query, head) rows), the
// rows being r = t * G + h over the chunk's T queries and the group's G
// heads: one CTA each. The unit's read range is the union of its rows'
// ranges, [lo, hi] with lo the first row's window start and hi the last
// row's position; it is walked in K/V tiles of 64 tokens (four 16-token
// slices, each inside one physical block, fetched by TMA through the block
// table).
//
// Per K/V tile n, with one control warp and four softmax warps (one row per
// thread):
//   control : S = Q . K_n^T           tcgen05.mma M128 N64  K128 -> TMEM
//   softmax : S from TMEM; per-row causal/window mask; online softmax in the
//             log2 domain; P (16-bit) -> shared memory, 128-byte swizzle
//   control : O_n = P . V_n           tcgen05.mma M128 N128 K64  -> TMEM
//             (V MN-major: its rows are tokens, head dims contiguous)
//   softmax : O = alpha O + O_n in registers
// Q (128 rows x 128 dims) stays in shared memory for the whole unit; K/V
// tiles stream through a three-stage ring; the control warp issues S_{n+1}
// while the softmax warps fold O_n. V rows of an edge tile that lie outside
// [lo, hi] (not loaded, or NaN-poisoned slots past the sequence or before
// the window) are zeroed in shared memory before the P . V product, so only
// attended rows reach the tensor core. Head dim 128, f16 or bf16 caches.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "pa_internal.h"
#include "ptx.cuh"
#include "tc.cuh"

namespace pa {
namespace {

constexpr int kRows = 128;      // (query, head) rows per unit: the MMA M
constexpr int kKv = 64;         // tokens per K/V tile
constexpr int kHd = 128;        // head dim
constexpr int kStages = 3;      // K/V ring depth
constexpr int kSoftWarps = 4;
constexpr int kThreads = (kSoftWarps + 1) * 32;
constexpr uint32_t kQBytes = kRows * kHd * 2;   // [2 boxes][128 rows][128 B]
constexpr uint32_t kKvBytes = kKv * kHd * 2;    // [2 boxes][64 rows][128 B]
constexpr uint32_t kPBytes = kRows * kKv * 2;   // [128 rows][128 B]
constexpr uint32_t kOffQ = 0;
constexpr uint32_t kOffK = kOffQ + kQBytes;
constexpr uint32_t kOffV = kOffK + kStages * kKvBytes;
constexpr uint32_t kOffP = kOffV + kStages * kKvBytes;
constexpr uint32_t kOffBar = kOffP + kPBytes;
constexpr int kBarFull = 0, kBarEmpty = kStages, kBarS = 2 * kStages, kBarP = kBarS + 1,
              kBarO = kBarS + 2, kBarQ = kBarS + 3, kNumBars = kBarS + 4;
constexpr uint32_t kOffSlot = kOffBar + 8 * kNumBars;
constexpr uint32_t kSmemBytes = kOffSlot + 16 + 1024;  // + room to align the base to 1 KB
constexpr uint32_t kTmemCols = 256;                    // S: columns [0, 64); O_n: [128, 256)
constexpr uint32_t kColS = 0, kColO = 128;
constexpr uint64_t kWaitNs = 2000000000ull;            // bound of every wait (2 s)
constexpr float kFloor = -1e30f;                       // running-max start
constexpr unsigned kFull = 0xffffffffu;

__device__ __forceinline__ void sts_v4(uint32_t addr, uint4 v) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(v.x), "r"(v.y),
               "r"(v.z), "r"(v.w)
               : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
template <bool BF16>
__device__ __forceinline__ uint32_t pack16x2(float lo, float hi) {
  if constexpr (BF16) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
  } else {
    __half2 v = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
  }
}
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

template <int QT>
__global__ void __launch_bounds__(kThreads, 1)
    chunk_attn_tc_kernel(const __grid_constant__ CUtensorMap tmK,
                         const __grid_constant__ CUtensorMap tmV, const ChunkArgs a) {
  constexpr bool kBf16 = QT == kBF16;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_addr(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  const uint32_t sQ = base + kOffQ, sK = base + kOffK, sV = base + kOffV, sP = base + kOffP;
  auto bar = [&](int i) -> uint32_t { return base + kOffBar + 8u * i; };
  const uint32_t* tslot = reinterpret_cast<const uint32_t*>(smem_raw + (base - raw) + kOffSlot);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int qt = blockIdx.x % a.QT;
  const int kvh = (blockIdx.x / a.QT) % a.Hkv;
  const int b = blockIdx.x / (a.QT * a.Hkv);

  if (tid == 0) {
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
    for (int i = 0; i < kStages; ++i) {
      mbar_init(bar(kBarFull + i), 1);
      mbar_init(bar(kBarEmpty + i), 1);
    }
    mbar_init(bar(kBarS), 1);
    mbar_init(bar(kBarP), kSoftWarps * 32);
    mbar_init(bar(kBarO), 1);
    mbar_init(bar(kBarQ), kSoftWarps * 32);
    fence_mbar_init();
  }
  if (warp == 0) tc::tmem_alloc(base + kOffSlot, kTmemCols);
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *tslot;
  griddep_wait();
  griddep_launch_dependents();

  // the unit's rows and read range
  const int cap = a.MB * a.bs;
  int L = a.seq_lens[b];
  if (L < 0 || L > cap) {
    if (tid == 0) atomicOr(a.err, PA_DEVERR_SEQ_LEN);
    L = L < 0 ? 0 : cap;
  }
  const int r0 = qt * kRows;
  const int r1 = min(r0 + kRows, a.T * a.G);  // valid rows [r0, r1)
  const int p_first = L - a.T + r0 / a.G;
  const int hi = L - a.T + (r1 - 1) / a.G;    // last position read
  const int lo = (a.window > 0 && p_first + 1 > a.window) ? p_first + 1 - a.window : 0;
  const int lo16 = lo & ~15;
  const int ntiles = hi >= lo ? (hi + 1 - lo16 + kKv - 1) / kKv : 0;

  if (warp == kSoftWarps) {
    // ------------------------------------------------------------ control
    // Loads K/V tile n into `stage`: lanes 0..3 each look up one 16-token
    // slice in the block table and copy it (two 64-dim boxes of K and of V).
    auto load_tile = [&](int n, int stage) {
      const int pos0 = lo16 + n * kKv + 16 * lane;
      int row = -1;
      if (lane < 4 && pos0 <= hi) {
        int blk = __ldg(a.block_tables + static_cast<size_t>(b) * a.MB + pos0 / a.bs);
        if (static_cast<unsigned>(blk) >= static_cast<unsigned>(a.NB)) {
          atomicOr(a.err, PA_DEVERR_BLOCK_ID);
          blk = 0;
        }
        row = (blk * a.Hkv + kvh) * a.bs + pos0 % a.bs;
      }
      const int nslices = __popc(__ballot_sync(kFull, row >= 0));
      if (lane == 0) mbar_arrive_expect_tx(bar(kBarFull + stage), nslices * 4 * 2048);
      __syncwarp();
      if (row >= 0) {
        const uint32_t kd = sK + stage * kKvBytes + lane * 2048;
        const uint32_t vd = sV + stage * kKvBytes + lane * 2048;
#pragma unroll
        for (int box = 0; box < 2; ++box) {
          tma_load_2d(kd + box * 8192, &tmK, box * 64, row, bar(kBarFull + stage));
          tma_load_2d(vd + box * 8192, &tmV, box * 64, row, bar(kBarFull + stage));
        }
      }
      __syncwarp();
    };
    constexpr uint32_t idS = tc::idesc_f16(kRows, kKv, kBf16, false);
    constexpr uint32_t idO = tc::idesc_f16(kRows, kHd, kBf16, true);
    // S = Q . K_n^T over the 128 head dims (8 steps of 16)
    auto issue_s = [&](int n) {
      const int st = n % kStages;
      if (lane == 0) {
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
          const uint32_t box = ks >> 2, kk = (ks & 3) * 32;
          const uint64_t ad = tc::sdesc_sw128(sQ + box * 16384 + kk, 16, 1024);
          const uint64_t bd = tc::sdesc_sw128(sK + st * kKvBytes + box * 8192 + kk, 16, 1024);
          tc::mma_f16(tmem + kColS, ad, bd, idS, ks > 0);
        }
        tc::commit(bar(kBarS));
      }
      __syncwarp();
    };
    bool ok = true;
    for (int i = 0; i < kStages && i < ntiles; ++i) load_tile(i, i);
    if (ntiles > 0) {
      ok = __all_sync(kFull, mbar_wait_bounded(bar(kBarQ), 0, kWaitNs)) &&
           __all_sync(kFull, mbar_wait_bounded(bar(kBarFull), 0, kWaitNs));
      if (ok) {
        tc::fence_after_sync();
        issue_s(0);
      }
    }
    for (int n = 0; ok && n < ntiles; ++n) {
      const int st = n % kStages;
      // P_n written (and V_n cleaned) by the softmax warps
      ok = __all_sync(kFull, mbar_wait_bounded(bar(kBarP), n & 1, kWaitNs));
      if (!ok) break;
      tc::fence_after_sync();
      if (lane == 0) {
#pragma unroll
        for (int ks = 0; ks < 4; ++ks) {  // O_n = P . V_n over 64 tokens (4 steps of 16)
          const uint64_t ad = tc::sdesc_sw128(sP + ks * 32, 16, 1024);
          const uint64_t bd = tc::sdesc_sw128(sV + st * kKvBytes + ks * 2048, 8192, 1024);
          tc::mma_f16(tmem + kColO, ad, bd, idO, ks > 0);
        }
        tc::commit(bar(kBarO));
        tc::commit(bar(kBarEmpty + st));
      }
      __syncwarp();
      if (n + 1 < ntiles) {
        ok = __all_sync(kFull, mbar_wait_bounded(bar(kBarFull + (n + 1) % kStages),
                                                 ((n + 1) / kStages) & 1, kWaitNs));
        if (!ok) break;
        tc::fence_after_sync();
        issue_s(n + 1);
      }
      if (n + kStages < ntiles) {
        ok = __all_sync(kFull, mbar_wait_bounded(bar(kBarEmpty + st), (n / kStages) & 1, kWaitNs));
        if (!ok) break;
        load_tile(n + kStages, st);
      }
    }
    if (!ok && lane == 0) atomicOr(a.err, PA_DEVERR_TIMEOUT);
  } else {
    // ------------------------------------------------------------ softmax
    const int r = tid;  // row of the unit = tensor-memory lane
    const int gr = r0 + r;
    const bool valid = gr < r1;
    const int tq = valid ? gr / a.G : 0;
    const int hq = gr - tq * a.G;
    const int hi_r = valid ? L - a.T + tq : -1;  // this row's query position
    const int lo_r = (a.window > 0 && hi_r + 1 > a.window) ? hi_r + 1 - a.window : 0;
    const size_t orow =
        ((static_cast<size_t>(b) * a.T + tq) * a.Hq + static_cast<size_t>(kvh) * a.G + hq) * kHd;
    {  // Q row -> shared memory (K-major, 128-byte swizzle)
      const uint4* src = reinterpret_cast<const uint4*>(reinterpret_cast<const uint16_t*>(a.q) + orow);
#pragma unroll
      for (int c = 0; c < 16; ++c) {
        const uint4 x = valid ? src[c] : make_uint4(0u, 0u, 0u, 0u);
        sts_v4(sQ + (c >> 3) * 16384 + r * 128 + (((c & 7) ^ (r & 7)) << 4), x);
      }
      fence_proxy_async();
      mbar_arrive(bar(kBarQ));
    }
    const uint32_t trow = tmem + (static_cast<uint32_t>(warp * 32) << 16);
    float m = kFloor, l = 0.f;
    float o[kHd];
#pragma unroll
    for (int i = 0; i < kHd; ++i) o[i] = 0.f;
    bool ok = true;
    for (int n = 0; n < ntiles; ++n) {
      const int st = n % kStages;
      const int t0 = lo16 + n * kKv;  // position of the tile's first token
      ok = __all_sync(kFull, mbar_wait_bounded(bar(kBarS), n & 1, kWaitNs));
      if (!ok) break;
      tc::fence_after_sync();
      float s[kKv];
      tc::ld32(trow + kColS, s);
      tc::ld32(trow + kColS + 32, s + 32);
      const bool inside = t0 >= lo_r && t0 + kKv - 1 <= hi_r;
      float mx = kFloor;
#pragma unroll
      for (int j = 0; j < kKv; ++j) {
        const bool keep = inside || (t0 + j >= lo_r && t0 + j <= hi_r);
        s[j] = keep ? s[j] * a.score_scale : -INFINITY;
        mx = fmaxf(mx, s[j]);
      }
      const float m_new = fmaxf(m, mx);
      const float alpha = ex2(m - m_new);
      float sum = 0.f;
      uint32_t pk[kKv / 2];
#pragma unroll
      for (int j = 0; j < kKv / 2; ++j) {
        const float p0 = ex2(s[2 * j] - m_new), p1 = ex2(s[2 * j + 1] - m_new);
        sum += p0 + p1;
        pk[j] = pack16x2<kBf16>(p0, p1);
      }
      l = l * alpha + sum;
      m = m_new;
      if (t0 < lo || t0 + kKv - 1 > hi) {
        // edge tile: once it has landed, zero the V rows outside [lo, hi]
        ok = __all_sync(kFull, mbar_wait_bounded(bar(kBarFull + st), (n / kStages) & 1, kWaitNs));
        if (!ok) break;
        for (int i = r; i < kKv * 16; i += kSoftWarps * 32) {
          const int row = i >> 4, box = (i >> 3) & 1, ch = i & 7;
          const int pos = t0 + row;
          if (pos < lo || pos > hi)
            sts_v4(sV + st * kKvBytes + box * 8192 + row * 128 + ch * 16, make_uint4(0u, 0u, 0u, 0u));
        }
      }
#pragma unroll
      for (int c = 0; c < 8; ++c)
        sts_v4(sP + r * 128 + ((c ^ (r & 7)) << 4),
               make_uint4(pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]));
      fence_proxy_async();  // P and the cleaned V rows, visible to the tensor core
      tc::fence_before_sync();
      mbar_arrive(bar(kBarP));
      ok = __all_sync(kFull, mbar_wait_bounded(bar(kBarO), n & 1, kWaitNs));
      if (!ok) break;
      tc::fence_after_sync();
#pragma unroll
      for (int c0 = 0; c0 < kHd; c0 += 32) {
        float ot[32];
        tc::ld32(trow + kColO + c0, ot);
#pragma unroll
        for (int i = 0; i < 32; ++i) o[c0 + i] = o[c0 + i] * alpha + ot[i];
      }
    }
    if (!ok && lane == 0) atomicOr(a.err, PA_DEVERR_TIMEOUT);
    if (valid) {
      const float inv = l > 0.f ? 1.f / l : 0.f;
      uint4* dst = reinterpret_cast<uint4*>(reinterpret_cast<uint16_t*>(a.out) + orow);
#pragma unroll
      for (int c = 0; c < 16; ++c)
        dst[c] = make_uint4(pack16x2<kBf16>(o[8 * c] * inv, o[8 * c + 1] * inv),
                            pack16x2<kBf16>(o[8 * c + 2] * inv, o[8 * c + 3] * inv),
                            pack16x2<kBf16>(o[8 * c + 4] * inv, o[8 * c + 5] * inv),
                            pack16x2<kBf16>(o[8 * c + 6] * inv, o[8 * c + 7] * inv));
    }
  }

  // every MMA has completed (the softmax warps waited for the last one)
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 0) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, kTmemCols);
  }
}

template <int QT>
cudaError_t launch_typed(const CUtensorMap& tk, const CUtensorMap& tv, const ChunkArgs& a,
                         int grid, cudaStream_t s, bool pdl) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, chunk_attn_tc_kernel<QT>, tk, tv, a);
}

}  // namespace

cudaError_t chunk_tc_prepare() {
  cudaError_t e = cudaFuncSetAttribute(chunk_attn_tc_kernel<kBF16>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(chunk_attn_tc_kernel<kF16>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
}

cudaError_t chunk_tc_launch(int qt, const CUtensorMap& tk, const CUtensorMap& tv,
                            const ChunkArgs& a, cudaStream_t s, bool pdl) {
  const long long grid = static_cast<long long>(a.B) * a.Hkv * a.QT;
  if (grid <= 0) return cudaSuccess;
  if (grid > 0x7fffffffLL) return cudaErrorInvalidValue;
  return qt == kBF16 ? launch_typed<kBF16>(tk, tv, a, static_cast<int>(grid), s, pdl)
                     : launch_typed<kF16>(tk, tv, a, static_cast<int>(grid), s, pdl);
}

}  // namespace pa
