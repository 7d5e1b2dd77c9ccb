// Tensor-memory kernel for chunked causal queries over an FP8 e4m3 paged
// cache, 64-token K/V tiles (16-bit caches take the 128-token kernel of
// chunk_tc.cu; this one is instantiated with FP8 = true only). The
// chunked-prefill step of "vLLM 0.5 深度解析" §5.2; the attention itself
// is the block-wise scaled dot product with a running max/sum of §2.3 of
// the same page), on the 5th-generation tensor cores of sm_103a.
//
// Work unit: one (sequence b, KV head, 256 (query, head) rows), the rows
// being r = t * G + h over the chunk's T queries and the group's G heads: one
// CTA each, holding two 128-row tiles A and B. The unit's read range is the
// union of its rows' ranges, [lo, hi] with lo the first row's window start
// and hi the last row's position; it is walked in K/V tiles of 64 tokens
// (four 16-token slices, each inside one physical block, fetched by TMA
// through the block table), each shared by both row tiles.
//
// Roles: a producer warp streams K/V tiles through a three-stage ring (block
// table lookups and TMA), an MMA warp issues every product, and two groups
// of four softmax warps (one row per thread)
// serve tiles A and B, so the tensor core works for one group while the
// other runs its softmax. Per K/V tile n and row tile X:
//   S_X  = Q_X . K_n^T        tcgen05.mma M128 N64  K128 -> TMEM
//   softmax X: S_X from TMEM; per-row causal/window mask; online softmax in
//          the log2 domain against the row's reference max m; P_X (16-bit,
//          packed in pairs) -> tensor memory
//   O_X += P_X . V_n          tcgen05.mma M128 N128 K64, A = P_X from TMEM,
//                             B = V_n (MN-major) -> TMEM
// The output accumulates in tensor memory. A row's reference max moves only
// when its running max exceeds it by more than 8 (log2 units); the warp then
// rescales those rows of O_X in tensor memory (load, scale, store) before the
// next product, so P stays below 2^8 and most tiles never touch O. V rows of
// an edge tile that lie outside [lo, hi] (not loaded, or NaN-poisoned slots
// past the sequence or before the window) are zeroed in shared memory before
// the products, so only attended rows reach the tensor core. Head dim 128.
//
// FP8 e4m3 caches (FP8 = true): the ring holds the raw e4m3 tiles (8 KB of K
// and of V per tile), and two converter warps turn each into f16 tiles of the
// same swizzled layouts (exact), in a double buffer the products read; they
// write zeros for the V rows outside [lo, hi]. Q is converted per row to f16
// after a power-of-two rescale that brings its largest magnitude into
// [2^14, 2^15); the rescale and k_scale fold into the row's score scale, and
// v_scale is applied to the output.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "pa_internal.h"
#include "ptx.cuh"
#include "tc.cuh"

namespace pa {
namespace {

constexpr int kRows = 128;      // rows per row tile: the MMA M
constexpr int kUnitRows = 2 * kRows;
constexpr int kKv = 64;         // tokens per K/V tile
constexpr int kHd = 128;        // head dim
constexpr int kStages = 3;      // K/V ring depth
constexpr int kGroupWarps = 4;  // softmax warps per row tile
constexpr int kCtrlWarp = 2 * kGroupWarps;  // issues the MMAs
constexpr int kLoadWarp = kCtrlWarp + 1;     // streams K/V tiles
constexpr int kConvWarp0 = kLoadWarp + 1;    // FP8: e4m3 -> f16 converters
constexpr int kConvWarps = 2;
constexpr uint32_t kQBytes = kRows * kHd * 2;   // per row tile: [2 boxes][128 rows][128 B]
constexpr uint32_t kKvBytes = kKv * kHd * 2;    // 16-bit tile: [2 boxes][64 rows][128 B]
constexpr uint32_t kRawBytes = kKv * kHd;       // e4m3 tile: [64 rows][128 B]
constexpr int kBarFull = 0, kBarEmpty = kStages, kBarS = 2 * kStages,  // S_A, S_B
    kBarP = kBarS + 2, kBarO = kBarS + 4, kBarQ = kBarS + 6,
    kBarCFull = kBarS + 7, kBarCEmpty = kBarS + 9,  // FP8: converted buffers 0, 1
    kNumBars = kBarS + 11;

// Shared-memory layout: Q_A, Q_B, the ring, (FP8: the converted double
// buffer of K and V), barriers, the tensor-memory address.
template <bool FP8>
struct Smem {
  static constexpr uint32_t kThreads = (kConvWarp0 + (FP8 ? kConvWarps : 0)) * 32;
  static constexpr uint32_t kTileK = FP8 ? kRawBytes : kKvBytes;  // one ring tile of K (or V)
  static constexpr uint32_t kQ = 0;
  static constexpr uint32_t kK = kQ + 2 * kQBytes;               // ring: K tiles
  static constexpr uint32_t kV = kK + kStages * kTileK;          // ring: V tiles
  static constexpr uint32_t kKc = kV + kStages * kTileK;         // FP8: f16 K tiles [2]
  static constexpr uint32_t kVc = kKc + (FP8 ? 2 * kKvBytes : 0);
  static constexpr uint32_t kBar = kVc + (FP8 ? 2 * kKvBytes : 0);
  static constexpr uint32_t kSlot = kBar + 8 * kNumBars;
  static constexpr uint32_t kBytes = kSlot + 16 + 1024;  // + room to align the base to 1 KB
};
// tensor memory: S_A [0,64) S_B [64,128) O_A [128,256) O_B [256,384)
// P_A [384,416) P_B [416,448)
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColS = 0, kColO = 128, kColP = 384;
constexpr uint64_t kWaitNs = 2000000000ull;  // bound of every wait (2 s)
constexpr float kFloor = -1e30f;             // reference-max start
constexpr float kRescaleAbove = 8.f;         // log2 units
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
__device__ __forceinline__ bool wait_all(uint32_t bar, uint32_t parity) {
  return __all_sync(kFull, mbar_wait_bounded(bar, parity, kWaitNs));
}

template <int QT, bool FP8>
__global__ void __launch_bounds__(Smem<FP8>::kThreads, 1)
    chunk_attn_tc_kernel(const __grid_constant__ CUtensorMap tmK,
                         const __grid_constant__ CUtensorMap tmV, const ChunkArgs a) {
  using SL = Smem<FP8>;
  // operand type of the products: the q type, or f16 for FP8 caches
  constexpr bool kBf16 = !FP8 && QT == kBF16;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_addr(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  const uint32_t sQ = base + SL::kQ, sK = base + SL::kK, sV = base + SL::kV;
  const uint32_t sKc = base + SL::kKc, sVc = base + SL::kVc;
  auto bar = [&](int i) -> uint32_t { return base + SL::kBar + 8u * i; };
  const uint32_t* tslot = reinterpret_cast<const uint32_t*>(smem_raw + (base - raw) + SL::kSlot);
  // the f16/bf16 K and V tiles the products read for K/V tile n
  auto tile_k = [&](int n) -> uint32_t {
    return FP8 ? sKc + (n & 1) * kKvBytes : sK + (n % kStages) * kKvBytes;
  };
  auto tile_v = [&](int n) -> uint32_t {
    return FP8 ? sVc + (n & 1) * kKvBytes : sV + (n % kStages) * kKvBytes;
  };
  // barrier (and parity) that says tile n is ready for the products
  auto ready_bar = [&](int n) -> uint32_t { return FP8 ? bar(kBarCFull + (n & 1)) : bar(kBarFull + n % kStages); };
  auto ready_par = [&](int n) -> uint32_t { return FP8 ? (n >> 1) & 1 : (n / kStages) & 1; };

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int ut = blockIdx.x % a.QT;  // unit (256 rows) within the (sequence, KV head)
  const int kvh = (blockIdx.x / a.QT) % a.Hkv;
  const int b = blockIdx.x / (a.QT * a.Hkv);

  if (tid == 0) {
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
    for (int i = 0; i < kStages; ++i) {
      mbar_init(bar(kBarFull + i), 1);
      // freed by the products' commit, or (FP8) by the converters
      mbar_init(bar(kBarEmpty + i), FP8 ? kConvWarps * 32 : 1);
    }
    for (int x = 0; x < 2; ++x) {
      mbar_init(bar(kBarS + x), 1);
      mbar_init(bar(kBarP + x), kGroupWarps * 32);
      mbar_init(bar(kBarO + x), 1);
    }
    mbar_init(bar(kBarQ), 2 * kGroupWarps * 32);
    if constexpr (FP8) {
      for (int j = 0; j < 2; ++j) {
        mbar_init(bar(kBarCFull + j), kConvWarps * 32);
        mbar_init(bar(kBarCEmpty + j), 1);
      }
    }
    fence_mbar_init();
  }
  if (warp == 0) tc::tmem_alloc(base + SL::kSlot, kTmemCols);
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
  const int nrows = a.T * a.G;
  const int r0 = ut * kUnitRows;
  const int r1 = min(r0 + kUnitRows, nrows);  // valid rows [r0, r1)
  const bool hasB = r0 + kRows < r1;
  const int p_first = L - a.T + r0 / a.G;
  const int hi = L - a.T + (r1 - 1) / a.G;  // last position read
  const int lo = (a.window > 0 && p_first + 1 > a.window) ? p_first + 1 - a.window : 0;
  const int lo16 = lo & ~15;
  const int ntiles = hi >= lo ? (hi + 1 - lo16 + kKv - 1) / kKv : 0;

  if (warp == kLoadWarp) {
    // ------------------------------------------------------------ producer
    // Loads K/V tile n into `stage`: lanes 0..3 each look up one 16-token
    // slice in the block table and copy it (16-bit: two 64-dim boxes of K and
    // of V; e4m3: one 128-dim box each).
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
      if (lane == 0)
        mbar_arrive_expect_tx(bar(kBarFull + stage), nslices * (FP8 ? 2 : 4) * 2048);
      __syncwarp();
      if (row >= 0) {
        const uint32_t kd = sK + stage * SL::kTileK + lane * 2048;
        const uint32_t vd = sV + stage * SL::kTileK + lane * 2048;
        if constexpr (FP8) {
          tma_load_2d(kd, &tmK, 0, row, bar(kBarFull + stage));
          tma_load_2d(vd, &tmV, 0, row, bar(kBarFull + stage));
        } else {
#pragma unroll
          for (int box = 0; box < 2; ++box) {
            tma_load_2d(kd + box * 8192, &tmK, box * 64, row, bar(kBarFull + stage));
            tma_load_2d(vd + box * 8192, &tmV, box * 64, row, bar(kBarFull + stage));
          }
        }
      }
      __syncwarp();
    };
    bool ok = true;
    for (int n = 0; n < ntiles; ++n) {
      const int st = n % kStages;
      if (n >= kStages && !(ok = wait_all(bar(kBarEmpty + st), ((n - kStages) / kStages) & 1)))
        break;
      load_tile(n, st);
    }
    if (!ok && lane == 0) atomicOr(a.err, PA_DEVERR_TIMEOUT);
  } else if (warp == kCtrlWarp) {
    // ------------------------------------------------------------ MMA issue
    constexpr uint32_t idS = tc::idesc_f16(kRows, kKv, kBf16, false);
    constexpr uint32_t idO = tc::idesc_f16(kRows, kHd, kBf16, true);
    // S_X = Q_X . K_n^T over the 128 head dims (8 steps of 16)
    auto issue_s = [&](int x, int n) {
      if (lane == 0) {
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
          const uint32_t box = ks >> 2, kk = (ks & 3) * 32;
          const uint64_t ad = tc::sdesc_sw128(sQ + x * kQBytes + box * 16384 + kk, 16, 1024);
          const uint64_t bd = tc::sdesc_sw128(tile_k(n) + box * 8192 + kk, 16, 1024);
          tc::mma_f16(tmem + kColS + 64 * x, ad, bd, idS, ks > 0);
        }
        tc::commit(bar(kBarS + x));
      }
      __syncwarp();
    };
    // O_X (+)= P_X . V_n over 64 tokens (4 steps of 16); P_X in tensor
    // memory, 8 columns (16 tokens) per step
    auto issue_o = [&](int x, int n) {
      if (lane == 0) {
#pragma unroll
        for (int ks = 0; ks < 4; ++ks) {
          const uint64_t bd = tc::sdesc_sw128(tile_v(n) + ks * 2048, 8192, 1024);
          tc::mma_f16_ta(tmem + kColO + 128 * x, tmem + kColP + 32 * x + 8 * ks, bd, idO,
                         (n > 0 || ks > 0) ? 1u : 0u);
        }
        tc::commit(bar(kBarO + x));
      }
      __syncwarp();
    };
    bool ok = true;
    if (ntiles > 0) {
      ok = wait_all(bar(kBarQ), 0) && wait_all(ready_bar(0), ready_par(0));
      if (ok) {
        tc::fence_after_sync();
        issue_s(0, 0);
        if (hasB) issue_s(1, 0);
      }
    }
    for (int n = 0; ok && n < ntiles; ++n) {
      const int st = n % kStages;
      const bool more = n + 1 < ntiles;
      if (!(ok = wait_all(bar(kBarP), n & 1))) break;  // P_A(n) written, V_n cleaned
      tc::fence_after_sync();
      issue_o(0, n);
      if (more) {
        if (!(ok = wait_all(ready_bar(n + 1), ready_par(n + 1)))) break;
        tc::fence_after_sync();
        issue_s(0, n + 1);
      }
      if (hasB) {
        if (!(ok = wait_all(bar(kBarP + 1), n & 1))) break;
        tc::fence_after_sync();
        issue_o(1, n);
      }
      // both products of tile n issued: its ring stage (FP8: converted buffer)
      // is free once they complete
      if (lane == 0) tc::commit(FP8 ? bar(kBarCEmpty + (n & 1)) : bar(kBarEmpty + st));
      __syncwarp();
      if (hasB && more) issue_s(1, n + 1);
    }
    if (!ok && lane == 0) atomicOr(a.err, PA_DEVERR_TIMEOUT);
  } else if (warp >= kConvWarp0) {
    // ------------------------------------------------------------ FP8 converters
    // e4m3 tile n (ring stage n % kStages) -> f16 tiles in converted buffer
    // n & 1: each 16-byte chunk of 16 e4m3 codes becomes two 16-byte chunks
    // of f16 in the 64-dim box that holds them; V rows outside [lo, hi] are
    // written as zeros.
    if constexpr (FP8) {
      const int ct = tid - kConvWarp0 * 32;
      bool ok = true;
      for (int n = 0; n < ntiles; ++n) {
        const int st = n % kStages, cb = n & 1;
        const int t0 = lo16 + n * kKv;
        if (!(ok = wait_all(bar(kBarFull + st), (n / kStages) & 1))) break;
        if (n >= 2 && !(ok = wait_all(bar(kBarCEmpty + cb), ((n - 2) >> 1) & 1))) break;
        for (int i = ct; i < 2 * kKv * 8; i += kConvWarps * 32) {
          const bool is_v = i >= kKv * 8;
          const int j = i & (kKv * 8 - 1), row = j >> 3, c = j & 7;
          const uint32_t src = (is_v ? sV : sK) + st * kRawBytes + row * 128 + ((c ^ (row & 7)) << 4);
          uint4 lo4 = make_uint4(0u, 0u, 0u, 0u), hi4 = lo4;
          const int pos = t0 + row;
          if (!is_v || (pos >= lo && pos <= hi)) {
            uint32_t w0, w1, w2, w3;
            lds_v4(src, w0, w1, w2, w3);
            lo4 = make_uint4(e4m3x2_to_f16x2(static_cast<uint16_t>(w0 & 0xffffu)),
                             e4m3x2_to_f16x2(static_cast<uint16_t>(w0 >> 16)),
                             e4m3x2_to_f16x2(static_cast<uint16_t>(w1 & 0xffffu)),
                             e4m3x2_to_f16x2(static_cast<uint16_t>(w1 >> 16)));
            hi4 = make_uint4(e4m3x2_to_f16x2(static_cast<uint16_t>(w2 & 0xffffu)),
                             e4m3x2_to_f16x2(static_cast<uint16_t>(w2 >> 16)),
                             e4m3x2_to_f16x2(static_cast<uint16_t>(w3 & 0xffffu)),
                             e4m3x2_to_f16x2(static_cast<uint16_t>(w3 >> 16)));
          }
          const uint32_t dst = (is_v ? sVc : sKc) + cb * kKvBytes + (c >> 2) * 8192 + row * 128;
          const int c0 = 2 * (c & 3);
          sts_v4(dst + ((c0 ^ (row & 7)) << 4), lo4);
          sts_v4(dst + (((c0 + 1) ^ (row & 7)) << 4), hi4);
        }
        fence_proxy_async();  // the f16 tiles, visible to the tensor core
        mbar_arrive(bar(kBarCFull + cb));
        mbar_arrive(bar(kBarEmpty + st));  // the e4m3 stage may be reloaded
      }
      if (!ok && lane == 0) atomicOr(a.err, PA_DEVERR_TIMEOUT);
    }
  } else {
    // ------------------------------------------------------------ softmax
    const int x = warp / kGroupWarps;  // row tile: 0 = A, 1 = B
    const int r = tid - x * kRows;     // row within the tile = tensor-memory lane
    const int gr = r0 + x * kRows + r;
    const bool valid = gr < r1;
    const bool active = x == 0 || hasB;
    const int tq = valid ? gr / a.G : 0;
    const int hq = gr - tq * a.G;
    const int hi_r = valid ? L - a.T + tq : -1;  // this row's query position
    const int lo_r = (a.window > 0 && hi_r + 1 > a.window) ? hi_r + 1 - a.window : 0;
    const size_t orow =
        ((static_cast<size_t>(b) * a.T + tq) * a.Hq + static_cast<size_t>(kvh) * a.G + hq) * kHd;
    const uint32_t q_tile = sQ + x * kQBytes;
    float sc = a.score_scale;  // this row's score scale (log2 domain)
    {  // Q row -> shared memory (K-major, 128-byte swizzle)
      const uint4* src =
          reinterpret_cast<const uint4*>(reinterpret_cast<const uint16_t*>(a.q) + orow);
      uint4 qv[16];
#pragma unroll
      for (int c = 0; c < 16; ++c) qv[c] = valid ? src[c] : make_uint4(0u, 0u, 0u, 0u);
      if constexpr (FP8) {
        // f16 after a power-of-two rescale: largest magnitude in [2^14, 2^15)
        auto f = [&](uint32_t w, int hi) -> float {
          const uint16_t h = static_cast<uint16_t>(hi ? w >> 16 : w & 0xffffu);
          return QT == kBF16 ? __uint_as_float(static_cast<uint32_t>(h) << 16)
                             : __half2float(__ushort_as_half(h));
        };
        float amax = 0.f;
#pragma unroll
        for (int c = 0; c < 16; ++c) {
          const uint32_t w4[4] = {qv[c].x, qv[c].y, qv[c].z, qv[c].w};
#pragma unroll
          for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(f(w4[i >> 1], i & 1)));
        }
        int sh = 0;
        if (amax > 0.f && amax < INFINITY) {
          int e;
          frexpf(amax, &e);
          sh = e - 15;
        }
        sc = ldexpf(a.score_scale, sh);
#pragma unroll
        for (int c = 0; c < 16; ++c) {
          const uint32_t w4[4] = {qv[c].x, qv[c].y, qv[c].z, qv[c].w};
          uint32_t o4[4];
#pragma unroll
          for (int i = 0; i < 4; ++i)
            o4[i] = pack16x2<false>(ldexpf(f(w4[i], 0), -sh), ldexpf(f(w4[i], 1), -sh));
          qv[c] = make_uint4(o4[0], o4[1], o4[2], o4[3]);
        }
      }
#pragma unroll
      for (int c = 0; c < 16; ++c)
        sts_v4(q_tile + (c >> 3) * 16384 + r * 128 + (((c & 7) ^ (r & 7)) << 4), qv[c]);
      fence_proxy_async();
      mbar_arrive(bar(kBarQ));
    }
    const uint32_t trow = tmem + (static_cast<uint32_t>((warp % 4) * 32) << 16);
    const uint32_t tS = trow + kColS + 64 * x, tO = trow + kColO + 128 * x;
    float m = kFloor, l = 0.f;  // reference max and running sum of the row
    bool ok = true;
    for (int n = 0; active && n < ntiles; ++n) {
      const int st = n % kStages;
      const int t0 = lo16 + n * kKv;  // position of the tile's first token
      if (!(ok = wait_all(bar(kBarS + x), n & 1))) break;
      tc::fence_after_sync();
      uint32_t sr[2][32];
      tc::ld32_async(tS, sr[0]);
      tc::ld32_async(tS + 32, sr[1]);
      tc::wait_ld(sr[0], sr[1]);
      float s[kKv];
      const bool inside = t0 >= lo_r && t0 + kKv - 1 <= hi_r;
      float mxp[8];  // eight independent partial maxima: short dependency chains
#pragma unroll
      for (int i = 0; i < 8; ++i) mxp[i] = kFloor;
      if (inside) {
#pragma unroll
        for (int j = 0; j < kKv; ++j) {
          s[j] = __uint_as_float(sr[j >> 5][j & 31]) * sc;
          mxp[j & 7] = fmaxf(mxp[j & 7], s[j]);
        }
      } else {
#pragma unroll
        for (int j = 0; j < kKv; ++j) {
          const bool keep = t0 + j >= lo_r && t0 + j <= hi_r;
          s[j] = keep ? __uint_as_float(sr[j >> 5][j & 31]) * sc : -INFINITY;
          mxp[j & 7] = fmaxf(mxp[j & 7], s[j]);
        }
      }
      const float mx = fmaxf(fmaxf(fmaxf(mxp[0], mxp[1]), fmaxf(mxp[2], mxp[3])),
                             fmaxf(fmaxf(mxp[4], mxp[5]), fmaxf(mxp[6], mxp[7])));
      // the previous product of this tile X is done: P_X and O_X are free
      if (n > 0 && !(ok = wait_all(bar(kBarO + x), (n - 1) & 1))) break;
      tc::fence_after_sync();
      const bool grow = mx > m + kRescaleAbove;
      if (n == 0) {
        m = mx;  // nothing accumulated yet
      } else if (__any_sync(kFull, grow)) {
        const float alpha = grow ? ex2(m - mx) : 1.f;
#pragma unroll
        for (int c0 = 0; c0 < kHd; c0 += 32) {
          uint32_t ov[32];
          tc::ld32_async(tO + c0, ov);
          tc::wait_ld(ov);
#pragma unroll
          for (int i = 0; i < 32; ++i) ov[i] = __float_as_uint(__uint_as_float(ov[i]) * alpha);
          tc::st32(tO + c0, ov);
        }
        tc::wait_st();
        l *= alpha;
        if (grow) m = mx;
      }
      float sp[8];  // eight independent partial sums
#pragma unroll
      for (int i = 0; i < 8; ++i) sp[i] = 0.f;
      uint32_t pk[kKv / 2];
#pragma unroll
      for (int j = 0; j < kKv / 2; ++j) {
        const float p0 = ex2(s[2 * j] - m), p1 = ex2(s[2 * j + 1] - m);
        sp[j & 7] += p0 + p1;
        pk[j] = pack16x2<kBf16>(p0, p1);
      }
      l += ((sp[0] + sp[1]) + (sp[2] + sp[3])) + ((sp[4] + sp[5]) + (sp[6] + sp[7]));
      if (!FP8 && x == 0 && (t0 < lo || t0 + kKv - 1 > hi)) {
        // edge tile: once it has landed, zero the V rows outside [lo, hi]
        // (with FP8 caches the converters write those rows as zeros)
        if (!(ok = wait_all(bar(kBarFull + st), (n / kStages) & 1))) break;
        for (int i = r; i < kKv * 16; i += kRows) {
          const int row = i >> 4, box = (i >> 3) & 1, ch = i & 7;
          const int pos = t0 + row;
          if (pos < lo || pos > hi)
            sts_v4(sV + st * kKvBytes + box * 8192 + row * 128 + ch * 16,
                   make_uint4(0u, 0u, 0u, 0u));
        }
        fence_proxy_async();  // the cleaned V rows, visible to the tensor core
      }
      // P_X: free, since the previous product of this tile completed above
      tc::st32(trow + kColP + 32 * x, pk);
      tc::wait_st();
      tc::fence_before_sync();
      mbar_arrive(bar(kBarP + x));
    }
    if (!ok && lane == 0) atomicOr(a.err, PA_DEVERR_TIMEOUT);
    if (active) {
      // the last product, then the output row
      if (ok && ntiles > 0) ok = wait_all(bar(kBarO + x), (ntiles - 1) & 1);
      tc::fence_after_sync();
      const float inv = (ok && ntiles > 0 && l > 0.f) ? (FP8 ? a.v_scale : 1.f) / l : 0.f;
      uint4* dst = reinterpret_cast<uint4*>(reinterpret_cast<uint16_t*>(a.out) + orow);
#pragma unroll
      for (int c0 = 0; c0 < kHd; c0 += 32) {
        uint32_t ov[32];
        if (ntiles > 0) {
          tc::ld32_async(tO + c0, ov);
          tc::wait_ld(ov);
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i) ov[i] = 0u;
        }
        if (valid) {
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            const float* f = reinterpret_cast<const float*>(ov) + 8 * c;
            constexpr bool kOutBf16 = QT == kBF16;
            dst[c0 / 8 + c] = make_uint4(pack16x2<kOutBf16>(f[0] * inv, f[1] * inv),
                                         pack16x2<kOutBf16>(f[2] * inv, f[3] * inv),
                                         pack16x2<kOutBf16>(f[4] * inv, f[5] * inv),
                                         pack16x2<kOutBf16>(f[6] * inv, f[7] * inv));
          }
        }
      }
    }
  }

  // every MMA has completed (each active group waited for its last product)
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 0) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, kTmemCols);
  }
}

template <int QT, bool FP8>
cudaError_t launch_typed(const CUtensorMap& tk, const CUtensorMap& tv, const ChunkArgs& a,
                         int grid, cudaStream_t s, bool pdl) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(Smem<FP8>::kThreads);
  cfg.dynamicSmemBytes = Smem<FP8>::kBytes;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, chunk_attn_tc_kernel<QT, FP8>, tk, tv, a);
}

}  // namespace

static_assert(kUnitRows == 256, "both chunk kernels take 256 rows per CTA");

template <int QT, bool FP8>
cudaError_t set_smem() {
  return cudaFuncSetAttribute(chunk_attn_tc_kernel<QT, FP8>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize, Smem<FP8>::kBytes);
}

cudaError_t chunk_tc_fp8_prepare() {
  cudaError_t e;
  if ((e = set_smem<kBF16, true>()) != cudaSuccess || (e = set_smem<kF16, true>()) != cudaSuccess)
    return e;
  return cudaSuccess;
}

cudaError_t chunk_tc_fp8_launch(int qt, const CUtensorMap& tk, const CUtensorMap& tv,
                                const ChunkArgs& a, int grid, cudaStream_t s, bool pdl) {
  return qt == kBF16 ? launch_typed<kBF16, true>(tk, tv, a, grid, s, pdl)
                     : launch_typed<kF16, true>(tk, tv, a, grid, s, pdl);
}

}  // namespace pa
