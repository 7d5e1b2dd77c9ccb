// Tensor-memory kernel for chunked causal queries over the paged cache
// (the chunked-prefill step of "vLLM 0.5 深度解析" §5.2; the attention itself
// is the block-wise scaled dot product with a running max/sum of §2.3 of
// the same page), on the 5th-generation tensor cores of sm_103a; 16-bit or
// FP8 e4m3 caches.
//
// Work unit: one (sequence b, KV head, 256 (query, head) rows), the rows
// being r = t * G + h over the chunk's T queries and the group's G heads: one
// CTA each, holding two 128-row tiles A and B. The unit's read range is the
// union of its rows' ranges, [lo, hi] with lo the first row's window start
// and hi the last row's position; it is walked in K/V tiles of 128 tokens
// (eight 16-token slices, each inside one physical block, fetched by TMA
// through the block table), each shared by both row tiles.
//
// Roles: a producer warp streams K and V tiles through two-stage rings, an
// MMA warp issues every product, and two groups of four softmax warps (one
// row per thread) serve tiles A and B, so the tensor core works for one
// group while the other runs its softmax. Per K/V tile n and row tile X:
//   S_X  = Q_X . K_n^T     tcgen05.mma M128 N128 K128 -> TMEM
//   softmax X: S_X from TMEM; per-row causal/window mask; online softmax in
//          the log2 domain against the row's reference max m; P_X (16-bit,
//          packed in pairs) written back over columns 0-31 and 64-95 of S_X
//   O_X += P_X . V_n       tcgen05.mma M128 N128 K128, A = P_X from TMEM,
//                          B = V_n (MN-major) -> TMEM
// S_X(n+1) overwrites P_X(n), so the MMA warp issues it only once the product
// that reads P_X(n) has completed (its commit barrier); products into
// different accumulators carry no ordering of their own. A completed S_X(n)
// therefore also means O_X is complete up to tile n-1, which the softmax
// relies on when it rescales O_X.
//
// Per-tile shapes: 128-token tiles keep every product at N = 128 or K = 128,
// where one M128 K16 step costs about the same as at N = 64, and halve the
// hand-offs between the softmax groups and the MMA warp per token. A thread
// reads its 128 scores from tensor memory 64 at a time for the row max,
// keeping the second half in registers; the exponentials of that half go
// over columns 64-95 (scores it holds), then the first half is read again
// and its P goes over columns 0-31. 64 scores live in registers, and the loop
// bodies stay small enough for the instruction cache. A warp takes the
// masked form of a half only when one of its rows needs it.
//
// The output accumulates in tensor memory. A row's reference max moves only
// when its running max exceeds it by more than 8 (log2 units); the warp then
// rescales those rows of O_X in tensor memory before the product that adds
// the tile, so P stays below 2^8 and most tiles never touch O. V rows of an
// edge tile that lie outside [lo, hi] (not loaded, or NaN-poisoned slots past
// the sequence or before the window) are zeroed in shared memory before the
// products, so only attended rows reach the tensor core. Scores enter the
// exponent through one fused multiply-add against the scaled reference max,
// issued on score pairs (the two-wide fp32 FMA of sm_100+; the row sums use
// the two-wide add); a negative softmax scale is carried by flipping the sign of Q (exact), so
// the row max is taken on the raw scores. Head dim 128.
//
// FP8 e4m3 caches (FP8 = true): the rings hold the raw e4m3 tiles (16 KB of
// K and of V per tile), and two converter warps turn each into an f16 tile
// of the layout above (exact), in one buffer for K and two for V that the
// products read; they write zeros for the V rows outside [lo, hi]. A
// converted buffer is refilled once the products that read it completed
// (V is double-buffered: its products come last in a tile's chain). K is
// converted head dims 0-63 first: S's first four steps start on them while
// dims 64-127 are converted.
// Q is converted per row to f16 after a power-of-two rescale that brings its
// largest magnitude into [2^14, 2^15); the rescale and k_scale fold into the
// row's score scale, and v_scale is applied to the output.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "pa_internal.h"
#include "ptx.cuh"
#include "tc.cuh"

namespace pa {
namespace {

constexpr int kRows = 128;      // rows per row tile: the MMA M
constexpr int kUnitRows = 2 * kRows;
constexpr int kKv = 128;        // tokens per K/V tile
constexpr int kSlices = kKv / 16;
constexpr int kHd = 128;        // head dim
constexpr int kGroupWarps = 4;  // softmax warps per row tile
constexpr int kCtrlWarp = 2 * kGroupWarps;  // issues the MMAs
constexpr int kLoadWarp = kCtrlWarp + 1;     // streams K/V tiles
constexpr int kConvWarp0 = kLoadWarp + 1;    // FP8: e4m3 -> f16 converters
constexpr int kConvWarps = 2;
constexpr uint32_t kQBytes = kRows * kHd * 2;   // per row tile: [2 boxes][128 rows][128 B]
constexpr uint32_t kBoxBytes = kKv * 128;       // one 64-dim box of a K or V tile
constexpr uint32_t kTileBytes = 2 * kBoxBytes;  // K or V tile: [2 boxes][128 tokens][128 B]
constexpr uint32_t kRawBytes = kKv * kHd;       // e4m3 tile: [128 tokens][128 B]
// barriers: K and V rings (full, empty; two stages each); per row tile X:
// S_X computed, P_X written, O_X product complete; Q staged; FP8: the
// converted K buffer and the two V buffers written (full) and read by their
// products (free)
constexpr int kBarKFull = 0, kBarKEmpty = 2, kBarVFull = 4, kBarVEmpty = 6, kBarS = 8,
              kBarP = 10, kBarO = 12, kBarQ = 14, kBarCKFull = 15 /* dims 0-63 */,
              kBarCKFree = 16, kBarCVFull = 17, kBarCVFree = 19, kBarCKFull1 = 21 /* 64-127 */,
              kNumBars = 22;

// Shared-memory layout: Q_A, Q_B, the K ring, the V ring, (FP8: the
// converted K and V tiles), barriers, the tensor-memory address.
template <bool FP8>
struct Smem {
  static constexpr uint32_t kThreads = (kConvWarp0 + (FP8 ? kConvWarps : 0)) * 32;
  static constexpr uint32_t kRing = FP8 ? kRawBytes : kTileBytes;  // one ring tile
  static constexpr uint32_t kQ = 0;
  static constexpr uint32_t kK = kQ + 2 * kQBytes;
  static constexpr uint32_t kV = kK + 2 * kRing;
  static constexpr uint32_t kKc = kV + 2 * kRing;
  static constexpr uint32_t kVc = kKc + (FP8 ? kTileBytes : 0);
  static constexpr uint32_t kBar = kVc + (FP8 ? 2 * kTileBytes : 0);
  static constexpr uint32_t kSlot = kBar + 8 * kNumBars;
  static constexpr uint32_t kBytes = kSlot + 16 + 1024;  // + room to align the base to 1 KB
};
static_assert(Smem<false>::kBytes <= 227 * 1024 && Smem<true>::kBytes <= 227 * 1024,
              "shared memory per CTA");
// tensor memory: S_A [0,128) S_B [128,256) O_A [256,384) O_B [384,512);
// P_X over columns 0-31 (tokens 0-63) and 64-95 (tokens 64-127) of S_X
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColS = 0, kColO = 256;
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
// max of three (one instruction on sm_103a)
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}
// Two consecutive 32-bit tensor-memory values as an fp32 pair.
__device__ __forceinline__ float2 score_pair(const uint32_t* v, int i) {
  return make_float2(__uint_as_float(v[i]), __uint_as_float(v[i + 1]));
}

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ bool wait_all(uint32_t bar, uint32_t parity) {
  return __all_sync(kFull, mbar_wait_bounded(bar, parity, kWaitNs));
}

// K/V tiles a unit reads: rows [r0, r1) of a sequence of length L (clamped
// to [0, cap]), the same range the kernel derives below.
__device__ __forceinline__ int unit_tiles(const ChunkArgs& a, int L, int cap, int r0, int r1) {
  L = L < 0 ? 0 : (L > cap ? cap : L);
  const int p_first = L - a.T + r0 / a.G;
  const int hi = L - a.T + (r1 - 1) / a.G;
  const int lo = (a.window > 0 && p_first + 1 > a.window) ? p_first + 1 - a.window : 0;
  return hi >= lo ? (hi + 1 - (lo & ~15) + kKv - 1) / kKv : 0;
}

// The work item of CTA `cta`, heaviest first: CTAs start in index order, so
// handing out the long units first makes the grid a longest-first list
// schedule (on 512 units of uniform [512, 8192]-token sequences the makespan
// drops by about 7% against the plain (sequence, KV head, unit) order).
// Sequences are ranked by the tiles of their last unit (most first, then by
// index); within one, units from the last (the most causal work) down, each
// for every KV head. Ranking costs every thread O(B) loads, so beyond
// kRankMax sequences they go in index order. Block-wide: every thread calls
// it; *s_b receives the sequence.
constexpr int kRankMax = 64;
__device__ __forceinline__ void unit_of_cta(const ChunkArgs& a, int cta, int* s_b, int* b,
                                            int* kvh, int* ut) {
  const int cap = a.MB * a.bs;
  const int per_seq = a.QT * a.Hkv;
  const int r = cta / per_seq;  // rank of the sequence
  const int i = cta - r * per_seq;
  const int nrows = a.T * a.G;
  const int lr0 = (a.QT - 1) * kUnitRows, lr1 = nrows;  // the last unit's rows
  if (a.B > kRankMax && threadIdx.x == 0) *s_b = r;
  for (int c = threadIdx.x; a.B <= kRankMax && c < a.B; c += blockDim.x) {
    const int wc = unit_tiles(a, __ldg(a.seq_lens + c), cap, lr0, lr1);
    int rank = 0;
    for (int o = 0; o < a.B; ++o) {
      const int wo = unit_tiles(a, __ldg(a.seq_lens + o), cap, lr0, lr1);
      rank += (wo > wc || (wo == wc && o < c)) ? 1 : 0;
    }
    if (rank == r) *s_b = c;
  }
  __syncthreads();
  *b = *s_b;
  *ut = a.QT - 1 - i / a.Hkv;
  *kvh = i % a.Hkv;
}


// Eight M128 K16 steps of one product group from one asm block, A and B in
// shared memory: step k reads A at descriptor a + a_off(k) and B at
// b + b_off(k) (offsets in 16-byte units, added to the low half: the
// address field cannot carry), the first step overwrites D, the others
// accumulate.
__device__ __forceinline__ void mma8_ss(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc) {
  const uint32_t alo = static_cast<uint32_t>(a), ahi = static_cast<uint32_t>(a >> 32);
  const uint32_t blo = static_cast<uint32_t>(b), bhi = static_cast<uint32_t>(b >> 32);
  asm volatile(
      "{\n.reg .pred p0, p1;\n.reg .b32 al, bl;\n.reg .b64 ad, bd;\n"
      "setp.ne.b32 p0, 0, 0;\nsetp.eq.b32 p1, 0, 0;\n"
      "mov.b64 ad, {%1, %2};\nmov.b64 bd, {%3, %4};\n"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], ad, bd, %5, p0;\n"
      "add.u32 al, %1, 2;\nadd.u32 bl, %3, 2;\nmov.b64 ad, {al, %2};\nmov.b64 bd, {bl, %4};\n"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], ad, bd, %5, p1;\n"
      "add.u32 al, %1, 4;\nadd.u32 bl, %3, 4;\nmov.b64 ad, {al, %2};\nmov.b64 bd, {bl, %4};\n"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], ad, bd, %5, p1;\n"
      "add.u32 al, %1, 6;\nadd.u32 bl, %3, 6;\nmov.b64 ad, {al, %2};\nmov.b64 bd, {bl, %4};\n"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], ad, bd, %5, p1;\n"
      "add.u32 al, %1, 1024;\nadd.u32 bl, %3, 1024;\nmov.b64 ad, {al, %2};\nmov.b64 bd, {bl, %4};\n"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], ad, bd, %5, p1;\n"
      "add.u32 al, %1, 1026;\nadd.u32 bl, %3, 1026;\nmov.b64 ad, {al, %2};\nmov.b64 bd, {bl, %4};\n"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], ad, bd, %5, p1;\n"
      "add.u32 al, %1, 1028;\nadd.u32 bl, %3, 1028;\nmov.b64 ad, {al, %2};\nmov.b64 bd, {bl, %4};\n"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], ad, bd, %5, p1;\n"
      "add.u32 al, %1, 1030;\nadd.u32 bl, %3, 1030;\nmov.b64 ad, {al, %2};\nmov.b64 bd, {bl, %4};\n"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], ad, bd, %5, p1;\n}" ::"r"(d),
      "r"(alo), "r"(ahi), "r"(blo), "r"(bhi), "r"(idesc)
      : "memory");
}
// Eight M128 K16 steps with A in tensor memory: step k reads A at column
// a + (k < 4 ? 8 k : 32 + 8 k) and B at descriptor b + 128 k; the first
// step accumulates iff acc0 != 0, the others always.
__device__ __forceinline__ void mma8_ts(uint32_t d, uint32_t a, uint64_t b, uint32_t idesc,
                                        uint32_t acc0) {
  const uint32_t blo = static_cast<uint32_t>(b), bhi = static_cast<uint32_t>(b >> 32);
  asm volatile(
      "{\n.reg .pred p0, p1;\n.reg .b32 ac, bl;\n.reg .b64 bd;\n"
      "setp.ne.b32 p0, %5, 0;\nsetp.eq.b32 p1, 0, 0;\n"
      "mov.b64 bd, {%2, %3};\n"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], bd, %4, p0;\n"
      "add.u32 ac, %1, 8;\nadd.u32 bl, %2, 128;\nmov.b64 bd, {bl, %3};\n"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [ac], bd, %4, p1;\n"
      "add.u32 ac, %1, 16;\nadd.u32 bl, %2, 256;\nmov.b64 bd, {bl, %3};\n"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [ac], bd, %4, p1;\n"
      "add.u32 ac, %1, 24;\nadd.u32 bl, %2, 384;\nmov.b64 bd, {bl, %3};\n"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [ac], bd, %4, p1;\n"
      "add.u32 ac, %1, 64;\nadd.u32 bl, %2, 512;\nmov.b64 bd, {bl, %3};\n"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [ac], bd, %4, p1;\n"
      "add.u32 ac, %1, 72;\nadd.u32 bl, %2, 640;\nmov.b64 bd, {bl, %3};\n"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [ac], bd, %4, p1;\n"
      "add.u32 ac, %1, 80;\nadd.u32 bl, %2, 768;\nmov.b64 bd, {bl, %3};\n"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [ac], bd, %4, p1;\n"
      "add.u32 ac, %1, 88;\nadd.u32 bl, %2, 896;\nmov.b64 bd, {bl, %3};\n"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [ac], bd, %4, p1;\n}" ::"r"(d),
      "r"(a), "r"(blo), "r"(bhi), "r"(idesc), "r"(acc0)
      : "memory");
}
template <int QT, bool FP8>
__global__ void __launch_bounds__(Smem<FP8>::kThreads, 1)
    chunk_attn_tc128_kernel(const __grid_constant__ CUtensorMap tmK,
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
  const uint32_t* tslot =
      reinterpret_cast<const uint32_t*>(smem_raw + (base - raw) + SL::kSlot);
  // the 16-bit K and V tiles the products read for K/V tile n, and the
  // barrier (with parity) that says they are ready
  auto tile_k = [&](int n) -> uint32_t { return FP8 ? sKc : sK + (n & 1) * kTileBytes; };
  auto tile_v = [&](int n) -> uint32_t {
    return (FP8 ? sVc : sV) + (n & 1) * kTileBytes;
  };
  auto k_ready = [&](int n) -> uint32_t { return FP8 ? bar(kBarCKFull) : bar(kBarKFull + (n & 1)); };
  auto v_ready = [&](int n) -> uint32_t {
    return bar((FP8 ? kBarCVFull : kBarVFull) + (n & 1));
  };
  auto k_par = [&](int n) -> uint32_t { return FP8 ? n & 1 : (n >> 1) & 1; };
  auto v_par = [&](int n) -> uint32_t { return (n >> 1) & 1; };

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // sequence, KV head and unit (256 rows) of this CTA; seq_lens is an input
  // the previous kernel does not write
  __shared__ int s_b;
  int b, kvh, ut;
  unit_of_cta(a, blockIdx.x, &s_b, &b, &kvh, &ut);

  if (tid == 0) {
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar(kBarKFull + i), 1);
      // a ring stage is freed by the products' commit, or (FP8) by the converters
      mbar_init(bar(kBarKEmpty + i), FP8 ? kConvWarps * 32 : 1);
      mbar_init(bar(kBarVFull + i), 1);
      mbar_init(bar(kBarVEmpty + i), FP8 ? kConvWarps * 32 : 1);
      mbar_init(bar(kBarS + i), 1);
      mbar_init(bar(kBarP + i), kGroupWarps * 32);
      mbar_init(bar(kBarO + i), 1);
    }
    mbar_init(bar(kBarQ), 2 * kGroupWarps * 32);
    if constexpr (FP8) {
      mbar_init(bar(kBarCKFull), kConvWarps * 32);
      mbar_init(bar(kBarCKFull1), kConvWarps * 32);
      mbar_init(bar(kBarCKFree), 1);
      for (int j = 0; j < 2; ++j) {
        mbar_init(bar(kBarCVFull + j), kConvWarps * 32);
        mbar_init(bar(kBarCVFree + j), 1);
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
  const int nx = hasB ? 2 : 1;  // row tiles in use
  const int p_first = L - a.T + r0 / a.G;
  const int hi = L - a.T + (r1 - 1) / a.G;  // last position read
  const int lo = (a.window > 0 && p_first + 1 > a.window) ? p_first + 1 - a.window : 0;
  const int lo16 = lo & ~15;
  const int ntiles = hi >= lo ? (hi + 1 - lo16 + kKv - 1) / kKv : 0;

  if (warp == kLoadWarp) {
    // ------------------------------------------------------------ producer
    // K (or V) tile n into ring stage n & 1: lanes 0..7 each look up one
    // 16-token slice in the block table and copy it (16-bit: two 64-dim
    // boxes; e4m3: one 128-dim box).
    auto load = [&](int n, bool is_v) {
      const uint32_t full = bar((is_v ? kBarVFull : kBarKFull) + (n & 1));
      const int pos0 = lo16 + n * kKv + 16 * lane;
      int row = -1;
      if (lane < kSlices && pos0 <= hi) {
        int blk = __ldg(a.block_tables + static_cast<size_t>(b) * a.MB + pos0 / a.bs);
        if (static_cast<unsigned>(blk) >= static_cast<unsigned>(a.NB)) {
          atomicOr(a.err, PA_DEVERR_BLOCK_ID);
          blk = 0;
        }
        row = (blk * a.Hkv + kvh) * a.bs + pos0 % a.bs;
      }
      const int nslices = __popc(__ballot_sync(kFull, row >= 0));
      if (lane == 0) mbar_arrive_expect_tx(full, nslices * (FP8 ? 1 : 2) * 2048);
      __syncwarp();
      if (row >= 0) {
        const uint32_t dst = (is_v ? sV : sK) + (n & 1) * SL::kRing + lane * 2048;
        if constexpr (FP8) {
          tma_load_2d(dst, is_v ? &tmV : &tmK, 0, row, full);
        } else {
#pragma unroll
          for (int box = 0; box < 2; ++box)
            tma_load_2d(dst + box * kBoxBytes, is_v ? &tmV : &tmK, box * 64, row, full);
        }
      }
      __syncwarp();
    };
    bool ok = true;
    for (int n = 0; n < ntiles; ++n) {
      const uint32_t par = ((n - 2) >> 1) & 1;  // tile n-2's release
      if (n >= 2 && !(ok = wait_all(bar(kBarKEmpty + (n & 1)), par))) break;
      load(n, false);
      if (n >= 2 && !(ok = wait_all(bar(kBarVEmpty + (n & 1)), par))) break;
      load(n, true);
    }
    if (!ok && lane == 0) atomicOr(a.err, PA_DEVERR_TIMEOUT);
  } else if (warp == kCtrlWarp) {
    // ------------------------------------------------------------ MMA issue
    constexpr uint32_t idS = tc::idesc_f16(kRows, kKv, kBf16, false);
    constexpr uint32_t idO = tc::idesc_f16(kRows, kHd, kBf16, true);
    // S_X = Q_X . K_n^T over head dims [64 b0, 64 b1) (4 steps of 16 per
    // 64-dim box); the commit once all 8 steps are issued
    // descriptors of the tiles' starts; a step's operand is the start plus a
    // constant (in 16-byte units, within the 14-bit address field)
    const uint64_t dQ0 = tc::sdesc_sw128(sQ, 16, 1024);
    auto issue_s_part = [&](int x, int n, int b0, int b1) {
      if (lane == 0) {
        const uint64_t dQ = dQ0 + ((x * kQBytes) >> 4);
        const uint64_t dK = tc::sdesc_sw128(tile_k(n), 16, 1024);
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
          if (ks < 4 * b0 || ks >= 4 * b1) continue;
          const uint32_t box = ks >> 2, kk = (ks & 3) * 32;
          const uint64_t ad = dQ + ((box * 16384 + kk) >> 4);
          const uint64_t bd = dK + ((box * kBoxBytes + kk) >> 4);
          tc::mma_f16(tmem + kColS + 128 * x, ad, bd, idS, ks > 0);
        }
        if (b1 == 2) tc::commit(bar(kBarS + x));
      }
      __syncwarp();
    };
    auto issue_s = [&](int x, int n) {
      if constexpr (FP8) {
        issue_s_part(x, n, 0, 2);
      } else {
        if (lane == 0) {
          mma8_ss(tmem + kColS + 128 * x, dQ0 + ((x * kQBytes) >> 4),
                  tc::sdesc_sw128(tile_k(n), 16, 1024), idS);
          tc::commit(bar(kBarS + x));
        }
        __syncwarp();
      }
    };
    // O_X (+)= P_X . V_n over 128 tokens (8 steps of 16); P_X in columns
    // 0-31 and 64-95 of S_X, 8 columns (16 tokens) per step
    auto issue_o = [&](int x, int n) {
      if (lane == 0) {
        const uint64_t dV = tc::sdesc_sw128(tile_v(n), kBoxBytes, 1024);
        // P columns of tokens 16 k ..: 8 k for k < 4, 32 + 8 k after
        mma8_ts(tmem + kColO + 128 * x, tmem + kColS + 128 * x, dV, idO, n > 0 ? 1u : 0u);
        tc::commit(bar(kBarO + x));
      }
      __syncwarp();
    };
    // K_t (V_t) is released once both products of tile t that read it
    // complete: its ring stage (16-bit), or the converted buffer (FP8). A
    // release is committed only when something will wait for it, so no
    // arrive outlives the CTA.
    auto release_k = [&](int t) {
      if (lane == 0) {
        if (FP8 && t + 1 < ntiles) tc::commit(bar(kBarCKFree));
        if (!FP8 && t + 2 < ntiles) tc::commit(bar(kBarKEmpty + (t & 1)));
      }
      __syncwarp();
    };
    auto release_v = [&](int t) {
      if (lane == 0) {
        if (FP8 && t + 2 < ntiles) tc::commit(bar(kBarCVFree + (t & 1)));
        if (!FP8 && t + 2 < ntiles) tc::commit(bar(kBarVEmpty + (t & 1)));
      }
      __syncwarp();
    };
    bool ok = true;
    if (ntiles > 0) {
      ok = wait_all(bar(kBarQ), 0) && wait_all(k_ready(0), k_par(0)) &&
           (!FP8 || wait_all(bar(kBarCKFull1), 0));
      if (ok) {
        tc::fence_after_sync();
        for (int x = 0; x < nx; ++x) issue_s(x, 0);
        release_k(0);
      }
    }
    // per row tile in turn: O_X += P_X(n) . V_n, then (once that product has
    // completed) S_X(n+1)
    for (int n = 0; ok && n < ntiles; ++n) {
      for (int x = 0; x < nx; ++x) {
        // P_X(n) written (by group A: the V rows of an edge tile cleaned)
        if (!(ok = wait_all(bar(kBarP + x), n & 1))) break;
        if (x == 0 && !(ok = wait_all(v_ready(n), v_par(n)))) break;
        tc::fence_after_sync();
        issue_o(x, n);
        if (x == nx - 1) release_v(n);
        if (n + 1 < ntiles) {
          if (x == 0 && !(ok = wait_all(k_ready(n + 1), k_par(n + 1)))) break;
          if (!(ok = wait_all(bar(kBarO + x), n & 1))) break;  // P_X(n) consumed
          tc::fence_after_sync();
          if (FP8 && x == 0) {
            // dims 0-63 of K_{n+1} are converted; 64-127 may still be under way
            issue_s_part(0, n + 1, 0, 1);
            if (!(ok = wait_all(bar(kBarCKFull1), (n + 1) & 1))) break;
            tc::fence_after_sync();
            issue_s_part(0, n + 1, 1, 2);
          } else {
            issue_s(x, n + 1);
          }
          if (x == nx - 1) release_k(n + 1);
        }
      }
    }
    if (!ok && lane == 0) atomicOr(a.err, PA_DEVERR_TIMEOUT);
  } else if (warp >= kConvWarp0) {
    // ------------------------------------------------------------ FP8 converters
    // e4m3 K (V) tile n, ring stage n & 1 -> the f16 K (V) buffer: each
    // 16-byte chunk of 16 codes becomes two 16-byte chunks of f16 in the
    // 64-dim box that holds them; V rows outside [lo, hi] are written as zeros.
    if constexpr (FP8) {
      const int ct = tid - kConvWarp0 * 32;
      bool ok = true;
      for (int n = 0; ok && n < ntiles; ++n) {
        const int t0 = lo16 + n * kKv;
        for (int is_v = 0; is_v < 2; ++is_v) {
          if (!(ok = wait_all(bar((is_v ? kBarVFull : kBarKFull) + (n & 1)), (n >> 1) & 1))) break;
          // the buffer's previous tile (K: n-1; V: n-2): its products completed
          if (!is_v && n > 0 && !(ok = wait_all(bar(kBarCKFree), (n - 1) & 1))) break;
          if (is_v && n > 1 && !(ok = wait_all(bar(kBarCVFree + (n & 1)), ((n - 2) >> 1) & 1)))
            break;
          const uint32_t src0 = (is_v ? sV : sK) + (n & 1) * kRawBytes;
          const uint32_t dst0 = is_v ? sVc + (n & 1) * kTileBytes : sKc;
          // a pass converts 16-byte chunks [c_lo, c_lo + nc) of every row:
          // thread ct takes chunk c_lo + ct % nc of rows r0, r0 + per, ...
          // (per = 64 / nc, so row & 7 == r0 & 7: one swizzle per thread)
          static_assert(kConvWarps * 32 == 64, "64 converter threads");
          auto convert = [&](int c_lo, int nc) {
            const int per = 64 / nc;
            const int c = c_lo + ct % nc, r0 = ct / nc, c0 = 2 * (c & 3);
            const uint32_t src = src0 + r0 * 128 + ((c ^ (r0 & 7)) << 4);
            const uint32_t dst = dst0 + (c >> 2) * kBoxBytes + r0 * 128;
            const uint32_t d_lo = dst + ((c0 ^ (r0 & 7)) << 4);
            const uint32_t d_hi = dst + (((c0 + 1) ^ (r0 & 7)) << 4);
            // V rows outside [lo, hi] are written as zeros (edge tiles only)
            const bool edge = is_v && (t0 < lo || t0 + kKv - 1 > hi);
#pragma unroll
            for (int k = 0; k < kKv / per; ++k) {
              uint32_t w0, w1, w2, w3;
              lds_v4(src + per * k * 128, w0, w1, w2, w3);
              uint4 lo4 = make_uint4(e4m3x2_to_f16x2(static_cast<uint16_t>(w0 & 0xffffu)),
                                     e4m3x2_to_f16x2(static_cast<uint16_t>(w0 >> 16)),
                                     e4m3x2_to_f16x2(static_cast<uint16_t>(w1 & 0xffffu)),
                                     e4m3x2_to_f16x2(static_cast<uint16_t>(w1 >> 16)));
              uint4 hi4 = make_uint4(e4m3x2_to_f16x2(static_cast<uint16_t>(w2 & 0xffffu)),
                                     e4m3x2_to_f16x2(static_cast<uint16_t>(w2 >> 16)),
                                     e4m3x2_to_f16x2(static_cast<uint16_t>(w3 & 0xffffu)),
                                     e4m3x2_to_f16x2(static_cast<uint16_t>(w3 >> 16)));
              if (edge) {
                const int pos = t0 + r0 + per * k;
                if (pos < lo || pos > hi) lo4 = hi4 = make_uint4(0u, 0u, 0u, 0u);
              }
              sts_v4(d_lo + per * k * 128, lo4);
              sts_v4(d_hi + per * k * 128, hi4);
            }
          };
          if (is_v) {
            convert(0, 8);
          } else {
            convert(0, 4);  // dims 0-63 first: S can start on them
            fence_proxy_async();
            mbar_arrive(bar(kBarCKFull));
            convert(4, 4);
          }
          fence_proxy_async();  // the f16 tile, visible to the tensor core
          mbar_arrive(bar(is_v ? kBarCVFull + (n & 1) : kBarCKFull1));
          mbar_arrive(bar((is_v ? kBarVEmpty : kBarKEmpty) + (n & 1)));  // reload the stage
        }
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
    // positions this row attends to (none for a query before its sequence)
    const int cnt = valid ? max(hi_r - lo_r + 1, 0) : 0;
    const size_t orow =
        ((static_cast<size_t>(b) * a.T + tq) * a.Hq + static_cast<size_t>(kvh) * a.G + hq) * kHd;
    // this row's score scale (log2 domain); a negative scale flips the sign
    // of Q instead, so sc >= 0
    float sc = fabsf(a.score_scale);
    {  // Q row -> shared memory (K-major, 128-byte swizzle)
      const uint32_t flip = a.score_scale < 0.f ? 0x80008000u : 0u;
      const uint4* src =
          reinterpret_cast<const uint4*>(reinterpret_cast<const uint16_t*>(a.q) + orow);
      const uint32_t q_tile = sQ + x * kQBytes;
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
        sc = ldexpf(sc, sh);
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
      for (int c = 0; c < 16; ++c) {
        uint4 v = qv[c];
        v.x ^= flip, v.y ^= flip, v.z ^= flip, v.w ^= flip;
        sts_v4(q_tile + (c >> 3) * 16384 + r * 128 + (((c & 7) ^ (r & 7)) << 4), v);
      }
      fence_proxy_async();
      mbar_arrive(bar(kBarQ));
    }
    const uint32_t trow = tmem + (static_cast<uint32_t>((warp % 4) * 32) << 16);
    const uint32_t tS = trow + kColS + 128 * x, tO = trow + kColO + 128 * x;
    float ms = kFloor, l = 0.f;  // reference max (scaled, log2 units) and running sum
    bool ok = true;
    for (int n = 0; active && n < ntiles; ++n) {
      const int t0 = lo16 + n * kKv;  // position of the tile's first token
      if (!(ok = wait_all(bar(kBarS + x), n & 1))) break;
      tc::fence_after_sync();
      // warp-uniform: every row of the warp attends to the whole tile
      const bool all_in = __all_sync(kFull, t0 >= lo_r && t0 + kKv - 1 <= hi_r);
      const int d0 = t0 - lo_r;  // token j of the tile is attended iff (unsigned)(d0 + j) < cnt
      uint32_t sv[2][32];
      float mxp[8];  // eight independent partial maxima (raw scores)
#pragma unroll
      for (int i = 0; i < 8; ++i) mxp[i] = -INFINITY;
#pragma unroll 1
      for (int h = 0; h < 2; ++h) {
        tc::ld32_async(tS + 64 * h, sv[0]);
        tc::ld32_async(tS + 64 * h + 32, sv[1]);
        tc::wait_ld(sv[0], sv[1]);
        if (all_in) {
#pragma unroll
          for (int j = 0; j < 32; ++j)
            mxp[j & 7] = fmax3(mxp[j & 7], __uint_as_float(sv[j >> 4][(2 * j) & 31]),
                               __uint_as_float(sv[j >> 4][(2 * j + 1) & 31]));
        } else {
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            const int e = d0 + 64 * h + 2 * j;
            const float v0 = __uint_as_float(sv[j >> 4][(2 * j) & 31]);
            const float v1 = __uint_as_float(sv[j >> 4][(2 * j + 1) & 31]);
            mxp[j & 7] = fmax3(mxp[j & 7],
                               static_cast<unsigned>(e) < static_cast<unsigned>(cnt) ? v0 : -INFINITY,
                               static_cast<unsigned>(e + 1) < static_cast<unsigned>(cnt) ? v1 : -INFINITY);
          }
        }
      }
      const float mxr = fmaxf(fmaxf(fmaxf(mxp[0], mxp[1]), fmaxf(mxp[2], mxp[3])),
                              fmaxf(fmaxf(mxp[4], mxp[5]), fmaxf(mxp[6], mxp[7])));
      const float mx = fmaxf(mxr * sc, kFloor);  // NaN (all masked, sc = 0) -> floor
      const bool grow = mx > ms + kRescaleAbove;
      if (n == 0) {
        ms = mx;  // nothing accumulated yet
      } else if (__any_sync(kFull, grow)) {
        // O_X holds tiles < n complete: S_X(n) was issued after their products
        const float alpha = grow ? ex2(ms - mx) : 1.f;
#pragma unroll 1
        for (int c0 = 0; c0 < kHd; c0 += 32) {
          uint32_t ov[32];
          tc::ld32_async(tO + c0, ov);
          tc::wait_ld(ov);
          const float2 a2 = make_float2(alpha, alpha);
#pragma unroll
          for (int i = 0; i < 32; i += 2) {
            const float2 o = __fmul2_rn(score_pair(ov, i), a2);
            ov[i] = __float_as_uint(o.x);
            ov[i + 1] = __float_as_uint(o.y);
          }
          tc::st32(tO + c0, ov);
        }
        l *= alpha;
        if (grow) ms = mx;
      }
      // P = 2^(s * sc - ms), packed in pairs: scores 64 h + j -> column
      // 64 h + j / 2; the second half first, from registers. The scale FMA
      // and the running sums work on score pairs (two-wide fp32 FMA / add,
      // one instruction per pair).
      const float2 sc2 = make_float2(sc, sc), nms2 = make_float2(-ms, -ms);
      float2 sp[4];  // four independent partial sums of score pairs
#pragma unroll
      for (int i = 0; i < 4; ++i) sp[i] = make_float2(0.f, 0.f);
#pragma unroll 1
      for (int h = 1; h >= 0; --h) {
        if (h == 0) {
          tc::ld32_async(tS, sv[0]);
          tc::ld32_async(tS + 32, sv[1]);
          tc::wait_ld(sv[0], sv[1]);
        }
        uint32_t pk[32];
        if (all_in) {
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            const float2 t = __ffma2_rn(score_pair(sv[j >> 4], (2 * j) & 31), sc2, nms2);
            const float p0 = ex2(t.x), p1 = ex2(t.y);
            sp[j & 3] = __fadd2_rn(sp[j & 3], make_float2(p0, p1));
            pk[j] = pack16x2<kBf16>(p0, p1);
          }
        } else {  // masked scores give exactly 0 (also when sc = 0)
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            const int e = d0 + 64 * h + 2 * j;
            const float2 t = __ffma2_rn(score_pair(sv[j >> 4], (2 * j) & 31), sc2, nms2);
            float p0 = ex2(t.x), p1 = ex2(t.y);
            p0 = static_cast<unsigned>(e) < static_cast<unsigned>(cnt) ? p0 : 0.f;
            p1 = static_cast<unsigned>(e + 1) < static_cast<unsigned>(cnt) ? p1 : 0.f;
            sp[j & 3] = __fadd2_rn(sp[j & 3], make_float2(p0, p1));
            pk[j] = pack16x2<kBf16>(p0, p1);
          }
        }
        tc::st32(tS + 64 * h, pk);
      }
      const float2 s01 = __fadd2_rn(sp[0], sp[1]), s23 = __fadd2_rn(sp[2], sp[3]);
      const float2 st = __fadd2_rn(s01, s23);
      l += st.x + st.y;
      if (!FP8 && x == 0 && (t0 < lo || t0 + kKv - 1 > hi)) {
        // edge tile: once it has landed, zero the V rows outside [lo, hi]
        // (with FP8 caches the converters write those rows as zeros)
        if (!(ok = wait_all(bar(kBarVFull + (n & 1)), (n >> 1) & 1))) break;
        const uint32_t vt = sV + (n & 1) * kTileBytes;
        for (int i = r; i < kKv * 16; i += kRows) {
          const int row = i >> 4, box = (i >> 3) & 1, ch = i & 7;
          const int pos = t0 + row;
          if (pos < lo || pos > hi)
            sts_v4(vt + box * kBoxBytes + row * 128 + ch * 16, make_uint4(0u, 0u, 0u, 0u));
        }
        fence_proxy_async();  // the cleaned V rows, visible to the tensor core
      }
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
          constexpr bool kOutBf16 = QT == kBF16;
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            const float* f = reinterpret_cast<const float*>(ov) + 8 * c;
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
  return cudaLaunchKernelEx(&cfg, chunk_attn_tc128_kernel<QT, FP8>, tk, tv, a);
}

template <int QT, bool FP8>
cudaError_t set_smem() {
  return cudaFuncSetAttribute(chunk_attn_tc128_kernel<QT, FP8>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize, Smem<FP8>::kBytes);
}

}  // namespace

int chunk_tc_unit_rows() { return kUnitRows; }

cudaError_t chunk_tc_prepare() {
  cudaError_t e;
  if ((e = set_smem<kBF16, false>()) != cudaSuccess || (e = set_smem<kF16, false>()) != cudaSuccess ||
      (e = set_smem<kBF16, true>()) != cudaSuccess || (e = set_smem<kF16, true>()) != cudaSuccess)
    return e;
  return cudaSuccess;
}

cudaError_t chunk_tc_launch(int qt, bool fp8, const CUtensorMap& tk, const CUtensorMap& tv,
                            const ChunkArgs& a, cudaStream_t s, bool pdl) {
  const long long grid = static_cast<long long>(a.B) * a.Hkv * a.QT;
  if (grid <= 0) return cudaSuccess;
  if (grid > 0x7fffffffLL) return cudaErrorInvalidValue;
  const int g = static_cast<int>(grid);
  if (fp8)
    return qt == kBF16 ? launch_typed<kBF16, true>(tk, tv, a, g, s, pdl)
                       : launch_typed<kF16, true>(tk, tv, a, g, s, pdl);
  return qt == kBF16 ? launch_typed<kBF16, false>(tk, tv, a, g, s, pdl)
                     : launch_typed<kF16, false>(tk, tv, a, g, s, pdl);
}

}  // namespace pa
