// Persistent paged-decode kernel for sm_103a.
//
// Work decomposition (balanced split-KV). Every (sequence b, KV head) pair
// owns the 16-token tiles that cover its attended positions [start, L); tiles
// never straddle a physical block because block_size is a multiple of 16.
// All tiles of all pairs form one flat index space (pair-major). The first
// part of it (about 90%) is split into equal contiguous static ranges, one per
// worker warp; the rest is a pool of pieces that warps claim with one
// atomicAdd each once their static range is done (the claim for the next
// piece is issued a piece ahead, so the copy pipeline never drains). Warps on
// SMs that get less bandwidth thus take fewer pieces and all warps finish
// together. The pool only covers the trailing run of
// sequences no longer than four times the mean, so a long sequence is never
// cut into small pieces (plan.cuh). A run of one warp's tiles inside one pair
// is a segment; each segment writes one partial (running max m, running sum
// l, unnormalised output) to a slot fixed by arithmetic: pair + warp for
// static segments, pair + piece (in a second region) for pool segments --
// unique because the walk through the (pair, warp) and (pair, piece) grids is
// a monotone staircase. A merge kernel combines each pair's partials by their
// log-sum-exp weights.
//
// Data movement. Each warp owns a ring of STAGES shared-memory stages; one
// stage holds the K tile and the V tile [16 rows x D] of one (block, KV head),
// loaded by TMA boxes of [16 rows x 128 bytes] with the 128-byte swizzle, and
// signalled on an mbarrier. Block ids are read 32 at a time per warp, the next
// window prefetched, and broadcast with shuffles. Each K/V byte of the step
// is loaded once and used by all G query heads of its group. Blocks wholly
// outside the window are never loaded ("vLLM 0.7.2深度解析" §2.3).
//
// Math (per tile, per warp), on the tensor cores with fp32 accumulation:
//   S^T[16 tok x 8 heads] = K[16 x D] . Q^T[D x 8]     (mma m16n8k16, M = tokens)
//   online softmax on S in the log2 domain (scale * log2 e folded in), with a
//     lazy reference max per column: it moves (cross-lane max, rescale of
//     l and O) only on tiles where a score exceeds it by more than 8
//   O^T[D x 8 heads] += V^T[D x 16 tok] . P^T[16 x 8]  (P^T via movmatrix)
// i.e. the block-wise scaled dot product, max/sum state and V-weighted sum of
// "vLLM 0.5 深度解析" §2.3, done in one pass. With bf16 caches P enters P.V
// as a bf16 high part plus a bf16 remainder (two mma), about 16 bits. Positions
// outside [start, L) in the first and last tile of a pair get score -inf and
// their V rows are zeroed in the fragment, so poisoned slots never reach the
// result.
//
// Chunked queries (MQ = true). A sequence may bring T query tokens at its
// last T positions, each attending causally to its own prefix (clipped by
// the window), as in the chunked prefill of "vLLM 0.5 深度解析" §5.2. The mma
// n-columns of a pair are then (query, head) columns c = t * G + h, at most
// 16 per pair; with more, the columns are cut into NCG groups of 16 and each
// group is a pair of its own (a "virtual" KV head vh = kvh * NCG + group), so
// the same K/V tile is read once per group. A pair's tiles cover the union of
// its queries' ranges; scores outside a column's own range get -inf, and the
// running maxima start at a finite floor so that a column with no position in
// a segment yields m = floor, l = 0 and a zero output.
//
// FP8 e4m3 caches: codes are converted to f16 in registers (exact), Q is
// converted once per segment to f16 after a power-of-two rescale so its
// largest magnitude lies in [2^14, 2^15), and k_scale, v_scale and the rescale
// are folded into the score scale and the partial outputs.
#pragma once

#include <type_traits>

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "pa_internal.h"
#include "plan.cuh"
#include "ptx.cuh"

namespace pa {

constexpr uint64_t kWaitLimitNs = 2000000000ull;   // pipeline wait bound (2 s)
constexpr uint64_t kDrainLimitNs = 200000000ull;   // bound while draining after an error
constexpr int kErrBlockId = PA_DEVERR_BLOCK_ID, kErrTimeout = PA_DEVERR_TIMEOUT;

template <int CT, int D, int STAGES>
struct Geometry {
  static constexpr int ELT = (CT == kE4M3) ? 1 : 2;
  static constexpr int ROW_BYTES = D * ELT;
  static constexpr int BOXES = ROW_BYTES / 128;   // 128-byte column boxes per row
  static constexpr int BOX_ELEMS = 128 / ELT;
  static constexpr int TILE_BYTES = kTile * ROW_BYTES;
  static constexpr int STAGE_BYTES = 2 * TILE_BYTES;
  static constexpr int RING_BYTES = STAGES * STAGE_BYTES;
  static constexpr int MT = D / 16;
  static_assert(ROW_BYTES % 128 == 0, "rows must be whole 128-byte boxes");
};

// Shared-memory byte offset of 16-byte chunk c (counted along the full row) of
// tile row r. A tile is stored as [box][16 rows][128 B]; within a box the TMA
// 128-byte swizzle places chunk j of row r at position j ^ (r & 7).
__device__ __forceinline__ uint32_t tile_off(int r, int c) {
  return (static_cast<uint32_t>(c >> 3) << 11) + (static_cast<uint32_t>(r) << 7) +
         (static_cast<uint32_t>((c & 7) ^ (r & 7)) << 4);
}

struct Cursor {
  int b, kvh, t, nt;
};

// Places the cursor on flat tile f (f < total): pair (b, kvh), tile t of nt.
__device__ __forceinline__ void cursor_locate(Cursor& c, int f, const int* pref, int B,
                                              int Hkv) {
  int lo = 0, hi = B;
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (Hkv * pref[mid] <= f) lo = mid; else hi = mid;
  }
  c.b = lo;
  c.nt = pref[lo + 1] - pref[lo];
  const int rem = f - Hkv * pref[lo];
  c.kvh = rem / c.nt;
  c.t = rem - c.kvh * c.nt;
}

__device__ __forceinline__ void cursor_next(Cursor& c, const int* pref, int B, int Hkv) {
  if (++c.t < c.nt) return;
  c.t = 0;
  if (++c.kvh < Hkv) return;
  c.kvh = 0;
  do {
    ++c.b;
  } while (c.b < B && pref[c.b + 1] == pref[c.b]);
  if (c.b < B) c.nt = pref[c.b + 1] - pref[c.b];
}

template <bool BF16>
__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
  if constexpr (BF16) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
  } else {
    __half2 v = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
  }
}

template <int QT>
__device__ __forceinline__ float to_float(uint16_t x) {
  if constexpr (QT == kBF16) {
    return __uint_as_float(static_cast<uint32_t>(x) << 16);
  } else {
    return __half2float(__ushort_as_half(x));
  }
}

// Head-dim index held by accumulator row (m-tile mt, fragment row g + 8 * hi).
template <bool FP8>
__device__ __forceinline__ int acc_dim(int mt, int g, int hi) {
  if constexpr (FP8) {
    return 32 * (mt >> 1) + 4 * g + 2 * (mt & 1) + hi;
  } else {
    return 16 * mt + g + 8 * hi;
  }
}

constexpr unsigned kFlagStart = 1, kFlagEnd = 2, kFlagPool = 4;

constexpr float kMaskedFloor = -1e30f;  // running-max start of chunked columns
constexpr float kRefSlack = 8.f;        // log2 units a score may exceed the reference max

template <int CT, int QT, int D, int NT, int WARPS, int STAGES, bool MQ>
__global__ void __launch_bounds__(WARPS * 32, 2)
    paged_decode_kernel(const __grid_constant__ CUtensorMap tmK,
                        const __grid_constant__ CUtensorMap tmV, const DecodeArgs a) {
  using Gm = Geometry<CT, D, STAGES>;
  constexpr bool kFp8 = (CT == kE4M3);
  constexpr bool kBf16Mma = (CT == kBF16);
  constexpr int MT = Gm::MT;
  constexpr unsigned FULL = 0xffffffffu;

  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_addr(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - raw);
  const uint32_t bars = base + WARPS * Gm::RING_BYTES;
  int* s_meta = reinterpret_cast<int*>(gbase + WARPS * Gm::RING_BYTES + WARPS * STAGES * 8);
  int* s_len = s_meta + 2 * WARPS * STAGES;
  int* s_pref = s_len + a.B;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, t4 = lane & 3;

  // Programmatic launch: the work before griddep_wait() below (planning from
  // seq_lens) overlaps the previous kernel of the stream.
  // A kernel of this library that lets dependents start early (the write
  // path) does so only once its own predecessors have finished, and it
  // writes none of q, seq_lens, block_tables or this workspace, only the
  // caches, which are first read after the wait.
  griddep_launch_dependents();

  if (tid == 0) {
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
    for (int i = 0; i < WARPS * STAGES; ++i) mbar_init(bars + 8 * i, 1);
    fence_mbar_init();
    fence_proxy_async();
  }
  // sequence lengths clamped to the block-table capacity, tile prefix and
  // split (the merge kernel derives the same plan from the same inputs)
  PlanIn pin;
  pin.seq_lens = a.seq_lens;
  pin.err = a.err;
  pin.B = a.B;
  pin.cap = a.MB * a.bs;
  pin.span = a.span;
  pin.Hv = a.Hv;
  pin.nw = gridDim.x * WARPS;
  pin.pool_permille = a.pool_permille;
  pin.min_tiles = a.min_tiles;
  pin.np_max = a.np_max;
  pin.piece_min = a.piece_min;
  const StepPlan pl = plan_step(pin, s_len, s_pref);
  const int total = pl.total, ws = pl.ws, ts = pl.ts;
  const int nw = pin.nw;
  const int pool_tiles = total - ts;
  if (blockIdx.x == 0) {
    // the plan, for the merge kernel (kept in L2: every merge CTA reads it)
    const uint64_t keep = l2_evict_last();
    int32_t* dst = a.plan;
    if (tid < kPlanScalars) {
      const int v[kPlanScalars] = {pl.total, pl.ws, pl.ts, pl.piece, pl.n_pool, 0, 0, 0};
      st_s32_hint(dst + tid, v[tid], keep);
    }
    for (int b = tid; b <= a.B; b += blockDim.x) st_s32_hint(dst + kPlanScalars + b, s_pref[b], keep);
    // publish it: merge CTAs that start before this kernel ends may then
    // load it before their dependency wait
    __syncthreads();
    if (tid == 0) {
      __threadfence();
      st_release_gpu(reinterpret_cast<int32_t*>(a.pool) + 1, 1);
    }
  }
  const int w = blockIdx.x * WARPS + warp;
  const int f0 = static_cast<int>(min(static_cast<long long>(w) * ws, static_cast<long long>(ts)));
  const int f1 = min(f0 + ws, ts);

  const uint32_t ring = base + warp * Gm::RING_BYTES;
  const uint32_t wbars = bars + warp * STAGES * 8;
  int* meta_f = s_meta + warp * 2 * STAGES;
  int* meta_fl = meta_f + STAGES;
  const int npairs = a.B * a.Hv;

  // ---------------------------------------------------------------- producer
  // Runs: the static range [f0, f1), then pool pieces. np = next flat tile to
  // load, run_end = end of the current run, run_id = piece index (pool runs).
  Cursor pc;
  pc.b = pc.kvh = pc.t = pc.nt = 0;
  int phase = 0;  // 0 static, 1 pool, 2 done
  int np = f0, run_end = f1, run_id = -1;
  bool run_first = true;
  bool claim_issued = false;
  uint32_t pending = 0;  // lane 0: prefetched pool claim

  auto issue_claim = [&]() {
    if (lane == 0) pending = atomicAdd(a.pool, 1u);
    claim_issued = true;
  };

  int id_b = -1, id_lb0 = 0, id_val = 0;  // current block-id window
  int pf_b = -1, pf_lb0 = 0, pf_val = 0;  // prefetched next window
  int produced = 0, consumed = 0;

  // Makes the block-id window hold logical block lb of sequence b: 32 table
  // entries per warp, one per lane, with the following window prefetched.
  auto refresh_window = [&](int b, int lb) {
    if (b != id_b || lb < id_lb0 || lb >= id_lb0 + 32) {
      if (b == pf_b && lb >= pf_lb0 && lb < pf_lb0 + 32) {
        id_b = pf_b;
        id_lb0 = pf_lb0;
        id_val = pf_val;
      } else {
        id_b = b;
        id_lb0 = lb;
        const int e = lb + lane;
        id_val = (e < a.MB) ? __ldg(a.block_tables + static_cast<size_t>(b) * a.MB + e) : 0;
      }
      // prefetch the following window of this sequence's table
      pf_b = id_b;
      pf_lb0 = id_lb0 + 32;
      const int e2 = pf_lb0 + lane;
      pf_val = (e2 < a.MB) ? __ldg(a.block_tables + static_cast<size_t>(pf_b) * a.MB + e2) : 0;
    }
  };

  // Produces the next tile into stage `slot`; false when no work is left.
  auto produce = [&](int slot) -> bool {
    while (np >= run_end) {
      if (phase == 2) return false;
      if (pool_tiles == 0) {
        phase = 2;
        return false;
      }
      if (!claim_issued) issue_claim();
      const unsigned i = __shfl_sync(FULL, pending, 0);
      claim_issued = false;
      if (i >= static_cast<unsigned>(pl.n_pool)) {
        phase = 2;
        return false;
      }
      phase = 1;
      piece_range(static_cast<int>(i), pl, &np, &run_end);
      run_id = static_cast<int>(i);
      run_first = true;
      issue_claim();  // the next piece, one piece ahead
    }
    const int f = np++;
    unsigned flags = (phase == 1) ? kFlagPool : 0u;
    if (run_first) {
      flags |= kFlagStart;
      cursor_locate(pc, f, s_pref, a.B, a.Hv);
      run_first = false;
    } else {
      cursor_next(pc, s_pref, a.B, a.Hv);
    }
    if (np == run_end) {
      flags |= kFlagEnd;
      // static range about to end: claim the first pool piece now
      if (phase == 0 && pool_tiles > 0 && !claim_issued) issue_claim();
    }
    const int L = s_len[pc.b];
    const int pt = win_start(L, a.span) / kTile + pc.t;  // tile index in position space
    const int lb = (pt * kTile) / a.bs;
    refresh_window(pc.b, lb);
    int phys = __shfl_sync(FULL, id_val, lb - id_lb0);
    if (static_cast<unsigned>(phys) >= static_cast<unsigned>(a.NB)) {
      if (lane == 0) atomicOr(a.err, kErrBlockId);
      phys = 0;
    }
    const int kvh = MQ ? pc.kvh / a.NCG : pc.kvh;
    const int row = (phys * a.Hkv + kvh) * a.bs + (pt * kTile) % a.bs;
    if (lane == 0) {
      meta_f[slot] = f;
      meta_fl[slot] = static_cast<int>(flags) | ((phase == 1 ? run_id : 0) << 3);
      const uint32_t bar = wbars + 8 * slot;
      const uint32_t kd = ring + slot * Gm::STAGE_BYTES;
      mbar_arrive_expect_tx(bar, Gm::STAGE_BYTES);
      // K/V are read once per step: evict them first, so the stream does not
      // push the partials (read by the merge right after) out of L2
      const uint64_t kv_policy = l2_evict_first();
#pragma unroll
      for (int j = 0; j < Gm::BOXES; ++j) {
        tma_load_2d_hint(kd + j * 2048, &tmK, j * Gm::BOX_ELEMS, row, bar, kv_policy);
        tma_load_2d_hint(kd + Gm::TILE_BYTES + j * 2048, &tmV, j * Gm::BOX_ELEMS, row, bar,
                         kv_policy);
      }
    }
    __syncwarp();
    return true;
  };

  // The block tables are inputs that the write path never touches: load the
  // window of this warp's first tile before waiting for the previous kernel,
  // so that its first K/V copies issue right after the wait.
  if (f0 < f1) {
    Cursor c0;
    cursor_locate(c0, f0, s_pref, a.B, a.Hv);
    const int pt0 = win_start(s_len[c0.b], a.span) / kTile + c0.t;
    refresh_window(c0.b, (pt0 * kTile) / a.bs);
  }
  griddep_wait();  // the caches may have been written by the previous kernel
  for (int i = 0; i < STAGES; ++i) {
    if (!produce(produced % STAGES)) break;
    ++produced;
  }

  // ---------------------------------------------------------------- consumer
  uint32_t qf[MT][NT][2];
  float m_run[NT][2], l_run[NT][2];
  int qlo[NT][2], qhi[NT][2];  // chunked: attended positions [lo, hi] per score column
  int lo_max = 0, hi_min = 0;  // chunked: tiles inside [lo_max, hi_min] need no column mask
  float acc[MT][NT][4];
  float sc = a.score_scale;
  bool ok = true;
  Cursor cc;
  cc.b = cc.kvh = cc.t = cc.nt = 0;

  while (consumed < produced) {
    const int slot = consumed % STAGES;
    const uint32_t parity = (consumed / STAGES) & 1;
    const int f = meta_f[slot];
    const int mf = meta_fl[slot];
    const unsigned flags = static_cast<unsigned>(mf) & 7u;
    const int piece_id = mf >> 3;
    if (flags & kFlagStart) cursor_locate(cc, f, s_pref, a.B, a.Hv);
    else cursor_next(cc, s_pref, a.B, a.Hv);
    const bool seg_start = (flags & kFlagStart) || (cc.t == 0);
    if (seg_start) {
      // Query fragments of this pair's columns (B operand, k = head dim).
      // Column c is q head kvh * G + c (T = 1), or, chunked, column
      // gc = group * CG + c of the kv head's T * G (query, head) columns.
      const uint16_t* q0 = reinterpret_cast<const uint16_t*>(a.q);
      const int kvh = MQ ? cc.kvh / a.NCG : cc.kvh;
      const int grp = MQ ? cc.kvh - kvh * a.NCG : 0;
      auto qrow = [&](int c) -> const uint16_t* {
        if (c >= a.CG) return nullptr;
        if constexpr (!MQ) {
          return q0 + (static_cast<size_t>(cc.b) * a.Hq + kvh * a.G + c) * D;
        } else {
          const int gc = grp * a.CG + c;
          if (gc >= a.T * a.G) return nullptr;
          const int t = gc / a.G;
          return q0 + ((static_cast<size_t>(cc.b) * a.T + t) * a.Hq + kvh * a.G + (gc - t * a.G)) * D;
        }
      };
      if constexpr (MQ) {
        const int L = s_len[cc.b];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const int c = 8 * nt + 2 * t4 + e;
            const int gc = grp * a.CG + c;
            if (c < a.CG && gc < a.T * a.G) {
              const int p = L - a.T + gc / a.G;  // this query's position
              qhi[nt][e] = p;
              qlo[nt][e] = (a.window > 0 && p + 1 > a.window) ? p + 1 - a.window : 0;
            } else {
              qhi[nt][e] = -1;
              qlo[nt][e] = 0x7fffffff;  // padding column: every score masked
            }
          }
        lo_max = win_start(L, a.window);  // range start of the last query
        hi_min = L - a.T;                 // position of the first query
      }
      sc = a.score_scale;
      if constexpr (!kFp8) {
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          const uint32_t* qh = reinterpret_cast<const uint32_t*>(qrow(8 * nt + g));
#pragma unroll
          for (int ks = 0; ks < MT; ++ks) {
            qf[ks][nt][0] = qh ? qh[(16 * ks + 2 * t4) >> 1] : 0u;
            qf[ks][nt][1] = qh ? qh[(16 * ks + 8 + 2 * t4) >> 1] : 0u;
          }
        }
      } else {
        // k-step ks = 4 * qd + j covers head dims 64 qd + 16 t4 + 4 j + {0..3}
        float qv[MT][NT][4];
        float amax = 0.f;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          const uint16_t* qh = qrow(8 * nt + g);
#pragma unroll
          for (int ks = 0; ks < MT; ++ks) {
            const int d = 64 * (ks >> 2) + 16 * t4 + 4 * (ks & 3);
            uint2 raw2 = make_uint2(0u, 0u);
            if (qh) raw2 = *reinterpret_cast<const uint2*>(qh + d);
            qv[ks][nt][0] = to_float<QT>(static_cast<uint16_t>(raw2.x & 0xffffu));
            qv[ks][nt][1] = to_float<QT>(static_cast<uint16_t>(raw2.x >> 16));
            qv[ks][nt][2] = to_float<QT>(static_cast<uint16_t>(raw2.y & 0xffffu));
            qv[ks][nt][3] = to_float<QT>(static_cast<uint16_t>(raw2.y >> 16));
#pragma unroll
            for (int i = 0; i < 4; ++i) amax = fmaxf(amax, fabsf(qv[ks][nt][i]));
          }
        }
        // warp max in one redux.sync: every lane's amax is a non-negative,
        // non-NaN float (fmaxf from +0 drops NaN), whose bits order as unsigned
        amax = __uint_as_float(__reduce_max_sync(FULL, __float_as_uint(amax)));
        int sh = 0;
        if (amax > 0.f && amax < INFINITY) {
          int e;
          frexpf(amax, &e);  // amax = m * 2^e, m in [0.5, 1)
          sh = (e - 1) - 14;
        }
        if (sh >= -126 && sh <= 127) {
          // 2^-sh from its exponent bits: one exact multiply per element
          const float r = __int_as_float((127 - sh) << 23);
#pragma unroll
          for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int ks = 0; ks < MT; ++ks) {
              qf[ks][nt][0] = pack2<false>(qv[ks][nt][0] * r, qv[ks][nt][1] * r);
              qf[ks][nt][1] = pack2<false>(qv[ks][nt][2] * r, qv[ks][nt][3] * r);
            }
        } else {  // |q| below 2^-112: 2^-sh is not a normal float
#pragma unroll
          for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int ks = 0; ks < MT; ++ks) {
              qf[ks][nt][0] = pack2<false>(ldexpf(qv[ks][nt][0], -sh), ldexpf(qv[ks][nt][1], -sh));
              qf[ks][nt][1] = pack2<false>(ldexpf(qv[ks][nt][2], -sh), ldexpf(qv[ks][nt][3], -sh));
            }
        }
        sc = ldexpf(a.score_scale, sh);
      }
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        m_run[nt][0] = m_run[nt][1] = MQ ? kMaskedFloor : -INFINITY;
        l_run[nt][0] = l_run[nt][1] = 0.f;
#pragma unroll
        for (int mt = 0; mt < MT; ++mt)
#pragma unroll
          for (int i = 0; i < 4; ++i) acc[mt][nt][i] = 0.f;
      }
    }

    const bool got = mbar_wait_bounded(wbars + 8 * slot, parity, kWaitLimitNs);
    if (!__all_sync(FULL, got)) {
      ok = false;
      break;
    }
    const uint32_t kt = ring + slot * Gm::STAGE_BYTES;
    const uint32_t vt = kt + Gm::TILE_BYTES;

    // tile position and edge masks
    const int L = s_len[cc.b];
    const int st = win_start(L, a.span);
    const int p0 = (st / kTile + cc.t) * kTile;
    const bool edge = (p0 < st) || (p0 + kTile > L);  // outside the pair's union range
    auto valid = [&](int r) { return !edge || (p0 + r >= st && p0 + r < L); };

    // ---- S^T = K . Q^T
    float sacc[NT][4];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int i = 0; i < 4; ++i) sacc[nt][i] = 0.f;
    if constexpr (!kFp8) {
#pragma unroll
      for (int ks = 0; ks < MT; ++ks) {
        uint32_t a0, a1, a2, a3;
        ldsm_x4(kt + tile_off(lane & 15, 2 * ks + (lane >> 4)), a0, a1, a2, a3);
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
          mma_16816<kBf16Mma>(sacc[nt], a0, a1, a2, a3, qf[ks][nt][0], qf[ks][nt][1]);
      }
    } else {
#pragma unroll
      for (int qd = 0; qd < D / 64; ++qd) {
        uint32_t wlo[4], whi[4];
        const int c = (64 * qd + 16 * t4) >> 4;
        lds_v4(kt + tile_off(g, c), wlo[0], wlo[1], wlo[2], wlo[3]);
        lds_v4(kt + tile_off(g + 8, c), whi[0], whi[1], whi[2], whi[3]);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const uint32_t a0 = e4m3x2_to_f16x2(static_cast<uint16_t>(wlo[j] & 0xffffu));
          const uint32_t a2 = e4m3x2_to_f16x2(static_cast<uint16_t>(wlo[j] >> 16));
          const uint32_t a1 = e4m3x2_to_f16x2(static_cast<uint16_t>(whi[j] & 0xffffu));
          const uint32_t a3 = e4m3x2_to_f16x2(static_cast<uint16_t>(whi[j] >> 16));
#pragma unroll
          for (int nt = 0; nt < NT; ++nt)
            mma_16816<false>(sacc[nt], a0, a1, a2, a3, qf[4 * qd + j][nt][0],
                             qf[4 * qd + j][nt][1]);
        }
      }
    }

    // ---- online softmax (log2 domain), P^T fragments
    const bool vlo = valid(g), vhi = valid(g + 8);
    // chunked: does some column's own range cut this tile?
    const bool cedge = MQ && (p0 < lo_max || p0 + kTile - 1 > hi_min);
    uint32_t pb[NT][2];
    // bf16 caches: P is split into a bf16 high part and a bf16 remainder, and
    // P.V runs on both, so P enters the product with ~16 bits instead of 8
    // (f16 P, used with f16 and FP8 caches, already has 11)
    uint32_t pr[NT][2];
    // scores (log2 domain) of the lane's rows g, g + 8 in columns 2 t4, 2 t4 + 1
    float sv[NT][4];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      if (MQ && cedge) {
        const int r0 = p0 + g, r1 = p0 + g + 8;
        sv[nt][0] = (r0 >= qlo[nt][0] && r0 <= qhi[nt][0]) ? sacc[nt][0] * sc : -INFINITY;
        sv[nt][1] = (r0 >= qlo[nt][1] && r0 <= qhi[nt][1]) ? sacc[nt][1] * sc : -INFINITY;
        sv[nt][2] = (r1 >= qlo[nt][0] && r1 <= qhi[nt][0]) ? sacc[nt][2] * sc : -INFINITY;
        sv[nt][3] = (r1 >= qlo[nt][1] && r1 <= qhi[nt][1]) ? sacc[nt][3] * sc : -INFINITY;
      } else {
        sv[nt][0] = vlo ? sacc[nt][0] * sc : -INFINITY;
        sv[nt][1] = vlo ? sacc[nt][1] * sc : -INFINITY;
        sv[nt][2] = vhi ? sacc[nt][2] * sc : -INFINITY;
        sv[nt][3] = vhi ? sacc[nt][3] * sc : -INFINITY;
      }
    }
    // A column's reference max m_run moves only when one of its scores
    // exceeds it by more than kRefSlack: the warp then takes the column maxima
    // across its lanes and rescales l and O (always on a segment's first
    // tile, whose reference starts at -inf or the floor). Every other tile
    // uses the reference as it is, so P stays below 2^kRefSlack.
    bool grow = false;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
      grow = grow || fmaxf(sv[nt][0], sv[nt][2]) > m_run[nt][0] + kRefSlack ||
             fmaxf(sv[nt][1], sv[nt][3]) > m_run[nt][1] + kRefSlack;
    if (__any_sync(FULL, grow)) {
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        float mx0 = fmaxf(sv[nt][0], sv[nt][2]), mx1 = fmaxf(sv[nt][1], sv[nt][3]);
#pragma unroll
        for (int o = 4; o < 32; o <<= 1) {
          mx0 = fmaxf(mx0, __shfl_xor_sync(FULL, mx0, o));
          mx1 = fmaxf(mx1, __shfl_xor_sync(FULL, mx1, o));
        }
        const float mn0 = fmaxf(m_run[nt][0], mx0), mn1 = fmaxf(m_run[nt][1], mx1);
        const float al0 = fast_exp2(m_run[nt][0] - mn0), al1 = fast_exp2(m_run[nt][1] - mn1);
        m_run[nt][0] = mn0;
        m_run[nt][1] = mn1;
        l_run[nt][0] *= al0;
        l_run[nt][1] *= al1;
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
          acc[mt][nt][0] *= al0;
          acc[mt][nt][1] *= al1;
          acc[mt][nt][2] *= al0;
          acc[mt][nt][3] *= al1;
        }
      }
    }
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      const float mn0 = m_run[nt][0], mn1 = m_run[nt][1];
      const float p0v = fast_exp2(sv[nt][0] - mn0), p1v = fast_exp2(sv[nt][1] - mn1);
      const float p2v = fast_exp2(sv[nt][2] - mn0), p3v = fast_exp2(sv[nt][3] - mn1);
      l_run[nt][0] += p0v + p2v;
      l_run[nt][1] += p1v + p3v;
      if constexpr (kBf16Mma) {
        const uint32_t h01 = pack2<true>(p0v, p1v), h23 = pack2<true>(p2v, p3v);
        pr[nt][0] = movmatrix_trans(pack2<true>(p0v - __uint_as_float(h01 << 16),
                                                p1v - __uint_as_float(h01 & 0xffff0000u)));
        pr[nt][1] = movmatrix_trans(pack2<true>(p2v - __uint_as_float(h23 << 16),
                                                p3v - __uint_as_float(h23 & 0xffff0000u)));
      }
      pb[nt][0] = movmatrix_trans(pack2<kBf16Mma>(p0v, p1v));
      pb[nt][1] = movmatrix_trans(pack2<kBf16Mma>(p2v, p3v));
    }

    // ---- O^T += V^T . P^T (the V rows of positions outside [start, L) are
    // zeroed in edge tiles only; interior tiles skip the masking work)
    auto pv = [&](auto masked) {
      constexpr bool kMask = decltype(masked)::value;
      uint32_t mlo = 0xffffffffu, mhi = 0xffffffffu;
      if constexpr (kMask) {
        mlo = (valid(2 * t4) ? 0x0000ffffu : 0u) | (valid(2 * t4 + 1) ? 0xffff0000u : 0u);
        mhi = (valid(2 * t4 + 8) ? 0x0000ffffu : 0u) | (valid(2 * t4 + 9) ? 0xffff0000u : 0u);
      }
      if constexpr (!kFp8) {
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
          uint32_t a0, a1, a2, a3;
          ldsm_x4_trans(vt + tile_off((lane & 7) + ((lane >> 4) << 3), 2 * mt + ((lane >> 3) & 1)),
                        a0, a1, a2, a3);
          if constexpr (kMask) {
            a0 &= mlo;
            a1 &= mlo;
            a2 &= mhi;
            a3 &= mhi;
          }
#pragma unroll
          for (int nt = 0; nt < NT; ++nt)
          {
            mma_16816<kBf16Mma>(acc[mt][nt], a0, a1, a2, a3, pb[nt][0], pb[nt][1]);
            if constexpr (kBf16Mma)
              mma_16816<true>(acc[mt][nt], a0, a1, a2, a3, pr[nt][0], pr[nt][1]);
          }
        }
      } else {
#pragma unroll
        for (int u = 0; u < D / 32; ++u) {
          const int dby = 32 * u + 4 * g;  // byte (= element) offset in the row
          const uint32_t co = (dby & 15);
          const int c = dby >> 4;
          const uint32_t w0 = lds_b32(vt + tile_off(2 * t4, c) + co);
          const uint32_t w1 = lds_b32(vt + tile_off(2 * t4 + 1, c) + co);
          const uint32_t w8 = lds_b32(vt + tile_off(2 * t4 + 8, c) + co);
          const uint32_t w9 = lds_b32(vt + tile_off(2 * t4 + 9, c) + co);
          const uint32_t x01a = __byte_perm(w0, w1, 0x5140), x01b = __byte_perm(w0, w1, 0x7362);
          const uint32_t x89a = __byte_perm(w8, w9, 0x5140), x89b = __byte_perm(w8, w9, 0x7362);
          // m-tile 2u: rows g, g+8 hold dims dby, dby+1; m-tile 2u+1: dby+2, dby+3
          uint32_t e0 = e4m3x2_to_f16x2(static_cast<uint16_t>(x01a & 0xffffu));
          uint32_t e1 = e4m3x2_to_f16x2(static_cast<uint16_t>(x01a >> 16));
          uint32_t e2 = e4m3x2_to_f16x2(static_cast<uint16_t>(x89a & 0xffffu));
          uint32_t e3 = e4m3x2_to_f16x2(static_cast<uint16_t>(x89a >> 16));
          uint32_t f0v = e4m3x2_to_f16x2(static_cast<uint16_t>(x01b & 0xffffu));
          uint32_t f1v = e4m3x2_to_f16x2(static_cast<uint16_t>(x01b >> 16));
          uint32_t f2v = e4m3x2_to_f16x2(static_cast<uint16_t>(x89b & 0xffffu));
          uint32_t f3v = e4m3x2_to_f16x2(static_cast<uint16_t>(x89b >> 16));
          if constexpr (kMask) {
            e0 &= mlo;
            e1 &= mlo;
            e2 &= mhi;
            e3 &= mhi;
            f0v &= mlo;
            f1v &= mlo;
            f2v &= mhi;
            f3v &= mhi;
          }
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) {
            mma_16816<false>(acc[2 * u][nt], e0, e1, e2, e3, pb[nt][0], pb[nt][1]);
            mma_16816<false>(acc[2 * u + 1][nt], f0v, f1v, f2v, f3v, pb[nt][0], pb[nt][1]);
          }
        }
      }
    };
    if (edge) pv(std::true_type{});
    else pv(std::false_type{});
    __syncwarp();
    ++consumed;
    // refill the stage just consumed
    if (produce(produced % STAGES)) ++produced;

    // ---- segment end: write the partial (m, l, unnormalised output)
    const bool seg_end = (flags & kFlagEnd) || (cc.t == cc.nt - 1);
    if (seg_end) {
      const int pair = cc.b * a.Hv + cc.kvh;
      const size_t pslot = (flags & kFlagPool)
                               ? static_cast<size_t>(npairs) + nw + pair + piece_id
                               : static_cast<size_t>(pair) + w;
      float* P = a.part + pslot * part_stride(a.CG, D);
      const float vs = kFp8 ? a.v_scale : 1.f;
      // kept in L2 for the merge kernel, which reads them right after
      const uint64_t keep = l2_evict_last();
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          float l = l_run[nt][e];
          l += __shfl_xor_sync(FULL, l, 4);
          l += __shfl_xor_sync(FULL, l, 8);
          l += __shfl_xor_sync(FULL, l, 16);
          const int h = 8 * nt + 2 * t4 + e;
          if (h < a.CG) {
            float* Ph = P + h * D;
#pragma unroll
            for (int mt = 0; mt < MT; ++mt) {
              st_f32_hint(Ph + acc_dim<kFp8>(mt, g, 0), acc[mt][nt][e] * vs, keep);
              st_f32_hint(Ph + acc_dim<kFp8>(mt, g, 1), acc[mt][nt][2 + e] * vs, keep);
            }
            if (g == 0) {
              st_f32_hint(P + a.CG * D + h, m_run[nt][e], keep);
              st_f32_hint(P + a.CG * D + a.CG + h, l, keep);
            }
          }
        }
      }
    }
  }

  if (!ok) {
    // Record the failure, then give the copies still in flight a bounded
    // chance to land before the warp leaves.
    if (lane == 0) atomicOr(a.err, kErrTimeout);
    for (int k = consumed; k < produced; ++k)
      (void)mbar_wait_bounded(wbars + 8 * (k % STAGES), (k / STAGES) & 1, kDrainLimitNs);
  }
}

// ---------------------------------------------------------------- host side

template <int CT, int QT, int D, int NT, int WARPS, int STAGES, bool MQ>
struct DecodeKernel {
  using Gm = Geometry<CT, D, STAGES>;
  static void* fn() {
    return reinterpret_cast<void*>(&paged_decode_kernel<CT, QT, D, NT, WARPS, STAGES, MQ>);
  }
  static DecodeVariant variant() { return DecodeVariant{WARPS, STAGES, WARPS * Gm::RING_BYTES}; }
  static cudaError_t prepare(int smem, int* ctas_per_sm) {
    cudaError_t e =
        cudaFuncSetAttribute(fn(), cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(ctas_per_sm, fn(), WARPS * 32, smem);
  }
  static cudaError_t launch(const CUtensorMap& tk, const CUtensorMap& tv, const DecodeArgs& a,
                            int grid, int smem, cudaStream_t s, bool pdl) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(WARPS * 32);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, paged_decode_kernel<CT, QT, D, NT, WARPS, STAGES, MQ>, tk,
                              tv, a);
  }
};

// Worker warps per CTA and pipeline stages per warp. Two CTAs share an SM.
// The e4m3 path with one n-tile at D = 128 spends about three times the
// instructions per byte of the 16-bit path, so it runs 8 warps of 3 stages
// (12 KB of ring each); every other variant runs 4 warps with about 24 KB of
// ring each (two stages at least).
template <int CT, int D, int NT>
constexpr int warps_for() {
  return (CT == kE4M3 && D == 128 && NT == 1) ? 8 : 4;
}

template <int CT, int D, int NT>
constexpr int stages_for() {
  constexpr int pair = 2 * kTile * D * ((CT == kE4M3) ? 1 : 2);
  constexpr int ring = (warps_for<CT, D, NT>() == 8) ? 12 * 1024 : 24 * 1024;
  constexpr int s = ring / pair;
  return s < 2 ? 2 : s;
}

// Expands `BODY` with the kernel type K for a runtime (D, NT) pair.
#define PA_DECODE_DISPATCH(CT, QT, MQ, D_, NT_, BODY)                             \
  do {                                                                            \
    if ((D_) == 64 && (NT_) == 1 && (CT) != kE4M3) {                              \
      constexpr int D0 = (CT) != kE4M3 ? 64 : 128;                                \
      using K = DecodeKernel<CT, QT, D0, 1, warps_for<CT, D0, 1>(),               \
                             stages_for<CT, D0, 1>(), MQ>;                        \
      BODY;                                                                       \
    } else if ((D_) == 64 && (NT_) == 2 && (CT) != kE4M3) {                       \
      constexpr int D0 = (CT) != kE4M3 ? 64 : 128;                                \
      using K = DecodeKernel<CT, QT, D0, 2, warps_for<CT, D0, 2>(),               \
                             stages_for<CT, D0, 2>(), MQ>;                        \
      BODY;                                                                       \
    } else if ((D_) == 128 && (NT_) == 1) {                                       \
      using K = DecodeKernel<CT, QT, 128, 1, warps_for<CT, 128, 1>(),            \
                             stages_for<CT, 128, 1>(), MQ>;                      \
      BODY;                                                                       \
    } else if ((D_) == 128 && (NT_) == 2) {                                       \
      using K = DecodeKernel<CT, QT, 128, 2, warps_for<CT, 128, 2>(),            \
                             stages_for<CT, 128, 2>(), MQ>;                      \
      BODY;                                                                       \
    } else if ((D_) == 256 && (NT_) == 1) {                                       \
      using K = DecodeKernel<CT, QT, 256, 1, warps_for<CT, 256, 1>(),            \
                             stages_for<CT, 256, 1>(), MQ>;                      \
      BODY;                                                                       \
    } else if ((D_) == 256 && (NT_) == 2) {                                       \
      using K = DecodeKernel<CT, QT, 256, 2, warps_for<CT, 256, 2>(),            \
                             stages_for<CT, 256, 2>(), MQ>;                      \
      BODY;                                                                       \
    } else {                                                                      \
      return cudaErrorInvalidValue;                                               \
    }                                                                             \
  } while (0)

// The three entry points of one (cache type, q type, chunked) family; each
// translation unit defines one or two families so that they build in parallel.
#define PA_DECODE_FAMILY(NAME, CT, QT, MQ)                                             \
  cudaError_t decode_variant_##NAME(int D, int nt, DecodeVariant* v) {                  \
    PA_DECODE_DISPATCH(CT, QT, MQ, D, nt, {                                            \
      *v = K::variant();                                                               \
      return cudaSuccess;                                                              \
    });                                                                                \
  }                                                                                    \
  cudaError_t decode_prepare_##NAME(int D, int nt, int smem, int* ctas_per_sm) {        \
    PA_DECODE_DISPATCH(CT, QT, MQ, D, nt, { return K::prepare(smem, ctas_per_sm); });  \
  }                                                                                    \
  cudaError_t decode_launch_##NAME(int D, int nt, const CUtensorMap& tk,                \
                                   const CUtensorMap& tv, const DecodeArgs& a, int grid, \
                                   int smem, cudaStream_t s, bool pdl) {               \
    PA_DECODE_DISPATCH(CT, QT, MQ, D, nt,                                              \
                       { return K::launch(tk, tv, a, grid, smem, s, pdl); });          \
  }

}  // namespace pa
