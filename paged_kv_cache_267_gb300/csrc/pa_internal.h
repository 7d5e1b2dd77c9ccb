// Internal declarations shared by the C-ABI layer and the kernel translation
// units. Host-only types; no kernel code here.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace pa {

// Element type codes used inside the library (same values as the ABI enums).
enum ElemType { kF16 = 0, kBF16 = 1, kE4M3 = 2 };

constexpr int kTile = 16;  // tokens per pipeline tile (one mma m-tile)

// Floats per decode partial slot: acc[G][D], m[G], l[G], rounded up to a
// multiple of 4 so that slots can be read with 16-byte vector loads.
__host__ __device__ constexpr inline int part_stride(int G, int D) {
  return G * D + ((2 * G + 3) & ~3);
}

// Decode workspace layout (device memory, all sections 256-byte aligned):
//   pool  u32 [3] at offset 0, at the same place for any shape, all zero
//         between calls (the merge kernel resets them after each step):
//         [0] the pool piece counter; [1] the plan flag, set to 1 (release)
//         by the decode kernel's first CTA once the plan below is stored;
//         [2] the merge CTAs that have read the flag
//   plan  int32 [plan_words(B)] at offset 256: the step's plan, written by the
//         decode kernel's first CTA before it streams, read by the merge
//         kernel: kPlanScalars scalars (tiles, static tiles per warp, end of
//         the static region, piece size, pieces, unused) and the tile prefix
//         over the sequences (B + 1)
//   part  f32 [NSLOT][part_stride(CG, D)]: acc[CG][D], m[CG], l[CG], padding
//         to a multiple of 4 floats so every slot starts 16-byte aligned
// with S = B * Hv pairs, NW worker warps, NSLOT = 2 S + NW + NPMAX. For
// single-query decode Hv = Hkv and CG = G (columns are the group's q heads).
// A segment is a run of one warp's tiles inside one pair. Static segments of
// pair s by warp w use slot s + w; segments of pool piece i use slot
// S + NW + s + i. Both are unique because the walk through the (pair, warp)
// and (pair, piece) grids is a monotone staircase.
constexpr int kPlanScalars = 8;
__host__ __device__ constexpr inline int plan_words(int B) { return kPlanScalars + B + 1; }
constexpr int kMergeNarrow = 8;  // partials one merge warp folds in one round trip

struct DecodeArgs {
  const void* q;                 // [B, T, Hq, D] ([B, Hq, D] when T = 1)
  const int32_t* block_tables;   // [B, MB]
  const int32_t* seq_lens;       // [B]
  uint32_t* pool;
  int32_t* plan;                 // plan region, written by the first CTA
  float* part;
  int32_t* err;                  // device error word
  int B, Hq, Hkv, G, D, bs, MB, NB, window;
  int T;                         // queries per sequence, at its last T positions
  int NCG;                       // column groups per kv head (1 when T * G <= 16)
  int CG;                        // (query, head) columns per pair: T * G, or 16
  int Hv;                        // pairs per sequence: Hkv * NCG
  int span;                      // window of the pairs' tile ranges: W + T - 1, 0 if W = 0
  float score_scale;             // scale * log2(e) (* k_scale for FP8)
  float v_scale;                 // FP8: applied to the partial outputs
  int min_tiles;                 // least tiles per warp in the static split
  int pool_permille;             // share of tiles handed out dynamically
  int piece_min;                 // least tiles per pool piece
  int np_max;                    // most pool pieces (bounds the slots)
};

struct MergeArgs {
  void* out;                     // [B, T, Hq, D], dtype of q
  const float* part;
  const int32_t* plan;           // the decode kernel's plan region
  uint32_t* pool;                // reset to zero for the next step
  int B, Hq, Hkv, G, D, NW;
  int T, NCG, CG, Hv;            // as in DecodeArgs
};

// Bound on output columns (batch * q heads * queries) of one call.
constexpr int kMaxColumns = 1 << 19;

struct ReshapeArgs {
  const void* k;
  const void* v;
  void* kc;
  void* vc;
  const int64_t* slots;
  int32_t* err;
  int64_t k_stride_t, k_stride_h, v_stride_t, v_stride_h;  // elements
  int T, H, D, bs;
  int64_t NB;
  float k_scale, v_scale;
};

// Chunked queries on the tensor-memory kernel (chunk_tc.cu): one CTA per
// (sequence, KV head, unit of chunk_tc_unit_rows() (query, head) rows); head
// dim 128, 16-bit or e4m3 caches.
struct ChunkArgs {
  const void* q;                 // [B, T, Hq, D]
  void* out;                     // [B, T, Hq, D]
  const int32_t* block_tables;   // [B, MB]
  const int32_t* seq_lens;       // [B]
  int32_t* err;                  // device error word
  int B, T, Hq, Hkv, G, bs, MB, NB, window;
  int QT;                        // units per (sequence, KV head): ceil(T * G / unit rows)
  float score_scale;             // scale * log2(e) (* k_scale for FP8)
  float v_scale;                 // FP8: applied to the output
};
int chunk_tc_unit_rows();
cudaError_t chunk_tc_prepare();  // once per device: the kernel's shared-memory size
cudaError_t chunk_tc_launch(int qt, bool fp8, const CUtensorMap& tk, const CUtensorMap& tv,
                            const ChunkArgs& a, cudaStream_t s, bool pdl);

// Kernel configuration chosen for a (cache type, q type, D, n-tiles) variant.
struct DecodeVariant {
  int warps;          // worker warps per CTA
  int stages;         // pipeline stages per warp
  int ring_bytes;     // shared memory for the K/V rings of one CTA
};

// Per-variant entry points of one (cache type, q type, chunked) family,
// implemented in decode_[mq_]<type>.cu. Each returns cudaErrorInvalidValue for
// an unsupported (D, NT) combination.
#define PA_DECLARE_DECODE_FAMILY(NAME)                                                   \
  cudaError_t decode_variant_##NAME(int D, int nt, DecodeVariant* v);                    \
  cudaError_t decode_prepare_##NAME(int D, int nt, int smem_bytes, int* ctas_per_sm);    \
  cudaError_t decode_launch_##NAME(int D, int nt, const CUtensorMap& tk,                 \
                                   const CUtensorMap& tv, const DecodeArgs& a, int grid, \
                                   int smem, cudaStream_t s, bool pdl);
PA_DECLARE_DECODE_FAMILY(f16)
PA_DECLARE_DECODE_FAMILY(bf16)
PA_DECLARE_DECODE_FAMILY(fp8_f16)
PA_DECLARE_DECODE_FAMILY(fp8_bf16)
PA_DECLARE_DECODE_FAMILY(mq_f16)
PA_DECLARE_DECODE_FAMILY(mq_bf16)
PA_DECLARE_DECODE_FAMILY(mq_fp8_f16)
PA_DECLARE_DECODE_FAMILY(mq_fp8_bf16)
#undef PA_DECLARE_DECODE_FAMILY

// merge_reshape.cu
cudaError_t merge_launch(int out_type, const MergeArgs& a, int grid, cudaStream_t s, bool pdl);
cudaError_t reshape_launch(int src_type, bool fp8, const ReshapeArgs& a, cudaStream_t s);
cudaError_t device_error_word(int32_t** ptr);  // address of this device's error word

}  // namespace pa

#include "pa.h"

#include <exception>
#include <new>

namespace pa {

// Records a message for pa_last_error() on the calling thread and returns
// `code` (pa_api.cpp; never throws).
pa_status set_error(pa_status code, const char* msg);
pa_status set_cuda_error(cudaError_t e, const char* what);

// Runs an entry point's body so that no C++ exception leaves it: host memory
// exhaustion becomes PA_ERR_HOST_MEMORY, any other exception from the C++
// runtime (a mutex that cannot be locked, for one) PA_ERR_CUDA.
template <typename F>
pa_status abi_guard(F&& body) noexcept {
  try {
    return body();
  } catch (const std::bad_alloc&) {
    return set_error(PA_ERR_HOST_MEMORY, "host memory exhausted");
  } catch (const std::exception& ex) {
    return set_error(PA_ERR_CUDA, ex.what());
  } catch (...) {
    return set_error(PA_ERR_CUDA, "unexpected host exception");
  }
}

// pa_decode with the scratch in a given device buffer (pa_api.cpp).
pa_status decode_in_buffer(const pa_tensor* out, const pa_tensor* q, const pa_tensor* key_cache,
                           const pa_tensor* value_cache, const pa_tensor* block_tables,
                           const pa_tensor* seq_lens, int32_t num_kv_heads, float scale,
                           int32_t block_size, int32_t window, int32_t kv_dtype, float k_scale,
                           float v_scale, pa_stream stream, void* buffer, size_t capacity);

}  // namespace pa
