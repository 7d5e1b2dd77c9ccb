// C-ABI layer of libpa: argument validation, workspace management, TMA
// descriptor encoding, variant dispatch and launch on the caller's stream.
// All validation happens on the host before any CUDA call, so argument
// errors are reported without touching the device.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <initializer_list>
#include <map>
#include <mutex>
#include <new>
#include <tuple>

#include "pa.h"
#include "pa_internal.h"

namespace pa {
// Defined in selftest.cu: one CTA whose two waits (an mbarrier phase, a
// device flag) can never be satisfied; each gives up after limit_ns, sets
// PA_DEVERR_TIMEOUT in *err and stores its duration in elapsed[0 .. 2)
// (elapsed may be null).
cudaError_t bounded_wait_selftest(int32_t* err, uint64_t limit_ns, uint64_t* elapsed,
                                  cudaStream_t s);
}  // namespace pa

namespace {

thread_local char g_last_error[512] = "";  // no host allocation on any error path
std::atomic<uint64_t> g_launches{0};
std::atomic<int32_t> g_tune_max_ctas{0};
std::atomic<int32_t> g_tune_min_tiles{0};
std::atomic<int32_t> g_tune_pool{0};
std::atomic<int32_t> g_tune_piece{0};
std::atomic<int32_t> g_chunk_path{0};  // 0 auto, 1 persistent kernel, 2 tensor-memory kernel
thread_local void* g_prof_before = nullptr;
thread_local void* g_prof_after = nullptr;

constexpr int kDefaultMinTiles = 1;  // small steps: as many warps as tiles (latency)
constexpr int kDefaultPoolPermille = 100;  // share of tiles handed out dynamically
constexpr int kDefaultPiece = 4;           // least tiles per pool piece
// e4m3 caches, one query: every piece is a segment whose start (q converted
// and rescaled to f16) costs issue slots in that issue-bound variant
constexpr int kDefaultPieceFp8 = 8;
constexpr int kPiecesPerWorker = 4;        // pool pieces per worker warp, at most
constexpr int kMaxCtasPerSm = 2;
constexpr int kWarpsPerCta = 8;  // most worker warps of any decode variant
constexpr int64_t kMaxBatch = 4096;
constexpr int64_t kMaxChunk = 4096;        // query tokens per sequence in a chunk call
constexpr double kMaxTensorBytes = 1125899906842624.0;  // 2^50: no tensor is larger
// Chunks with more (query, head) columns per KV head than this go to the
// tensor-memory kernel (head dim 128, 16-bit or e4m3 caches): the persistent kernel
// reads each K/V tile once per 16 columns.
constexpr int64_t kTcMinColumns = 32;

pa_status fail(pa_status code, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_last_error, sizeof(g_last_error), fmt, ap);
  va_end(ap);
  return code;
}

pa_status ok() {
  g_last_error[0] = '\0';
  return PA_OK;
}

pa_status cuda_fail(cudaError_t e, const char* what) {
  return fail(PA_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

int elem_size(int32_t dt) {
  switch (dt) {
    case PA_F16:
    case PA_BF16: return 2;
    case PA_FP8_E4M3: return 1;
    case PA_I32: return 4;
    case PA_I64: return 8;
    default: return 0;
  }
}

// A tensor with no elements has no layout to get wrong (torch gives empty
// views strides of 0), so it counts as contiguous.
bool is_contiguous(const pa_tensor* t) {
  for (int i = 0; i < t->ndim; ++i)
    if (t->shape[i] == 0) return true;
  int64_t expect = 1;
  for (int i = t->ndim - 1; i >= 0; --i) {
    if (t->shape[i] != 1 && t->strides[i] != expect) return false;
    expect *= t->shape[i];
  }
  return true;
}

int64_t numel(const pa_tensor* t) {
  int64_t n = 1;
  for (int i = 0; i < t->ndim; ++i) n *= t->shape[i];
  return n;
}

// Byte span [lo, hi) covered by a tensor (assumes non-negative strides).
void span(const pa_tensor* t, uintptr_t* lo, uintptr_t* hi) {
  int64_t last = 0;
  for (int i = 0; i < t->ndim; ++i) last += (t->shape[i] - 1) * t->strides[i];
  *lo = reinterpret_cast<uintptr_t>(t->data);
  *hi = *lo + static_cast<uintptr_t>((last + 1) * elem_size(t->dtype));
}

bool overlaps(const pa_tensor* a, const pa_tensor* b) {
  if (numel(a) == 0 || numel(b) == 0) return false;
  uintptr_t alo, ahi, blo, bhi;
  span(a, &alo, &ahi);
  span(b, &blo, &bhi);
  return alo < bhi && blo < ahi;
}

pa_status check_tensor(const pa_tensor* t, const char* name, int ndim) {
  if (!t) return fail(PA_ERR_INVALID_ARG, "%s: null tensor", name);
  if (t->ndim != ndim) return fail(PA_ERR_INVALID_ARG, "%s: expected %d dims, got %d", name, ndim, t->ndim);
  if (elem_size(t->dtype) == 0) return fail(PA_ERR_INVALID_ARG, "%s: bad dtype %d", name, t->dtype);
  for (int i = 0; i < ndim; ++i) {
    if (t->shape[i] < 0) return fail(PA_ERR_INVALID_ARG, "%s: negative extent", name);
    if (t->strides[i] < 0) return fail(PA_ERR_LAYOUT, "%s: negative stride", name);
  }
  // Extents and spans beyond any memory are rejected here (counted in double,
  // which cannot overflow), so the 64-bit size arithmetic after this check
  // stays in range for any descriptor.
  double n = 1.0, last = 0.0;
  for (int i = 0; i < ndim; ++i) {
    n *= static_cast<double>(t->shape[i]);
    if (t->shape[i] > 0)
      last += static_cast<double>(t->shape[i] - 1) * static_cast<double>(t->strides[i]);
  }
  const double elt = static_cast<double>(elem_size(t->dtype));
  if (n * elt >= kMaxTensorBytes || (n > 0 && (last + 1.0) * elt >= kMaxTensorBytes))
    return fail(PA_ERR_UNSUPPORTED, "%s: extent or span beyond 2^50 bytes", name);
  if (!t->data && numel(t) > 0) return fail(PA_ERR_INVALID_ARG, "%s: null data", name);
  return PA_OK;
}

// Product of sizes in double, for limit checks that must not overflow.
double dprod(std::initializer_list<double> f) {
  double p = 1.0;
  for (double x : f) p *= x;
  return p;
}

// The kernels may only touch memory of the current device, or pinned host
// memory mapped into its address space at the same address (on GB300 the
// kernels then read and write it over the CPU-GPU link). Anything else
// (pageable host memory, another device's memory) is rejected before launch.
pa_status check_accessible_ptr(const void* p, const char* name) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  cudaPointerAttributes at;
  e = cudaPointerGetAttributes(&at, p);
  if (e != cudaSuccess) return cuda_fail(e, "cudaPointerGetAttributes");
  if ((at.type == cudaMemoryTypeDevice || at.type == cudaMemoryTypeManaged) && at.device == dev)
    return PA_OK;
  if (at.type == cudaMemoryTypeHost && at.devicePointer == p) return PA_OK;
  return fail(PA_ERR_INVALID_ARG,
              "%s: memory not accessible from the current device (use device memory or pinned, "
              "mapped host memory)",
              name);
}

pa_status check_accessible(const pa_tensor* t, const char* name) {
  if (!t || numel(t) == 0 || !t->data) return PA_OK;
  return check_accessible_ptr(t->data, name);
}

// ------------------------------------------------------------ device state

struct Workspace {
  void* ptr = nullptr;
  size_t bytes = 0;
  bool dirty = false;  // the pool counter may be nonzero (a merge launch failed)
};

struct DeviceState {
  bool init = false;
  int num_sms = 0;
  int32_t* err_word = nullptr;
  bool chunk_tc_ready = false;              // tensor-memory kernel configured
  Workspace user_ws;                        // caller-owned (pa_set_workspace)
  std::map<uintptr_t, Workspace> lib_ws;    // library-owned, one per stream
  std::map<std::tuple<int, int, int, int, int, bool>, int> occupancy;
};

std::mutex g_mu;
std::map<int, DeviceState> g_dev;

pa_status device_state(DeviceState** out, int* dev_out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  DeviceState* stp;
  try {
    stp = &g_dev[dev];
  } catch (const std::bad_alloc&) {
    return fail(PA_ERR_HOST_MEMORY, "host memory exhausted");
  }
  DeviceState& st = *stp;
  if (!st.init) {
    e = cudaDeviceGetAttribute(&st.num_sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceGetAttribute");
    e = pa::device_error_word(&st.err_word);
    if (e != cudaSuccess) return cuda_fail(e, "device error word");
    st.init = true;
  }
  *out = &st;
  if (dev_out) *dev_out = dev;
  return PA_OK;
}

size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Section offsets of the decode workspace (layout described in pa_internal.h).
struct WsLayout {
  size_t pool, plan, part, total;
};

// Hv pairs per sequence with CG columns each (Hkv and G for single-query decode).
WsLayout ws_layout(int64_t B, int Hv, int CG, int D, int64_t workers) {
  const size_t S = static_cast<size_t>(B) * Hv;
  const size_t nslot = 2 * S + workers + static_cast<size_t>(workers) * kPiecesPerWorker;
  WsLayout L;
  size_t o = 0;
  // The pool counter sits at a fixed offset: it must stay zero between calls
  // whatever their shapes, and each step's merge only resets its own copy.
  L.pool = o;  o += 256;
  L.plan = o;  o += round_up(static_cast<size_t>(pa::plan_words(static_cast<int>(B))) * 4, 256);
  L.part = o;  o += nslot * static_cast<size_t>(pa::part_stride(CG, D)) * sizeof(float);
  L.total = o;
  return L;
}

int tuned_pool_permille() {
  const int v = g_tune_pool.load();
  return v == 0 ? kDefaultPoolPermille : (v < 0 ? 0 : v);
}

int tuned_piece(bool fp8_decode) {
  const int v = g_tune_piece.load();
  return v > 0 ? v : (fp8_decode ? kDefaultPieceFp8 : kDefaultPiece);
}

// ------------------------------------------------------------ TMA descriptors

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// 2-D view of a cache [NB * Hkv * bs rows, D]: box of 16 rows x 128 bytes,
// 128-byte swizzle.
pa_status make_cache_map(CUtensorMap* map, const void* base, int64_t rows, int D, int elt) {
  auto fn = encode_fn();
  if (!fn) return fail(PA_ERR_CUDA, "cuTensorMapEncodeTiled is not available");
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(D) * elt};
  cuuint32_t box[2] = {static_cast<cuuint32_t>(128 / elt), static_cast<cuuint32_t>(pa::kTile)};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(map, elt == 1 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_UINT16,
                  2, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(PA_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", (int)r);
  return PA_OK;
}

// ------------------------------------------------------------ dispatch glue

// The kernel family of a (cache type, q type, chunked) combination.
struct Family {
  cudaError_t (*variant)(int D, int nt, pa::DecodeVariant* v);
  cudaError_t (*prepare)(int D, int nt, int smem, int* ctas_per_sm);
  cudaError_t (*launch)(int D, int nt, const CUtensorMap& tk, const CUtensorMap& tv,
                        const pa::DecodeArgs& a, int grid, int smem, cudaStream_t s, bool pdl);
};

#define PA_FAMILY(NAME) \
  Family { pa::decode_variant_##NAME, pa::decode_prepare_##NAME, pa::decode_launch_##NAME }

Family family_of(int ct, int qt, bool mq) {
  if (ct == pa::kE4M3) {
    if (qt == pa::kBF16) return mq ? PA_FAMILY(mq_fp8_bf16) : PA_FAMILY(fp8_bf16);
    return mq ? PA_FAMILY(mq_fp8_f16) : PA_FAMILY(fp8_f16);
  }
  if (ct == pa::kBF16) return mq ? PA_FAMILY(mq_bf16) : PA_FAMILY(bf16);
  return mq ? PA_FAMILY(mq_f16) : PA_FAMILY(f16);
}
#undef PA_FAMILY

struct DecodePlan {
  Family fam;
  int nt;
  int smem, grid, workers, min_tiles, pool_permille, piece;
  pa::DecodeVariant var;
};

// Shape validation shared by pa_decode and the workspace query.
pa_status check_heads(int64_t Hq, int64_t Hkv, int64_t D) {
  if (Hkv <= 0 || Hq <= 0) return fail(PA_ERR_INVALID_ARG, "head counts must be positive");
  if (Hq % Hkv) return fail(PA_ERR_INVALID_ARG, "num_q_heads %% num_kv_heads != 0");
  if (Hq / Hkv > 16) return fail(PA_ERR_UNSUPPORTED, "GQA group %lld > 16", (long long)(Hq / Hkv));
  if (D != 64 && D != 128 && D != 256) return fail(PA_ERR_UNSUPPORTED, "head_dim %lld", (long long)D);
  return PA_OK;
}

// Columns per pair and column groups for T queries of a G-head group.
void chunk_columns(int64_t T, int G, int* CG, int* NCG) {
  const int64_t cols = T * G;
  *NCG = static_cast<int>((cols + 15) / 16);
  *CG = *NCG == 1 ? static_cast<int>(cols) : 16;
}

pa_status plan_decode(DeviceState* st, int ct, int qt, bool mq, int64_t B, int CG, int D,
                      DecodePlan* p) {
  p->fam = family_of(ct, qt, mq);
  p->nt = CG > 8 ? 2 : 1;
  cudaError_t e = p->fam.variant(D, p->nt, &p->var);
  if (e != cudaSuccess) return fail(PA_ERR_UNSUPPORTED, "no decode kernel for this dtype/head_dim");
  const size_t smem = 1024 + p->var.ring_bytes + p->var.warps * p->var.stages * (8 + 8) +
                      static_cast<size_t>(2 * B + 1) * sizeof(int32_t);
  p->smem = static_cast<int>(round_up(smem, 1024));
  auto key = std::make_tuple(ct, qt, D, p->nt, p->smem, mq);
  auto it = st->occupancy.find(key);
  int ctas = 0;
  if (it == st->occupancy.end()) {
    e = p->fam.prepare(D, p->nt, p->smem, &ctas);
    if (e != cudaSuccess) return cuda_fail(e, "decode kernel setup");
    try {
      st->occupancy[key] = ctas;
    } catch (const std::bad_alloc&) {
      return fail(PA_ERR_HOST_MEMORY, "host memory exhausted");
    }
  } else {
    ctas = it->second;
  }
  if (ctas < 1) return fail(PA_ERR_UNSUPPORTED, "decode kernel does not fit on an SM (smem %d)", p->smem);
  if (ctas > kMaxCtasPerSm) ctas = kMaxCtasPerSm;
  p->grid = st->num_sms * ctas;
  const int cap = g_tune_max_ctas.load();
  if (cap > 0 && p->grid > cap) p->grid = cap;
  p->workers = p->grid * p->var.warps;
  const int mt = g_tune_min_tiles.load();
  p->min_tiles = mt > 0 ? mt : kDefaultMinTiles;
  p->pool_permille = tuned_pool_permille();
  p->piece = tuned_piece(ct == pa::kE4M3 && !mq);
  return PA_OK;
}

// Picks the workspace for this call (zeroed on allocation: the pool counter
// starts at zero, and each step's merge kernel leaves it at zero).
pa_status get_workspace(DeviceState* st, cudaStream_t stream, const WsLayout& lay, void** ws,
                        Workspace** wsp) {
  Workspace* w;
  const size_t need = lay.total;
  if (st->user_ws.ptr) {
    if (st->user_ws.bytes < need)
      return fail(PA_ERR_WORKSPACE, "workspace too small: %zu bytes set, %zu needed",
                  st->user_ws.bytes, need);
    w = &st->user_ws;
  } else {
    try {
      w = &st->lib_ws[reinterpret_cast<uintptr_t>(stream)];
    } catch (const std::bad_alloc&) {
      return fail(PA_ERR_HOST_MEMORY, "host memory exhausted");
    }
    if (w->bytes < need) {
      cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
      cudaError_t e = cudaStreamIsCapturing(stream, &cap);
      if (e != cudaSuccess) return cuda_fail(e, "cudaStreamIsCapturing");
      if (cap != cudaStreamCaptureStatusNone)
        return fail(PA_ERR_WORKSPACE,
                    "decode workspace must grow to %zu bytes during stream capture; run one "
                    "step before capturing or call pa_set_workspace",
                    need);
      if (w->ptr) {
        e = cudaStreamSynchronize(stream);
        if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
        cudaFree(w->ptr);
        *w = Workspace{};
      }
      const size_t bytes = round_up(need + need / 4, 1 << 20);
      void* p = nullptr;
      e = cudaMalloc(&p, bytes);
      if (e != cudaSuccess) return cuda_fail(e, "cudaMalloc(workspace)");
      e = cudaMemsetAsync(p, 0, bytes, stream);
      if (e != cudaSuccess) {
        cudaFree(p);
        return cuda_fail(e, "cudaMemsetAsync(workspace)");
      }
      w->ptr = p;
      w->bytes = bytes;
    }
  }
  if (w->dirty) {
    cudaError_t e = cudaMemsetAsync(static_cast<char*>(w->ptr) + lay.pool, 0,
                                    lay.plan - lay.pool, stream);
    if (e != cudaSuccess) return cuda_fail(e, "cudaMemsetAsync(pool counter)");
    w->dirty = false;
  }
  *ws = w->ptr;
  *wsp = w;
  return PA_OK;
}

}  // namespace

extern "C" {

const char* pa_last_error(void) { return g_last_error; }

int32_t pa_version(void) { return 10000; }

uint64_t pa_launch_count(void) { return g_launches.load(); }

pa_status pa_set_decode_tuning(int32_t max_ctas, int32_t min_tiles, int32_t pool_permille,
                               int32_t piece_tiles) {
  if (max_ctas < 0 || min_tiles < 0 || piece_tiles < 0)
    return fail(PA_ERR_INVALID_ARG, "negative tuning value");
  if (pool_permille > 1000 || piece_tiles > (1 << 20) || min_tiles > (1 << 20))
    return fail(PA_ERR_INVALID_ARG, "tuning value out of range");
  g_tune_max_ctas = max_ctas;
  g_tune_min_tiles = min_tiles;
  g_tune_pool = pool_permille;
  g_tune_piece = piece_tiles;
  return ok();
}

pa_status pa_set_prefill_path(int32_t path) {
  if (path < 0 || path > 2) return fail(PA_ERR_INVALID_ARG, "path must be 0, 1 or 2");
  g_chunk_path = path;
  return ok();
}

pa_status pa_profile_events(void* ev_before, void* ev_after) {
  if ((ev_before == nullptr) != (ev_after == nullptr))
    return fail(PA_ERR_INVALID_ARG, "give both events or neither");
  g_prof_before = ev_before;
  g_prof_after = ev_after;
  return ok();
}

pa_status pa_set_workspace(void* ptr, size_t bytes) {
  return pa::abi_guard([&]() -> pa_status {
    if (ptr && (reinterpret_cast<uintptr_t>(ptr) % 256))
      return fail(PA_ERR_LAYOUT, "workspace must be 256-byte aligned");
    std::lock_guard<std::mutex> lk(g_mu);
    DeviceState* st;
    pa_status s = device_state(&st, nullptr);
    if (s) return s;
    if (ptr && bytes) {
      // The pool counter must start at zero; zero the whole buffer.
      cudaError_t e = cudaMemset(ptr, 0, bytes);
      if (e == cudaSuccess) e = cudaDeviceSynchronize();
      if (e != cudaSuccess) return cuda_fail(e, "zeroing the workspace");
    }
    st->user_ws = Workspace{};
    if (ptr) {
      st->user_ws.ptr = ptr;
      st->user_ws.bytes = bytes;
    }
    return ok();
  });
}

}  // extern "C"

namespace {

pa_status workspace_size(int64_t batch, int64_t num_queries, int32_t num_q_heads,
                         int32_t num_kv_heads, int32_t head_dim, size_t* bytes) {
  if (!bytes) return fail(PA_ERR_INVALID_ARG, "bytes is null");
  if (num_queries < 1 || num_queries > kMaxChunk)
    return fail(PA_ERR_UNSUPPORTED, "num_queries %lld", (long long)num_queries);
  if (batch < 0 || batch > kMaxBatch) return fail(PA_ERR_UNSUPPORTED, "batch %lld", (long long)batch);
  pa_status s = check_heads(num_q_heads, num_kv_heads, head_dim);
  if (s) return s;
  int CG, NCG;
  chunk_columns(num_queries, num_q_heads / num_kv_heads, &CG, &NCG);
  const int64_t Hv = static_cast<int64_t>(num_kv_heads) * NCG;
  if (dprod({double(batch), double(Hv), double(CG)}) > pa::kMaxColumns)
    return fail(PA_ERR_UNSUPPORTED, "batch * num_q_heads * num_queries too large");
  std::lock_guard<std::mutex> lk(g_mu);
  DeviceState* st;
  s = device_state(&st, nullptr);
  if (s) return s;
  int64_t workers = static_cast<int64_t>(st->num_sms) * kMaxCtasPerSm * kWarpsPerCta;
  const int cap = g_tune_max_ctas.load();
  if (cap > 0 && cap * kWarpsPerCta < workers) workers = static_cast<int64_t>(cap) * kWarpsPerCta;
  *bytes = ws_layout(batch, static_cast<int>(Hv), CG, head_dim, workers).total;
  return ok();
}

}  // namespace

extern "C" {

pa_status pa_decode_workspace_size(int64_t batch, int32_t num_q_heads, int32_t num_kv_heads,
                                   int32_t head_dim, size_t* bytes) {
  return pa::abi_guard([&]() -> pa_status {
    return workspace_size(batch, 1, num_q_heads, num_kv_heads, head_dim, bytes);
  });
}

pa_status pa_prefill_chunk_workspace_size(int64_t batch, int32_t num_queries, int32_t num_q_heads,
                                          int32_t num_kv_heads, int32_t head_dim, size_t* bytes) {
  return pa::abi_guard([&]() -> pa_status {
    return workspace_size(batch, num_queries, num_q_heads, num_kv_heads, head_dim, bytes);
  });
}

pa_status pa_check_device_error(int32_t* bits, pa_stream stream) {
  return pa::abi_guard([&]() -> pa_status {
    if (!bits) return fail(PA_ERR_INVALID_ARG, "bits is null");
    DeviceState* st;
    {
      std::lock_guard<std::mutex> lk(g_mu);
      pa_status s = device_state(&st, nullptr);
      if (s) return s;
    }
    cudaStream_t cs = static_cast<cudaStream_t>(stream);
    int32_t v = 0;
    cudaError_t e = cudaMemcpyAsync(&v, st->err_word, sizeof(v), cudaMemcpyDeviceToHost, cs);
    if (e == cudaSuccess) e = cudaMemsetAsync(st->err_word, 0, sizeof(int32_t), cs);
    if (e == cudaSuccess) e = cudaStreamSynchronize(cs);
    if (e != cudaSuccess) return cuda_fail(e, "reading the device error word");
    *bits = v;
    return ok();
  });
}

pa_status pa_selftest_bounded_wait(uint32_t limit_us, uint64_t* elapsed_ns, pa_stream stream) {
  return pa::abi_guard([&]() -> pa_status {
    if (limit_us < 1 || limit_us > 1000000)
      return fail(PA_ERR_INVALID_ARG, "limit_us must be in [1, 1000000]");
    pa_status s;
    if (elapsed_ns && reinterpret_cast<uintptr_t>(elapsed_ns) % alignof(uint64_t))
      return fail(PA_ERR_INVALID_ARG, "elapsed_ns must be 8-byte aligned");
    if (elapsed_ns && (s = check_accessible_ptr(elapsed_ns, "elapsed_ns"))) return s;
    DeviceState* st;
    {
      std::lock_guard<std::mutex> lk(g_mu);
      s = device_state(&st, nullptr);
      if (s) return s;
    }
    cudaError_t e = pa::bounded_wait_selftest(st->err_word, 1000ull * limit_us, elapsed_ns,
                                              static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "self-test launch");
    g_launches += 1;
    return ok();
  });
}

pa_status pa_reshape_and_cache(const pa_tensor* k, const pa_tensor* v, const pa_tensor* key_cache,
                               const pa_tensor* value_cache, const pa_tensor* slot_mapping,
                               int32_t kv_dtype, float k_scale, float v_scale, pa_stream stream) {
  return pa::abi_guard([&]() -> pa_status {
    pa_status s;
    if ((s = check_tensor(k, "k", 3)) || (s = check_tensor(v, "v", 3)) ||
        (s = check_tensor(key_cache, "key_cache", 4)) ||
        (s = check_tensor(value_cache, "value_cache", 4)) ||
        (s = check_tensor(slot_mapping, "slot_mapping", 1)))
      return s;
    if (k->dtype != PA_F16 && k->dtype != PA_BF16)
      return fail(PA_ERR_UNSUPPORTED, "k must be f16 or bf16");
    if (v->dtype != k->dtype) return fail(PA_ERR_INVALID_ARG, "k and v dtypes differ");
    for (int i = 0; i < 3; ++i)
      if (k->shape[i] != v->shape[i]) return fail(PA_ERR_INVALID_ARG, "k and v shapes differ");
    const int64_t T = k->shape[0], H = k->shape[1], D = k->shape[2];
    if (kv_dtype != PA_KV_AUTO && kv_dtype != PA_KV_FP8_E4M3)
      return fail(PA_ERR_INVALID_ARG, "bad kv_dtype %d", kv_dtype);
    const bool fp8 = kv_dtype == PA_KV_FP8_E4M3;
    const int32_t cdt = fp8 ? PA_FP8_E4M3 : k->dtype;
    if (key_cache->dtype != cdt || value_cache->dtype != cdt)
      return fail(PA_ERR_INVALID_ARG, "cache dtype does not match kv_dtype");
    for (int i = 0; i < 4; ++i)
      if (key_cache->shape[i] != value_cache->shape[i])
        return fail(PA_ERR_INVALID_ARG, "key and value cache shapes differ");
    if (key_cache->shape[1] != H || key_cache->shape[3] != D)
      return fail(PA_ERR_INVALID_ARG, "cache [NB, Hkv, bs, D] does not match k [T, Hkv, D]");
    if (slot_mapping->dtype != PA_I64 || slot_mapping->shape[0] != T)
      return fail(PA_ERR_INVALID_ARG, "slot_mapping must be int64 [T]");
    if (D % 8) return fail(PA_ERR_UNSUPPORTED, "head_dim must be a multiple of 8");
    if (!is_contiguous(key_cache) || !is_contiguous(value_cache) || !is_contiguous(slot_mapping))
      return fail(PA_ERR_LAYOUT, "caches and slot_mapping must be contiguous");
    for (const pa_tensor* x : {k, v}) {
      if (T == 0) break;  // no rows: nothing is read
      if (x->strides[2] != 1 || (H > 1 && x->strides[1] != D))
        return fail(PA_ERR_LAYOUT, "k/v rows [Hkv, D] must be contiguous");
      if ((reinterpret_cast<uintptr_t>(x->data) % 16) || (x->strides[0] % 8))
        return fail(PA_ERR_LAYOUT, "k/v rows must be 16-byte aligned");
    }
    if ((reinterpret_cast<uintptr_t>(key_cache->data) % 16) ||
        (reinterpret_cast<uintptr_t>(value_cache->data) % 16))
      return fail(PA_ERR_LAYOUT, "caches must be 16-byte aligned");
    if (fp8 && !(std::isfinite(k_scale) && std::isfinite(v_scale) && k_scale > 0 && v_scale > 0))
      return fail(PA_ERR_INVALID_ARG, "fp8 scales must be finite and positive");
    if (key_cache->data == value_cache->data && numel(key_cache) > 0)
      return fail(PA_ERR_INVALID_ARG, "key and value caches alias");
    if (T > (int64_t(1) << 30) || H > 65535) return fail(PA_ERR_UNSUPPORTED, "too many tokens/heads");
    if (T == 0 || H == 0) return ok();
    if ((s = check_accessible(k, "k")) || (s = check_accessible(v, "v")) ||
        (s = check_accessible(key_cache, "key_cache")) ||
        (s = check_accessible(value_cache, "value_cache")) ||
        (s = check_accessible(slot_mapping, "slot_mapping")))
      return s;
  
    DeviceState* st;
    {
      std::lock_guard<std::mutex> lk(g_mu);
      if ((s = device_state(&st, nullptr))) return s;
    }
    pa::ReshapeArgs a;
    a.k = k->data;
    a.v = v->data;
    a.kc = key_cache->data;
    a.vc = value_cache->data;
    a.slots = static_cast<const int64_t*>(slot_mapping->data);
    a.err = st->err_word;
    a.k_stride_t = k->strides[0];
    a.k_stride_h = D;
    a.v_stride_t = v->strides[0];
    a.v_stride_h = D;
    a.T = static_cast<int>(T);
    a.H = static_cast<int>(H);
    a.D = static_cast<int>(D);
    a.bs = static_cast<int>(key_cache->shape[2]);
    a.NB = key_cache->shape[0];
    a.k_scale = k_scale;
    a.v_scale = v_scale;
    cudaError_t e = pa::reshape_launch(k->dtype, fp8, a, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "reshape_and_cache launch");
    g_launches += 1;
    return ok();
  });
}

}  // extern "C"

namespace {

// A validated decode or chunk call.
struct DecodeCall {
  const pa_tensor *out, *q, *kc, *vc, *bt, *sl;
  int64_t B, T, Hq, Hkv, D, NB, MB;
  int G, CG, NCG, Hv;
  int32_t bs, window;
  bool fp8;
  int ct, qt;
  float scale, k_scale, v_scale;
};

// Host validation shared by the decode entry points: q and out are
// [B, Hq, D] (chunked = false) or [B, T, Hq, D] (chunked = true).
pa_status check_decode(const pa_tensor* out, const pa_tensor* q, const pa_tensor* key_cache,
                       const pa_tensor* value_cache, const pa_tensor* block_tables,
                       const pa_tensor* seq_lens, int32_t num_kv_heads, float scale,
                       int32_t block_size, int32_t window, int32_t kv_dtype, float k_scale,
                       float v_scale, bool chunked, DecodeCall* c) {
  pa_status s;
  const int qd = chunked ? 4 : 3;
  if ((s = check_tensor(out, "out", qd)) || (s = check_tensor(q, "q", qd)) ||
      (s = check_tensor(key_cache, "key_cache", 4)) ||
      (s = check_tensor(value_cache, "value_cache", 4)) ||
      (s = check_tensor(block_tables, "block_tables", 2)) ||
      (s = check_tensor(seq_lens, "seq_lens", 1)))
    return s;
  if (q->dtype != PA_F16 && q->dtype != PA_BF16) return fail(PA_ERR_UNSUPPORTED, "q must be f16 or bf16");
  if (out->dtype != q->dtype) return fail(PA_ERR_INVALID_ARG, "out dtype must equal q dtype");
  for (int i = 0; i < qd; ++i)
    if (out->shape[i] != q->shape[i]) return fail(PA_ERR_INVALID_ARG, "out shape != q shape");
  const int64_t B = q->shape[0], T = chunked ? q->shape[1] : 1;
  const int64_t Hq = q->shape[qd - 2], D = q->shape[qd - 1];
  if (chunked && (T < 1 || T > kMaxChunk))
    return fail(PA_ERR_UNSUPPORTED, "num_queries %lld not in [1, %lld]", (long long)T,
                (long long)kMaxChunk);
  if (kv_dtype != PA_KV_AUTO && kv_dtype != PA_KV_FP8_E4M3)
    return fail(PA_ERR_INVALID_ARG, "bad kv_dtype %d", kv_dtype);
  const bool fp8 = kv_dtype == PA_KV_FP8_E4M3;
  const int32_t cdt = fp8 ? PA_FP8_E4M3 : q->dtype;
  if (key_cache->dtype != cdt || value_cache->dtype != cdt)
    return fail(PA_ERR_INVALID_ARG, "cache dtype does not match q dtype / kv_dtype");
  for (int i = 0; i < 4; ++i)
    if (key_cache->shape[i] != value_cache->shape[i])
      return fail(PA_ERR_INVALID_ARG, "key and value cache shapes differ");
  const int64_t NB = key_cache->shape[0], Hkv = key_cache->shape[1];
  if (num_kv_heads != Hkv) return fail(PA_ERR_INVALID_ARG, "num_kv_heads != key_cache.shape[1]");
  if (block_size != key_cache->shape[2]) return fail(PA_ERR_INVALID_ARG, "block_size != key_cache.shape[2]");
  if (key_cache->shape[3] != D) return fail(PA_ERR_INVALID_ARG, "cache head_dim != q head_dim");
  if ((s = check_heads(Hq, Hkv, D))) return s;
  if (fp8 && D == 64) return fail(PA_ERR_UNSUPPORTED, "fp8 caches need head_dim 128 or 256");
  if (block_size <= 0 || block_size % 16 || block_size > 1024)
    return fail(PA_ERR_UNSUPPORTED, "block_size must be a multiple of 16 in [16, 1024]");
  if (block_tables->dtype != PA_I32 || seq_lens->dtype != PA_I32)
    return fail(PA_ERR_INVALID_ARG, "block_tables and seq_lens must be int32");
  if (block_tables->shape[0] != B || seq_lens->shape[0] != B)
    return fail(PA_ERR_INVALID_ARG, "block_tables / seq_lens batch != q batch");
  const int64_t MB = block_tables->shape[1];
  if (B > kMaxBatch) return fail(PA_ERR_UNSUPPORTED, "batch %lld > %lld", (long long)B, (long long)kMaxBatch);
  if (!is_contiguous(out) || !is_contiguous(q) || !is_contiguous(key_cache) ||
      !is_contiguous(value_cache) || !is_contiguous(block_tables) || !is_contiguous(seq_lens))
    return fail(PA_ERR_LAYOUT, "decode needs contiguous tensors");
  for (const pa_tensor* x : {key_cache, value_cache, q, out})
    if (reinterpret_cast<uintptr_t>(x->data) % 16)
      return fail(PA_ERR_LAYOUT, "q, out and caches must be 16-byte aligned");
  if (!std::isfinite(scale)) return fail(PA_ERR_INVALID_ARG, "scale must be finite");
  if (fp8 && !(std::isfinite(k_scale) && std::isfinite(v_scale) && k_scale > 0 && v_scale > 0))
    return fail(PA_ERR_INVALID_ARG, "fp8 scales must be finite and positive");
  const int G = static_cast<int>(Hq / Hkv);
  int CG, NCG;
  chunk_columns(T, G, &CG, &NCG);
  const int64_t Hv = Hkv * NCG;
  // 32-bit index limits inside the kernels
  const double k2p31 = 2147483648.0;
  const double dNB = static_cast<double>(NB), dMB = static_cast<double>(MB);
  const double dB = static_cast<double>(B), dHv = static_cast<double>(Hv);
  if (dprod({dNB, double(Hkv), double(block_size)}) >= k2p31 ||
      dprod({dMB, double(block_size)}) >= k2p31 ||
      dprod({dB, dHv}) * (dprod({dMB, double(block_size)}) / 16 + 1) >= k2p31 ||
      dprod({dB, dMB}) >= k2p31 ||
      dprod({dB, double(T), double(Hq), double(D)}) >= 1099511627776.0)
    return fail(PA_ERR_UNSUPPORTED, "pool or tables exceed 32-bit indexing");
  for (const pa_tensor* x : {q, key_cache, value_cache, block_tables, seq_lens})
    if (overlaps(out, x)) return fail(PA_ERR_INVALID_ARG, "out overlaps an input");
  if (dprod({dB, dHv, double(CG)}) > pa::kMaxColumns)
    return fail(PA_ERR_UNSUPPORTED, "batch * num_q_heads * num_queries too large");
  if (B > 0 && MB == 0) return fail(PA_ERR_INVALID_ARG, "block_tables has no columns");
  if (B > 0 && NB == 0) return fail(PA_ERR_INVALID_ARG, "empty block pool");
  if (B > 0 && ((s = check_accessible(out, "out")) || (s = check_accessible(q, "q")) ||
                (s = check_accessible(key_cache, "key_cache")) ||
                (s = check_accessible(value_cache, "value_cache")) ||
                (s = check_accessible(block_tables, "block_tables")) ||
                (s = check_accessible(seq_lens, "seq_lens"))))
    return s;
  *c = DecodeCall{out, q, key_cache, value_cache, block_tables, seq_lens, B, T, Hq, Hkv, D, NB,
                  MB, G, CG, NCG, static_cast<int>(Hv), block_size, window > 0 ? window : 0,
                  fp8, fp8 ? pa::kE4M3 : (q->dtype == PA_BF16 ? pa::kBF16 : pa::kF16),
                  q->dtype, scale, k_scale, v_scale};
  return PA_OK;
}

pa_status plan_call(DeviceState* st, const DecodeCall& c, DecodePlan* plan, WsLayout* layout) {
  pa_status s = plan_decode(st, c.ct, c.qt, c.T > 1, c.B, c.CG, static_cast<int>(c.D), plan);
  if (s) return s;
  // No more worker warps than the step can fill at min_tiles each: its
  // tiles are at most B * Hv pairs times the 16-token tiles of the longest
  // read range the tables (or the window) allow, plus one for a window
  // start inside a tile. Small batches then launch fewer CTAs and need
  // less scratch; large ones keep the full grid.
  int64_t span = c.MB * c.bs;
  if (c.window > 0) span = std::min<int64_t>(span, int64_t(c.window) + c.T - 1);
  const int64_t tiles = c.B * c.Hv * ((span + 15) / 16 + 1);
  const int64_t warps = (tiles + plan->min_tiles - 1) / plan->min_tiles;
  const int64_t ctas = (warps + plan->var.warps - 1) / plan->var.warps;
  if (ctas < plan->grid) {
    plan->grid = static_cast<int>(std::max<int64_t>(ctas, 1));
    plan->workers = plan->grid * plan->var.warps;
  }
  *layout = ws_layout(c.B, c.Hv, c.CG, static_cast<int>(c.D), plan->workers);
  return PA_OK;
}

// Encodes the cache maps and launches the decode and merge kernels with the
// scratch at `ws`. `wsp` (if given) is marked dirty when the merge launch
// fails after the decode kernel ran, so that its pool counter is cleared
// before the next use.
pa_status run_decode(const DecodeCall& c, DeviceState* st, const DecodePlan& plan,
                     const WsLayout& layout, void* ws, Workspace* wsp, cudaStream_t cs) {
  pa_status s;
  const int elt = c.fp8 ? 1 : 2;
  const int D = static_cast<int>(c.D);
  CUtensorMap tk, tv;
  if ((s = make_cache_map(&tk, c.kc->data, c.NB * c.Hkv * c.bs, D, elt)) ||
      (s = make_cache_map(&tv, c.vc->data, c.NB * c.Hkv * c.bs, D, elt)))
    return s;

  const double log2e = 1.4426950408889634;
  pa::DecodeArgs a;
  a.q = c.q->data;
  a.block_tables = static_cast<const int32_t*>(c.bt->data);
  a.seq_lens = static_cast<const int32_t*>(c.sl->data);
  char* wsb = static_cast<char*>(ws);
  a.pool = reinterpret_cast<uint32_t*>(wsb + layout.pool);
  a.plan = reinterpret_cast<int32_t*>(wsb + layout.plan);
  a.part = reinterpret_cast<float*>(wsb + layout.part);
  a.err = st->err_word;
  a.B = static_cast<int>(c.B);
  a.Hq = static_cast<int>(c.Hq);
  a.Hkv = static_cast<int>(c.Hkv);
  a.G = c.G;
  a.D = D;
  a.bs = c.bs;
  a.MB = static_cast<int>(c.MB);
  a.NB = static_cast<int>(c.NB);
  a.window = c.window;
  a.T = static_cast<int>(c.T);
  a.NCG = c.NCG;
  a.CG = c.CG;
  a.Hv = c.Hv;
  // a window at least as long as the table covers acts as no window
  a.span = c.window > 0
               ? static_cast<int>(std::min<int64_t>(int64_t(c.window) + c.T - 1, c.MB * c.bs))
               : 0;
  a.score_scale = static_cast<float>(static_cast<double>(c.scale) * log2e *
                                     (c.fp8 ? static_cast<double>(c.k_scale) : 1.0));
  a.v_scale = c.fp8 ? c.v_scale : 1.f;
  a.min_tiles = plan.min_tiles;
  a.pool_permille = plan.pool_permille;
  a.piece_min = plan.piece;
  a.np_max = plan.workers * kPiecesPerWorker;

  const bool prof = g_prof_before && g_prof_after;
  cudaError_t e;
  if (prof && (e = cudaEventRecord(static_cast<cudaEvent_t>(g_prof_before), cs)) != cudaSuccess)
    return cuda_fail(e, "profile event");
  e = plan.fam.launch(D, plan.nt, tk, tv, a, plan.grid, plan.smem, cs, !prof);
  if (e != cudaSuccess) return cuda_fail(e, "decode kernel launch");
  if (prof && (e = cudaEventRecord(static_cast<cudaEvent_t>(g_prof_after), cs)) != cudaSuccess)
    return cuda_fail(e, "profile event");
  pa::MergeArgs m;
  m.out = c.out->data;
  m.part = a.part;
  m.plan = a.plan;
  m.pool = a.pool;
  m.NW = plan.workers;
  m.B = a.B;
  m.Hq = a.Hq;
  m.Hkv = a.Hkv;
  m.G = a.G;
  m.D = a.D;
  m.T = a.T;
  m.NCG = a.NCG;
  m.CG = a.CG;
  m.Hv = a.Hv;
  // three CTAs per SM, and no more than output columns (a wide column takes
  // one CTA, a narrow one a warp)
  const int64_t cols = static_cast<int64_t>(m.B) * m.Hv * m.CG;
  const int merge_grid =
      static_cast<int>(std::min<int64_t>(int64_t(st->num_sms) * 3, std::max<int64_t>(cols, 1)));
  e = pa::merge_launch(c.qt, m, merge_grid, cs, !prof);
  if (e != cudaSuccess) {
    if (wsp) {
      std::lock_guard<std::mutex> lk(g_mu);
      wsp->dirty = true;  // the decode kernel ran; its pool counter was not reset
    }
    return cuda_fail(e, "merge kernel launch");
  }
  g_launches += 2;
  return ok();
}

bool use_chunk_tc(const DecodeCall& c) {
  const int path = g_chunk_path.load();
  if (path == 1 || c.D != 128) return false;
  return path == 2 || c.T * c.G > kTcMinColumns;
}

// A chunk on the tensor-memory kernel: no workspace, one launch.
pa_status run_chunk_tc(const DecodeCall& c, cudaStream_t cs) {
  pa_status s;
  DeviceState* st;
  {
    std::lock_guard<std::mutex> lk(g_mu);
    if ((s = device_state(&st, nullptr))) return s;
    if (!st->chunk_tc_ready) {
      cudaError_t e = pa::chunk_tc_prepare();
      if (e != cudaSuccess) return cuda_fail(e, "chunk kernel setup");
      st->chunk_tc_ready = true;
    }
  }
  const int D = static_cast<int>(c.D);
  CUtensorMap tk, tv;
  const int elt = c.fp8 ? 1 : 2;
  if ((s = make_cache_map(&tk, c.kc->data, c.NB * c.Hkv * c.bs, D, elt)) ||
      (s = make_cache_map(&tv, c.vc->data, c.NB * c.Hkv * c.bs, D, elt)))
    return s;
  pa::ChunkArgs a;
  a.q = c.q->data;
  a.out = c.out->data;
  a.block_tables = static_cast<const int32_t*>(c.bt->data);
  a.seq_lens = static_cast<const int32_t*>(c.sl->data);
  a.err = st->err_word;
  a.B = static_cast<int>(c.B);
  a.T = static_cast<int>(c.T);
  a.Hq = static_cast<int>(c.Hq);
  a.Hkv = static_cast<int>(c.Hkv);
  a.G = c.G;
  a.bs = c.bs;
  a.MB = static_cast<int>(c.MB);
  a.NB = static_cast<int>(c.NB);
  a.window = c.window;
  const int unit = pa::chunk_tc_unit_rows();
  a.QT = static_cast<int>((c.T * c.G + unit - 1) / unit);
  a.score_scale = static_cast<float>(static_cast<double>(c.scale) * 1.4426950408889634 *
                                     (c.fp8 ? static_cast<double>(c.k_scale) : 1.0));
  a.v_scale = c.fp8 ? c.v_scale : 1.f;
  const bool prof = g_prof_before && g_prof_after;
  cudaError_t e;
  if (prof && (e = cudaEventRecord(static_cast<cudaEvent_t>(g_prof_before), cs)) != cudaSuccess)
    return cuda_fail(e, "profile event");
  e = pa::chunk_tc_launch(c.qt, c.fp8, tk, tv, a, cs, !prof);
  if (e != cudaSuccess) return cuda_fail(e, "chunk kernel launch");
  if (prof && (e = cudaEventRecord(static_cast<cudaEvent_t>(g_prof_after), cs)) != cudaSuccess)
    return cuda_fail(e, "profile event");
  g_launches += 1;
  return ok();
}

// Validation, planning and launch with the library's (or the caller's set)
// workspace.
pa_status decode_entry(const pa_tensor* out, const pa_tensor* q, const pa_tensor* key_cache,
                       const pa_tensor* value_cache, const pa_tensor* block_tables,
                       const pa_tensor* seq_lens, int32_t num_kv_heads, float scale,
                       int32_t block_size, int32_t window, int32_t kv_dtype, float k_scale,
                       float v_scale, pa_stream stream, bool chunked) {
  DecodeCall c;
  pa_status s = check_decode(out, q, key_cache, value_cache, block_tables, seq_lens,
                             num_kv_heads, scale, block_size, window, kv_dtype, k_scale, v_scale,
                             chunked, &c);
  if (s) return s;
  if (c.B == 0) return ok();
  cudaStream_t cs = static_cast<cudaStream_t>(stream);
  if (chunked && use_chunk_tc(c)) return run_chunk_tc(c, cs);
  DeviceState* st;
  DecodePlan plan;
  WsLayout layout;
  void* ws = nullptr;
  Workspace* wsp = nullptr;
  {
    std::lock_guard<std::mutex> lk(g_mu);
    if ((s = device_state(&st, nullptr)) || (s = plan_call(st, c, &plan, &layout)) ||
        (s = get_workspace(st, cs, layout, &ws, &wsp)))
      return s;
  }
  return run_decode(c, st, plan, layout, ws, wsp, cs);
}

}  // namespace

extern "C" {

pa_status pa_decode(const pa_tensor* out, const pa_tensor* q, const pa_tensor* key_cache,
                    const pa_tensor* value_cache, const pa_tensor* block_tables,
                    const pa_tensor* seq_lens, int32_t num_kv_heads, float scale,
                    int32_t block_size, int32_t window, int32_t kv_dtype, float k_scale,
                    float v_scale, pa_stream stream) {
  return pa::abi_guard([&]() -> pa_status {
    return decode_entry(out, q, key_cache, value_cache, block_tables, seq_lens, num_kv_heads, scale,
                        block_size, window, kv_dtype, k_scale, v_scale, stream, false);
  });
}

pa_status pa_prefill_chunk(const pa_tensor* out, const pa_tensor* q, const pa_tensor* key_cache,
                           const pa_tensor* value_cache, const pa_tensor* block_tables,
                           const pa_tensor* seq_lens, int32_t num_kv_heads, float scale,
                           int32_t block_size, int32_t window, int32_t kv_dtype, float k_scale,
                           float v_scale, pa_stream stream) {
  return pa::abi_guard([&]() -> pa_status {
    return decode_entry(out, q, key_cache, value_cache, block_tables, seq_lens, num_kv_heads, scale,
                        block_size, window, kv_dtype, k_scale, v_scale, stream, true);
  });
}

}  // extern "C"

// pa_decode with the scratch in a caller-given device buffer of `capacity`
// bytes instead of a library workspace; used by the allocation-free entry
// point (decode_noalloc.cu). Allocates nothing.
namespace pa {
pa_status decode_in_buffer(const pa_tensor* out, const pa_tensor* q, const pa_tensor* key_cache,
                           const pa_tensor* value_cache, const pa_tensor* block_tables,
                           const pa_tensor* seq_lens, int32_t num_kv_heads, float scale,
                           int32_t block_size, int32_t window, int32_t kv_dtype, float k_scale,
                           float v_scale, pa_stream stream, void* buffer, size_t capacity) {
  DecodeCall c;
  pa_status s = check_decode(out, q, key_cache, value_cache, block_tables, seq_lens,
                             num_kv_heads, scale, block_size, window, kv_dtype, k_scale, v_scale,
                             false, &c);
  if (s) return s;
  if (c.B == 0) return ok();
  cudaStream_t cs = static_cast<cudaStream_t>(stream);
  DeviceState* st;
  DecodePlan plan;
  WsLayout layout;
  {
    std::lock_guard<std::mutex> lk(g_mu);
    if ((s = device_state(&st, nullptr)) || (s = plan_call(st, c, &plan, &layout))) return s;
  }
  if (layout.total > capacity)
    return fail(PA_ERR_WORKSPACE,
                "this step needs %zu bytes of scratch; the built-in buffer holds %zu (use "
                "pa_decode with its own workspace for larger batches or head counts)",
                layout.total, capacity);
  // The piece counter must start at zero; the buffer keeps whatever the
  // previous call left there.
  cudaError_t e = cudaMemsetAsync(static_cast<char*>(buffer) + layout.pool, 0,
                                  layout.plan - layout.pool, cs);
  if (e != cudaSuccess) return cuda_fail(e, "clearing the scratch counter");
  return run_decode(c, st, plan, layout, buffer, nullptr, cs);
}
}  // namespace pa

namespace pa {
pa_status set_error(pa_status code, const char* msg) { return fail(code, "%s", msg); }
pa_status set_cuda_error(cudaError_t e, const char* what) { return cuda_fail(e, what); }
}  // namespace pa
