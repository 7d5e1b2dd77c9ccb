// Allocation-free decode entry point.
//
// Some callers cannot allocate device memory at the time they decode: code
// running inside a memory pool or arena that owns all of the GPU's memory,
// runtimes whose allocator is locked or must not be re-entered from this
// call, and hosts that forbid cudaMalloc after start-up so that memory use
// stays fixed. For them pa_decode_noalloc keeps its scratch in one fixed
// array in this file, compiled into the library. The array lives in the
// module's device memory on every GPU that loads the library, for as long as
// the process runs, and every call shares it.
#include <cuda_runtime.h>

#include <atomic>

#include "pa.h"
#include "pa_internal.h"

namespace {

constexpr size_t kNoallocScratchBytes = size_t(32) << 20;  // 32 MiB
constexpr int kMaxDevices = 64;  // device ordinals this entry point serves

// The scratch itself. Host code must not pass `g_noalloc_scratch` to a kernel:
// on the host that name is only a stand-in, not a device address. The device
// address comes from cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoallocScratchBytes];

// Device address of the array, per device ordinal (null until first looked
// up). A fixed table of atomics: the lookup takes no lock and allocates no
// host memory, so nothing here can throw. Two threads that race on the first
// call of a device both store the same address.
std::atomic<void*> g_noalloc_addr[kMaxDevices];

// Resolves the array's device address once per device, with that device
// current (the caller's current device).
pa_status noalloc_scratch(void** ptr) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return pa::set_cuda_error(e, "cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices)
    return pa::set_error(PA_ERR_UNSUPPORTED,
                         "pa_decode_noalloc serves device ordinals below 64 only");
  void* p = g_noalloc_addr[dev].load(std::memory_order_acquire);
  if (p == nullptr) {
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return pa::set_cuda_error(e, "cudaGetSymbolAddress(scratch array)");
    if (p == nullptr)
      return pa::set_error(PA_ERR_CUDA, "cudaGetSymbolAddress(scratch array) gave no address");
    g_noalloc_addr[dev].store(p, std::memory_order_release);
  }
  *ptr = p;
  return PA_OK;
}

}  // namespace

extern "C" pa_status pa_decode_noalloc(const pa_tensor* out, const pa_tensor* q,
                                       const pa_tensor* key_cache, const pa_tensor* value_cache,
                                       const pa_tensor* block_tables, const pa_tensor* seq_lens,
                                       int32_t num_kv_heads, float scale, int32_t block_size,
                                       int32_t window, int32_t kv_dtype, float k_scale,
                                       float v_scale, pa_stream stream) {
  return pa::abi_guard([&]() -> pa_status {
    void* scratch = nullptr;
    const pa_status s = noalloc_scratch(&scratch);
    if (s != PA_OK) return s;
    return pa::decode_in_buffer(out, q, key_cache, value_cache, block_tables, seq_lens,
                                num_kv_heads, scale, block_size, window, kv_dtype, k_scale,
                                v_scale, stream, scratch, kNoallocScratchBytes);
  });
}
