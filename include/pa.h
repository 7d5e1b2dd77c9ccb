/*
 * pa.h — C ABI of the GB300 paged-attention decode library (libpa.so).
 *
 * One decode step of PagedAttention: every sequence contributes one query
 * token per q head, which attends over that sequence's K/V rows stored in
 * fixed-size physical blocks of a shared pool and reached through a per-
 * sequence block table. Sources (page title and section):
 *   - "vLLM 0.5 深度解析" §2.1: blocks of block_size tokens, a block table per
 *     request mapping logical to physical blocks, ceil(n / block_size) blocks
 *     for n tokens; §2.2: scale = head_dim ** -0.5, the forward signature
 *     (query, key_cache, value_cache, block_table, seq_lens); §2.3: per
 *     physical block, K loaded, scaled dot product, softmax max/sum state,
 *     V-weighted sum.
 *   - "vLLM 0.7.2深度解析" §2.1: physical blocks shared by several sequences,
 *     ref-counted deferred reclamation; §2.2: GQA head groups and the FP8 e4m3
 *     KV cache; §2.3: masking of positions outside a sliding window and never
 *     loading blocks that lie wholly outside it; §5.3: a hard cap on pool
 *     blocks, requests beyond it rejected.
 *
 * Conventions for every entry point:
 *   - Returns PA_OK (0) or a negative pa_status; a message for the calling
 *     thread is available from pa_last_error(). No C++ exception crosses the
 *     ABI. Host-detectable errors are reported before anything is launched.
 *   - Tensors are described by pa_tensor: data pointer, dtype, rank, shape and
 *     strides in elements. A tensor lives in memory of the current CUDA device,
 *     or in pinned host memory mapped into the device's address space at the
 *     same address (cudaHostAlloc / cudaHostRegister with mapping, as every
 *     pinned allocation is under unified addressing); the kernels then read or
 *     write it in place over the CPU-GPU link, which on GB300 saves the copy
 *     engine's per-copy latency for a step's small inputs and outputs. Any
 *     other pointer (pageable host memory, another device) is rejected with
 *     PA_ERR_INVALID_ARG before launch. The caller owns every tensor; the
 *     library keeps no pointer to them after the call returns.
 *   - Launches are asynchronous on the given stream (a cudaStream_t; NULL is
 *     the legacy default stream). No entry point synchronises the stream
 *     except pa_check_device_error().
 *   - Device-side data errors (a block id outside the pool, a seq_len beyond
 *     max_blocks_per_seq * block_size, a slot beyond the pool) never cause an
 *     out-of-bounds access: the kernel substitutes a safe value, and records
 *     a bit in a device error word that pa_check_device_error() returns.
 */
#ifndef PA_H
#define PA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef int32_t pa_status;

enum {
  PA_OK = 0,
  PA_ERR_INVALID_ARG = -1,   /* null pointer, bad value, aliasing, mismatched shapes */
  PA_ERR_UNSUPPORTED = -2,   /* a shape or dtype this build has no kernel for */
  PA_ERR_LAYOUT = -3,        /* a tensor is not contiguous or not aligned as required
                                (a tensor with no elements counts as contiguous) */
  PA_ERR_CUDA = -4,          /* a CUDA runtime call or launch failed */
  PA_ERR_OUT_OF_BLOCKS = -5, /* allocator: the pool cannot cover the request */
  PA_ERR_WORKSPACE = -6,     /* decode workspace missing or too small */
  PA_ERR_NOT_FOUND = -7,     /* allocator: unknown sequence or block id */
  PA_ERR_HOST_MEMORY = -8    /* host memory exhausted; no C++ exception crosses this
                                ABI. An allocator that returns it has undefined
                                state: destroy it */
};

/* Element types. */
enum { PA_F16 = 0, PA_BF16 = 1, PA_FP8_E4M3 = 2, PA_I32 = 3, PA_I64 = 4 };

/* kv_dtype argument: cache elements have the dtype of k/q (PA_KV_AUTO), or are
 * OCP e4m3 codes (uint8) with per-tensor scales (PA_KV_FP8_E4M3). */
enum { PA_KV_AUTO = 0, PA_KV_FP8_E4M3 = 2 };

/* Bits of the device error word. */
enum {
  PA_DEVERR_BLOCK_ID = 1,  /* a block table entry outside [0, num_blocks) */
  PA_DEVERR_SEQ_LEN = 2,   /* seq_len < 0 or > max_blocks_per_seq * block_size */
  PA_DEVERR_SLOT = 4,      /* a slot_mapping entry >= num_blocks * block_size */
  PA_DEVERR_TIMEOUT = 8    /* a pipeline wait gave up (should never happen, except
                              in pa_selftest_bounded_wait) */
};

#define PA_MAX_DIMS 6

typedef struct pa_tensor {
  void* data;
  int32_t dtype;                  /* PA_F16 ... PA_I64 */
  int32_t ndim;                   /* 1 .. PA_MAX_DIMS */
  int64_t shape[PA_MAX_DIMS];
  int64_t strides[PA_MAX_DIMS];   /* in elements */
} pa_tensor;

typedef void* pa_stream; /* cudaStream_t */

/* ------------------------------------------------------------ write path */

/*
 * pa_reshape_and_cache — scatter new K/V rows into their cache slots.
 * For every t < T with slot = slot_mapping[t] >= 0 and every head h:
 *   key_cache[slot / bs, h, slot % bs, :]   = enc(k[t, h, :])
 *   value_cache[slot / bs, h, slot % bs, :] = enc(v[t, h, :])
 * enc is the identity (bit copy) for PA_KV_AUTO; for PA_KV_FP8_E4M3 it is
 * e4m3(round-to-nearest-even, saturating)(float(x) / scale) with the division
 * in IEEE fp32, k_scale for K and v_scale for V. Slots < 0 are skipped; slots
 * beyond the pool are skipped and flagged (PA_DEVERR_SLOT). Duplicate
 * non-negative slots are a caller error (the surviving row is unspecified).
 *
 *   k, v          [T, Hkv, D] f16/bf16; dims 1 and 2 contiguous, dim 0 any
 *                 stride; rows 16-byte aligned.
 *   key_cache,    [NB, Hkv, bs, D] contiguous; dtype of k (PA_KV_AUTO) or
 *   value_cache   PA_FP8_E4M3 (uint8 codes).
 *   slot_mapping  [T] int64, slot = physical_block * bs + offset.
 *   k_scale, v_scale  used only for FP8 (finite, > 0).
 * D must be a multiple of 8 (16 for FP8).
 */
pa_status pa_reshape_and_cache(const pa_tensor* k, const pa_tensor* v,
                               const pa_tensor* key_cache, const pa_tensor* value_cache,
                               const pa_tensor* slot_mapping, int32_t kv_dtype,
                               float k_scale, float v_scale, pa_stream stream);

/* ---------------------------------------------------------------- decode */

/*
 * pa_decode — one decode step of paged attention.
 * For every sequence b and q head h, with G = Hq / Hkv, kvh = h / G,
 * L = seq_lens[b], start = (window > 0 && L > window) ? L - window : 0:
 *   out[b, h, :] = sum_{j in [start, L)} softmax_j(scale * q[b,h,:] . K_j) V_j
 * where K_j, V_j are the rows at block_tables[b][j / bs], offset j % bs, KV
 * head kvh (for FP8: decode(code) * k_scale, resp. * v_scale). An empty range
 * (L == 0) gives a row of zeros. Blocks wholly outside [start, L) are never
 * read; table entries past ceil(L / bs) are never read.
 *
 *   out           [B, Hq, D] contiguous, dtype of q; must not overlap inputs.
 *   q             [B, Hq, D] contiguous, f16 or bf16.
 *   key_cache,    [NB, Hkv, bs, D] contiguous, base 16-byte aligned; dtype of
 *   value_cache   q (PA_KV_AUTO) or PA_FP8_E4M3.
 *   block_tables  [B, MB] int32 contiguous.
 *   seq_lens      [B] int32.
 *   num_kv_heads  Hkv (== key_cache.shape[1]); Hq % Hkv == 0, G <= 16.
 *   block_size    bs (== key_cache.shape[2]), a multiple of 16, <= 1024.
 *   window        <= 0: no window.
 * Supported D: 64, 128, 256 for 16-bit caches; 128, 256 for FP8. B <= 4096.
 *
 * Most tiles are split evenly over the worker warps of a persistent grid; the
 * rest are handed out in small pieces to whichever warps finish first, so the
 * summation order, and with it the last bits of the output, can differ from
 * run to run (pa_set_decode_tuning can turn the dynamic share off).
 *
 * Ordering: the kernels use programmatic dependent launch. The decode kernel
 * reads q, block_tables and seq_lens (and plans the step) before it waits for
 * the previous kernel of the stream, and reads the caches only after. A
 * predecessor that lets its dependents start early (as pa_reshape_and_cache
 * does) must therefore have written q, block_tables and seq_lens before doing
 * so; ordinary kernels and copies are waited for in full.
 *
 * Workspace: the step writes per-segment partial results (running max, sum
 * and unnormalised output), its plan and three counter words (zero again
 * when the step ends) to a device workspace of pa_decode_workspace_size()
 * bytes. It is the buffer
 * given to pa_set_workspace() for the current device, or else a buffer the
 * library allocates (and zeroes) once per (device, stream) outside stream
 * capture and keeps. Calls that overlap on the GPU must not share a
 * workspace.
 */
pa_status pa_decode(const pa_tensor* out, const pa_tensor* q, const pa_tensor* key_cache,
                    const pa_tensor* value_cache, const pa_tensor* block_tables,
                    const pa_tensor* seq_lens, int32_t num_kv_heads, float scale,
                    int32_t block_size, int32_t window, int32_t kv_dtype, float k_scale,
                    float v_scale, pa_stream stream);

/*
 * pa_decode_noalloc — pa_decode for callers that cannot allocate device
 * memory when they decode: code that runs inside a memory pool or arena
 * owning all of the GPU's memory, runtimes whose allocator must not be
 * re-entered from this call, and services that forbid cudaMalloc after
 * start-up so that their memory use stays fixed. (The paged-attention pages
 * describe no such variant; it is a property of this library.)
 *
 * Arguments, results and errors are those of pa_decode. Instead of a
 * workspace, the call keeps its scratch in one 32 MiB array compiled into the
 * library; every GPU that loads the library holds that array until the
 * process exits. The call allocates and frees nothing (no cudaMalloc or
 * cudaFree, directly or through another library). The scratch a step needs
 * is about 512 + 4 * batch bytes of counters and plan, plus
 *   4 * (G * head_dim + 2 * G rounded up to 4) * (2 * batch * num_kv_heads + 5 * W)
 * bytes of partial results, where W is the number of worker warps of the
 * decode kernel: 2 * (SM count) * 4, or * 8 for e4m3 caches with head_dim 128
 * (W = 1216 or 2432 on a 152-SM GB300), but no more than a step can fill:
 * about batch * num_kv_heads * (block_tables' width * block_size / 16 + 1),
 * rounded up to whole CTAs (the window's span instead of the tables' when it
 * is shorter). The per-warp term dominates batches of moderate size: a batch
 * of 64 with 8 KV heads, G = 4 and head_dim 128 needs about 14.8 MB; a batch
 * of 256 of that shape with an e4m3 cache needs about 33.8 MB; four
 * sequences of at most 208 positions with 2 KV heads and head_dim 64 need
 * about 0.6 MB. A step beyond 32 MiB is rejected with PA_ERR_WORKSPACE and a
 * message giving the bytes needed.
 *
 * The first call on a device looks up that device's address of the array
 * (cudaGetSymbolAddress, with that device current); make that first call
 * before any stream capture. All calls share the one array and find the last
 * call's contents in it; each call clears, on its stream, the counter that
 * must start at zero. Calls that overlap on the GPU (on different streams, or
 * different host threads, of one device) race on the array and must not be
 * issued.
 */
pa_status pa_decode_noalloc(const pa_tensor* out, const pa_tensor* q,
                            const pa_tensor* key_cache, const pa_tensor* value_cache,
                            const pa_tensor* block_tables, const pa_tensor* seq_lens,
                            int32_t num_kv_heads, float scale, int32_t block_size,
                            int32_t window, int32_t kv_dtype, float k_scale, float v_scale,
                            pa_stream stream);

/* Workspace bytes pa_decode needs on the current device for a batch of
 * `batch` sequences with these head counts and head_dim. */
pa_status pa_decode_workspace_size(int64_t batch, int32_t num_q_heads, int32_t num_kv_heads,
                                   int32_t head_dim, size_t* bytes);

/*
 * pa_prefill_chunk — attention of a chunk of T new query tokens per sequence
 * over the paged cache, causal within the chunk: the chunked-prefill step
 * that "vLLM 0.5 深度解析" §5.2 switches on in its batching configuration
 * (the pages give only the switch; the computation below is the plain
 * reading), and equally the verification step of T drafted tokens.
 * The chunk's own K/V rows are written to the cache first (pa_reshape_and_cache
 * with B * T rows); seq_lens[b] counts them. Query t of sequence b sits at
 * position p = seq_lens[b] - T + t and, with
 * start = (window > 0 && p + 1 > window) ? p + 1 - window : 0,
 *   out[b, t, h, :] = sum_{j in [start, p]} softmax_j(scale * q[b,t,h,:] . K_j) V_j
 * with K_j, V_j as in pa_decode. A query with p < 0 (seq_lens[b] < T) gives a
 * row of zeros. With T = 1 the result equals pa_decode's.
 *
 *   out, q        [B, T, Hq, D] contiguous (q f16 or bf16, out the same),
 *                 1 <= T <= 4096; every other argument as for pa_decode.
 * The persistent kernel processes the (query, head) pairs of one KV head 16
 * at a time, so it reads each attended K/V byte ceil(T * G / 16) times (from
 * L2 where they are close together); for T * G <= 16 it reads it once. The
 * tensor-memory kernel (head_dim 128, T * G > 32 by default) reads it
 * ceil(T * G / 256) times. Workspace:
 * pa_prefill_chunk_workspace_size() bytes, from the same source as
 * pa_decode's. Errors as for pa_decode, plus PA_ERR_UNSUPPORTED for T out of
 * range or B * Hkv * ceil(T * G / 16) * 16 > 2^19.
 */
pa_status pa_prefill_chunk(const pa_tensor* out, const pa_tensor* q, const pa_tensor* key_cache,
                           const pa_tensor* value_cache, const pa_tensor* block_tables,
                           const pa_tensor* seq_lens, int32_t num_kv_heads, float scale,
                           int32_t block_size, int32_t window, int32_t kv_dtype, float k_scale,
                           float v_scale, pa_stream stream);

/* Kernel choice for pa_prefill_chunk, process-wide: 0 (default) picks per
 * call; 1 always uses the persistent split-KV kernel (16 (query, head)
 * columns per pass over K/V, any head dim); 2 uses the tensor-memory kernel
 * wherever it applies (head_dim 128; 16-bit or e4m3 caches),
 * which tiles 128 (query, head) rows against 128-token K/V tiles on the
 * tcgen05 tensor cores and reads each K/V tile once per 256 rows. The
 * default takes the tensor-memory kernel for chunks of more than 32 (query,
 * head) columns per KV head. */
pa_status pa_set_prefill_path(int32_t path);

/* Workspace bytes pa_prefill_chunk needs on the current device (the
 * tensor-memory kernel needs none). */
pa_status pa_prefill_chunk_workspace_size(int64_t batch, int32_t num_queries,
                                          int32_t num_q_heads, int32_t num_kv_heads,
                                          int32_t head_dim, size_t* bytes);

/* Use caller-owned device memory [ptr, ptr + bytes) as the decode workspace on
 * the current device (ptr 256-byte aligned). The call zeroes the buffer and
 * synchronises the device; each step leaves its piece counter at zero. ptr == NULL returns to the library-managed
 * workspace. The caller keeps the memory alive while decode steps that use it
 * are in flight, and does not write to it between calls. */
pa_status pa_set_workspace(void* ptr, size_t bytes);

/* Test and tuning knobs, process-wide for later pa_decode calls; 0 keeps the
 * default of each:
 *   max_ctas       caps the persistent decode grid (default: 2 CTAs per SM);
 *   min_tiles      least number of 16-token tiles per warp's static range,
 *                  which also caps the grid at the warps a step can fill
 *                  (default 1);
 *   pool_permille  share of the tiles handed out dynamically in small pieces
 *                  after the static ranges (default 100; the pool only
 *                  covers the trailing run of sequences no longer than 4x the
 *                  mean length); negative turns the pool off, which makes
 *                  results bit-reproducible;
 *   piece_tiles    least tiles per pool piece (default 4; 8 for single-query
 *                  decode on e4m3 caches). */
pa_status pa_set_decode_tuning(int32_t max_ctas, int32_t min_tiles, int32_t pool_permille,
                               int32_t piece_tiles);

/* Profiling hook: when both are non-NULL, the next pa_decode calls on this
 * thread record the CUDA events (cudaEvent_t) immediately before and after the
 * main decode kernel on the call's stream. NULL, NULL turns it off. */
pa_status pa_profile_events(void* ev_before, void* ev_after);

/* Reads and clears the device error word of the current device (PA_DEVERR_*
 * bits); synchronises `stream`. */
pa_status pa_check_device_error(int32_t* bits, pa_stream stream);

/* Self-test of the kernels' bounded waits. Every wait in this library's
 * kernels (for a copy to land, for a product to complete, for another CTA's
 * flag) gives up after a limit of device wall time, sets PA_DEVERR_TIMEOUT
 * and lets the kernel return, so that a wait that cannot be satisfied ends
 * with an error the host reads instead of a hung context. This call launches
 * one CTA on `stream` whose two waits can never be satisfied, through the
 * same bounded-wait code: an mbarrier phase that nothing completes, then a
 * device word that nothing writes. Each gives up after `limit_us`
 * microseconds (1 .. 1,000,000), the kernel sets PA_DEVERR_TIMEOUT and exits
 * normally. `elapsed_ns` (NULL, or two uint64_t in memory the device can
 * write, 8-byte aligned) receives each wait's duration in nanoseconds of the
 * device's global timer. Asynchronous like every launch: read the bit with
 * pa_check_device_error(), which also clears it.
 * Errors: PA_ERR_INVALID_ARG (limit out of range, elapsed_ns unaligned or not
 * accessible from the current device), PA_ERR_CUDA (launch failure). */
pa_status pa_selftest_bounded_wait(uint32_t limit_us, uint64_t* elapsed_ns, pa_stream stream);

/* Number of kernels this library has launched in this process. */
uint64_t pa_launch_count(void);

/* Message for the last error on the calling thread ("" if none). */
const char* pa_last_error(void);

/* Library version, major * 10000 + minor * 100 + patch. */
int32_t pa_version(void);

/* --------------------------------------------------- host block allocator */

/*
 * A fixed pool of num_blocks physical blocks of block_size tokens, used to
 * build block tables ("vLLM 0.5 深度解析" §2.1; "vLLM 0.7.2深度解析" §2.1, §5.3).
 *   - The free list starts as 0..NB-1 shuffled by Fisher-Yates driven by
 *     SplitMix64(seed); allocation pops from its end.
 *   - A sequence of n tokens holds ceil(n / block_size) blocks.
 *   - fork() shares every block of a sequence (reference count + 1 each).
 *   - append() grows a sequence; if its last block is partial and shared it is
 *     first copied (copy-on-write): *cow_src / *cow_dst name the blocks whose
 *     cached rows the caller must copy (-1 / -1 when no copy is needed).
 *   - free() drops one reference per block; blocks reaching zero wait in a
 *     pending list until reclaim() returns them to the free list (deferred
 *     reclamation: call it once the GPU work reading them has finished).
 *   - Every call is all-or-nothing: PA_ERR_OUT_OF_BLOCKS leaves the pool as it
 *     was (a hard cap: requests beyond it are rejected, not queued).
 *   - trim_window() releases blocks a sliding window has left behind.
 * Handles are not thread-safe; use one per thread or lock around calls.
 */
typedef struct pa_alloc pa_alloc;

pa_status pa_alloc_create(int32_t num_blocks, int32_t block_size, uint64_t seed, pa_alloc** out);
void pa_alloc_destroy(pa_alloc* a);
pa_status pa_alloc_add(pa_alloc* a, int64_t n_tokens, int32_t* seq_out);
pa_status pa_alloc_fork(pa_alloc* a, int32_t src_seq, int32_t* seq_out);
/* Prefix caching ("vLLM 0.7.2深度解析" §2.1 and §5.2; "vLLM 0.5 深度解析"
 * §4.4): a new sequence for n_tokens token ids that reuses cached full blocks
 * for its longest cached prefix. Full block i is keyed by
 * FNV-1a-64(key_{i-1} as 8 little-endian bytes || its token ids as 4
 * little-endian bytes each), key_{-1} = 0, and a hit also needs equal token
 * ids. Reused blocks gain a reference (one waiting for reclaim() is taken back);
 * the rest are allocated as by add(), and new full blocks are registered.
 * *n_cached (may be NULL) receives the number of tokens covered by reused
 * blocks: their K/V are already cached and need not be written again.
 * reclaim() drops the cache entries of the blocks it frees. */
pa_status pa_alloc_add_cached(pa_alloc* a, const int32_t* tokens, int64_t n_tokens,
                              int32_t* seq_out, int64_t* n_cached);
pa_status pa_alloc_append(pa_alloc* a, int32_t seq, int64_t n_tokens, int32_t* cow_src,
                          int32_t* cow_dst);
pa_status pa_alloc_free(pa_alloc* a, int32_t seq);
/* Releases the blocks of `seq` that lie wholly before its sliding window
 * [max(0, len - window), len) ("vLLM 0.7.2深度解析" §2.3: blocks known to be
 * outside the window need not stay allocated). Each drops one reference
 * (reaching zero, it waits for reclaim()) and its table entry becomes -1,
 * which a decode with that window never reads. fork() copies -1 entries and
 * free() skips them. window <= 0 releases nothing. *n_released (may be NULL)
 * receives the count. */
pa_status pa_alloc_trim_window(pa_alloc* a, int32_t seq, int32_t window, int32_t* n_released);
/* Returns the number of blocks moved from pending to free. */
int32_t pa_alloc_reclaim(pa_alloc* a);
/* Copies the sequence's block ids (logical order) into out[0 .. capacity);
 * *n_out receives the count; PA_ERR_INVALID_ARG if capacity is too small. */
pa_status pa_alloc_block_table(const pa_alloc* a, int32_t seq, int32_t* out, int32_t capacity,
                               int32_t* n_out);
pa_status pa_alloc_seq_len(const pa_alloc* a, int32_t seq, int64_t* len_out);
/* Writes a [n, max_blocks] int32 table matrix (-1 padded) and int32 lengths
 * for the listed sequences, the layout pa_decode reads. */
pa_status pa_alloc_fill_tables(const pa_alloc* a, const int32_t* seqs, int32_t n,
                               int32_t* tables, int32_t max_blocks, int32_t* lens_out);
int32_t pa_alloc_refcount(const pa_alloc* a, int32_t block); /* -1 for a bad id */
int32_t pa_alloc_num_free(const pa_alloc* a);
int32_t pa_alloc_num_pending(const pa_alloc* a);

#ifdef __cplusplus
}
#endif
#endif /* PA_H */
