/*
 * Plain fp64 CPU oracle for paged decode attention and its KV write path.
 *
 * TEST INFRASTRUCTURE ONLY. Only the tests, the smoke check and the CPU-baseline
 * leg of the benchmark may load this library. It shares no code, header, table
 * or helper with the CUDA library it judges.
 *
 * What it computes follows the pages on PagedAttention:
 *   - "vLLM 0.5 深度解析" §2.1 (block table: logical block i of a request maps
 *     to a physical block id; a request of n tokens holds ceil(n / block_size)
 *     blocks), §2.2 (scale = head_dim ** -0.5; the query attends over the cache
 *     reached through the block table), §2.3 (per physical block: load K, scaled
 *     dot product, softmax max/sum state, then the V-weighted sum).
 *   - "vLLM 0.7.2深度解析" §2.1 (several sequences may point at one physical
 *     block), §2.2 (GQA: several query heads share one KV head; FP8 e4m3 KV
 *     cache), §2.3 (positions outside the sliding window are masked).
 * The result is the plain definition softmax(scale * q K^T) V over the
 * sequence's attended positions, in fp64.
 */
#ifndef PA_ORACLE_H
#define PA_ORACLE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum { ORC_F16 = 0, ORC_BF16 = 1, ORC_E4M3 = 2 };
enum { ORC_OK = 0, ORC_EINVAL = -1, ORC_ERANGE = -2, ORC_ENOMEM = -3 };

/* Scalar codecs, written from the IEEE 754 binary16 definition, the bfloat16
 * definition (upper half of binary32) and the OCP 8-bit floating point E4M3
 * definition (bias 7, no infinities, S.1111.111 is NaN, max finite 448). */
double orc_f16_to_f64(uint16_t h);
double orc_bf16_to_f64(uint16_t h);
double orc_e4m3_to_f64(uint8_t c);
/* Round to nearest, ties to even; finite values beyond +-448 and infinities
 * saturate to +-448; NaN gives 0x7F; the sign of zero is kept. */
uint8_t orc_e4m3_from_f32(float x);

/* Array forms of the codecs (n elements). */
void orc_decode16_array(const uint16_t* src, int dtype, double* dst, int64_t n);
void orc_e4m3_decode_array(const uint8_t* src, double* dst, int64_t n);
void orc_e4m3_encode_array(const float* src, uint8_t* dst, int64_t n);

/*
 * Write path: for every token t with slot_mapping[t] >= 0,
 *   cache[slot / block_size, h, slot % block_size, :] = src[t, h, :]
 * for both K and V. Caches are [num_blocks, num_heads, block_size, head_dim].
 * src is 16-bit (src_dtype ORC_F16 / ORC_BF16). With cache_dtype == src_dtype
 * the bits are copied; with ORC_E4M3 each element is encoded from
 * float(x) / scale, the division done in fp32.
 * Returns ORC_ERANGE if a slot lies beyond the pool.
 */
int orc_reshape_and_cache(const uint16_t* k, const uint16_t* v, int64_t num_tokens,
                          int64_t num_heads, int64_t head_dim, int src_dtype,
                          void* key_cache, void* value_cache, int64_t num_blocks,
                          int64_t block_size, int cache_dtype, const int64_t* slot_mapping,
                          float k_scale, float v_scale, int threads);

/*
 * Decode: out[b, h, :] (fp64) for each requested (b, h); pairs holds n_pairs
 * distinct (b, h) couples (computed on parallel threads), or is NULL for all
 * B * Hq of them. q is [B, Hq, D] 16-bit,
 * block_tables is [B, max_blocks] int32, seq_lens [B] int32. q head h reads KV
 * head h / (Hq / Hkv). The attended positions are [start, L) with
 * start = max(0, L - window) when window > 0, else 0. For ORC_E4M3 caches the
 * element value is decode(code) * scale (k_scale for K, v_scale for V).
 * An empty range gives zeros. Returns ORC_ERANGE on a block id outside
 * [0, num_blocks) or a sequence longer than max_blocks * block_size.
 */
int orc_decode(double* out, const uint16_t* q, int q_dtype, const void* key_cache,
               const void* value_cache, int cache_dtype, const int32_t* block_tables,
               const int32_t* seq_lens, int64_t batch, int64_t num_q_heads,
               int64_t num_kv_heads, int64_t head_dim, int64_t num_blocks,
               int64_t block_size, int64_t max_blocks, double scale, int64_t window,
               double k_scale, double v_scale, const int32_t* pairs, int64_t n_pairs,
               int threads);

/*
 * Multi-token decode (chunked queries with a causal mask), the attention of
 * the chunked prefill that "vLLM 0.5 深度解析" §5.2 switches on; the pages
 * name only the switch, so this is the plain causal reading: q and out are
 * [B, T, Hq, D]; the T queries of sequence b sit at positions
 * p_t = seq_lens[b] - T + t (the last T positions of the sequence), and query
 * t attends to [start_t, p_t], start_t = max(0, p_t + 1 - window) when
 * window > 0, else 0. A query with p_t < 0 gives zeros. With T = 1 this is
 * orc_decode. triples lists distinct (b, t, h) rows (they are computed on
 * parallel threads), or is NULL for all of them.
 */
int orc_decode_multi(double* out, const uint16_t* q, int q_dtype, const void* key_cache,
                     const void* value_cache, int cache_dtype, const int32_t* block_tables,
                     const int32_t* seq_lens, int64_t batch, int64_t num_queries,
                     int64_t num_q_heads, int64_t num_kv_heads, int64_t head_dim,
                     int64_t num_blocks, int64_t block_size, int64_t max_blocks, double scale,
                     int64_t window, double k_scale, double v_scale, const int32_t* triples,
                     int64_t n_triples, int threads);

#ifdef __cplusplus
}
#endif
#endif
