// Chunked-query kernel instantiations for e4m3 caches with f16 or bf16 queries.
#include "decode.cuh"

namespace pa {

PA_DECODE_FAMILY(mq_fp8_bf16, kE4M3, kBF16, true)
PA_DECODE_FAMILY(mq_fp8_f16, kE4M3, kF16, true)

}  // namespace pa
