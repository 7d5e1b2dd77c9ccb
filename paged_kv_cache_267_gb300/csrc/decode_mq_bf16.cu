// Chunked-query kernel instantiations for bf16 caches.
#include "decode.cuh"

namespace pa {

PA_DECODE_FAMILY(mq_bf16, kBF16, kBF16, true)

}  // namespace pa
