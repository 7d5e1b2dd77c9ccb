// Chunked-query kernel instantiations for f16 caches.
#include "decode.cuh"

namespace pa {

PA_DECODE_FAMILY(mq_f16, kF16, kF16, true)

}  // namespace pa
