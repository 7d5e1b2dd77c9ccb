// Decode kernel instantiations for e4m3 caches with f16 or bf16 queries.
#include "decode.cuh"

namespace pa {

PA_DECODE_FAMILY(fp8_bf16, kE4M3, kBF16, false)
PA_DECODE_FAMILY(fp8_f16, kE4M3, kF16, false)

}  // namespace pa
