// Decode kernel instantiations for bf16 caches (q and out are bf16 too).
#include "decode.cuh"

namespace pa {

PA_DECODE_FAMILY(bf16, kBF16, kBF16, false)

}  // namespace pa
