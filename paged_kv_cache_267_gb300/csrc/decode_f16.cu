// Decode kernel instantiations for f16 caches (q and out are f16 too).
#include "decode.cuh"

namespace pa {

PA_DECODE_FAMILY(f16, kF16, kF16, false)

}  // namespace pa
