// Decode kernel instantiations for bf16 caches (q and out are bf16 too).
#include "decode.cuh"

namespace pa {

cudaError_t decode_variant_bf16(int D, int nt, DecodeVariant* v) {
  PA_DECODE_DISPATCH(kBF16, kBF16, D, nt, { *v = K::variant(); return cudaSuccess; });
}

cudaError_t decode_prepare_bf16(int D, int nt, int smem, int* ctas_per_sm) {
  PA_DECODE_DISPATCH(kBF16, kBF16, D, nt, { return K::prepare(smem, ctas_per_sm); });
}

cudaError_t decode_launch_bf16(int D, int nt, const CUtensorMap& tk, const CUtensorMap& tv,
                              const DecodeArgs& a, int grid, int smem, cudaStream_t s,
                              bool pdl) {
  PA_DECODE_DISPATCH(kBF16, kBF16, D, nt, { return K::launch(tk, tv, a, grid, smem, s, pdl); });
}

}  // namespace pa
