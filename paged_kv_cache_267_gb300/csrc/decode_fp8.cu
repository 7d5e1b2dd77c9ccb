// Decode kernel instantiations for e4m3 caches with f16 or bf16 queries.
#include "decode.cuh"

namespace pa {

cudaError_t decode_variant_fp8(int qt, int D, int nt, DecodeVariant* v) {
  if (D == 64) return cudaErrorInvalidValue;
  if (qt == kBF16) PA_DECODE_DISPATCH(kE4M3, kBF16, D, nt, { *v = K::variant(); return cudaSuccess; });
  PA_DECODE_DISPATCH(kE4M3, kF16, D, nt, { *v = K::variant(); return cudaSuccess; });
}

cudaError_t decode_prepare_fp8(int qt, int D, int nt, int smem, int* ctas_per_sm) {
  if (D == 64) return cudaErrorInvalidValue;
  if (qt == kBF16) PA_DECODE_DISPATCH(kE4M3, kBF16, D, nt, { return K::prepare(smem, ctas_per_sm); });
  PA_DECODE_DISPATCH(kE4M3, kF16, D, nt, { return K::prepare(smem, ctas_per_sm); });
}

cudaError_t decode_launch_fp8(int qt, int D, int nt, const CUtensorMap& tk, const CUtensorMap& tv,
                              const DecodeArgs& a, int grid, int smem, cudaStream_t s, bool pdl) {
  if (D == 64) return cudaErrorInvalidValue;
  if (qt == kBF16)
    PA_DECODE_DISPATCH(kE4M3, kBF16, D, nt, { return K::launch(tk, tv, a, grid, smem, s, pdl); });
  PA_DECODE_DISPATCH(kE4M3, kF16, D, nt, { return K::launch(tk, tv, a, grid, smem, s, pdl); });
}

}  // namespace pa
