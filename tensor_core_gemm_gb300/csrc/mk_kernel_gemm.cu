// GEMM-only specialisations of the persistent kernel (single CTAs and CTA pairs): plans made of
// tcgen05 GEMM tiles alone.
#include "mk_megakernel.cuh"

namespace mk {

KernelVariant variant_gemm(bool pair) {
  return pair ? make_variant<true, KS_GEMM>() : make_variant<false, KS_GEMM>();
}

}  // namespace mk
