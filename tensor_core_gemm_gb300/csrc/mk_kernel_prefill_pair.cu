// Prefill specialisation of the persistent kernel on CTA pairs: 256x256 GEMM tiles and 256-row
// causal attention tiles issued as cta_group::2 MMAs, and row instructions.
#include "mk_megakernel.cuh"

namespace mk {

KernelVariant variant_prefill_pair() { return make_variant<true, KS_PREFILL>(); }

}  // namespace mk
