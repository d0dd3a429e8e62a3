// Prefill specialisation of the persistent kernel: GEMM tiles, causal prefill attention and row
// instructions (no GEMV or split-KV attention path).
#include "mk_megakernel.cuh"

namespace mk {

KernelVariant variant_prefill() { return make_variant<false, KS_PREFILL>(); }

}  // namespace mk
