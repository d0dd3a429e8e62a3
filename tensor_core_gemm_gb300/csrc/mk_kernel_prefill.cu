// Prefill specialisation of the persistent kernel: GEMM tiles, causal prefill attention and row
// instructions (no GEMV or split-KV attention path). The CTA-pair form compiles in its own
// translation unit (mk_kernel_prefill_pair.cu), in parallel with this one.
#include "mk_megakernel.cuh"

namespace mk {

KernelVariant variant_prefill(bool pair) {
  return pair ? variant_prefill_pair() : make_variant<false, KS_PREFILL>();
}

}  // namespace mk
