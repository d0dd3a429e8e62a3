// Decode specialisation of the persistent kernel: GEMV tiles, split-KV attention partials and
// combines, and row instructions; no tensor-memory allocation, no tcgen05 path.
#include "mk_megakernel.cuh"

namespace mk {

KernelVariant variant_decode() { return make_variant<false, KS_DECODE>(); }

}  // namespace mk
