// Launch dispatcher of the persistent kernel and the general specialisation (every instruction
// kind). The GEMM-only, decode and prefill specialisations are instantiated by their own
// translation units (mk_kernel_gemm.cu, mk_kernel_decode.cu, mk_kernel_prefill.cu).
#include "mk_launch.h"
#include "mk_megakernel.cuh"

namespace mk {

KernelVariant variant_all(bool pair) {
  return pair ? make_variant<true, KS_ALL>() : make_variant<false, KS_ALL>();
}

size_t megakernel_smem_bytes() { return kMegakernelSmem; }

int launched_kernel_set(int ks, bool pair) {
  if (ks < KS_ALL || ks > KS_PREFILL) return KS_ALL;
  return pair && ks == KS_DECODE ? KS_ALL : ks;
}

static KernelVariant pick(int ks, bool pair) {
  switch (launched_kernel_set(ks, pair)) {
    case KS_GEMM: return variant_gemm(pair);
    case KS_DECODE: return variant_decode();
    case KS_PREFILL: return variant_prefill(pair);
    default: return variant_all(pair);
  }
}

cudaError_t configure_megakernel(size_t smem) {
  const KernelVariant all[] = {variant_all(false), variant_all(true), variant_gemm(false),
                               variant_gemm(true), variant_decode(), variant_prefill(false),
                               variant_prefill(true)};
  for (const KernelVariant& v : all) {
    const cudaError_t e = v.configure(smem);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

cudaError_t pair_clusters_resident(size_t smem, int ks, int* n) {
  return pick(ks, true).clusters_resident(smem, n);
}

cudaError_t launch_megakernel(const Params& p, int grid, size_t smem, cudaStream_t stream,
                              bool pair, int ks) {
  return pick(ks, pair).launch(p, grid, smem, stream);
}

}  // namespace mk
