// Host stubs of the persistent kernel, defined in mk_kernel.cu (which dispatches to the
// translation unit of each specialisation).
#pragma once
#include <cuda_runtime.h>
#include <stddef.h>

#include "mk_types.h"

namespace mk {

// Dynamic shared memory of one CTA (the same for every specialisation).
size_t megakernel_smem_bytes();
// Raise the dynamic shared-memory limit of every specialisation to `smem`.
cudaError_t configure_megakernel(size_t smem);
// 2-CTA clusters of the CTA-pair kernel of set `ks` that can be resident at once.
cudaError_t pair_clusters_resident(size_t smem, int ks, int* n);
// One persistent launch of `grid` CTAs of specialisation `ks` (a KernelSet) on `stream`:
// 2-CTA clusters when `pair`, a cooperative launch otherwise.
cudaError_t launch_megakernel(const Params& p, int grid, size_t smem, cudaStream_t stream,
                              bool pair, int ks);
// The KernelSet launched for `ks` and `pair`: pair kernels exist for KS_GEMM and KS_ALL only.
int launched_kernel_set(int ks, bool pair);

}  // namespace mk
