// Packed copies of GEMV weights. A GEMV tile streams its weight W (K x N, row-major, leading
// dimension ld elements) as 64-row stages of tw columns (256, or 128 per weight for the two
// weights of a SiLU·mul node), each stage a set of 64-column panels of 64 rows x 128 bytes in the
// layout a 128-byte-swizzled TMA copy leaves in shared memory (16-byte chunk c of row r at
// c ^ (r mod 8)). As a multi-dimensional TMA copy such a stage is 256 separate 128-byte lines,
// which streams from HBM at about half the rate of one contiguous copy; the packed copy stores
// every stage contiguously in that final layout, so the kernel loads it with one bulk copy:
//   unit(t, kb) at ((t * KB + kb) * (tw / 64) + p) * 8192, t = column tile, kb = 64-row block,
// panels p in order, zero beyond K and N (what the TMA copy reads out of bounds).
#include <cuda_runtime.h>
#include <stdint.h>

namespace mk {

__global__ void pack_gemv_kernel(const uint16_t* __restrict__ w, long long ld, int K, int N,
                                 int tw, int kb_n, long long chunks, uint8_t* __restrict__ dst) {
  const int panels = tw / 64;
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < chunks;
       i += (long long)gridDim.x * blockDim.x) {
    const int c = (int)(i & 7), r = (int)((i >> 3) & 63);
    long long rest = i >> 9;
    const int p = (int)(rest % panels);
    rest /= panels;
    const int kb = (int)(rest % kb_n);
    const long long t = rest / kb_n;
    const long long k = (long long)kb * 64 + r, n = t * tw + p * 64 + c * 8;
    uint16_t v[8] = {0, 0, 0, 0, 0, 0, 0, 0};
    if (k < K) {
      const uint16_t* row = w + k * ld;
      for (int e = 0; e < 8; ++e)
        if (n + e < N) v[e] = row[n + e];
    }
    uint4 q;
    q.x = (uint32_t)v[0] | ((uint32_t)v[1] << 16);
    q.y = (uint32_t)v[2] | ((uint32_t)v[3] << 16);
    q.z = (uint32_t)v[4] | ((uint32_t)v[5] << 16);
    q.w = (uint32_t)v[6] | ((uint32_t)v[7] << 16);
    uint8_t* unit = dst + (((t * kb_n + kb) * panels + p) * 64 + r) * 128;
    *reinterpret_cast<uint4*>(unit + ((c ^ (r & 7)) << 4)) = q;
  }
}

size_t packed_gemv_bytes(int K, int N, int tw) {
  const size_t t = (size_t)((N + tw - 1) / tw), kb = (size_t)((K + 63) / 64);
  return t * kb * (size_t)tw * 128;
}

cudaError_t pack_gemv_weight(const void* w, long long ld, int K, int N, int tw, void* dst,
                             cudaStream_t stream) {
  const int kb_n = (K + 63) / 64;
  const long long chunks = (long long)((N + tw - 1) / tw) * kb_n * (tw / 64) * 64 * 8;
  if (chunks == 0) return cudaSuccess;
  const long long blocks = (chunks + 255) / 256;
  pack_gemv_kernel<<<(unsigned)(blocks < 65535 * 4 ? blocks : 65535 * 4), 256, 0, stream>>>(
      reinterpret_cast<const uint16_t*>(w), ld, K, N, tw, kb_n, chunks,
      reinterpret_cast<uint8_t*>(dst));
  return cudaGetLastError();
}

}  // namespace mk
