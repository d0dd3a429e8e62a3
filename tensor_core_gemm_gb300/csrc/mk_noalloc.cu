// Allocation-free entry point: out = x @ w for a few rows (M <= 8), run as split-K GEMV tiles
// of the persistent kernel, with every piece of run state in one fixed, file-scope device array.
//
// Some callers cannot allocate device memory at the moment they need this product: a serving
// loop whose device memory was claimed up front by its own pool (cudaMalloc would fail or
// fragment that pool), code running inside such a pool's callbacks, or latency-bound paths
// where cudaMalloc / cudaFree would synchronise the device. mk_compile allocates a plan; this
// entry point allocates nothing. It calls no cudaMalloc, cudaFree or allocating library
// routine: the instruction records, node entry, tensor map, split semaphores, status words and
// fp32 split partials all live in g_noalloc_scratch below.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>
#include <string.h>

#include "mk_internal.h"
#include "mk_launch.h"


using namespace mk;

namespace {

// Fixed layout of the scratch array (bytes). Every GPU that loads the library holds the whole
// array until the process exits.
constexpr size_t kScratchBytes = 4u << 20;                              // 4 MiB
constexpr int kMaxTiles = 1024;                                         // N <= 262144
constexpr int kMaxInstr = 1024;                                         // tiles x splits
constexpr size_t kOffInstr = 0;
constexpr size_t kOffNode = kOffInstr + (size_t)kMaxInstr * sizeof(Instr);
constexpr size_t kOffMap = kOffNode + sizeof(Node);                     // 64-byte aligned
constexpr size_t kOffCtr = kOffMap + 128;                               // one semaphore per tile
constexpr size_t kOffStatus = kOffCtr + (size_t)kMaxTiles * 4;          // status, last, done
constexpr size_t kOffPart = (kOffStatus + (2 * kStatusWords + 1) * 4 + 255) & ~(size_t)255;
constexpr size_t kPartFloats = (kScratchBytes - kOffPart) / 4;          // split partials
static_assert(kOffMap % 64 == 0, "tensor map alignment");
static_assert(kOffPart < kScratchBytes, "layout fits");

constexpr int kTileN = 256;     // output columns per GEMV tile
constexpr int kKStep = kGemvRows;  // K chunks are multiples of the stage depth

// Host staging for the records copied into the array on every call (no heap use).
Instr h_instr[kMaxInstr];
Node h_node;
CUtensorMap h_map;

constexpr int kMaxDevices = 64;
char* g_scratch_dev[kMaxDevices];  // device address of the array, per device (set up once)

}  // namespace

// The scratch array. In host code this name is a host-side stand-in, never a device address;
// kernels receive the address that cudaGetSymbolAddress returns for the current device.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

static mk_status fail(mk_status code, const char* msg, cudaError_t e = cudaSuccess) {
  if (e != cudaSuccess)
    set_error("mk_gemv_noalloc: %s: %s", msg, cudaGetErrorString(e));
  else
    set_error("mk_gemv_noalloc: %s", msg);
  return code;
}

extern "C" mk_status mk_gemv_noalloc(const void* x, const void* w, void* out, int32_t m,
                                     int32_t n, int32_t k, int32_t dtype, void* stream,
                                     mk_device_status* status) {
  if (dtype != MK_F16 && dtype != MK_BF16)
    return fail(MK_ERR_UNSUPPORTED, "dtype must be MK_F16 or MK_BF16");
  if (m < 1 || m > 8) return fail(MK_ERR_UNSUPPORTED, "m must be 1..8");
  if (n < 1 || n % 8 || k < 0 || k % 8)
    return fail(MK_ERR_UNSUPPORTED, "n >= 1 and k >= 0 must be multiples of 8");
  const int64_t tiles = (n + kTileN - 1) / kTileN;
  if (tiles > kMaxTiles) {
    set_error("mk_gemv_noalloc: n = %d exceeds the maximum %d (fixed scratch holds %d tiles)",
              n, kMaxTiles * kTileN, kMaxTiles);
    return MK_ERR_UNSUPPORTED;
  }
  if (!x || !w || !out || ((uintptr_t)x | (uintptr_t)w | (uintptr_t)out) % 16)
    return fail(MK_ERR_INVALID_ARG, "x, w and out must be non-NULL and 16-byte aligned");

  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return fail(MK_ERR_CUDA, "no current CUDA device", e);
  if (dev >= kMaxDevices) return fail(MK_ERR_UNSUPPORTED, "device ordinal above 63");

  // Set-up, once per device, with that device current: the array's device address, and the
  // kernel's shared-memory limit. The first call on a device does this.
  if (!g_scratch_dev[dev]) {
    void* ptr = nullptr;
    e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
    if (e != cudaSuccess) return fail(MK_ERR_CUDA, "cudaGetSymbolAddress of the scratch array", e);
    e = configure_megakernel(megakernel_smem_bytes());
    if (e != cudaSuccess) return fail(MK_ERR_CUDA, "kernel attribute set-up", e);
    g_scratch_dev[dev] = static_cast<char*>(ptr);
  }
  char* base = g_scratch_dev[dev];

  // Split K the way a compiled plan does, then shrink the split count until the instruction
  // records and the partials fit the fixed array (one split needs no partials).
  int64_t s = std::max<int64_t>(1, sms / tiles);
  int64_t chunk = 0;
  for (;;) {
    chunk = std::max<int64_t>(kKStep, ((((int64_t)k + s - 1) / s + kKStep - 1) / kKStep) * kKStep);
    s = std::max<int64_t>(1, ((int64_t)k + chunk - 1) / chunk);
    const bool fits = tiles * s <= kMaxInstr &&
                      (s == 1 || (size_t)(s * m * (int64_t)n) <= kPartFloats);
    if (fits) break;
    s = s - 1;
  }

  // Records: one GEMV instruction per (column tile, split); no dependencies between them.
  int ni = 0;
  for (int64_t ct = 0; ct < tiles; ++ct) {
    for (int64_t si = 0; si < s; ++si) {
      Instr& in = h_instr[ni++];
      memset(&in, 0, sizeof in);
      in.op = OP_GEMV;
      in.n0 = (int32_t)(ct * kTileN);
      in.k0 = (int32_t)(si * chunk);
      in.klen = (int32_t)std::min<int64_t>(chunk, (int64_t)k - si * chunk);
      in.aux0 = (int32_t)si;
      in.aux1 = (int32_t)s;
      in.sem = (int32_t)ct;
    }
  }
  memset(&h_node, 0, sizeof h_node);
  h_node.kind = OP_GEMV;
  h_node.dtype = dtype;
  h_node.M = m;
  h_node.N = n;
  h_node.K = k;
  h_node.tile_n = kTileN;
  h_node.n_splits = (int32_t)s;
  h_node.ldp = m * n;
  h_node.a = Operand{(uint64_t)(uintptr_t)x, k, -1};
  h_node.b = Operand{(uint64_t)(uintptr_t)w, n, k > 0 ? 0 : -1};
  h_node.out = Operand{(uint64_t)(uintptr_t)out, n, -1};
  h_node.scratch = Operand{(uint64_t)(uintptr_t)(base + kOffPart), 0, -1};
  h_node.b2.tmap = h_node.bias.tmap = h_node.res.tmap = h_node.gamma.tmap = -1;
  h_node.out_k.tmap = h_node.out_v.tmap = -1;
  if (k > 0) {
    void* fnp = nullptr;
    cudaDriverEntryPointQueryResult q;
    e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fnp, 12000, cudaEnableDefault,
                                         &q);
    if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || !fnp)
      return fail(MK_ERR_CUDA, "cuTensorMapEncodeTiled is unavailable", e);
    auto encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fnp);
    cuuint64_t dims[2] = {(cuuint64_t)n, (cuuint64_t)k};
    cuuint64_t strides[1] = {(cuuint64_t)n * 2};
    cuuint32_t box[2] = {64u, (cuuint32_t)kGemvRows};  // four 64-column boxes per stage
    cuuint32_t estr[2] = {1, 1};
    CUresult r = encode(&h_map, dtype == MK_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                                 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
                        2, const_cast<void*>(w), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(MK_ERR_CUDA, "cuTensorMapEncodeTiled failed");
  }

  // Upload the records (from static host memory) and clear what must start at zero: the split
  // semaphores, the status words and the CTA completion count. The array keeps the last call's
  // contents otherwise.
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  e = cudaMemcpyAsync(base + kOffInstr, h_instr, (size_t)ni * sizeof(Instr),
                      cudaMemcpyHostToDevice, st);
  if (e == cudaSuccess)
    e = cudaMemcpyAsync(base + kOffNode, &h_node, sizeof h_node, cudaMemcpyHostToDevice, st);
  if (e == cudaSuccess && k > 0)
    e = cudaMemcpyAsync(base + kOffMap, &h_map, sizeof h_map, cudaMemcpyHostToDevice, st);
  if (e == cudaSuccess) e = cudaMemsetAsync(base + kOffCtr, 0, kOffPart - kOffCtr, st);
  if (e != cudaSuccess) return fail(MK_ERR_CUDA, "upload into the scratch array", e);

  Params p{};
  p.instrs = reinterpret_cast<const Instr*>(base + kOffInstr);
  p.nodes = reinterpret_cast<const Node*>(base + kOffNode);
  p.counters = reinterpret_cast<int32_t*>(base + kOffCtr);
  p.src_list = p.counters;  // no instruction has sources or arrivals
  p.dst_list = p.counters;
  p.status = reinterpret_cast<int32_t*>(base + kOffStatus);
  p.last_status = p.status + kStatusWords;
  p.done = p.last_status + kStatusWords;
  p.snapshot = nullptr;
  p.tmaps = base + kOffMap;
  p.n_instr = ni;
  p.n_sm = sms;
  p.n_tmaps = k > 0 ? 1 : 0;
  p.n_counters = (int32_t)tiles;
  p.timeout_ns = 2000000000ull;
  p.stages = kPairStages;  // GEMV tiles only: 32 KB stages
  e = launch_megakernel(p, sms, megakernel_smem_bytes(), st, false, KS_DECODE);
  if (e != cudaSuccess) return fail(MK_ERR_CUDA, "launch", e);

  if (status) {
    int32_t wds[kStatusWords];
    e = cudaStreamSynchronize(st);
    if (e == cudaSuccess)
      e = cudaMemcpy(wds, p.last_status, sizeof wds, cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return fail(MK_ERR_CUDA, "reading the run status", e);
    status->code = wds[ST_CODE];
    status->instr = wds[ST_INSTR];
    status->counter = wds[ST_COUNTER];
    status->observed = wds[ST_OBSERVED];
    status->expected = wds[ST_EXPECTED];
    status->sm = wds[ST_SM];
    status->role = wds[ST_ROLE];
    status->where = wds[ST_WHERE];
    if (status->code) {
      set_error("mk_gemv_noalloc: device reported status %d", status->code);
      return status->code;
    }
  }
  return MK_OK;
}
