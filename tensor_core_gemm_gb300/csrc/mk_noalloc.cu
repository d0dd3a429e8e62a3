// Allocation-free entry point: out = x @ w for a few rows (M <= 8), run as split-K GEMV tiles
// of the persistent kernel, with every piece of run state in one fixed, file-scope device array.
//
// Some callers cannot allocate device memory at the moment they need this product: a serving
// loop whose device memory was claimed up front by its own pool (cudaMalloc would fail or
// fragment that pool), code running inside such a pool's callbacks, or latency-bound paths
// where cudaMalloc / cudaFree would synchronise the device. mk_compile allocates a plan; this
// entry point allocates nothing. It calls no cudaMalloc, cudaFree or allocating library
// routine: the instruction records, node entry, tensor map, split semaphores, status words and
// fp32 split partials all live in g_noalloc_scratch below. A small set-up kernel, given the
// records by value, writes them there before each run, so the call reads no host buffer after
// it returns.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>
#include <string.h>

#include <algorithm>

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

constexpr int kMaxDevices = 64;
char* g_scratch_dev[kMaxDevices];  // device address of the array, per device (set up once)

// Everything a call writes into the array, passed to the set-up kernel by value: kernel
// parameters are copied when the launch is enqueued, so no host buffer is read after the call
// returns and calls from several host threads share no host state.
struct SetupArgs {
  CUtensorMap map;   // 64-byte aligned first member
  Node node;
  char* base;        // device address of the array
  int32_t tiles, splits, chunk, k, has_map;
};

// One CTA of 256 threads: the instruction records (one GEMV per column tile and K split, the
// same order and fields a compiled plan uses), the node entry, the tensor map, and zeros over
// the split semaphores, status words and CTA completion count.
__global__ void __launch_bounds__(256) noalloc_setup(const __grid_constant__ SetupArgs a) {
  Instr* ins = reinterpret_cast<Instr*>(a.base + kOffInstr);
  const int n = a.tiles * a.splits;
  for (int i = (int)threadIdx.x; i < n; i += (int)blockDim.x) {
    const int ct = i / a.splits, si = i % a.splits;
    Instr r;
    memset(&r, 0, sizeof r);
    r.op = OP_GEMV;
    r.n0 = ct * kTileN;
    r.k0 = si * a.chunk;
    r.klen = min(a.chunk, a.k - si * a.chunk);
    r.aux0 = si;
    r.aux1 = a.splits;
    r.sem = ct;
    ins[i] = r;
  }
  const uint32_t* nsrc = reinterpret_cast<const uint32_t*>(&a.node);
  uint32_t* ndst = reinterpret_cast<uint32_t*>(a.base + kOffNode);
  for (int i = (int)threadIdx.x; i < (int)(sizeof(Node) / 4); i += (int)blockDim.x)
    ndst[i] = nsrc[i];
  if (a.has_map) {
    const uint32_t* msrc = reinterpret_cast<const uint32_t*>(&a.map);
    uint32_t* mdst = reinterpret_cast<uint32_t*>(a.base + kOffMap);
    for (int i = (int)threadIdx.x; i < (int)(sizeof(CUtensorMap) / 4); i += (int)blockDim.x)
      mdst[i] = msrc[i];
  }
  uint32_t* z = reinterpret_cast<uint32_t*>(a.base + kOffCtr);
  for (int i = (int)threadIdx.x; i < (int)((kOffPart - kOffCtr) / 4); i += (int)blockDim.x)
    z[i] = 0u;
}

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

  // A capturing stream takes the set-up kernel and the launch as graph nodes (their arguments
  // are passed by value), but neither the per-device set-up nor the status read (a stream
  // synchronisation and a copy) is legal while the stream captures.
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  e = cudaStreamIsCapturing(st, &cap);
  if (e != cudaSuccess) return fail(MK_ERR_CUDA, "cudaStreamIsCapturing", e);
  if (cap != cudaStreamCaptureStatusNone && (status || !g_scratch_dev[dev]))
    return fail(MK_ERR_UNSUPPORTED,
                "a capturing stream needs status == NULL and an earlier uncaptured call on this "
                "device");

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

  // Records: one GEMV instruction per (column tile, split), no dependencies between them,
  // written on the device by the set-up kernel from the arguments below.
  SetupArgs sa;
  memset(&sa, 0, sizeof sa);
  sa.base = base;
  sa.tiles = (int32_t)tiles;
  sa.splits = (int32_t)s;
  sa.chunk = (int32_t)chunk;
  sa.k = k;
  sa.has_map = k > 0;
  const int ni = (int)(tiles * s);
  Node& nd = sa.node;
  nd.kind = OP_GEMV;
  nd.dtype = dtype;
  nd.M = m;
  nd.N = n;
  nd.K = k;
  nd.tile_n = kTileN;
  nd.n_splits = (int32_t)s;
  nd.ldp = m * n;
  nd.a = Operand{(uint64_t)(uintptr_t)x, k, -1};
  nd.b = Operand{(uint64_t)(uintptr_t)w, n, k > 0 ? 0 : -1};
  nd.out = Operand{(uint64_t)(uintptr_t)out, n, -1};
  nd.scratch = Operand{(uint64_t)(uintptr_t)(base + kOffPart), 0, -1};
  nd.b2.tmap = nd.bias.tmap = nd.res.tmap = nd.gamma.tmap = -1;
  nd.out_k.tmap = nd.out_v.tmap = nd.out_q.tmap = -1;
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
    CUresult r = encode(&sa.map, dtype == MK_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                                  : CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
                        2, const_cast<void*>(w), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(MK_ERR_CUDA, "cuTensorMapEncodeTiled failed");
  }

  // Write the records into the array and clear what must start at zero (the split
  // semaphores, the status words and the CTA completion count); the array keeps the previous
  // call's contents otherwise.
  noalloc_setup<<<1, 256, 0, st>>>(sa);
  e = cudaGetLastError();
  if (e != cudaSuccess) return fail(MK_ERR_CUDA, "set-up launch", e);

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
