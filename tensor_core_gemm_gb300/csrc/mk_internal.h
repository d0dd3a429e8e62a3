// Host-side structures shared by the compiler (mk_graph.cpp), the runtime (mk_runtime.cpp)
// and the launch stub (mk_kernel.cu).
#pragma once
#include <stdarg.h>
#include <stdint.h>

#include <algorithm>
#include <string>
#include <vector>

#include "mk.h"
#include "mk_types.h"

namespace mk {

// A registered tensor or a view of one. Views resolve to their base tensor plus an offset;
// `base == own id` for base tensors.
struct TensorRec {
  void* ptr = nullptr;   // first element of this tensor / view
  int dtype = 0;
  int64_t rows = 0, cols = 0, ld = 0;
  int base = -1;
  int64_t r0 = 0, c0 = 0;   // offset inside the base tensor
  bool internal = false;    // plan-owned scratch created by the lowering
  bool transient = false;   // plan-owned intermediate placed in the buffer pool (mk_add_transient)
};

enum NodeKind { NK_MATMUL = 0, NK_EW = 1, NK_RMSNORM = 2, NK_ROPE = 3, NK_ATTN = 4, NK_ARGMAX = 5 };

struct NodeRec {
  int kind = 0;
  int a = -1, b = -1, b2 = -1, out = -1, bias = -1, res = -1, gamma = -1;
  int out_k = -1, out_v = -1;
  int ins[2] = {-1, -1};
  int n_in = 0;
  int ewop = 0;
  uint32_t flags = 0;
  float eps = 0.f, theta = 0.f, scale = 0.f;
  int hq = 0, hkv = 0, hd = 0, pos0 = 0, causal = 0;
};

struct Box {
  int t = -1;
  int64_t r0 = 0, r1 = 0, c0 = 0, c1 = 0;
  bool empty() const { return r0 >= r1 || c0 >= c1; }
};

inline bool meets(const Box& a, const Box& b) {
  return a.t == b.t && !a.empty() && !b.empty() && a.r0 < b.r1 && b.r0 < a.r1 && a.c0 < b.c1 &&
         b.c0 < a.c1;
}

enum Role { ROLE_A = 0, ROLE_B = 1, ROLE_E = 2 };

struct HInstr {
  Instr rec{};
  std::vector<std::pair<Box, int>> reads;  // (box, role)
  std::vector<Box> writes;
  int tile = -1;  // split semaphore ordinal (GEMV tile, or GEMM split-tail tile and rank)
  std::vector<std::pair<int, int>> src;
  std::vector<int> dst;
};

// Lowered, scheduled plan on the host (no device state).
struct HostPlan {
  std::vector<Instr> instrs;
  std::vector<int32_t> src_list;  // pairs
  std::vector<int32_t> dst_list;
  std::vector<int32_t> targets;
  int n_dep = 0, n_sem = 0, n_sm = 0;
  std::vector<TensorRec> tensors;          // user tensors, then internal scratch tensors
  std::vector<int> node_scratch;           // per node: internal tensor id or -1
  std::vector<int> node_splits;            // per node: GEMV K splits (0 otherwise)
  std::vector<int> node_chunks;            // per node: attention decode chunks (0 otherwise)
  std::vector<int> node_tile_n;            // per node: output columns per tile
  std::vector<int> node_gsplit_slots;      // per node: fp32 partial slots of GEMM split tails
  std::vector<int> node_rope;              // per matmul node: the ROPE node fused into it, or -1
  std::vector<int64_t> pool_off;           // per tensor: byte offset in the buffer pool, or -1
  int64_t pool_bytes = 0;
  int n_reuse = 0;                         // reuse events (one reuse counter each)
};

void set_error(const char* fmt, ...);
int dtype_size(int dt);

// Compiler entry point: lower + schedule. Returns MK_OK or an error with mk_last_error set.
mk_status lower_graph(const std::vector<TensorRec>& tensors, const std::vector<NodeRec>& nodes,
                      const mk_compile_opts& o, HostPlan* out);

// Kernel-support checks for a graph that is about to run on the device.
mk_status check_kernel_support(const std::vector<TensorRec>& tensors,
                               const std::vector<NodeRec>& nodes, const mk_compile_opts& o);

}  // namespace mk

struct mk_graph {
  std::vector<mk::TensorRec> tensors;
  std::vector<mk::NodeRec> nodes;
};
