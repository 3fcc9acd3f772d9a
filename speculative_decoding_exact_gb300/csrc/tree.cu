// tree.cu — the decision of a token-tree verify step (Muser book Ch. 33 §33.7:
// a tree spends the verify batch on covering near-miss branches).
//
// Node 0 is the carried frontier; node i >= 1 holds the draft token tokens[i],
// proposed as the continuation of parent[i] < i.  The root is accepted; node
// i is accepted when its parent is and tokens[i] equals the parent's argmax.
// The deepest accepted node a (the lowest index among equals) ends the path
// root -> a: L = depth(a) drafts accepted, next = argmax of a.  The path's
// K/V rows (block slots path[d]) move to slots d, then the KV is rolled back
// to n_past + L + 1.  Up to 64 nodes (the section names trees of 24 to 64
// nodes): the forward runs in passes of up to 16 rows, each with the KV
// length set to the end of its rows, and every node's argmax is reduced
// before the decision.
//
// Kernels: the length of a pass (one thread), the decision (one thread), the
// K/V moves (one CTA per layer, K/V and KV head), the rollback and the result
// (one thread).
#include "common.cuh"
#include "internal.h"
#include "kvmeta.cuh"

namespace spec {

struct TreeScratch {
  int L, next, status, pad;
  int path[kTreeMax];
};
size_t tree_scratch_bytes() { return sizeof(TreeScratch); }

// before a pass over nodes [.., end): seq_len = the tree's first position +
// end, so that the step's kernels place row r of the pass at position
// seq_len - M + r (nothing when the step was aborted)
__global__ void tree_pass_kernel(KvView kv, const int32_t* step_state, const int32_t* status, int end) {
  pdl_trigger();
  pdl_wait();
  if (threadIdx.x == 0 && !(*status & kStepAbort) && step_state[1]) *kv.seq_len = step_state[0] + end;
}

cudaError_t launch_tree_pass(const KvView& kv, const int32_t* step_state, const int32_t* status, int end,
                             cudaStream_t st, bool pdl) {
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(1);
  cfg.blockDim = dim3(32);
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, tree_pass_kernel, kv, step_state, status, end);
}

// idx [n]: every node's argmax (lowest index among equal maxima)
__global__ void tree_decide_kernel(const int32_t* __restrict__ idx, const int32_t* __restrict__ tokens,
                                   const int32_t* __restrict__ parent, int n, int vocab,
                                   const int32_t* status, TreeScratch* sc, int32_t* idx_out) {
  pdl_trigger();
  pdl_wait();
  if (threadIdx.x != 0) return;
  int st = *status;
  for (int row = 0; row < n; ++row) {
    if (idx[row] < 0 || idx[row] >= vocab) st |= SPEC_ST_NONFINITE;
    if (idx_out) idx_out[row] = idx[row];
  }
  int L = 0, next = -1;
  if (!st) {
    int acc[kTreeMax], depth[kTreeMax], best = 0;
    acc[0] = 1;
    depth[0] = 0;
    for (int i = 1; i < n; ++i) {
      acc[i] = acc[parent[i]] && tokens[i] == idx[parent[i]];
      depth[i] = depth[parent[i]] + 1;
      if (acc[i] && depth[i] > depth[best]) best = i;
    }
    L = depth[best];
    next = idx[best];
    int a = best;
    for (int d = L; d >= 0; --d) {
      sc->path[d] = a;
      a = d > 0 ? parent[a] : a;
    }
  }
  sc->L = L;
  sc->next = next;
  sc->status = st;
}

// one CTA per (layer, K/V, KV head): the L rows are read first, then written
// (a destination slot d can be the source slot of an earlier path entry)
__global__ void tree_compact_kernel(KvView kv, const int32_t* step_state, const TreeScratch* sc) {
  pdl_trigger();
  pdl_wait();
  const int L = sc->L;
  if (sc->status || L == 0 || step_state[1] == 0) return;
  const int layer = blockIdx.x, which = blockIdx.y, head = blockIdx.z;
  const int n_past = step_state[0];
  const int t = threadIdx.x;                // (row d - 1, 16-byte chunk): up to 63 rows
  const int d = 1 + (t >> 4), ch = t & 15;
  auto row_ptr = [&](int slot) -> uint4* {
    const int page = kv.page_table[slot / kv.page_size];
    const size_t off = ((((size_t)page * kv.n_layers + layer) * 2 + which) * kv.n_kv + head) *
                           (size_t)kv.page_size * kv.head_dim +
                       (size_t)(slot % kv.page_size) * kv.head_dim;
    return reinterpret_cast<uint4*>(kv.pool + off);
  };
  uint4 v = make_uint4(0, 0, 0, 0);
  const bool mine = d <= L;
  if (mine) v = row_ptr(n_past + sc->path[d])[ch];
  __syncthreads();
  if (mine) row_ptr(n_past + d)[ch] = v;
}

__global__ void tree_finish_kernel(KvView kv, const int32_t* step_state, const TreeScratch* sc,
                                   int32_t* status, int32_t* res, int32_t* path_out, int path_len) {
  pdl_trigger();
  pdl_wait();
  if (threadIdx.x != 0) return;
  const int st = sc->status;
  int L = sc->L, next = sc->next;
  const bool appended = step_state[1] != 0;
  const int n_past = step_state[0];
  if (st) {
    L = 0;
    next = -1;
    if (appended) kv_rollback_dev(kv, n_past);
  } else if (appended) {
    kv_rollback_dev(kv, n_past + L + 1);
  }
  if (path_out)
    for (int d = 0; d < path_len; ++d) path_out[d] = (!st && d <= L) ? sc->path[d] : -1;
  *status = st;
  res[0] = L;
  res[1] = next;
  res[2] = st;
  res[3] = *kv.seq_len;
}

cudaError_t launch_tree_accept(const int32_t* idx, const int32_t* tokens, const int32_t* parent, int n,
                               int vocab, const KvView& kv, const int32_t* step_state, uint8_t* scratch,
                               int32_t* status, int32_t* res, int32_t* path_out, int32_t* idx_out,
                               cudaStream_t st, bool pdl) {
  if (kv.head_dim * 2 != 256 || n < 1 || n > kTreeMax) return cudaErrorInvalidValue;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  TreeScratch* sc = reinterpret_cast<TreeScratch*>(scratch);
  cfg.gridDim = dim3(1);
  cfg.blockDim = dim3(32);
  cudaError_t e = cudaLaunchKernelEx(&cfg, tree_decide_kernel, idx, tokens, parent, n, vocab,
                                     (const int32_t*)status, sc, idx_out);
  if (e != cudaSuccess) return e;
  cfg.gridDim = dim3(kv.n_layers, 2, kv.n_kv);
  cfg.blockDim = dim3(16 * max(n - 1, 1));  // (n - 1) rows x 16 chunks of 16 bytes
  e = cudaLaunchKernelEx(&cfg, tree_compact_kernel, kv, step_state, (const TreeScratch*)sc);
  if (e != cudaSuccess) return e;
  cfg.gridDim = dim3(1);
  cfg.blockDim = dim3(32);
  return cudaLaunchKernelEx(&cfg, tree_finish_kernel, kv, step_state, (const TreeScratch*)sc, status, res,
                            path_out, n > 16 ? n : 16);
}

}  // namespace spec
