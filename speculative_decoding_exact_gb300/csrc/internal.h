// internal.h — host-side launchers shared between the library's translation
// units.  Not part of the public ABI (include/spec_verify.h).
#pragma once
#include <cstdint>
#include <cuda_runtime.h>

#include "gemm_plan.h"

namespace spec {

// ---- launchers (all enqueue on `st`; `pdl` = programmatic dependent launch)
cudaError_t launch_repack(const void* src, void* dst, int N, int K, cudaStream_t st);
// withhold: the producer issues no copy (the self-test of the bounded waits:
// every consumer gives up after its limit with nothing in flight)
cudaError_t launch_gemm(const GemmPlan& p, const void* w_tiled, const uint8_t* act, float* pieces,
                        int32_t* isc, int32_t* imn, int m_sums, int32_t* status, cudaStream_t st,
                        bool pdl, bool withhold = false);
// y[m][n] = sum of the pieces, m < M
cudaError_t launch_sum_pieces(const GemmPlan& p, const float* pieces, float* y, int M,
                              cudaStream_t st, bool pdl);

// the CUDA-core (dp4a) GEMM of the tensor-core comparison: plain int8 codes q
// [M][K], d_a [M][K/256], sub-block sums A [M][K/32] -> y [M][N] (zeroed
// here, superblock ranges added with atomics)
cudaError_t launch_gemm_dp4a(const void* w_tiled, const int8_t* q, const float* da, const int32_t* A, int M,
                             int N, int K, float* y, int num_sms, cudaStream_t st);

// act buffer: (K/256) superblocks of kActSBBytes bytes (fragment-ordered f16 codes,
// min-term slot, d_a) produced from fp32 rows x[M][K]
cudaError_t launch_quantize(const float* x, int M, int K, uint8_t* act, int8_t* q_dbg,
                            float* da_dbg, int32_t* A_dbg, int32_t* status, cudaStream_t st,
                            bool pdl);

// residual add of GEMM pieces (optional), RMSNorm with gain, quantise -> act.
// x_out = x_in + pieces (x_out may equal x_in, or be NULL without pieces);
// xnorm_out (optional) receives the normalised rows.
cudaError_t launch_resid_norm_quant(const GemmPlan* p, const float* pieces, const float* x_in,
                                    float* x_out, const float* gamma, float eps, int M, int H,
                                    uint8_t* act, float* xnorm_out, int32_t* status,
                                    cudaStream_t st, bool pdl, float* cap = nullptr, int cap_ld = 0);

// h = silu(gate) * up from the gate|up GEMM pieces, quantised -> act (K = F)
cudaError_t launch_swiglu_quant(const GemmPlan& p, const float* pieces, int M, int F,
                                uint8_t* act, int32_t* status, cudaStream_t st, bool pdl);

// QKV pieces -> Q attention fragments; K,V rows -> bf16 cache at positions seq_len-M+i
struct KvView {
  uint16_t* pool;            // bf16 bits
  int32_t* page_table;
  int32_t* seq_len;
  int32_t* free_stack;
  int32_t* free_top;
  int num_pages, max_seq_pages, n_layers, n_kv, head_dim, page_size;
  // sliding-window layers (swa_window 0: none): ring [n_swa][K,V][n_kv][R][dh]
  // bf16 with R = swa_rows = W rounded up to 16, plus 16; swa_state = {the
  // last step's block position n (-1: none), its rows}
  uint16_t* swa_ring;
  int32_t* swa_state;
  int swa_window, swa_period, swa_rows;
  int max_ctx;               // positions >= max_ctx are refused (SPEC_ST_CTX_FULL)
};

// layer l is a sliding-window layer when l % period == period - 1; its index
// among those layers is l / period
__host__ __device__ __forceinline__ int swa_index(const KvView& kv, int layer) {
  if (kv.swa_window <= 0 || kv.swa_period <= 0 || layer % kv.swa_period != kv.swa_period - 1) return -1;
  return layer / kv.swa_period;
}
__host__ __device__ __forceinline__ int swa_layers(const KvView& kv) {
  return (kv.swa_window > 0 && kv.swa_period > 0) ? kv.n_layers / kv.swa_period : 0;
}
__host__ __device__ __forceinline__ int swa_ring_rows(int window) { return (window + 15) / 16 * 16 + 16; }
__host__ __device__ __forceinline__ size_t ring_row(const KvView& kv, int s, int which, int head, int slot) {
  return ((((size_t)s * 2 + which) * kv.n_kv + head) * kv.swa_rows + slot) * kv.head_dim;
}
// In a sliding-window layer the K,V rows go to the layer's ring (slot
// position mod swa_rows) instead of the paged pool.
// Optional per-head transforms of q and k before they are stored: QK-norm
// with gains gq / gk (nullptr: none) and RoPE from the table cs[pos][dh/2] of
// (cos, sin) for pos < cs_len (nullptr: none).
struct QkTransform {
  const float* gq = nullptr;
  const float* gk = nullptr;
  const float2* cs = nullptr;
  int cs_len = 0;
  float eps = 0.f;
};
cudaError_t launch_qkv_post(const GemmPlan& p, const float* pieces, int M, int nq, int nkv,
                            int dh, const KvView& kv, int layer, uint8_t* qtile, int tiles,
                            const int32_t* status, cudaStream_t st, bool pdl, bool late_trigger,
                            const QkTransform& qk = QkTransform{});

// verify attention: partials then merge (+ quantise for the O projection)
struct AttnPlan {
  int nq = 0, nkv = 0, dh = 0, max_ctx = 0, chunk = 0, max_chunks = 0;
  int sub = 64;                 // keys per sub-chunk: 64 or 128
  int group = 0, tiles = 0;     // query heads per kv head; 128-row MMA tiles per kv head
  // the chunk fits the K/V ring: the partial kernel reads the KV metadata and
  // copies the chunk's rows of earlier steps before its dependency wait, and
  // the QKV kernel before it signals only after its own wait
  bool early = false;
};
// max_ctx: the span of keys one block may see (the context length; for a
// sliding-window layer the window plus 32)
AttnPlan make_attn_plan(int nq, int nkv, int dh, int max_ctx);
size_t attn_partial_floats(const AttnPlan& a, int max_rows);
// Q tiles (bf16 hi/lo, 64 KB per (kv head, tile); layout at write_qtile) from
// fp32 q [M][nq][128]; rows >= M zero.  Rows of heads past the group are never
// written: the buffer is zeroed once at init.
size_t qtile_bytes(const AttnPlan& a);
cudaError_t launch_q_to_tile(const float* q, int M, const AttnPlan& a, uint8_t* qtile, cudaStream_t st,
                             bool pdl);
// tree_mask (DEVICE uint64 [M], optional): the tree nodes row i sees (bit j
// = node j at position *tree_base + j); NULL = causal.  A sliding-window
// layer (swa_index(kv, layer) >= 0) reads its ring, keeps the keys of the
// window, and places its chunks from the window's first page on (a plan made
// for the window).
cudaError_t launch_attention(const AttnPlan& a, const KvView& kv, int layer, const uint8_t* qtile,
                             int M, float* part, float* out, uint8_t* act, int32_t* status,
                             cudaStream_t st, bool pdl, const uint64_t* tree_mask = nullptr,
                             const int32_t* tree_base = nullptr);

// stochastic exact acceptance: row normalizers (stats fp32x2 [k+1]: max and
// sum of exp) then the decisions, the final draw and the rollback; mt is the
// 625-word MT19937 state (DEVICE), advanced by the draws
size_t sample_scratch_bytes();
cudaError_t launch_sample_accept(const float* logits, const float* q, const int32_t* draft, int k,
                                 int V, float2* stats, uint8_t* scratch, uint32_t* mt, const KvView* kv,
                                 const int32_t* step_state, int32_t* status, int32_t* res,
                                 cudaStream_t st, bool pdl);

// token-tree decision over n <= kTreeMax nodes from every node's argmax idx
// [n]: the accepted path, its K/V moves and the rollback; path_out (DEVICE
// int32 [max(16, n)], optional) = the path's nodes, -1 after it
size_t tree_scratch_bytes();
cudaError_t launch_tree_accept(const int32_t* idx, const int32_t* tokens, const int32_t* parent, int n,
                               int vocab, const KvView& kv, const int32_t* step_state, uint8_t* scratch,
                               int32_t* status, int32_t* res, int32_t* path_out, int32_t* idx_out,
                               cudaStream_t st, bool pdl);
// a pass of a tree forward over the nodes [.., end): seq_len = tree start + end
cudaError_t launch_tree_pass(const KvView& kv, const int32_t* step_state, const int32_t* status, int end,
                             cudaStream_t st, bool pdl);

// LM head argmax over the head GEMM pieces: per-(CTA,row) partial (value, index)
int head_argmax_blocks(int V);
cudaError_t launch_head_argmax(const GemmPlan& p, const float* pieces, int M, float* logits,
                               float* part_val, int32_t* part_idx, int32_t* status,
                               cudaStream_t st, bool pdl);
cudaError_t launch_argmax_final(const float* part_val, const int32_t* part_idx, int nparts, int M,
                                int32_t* idx, cudaStream_t st, bool pdl);

// KV metadata kernels
cudaError_t launch_kv_reset(const KvView& kv, cudaStream_t st);
// map pages for [seq_len, seq_len + n); commit seq_len += n when `commit`
// (a step reserves its block; extend commits).  `draft`/`k`/`vocab` (optional)
// validate the draft tokens first; on any failure nothing changes.
cudaError_t launch_kv_reserve(const KvView& kv, int n, int commit, const int32_t* draft, int k,
                              int vocab, int32_t* status, int32_t* step_state, cudaStream_t st,
                              bool pdl, const int32_t* parent = nullptr,
                              uint64_t* tree_mask = nullptr);
cudaError_t launch_kv_rollback(const KvView& kv, int new_len, int32_t* status, cudaStream_t st);
// accept + rollback; idx [k+1] from head_argmax final reduce (or given)
cudaError_t launch_accept(const int32_t* idx, const float* part_val, const int32_t* part_idx,
                          int nparts, const int32_t* draft, int k, int vocab, const KvView* kv,
                          const int32_t* step_state, int32_t* status, int32_t* res,
                          int32_t* idx_out, cudaStream_t st, bool pdl);

}  // namespace spec
