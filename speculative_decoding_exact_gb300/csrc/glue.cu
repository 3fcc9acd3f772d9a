// glue.cu — the small kernels around the GEMMs of the verify step:
// activation quantisation into the tensor-core operand order, residual add +
// RMSNorm + quantisation (one CTA per row), SwiGLU + quantisation,
// QKV split with the K/V append into the paged bf16 cache, the LM-head argmax,
// the greedy accept + KV rollback kernel and the KV metadata kernels.
//
// Sources (page titles and sections):
//   accept rule            Muser book Ch. 33 §33.2 (greedy = one-hot case)
//   carried frontier       Ch. 33 §33.7
//   verify lengths, rewind Ch. 8 §8.6 items 3 and 4
//   F32 residual, one fixed reduction order
//                          Ch. 32 "Precision across the handoff" (intro, §32.4)
#include "common.cuh"
#include "internal.h"
#include "quant.cuh"
#include "kvmeta.cuh"

namespace spec {

// number of pieces (CTA slots) of the group holding column col.  The GEMM
// plan splits U units over G CTAs in contiguous ranges: unit x belongs to CTA
// ((x+1)*G - 1)/U.  U*G stays far below 2^31 for every shape here (the LM
// head has U = 1024*26, G <= 152), so 32-bit arithmetic is exact.
__device__ __forceinline__ int piece_slots(int nb, int U, int G, int col) {
  const int gr = (col >> 4) / kTilesPerGroup;
  const int x0 = gr * nb, x1 = x0 + nb - 1;
  return ((x1 + 1) * G - 1) / U - ((x0 + 1) * G - 1) / U + 1;
}

// sum of the ns pieces of output (row, col), slots in order
__device__ __forceinline__ float piece_sum(const float* __restrict__ pieces, int N, int ns, int row,
                                           int col) {
  // independent loads of at most kMaxSlots slots, added in slot order
  float v[kMaxSlots];
#pragma unroll
  for (int k = 0; k < kMaxSlots; ++k) v[k] = k < ns ? pieces[((size_t)k * 16 + row) * N + col] : 0.f;
  float s = v[0];
#pragma unroll
  for (int k = 1; k < kMaxSlots; ++k)
    if (k < ns) s += v[k];
  return s;
}

// the same for 8 consecutive columns col0 .. col0+7 (col0 % 8 == 0, N % 8 == 0:
// one group, 32-byte aligned rows), each summed in slot order
__device__ __forceinline__ void piece_sum8(const float* __restrict__ pieces, int N, int ns, int row,
                                           int col0, float (&out)[8]) {
#pragma unroll
  for (int i = 0; i < 8; ++i) out[i] = 0.f;
#pragma unroll
  for (int k = 0; k < kMaxSlots; ++k) {
    if (k < ns) {
      const float4* p = reinterpret_cast<const float4*>(pieces + ((size_t)k * 16 + row) * N + col0);
      const float4 a = p[0], b = p[1];
      const float v[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
      for (int i = 0; i < 8; ++i) out[i] = k == 0 ? v[i] : out[i] + v[i];
    }
  }
}

template <class T>
__device__ __forceinline__ void load8(const T* p, float (&v)[8]) {
  const float4 a = reinterpret_cast<const float4*>(p)[0];
  const float4 c = reinterpret_cast<const float4*>(p)[1];
  v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
  v[4] = c.x; v[5] = c.y; v[6] = c.z; v[7] = c.w;
}

// ---- plain quantisation of x[M][K]: grid (ceil(nb/8), 16), 8 warps, warp = block
__global__ void quantize_kernel(const float* __restrict__ x, int M, int K, uint8_t* act,
                                int8_t* q_dbg, float* da_dbg, int32_t* A_dbg, int32_t* status) {
  pdl_trigger();
  pdl_wait();
  const int nb = K / 256;
  const int b = blockIdx.x * 8 + (threadIdx.x >> 5);
  const int row = blockIdx.y;
  if (b >= nb) return;
  if (row >= M) {
    zero_block_warp(row, b, act);
    return;
  }
  float v[8];
  load8(x + (size_t)row * K + 256 * b + 8 * (threadIdx.x & 31), v);
  quant_block_warp(v, row, b, K, act, q_dbg, da_dbg, A_dbg, status);
}

static cudaLaunchConfig_t make_cfg(dim3 grid, dim3 block, size_t smem, cudaStream_t st, bool pdl,
                                   cudaLaunchAttribute* attrs, int cluster_x = 0) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  int n = 0;
  if (pdl) {
    attrs[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attrs[n].val.programmaticStreamSerializationAllowed = 1;
    ++n;
  }
  if (cluster_x > 0) {
    attrs[n].id = cudaLaunchAttributeClusterDimension;
    attrs[n].val.clusterDim.x = cluster_x;
    attrs[n].val.clusterDim.y = 1;
    attrs[n].val.clusterDim.z = 1;
    ++n;
  }
  cfg.attrs = attrs;
  cfg.numAttrs = n;
  return cfg;
}

cudaError_t launch_quantize(const float* x, int M, int K, uint8_t* act, int8_t* q_dbg,
                            float* da_dbg, int32_t* A_dbg, int32_t* status, cudaStream_t st,
                            bool pdl) {
  const int nb = K / 256;
  cudaLaunchAttribute attrs[2];
  cudaLaunchConfig_t cfg = make_cfg(dim3((nb + 7) / 8, 16), dim3(256), 0, st, pdl, attrs);
  return cudaLaunchKernelEx(&cfg, quantize_kernel, x, M, K, act, q_dbg, da_dbg, A_dbg, status);
}

// ---------------------------------------------------------------------------
// residual + RMSNorm + quantisation.  A cluster of kNormSplit CTAs per row
// (16 rows: rows >= M write zero activation blocks); warp w of cluster rank c
// owns the 256-blocks b = c + kNormSplit*w and b = c + kNormSplit*(w + warps)
// (H/256 <= 64).  The row's sum of squares is reduced lane -> warp
// (butterfly, the warp's blocks in order); every warp sum is pushed into the
// shared memory of every CTA of the cluster, and after one cluster barrier
// each warp adds the kNormSplit*warps sums in a butterfly: one fixed order set
// by H alone.  x_out = x_in + sum(pieces) (fp32 add) when pieces are given;
// cap (optional) receives the same rows with row stride cap_ld.
// ---------------------------------------------------------------------------
constexpr int kNormSplit = 4;

__global__ void __launch_bounds__(1024)
resid_norm_quant_kernel(const float* __restrict__ pieces, int pN, int pnb, long long pU, int pG,
                        const float* x_in, float* x_out,
                        const float* __restrict__ gamma, float eps, int M, int H, uint8_t* act,
                        float* __restrict__ xnorm_out, float* __restrict__ cap, int cap_ld,
                        int32_t* status) {
  __shared__ float part_ss[64];
  const int row = blockIdx.y;
  const int c = kNormSplit > 1 ? (int)cluster_rank() : 0;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;
  const int nb = H / 256;
  // gamma does not depend on the previous kernel: fetch it before waiting
  float gm[2][8];
#pragma unroll
  for (int t = 0; t < 2; ++t) {
    const int b = c + kNormSplit * (warp + t * nw);
    if (gamma && b < nb) {
      load8(gamma + 256 * b + 8 * lane, gm[t]);
    } else {
#pragma unroll
      for (int i = 0; i < 8; ++i) gm[t][i] = 1.f;
    }
  }
  pdl_trigger();
  pdl_wait();
  float v[2][8];
  float ss = 0.f;
#pragma unroll
  for (int t = 0; t < 2; ++t) {
    const int b = c + kNormSplit * (warp + t * nw);
    if (row < M && b < nb) {
      const int col0 = 256 * b + 8 * lane;
      load8(x_in + (size_t)row * H + col0, v[t]);
      if (pieces) {
        float ps[8];
        piece_sum8(pieces, pN, piece_slots(pnb, (int)pU, pG, col0), row, col0, ps);
#pragma unroll
        for (int i = 0; i < 8; ++i) v[t][i] = v[t][i] + ps[i];
      }
#pragma unroll
      for (int i = 0; i < 8; ++i) ss += v[t][i] * v[t][i];
    }
  }
  ss = warp_sum(ss);
  // warp sum -> slot c*nw + warp of every CTA of the cluster
  if (lane < kNormSplit) {
    if (kNormSplit > 1) {
      st_cluster_f32(&part_ss[c * nw + warp], (uint32_t)lane, ss);
    } else {
      part_ss[warp] = ss;
    }
  }
  // the residual stores go out while the partial sums travel
#pragma unroll
  for (int t = 0; t < 2; ++t) {
    const int b = c + kNormSplit * (warp + t * nw);
    if (row < M && b < nb && x_out && (pieces || x_out != x_in)) {
      float4* o = reinterpret_cast<float4*>(x_out + (size_t)row * H + 256 * b + 8 * lane);
      o[0] = make_float4(v[t][0], v[t][1], v[t][2], v[t][3]);
      o[1] = make_float4(v[t][4], v[t][5], v[t][6], v[t][7]);
    }
    if (row < M && b < nb && cap) {           // hidden-state capture (row stride cap_ld)
      float4* o = reinterpret_cast<float4*>(cap + (size_t)row * cap_ld + 256 * b + 8 * lane);
      o[0] = make_float4(v[t][0], v[t][1], v[t][2], v[t][3]);
      o[1] = make_float4(v[t][4], v[t][5], v[t][6], v[t][7]);
    }
  }
  if (kNormSplit > 1) {
    cluster_sync_all();
  } else {
    __syncthreads();
  }
  const int np = kNormSplit * nw;
  const float total = warp_sum((lane < np ? part_ss[lane] : 0.f) + (lane + 32 < np ? part_ss[lane + 32] : 0.f));
  const float rinv = 1.0f / sqrtf(total / (float)H + eps);
#pragma unroll
  for (int t = 0; t < 2; ++t) {
    const int b = c + kNormSplit * (warp + t * nw);
    if (b >= nb) continue;
    if (row < M) {
      const int col0 = 256 * b + 8 * lane;
#pragma unroll
      for (int i = 0; i < 8; ++i) v[t][i] = v[t][i] * rinv * gm[t][i];
      if (xnorm_out) {
        float4* o = reinterpret_cast<float4*>(xnorm_out + (size_t)row * H + col0);
        o[0] = make_float4(v[t][0], v[t][1], v[t][2], v[t][3]);
        o[1] = make_float4(v[t][4], v[t][5], v[t][6], v[t][7]);
      }
      quant_block_warp(v[t], row, b, H, act, nullptr, nullptr, nullptr, status);
    } else {
      zero_block_warp(row, b, act);
    }
  }
}

cudaError_t launch_resid_norm_quant(const GemmPlan* p, const float* pieces, const float* x_in,
                                    float* x_out, const float* gamma, float eps, int M, int H,
                                    uint8_t* act, float* xnorm_out, int32_t* status,
                                    cudaStream_t st, bool pdl, float* cap, int cap_ld) {
  const int nb = H / 256;
  const int per = (nb + kNormSplit - 1) / kNormSplit;       // blocks per CTA
  const int warps = per < 32 ? per : 32;
  if (per > 2 * warps || kNormSplit * warps > 64) return cudaErrorInvalidValue;
  cudaLaunchAttribute attrs[2];
  cudaLaunchConfig_t cfg = make_cfg(dim3(kNormSplit, 16), dim3(32 * warps), 0, st, pdl, attrs,
                                    kNormSplit > 1 ? kNormSplit : 0);
  const int pN = p ? p->N : 0, pnb = p ? p->nb : 1, pG = p ? p->G : 1;
  const long long pU = p ? p->U : 1;
  return cudaLaunchKernelEx(&cfg, resid_norm_quant_kernel, pieces, pN, pnb, pU, pG, x_in, x_out,
                            gamma, eps, M, H, act, xnorm_out, cap, cap_ld, status);
}

// ---------------------------------------------------------------------------
// SwiGLU + quantisation: grid (ceil(nbF/8), 16), warp = one 256-block of h.
// h = silu(g) * u, silu(g) = g / (1 + exp(-g)), fp32.
// ---------------------------------------------------------------------------
__global__ void swiglu_quant_kernel(const float* __restrict__ pieces, int pN, int pnb, long long pU,
                                    int pG, int M, int F, uint8_t* act, int32_t* status) {
  pdl_trigger();
  pdl_wait();
  const int nb = F / 256;
  const int b = blockIdx.x * 8 + (threadIdx.x >> 5);
  const int row = blockIdx.y;
  if (b >= nb) return;
  if (row >= M) {
    zero_block_warp(row, b, act);
    return;
  }
  const int col0 = 256 * b + 8 * (threadIdx.x & 31);
  float gt[8], up[8], v[8];
  piece_sum8(pieces, pN, piece_slots(pnb, (int)pU, pG, col0), row, col0, gt);
  piece_sum8(pieces, pN, piece_slots(pnb, (int)pU, pG, F + col0), row, F + col0, up);
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const float sl = gt[i] / (1.0f + expf(-gt[i]));
    v[i] = sl * up[i];
  }
  quant_block_warp(v, row, b, F, act, nullptr, nullptr, nullptr, status);
}

cudaError_t launch_swiglu_quant(const GemmPlan& p, const float* pieces, int M, int F, uint8_t* act,
                                int32_t* status, cudaStream_t st, bool pdl) {
  const int nb = F / 256;
  cudaLaunchAttribute attrs[2];
  cudaLaunchConfig_t cfg = make_cfg(dim3((nb + 7) / 8, 16), dim3(256), 0, st, pdl, attrs);
  return cudaLaunchKernelEx(&cfg, swiglu_quant_kernel, pieces, p.N, p.nb, p.U, p.G, M, F, act,
                            status);
}

// ---------------------------------------------------------------------------
// QKV split: Q -> bf16 hi/lo attention fragments (rows >= M zero); K, V ->
// bf16 (round to nearest even) into the page of position n_past + row,
// n_past = seq_len - M (the reserve kernel has already appended the block).
// Skips the cache when the step is invalid.  With a QkTransform, each q and
// k head is first QK-normed and/or rotated (RoPE) at its row's position.
// ---------------------------------------------------------------------------
constexpr int kQkvThreads = 256;     // columns per CTA; one more warp prefetches the KV

// QK-norm and RoPE of one head (Ch. 8 §8.2), computed by the 128 threads
// that hold its elements (thread d of the group holds element d): the group's
// sum of squares (warp shuffles, then the four warp sums in order), then
// y = x * g / sqrt(mean + eps), then the rotation of pair (i, i + 64) by the
// table's (cos, sin) of row pos, element i.  The groups of a CTA synchronise
// on their own named barriers (1 and 2), so a group whose columns lie past the
// end may leave early.
// named barrier of one 128-thread group (ids 1 and 2: immediates, so the
// kernel reserves two hardware barriers, not all sixteen)
__device__ __forceinline__ void group_bar(int grp) {
  if (grp == 0)
    asm volatile("bar.sync 1, 128;" ::: "memory");
  else
    asm volatile("bar.sync 2, 128;" ::: "memory");
}
__device__ __forceinline__ float head_norm_rope(float x, const float* g, const float2* cs, int d, float eps) {
  __shared__ float red[2][4];
  __shared__ float xch[2][128];
  const int grp = threadIdx.x >> 7, w = (threadIdx.x >> 5) & 3;
  if (g) {
    float s = x * x;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    if ((threadIdx.x & 31) == 0) red[grp][w] = s;
    group_bar(grp);
    const float ss = ((red[grp][0] + red[grp][1]) + red[grp][2]) + red[grp][3];
    x = x * (1.0f / sqrtf(ss / 128.0f + eps)) * g[d];
  }
  if (cs) {
    xch[grp][d] = x;
    group_bar(grp);
    const float other = xch[grp][d ^ 64];
    const float2 t = cs[d & 63];
    x = d < 64 ? x * t.x - other * t.y : x * t.x + other * t.y;
  }
  return x;
}

__global__ void qkv_post_kernel(const float* __restrict__ pieces, int pN, int pnb, long long pU,
                                int pG, int M, int nq, int nkv, int dh, KvView kv, int layer,
                                uint8_t* __restrict__ qtile, int tiles, const int32_t* status,
                                int late_trigger, QkTransform qk) {
  // With late_trigger the attention that follows reads the KV metadata before
  // its own wait: signalling it only after this wait means that every kernel
  // before this one has completed when it starts.
  if (!late_trigger) pdl_trigger();
  pdl_wait();
  if (late_trigger) pdl_trigger();
  // The attention that follows reads this layer's K and V of every page up to
  // the length: one 32 KB slab per page ([K, V][n_kv][16][128] bf16).  An
  // extra warp sends them to L2 now, while HBM has nothing else to do: lane l
  // of CTA c takes page c + l * (number of CTAs), spreading the copies over
  // the SMs' copy engines; its loads run alongside the other warps' loads.
  const int swa = swa_index(kv, layer);
  if (threadIdx.x >= kQkvThreads) {
    if (swa >= 0) return;                    // a ring layer reads no pages
    const int ncta = gridDim.x * gridDim.y;
    const int gi = blockIdx.y * gridDim.x + blockIdx.x + (threadIdx.x - kQkvThreads) * ncta;
    const int lp = gi < kv.max_seq_pages ? gi : kv.max_seq_pages - 1;
    const int page = kv.page_table[lp];
    const int npg = (*kv.seq_len + kv.page_size - 1) / kv.page_size;
    const uint32_t slab = (uint32_t)(2 * kv.n_kv * kv.page_size * kv.head_dim * 2);
    if (gi < npg && gi < kv.max_seq_pages && page >= 0 && page < kv.num_pages)
      asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;\n" ::"l"(
                       kv.pool + ((size_t)page * kv.n_layers + layer) * (slab / 2)),
                   "r"(slab)
                   : "memory");
    return;
  }
  const int row = blockIdx.y;
  const int col = blockIdx.x * kQkvThreads + threadIdx.x;
  const int qcols = nq * dh;
  if (col >= pN) return;
  if (row >= M) {
    if (col < qcols) write_qtile(qtile, row, col / dh, col % dh, 0.f, nq / nkv, tiles);
    return;
  }
  float v = piece_sum(pieces, pN, piece_slots(pnb, (int)pU, pG, col), row, col);
  const int pos = *kv.seq_len - M + row;
  if (col < qcols + nkv * dh) {
    // a q or k head: all 128 threads of this thread's group take this branch
    const float* g = col < qcols ? qk.gq : qk.gk;
    const float2* cs = nullptr;
    if (qk.cs) cs = qk.cs + (size_t)min(max(pos, 0), qk.cs_len - 1) * 64;
    if (g || cs) v = head_norm_rope(v, g, cs, col % dh, qk.eps);
  }
  if (col < qcols) {
    write_qtile(qtile, row, col / dh, col % dh, v, nq / nkv, tiles);
    return;
  }
  if (*status & kStepAbort) return;
  const int c = col - qcols;
  const int which = c / (nkv * dh);          // 0 = K, 1 = V
  const int head = (c % (nkv * dh)) / dh, d = c % dh;
  if (swa >= 0) {
    // the ring slot pos mod R: it held position pos - R, which no window of
    // this block or a later one sees
    if (pos >= 0)
      kv.swa_ring[ring_row(kv, swa, which, head, pos % kv.swa_rows) + d] =
          __bfloat16_as_ushort(__float2bfloat16_rn(v));
    return;
  }
  const int lp = pos / kv.page_size;
  if (pos < 0 || lp >= kv.max_seq_pages) return;
  const int page = kv.page_table[lp];
  if (page < 0 || page >= kv.num_pages) return;
  const size_t off = ((((size_t)page * kv.n_layers + layer) * 2 + which) * kv.n_kv + head) *
                         (size_t)kv.page_size * kv.head_dim +
                     (size_t)(pos % kv.page_size) * kv.head_dim + d;
  kv.pool[off] = __bfloat16_as_ushort(__float2bfloat16_rn(v));
}

cudaError_t launch_qkv_post(const GemmPlan& p, const float* pieces, int M, int nq, int nkv, int dh,
                            const KvView& kv, int layer, uint8_t* qtile, int tiles,
                            const int32_t* status, cudaStream_t st, bool pdl, bool late_trigger,
                            const QkTransform& qk) {
  // the per-head transforms assume 128-element heads, two per CTA
  if ((qk.gq || qk.gk || qk.cs) && (dh != 128 || (qk.cs && qk.cs_len < 1))) return cudaErrorInvalidValue;
  cudaLaunchAttribute attrs[2];
  cudaLaunchConfig_t cfg = make_cfg(dim3((p.N + kQkvThreads - 1) / kQkvThreads, 16), dim3(kQkvThreads + 32), 0,
                                    st, pdl, attrs);
  return cudaLaunchKernelEx(&cfg, qkv_post_kernel, pieces, p.N, p.nb, p.U, p.G, M, nq, nkv, dh, kv,
                            layer, qtile, tiles, status, (int)late_trigger, qk);
}

// ---------------------------------------------------------------------------
// LM head argmax: CTA c scans columns [c*kArgCols, (c+1)*kArgCols) of every
// row: logit = sum of the head GEMM pieces; keeps (max, lowest index).
// ---------------------------------------------------------------------------
constexpr int kArgCols = 512;

int head_argmax_blocks(int V) { return (V + kArgCols - 1) / kArgCols; }

__device__ __forceinline__ void better(float& bv, int& bi, float v, int i) {
  // larger value wins; equal values: lower index wins
  if (v > bv || (v == bv && i < bi)) {
    bv = v;
    bi = i;
  }
}

// CTA c scans columns [c*kArgCols, (c+1)*kArgCols) of every row; thread t
// owns columns t + 256k (k < kArgCols/256) of every row, all rows loaded in
// one round; per-row (max, lowest index) reduced
// warp -> CTA in a fixed order.
__global__ void __launch_bounds__(256)
head_argmax_kernel(const float* __restrict__ pieces, int pN, int pnb, long long pU, int pG, int M,
                   float* __restrict__ logits, float* __restrict__ part_val,
                   int32_t* __restrict__ part_idx, int32_t* status) {
  pdl_trigger();
  pdl_wait();
  __shared__ float sv[16][8];
  __shared__ int si[16][8];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int col_base = blockIdx.x * kArgCols;
  int nsl[kArgCols / 256];
#pragma unroll
  for (int k = 0; k < kArgCols / 256; ++k) {
    const int col = col_base + threadIdx.x + 256 * k;
    nsl[k] = col < pN ? piece_slots(pnb, (int)pU, pG, col) : 1;
  }
  // the logits of both columns for every row: slot 0 of all rows in one
  // round of loads, then the further slots, each added in slot order
  constexpr int kC = kArgCols / 256;
  float lv[kC][16];
#pragma unroll
  for (int k = 0; k < kC; ++k) {
    const int col = col_base + threadIdx.x + 256 * k;
#pragma unroll
    for (int row = 0; row < 16; ++row)
      lv[k][row] = (col < pN && row < M) ? pieces[(size_t)row * pN + col] : 0.f;
  }
  int nsmax = 1;
#pragma unroll
  for (int k = 0; k < kC; ++k) nsmax = max(nsmax, nsl[k]);
  for (int sl = 1; sl < nsmax; ++sl) {
#pragma unroll
    for (int k = 0; k < kC; ++k) {
      const int col = col_base + threadIdx.x + 256 * k;
      if (col < pN && sl < nsl[k]) {
#pragma unroll
        for (int row = 0; row < 16; ++row)
          if (row < M) lv[k][row] += pieces[((size_t)sl * 16 + row) * pN + col];
      }
    }
  }
  bool bad = false;
#pragma unroll
  for (int row = 0; row < 16; ++row) {
    float bv = -INFINITY;
    int bi = 0x7fffffff;
    if (row < M) {
#pragma unroll
      for (int k = 0; k < kC; ++k) {
        const int col = col_base + threadIdx.x + 256 * k;
        if (col < pN) {
          const float v = lv[k][row];
          if (logits) logits[(size_t)row * pN + col] = v;
          if (!isfinite(v)) bad = true;
          better(bv, bi, v, col);
        }
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
      const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
      better(bv, bi, ov, oi);
    }
    if (lane == 0) {
      sv[row][warp] = bv;
      si[row][warp] = bi;
    }
  }
  if (bad) atomicOr(status, SPEC_ST_NONFINITE);
  __syncthreads();
  if (threadIdx.x < 16) {
    const int row = threadIdx.x;
    float v = sv[row][0];
    int i = si[row][0];
    for (int w = 1; w < 8; ++w) better(v, i, sv[row][w], si[row][w]);
    part_val[(size_t)blockIdx.x * 16 + row] = v;
    part_idx[(size_t)blockIdx.x * 16 + row] = i;
  }
}

cudaError_t launch_head_argmax(const GemmPlan& p, const float* pieces, int M, float* logits,
                               float* part_val, int32_t* part_idx, int32_t* status, cudaStream_t st,
                               bool pdl) {
  cudaLaunchAttribute attrs[2];
  cudaLaunchConfig_t cfg = make_cfg(dim3(head_argmax_blocks(p.N)), dim3(256), 0, st, pdl, attrs);
  return cudaLaunchKernelEx(&cfg, head_argmax_kernel, pieces, p.N, p.nb, p.U, p.G, M, logits,
                            part_val, part_idx, status);
}

// final reduction of the per-CTA partials: idx[row], lowest index on ties
__global__ void argmax_final_kernel(const float* __restrict__ part_val,
                                    const int32_t* __restrict__ part_idx, int nparts, int M,
                                    int32_t* __restrict__ idx) {
  pdl_trigger();
  pdl_wait();
  const int row = threadIdx.x >> 5, lane = threadIdx.x & 31;   // one warp per row
  if (row >= M) return;
  float bv = -INFINITY;
  int bi = 0x7fffffff;
  for (int c = lane; c < nparts; c += 32)
    better(bv, bi, part_val[(size_t)c * 16 + row], part_idx[(size_t)c * 16 + row]);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
    const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
    better(bv, bi, ov, oi);
  }
  if (lane == 0) idx[row] = bi;
}

cudaError_t launch_argmax_final(const float* part_val, const int32_t* part_idx, int nparts, int M,
                                int32_t* idx, cudaStream_t st, bool pdl) {
  cudaLaunchAttribute attrs[2];
  cudaLaunchConfig_t cfg = make_cfg(dim3(1), dim3(32 * 16), 0, st, pdl, attrs);
  return cudaLaunchKernelEx(&cfg, argmax_final_kernel, part_val, part_idx, nparts, M, idx);
}

// ---------------------------------------------------------------------------
// KV metadata (Ch. 8 §8.6 item 4).  The reserve scans the page table with a
// warp; a rollback touches at most ceil(16/16)+1 pages and runs on one thread.
// ---------------------------------------------------------------------------
__global__ void kv_reset_kernel(KvView kv) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < kv.max_seq_pages) kv.page_table[i] = -1;
  if (i < kv.num_pages) kv.free_stack[i] = kv.num_pages - 1 - i;
  if (i == 0) {
    *kv.free_top = kv.num_pages;
    *kv.seq_len = 0;
    if (kv.swa_state) {
      kv.swa_state[0] = -1;                  // no block to roll back into
      kv.swa_state[1] = 0;
    }
  }
}

cudaError_t launch_kv_reset(const KvView& kv, cudaStream_t st) {
  const int n = kv.max_seq_pages > kv.num_pages ? kv.max_seq_pages : kv.num_pages;
  kv_reset_kernel<<<(n + 255) / 256, 256, 0, st>>>(kv);
  return cudaGetLastError();
}

// step_state: [0] = n_past, [1] = 1 when the block was appended
__global__ void kv_reserve_kernel(KvView kv, int n, int commit, const int32_t* __restrict__ draft,
                                  int k, int vocab, int32_t* status, int32_t* step_state,
                                  const int32_t* __restrict__ parent, uint64_t* tree_mask) {
  pdl_trigger();
  pdl_wait();
  if (blockIdx.x != 0) return;
  const int lane = threadIdx.x;              // one warp
  const int len = *kv.seq_len;
  int st = 0;
  if (lane == 0) {
    if (step_state) {
      step_state[0] = len;
      step_state[1] = 0;
    }
    if (parent) {
      // a token tree of n <= 64 nodes: parent[0] = -1, 0 <= parent[i] < i;
      // the mask of node i = its ancestors and itself (Ch. 33 §33.7), built
      // in place (a parent's mask is final before its children's)
      if (n < 1 || n > kTreeMax || parent[0] != -1) st |= SPEC_ST_BAD_TREE;
      for (int i = 1; i < n && !st; ++i)
        if (parent[i] < 0 || parent[i] >= i) st |= SPEC_ST_BAD_TREE;
      if (!st) {
        tree_mask[0] = 1ull;
        for (int i = 1; i < n; ++i) tree_mask[i] = tree_mask[parent[i]] | (1ull << i);
      }
    }
    if (draft) {
      for (int i = 0; i < k; ++i)
        if (draft[i] < 0 || draft[i] >= vocab) st |= SPEC_ST_TOKEN_RANGE;
    }
  }
  st = __shfl_sync(0xffffffffu, st, 0);
  const int upto = len + n;
  const int pages = (upto + kv.page_size - 1) / kv.page_size;
  // beyond the page table, or beyond the positions the context was sized for
  // (the attention's chunk plan and the rotary table end at max_ctx)
  if (!st && (pages > kv.max_seq_pages || (kv.max_ctx > 0 && upto > kv.max_ctx))) st |= SPEC_ST_CTX_FULL;
  // the unmapped pages below `pages`, counted by the warp; the r-th of them in
  // page order gets free_stack[top - 1 - r] (the pops of a serial walk)
  int need = 0;
  if (!st)
    for (int base = 0; base < pages; base += 32) {
      const int p = base + lane;
      need += __popc(__ballot_sync(0xffffffffu, p < pages && kv.page_table[p] < 0));
    }
  const int top = *kv.free_top;
  if (!st && need > top) st |= SPEC_ST_POOL_EMPTY;
  if (!st) {
    int before = 0;
    for (int base = 0; base < pages; base += 32) {
      const int p = base + lane;
      const bool hole = p < pages && kv.page_table[p] < 0;
      const uint32_t holes = __ballot_sync(0xffffffffu, hole);
      if (hole) kv.page_table[p] = kv.free_stack[top - 1 - before - __popc(holes & ((1u << lane) - 1u))];
      before += __popc(holes);
    }
    if (lane == 0) {
      *kv.free_top = top - need;
      if (commit || step_state) *kv.seq_len = upto;
      if (step_state) step_state[1] = 1;
      if (kv.swa_state) {
        // a step's block: rollbacks down to its first position are served by
        // the rings' spare slots.  Rows laid down by an extend are not a
        // speculative block: no rollback below the new length.
        kv.swa_state[0] = step_state ? len : (commit ? -1 : kv.swa_state[0]);
        if (step_state) kv.swa_state[1] = n;
      }
    }
  }
  if (lane != 0) return;
  if (step_state) {
    *status = st;           // first kernel of a step: resets the step status
  } else if (st) {
    atomicOr(status, st);
  }
}

cudaError_t launch_kv_reserve(const KvView& kv, int n, int commit, const int32_t* draft, int k,
                              int vocab, int32_t* status, int32_t* step_state, cudaStream_t st,
                              bool pdl, const int32_t* parent, uint64_t* tree_mask) {
  cudaLaunchAttribute attrs[2];
  cudaLaunchConfig_t cfg = make_cfg(dim3(1), dim3(32), 0, st, pdl, attrs);
  return cudaLaunchKernelEx(&cfg, kv_reserve_kernel, kv, n, commit, draft, k, vocab, status,
                            step_state, parent, tree_mask);
}

__global__ void kv_rollback_kernel(KvView kv, int new_len, int32_t* status) {
  if (threadIdx.x != 0 || blockIdx.x != 0) return;
  const int len = *kv.seq_len;
  bool bad = new_len < 0 || new_len > len;
  // a sliding-window ring can be wound back only over the rows its spare
  // slots keep: to lengths at or above the last step's n_past
  if (swa_layers(kv) > 0 && new_len < len && (kv.swa_state[0] < 0 || new_len < kv.swa_state[0])) bad = true;
  if (bad) {
    atomicOr(status, SPEC_ST_ROLLBACK);
    return;
  }
  kv_rollback_dev(kv, new_len);
}

cudaError_t launch_kv_rollback(const KvView& kv, int new_len, int32_t* status, cudaStream_t st) {
  kv_rollback_kernel<<<1, 32, 0, st>>>(kv, new_len, status);
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// Accept + rollback: final argmax reduction over the head partials (or the
// given idx), L = first i < k with draft[i] != idx[i] (else k), next = idx[L];
// seq_len := n_past + L + 1 and the pages past it are freed.  On any device
// error the block is rolled back entirely (seq_len := n_past).
// res = {accepted_len, next_token, status, seq_len}.
// ---------------------------------------------------------------------------
__global__ void accept_kernel(const int32_t* __restrict__ idx_in, const float* __restrict__ part_val,
                              const int32_t* __restrict__ part_idx, int nparts,
                              const int32_t* __restrict__ draft, int k, int vocab, KvView kv,
                              int has_kv, const int32_t* step_state, int32_t* status, int32_t* res,
                              int32_t* idx_out) {
  pdl_trigger();
  pdl_wait();
  __shared__ int idx_s[16];
  const int row = threadIdx.x >> 5, lane = threadIdx.x & 31;   // one warp per row
  if (row <= k) {
    if (idx_in) {
      if (lane == 0) idx_s[row] = idx_in[row];
    } else {
      float bv = -INFINITY;
      int bi = 0x7fffffff;
      for (int c = lane; c < nparts; c += 32) better(bv, bi, part_val[(size_t)c * 16 + row], part_idx[(size_t)c * 16 + row]);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
        const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
        better(bv, bi, ov, oi);
      }
      if (lane == 0) idx_s[row] = bi;
    }
  }
  __syncthreads();
  if (threadIdx.x != 0) return;
  int st = step_state ? *status : 0;
  for (int i = 0; i < k; ++i)
    if (draft[i] < 0 || draft[i] >= vocab) st |= SPEC_ST_TOKEN_RANGE;
  for (int row = 0; row <= k; ++row) {
    if (idx_s[row] < 0 || idx_s[row] >= vocab) st |= SPEC_ST_NONFINITE;
    if (idx_out) idx_out[row] = idx_s[row];
  }
  int L = k;
  for (int i = 0; i < k; ++i)
    if (draft[i] != idx_s[i]) {
      L = i;
      break;
    }
  int next = idx_s[L];
  const bool appended = step_state ? step_state[1] != 0 : has_kv != 0;
  const int n_past = step_state ? step_state[0] : (has_kv ? *kv.seq_len - (k + 1) : 0);
  if (st) {
    L = 0;
    next = -1;
    if (has_kv && appended) kv_rollback_dev(kv, n_past);
  } else if (has_kv && appended) {
    kv_rollback_dev(kv, n_past + L + 1);
  }
  *status = st;
  res[0] = L;
  res[1] = next;
  res[2] = st;
  res[3] = has_kv ? *kv.seq_len : 0;
}

cudaError_t launch_accept(const int32_t* idx, const float* part_val, const int32_t* part_idx,
                          int nparts, const int32_t* draft, int k, int vocab, const KvView* kv,
                          const int32_t* step_state, int32_t* status, int32_t* res,
                          int32_t* idx_out, cudaStream_t st, bool pdl) {
  cudaLaunchAttribute attrs[2];
  cudaLaunchConfig_t cfg = make_cfg(dim3(1), dim3(32 * 16), 0, st, pdl, attrs);
  KvView v = kv ? *kv : KvView{};
  return cudaLaunchKernelEx(&cfg, accept_kernel, idx, part_val, part_idx, nparts, draft, k, vocab, v,
                            kv ? 1 : 0, step_state, status, res, idx_out);
}

}  // namespace spec
