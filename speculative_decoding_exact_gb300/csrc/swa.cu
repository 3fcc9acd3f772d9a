// swa.cu — sliding-window layers: a ring of W K/V rows per layer and the
// checkpoint of the rows a verify block overwrites.
//
// Muser book Ch. 8 ("The DFlash draft") §8.6 item 4: a speculation round may
// fail and roll back, so the target's KV planes checkpoint before the block;
// the NoPE planes (the paged cache) rewind their metadata only, while the
// sliding-window rings keep the at most 16 rows a block may overwrite.
//
// A sliding-window layer of window W stores position t in slot t mod W of its
// ring, so its storage does not grow with the context; its row at position p
// sees positions p-W+1..p.  A block of M <= 16 rows at positions n..n+M-1
// overwrites the slots of positions n-W..n+M-1-W.  Those rows are still
// inside the windows of the block's own earlier rows and, after a rollback,
// of the rows that follow.  So:
//   * before the block is written, the checkpoint kernel copies the M slots it
//     will overwrite (the checkpoint: [layer][K,V][kv head][16][128] bf16,
//     and its position n and row count M in swa_state);
//   * the attention reads key t from the ring, except an old position that a
//     block row overwrote (n-W <= t <= n+M-1-W), which it reads from the
//     checkpoint;
//   * every rollback to a length len >= n writes the checkpoint rows
//     len-n..M-1 back into their slots; a rollback below n cannot be served
//     (the rows it would need are gone) and is refused.
//
// The attention is a CUDA-core kernel in fp32: CTA (query head, split of 128
// keys) stages 32-key tiles of K (transposed) and V as fp32 in shared memory,
// keeps an online (max, sum) per row, and writes partials [split][head][row]
// [o 128 | max | sum | pad 2]; a merge kernel combines the splits in split order,
// normalises and quantises the rows for the output projection.  The splits
// are fixed by the window and the block position alone, so row i's result is
// the same for every M.
#include "common.cuh"
#include "internal.h"
#include "quant.cuh"

namespace spec {

constexpr int kSwaTile = 32;              // keys per staged tile
constexpr int kSwaSplit = 128;            // keys per CTA
constexpr int kSwaThreads = 128;
constexpr int kSwaStride = 132;           // floats per partial row: o[128], max, sum, 2 pad (16-byte rows)
constexpr int kKtPad = 36;                // K^T row length in floats (16-byte aligned)

int swa_splits(int window) { return (window + 15 + kSwaSplit - 1) / kSwaSplit; }
size_t swa_partial_floats(int window, int nq) {
  return window > 0 ? (size_t)swa_splits(window) * nq * 16 * kSwaStride : 0;
}

// ---- checkpoint: grid (n_swa * 2 * n_kv), 256 threads; thread t copies the
// 16-byte chunk t % 16 of row t / 16.  Nothing is saved when the step was
// aborted before its reservation (nothing will be written either).
__global__ void swa_checkpoint_kernel(KvView kv, int M, const int32_t* step_state, const int32_t* status) {
  pdl_trigger();
  pdl_wait();
  if (*status & kStepAbort) return;
  const int n = step_state[0];
  const int b = blockIdx.x;
  const int s = b / (2 * kv.n_kv), which = (b / kv.n_kv) % 2, head = b % kv.n_kv;
  const int j = threadIdx.x >> 4, c = threadIdx.x & 15;
  if (j < M) {
    const int slot = (n + j) % kv.swa_window;
    const uint4 v = *reinterpret_cast<const uint4*>(kv.swa_ring + ring_row(kv, s, which, head, slot) + 8 * c);
    *reinterpret_cast<uint4*>(kv.swa_ckpt + ckpt_row(kv, s, which, head, j) + 8 * c) = v;
  }
  if (b == 0 && threadIdx.x == 0) {
    kv.swa_state[0] = n;
    kv.swa_state[1] = M;
  }
}

// ---- restore after a rollback (the step's accept, or spec_kv_rollback): the
// checkpoint rows j >= seq_len - n go back into their slots.  Same grid.
__global__ void swa_restore_kernel(KvView kv) {
  pdl_trigger();
  pdl_wait();
  const int n = kv.swa_state[0], m = kv.swa_state[1];
  if (n < 0) return;
  const int len = *kv.seq_len;
  const int b = blockIdx.x;
  const int s = b / (2 * kv.n_kv), which = (b / kv.n_kv) % 2, head = b % kv.n_kv;
  const int j = threadIdx.x >> 4, c = threadIdx.x & 15;
  if (j < m && n + j >= len) {
    const int slot = (n + j) % kv.swa_window;
    const uint4 v = *reinterpret_cast<const uint4*>(kv.swa_ckpt + ckpt_row(kv, s, which, head, j) + 8 * c);
    *reinterpret_cast<uint4*>(kv.swa_ring + ring_row(kv, s, which, head, slot) + 8 * c) = v;
  }
}

// K or V row of position t for the current block (n, M): the checkpoint row
// when a block row overwrote t's slot, the ring row otherwise
SPEC_DEV const uint16_t* swa_key_row(const KvView& kv, int s, int which, int head, int t, int n, int M) {
  const int j = t + kv.swa_window - n;      // the block row that shares t's slot, if t < n
  if (t < n && j >= 0 && j < M) return kv.swa_ckpt + ckpt_row(kv, s, which, head, j);
  return kv.swa_ring + ring_row(kv, s, which, head, t % kv.swa_window);
}

// ---- partials: grid (splits, nq), kSwaThreads threads.  Split sp takes the
// keys [lo + 128 sp, lo + 128 (sp + 1)) with lo = max(0, n - W + 1), the
// first position any block row sees.  Thread t: row r = t / 8, keys
// 4 (t % 8) .. +3 of a tile for the scores, dims 16 (t % 8) .. +15 for o.
__global__ void __launch_bounds__(kSwaThreads)
swa_partial_kernel(const float* __restrict__ q32, int M, int nq, KvView kv, int s, float* __restrict__ part,
                   const int32_t* status) {
  pdl_trigger();
  pdl_wait();
  __shared__ __align__(16) float q_s[16][128];
  __shared__ __align__(16) float kt_s[128][kKtPad];     // K^T of the tile
  __shared__ __align__(16) float v_s[kSwaTile][128];
  __shared__ __align__(16) float p_s[16][kSwaTile];
  const int sp = blockIdx.x, h = blockIdx.y, tid = threadIdx.x;
  const int group = nq / kv.n_kv, g = h / group;
  const int W = kv.swa_window, dh = kv.head_dim;
  const int r = tid >> 3, kq = tid & 7;
  const bool abort = (*status & kStepAbort) != 0;
  const int n = *kv.seq_len - M;
  const int lo = max(0, n - W + 1);
  const int k0 = lo + kSwaSplit * sp;
  const int k1 = min(k0 + kSwaSplit, n + M);       // keys past the block are nobody's
  // the row's window: [max(0, n + r - W + 1), n + r]
  const int rlo = max(0, n + r - W + 1), rhi = n + r;
  for (int i = tid; i < 16 * 128; i += kSwaThreads) {
    const int rr = i >> 7, d = i & 127;
    q_s[rr][d] = (rr < M && !abort) ? q32[(size_t)rr * nq * dh + (size_t)h * dh + d] : 0.f;
  }
  float m = -INFINITY, l = 0.f;
  float o[16];
#pragma unroll
  for (int e = 0; e < 16; ++e) o[e] = 0.f;
  const float scale = 0.08838834764831845f;        // 1 / sqrt(128)
  for (int t0 = k0; t0 < k1 && !abort; t0 += kSwaTile) {
    __syncthreads();                               // the previous tile is consumed
    // stage K^T and V as fp32: thread t loads key t / 4, dims 32 (t % 4) .. +31
    {
      const int key = tid >> 2, d0 = 32 * (tid & 3), t = t0 + key;
      const bool live = t < k1;
      const uint16_t* kr = live ? swa_key_row(kv, s, 0, g, t, n, M) : nullptr;
      const uint16_t* vr = live ? swa_key_row(kv, s, 1, g, t, n, M) : nullptr;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint4 kw = make_uint4(0, 0, 0, 0), vw = make_uint4(0, 0, 0, 0);
        if (live) {
          kw = *reinterpret_cast<const uint4*>(kr + d0 + 8 * c);
          vw = *reinterpret_cast<const uint4*>(vr + d0 + 8 * c);
        }
        const uint32_t kk[4] = {kw.x, kw.y, kw.z, kw.w}, vv[4] = {vw.x, vw.y, vw.z, vw.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int d = d0 + 8 * c + 2 * e;
          kt_s[d][key] = __uint_as_float(kk[e] << 16);
          kt_s[d + 1][key] = __uint_as_float(kk[e] & 0xffff0000u);
          v_s[key][d] = __uint_as_float(vv[e] << 16);
          v_s[key][d + 1] = __uint_as_float(vv[e] & 0xffff0000u);
        }
      }
    }
    __syncthreads();
    // scores of row r against keys 4kq .. 4kq+3
    float sc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 8
    for (int d = 0; d < 128; d += 4) {
      const float4 qv = *reinterpret_cast<const float4*>(&q_s[r][d]);
      const float qa[4] = {qv.x, qv.y, qv.z, qv.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float4 kv4 = *reinterpret_cast<const float4*>(&kt_s[d + e][4 * kq]);
        sc[0] = fmaf(qa[e], kv4.x, sc[0]);
        sc[1] = fmaf(qa[e], kv4.y, sc[1]);
        sc[2] = fmaf(qa[e], kv4.z, sc[2]);
        sc[3] = fmaf(qa[e], kv4.w, sc[3]);
      }
    }
    float tmax = -INFINITY;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int t = t0 + 4 * kq + e;
      sc[e] = (t >= rlo && t <= rhi && t < k1) ? sc[e] * scale : -INFINITY;
      tmax = fmaxf(tmax, sc[e]);
    }
    // the row's 8 threads are 8 consecutive lanes
#pragma unroll
    for (int off = 1; off < 8; off <<= 1) tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, off));
    const float mn = fmaxf(m, tmax);
    const float alpha = (m == -INFINITY) ? 0.f : expf(m - mn);
    float psum = 0.f;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float p = (sc[e] == -INFINITY) ? 0.f : expf(sc[e] - mn);
      p_s[r][4 * kq + e] = p;
      psum += p;
    }
#pragma unroll
    for (int off = 1; off < 8; off <<= 1) psum += __shfl_xor_sync(0xffffffffu, psum, off);
    if (mn != -INFINITY) {
      l = l * alpha + psum;
#pragma unroll
      for (int e = 0; e < 16; ++e) o[e] *= alpha;
      m = mn;
    }
    __syncwarp();
    // o[r][16 kq .. +15] += sum_j p[r][j] v[j]
#pragma unroll 4
    for (int j = 0; j < kSwaTile; ++j) {
      const float p = p_s[r][j];
      const float4* vp = reinterpret_cast<const float4*>(&v_s[j][16 * kq]);
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const float4 v4 = vp[c];
        o[4 * c] = fmaf(p, v4.x, o[4 * c]);
        o[4 * c + 1] = fmaf(p, v4.y, o[4 * c + 1]);
        o[4 * c + 2] = fmaf(p, v4.z, o[4 * c + 2]);
        o[4 * c + 3] = fmaf(p, v4.w, o[4 * c + 3]);
      }
    }
  }
  float* dst = part + (((size_t)sp * nq + h) * 16 + r) * kSwaStride;
#pragma unroll
  for (int c = 0; c < 4; ++c)
    *reinterpret_cast<float4*>(dst + 16 * kq + 4 * c) = make_float4(o[4 * c], o[4 * c + 1], o[4 * c + 2], o[4 * c + 3]);
  if (kq == 0) {
    dst[128] = m;
    dst[129] = l;
  }
}

// ---- merge: grid (nq * 128 / 256, 16 rows), 256 threads = 2 heads x 128
// dims.  The splits are combined in split order: M = max m_s, w_s =
// exp(m_s - M), out = sum_s w_s o_s / sum_s w_s l_s; then the 256-block of the
// row is quantised for the output projection.
__global__ void __launch_bounds__(256)
swa_merge_kernel(const float* __restrict__ part, int M, int nq, int splits, const int32_t* seq_len,
                 float* __restrict__ out, uint8_t* act, int32_t* status) {
  pdl_trigger();
  pdl_wait();
  __shared__ float vals[256];
  const int b = blockIdx.x, row = blockIdx.y;
  const int hh = threadIdx.x >> 7, d = threadIdx.x & 127, h = 2 * b + hh;
  const bool valid = row < M && !(*status & kStepAbort);
  float res = 0.f;
  if (valid) {
    float mx = -INFINITY;
    for (int sp = 0; sp < splits; ++sp) mx = fmaxf(mx, part[(((size_t)sp * nq + h) * 16 + row) * kSwaStride + 128]);
    float L = 0.f, o = 0.f;
    for (int sp = 0; sp < splits; ++sp) {
      const float* pp = part + (((size_t)sp * nq + h) * 16 + row) * kSwaStride;
      const float ms = pp[128];
      const float w = (ms == -INFINITY) ? 0.f : expf(ms - mx);
      L += w * pp[129];
      o += w * pp[d];
    }
    res = o / L;
  }
  vals[threadIdx.x] = res;
  if (out && row < M) out[(size_t)row * nq * 128 + 256 * b + threadIdx.x] = res;
  __syncthreads();
  if (act && threadIdx.x < 32) {
    if (row < M) {
      float v[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) v[i] = vals[8 * threadIdx.x + i];
      quant_block_warp(v, row, b, nq * 128, act, nullptr, nullptr, nullptr, status);
    } else {
      zero_block_warp(row, b, act);
    }
  }
}

static cudaLaunchConfig_t swa_cfg(dim3 grid, dim3 block, cudaStream_t st, bool pdl, cudaLaunchAttribute* attr) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.stream = st;
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cfg;
}

cudaError_t launch_swa_checkpoint(const KvView& kv, int M, const int32_t* step_state, const int32_t* status,
                                  cudaStream_t st, bool pdl) {
  const int nb = swa_layers(kv) * 2 * kv.n_kv;
  if (nb == 0) return cudaSuccess;
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t cfg = swa_cfg(dim3(nb), dim3(256), st, pdl, attr);
  return cudaLaunchKernelEx(&cfg, swa_checkpoint_kernel, kv, M, step_state, status);
}

cudaError_t launch_swa_restore(const KvView& kv, cudaStream_t st, bool pdl) {
  const int nb = swa_layers(kv) * 2 * kv.n_kv;
  if (nb == 0) return cudaSuccess;
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t cfg = swa_cfg(dim3(nb), dim3(256), st, pdl, attr);
  return cudaLaunchKernelEx(&cfg, swa_restore_kernel, kv);
}

cudaError_t launch_swa_attention(const KvView& kv, int layer, const float* q32, int M, int nq, float* part,
                                 float* out, uint8_t* act, int32_t* status, cudaStream_t st, bool pdl) {
  const int s = swa_index(kv, layer);
  if (s < 0) return cudaErrorInvalidValue;
  const int splits = swa_splits(kv.swa_window);
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t cfg = swa_cfg(dim3(splits, nq), dim3(kSwaThreads), st, pdl, attr);
  cudaError_t e = cudaLaunchKernelEx(&cfg, swa_partial_kernel, q32, M, nq, kv, s, part, (const int32_t*)status);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg2 = swa_cfg(dim3(nq * 128 / 256, 16), dim3(256), st, pdl, attr);
  return cudaLaunchKernelEx(&cfg2, swa_merge_kernel, (const float*)part, M, nq, splits,
                            (const int32_t*)kv.seq_len, out, act, status);
}

}  // namespace spec
