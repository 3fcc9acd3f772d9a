// sample.cu — stochastic exact acceptance on the device (Muser book Ch. 33
// §33.2: the accept rule of which the greedy accept is the one-hot case).
//
//   for i < k: x = draft[i], p = p_i(x), q = q_i(x), a = 1 if q <= 0 else
//       min(p / q, 1), one uniform u; u <= a accepts and goes on; otherwise
//       stop: the next token is drawn from max(p_i - q_i, 0) / total (from p_i
//       itself when total <= 0);
//   all accepted: the next token is drawn from p_k.
// p_i = softmax of the target logits of row i (temperature 1); q_i = the
// draft's distribution at position i.  Every uniform comes from a caller-owned
// MT19937 stream (Matsumoto & Nishimura 1998), one per attempted draft and one
// for the final draw, in that order; uniform = top 24 bits x 2^-24.  A draw
// walks the tokens in index order and returns the first whose running sum
// exceeds u (the last token of positive weight if rounding leaves none).
#include "common.cuh"
#include "internal.h"
#include "kvmeta.cuh"

namespace spec {

constexpr int kMtN = 624, kMtM = 397;
constexpr int kSampleThreads = 1024;

// ---- MT19937 on a 625-word state in shared memory (624 words + the index of
// the next word to temper); one thread draws.
SPEC_DEV void mt_regenerate(uint32_t* st) {
  for (int i = 0; i < kMtN; ++i) {
    const uint32_t x = (st[i] & 0x80000000u) | (st[i + 1 < kMtN ? i + 1 : 0] & 0x7fffffffu);
    const uint32_t xa = (x >> 1) ^ ((x & 1u) ? 0x9908B0DFu : 0u);
    st[i] = st[i + kMtM < kMtN ? i + kMtM : i + kMtM - kMtN] ^ xa;
  }
  st[kMtN] = 0;
}
SPEC_DEV uint32_t mt_draw(uint32_t* st) {
  if (st[kMtN] >= (uint32_t)kMtN) mt_regenerate(st);
  uint32_t y = st[st[kMtN]++];
  y ^= y >> 11;
  y ^= (y << 7) & 0x9D2C5680u;
  y ^= (y << 15) & 0xEFC60000u;
  y ^= y >> 18;
  return y;
}
SPEC_DEV float mt_uniform(uint32_t* st) { return (float)(mt_draw(st) >> 8) * 0x1p-24f; }

// ---- row normalizers: grid (rows), kSampleThreads threads; per row the max
// m and s = sum exp(l - m) of the logits, thread-strided online pairs combined
// lane -> warp (butterfly) -> CTA (warp order).  A row with a non-finite logit
// gets (NaN, NaN), which the decision kernel reports as SPEC_ST_NONFINITE.
SPEC_DEV void ms_merge(float& m, float& s, float m2, float s2) {
  const float mn = fmaxf(m, m2);
  if (mn == -INFINITY) return;
  s = s * expf(m - mn) + s2 * expf(m2 - mn);
  m = mn;
}

__global__ void __launch_bounds__(kSampleThreads)
softmax_stats_kernel(const float* __restrict__ logits, int V, float2* __restrict__ stats) {
  pdl_trigger();
  pdl_wait();
  __shared__ float wm[32], ws[32];
  const int row = blockIdx.x, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const float* l = logits + (size_t)row * V;
  float m = -INFINITY, s = 0.f;
  bool bad = false;                        // NaN or inf anywhere in the row
  for (int x = threadIdx.x; x < V; x += kSampleThreads) {
    const float v = l[x];
    bad = bad || !(fabsf(v) <= 3.40282347e38f);
    ms_merge(m, s, v, 1.f);
  }
  bad = __syncthreads_or(bad);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float m2 = __shfl_xor_sync(0xffffffffu, m, o), s2 = __shfl_xor_sync(0xffffffffu, s, o);
    ms_merge(m, s, m2, s2);
  }
  if (lane == 0) {
    wm[warp] = m;
    ws[warp] = s;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    float M = wm[0], S = ws[0];
    for (int w = 1; w < kSampleThreads / 32; ++w) ms_merge(M, S, wm[w], ws[w]);
    stats[row] = bad ? make_float2(NAN, NAN) : make_float2(M, S);
  }
}

// ---- block-wide exclusive scan of one float per thread (fixed order: warp
// Kogge-Stone, then the warp totals by warp 0); returns the exclusive prefix,
// *total = the sum of all.
SPEC_DEV float block_exclusive_scan(float v, float* sh, float* total) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  float inc = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const float t = __shfl_up_sync(0xffffffffu, inc, o);
    if (lane >= o) inc += t;
  }
  if (lane == 31) sh[warp] = inc;
  __syncthreads();
  if (warp == 0) {
    float w = sh[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const float t = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += t;
    }
    sh[32 + lane] = w;                       // inclusive prefix of the warp totals
  }
  __syncthreads();
  const float before = warp > 0 ? sh[32 + warp - 1] : 0.f;
  *total = sh[32 + 31];
  const float r = before + (inc - v);
  __syncthreads();                           // sh may be reused by the caller
  return r;
}

// ---- decisions, the final draw and the rollback: one CTA, kSampleThreads.
// Thread t owns the tokens [t*C, (t+1)*C) of a row, C = ceil(V / threads).
__global__ void __launch_bounds__(kSampleThreads)
sample_accept_kernel(const float* __restrict__ logits, const float* __restrict__ q,
                     const int32_t* __restrict__ draft, int k, int V,
                     const float2* __restrict__ stats, uint32_t* mt, KvView kv, int has_kv,
                     const int32_t* step_state, int32_t* status, int32_t* res) {
  pdl_trigger();
  pdl_wait();
  __shared__ uint32_t st[kMtN + 1];
  __shared__ float sh[64];
  __shared__ int sL, sst, best;
  __shared__ float su;
  const int tid = threadIdx.x;
  for (int i = tid; i <= kMtN; i += kSampleThreads) st[i] = mt[i];
  __syncthreads();
  if (tid == 0) {
    int s = step_state ? *status : 0;
    for (int i = 0; i < k; ++i)
      if (draft[i] < 0 || draft[i] >= V) s |= SPEC_ST_TOKEN_RANGE;
    for (int row = 0; row <= k; ++row) {
      const float2 ms = stats[row];
      if (!(ms.y > 0.f) || !isfinite(ms.x) || !isfinite(ms.y)) s |= SPEC_ST_NONFINITE;
    }
    int L = k;
    if (!s) {
      for (int i = 0; i < k; ++i) {
        const int x = draft[i];
        const float2 ms = stats[i];
        const float p = expf(logits[(size_t)i * V + x] - ms.x) / ms.y;
        const float qx = q[(size_t)i * V + x];
        const float a = qx <= 0.f ? 1.f : fminf(p / qx, 1.f);
        if (mt_uniform(st) <= a) continue;
        L = i;
        break;
      }
    }
    sL = L;
    sst = s;
    best = 0x7fffffff;
  }
  __syncthreads();
  const int L = sL;
  int next = -1;
  if (!sst) {
    // weights of the row drawn from: the residual of row L, or p_k
    const int row = L;
    const bool resid = L < k;
    const float2 ms = stats[row];
    const float* lr = logits + (size_t)row * V;
    const float* qr = resid ? q + (size_t)row * V : nullptr;
    const int C = (V + kSampleThreads - 1) / kSampleThreads;
    const int x0 = min(tid * C, V), x1 = min(x0 + C, V);
    bool use_p = !resid;
    float part = 0.f;
    for (int x = x0; x < x1; ++x) {
      const float p = expf(lr[x] - ms.x) / ms.y;
      part += use_p ? p : fmaxf(p - qr[x], 0.f);
    }
    float total;
    block_exclusive_scan(part, sh, &total);
    if (resid && !(total > 0.f)) {          // residual all zero: draw from p_L itself
      use_p = true;
      part = 0.f;
      for (int x = x0; x < x1; ++x) part += expf(lr[x] - ms.x) / ms.y;
      block_exclusive_scan(part, sh, &total);
    }
    // normalised weights r = w / total; their running sum in index order:
    // chunk sums scanned across threads, then each chunk walked in order
    float rpart = 0.f;
    for (int x = x0; x < x1; ++x) {
      const float p = expf(lr[x] - ms.x) / ms.y;
      rpart += (use_p ? p : fmaxf(p - qr[x], 0.f)) / total;
    }
    float rtot;
    const float before = block_exclusive_scan(rpart, sh, &rtot);
    if (tid == 0) su = mt_uniform(st);
    __syncthreads();
    const float u = su;
    float c = 0.f;
    int last = -1, hit = 0x7fffffff;
    for (int x = x0; x < x1; ++x) {
      const float p = expf(lr[x] - ms.x) / ms.y;
      const float r = (use_p ? p : fmaxf(p - qr[x], 0.f)) / total;
      if (r > 0.f) last = x;
      c += r;
      if (u < before + c) {
        hit = x;
        break;
      }
    }
    if (hit != 0x7fffffff) atomicMin(&best, hit);
    __syncthreads();
    const int found = best;
    __syncthreads();
    if (found == 0x7fffffff) {
      // rounding left no crossing: the last token of positive weight (no
      // thread stopped early, so every thread saw its whole chunk)
      if (tid == 0) best = -1;
      __syncthreads();
      if (last >= 0) atomicMax(&best, last);
      __syncthreads();
      next = best;
    } else {
      next = found;
    }
  }
  // the MT state and the result
  __syncthreads();
  for (int i = tid; i <= kMtN; i += kSampleThreads) mt[i] = st[i];
  if (tid != 0) return;
  int s = sst;
  int Lr = L;
  const bool appended = step_state ? step_state[1] != 0 : has_kv != 0;
  const int n_past = step_state ? step_state[0] : (has_kv ? *kv.seq_len - (k + 1) : 0);
  if (s) {
    Lr = 0;
    next = -1;
    if (has_kv && appended) kv_rollback_dev(kv, n_past);
  } else if (has_kv && appended) {
    kv_rollback_dev(kv, n_past + Lr + 1);
  }
  *status = s;
  res[0] = Lr;
  res[1] = next;
  res[2] = s;
  res[3] = has_kv ? *kv.seq_len : 0;
}

cudaError_t launch_sample_accept(const float* logits, const float* q, const int32_t* draft, int k,
                                 int V, float2* stats, uint32_t* mt, const KvView* kv,
                                 const int32_t* step_state, int32_t* status, int32_t* res,
                                 cudaStream_t st, bool pdl) {
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(k + 1);
  cfg.blockDim = dim3(kSampleThreads);
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  cudaError_t e = cudaLaunchKernelEx(&cfg, softmax_stats_kernel, logits, V, stats);
  if (e != cudaSuccess) return e;
  cfg.gridDim = dim3(1);
  KvView v = kv ? *kv : KvView{};
  return cudaLaunchKernelEx(&cfg, sample_accept_kernel, logits, q, draft, k, V, (const float2*)stats, mt, v,
                            kv ? 1 : 0, step_state, status, res);
}

}  // namespace spec
