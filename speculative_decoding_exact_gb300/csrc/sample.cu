// sample.cu — stochastic exact acceptance on the device (Muser book Ch. 33
// §33.2: the accept rule of which the greedy accept is the one-hot case).
//
//   for i < k: x = draft[i], p = p_i(x), q = q_i(x), a = 1 if q <= 0 else
//       min(p / q, 1), one uniform u; u <= a accepts and goes on; otherwise
//       stop: the next token is drawn from the weights max(p_i - q_i, 0)
//       (from p_i itself when they sum to 0);
//   all accepted: the next token is drawn from the weights p_k.
// p_i = softmax of the target logits of row i (temperature 1); q_i = the
// draft's distribution at position i.  Every uniform comes from a caller-owned
// MT19937 stream (Matsumoto & Nishimura 1998), one per attempted draft and one
// for the final draw, in that order; uniform = top 24 bits x 2^-24.  As the
// listing of §33.2 does, a rejection's residual r = max(p_i - q_i, 0) is
// summed (total) and every entry divided by total, unless total <= 0, when
// the draw uses p_i itself.  A draw walks the tokens in index order and
// returns the first whose running sum of the draw weights exceeds u (the last
// token of positive weight if rounding leaves none).  The device sums in a
// fixed tree order, not token by token, so totals may differ from a serial
// sum by rounding.
//
// Kernels: row normalizers (8 CTAs per row), the decisions and the final
// uniform (one CTA), per-tile sums of the drawn row's raw weights (one CTA
// per kSampleThreads tokens, coalesced), per-tile sums of its draw weights
// (the same tiles, after the total is known), the draw and the rollback (one
// CTA).
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

// ---- row normalizers: grid (kStatParts, rows), kSampleThreads threads.  CTA
// (part, row) takes the logits [part*Vp, min(V, (part+1)*Vp)), Vp =
// ceil(V / kStatParts): their max m (one pass), then s = sum exp(l - m) (a
// second pass over the same 64 KB, served from L1), each reduced lane -> warp
// (butterfly) -> CTA (warp order).  A part with a non-finite logit gets (NaN,
// NaN); an empty part (-inf, 0).  The decision kernel merges a row's parts
// in part order.
SPEC_DEV void ms_merge(float& m, float& s, float m2, float s2) {
  const float mn = fmaxf(m, m2);
  if (mn == -INFINITY) return;
  s = s * expf(m - mn) + s2 * expf(m2 - mn);
  m = mn;
}

constexpr int kStatParts = 8;

__global__ void __launch_bounds__(kSampleThreads)
softmax_stats_kernel(const float* __restrict__ logits, int V, float2* __restrict__ pstats) {
  pdl_trigger();
  pdl_wait();
  __shared__ float red[32];
  const int part = blockIdx.x, row = blockIdx.y, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int Vp = (V + kStatParts - 1) / kStatParts;
  const int x0 = part * Vp, x1 = min(V, x0 + Vp);
  const float* l = logits + (size_t)row * V;
  float m = -INFINITY;
  bool bad = false;                        // NaN or inf anywhere in the part
  for (int x = x0 + threadIdx.x; x < x1; x += kSampleThreads) {
    const float v = l[x];
    bad = bad || !(fabsf(v) <= 3.40282347e38f);
    m = fmaxf(m, v);
  }
  bad = __syncthreads_or(bad);
  m = warp_max(m);
  if (lane == 0) red[warp] = m;
  __syncthreads();
  m = red[0];
  for (int w = 1; w < kSampleThreads / 32; ++w) m = fmaxf(m, red[w]);
  __syncthreads();                         // red is reused below
  float s = 0.f;
  if (m != -INFINITY)
    for (int x = x0 + threadIdx.x; x < x1; x += kSampleThreads) s += expf(l[x] - m);
  s = warp_sum(s);
  if (lane == 0) red[warp] = s;
  __syncthreads();
  if (threadIdx.x == 0) {
    float S = red[0];
    for (int w = 1; w < kSampleThreads / 32; ++w) S += red[w];
    pstats[row * kStatParts + part] = bad ? make_float2(NAN, NAN) : make_float2(m, S);
  }
}

// ---- block-wide inclusive scan of one float per thread in a fixed order
// (warp Kogge-Stone, then the warp totals scanned by warp 0 and added);
// *total = the last thread's inclusive value.  sh: 64 floats of shared memory.
SPEC_DEV float block_inclusive_scan(float v, float* sh, float* total) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;
  float inc = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const float t = __shfl_up_sync(0xffffffffu, inc, o);
    if (lane >= o) inc += t;
  }
  if (lane == 31) sh[warp] = inc;
  __syncthreads();
  if (warp == 0) {
    float w = lane < nw ? sh[lane] : 0.f;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const float t = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += t;
    }
    sh[32 + lane] = w;                       // inclusive prefix of the warp totals
  }
  __syncthreads();
  const float r = warp > 0 ? sh[32 + warp - 1] + inc : inc;
  __syncthreads();
  if (threadIdx.x == blockDim.x - 1) sh[0] = r;
  __syncthreads();
  *total = sh[0];
  __syncthreads();                           // sh may be reused by the caller
  return r;
}

// Scratch of one decision (device): L, the final uniform, the status, then
// per tile of kSampleThreads tokens the sums and the last positive index of
// the raw weights w (the residual or p_k) and of p, and the sums of the draw
// weights (w / total, or p).
struct SampleScratch {
  int L;
  float u;
  int status;
  int pad;
};
constexpr int kMaxTiles = 1024;              // V <= 1024 * kSampleThreads
// then the row normalizers' parts: float2 [16 rows][kStatParts]
constexpr size_t kPstatsOffset = sizeof(SampleScratch) + 5 * sizeof(float) * kMaxTiles;
size_t sample_scratch_bytes() { return kPstatsOffset + sizeof(float2) * 16 * kStatParts; }

// weight of token x of the drawn row: max(p - q, 0) for a rejection, p else
SPEC_DEV float sample_weight(const float* lr, const float* qr, float2 ms, int x, int V, bool resid, bool use_p) {
  if (x >= V) return 0.f;
  const float p = expf(lr[x] - ms.x) / ms.y;
  return (resid && !use_p) ? fmaxf(p - qr[x], 0.f) : p;
}

// ---- decisions and the final uniform: one CTA (the MT state is staged in
// shared memory by all threads; thread 0 draws)
__global__ void __launch_bounds__(kSampleThreads)
sample_decide_kernel(const float* __restrict__ logits, const float* __restrict__ q,
                     const int32_t* __restrict__ draft, int k, int V,
                     uint32_t* mt, const int32_t* step_state, const int32_t* status, SampleScratch* sc,
                     const float2* __restrict__ pstats, float2* __restrict__ stats_out) {
  pdl_trigger();
  pdl_wait();
  __shared__ uint32_t st[kMtN + 1];
  __shared__ float2 rs[16];
  const int tid = threadIdx.x;
  for (int i = tid; i <= kMtN; i += kSampleThreads) st[i] = mt[i];
  // thread r merges row r's normalizer parts in part order (any NaN part
  // makes the row NaN); the tile and finish kernels read the result
  if (tid <= k) {
    float M = -INFINITY, S = 0.f;
    bool nan = false;
    for (int p = 0; p < kStatParts; ++p) {
      const float2 v = pstats[tid * kStatParts + p];
      if (isnan(v.x) || isnan(v.y)) nan = true;
      else ms_merge(M, S, v.x, v.y);
    }
    const float2 r = nan ? make_float2(NAN, NAN) : make_float2(M, S);
    rs[tid] = r;
    stats_out[tid] = r;
  }
  __syncthreads();
  if (tid == 0) {
    int s = step_state ? *status : 0;
    for (int i = 0; i < k; ++i)
      if (draft[i] < 0 || draft[i] >= V) s |= SPEC_ST_TOKEN_RANGE;
    for (int row = 0; row <= k; ++row) {
      const float2 ms = rs[row];
      if (!(ms.y > 0.f) || !isfinite(ms.x) || !isfinite(ms.y)) s |= SPEC_ST_NONFINITE;
    }
    int L = k;
    float u = 0.f;
    if (!s) {
      for (int i = 0; i < k; ++i) {
        const int x = draft[i];
        const float2 ms = rs[i];
        const float p = expf(logits[(size_t)i * V + x] - ms.x) / ms.y;
        const float qx = q[(size_t)i * V + x];
        const float a = qx <= 0.f ? 1.f : fminf(p / qx, 1.f);
        if (mt_uniform(st) <= a) continue;
        L = i;
        break;
      }
      u = mt_uniform(st);                    // the final draw
    }
    sc->L = L;
    sc->u = u;
    sc->status = s;
  }
  __syncthreads();
  for (int i = tid; i <= kMtN; i += kSampleThreads) mt[i] = st[i];
}

// ---- per tile of kSampleThreads tokens of the drawn row (coalesced): the sum
// of the weights w and of p (the block scan's last value) and the last
// positive index of each
__global__ void __launch_bounds__(kSampleThreads)
sample_tiles_kernel(const float* __restrict__ logits, const float* __restrict__ q, int k, int V,
                    const float2* __restrict__ stats, SampleScratch* sc) {
  pdl_trigger();
  pdl_wait();
  __shared__ float sh[64];
  __shared__ int lw, lp;
  if (sc->status) return;
  const int L = sc->L, j = blockIdx.x, tid = threadIdx.x;
  const bool resid = L < k;
  const int x = j * kSampleThreads + tid;
  const float* lr = logits + (size_t)L * V;
  const float* qr = resid ? q + (size_t)L * V : nullptr;
  const float2 ms = stats[L];
  const float w = sample_weight(lr, qr, ms, x, V, resid, false);
  const float p = sample_weight(lr, qr, ms, x, V, resid, true);
  if (tid == 0) {
    lw = -1;
    lp = -1;
  }
  float tw, tp;
  block_inclusive_scan(w, sh, &tw);
  block_inclusive_scan(p, sh, &tp);
  if (w > 0.f) atomicMax(&lw, x);
  if (p > 0.f) atomicMax(&lp, x);
  __syncthreads();
  if (tid == 0) {
    float* t = reinterpret_cast<float*>(sc + 1);
    t[j] = tw;
    t[kMaxTiles + j] = tp;
    reinterpret_cast<int*>(t)[2 * kMaxTiles + j] = lw;
    reinterpret_cast<int*>(t)[3 * kMaxTiles + j] = lp;
  }
}

// total of the raw weights: the block scan of the raw tile sums (thread t
// holds tile t), the same expression in every kernel that needs it
SPEC_DEV float raw_total(const float* t, int ntiles, float* sh) {
  float tot;
  block_inclusive_scan(threadIdx.x < ntiles ? t[threadIdx.x] : 0.f, sh, &tot);
  return tot;
}

// weight of token x in the draw: the residual divided by its total, or p
// (the residual summed to <= 0, or all drafts were accepted)
SPEC_DEV float draw_weight(const float* lr, const float* qr, float2 ms, int x, int V, bool resid,
                           bool use_p, float tot) {
  if (x >= V) return 0.f;
  const float p = expf(lr[x] - ms.x) / ms.y;
  return (resid && !use_p) ? __fdiv_rn(fmaxf(p - qr[x], 0.f), tot) : p;
}

// ---- per tile of kSampleThreads tokens of the drawn row: the sum of the
// draw weights (the block scan's last value), after the total is known
__global__ void __launch_bounds__(kSampleThreads)
sample_norm_tiles_kernel(const float* __restrict__ logits, const float* __restrict__ q, int k, int V,
                         const float2* __restrict__ stats, SampleScratch* sc) {
  pdl_trigger();
  pdl_wait();
  __shared__ float sh[64];
  if (sc->status) return;
  const int L = sc->L, j = blockIdx.x, tid = threadIdx.x;
  const bool resid = L < k;
  const int ntiles = (V + kSampleThreads - 1) / kSampleThreads;
  float* t = reinterpret_cast<float*>(sc + 1);
  const float tot = raw_total(t, ntiles, sh);
  const bool use_p = resid && !(tot > 0.f);
  const float* lr = logits + (size_t)L * V;
  const float* qr = resid ? q + (size_t)L * V : nullptr;
  const float v = draw_weight(lr, qr, stats[L], j * kSampleThreads + tid, V, resid, use_p, tot);
  float tv;
  block_inclusive_scan(v, sh, &tv);
  if (tid == 0) t[4 * kMaxTiles + j] = tv;
}

// ---- the draw and the rollback: one CTA.  With prefix_j the inclusive scan
// of the draw-weight tile sums up to tile j-1, the running sum at token x of
// tile j is prefix_j + (the tile's inclusive scan at x); the drawn token is
// the first with u < that sum, found in the first tile with
// u < prefix_j + tile_j (the same expression as its last token).
__global__ void __launch_bounds__(kSampleThreads)
sample_finish_kernel(const float* __restrict__ logits, const float* __restrict__ q, int k, int V,
                     const float2* __restrict__ stats, const SampleScratch* sc, KvView kv, int has_kv,
                     const int32_t* step_state, int32_t* status, int32_t* res) {
  pdl_trigger();
  pdl_wait();
  __shared__ float sh[64];
  __shared__ int hit_tile, hit_x, last;
  __shared__ float prefix_hit;
  __shared__ float incl[kMaxTiles];
  const int tid = threadIdx.x;
  const int s = sc->status;
  int next = -1;
  const int L = sc->L;
  if (!s) {
    const bool resid = L < k;
    const int ntiles = (V + kSampleThreads - 1) / kSampleThreads;
    const float* t = reinterpret_cast<const float*>(sc + 1);
    const int* ti = reinterpret_cast<const int*>(t);
    const float tot = raw_total(t, ntiles, sh);
    const bool use_p = resid && !(tot > 0.f);     // residual all zero: draw from p_L itself
    const float mine = tid < ntiles ? t[4 * kMaxTiles + tid] : 0.f;
    float all;
    const float inc = block_inclusive_scan(mine, sh, &all);
    if (tid == 0) {
      hit_tile = 0x7fffffff;
      hit_x = 0x7fffffff;
      last = -1;
    }
    // inclusive value of the previous tile (prefix_j), from the neighbour
    if (tid < ntiles) incl[tid] = inc;
    __syncthreads();
    const float prefix = tid > 0 && tid < ntiles ? incl[tid - 1] : 0.f;
    const float u = sc->u;
    if (tid < ntiles && u < prefix + mine) atomicMin(&hit_tile, tid);
    if (tid < ntiles) {
      const int lt = (resid && !use_p) ? ti[2 * kMaxTiles + tid] : ti[3 * kMaxTiles + tid];
      if (lt >= 0) atomicMax(&last, lt);
    }
    __syncthreads();
    const int j = hit_tile;
    if (j != 0x7fffffff) {
      if (tid == 0) prefix_hit = j > 0 ? incl[j - 1] : 0.f;
      __syncthreads();
      const float* lr = logits + (size_t)L * V;
      const float* qr = resid ? q + (size_t)L * V : nullptr;
      const int x = j * kSampleThreads + tid;
      const float v = draw_weight(lr, qr, stats[L], x, V, resid, use_p, tot);
      float tt;
      const float c = prefix_hit + block_inclusive_scan(v, sh, &tt);
      if (x < V && v > 0.f && u < c) atomicMin(&hit_x, x);
      __syncthreads();
      // a ragged last tile can miss by an ulp: its scan over the valid tokens
      // need not repeat the tile sum bit for bit
      next = hit_x != 0x7fffffff ? hit_x : last;
    } else {
      next = last;                           // rounding left no crossing
    }
  }
  if (tid != 0) return;
  int st = s;
  int Lr = L;
  const bool appended = step_state ? step_state[1] != 0 : has_kv != 0;
  const int n_past = step_state ? step_state[0] : (has_kv ? *kv.seq_len - (k + 1) : 0);
  if (st) {
    Lr = 0;
    next = -1;
    if (has_kv && appended) kv_rollback_dev(kv, n_past);
  } else if (has_kv && appended) {
    kv_rollback_dev(kv, n_past + Lr + 1);
  }
  *status = st;
  res[0] = Lr;
  res[1] = next;
  res[2] = st;
  res[3] = has_kv ? *kv.seq_len : 0;
}

cudaError_t launch_sample_accept(const float* logits, const float* q, const int32_t* draft, int k,
                                 int V, float2* stats, uint8_t* scratch, uint32_t* mt, const KvView* kv,
                                 const int32_t* step_state, int32_t* status, int32_t* res,
                                 cudaStream_t st, bool pdl) {
  if ((V + kSampleThreads - 1) / kSampleThreads > kMaxTiles) return cudaErrorInvalidValue;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(kStatParts, k + 1);
  cfg.blockDim = dim3(kSampleThreads);
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  SampleScratch* sc = reinterpret_cast<SampleScratch*>(scratch);
  float2* pstats = reinterpret_cast<float2*>(scratch + kPstatsOffset);
  cudaError_t e = cudaLaunchKernelEx(&cfg, softmax_stats_kernel, logits, V, pstats);
  if (e != cudaSuccess) return e;
  cfg.gridDim = dim3(1);
  e = cudaLaunchKernelEx(&cfg, sample_decide_kernel, logits, q, draft, k, V, mt, step_state,
                         (const int32_t*)status, sc, (const float2*)pstats, stats);
  if (e != cudaSuccess) return e;
  cfg.gridDim = dim3((V + kSampleThreads - 1) / kSampleThreads);
  e = cudaLaunchKernelEx(&cfg, sample_tiles_kernel, logits, q, k, V, (const float2*)stats, sc);
  if (e != cudaSuccess) return e;
  e = cudaLaunchKernelEx(&cfg, sample_norm_tiles_kernel, logits, q, k, V, (const float2*)stats, sc);
  if (e != cudaSuccess) return e;
  cfg.gridDim = dim3(1);
  KvView v = kv ? *kv : KvView{};
  return cudaLaunchKernelEx(&cfg, sample_finish_kernel, logits, q, k, V, (const float2*)stats,
                            (const SampleScratch*)sc, v, kv ? 1 : 0, step_state, status, res);
}

}  // namespace spec
