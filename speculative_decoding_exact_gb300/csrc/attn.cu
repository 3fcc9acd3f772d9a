// attn.cu — verify attention of k+1 query rows against the paged bf16 KV cache.
//
// Row i of the block sits at position n_past + i and sees positions
// 0..n_past+i (the carried-frontier row first, then the drafts: Muser book
// Ch. 33 §33.7).  Query head h reads KV head h / (n_q/n_kv).
// s = q.k / sqrt(head_dim), softmax over the visible positions, o = sum p v.
//
// Decomposition (flash-decoding): CTA (chunk c, kv head, head half) takes the
// keys [c*C, (c+1)*C) for its query heads of that kv head (one warp per head,
// the 16 rows of the block are the MMA's 16 rows), walking them in 64-key
// sub-chunks with a running (max, sum, unnormalised o) per row (online
// softmax), and writes those partials.  C is 64 times the number of
// sub-chunks per chunk, set from max_ctx alone so that a long context still
// uses at most about 48 chunks (the partials would otherwise outgrow the KV
// they summarise).  A merge kernel combines the chunks in chunk order,
// normalises, and quantises the rows for the output projection.  Chunk and
// sub-chunk boundaries are fixed by max_ctx and masked keys contribute exact
// zeros, so row i's result is the same for every M (batch-height invariance:
// "The Two-Fifteen That Wasn't").
//
// Precision: K and V are exact bf16; q and p are split into bf16 hi + lo parts
// (two MMAs each) so the products carry ~16 significant bits; accumulation is
// fp32.
#include "common.cuh"
#include "internal.h"
#include "quant.cuh"

namespace spec {

constexpr int kChunk = 64;
constexpr int kRowPad = 136;         // bf16 per padded K/V row in shared memory (272 B)
constexpr int kMaxGroup = 13;        // max query heads per kv head

constexpr int kTargetChunks = 48;    // chunks per context at most (about)

AttnPlan make_attn_plan(int nq, int nkv, int dh, int max_ctx) {
  AttnPlan a;
  a.nq = nq;
  a.nkv = nkv;
  a.dh = dh;
  a.max_ctx = max_ctx;
  const int subs64 = (max_ctx + kChunk - 1) / kChunk;
  const int subs = (subs64 + kTargetChunks - 1) / kTargetChunks;   // 64-key sub-chunks per chunk
  a.chunk = kChunk * (subs > 0 ? subs : 1);
  a.max_chunks = (max_ctx + a.chunk - 1) / a.chunk;
  return a;
}
size_t attn_smem_bytes() { return (size_t)2 * 2 * kChunk * kRowPad * sizeof(__nv_bfloat16); }

size_t attn_partial_floats(const AttnPlan& a, int max_rows) {
  (void)max_rows;
  return (size_t)a.max_chunks * a.nq * 16 * (a.dh + 2);
}

SPEC_DEV void ldsm_x4(uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3, const void* p) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(smem_u32(p)));
}
SPEC_DEV void ldsm_x4_t(uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3, const void* p) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(smem_u32(p)));
}

SPEC_DEV uint32_t pack_bf16(float lo, float hi) {
  return (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(lo)) |
         ((uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(hi)) << 16);
}
// split x into bf16 hi + bf16 lo (x - hi), packed pairs
SPEC_DEV void split2(float x0, float x1, uint32_t& hi, uint32_t& lo) {
  const __nv_bfloat16 h0 = __float2bfloat16_rn(x0), h1 = __float2bfloat16_rn(x1);
  hi = (uint32_t)__bfloat16_as_ushort(h0) | ((uint32_t)__bfloat16_as_ushort(h1) << 16);
  lo = pack_bf16(x0 - __bfloat162float(h0), x1 - __bfloat162float(h1));
}

// dh is fixed to 128 (8 k-steps of 16 for q.k, 16 n-tiles of 8 for p.v).
// grid (chunk, kv head, head part): the query heads of a kv head are split
// over HS CTAs (the K/V chunk is read HS times, all but once from L2).  One
// 64-key sub-chunk per chunk (short contexts): HS = 2, 7 warps.  Several
// sub-chunks: HS = 3, at most 5 warps, so that two CTAs per SM fit the
// registers of the running softmax state.
__host__ __device__ constexpr int head_split(bool multi) { return multi ? 3 : 2; }
__host__ __device__ constexpr int warps_per_cta(bool multi) {
  return (kMaxGroup + head_split(multi) - 1) / head_split(multi);
}

size_t qfrag_bytes(int nq) { return (size_t)nq * 8 * 2 * 32 * 16; }

__global__ void q_to_frag_kernel(const float* __restrict__ q, int M, int nq, uint8_t* qfrag) {
  pdl_trigger();
  pdl_wait();
  const int row = blockIdx.y;
  const int col = blockIdx.x * blockDim.x + threadIdx.x;
  if (col >= nq * 128) return;
  write_qfrag(qfrag, row, col >> 7, col & 127, row < M ? q[(size_t)row * nq * 128 + col] : 0.f);
}

cudaError_t launch_q_to_frag(const float* q, int M, int nq, uint8_t* qfrag, cudaStream_t st, bool pdl) {
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((nq * 128 + 255) / 256, 16);
  cfg.blockDim = dim3(256);
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, q_to_frag_kernel, q, M, nq, qfrag);
}

// a Q-fragment load the compiler re-issues per use (kept out of the registers
// across the key loop: the fragments are L1/L2 hits)
SPEC_DEV uint4 ldg_frag(const uint4* p) {
  uint4 v;
  asm volatile("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

template <bool MULTI>
__global__ void __launch_bounds__(warps_per_cta(MULTI) * 32, 2)
attn_partial_kernel(const uint4* __restrict__ qf, int M, int nq, int nkv, int chunk_keys, KvView kv,
                    int layer, float* __restrict__ part, const int32_t* status) {
  constexpr int kHeadSplit = head_split(MULTI);
  // [buffer][K, V][64 keys][padded 136 bf16]
  extern __shared__ __align__(128) __nv_bfloat16 kvs[];

  pdl_trigger();
  pdl_wait();
  const int chunk = blockIdx.x, kvh = blockIdx.y;
  const int group = nq / nkv;
  const int per = (group + kHeadSplit - 1) / kHeadSplit;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, t = lane & 3;
  if (*status & (SPEC_ST_TOKEN_RANGE | SPEC_ST_POOL_EMPTY | SPEC_ST_CTX_FULL)) return;
  const int len = *kv.seq_len;             // block appended: n_past + M
  const int n_past = len - M;
  const int key0 = chunk * chunk_keys;
  if (key0 >= len) return;
  // sub-chunks with keys (exactly one when the chunk is one sub-chunk long)
  const int nsub = MULTI ? min(chunk_keys, len - key0 + kChunk - 1) / kChunk : 1;

  // ---- K, V sub-chunk sc -> shared buffer sc % 2 (rows beyond len are zero)
  auto load_sub = [&](int sc) {
    __nv_bfloat16* buf = kvs + (size_t)(sc & 1) * 2 * kChunk * kRowPad;
    const int ks0 = key0 + sc * kChunk;
    for (int i = threadIdx.x; i < 2 * kChunk * 16; i += blockDim.x) {
      const int which = i / (kChunk * 16), r = (i / 16) % kChunk, c16 = i % 16;
      __nv_bfloat16* dst = buf + which * kChunk * kRowPad + r * kRowPad + c16 * 8;
      const int pos = ks0 + r;
      const int lp = pos / kv.page_size;
      const int page = (pos < len && lp < kv.max_seq_pages) ? kv.page_table[lp] : -1;
      if (page >= 0 && page < kv.num_pages) {
        const size_t off = ((((size_t)page * kv.n_layers + layer) * 2 + which) * kv.n_kv + kvh) *
                               (size_t)kv.page_size * kv.head_dim +
                           (size_t)(pos % kv.page_size) * kv.head_dim + c16 * 8;
        cp_async16(dst, kv.pool + off);
      } else {
        *reinterpret_cast<uint4*>(dst) = make_uint4(0, 0, 0, 0);
      }
    }
    cp_async_commit();
  };

  const int hl = blockIdx.z * per + warp;          // head within the kv group
  const bool active = warp < per && hl < group;
  const int head = kvh * group + (active ? hl : 0);
  const uint4* Qf = qf + (size_t)head * 8 * 2 * 32;   // [8 ksteps][hi, lo][32 lanes]
  const float scale = 1.0f / sqrtf(128.0f);

  // running per-row state (rows g and g+8): max, sum, unnormalised o
  float mrun[2] = {-INFINITY, -INFINITY}, lrun[2] = {0.f, 0.f};
  float o[16][4];
#pragma unroll
  for (int nd = 0; nd < 16; ++nd)
#pragma unroll
    for (int e = 0; e < 4; ++e) o[nd][e] = 0.f;

  load_sub(0);
  for (int sc = 0; sc < nsub; ++sc) {
    if (sc + 1 < nsub) {
      load_sub(sc + 1);
      cp_async_wait<1>();
    } else {
      cp_async_wait<0>();
    }
    __syncthreads();
    const __nv_bfloat16* Ks = kvs + (size_t)(sc & 1) * 2 * kChunk * kRowPad;
    const __nv_bfloat16* Vs = Ks + kChunk * kRowPad;
    const int ks0 = key0 + sc * kChunk;
    if (active) {
      // ---- scores S = q.k for 64 keys: 8 n-tiles x 4
      float s[8][4];
#pragma unroll
      for (int nt = 0; nt < 8; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) s[nt][e] = 0.f;
#pragma unroll
      for (int kp = 0; kp < 4; ++kp) {          // pairs of k-steps
        const uint4 qh0 = ldg_frag(Qf + ((2 * kp) * 2 + 0) * 32 + lane);
        const uint4 ql0 = ldg_frag(Qf + ((2 * kp) * 2 + 1) * 32 + lane);
        const uint4 qh1 = ldg_frag(Qf + ((2 * kp + 1) * 2 + 0) * 32 + lane);
        const uint4 ql1 = ldg_frag(Qf + ((2 * kp + 1) * 2 + 1) * 32 + lane);
#pragma unroll
        for (int nt = 0; nt < 8; ++nt) {
          uint32_t b0, b1, b2, b3;
          const int krow = 8 * nt + (lane & 7);
          const int kcol = 32 * kp + 8 * (lane >> 3);
          ldsm_x4(b0, b1, b2, b3, Ks + krow * kRowPad + kcol);
          mma16816_bf16(s[nt], qh0.x, qh0.y, qh0.z, qh0.w, b0, b1);
          mma16816_bf16(s[nt], ql0.x, ql0.y, ql0.z, ql0.w, b0, b1);
          mma16816_bf16(s[nt], qh1.x, qh1.y, qh1.z, qh1.w, b2, b3);
          mma16816_bf16(s[nt], ql1.x, ql1.y, ql1.z, ql1.w, b2, b3);
        }
      }

      // ---- mask, running max, p = exp(s - max), rescale of the running state
      float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
      for (int nt = 0; nt < 8; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int row = g + 8 * (e >> 1);
          const int key = ks0 + 8 * nt + 2 * t + (e & 1);
          const bool vis = row < M && key <= n_past + row;
          const float v = vis ? s[nt][e] * scale : -INFINITY;
          s[nt][e] = v;
          mx[e >> 1] = fmaxf(mx[e >> 1], v);
        }
      float alpha[2];
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], 1));
        mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], 2));
        const float mnew = fmaxf(mrun[r], mx[r]);
        alpha[r] = (mrun[r] == -INFINITY) ? 0.f : expf(mrun[r] - mnew);
        mrun[r] = mnew;
      }
      float sum[2] = {0.f, 0.f};
#pragma unroll
      for (int nt = 0; nt < 8; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float m = mrun[e >> 1];
          const float p = (s[nt][e] == -INFINITY) ? 0.f : expf(s[nt][e] - m);
          s[nt][e] = p;
          sum[e >> 1] += p;
        }
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        sum[r] += __shfl_xor_sync(0xffffffffu, sum[r], 1);
        sum[r] += __shfl_xor_sync(0xffffffffu, sum[r], 2);
        lrun[r] = lrun[r] * alpha[r] + sum[r];
      }
#pragma unroll
      for (int nd = 0; nd < 16; ++nd)
#pragma unroll
        for (int e = 0; e < 4; ++e) o[nd][e] *= alpha[e >> 1];

      // ---- o += p.v : 16 n-tiles of 8 dims
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {           // 16 keys per k-step
        uint32_t ph[4], pl[4];
        split2(s[2 * kk][0], s[2 * kk][1], ph[0], pl[0]);
        split2(s[2 * kk][2], s[2 * kk][3], ph[1], pl[1]);
        split2(s[2 * kk + 1][0], s[2 * kk + 1][1], ph[2], pl[2]);
        split2(s[2 * kk + 1][2], s[2 * kk + 1][3], ph[3], pl[3]);
#pragma unroll
        for (int np = 0; np < 8; ++np) {          // pairs of dim tiles
          uint32_t b0, b1, b2, b3;
          const int vrow = 16 * kk + (lane & 7) + 8 * ((lane >> 3) & 1);
          const int vcol = 16 * np + 8 * (lane >> 4);
          ldsm_x4_t(b0, b1, b2, b3, Vs + vrow * kRowPad + vcol);
          mma16816_bf16(o[2 * np], ph[0], ph[1], ph[2], ph[3], b0, b1);
          mma16816_bf16(o[2 * np], pl[0], pl[1], pl[2], pl[3], b0, b1);
          mma16816_bf16(o[2 * np + 1], ph[0], ph[1], ph[2], ph[3], b2, b3);
          mma16816_bf16(o[2 * np + 1], pl[0], pl[1], pl[2], pl[3], b2, b3);
        }
      }
    }
    __syncthreads();            // the next prefetch overwrites this buffer
  }
  if (!active) return;

  // ---- partials: [chunk][head][row][128 o | max | sum]
  const int stride = 130;
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    const int row = g + 8 * r;
    float* base = part + (((size_t)chunk * nq + head) * 16 + row) * stride;
#pragma unroll
    for (int nd = 0; nd < 16; ++nd)
      *reinterpret_cast<float2*>(base + 8 * nd + 2 * t) = make_float2(o[nd][2 * r], o[nd][2 * r + 1]);
    if (t == 0) {
      base[128] = mrun[r];
      base[129] = lrun[r];
    }
  }
}


// merge: grid (nq*128/256 blocks, 16 rows), 256 threads = 2 heads x 128 dims.
// For row i the chunks 0 .. (n_past+i)/C are combined:
//   M = max_c m_c;  w_c = exp(m_c - M);  L = sum_c w_c l_c;  o = sum_c w_c o_c;
// out = o / L.  Warp hh (one per head) computes M, the weights and L with
// warp shuffles in a fixed butterfly order; o is summed in chunk order.  The
// chunk count depends on the row's position only, so the result is the same
// for every M.
__global__ void __launch_bounds__(256)
attn_merge_kernel(const float* __restrict__ part, int M, int nq, int max_chunks, int chunk_keys,
                  const int32_t* seq_len, float* __restrict__ out, uint8_t* act, int32_t* status) {
  pdl_trigger();
  pdl_wait();
  extern __shared__ float msh[];          // [2][max_chunks] weights, then [2][max_chunks] sums
  __shared__ float vals[256];
  __shared__ float lsum[2];
  const int b = blockIdx.x, row = blockIdx.y;
  const int H = nq * 128;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const bool valid = row < M && !(*status & (SPEC_ST_TOKEN_RANGE | SPEC_ST_POOL_EMPTY | SPEC_ST_CTX_FULL));
  const int n_past = *seq_len - M;
  const int nchunks = valid ? (n_past + row) / chunk_keys + 1 : 0;
  const size_t cstride = (size_t)nq * 16 * 130;
  if (warp < 2) {
    const int hh = warp;
    const float* st = part + (((size_t)(2 * b + hh)) * 16 + row) * 130;
    // lane takes the chunks lane, lane + 32, ...: maxima first (kept in
    // shared memory), then the weights and the weighted sums
    // (max, sum) of chunk c are adjacent: one 8-byte load per chunk
    float m = -INFINITY;
    float* lsh = msh + 2 * max_chunks;      // the chunk sums, [2][max_chunks]
    for (int c = lane; c < nchunks; c += 32) {
      const float2 ml = *reinterpret_cast<const float2*>(st + c * cstride + 128);
      msh[hh * max_chunks + c] = ml.x;
      lsh[hh * max_chunks + c] = ml.y;
      m = fmaxf(m, ml.x);
    }
    m = warp_max(m);
    float L = 0.f;
    for (int c = lane; c < nchunks; c += 32) {
      const float mc = msh[hh * max_chunks + c];
      const float w = (mc == -INFINITY) ? 0.f : expf(mc - m);
      msh[hh * max_chunks + c] = w;
      L += w * lsh[hh * max_chunks + c];
    }
    L = warp_sum(L);
    if (lane == 0) lsum[hh] = L;
  }
  __syncthreads();
  // weighted sum of the unnormalised outputs, in chunk order
  const int hh = threadIdx.x >> 7, d = threadIdx.x & 127;
  const float* pp = part + (((size_t)(2 * b + hh)) * 16 + row) * 130 + d;
  const float* w = msh + hh * max_chunks;
  float o = 0.f;
  int c = 0;
  for (; c + 8 <= nchunks; c += 8) {        // 8 loads in flight, then the sums in chunk order
    float oc[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) oc[k] = pp[(c + k) * cstride];
#pragma unroll
    for (int k = 0; k < 8; ++k) o += w[c + k] * oc[k];
  }
  for (; c < nchunks; ++c) o += w[c] * pp[c * cstride];
  const float res = valid ? o / lsum[hh] : 0.f;
  vals[threadIdx.x] = res;
  if (out && row < M) out[(size_t)row * H + 256 * b + threadIdx.x] = res;
  __syncthreads();
  if (act && threadIdx.x < 32) {
    if (row < M) {
      float v[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) v[i] = vals[8 * threadIdx.x + i];
      quant_block_warp(v, row, b, H, act, nullptr, nullptr, nullptr, status);
    } else {
      zero_block_warp(row, b, act);
    }
  }
}

cudaError_t launch_attention(const AttnPlan& a, const KvView& kv, int layer, const uint8_t* qfrag,
                             int M, float* part, float* out, uint8_t* act, int32_t* status,
                             cudaStream_t st, bool pdl) {
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  const bool multi = a.chunk > kChunk;
  auto kern = multi ? attn_partial_kernel<true> : attn_partial_kernel<false>;
  static bool smem_attr[2] = {false, false};
  if (!smem_attr[multi]) {
    cudaError_t ea = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                          (int)attn_smem_bytes());
    if (ea != cudaSuccess) return ea;
    smem_attr[multi] = true;
  }
  cfg.gridDim = dim3(a.max_chunks, a.nkv, head_split(multi));
  cfg.blockDim = dim3(32 * warps_per_cta(multi));
  cfg.dynamicSmemBytes = attn_smem_bytes();
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  cudaError_t e = cudaLaunchKernelEx(&cfg, kern, reinterpret_cast<const uint4*>(qfrag),
                                     M, a.nq, a.nkv, a.chunk, kv, layer, part, (const int32_t*)status);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg2 = {};
  cfg2.gridDim = dim3(a.nq * 128 / 256, 16);
  cfg2.blockDim = dim3(256);
  cfg2.dynamicSmemBytes = sizeof(float) * (4 * (size_t)a.max_chunks + 2);
  cfg2.stream = st;
  cfg2.attrs = attr;
  cfg2.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg2, attn_merge_kernel, (const float*)part, M, a.nq, a.max_chunks,
                            a.chunk, (const int32_t*)kv.seq_len, out, act, status);
}

}  // namespace spec
