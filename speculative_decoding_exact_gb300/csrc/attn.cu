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
#include <cuda.h>

#include "common.cuh"
#include "internal.h"
#include "quant.cuh"

namespace spec {

constexpr int kChunk = 64;
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
// Shared memory of the partial kernel: a double buffer of K and V sub-chunks,
// each [d half (2)][64 keys][128 bytes] with the 16-byte chunks of a row
// permuted by the 128-byte swizzle of the tensor copies (chunk j of row r at
// j ^ (r % 8)), then the chunk's page ids (16 keys per page).  1 KB of slack
// aligns the buffers to the 1 KB swizzle period.
constexpr int kHalfBytes = kChunk * 128;              // one d half of a K or V sub-chunk
constexpr int kKvBufBytes = 2 * 2 * kHalfBytes;       // K and V of one buffer
constexpr size_t kKvSmemBytes = 1024 + 2 * (size_t)kKvBufBytes;
size_t attn_smem_bytes(int chunk) { return kKvSmemBytes + sizeof(int) * (size_t)(chunk / 16); }

// byte offset of 16-byte chunk j (0..7) of row r in a swizzled [rows][128 B] half
SPEC_DEV uint32_t swz(int r, int j) { return (uint32_t)(r * 128 + ((j ^ (r & 7)) << 4)); }

// 2-D tensor copy global -> shared: box at (x, y) of the map, completion on mbar
SPEC_DEV void tma_load_2d(void* dst_smem, const CUtensorMap* map, int x, int y, uint64_t* mbar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];\n" ::"r"(
          smem_u32(dst_smem)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(mbar))
      : "memory");
}

// The KV pool [num_pages][n_layers][K, V][n_kv][16 positions][128] bf16 seen as
// one 2-D tensor of 256-byte rows (row = ((page*n_layers + layer)*2 + kv)*n_kv
// + head, times 16, plus the position in the page); boxes of 16 rows x 64
// values (one d half of one page), 128-byte swizzle.
static cudaError_t make_kv_tmap(const KvView& kv, CUtensorMap* map) {
  using EncodeFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
  static EncodeFn encode = nullptr;
  if (!encode) {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
    if (e != cudaSuccess) return e;
    if (q != cudaDriverEntryPointSuccess || !fn) return cudaErrorNotSupported;
    encode = reinterpret_cast<EncodeFn>(fn);
  }
  const unsigned long long rows = (unsigned long long)kv.num_pages * kv.n_layers * 2 * kv.n_kv * 16;
  if (rows == 0 || rows >= (1ull << 31)) return cudaErrorInvalidValue;   // y coordinates are int32
  const cuuint64_t dims[2] = {128, rows};
  const cuuint64_t strides[1] = {256};
  const cuuint32_t box[2] = {64, 16};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, kv.pool, dims, strides, box, estr,
                            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

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
// split x into bf16 hi + bf16 lo (x - hi), packed pairs (x0 in the low half)
SPEC_DEV void split2(float x0, float x1, uint32_t& hi, uint32_t& lo) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(x0, x1);
  const __nv_bfloat162 l = __floats2bfloat162_rn(x0 - __low2float(h), x1 - __high2float(h));
  hi = *reinterpret_cast<const uint32_t*>(&h);
  lo = *reinterpret_cast<const uint32_t*>(&l);
}
// 2^x (PTX ex2.approx: relative error about 2^-22; 2^-inf = 0)
SPEC_DEV float exp2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;\n" : "=f"(y) : "f"(x));
  return y;
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
                    const __grid_constant__ CUtensorMap kvmap, int layer, float* __restrict__ part,
                    int32_t* status) {
  constexpr int kHeadSplit = head_split(MULTI);
  extern __shared__ __align__(128) uint8_t dsm[];
  uint8_t* kvs = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(dsm) + 1023) & ~(uintptr_t)1023);
  int* pg = reinterpret_cast<int*>(dsm + kKvSmemBytes);
  __shared__ __align__(8) uint64_t kvbar[2];     // K/V of buffer b landed (bulk copies)
  __shared__ int copy_ok;

  pdl_trigger();
  pdl_wait();
  const int chunk = blockIdx.x, kvh = blockIdx.y;
  const int group = nq / nkv;
  const int per = (group + kHeadSplit - 1) / kHeadSplit;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, t = lane & 3;
  const int key0 = chunk * chunk_keys;
  // status, length and the chunk's page ids in one round of loads
  const int32_t st = *status;
  const int len = *kv.seq_len;             // block appended: n_past + M
  for (int i = threadIdx.x; i < chunk_keys / 16; i += blockDim.x) {
    const int lp = key0 / 16 + i;
    pg[i] = lp < kv.max_seq_pages ? kv.page_table[lp] : -1;
  }
  if (threadIdx.x == 0) {
    mbar_init(&kvbar[0], 1);
    mbar_init(&kvbar[1], 1);
    fence_mbarrier_init();
  }
  __syncthreads();
  if (st & (SPEC_ST_TOKEN_RANGE | SPEC_ST_POOL_EMPTY | SPEC_ST_CTX_FULL)) return;
  const int n_past = len - M;
  if (key0 >= len) return;
  // sub-chunks with keys (exactly one when the chunk is one sub-chunk long)
  const int nsub = MULTI ? min(chunk_keys, len - key0 + kChunk - 1) / kChunk : 1;

  // ---- K, V sub-chunk sc -> shared buffer sc % 2: lanes 0..15 of warp 0 each
  // copy one d half of the K or V rows of one page (16 keys) with a tensor
  // copy; lane 0 arms the buffer's barrier with the bytes of the pages copied.
  // Pages past len or with an out-of-range id are not copied; their rows, and
  // the rows at or past len in a copied page, are zeroed once the copies have
  // landed (fix_sub).
  auto page_of = [&](int pos0) -> int {
    const int page = pos0 < len ? pg[(pos0 - key0) >> 4] : -1;
    return (page >= 0 && page < kv.num_pages) ? page : -1;
  };
  auto load_sub = [&](int sc) {
    if (warp != 0) return;
    uint8_t* buf = kvs + (size_t)(sc & 1) * kKvBufBytes;
    uint64_t* bar = &kvbar[sc & 1];
    const int ks0 = key0 + sc * kChunk;
    const int pp = (lane >> 2) & 3, which = (lane >> 1) & 1, half = lane & 1;
    const int page = page_of(ks0 + 16 * pp);
    const bool go = lane < 16 && page >= 0;
    const uint32_t ops = __popc(__ballot_sync(0xffffffffu, go));
    if (lane == 0) mbar_arrive_expect_tx(bar, ops * 2048u);
    if (go) {
      const int y = (((page * kv.n_layers + layer) * 2 + which) * kv.n_kv + kvh) * 16;
      tma_load_2d(buf + which * 2 * kHalfBytes + half * kHalfBytes + pp * 2048, &kvmap, 64 * half, y, bar);
    }
  };
  // rows of sub-chunk sc that must read as zero: keys at or past len, keys of a
  // page with an out-of-range id (CTA-uniform)
  auto sub_needs_fix = [&](int sc) -> bool {
    const int ks0 = key0 + sc * kChunk;
    if (ks0 + kChunk > len) return true;
#pragma unroll
    for (int pp = 0; pp < kChunk / 16; ++pp)
      if (page_of(ks0 + 16 * pp) < 0) return true;
    return false;
  };
  auto fix_sub = [&](int sc) {
    uint8_t* buf = kvs + (size_t)(sc & 1) * kKvBufBytes;
    const int ks0 = key0 + sc * kChunk;
    for (int i = threadIdx.x; i < kChunk * 4; i += blockDim.x) {     // (row, K/V, half)
      const int r = i >> 2, which = (i >> 1) & 1, half = i & 1;
      const int pos = ks0 + r;
      if (pos < len && page_of(ks0 + 16 * (r >> 4)) >= 0) continue;
      uint4* row = reinterpret_cast<uint4*>(buf + which * 2 * kHalfBytes + half * kHalfBytes + r * 128);
#pragma unroll
      for (int c16 = 0; c16 < 8; ++c16) row[c16] = make_uint4(0, 0, 0, 0);
    }
    fence_proxy_async();      // ordered before the tensor copies that later refill the buffer
  };

  const int hl = blockIdx.z * per + warp;          // head within the kv group
  const bool active = warp < per && hl < group;
  const int head = kvh * group + (active ? hl : 0);
  const uint4* Qf = qf + (size_t)head * 8 * 2 * 32;   // [8 ksteps][hi, lo][32 lanes]
  // scores in base-2 units: u = (q.k / sqrt(128)) * log2(e), p = 2^(u - max)
  const float c2 = 1.4426950408889634f / sqrtf(128.0f);

  // running per-row state (rows g and g+8): max, sum, unnormalised o
  float mrun[2] = {-INFINITY, -INFINITY}, lrun[2] = {0.f, 0.f};
  float o[16][4];
#pragma unroll
  for (int nd = 0; nd < 16; ++nd)
#pragma unroll
    for (int e = 0; e < 4; ++e) o[nd][e] = 0.f;

  load_sub(0);
  for (int sc = 0; sc < nsub; ++sc) {
    if (sc + 1 < nsub) load_sub(sc + 1);
    // one thread waits (bounded) for the buffer; the CTA barrier passes the
    // result and the landed rows to all threads
    if (threadIdx.x == 0) copy_ok = mbar_wait_ns(&kvbar[sc & 1], (sc >> 1) & 1, 2000000000ull) ? 1 : 0;
    __syncthreads();
    if (!copy_ok) {
      if (threadIdx.x == 0) {          // flag it; let the other buffer's copies land (bounded)
        atomicOr(status, SPEC_ST_DEVICE_WAIT);
        if (sc + 1 < nsub) mbar_wait_ns(&kvbar[(sc + 1) & 1], ((sc + 1) >> 1) & 1, 2000000000ull);
      }
      return;
    }
    if (sub_needs_fix(sc)) {
      fix_sub(sc);
      __syncthreads();
    }
    const uint8_t* Ks = kvs + (size_t)(sc & 1) * kKvBufBytes;
    const uint8_t* Vs = Ks + 2 * kHalfBytes;
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
          const int krow = 8 * nt + (lane & 7);   // d = 32 kp + 8 (lane / 8): half kp / 2
          ldsm_x4(b0, b1, b2, b3, Ks + (kp >> 1) * kHalfBytes + swz(krow, 4 * (kp & 1) + (lane >> 3)));
          mma16816_bf16(s[nt], qh0.x, qh0.y, qh0.z, qh0.w, b0, b1);
          mma16816_bf16(s[nt], ql0.x, ql0.y, ql0.z, ql0.w, b0, b1);
          mma16816_bf16(s[nt], qh1.x, qh1.y, qh1.z, qh1.w, b2, b3);
          mma16816_bf16(s[nt], ql1.x, ql1.y, ql1.z, ql1.w, b2, b3);
        }
      }

      // ---- mask, running max, p = 2^(u - max), rescale of the running state.
      // A sub-chunk whose keys all precede the block is visible to every row.
      const bool full = ks0 + kChunk - 1 <= n_past;
      float mx[2] = {-INFINITY, -INFINITY};
      if (full) {
#pragma unroll
        for (int nt = 0; nt < 8; ++nt)
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            s[nt][e] *= c2;
            mx[e >> 1] = fmaxf(mx[e >> 1], s[nt][e]);
          }
      } else {
        // key ks0 + 8nt + 2t + (e&1) is visible to row g + 8(e>>1) < M when
        // 8nt + (e&1) <= n_past + row - ks0 - 2t
        int lim[2];
#pragma unroll
        for (int r = 0; r < 2; ++r) lim[r] = (g + 8 * r < M) ? n_past + g + 8 * r - ks0 - 2 * t : -1;
#pragma unroll
        for (int nt = 0; nt < 8; ++nt)
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float v = (8 * nt + (e & 1) <= lim[e >> 1]) ? s[nt][e] * c2 : -INFINITY;
            s[nt][e] = v;
            mx[e >> 1] = fmaxf(mx[e >> 1], v);
          }
      }
      float alpha[2], mbase[2];
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], 1));
        mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], 2));
        const float mnew = fmaxf(mrun[r], mx[r]);
        alpha[r] = (mrun[r] == -INFINITY) ? 0.f : exp2_approx(mrun[r] - mnew);
        mrun[r] = mnew;
        mbase[r] = mnew == -INFINITY ? 0.f : mnew;    // a row with no visible key yet: p = 2^-inf = 0
      }
      float sum[2] = {0.f, 0.f};
#pragma unroll
      for (int nt = 0; nt < 8; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float p = exp2_approx(s[nt][e] - mbase[e >> 1]);
          s[nt][e] = p;
          sum[e >> 1] += p;
        }
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        sum[r] += __shfl_xor_sync(0xffffffffu, sum[r], 1);
        sum[r] += __shfl_xor_sync(0xffffffffu, sum[r], 2);
        lrun[r] = lrun[r] * alpha[r] + sum[r];
      }
      if (sc > 0) {
#pragma unroll
        for (int nd = 0; nd < 16; ++nd)
#pragma unroll
          for (int e = 0; e < 4; ++e) o[nd][e] *= alpha[e >> 1];
      }

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
          const int vrow = 16 * kk + (lane & 7) + 8 * ((lane >> 3) & 1);   // d = 16 np + 8 (lane / 16)
          ldsm_x4_t(b0, b1, b2, b3, Vs + (np >> 2) * kHalfBytes + swz(vrow, 2 * (np & 3) + (lane >> 4)));
          mma16816_bf16(o[2 * np], ph[0], ph[1], ph[2], ph[3], b0, b1);
          mma16816_bf16(o[2 * np], pl[0], pl[1], pl[2], pl[3], b0, b1);
          mma16816_bf16(o[2 * np + 1], ph[0], ph[1], ph[2], ph[3], b2, b3);
          mma16816_bf16(o[2 * np + 1], pl[0], pl[1], pl[2], pl[3], b2, b3);
        }
      }
    }
    if (sc + 1 < nsub) __syncthreads();     // the next prefetch overwrites this buffer
  }
  if (!active) return;

  // ---- partials: [chunk][head][row][128 o | max (base-2 units) | sum]
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
//   M = max_c m_c;  w_c = 2^(m_c - M) (maxima in base-2 units);  L = sum_c w_c l_c;
//   o = sum_c w_c o_c;
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
      const float w = (mc == -INFINITY) ? 0.f : exp2f(mc - m);
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
  alignas(64) CUtensorMap kvmap;
  cudaError_t em = make_kv_tmap(kv, &kvmap);
  if (em != cudaSuccess) return em;
  const bool multi = a.chunk > kChunk;
  auto kern = multi ? attn_partial_kernel<true> : attn_partial_kernel<false>;
  const size_t smem = attn_smem_bytes(a.chunk);
  static size_t smem_attr[2] = {0, 0};
  if (smem_attr[multi] < smem) {
    cudaError_t ea = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (ea != cudaSuccess) return ea;
    smem_attr[multi] = smem;
  }
  cfg.gridDim = dim3(a.max_chunks, a.nkv, head_split(multi));
  cfg.blockDim = dim3(32 * warps_per_cta(multi));
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  cudaError_t e = cudaLaunchKernelEx(&cfg, kern, reinterpret_cast<const uint4*>(qfrag),
                                     M, a.nq, a.nkv, a.chunk, kv, kvmap, layer, part, status);
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
