// attn.cu — verify attention of k+1 query rows against the paged bf16 KV cache.
//
// Row i of the block sits at position n_past + i and sees positions
// 0..n_past+i (the carried-frontier row first, then the drafts: Muser book
// Ch. 33 §33.7).  Query head h reads KV head h / (n_q/n_kv).
// s = q.k / sqrt(head_dim), softmax over the visible positions, o = sum p v.
//
// Decomposition (flash-decoding): CTA (chunk c, kv head, tile) takes the keys
// [c*C, (c+1)*C) for up to 8 query heads of that kv head.  The 8 heads x 16
// block rows are the 128 rows of tcgen05 MMAs:
//   S[128 x B keys]   = Q[128 x 128 d] . K^T      (A, B in shared memory)
//   O[128 x 128 d]   += P[128 x B keys] . V       (A = P in TMEM, B = V)
// walking the chunk in sub-chunks of B = 64 or 128 keys with a running
// (max, sum) per row and O accumulated in TMEM (online softmax), and writes
// the partials.  C is B times the sub-chunks per chunk, set from max_ctx
// alone so that one launch is one wave of at most kCtaBudget CTAs.  A merge
// kernel combines the chunks in chunk order, normalises, and quantises the
// rows for the output projection.  Chunk and sub-chunk boundaries are fixed by max_ctx and masked
// keys contribute exact zeros, so row i's result is the same for every M
// (batch-height invariance: "The Two-Fifteen That Wasn't").
//
// Precision: K and V are exact bf16; q and p are split into bf16 hi + lo parts
// (two MMAs each) so the products carry ~16 significant bits; accumulation is
// fp32.
#include <cuda.h>

#include "common.cuh"
#include "internal.h"
#include "quant.cuh"

namespace spec {

constexpr int kCtaBudget = 148;            // CTAs of one partial launch at most
constexpr int kHeadsPerTile = 8;           // 8 heads x 16 rows = 128 MMA rows
constexpr int kPartStride = 130;           // floats per partial row: o[128], max, sum
constexpr int kQHalfBytes = 128 * 128;     // 16 KB
constexpr int kQTileBytes = 4 * kQHalfBytes;   // 64 KB

// The layout of one sub-chunk size B (64 or 128 keys): its K/V ring in shared
// memory (K then V, each [d half][B keys][128 B]; 3 slots of 32 KB or 2 of
// 64 KB), and TMEM columns S (two buffers of B), P hi and lo (B/2 each), O
// (128) out of 512.  Each row thread holds B/2 score columns.
template <int B>
struct Sub {
  static_assert(B == 64 || B == 128, "sub-chunk of 64 or 128 keys");
  static constexpr int kKeys = B;
  static constexpr int kPages = B / 16;
  static constexpr int kCols = B / 2;
  static constexpr int kKvBufs = B == 64 ? 3 : 2;
  static constexpr int kHalfBytes = B * 128;
  static constexpr int kKvBufBytes = 4 * kHalfBytes;
  static constexpr uint32_t kTmS = 0, kTmP = 2 * B, kTmO = 3 * B;
  static constexpr size_t kSmemFixed = 1024 + kQTileBytes + (size_t)kKvBufs * kKvBufBytes;
  static_assert(128 * kPartStride * 4 <= kQTileBytes + kKvBufBytes, "partials staging");
  static_assert(kTmO + 128 <= 512, "TMEM columns");
};
int sub_bufs(int sub) { return sub == 64 ? Sub<64>::kKvBufs : Sub<128>::kKvBufs; }

AttnPlan make_attn_plan(int nq, int nkv, int dh, int max_ctx) {
  AttnPlan a;
  a.nq = nq;
  a.nkv = nkv;
  a.dh = dh;
  a.max_ctx = max_ctx;
  a.group = nkv > 0 ? nq / nkv : 0;
  a.tiles = (a.group + kHeadsPerTile - 1) / kHeadsPerTile;
  const int per_chunk = nkv * (a.tiles > 0 ? a.tiles : 1);
  const int budget = kCtaBudget / per_chunk > 0 ? kCtaBudget / per_chunk : 1;
  // Sub-chunks of 128 keys halve the hand-offs per key (one QK MMA of N =
  // 128 where 64-key sub-chunks need two); measured on the verify step at a
  // 32k context, 157.5 against 166.6 steps/s.  A chunk that would hold one
  // such sub-chunk takes two of 64 instead, which overlap (2k: 223.2 against
  // 222.4 steps/s).
  auto subs_of = [&](int b) {
    const int n = max_ctx > 0 ? (max_ctx + b - 1) / b : 1;
    return (n + budget - 1) / budget;                          // sub-chunks per chunk
  };
  a.sub = subs_of(128) > 1 ? 128 : 64;
  a.chunk = a.sub * subs_of(a.sub);
  a.max_chunks = (max_ctx + a.chunk - 1) / a.chunk;
  if (a.max_chunks < 1) a.max_chunks = 1;
  // Measured on the 52-block verify step: copying before the wait gains 0.4 %
  // at a 2k context (2 sub-chunks per chunk); at 16k (15 per chunk) the later
  // signal of the QKV kernel cost 1 % and the early copies gained nothing.
  a.early = a.chunk <= sub_bufs(a.sub) * a.sub;
  return a;
}

// Shared memory of the partial kernel (1 KB aligned; the 128-byte swizzle
// repeats every 1 KB): the Q tile (hi, lo; each [d half][128 rows][128 B]),
// the K/V ring of Sub<B>, then the chunk's page ids.  In every [rows][128 B]
// block the 16-byte chunk j of row r sits at j ^ (r % 8).  The partials of the
// tile are staged over the Q tile and the first ring slot once every MMA has
// completed.
size_t attn_smem_bytes(const AttnPlan& a) {
  return (a.sub == 64 ? Sub<64>::kSmemFixed : Sub<128>::kSmemFixed) + sizeof(int) * (size_t)(a.chunk / 16);
}
constexpr int kTmCols = 512;

// warps: 0-7 own the tile rows, two threads per row (warp w: rows 32(w%4)..,
// S columns (B/2)(w/4).., O columns 64(w/4)..) for the softmax, the O rescale
// and the partials; 8 issues the QK MMAs, 9 the PV MMAs, 10 the K copies and
// 11 the V copies.  Per-CTA timelines at a 32k context put each issuing role
// on the critical path when another role shared its warp: the 16 QK and 8 PV
// MMAs of a 64-key sub-chunk took about 1,500 cycles of one warp's issue, and
// the 16 tensor copies about 1,000.
constexpr int kRowWarps = 8;
constexpr int kRowThreads = 32 * kRowWarps;
constexpr int kAttnWarps = kRowWarps + 4;
constexpr int kWarpQk = kRowWarps, kWarpPv = kRowWarps + 1, kWarpKc = kRowWarps + 2, kWarpVc = kRowWarps + 3;
constexpr uint64_t kAttnWaitNs = 2000000000ull;

size_t qtile_bytes(const AttnPlan& a) { return (size_t)a.nkv * a.tiles * kQTileBytes; }

size_t attn_partial_floats(const AttnPlan& a, int max_rows) {
  (void)max_rows;
  return (size_t)a.max_chunks * a.nq * 16 * kPartStride;
}

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

// The sliding-window rings [n_swa][K, V][n_kv][R][128] bf16 as one 2-D tensor
// of 256-byte rows (row = ((s*2 + kv)*n_kv + head)*R + slot); the same boxes.
// R is a multiple of 16, so a 16-row box never straddles two rings.
static cudaError_t make_ring_tmap(const KvView& kv, CUtensorMap* map) {
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
  const unsigned long long rows = (unsigned long long)swa_layers(kv) * 2 * kv.n_kv * kv.swa_rows;
  if (rows == 0 || rows >= (1ull << 31) || kv.swa_rows % 16) return cudaErrorInvalidValue;
  const cuuint64_t dims[2] = {128, rows};
  const cuuint64_t strides[1] = {256};
  const cuuint32_t box[2] = {64, 16};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, kv.swa_ring, dims, strides, box, estr,
                            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// 2^x (PTX ex2.approx: relative error about 2^-22; 2^-inf = 0)
SPEC_DEV float exp2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;\n" : "=f"(y) : "f"(x));
  return y;
}
// split x into bf16 hi + bf16 lo, packed pairs (x0 in the low half): hi is x
// with the low 16 bits dropped (exact), lo = x - hi (exact in fp32, below
// 2^-7 |x|) rounded to bf16, so hi + lo carries about 16 significant bits
SPEC_DEV void split2(float x0, float x1, uint32_t& hi, uint32_t& lo) {
  const uint32_t b0 = __float_as_uint(x0), b1 = __float_as_uint(x1);
  hi = __byte_perm(b0, b1, 0x7632);
  const __nv_bfloat162 l = __floats2bfloat162_rn(x0 - __uint_as_float(b0 & 0xFFFF0000u),
                                                 x1 - __uint_as_float(b1 & 0xFFFF0000u));
  lo = *reinterpret_cast<const uint32_t*>(&l);
}
SPEC_DEV void tmem_st16(uint32_t taddr, const uint32_t* r) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};\n" ::"r"(
          taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
      "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]));
}
SPEC_DEV void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];\n"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
}
// shared-memory descriptor of a 128-byte-swizzled operand: lbo and sbo in bytes
SPEC_DEV uint64_t desc_sw128(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  return smem_desc(saddr, lbo, sbo) | ((uint64_t)2 << 61);
}
// D[tmem] (+)= A[smem] * B[smem]^T, kind::f16, issued by one thread
SPEC_DEV void mma_f16_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.u32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate));
}
// bulk copy shared -> global (bulk group of this thread)
SPEC_DEV void bulk_s2g(void* dst, const void* src_smem, uint32_t bytes) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;\n" ::"l"(dst),
               "r"(smem_u32(src_smem)), "r"(bytes)
               : "memory");
  asm volatile("cp.async.bulk.commit_group;\n" ::: "memory");
  asm volatile("cp.async.bulk.wait_group.read 0;\n" ::: "memory");
}

// ---- Q tiles from fp32 q [M][nq][128] (rows >= M zero), the standalone path
__global__ void q_to_tile_kernel(const float* __restrict__ q, int M, int nq, int group, int tiles,
                                 uint8_t* qtile) {
  pdl_trigger();
  pdl_wait();
  const int row = blockIdx.y;
  const int col = blockIdx.x * blockDim.x + threadIdx.x;
  if (col >= nq * 128) return;
  write_qtile(qtile, row, col >> 7, col & 127, row < M ? q[(size_t)row * nq * 128 + col] : 0.f, group,
              tiles);
}

cudaError_t launch_q_to_tile(const float* q, int M, const AttnPlan& a, uint8_t* qtile, cudaStream_t st,
                             bool pdl) {
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((a.nq * 128 + 255) / 256, 16);
  cfg.blockDim = dim3(256);
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, q_to_tile_kernel, q, M, a.nq, a.group, a.tiles, qtile);
}

// ---------------------------------------------------------------------------
// partials: grid (chunk, kv head, tile), kAttnWarps warps.
// ---------------------------------------------------------------------------
template <bool kTree, int kSub>
__global__ void __launch_bounds__(kAttnWarps * 32, 1)
attn_partial_kernel(const uint8_t* __restrict__ qtile, int M, int nq, int nkv, int group, int tiles,
                    int chunk_keys, KvView kv, const __grid_constant__ CUtensorMap kvmap, int layer,
                    const uint64_t* __restrict__ tree_mask, const int32_t* __restrict__ tree_base,
                    float* __restrict__ part, int32_t* status, int early, int ring_s) {
  using S = Sub<kSub>;
  constexpr int kChunk = S::kKeys, kPages = S::kPages, kCols = S::kCols, kKvBufs = S::kKvBufs;
  constexpr int kHalfBytes = S::kHalfBytes, kKvBufBytes = S::kKvBufBytes;
  constexpr uint32_t kTmS = S::kTmS, kTmP = S::kTmP, kTmO = S::kTmO;
  constexpr size_t kSmemFixed = S::kSmemFixed;
  extern __shared__ __align__(128) uint8_t dsm[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(dsm) + 1023) & ~(uintptr_t)1023);
  uint8_t* qs = sm;                                    // Q tile: hi [0, 32K), lo [32K, 64K)
  uint8_t* kvb = sm + kQTileBytes;                     // ring slot b at kvb + b * kKvBufBytes
  int* pg = reinterpret_cast<int*>(dsm + kSmemFixed);
  __shared__ uint32_t tmem_slot;
  __shared__ __align__(8) uint64_t q_full, k_full[kKvBufs], v_full[kKvBufs], k_free[kKvBufs], v_free[kKvBufs],
      s_full[2], s_free[2], p_full, pv_done;

  __shared__ float rowmax[2][2][128];       // [sub-chunk parity][column half][row]
  __shared__ float lpart[2][128];           // [column half][row]
  __shared__ int proceed, len_sh, tb_sh, key0_sh;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int chunk = blockIdx.x, kvh = blockIdx.y, tile = blockIdx.z;
  // a sliding-window layer (ring_s >= 0) reads ring ring_s; its chunks start
  // at the page of the first key any block row sees
  const bool ring = ring_s >= 0;
  // barriers and TMEM do not depend on the previous kernel
  if (warp == 0) tmem_alloc(&tmem_slot, kTmCols);
  if (tid == 0) {
    mbar_init(&q_full, 1);
    for (int b = 0; b < kKvBufs; ++b) {
      mbar_init(&k_full[b], 1);
      mbar_init(&v_full[b], 1);
      mbar_init(&k_free[b], 1);                  // K read by the QK MMAs
      mbar_init(&v_free[b], 1);                  // V read by the PV MMAs
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&s_full[b], 1);
      mbar_init(&s_free[b], kRowThreads);
    }
    mbar_init(&p_full, kRowThreads);
    mbar_init(&pv_done, 1);
    fence_mbarrier_init();
  }
  if ((warp == kWarpKc || warp == kWarpVc) && lane == 0)
    asm volatile("prefetch.tensormap [%0];\n" ::"l"(reinterpret_cast<uint64_t>(&kvmap)) : "memory");
  // Status, length and page ids were written by the reserve at the start of
  // the step.  With `early` the kernel launched before this one signals its
  // dependents only after its own dependency wait, so the reserve and
  // everything before it have completed when this kernel starts, and they
  // are read from L2 (.cg) before the wait; otherwise after it.  The abort
  // bits are the reserve's.
  if (!early) {
    pdl_trigger();
    pdl_wait();
  }
  {
    const int32_t st = __ldcg(status);
    const int len0 = __ldcg(kv.seq_len);
    const int k0 = (ring ? (max(0, len0 - M - kv.swa_window + 1) & ~15) : 0) + chunk * chunk_keys;
    if (!ring)
      for (int i = tid; i < chunk_keys / 16; i += blockDim.x) {
        const int lp = k0 / 16 + i;
        pg[i] = lp < kv.max_seq_pages ? __ldcg(kv.page_table + lp) : -1;
      }
    if (tid == 0) {
      proceed = !(st & kStepAbort) && k0 < len0;
      len_sh = len0;
      key0_sh = k0;
      tb_sh = kTree ? __ldcg(tree_base) : 0;
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_slot;
  const int len = len_sh;                  // block appended: n_past + M
  const int n_past = len - M;
  const int key0 = key0_sh;
  // sliding window: row r sees keys >= wlo + r; keys below wlo no row sees
  const int wlo = ring ? n_past - kv.swa_window + 1 : 0;
  // token tree: the tree's first position (node 0); a tree of more than 16
  // nodes runs in passes of up to 16 rows, and n_past is this pass's first
  // row, so earlier passes' nodes lie between the two
  const int tb = kTree ? tb_sh : n_past;
  // sub-chunks with keys (0 when the CTA has nothing to do)
  const int nsub = proceed ? min(chunk_keys, len - key0 + kChunk - 1) / kChunk : 0;
  // The first sub-chunks whose keys all precede the block (rows of earlier
  // steps, which the kernel before this one does not write) are copied
  // before the wait; the block's own K/V rows are written by that kernel.
  int npre = 0;
  while (early && npre < min(nsub, kKvBufs) && key0 + (npre + 1) * kChunk <= n_past) ++npre;

  // page id of the page holding pos0 (a multiple of 16), -1 past len or out
  // of range; a ring's page is its 16 slots from (pos0 mod R)
  auto page_of = [&](int pos0) -> int {
    if (ring) return pos0 < len ? (pos0 >> 4) % (kv.swa_rows >> 4) : -1;
    const int page = pos0 < len ? pg[(pos0 - key0) >> 4] : -1;
    return (page >= 0 && page < kv.num_pages) ? page : -1;
  };
  // copy warps: the K (warp kWarpKc) or V rows of sub-chunk sc into ring slot
  // sc % kKvBufs; lane l < 2 * kPages takes page l / 2, d half l % 2
  const int which = warp == kWarpVc ? 1 : 0;
  uint64_t* kv_full_w = which ? v_full : k_full;
  uint64_t* kv_free_w = which ? v_free : k_free;
  auto issue_kv = [&](int sc) {
    const int b = sc % kKvBufs;
    uint8_t* buf = kvb + (size_t)b * kKvBufBytes;
    const int ks0 = key0 + sc * kChunk;
    const int pp = (lane >> 1) % kPages, half = lane & 1;
    const int page = page_of(ks0 + 16 * pp);
    const bool go = lane < 2 * kPages && page >= 0;
    const uint32_t ops = __popc(__ballot_sync(0xffffffffu, go));
    if (lane == 0) mbar_arrive_expect_tx(&kv_full_w[b], ops * 2048u);
    if (go) {
      const int y = ring ? ((ring_s * 2 + which) * kv.n_kv + kvh) * kv.swa_rows + 16 * page
                         : (((page * kv.n_layers + layer) * 2 + which) * kv.n_kv + kvh) * 16;
      tma_load_2d(buf + which * 2 * kHalfBytes + half * kHalfBytes + pp * 2048, &kvmap, 64 * half, y,
                  &kv_full_w[b]);
    }
  };
  if (warp == kWarpKc || warp == kWarpVc)
    for (int sc = 0; sc < npre; ++sc) issue_kv(sc);
  if (early) {
    pdl_trigger();
    pdl_wait();
  }

  if (warp == kWarpKc || warp == kWarpVc) {
    // ------------------------------------------------------------ copies
    if (lane == 0 && which == 0) {
      mbar_arrive_expect_tx(&q_full, (uint32_t)kQTileBytes);
      bulk_g2s(qs, qtile + (size_t)(kvh * tiles + tile) * kQTileBytes, (uint32_t)kQTileBytes, &q_full);
    }
    bool ok = true;
    int issued = npre;
    for (int sc = npre; sc < nsub; ++sc) {
      const int b = sc % kKvBufs;
      if (sc >= kKvBufs)
        ok = __all_sync(0xffffffffu, mbar_wait_ns(&kv_free_w[b], ((sc / kKvBufs) - 1) & 1, kAttnWaitNs));
      if (!ok) break;
      issue_kv(sc);
      issued = sc + 1;
    }
    if (!ok && lane == 0) atomicOr(status, SPEC_ST_DEVICE_WAIT);
    // no copy may still be writing shared memory when the CTA exits
    if (lane == 0) {
      if (which == 0) mbar_wait_ns(&q_full, 0, kAttnWaitNs);
      for (int u = max(0, issued - kKvBufs); u < issued; ++u)
        mbar_wait_ns(&kv_full_w[u % kKvBufs], (u / kKvBufs) & 1, kAttnWaitNs);
    }
  } else if (warp == kWarpQk) {
    // ------------------------------------------------------------ QK issue
    // S[sc % 2] = Q . K(sc)^T: 8 d steps of 16, hi and lo parts of Q.
    // D f32 (bit 4), A and B bf16 (bits 7, 10), N >> 3 at 17, M >> 4 at 24.
    // The descriptors are built once; a step adds its byte offset / 16 to
    // the start-address field (addresses stay below 256 KB: no carry).
    constexpr uint32_t kIdQK =
        (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(kChunk >> 3) << 17) | ((128u >> 4) << 24);
    const uint32_t tm = __shfl_sync(0xffffffffu, tmem, 0);
    const uint64_t dq0 = desc_sw128(__shfl_sync(0xffffffffu, smem_u32(qs), 0), 16, 1024);
    const uint64_t dk0 = desc_sw128(__shfl_sync(0xffffffffu, smem_u32(kvb), 0), 16, 1024);
    bool ok = __all_sync(0xffffffffu, mbar_wait_ns(&q_full, 0, kAttnWaitNs));
    int last = -1;
    for (int sc = 0; ok && sc < nsub; ++sc) {
      const int b = sc % kKvBufs, sb = sc & 1;
      bool w = mbar_wait_ns(&k_full[b], (sc / kKvBufs) & 1, kAttnWaitNs);
      if (sc >= 2) w = w && mbar_wait_ns(&s_free[sb], ((sc >> 1) - 1) & 1, kAttnWaitNs);
      ok = __all_sync(0xffffffffu, w);
      if (!ok) break;
      tc_fence_after();
      if (elect_one()) {
        const uint64_t dk = dk0 + (uint64_t)((b * kKvBufBytes) >> 4);
        const uint32_t d = tm + kTmS + (uint32_t)kChunk * sb;
#pragma unroll
        for (int ks = 0; ks < 8; ++ks)
#pragma unroll
          for (int part = 0; part < 2; ++part)
            mma_f16_ss(d, dq0 + (uint64_t)((part * 2 * kQHalfBytes + (ks >> 2) * kQHalfBytes + (ks & 3) * 32) >> 4),
                       dk + (uint64_t)(((ks >> 2) * kHalfBytes + (ks & 3) * 32) >> 4), kIdQK, (ks | part) != 0);
        mma_commit(&s_full[sb]);
        mma_commit(&k_free[b]);
      }
      __syncwarp();
      last = sc;
    }
    if (!ok && lane == 0) atomicOr(status, SPEC_ST_DEVICE_WAIT);
    // TMEM is released at the end: this warp's MMAs must have finished
    if (last >= 0) mbar_wait_ns(&s_full[last & 1], (last >> 1) & 1, kAttnWaitNs);
  } else if (warp == kWarpPv) {
    // ------------------------------------------------------------ PV issue
    // O (+)= P . V(sc): key steps of 16, hi and lo parts of P; V (the B
    // operand) MN-major (bit 16): lbo = the d-half stride, sbo = 1 KB between
    // 8-key groups
    constexpr uint32_t kIdPV =
        (1u << 4) | (1u << 7) | (1u << 10) | (1u << 16) | ((128u >> 3) << 17) | ((128u >> 4) << 24);
    const uint32_t tm = __shfl_sync(0xffffffffu, tmem, 0);
    const uint64_t dv0 = desc_sw128(__shfl_sync(0xffffffffu, smem_u32(kvb), 0) + 2 * kHalfBytes, kHalfBytes, 1024);
    bool ok = true;
    int last = -1;
    for (int sc = 0; ok && sc < nsub; ++sc) {
      const int b = sc % kKvBufs;
      ok = __all_sync(0xffffffffu, mbar_wait_ns(&p_full, sc & 1, kAttnWaitNs) &&
                                       mbar_wait_ns(&v_full[b], (sc / kKvBufs) & 1, kAttnWaitNs));
      if (!ok) break;
      tc_fence_after();
      if (elect_one()) {
        const uint64_t dv = dv0 + (uint64_t)((b * kKvBufBytes) >> 4);
#pragma unroll
        for (int kk = 0; kk < kChunk / 16; ++kk)
#pragma unroll
          for (int part = 0; part < 2; ++part)
            mma_f16_ts(tm + kTmO, tm + kTmP + (uint32_t)(kChunk / 2) * part + 8u * kk,
                       dv + (uint64_t)((kk * 2048) >> 4), kIdPV, (sc | kk | part) != 0);
        mma_commit(&pv_done);
        mma_commit(&v_free[b]);
      }
      __syncwarp();
      last = sc;
    }
    if (!ok && lane == 0) atomicOr(status, SPEC_ST_DEVICE_WAIT);
    if (last >= 0) mbar_wait_ns(&pv_done, last & 1, kAttnWaitNs);
  } else {
    // ------------------------------------------------------------ tile rows
    const int r = 32 * (warp & 3) + lane;               // tile row = TMEM lane
    const int h = warp >> 2;                            // S columns kCols*h.., O columns 64h..
    const int hl = tile * kHeadsPerTile + (r >> 4);     // head within the kv group
    const int row = r & 15;                             // block row
    const bool live = hl < group && row < M;
    // token tree: the tree nodes this row sees (bit j = node j: its
    // ancestors and itself); the causal step sees rows 0..row
    const uint64_t tm = (kTree && live) ? tree_mask[row] : 0ull;
    const uint32_t lane_base = (uint32_t)(32 * (warp & 3)) << 16;
    const float c2 = 1.4426950408889634f / sqrtf(128.0f);   // log2(e) / sqrt(d)
    float mref = -INFINITY, lsum = 0.f;
    bool ok = true;
    // Every row thread passes the same named barriers in the same order: a
    // failed wait is carried to the next barrier (bar.red.and), where all
    // 256 threads leave together.
    for (int sc = 0; sc < nsub; ++sc) {
      const int sb = sc & 1, b = sc % kKvBufs;
      const int ks0 = key0 + sc * kChunk;
      const bool got = ok && __all_sync(0xffffffffu, mbar_wait_ns(&s_full[sb], (sc >> 1) & 1, kAttnWaitNs));
      float s[kCols];
      if (got) {
        tc_fence_after();
#pragma unroll
        for (int q = 0; q < kCols / 32; ++q) {
          uint32_t u[32];
          tmem_ld32(tmem + lane_base + kTmS + (uint32_t)kChunk * sb + (uint32_t)kCols * h + 32u * q, u);
          tmem_wait_ld();
#pragma unroll
          for (int c = 0; c < 32; ++c) s[32 * q + c] = __uint_as_float(u[c]);
        }
        tc_fence_before();
        mbar_arrive(&s_free[sb]);
      } else {
#pragma unroll
        for (int c = 0; c < kCols; ++c) s[c] = 0.f;
      }
      // pages of this sub-chunk: a key of a page past len or with an
      // out-of-range id is masked (and its V row zeroed below)
      bool pok[kPages];
      bool allpages = true;
#pragma unroll
      for (int pp = 0; pp < kPages; ++pp) {
        pok[pp] = page_of(ks0 + 16 * pp) >= 0;
        allpages = allpages && pok[pp];
      }
      const bool full = ks0 + kChunk - 1 <= tb && allpages && (!ring || ks0 >= wlo + M - 1);
      // scores in base-2 units, masked -> -inf.  A row past the block or a
      // head past the group is never stored: it takes the unmasked path too
      // (its q is zero), so that a warp with such rows does not split between
      // the two paths.  Measured at a 32k context: the second tile of a KV
      // head (5 heads, rows 80-127 dead) took 50 us against 32 us for the
      // first while its dead rows ran the masked path.
      float mx4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
      if (full || !live) {
#pragma unroll
        for (int c = 0; c < kCols; ++c) {
          s[c] *= c2;
          mx4[c & 3] = fmaxf(mx4[c & 3], s[c]);
        }
      } else {
        // tree: key ks0 + kCols*h + c is visible when it precedes the tree
        // (and the row is live), or when it is node rel = base + c with bit
        // rel of tm set, and its page is valid: bit c of vm
        const int lim = live ? n_past + row - ks0 : -1;
        const int lim_lo = ring ? wlo + row - ks0 : -(1 << 30);   // the window's first key
        uint64_t vm = 0ull;
        if (kTree) {
          const int base = ks0 + kCols * h - tb;
          const int nold = min(kCols, max(0, -base));
          const uint64_t mold = !live ? 0ull : (nold >= 64 ? ~0ull : (1ull << nold) - 1ull);
          const uint64_t blk = base >= 0 ? (base < 64 ? tm >> base : 0ull) : (-base < 64 ? tm << -base : 0ull);
          uint64_t pm = 0ull;
#pragma unroll
          for (int pp = 0; pp < kPages / 2; ++pp)
            if (pok[(kPages / 2) * h + pp]) pm |= 0xffffull << (16 * pp);
          vm = (mold | blk) & pm;
        }
#pragma unroll
        for (int c = 0; c < kCols; ++c) {
          const int key = kCols * h + c;
          // causal: key ks0 + key is visible to row when key <= n_past + row - ks0
          const bool vis = kTree ? ((vm >> c) & 1ull) != 0 : (key <= lim && key >= lim_lo && pok[key >> 4]);
          s[c] = vis ? s[c] * c2 : -INFINITY;
          mx4[c & 3] = fmaxf(mx4[c & 3], s[c]);
        }
      }
      // row max over both column halves (exchanged through shared memory)
      rowmax[sb][h][r] = fmaxf(fmaxf(mx4[0], mx4[1]), fmaxf(mx4[2], mx4[3]));
      ok = named_bar_and(1, kRowThreads, got);
      if (!ok) break;                                   // all row threads together
      const float mx = fmaxf(rowmax[sb][0][r], rowmax[sb][1][r]);
      // the reference max moves only when a score exceeds it by more than 8
      // (p <= 2^8): O is rescaled rarely.  Both threads of a row take the
      // same decision.
      float alpha = 1.f;
      if (mx > mref + 8.f) {
        alpha = mref == -INFINITY ? 0.f : exp2_approx(mref - mx);
        mref = mx;
        lsum *= alpha;
      }
      const float base = mref == -INFINITY ? 0.f : mref;
      float ps4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int c = 0; c < kCols; c += 2) {
        s[c] = exp2_approx(s[c] - base);                // p, in place
        s[c + 1] = exp2_approx(s[c + 1] - base);
        ps4[(c >> 1) & 3] += s[c] + s[c + 1];
      }
      lsum += (ps4[0] + ps4[1]) + (ps4[2] + ps4[3]);
      // P(sc) may be written, and O rescaled, once P.V(sc-1) has finished
      if (sc > 0) {
        ok = __all_sync(0xffffffffu, mbar_wait_ns(&pv_done, (sc - 1) & 1, kAttnWaitNs));
        if (!ok) continue;                              // carried to the next barrier
        tc_fence_after();
        if (__any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll 1
          for (int q = 0; q < 2; ++q) {
            uint32_t o[32];
            const uint32_t oa = tmem + lane_base + kTmO + 64u * h + 32u * q;
            tmem_ld32(oa, o);
            tmem_wait_ld();
#pragma unroll
            for (int c = 0; c < 32; ++c) o[c] = __float_as_uint(__uint_as_float(o[c]) * alpha);
            tmem_st32(oa, o);
          }
        }
      }
      // V rows of keys that must read as zero (past len, bad page id, below
      // every row's window), once the V copies of this buffer have landed
      if (ks0 + kChunk > len || !allpages || (ring && ks0 < wlo)) {
        if (!__all_sync(0xffffffffu, mbar_wait_ns(&v_full[b], (sc / kKvBufs) & 1, kAttnWaitNs))) {
          ok = false;
          continue;                                     // carried to the next barrier
        }
        uint8_t* vb = kvb + (size_t)b * kKvBufBytes + 2 * kHalfBytes;
#pragma unroll 1
        for (int i = 128 * h + r; i < kChunk * 16; i += kRowThreads) {   // (key, d half, 16-byte chunk)
          const int c = i >> 4, half = (i >> 3) & 1, ch = i & 7;
          if (ks0 + c < len && pok[c >> 4] && (!ring || ks0 + c >= wlo)) continue;
          *reinterpret_cast<uint4*>(vb + half * kHalfBytes + c * 128 + ch * 16) = make_uint4(0, 0, 0, 0);
        }
        fence_proxy_async();
      }
      // P hi / lo as bf16 pairs: the keys kCols*h + 32q .. at columns
      // (kCols/2)*h + 16q .. of each half
#pragma unroll
      for (int q = 0; q < kCols / 32; ++q) {
        uint32_t ph[16], pl[16];
#pragma unroll
        for (int c = 0; c < 16; ++c) split2(s[32 * q + 2 * c], s[32 * q + 2 * c + 1], ph[c], pl[c]);
        tmem_st16(tmem + lane_base + kTmP + (uint32_t)(kCols / 2) * h + 16u * q, ph);
        tmem_st16(tmem + lane_base + kTmP + (uint32_t)(kChunk / 2) + (uint32_t)(kCols / 2) * h + 16u * q, pl);
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(&p_full);
    }
    if (!ok && r == 0 && h == 0) atomicOr(status, SPEC_ST_DEVICE_WAIT);
    // ---- partials of the tile: [chunk][head][row][o 128 | max (base 2) | sum]
    const int nrows = min(kHeadsPerTile, group - tile * kHeadsPerTile) * 16;
    const bool done = ok && nsub > 0 && __all_sync(0xffffffffu, mbar_wait_ns(&pv_done, (nsub - 1) & 1, kAttnWaitNs));
    lpart[h][r] = lsum;
    if (done) {
      tc_fence_after();
      float* stage = reinterpret_cast<float*>(sm) + (size_t)r * kPartStride + 64 * h;
#pragma unroll 1
      for (int q = 0; q < 2; ++q) {
        uint32_t o[32];
        tmem_ld32(tmem + lane_base + kTmO + 64u * h + 32u * q, o);
        tmem_wait_ld();
        if (r < nrows) {
#pragma unroll
          for (int c = 0; c < 32; c += 2)
            *reinterpret_cast<float2*>(stage + 32 * q + c) =
                make_float2(__uint_as_float(o[c]), __uint_as_float(o[c + 1]));
        }
      }
    }
    // every row's sum = its two column halves, in that order
    const bool all_done = named_bar_and(1, kRowThreads, done);
    if (all_done && h == 0 && r < nrows)
      *reinterpret_cast<float2*>(reinterpret_cast<float*>(sm) + (size_t)r * kPartStride + 128) =
          make_float2(mref, lpart[0][r] + lpart[1][r]);
    fence_proxy_async();
    if (named_bar_and(1, kRowThreads, all_done) && r == 0 && h == 0) {
      float* dst = part + (((size_t)chunk * nq + (size_t)kvh * group + tile * kHeadsPerTile) * 16) * kPartStride;
      bulk_s2g(dst, sm, (uint32_t)(nrows * kPartStride * 4));
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmCols);
  }
}

// merge: grid (nq*128/256 blocks, 16 rows), 256 threads = 2 heads x 128 dims.
// For row i the chunks 0 .. (n_past+i)/C are combined:
//   M = max_c m_c;  w_c = 2^(m_c - M) (maxima in base-2 units);  L = sum_c w_c l_c;
//   o = sum_c w_c o_c;
// out = o / L.  Warp hh (one per head) computes M, the weights and L with
// warp shuffles in a fixed butterfly order; o is summed in chunk order.  The
// chunk count depends on the row's position only, so the result is the same
// for every M.  The o values of the first kMergeBatch chunks, the (max, sum)
// pairs, the status and the length are all loaded in one round: the o loads
// do not depend on the weights, and chunks past the row's count are loaded
// but not used.
constexpr int kMergeBatch = 24;

__global__ void __launch_bounds__(256)
attn_merge_kernel(const float* __restrict__ part, int M, int nq, int max_chunks, int chunk_keys,
                  const int32_t* seq_len, float* __restrict__ out, uint8_t* act, int32_t* status, int window) {
  pdl_trigger();
  pdl_wait();
  extern __shared__ float msh[];          // [2][max_chunks] weights
  __shared__ float vals[256];
  __shared__ float lsum[2];
  const int b = blockIdx.x, row = blockIdx.y;
  const int H = nq * 128;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const size_t cstride = (size_t)nq * 16 * kPartStride;
  const int hh = threadIdx.x >> 7, d = threadIdx.x & 127;
  const float* pp = part + (((size_t)(2 * b + hh)) * 16 + row) * kPartStride + d;
  float oc[kMergeBatch];
#pragma unroll
  for (int k = 0; k < kMergeBatch; ++k) oc[k] = k < max_chunks ? pp[k * cstride] : 0.f;
  float2 ml[2];                            // warps 0, 1: (max, sum) of chunks lane, lane + 32
  if (warp < 2) {
    const float* st = part + (((size_t)(2 * b + warp)) * 16 + row) * kPartStride + 128;
#pragma unroll
    for (int t = 0; t < 2; ++t) {
      const int c = lane + 32 * t;
      ml[t] = c < max_chunks ? *reinterpret_cast<const float2*>(st + c * cstride) : make_float2(0.f, 0.f);
    }
  }
  const bool valid = row < M && !(*status & kStepAbort);
  const int n_past = *seq_len - M;
  // a sliding-window layer's chunks start at its window's first page
  const int kbase = window > 0 ? (max(0, n_past - window + 1) & ~15) : 0;
  const int nchunks = valid ? min((n_past + row - kbase) / chunk_keys + 1, max_chunks) : 0;
  if (warp < 2) {
    const float* st = part + (((size_t)(2 * b + warp)) * 16 + row) * kPartStride + 128;
    auto ml_of = [&](int c, int t) -> float2 {
      return t == 0 ? ml[0] : (t == 1 ? ml[1] : *reinterpret_cast<const float2*>(st + c * cstride));
    };
    float m = -INFINITY;
#pragma unroll 1
    for (int c = lane, t = 0; c < nchunks; c += 32, ++t) m = fmaxf(m, ml_of(c, t).x);
    m = warp_max(m);
    float L = 0.f;
#pragma unroll 1
    for (int c = lane, t = 0; c < nchunks; c += 32, ++t) {
      const float2 v = ml_of(c, t);
      const float w = (v.x == -INFINITY) ? 0.f : exp2f(v.x - m);
      msh[warp * max_chunks + c] = w;
      L += w * v.y;
    }
    L = warp_sum(L);
    if (lane == 0) lsum[warp] = L;
  }
  __syncthreads();
  // weighted sum of the unnormalised outputs, in chunk order
  const float* w = msh + hh * max_chunks;
  float o = 0.f;
#pragma unroll
  for (int k = 0; k < kMergeBatch; ++k)
    if (k < nchunks) o += w[k] * oc[k];
  for (int c = kMergeBatch; c < nchunks; ++c) o += w[c] * pp[c * cstride];
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

cudaError_t launch_attention(const AttnPlan& a, const KvView& kv, int layer, const uint8_t* qtile,
                             int M, float* part, float* out, uint8_t* act, int32_t* status,
                             cudaStream_t st, bool pdl, const uint64_t* tree_mask, const int32_t* tree_base) {
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  const int ring_s = swa_index(kv, layer);
  if (ring_s >= 0 && tree_mask) return cudaErrorInvalidValue;   // trees: paged layers only
  alignas(64) CUtensorMap kvmap;
  cudaError_t em = ring_s >= 0 ? make_ring_tmap(kv, &kvmap) : make_kv_tmap(kv, &kvmap);
  if (em != cudaSuccess) return em;
  const size_t smem = attn_smem_bytes(a);
  // the causal kernel and the token-tree kernel (which tests every block key
  // against the row's ancestor mask), each for sub-chunks of 64 and 128 keys
  const int inst = (tree_mask != nullptr) * 2 + (a.sub == 128);
  auto kern = inst == 0 ? attn_partial_kernel<false, 64>
                        : inst == 1 ? attn_partial_kernel<false, 128>
                                    : inst == 2 ? attn_partial_kernel<true, 64> : attn_partial_kernel<true, 128>;
  // the shared-memory limit is a per-device attribute of each instance
  constexpr int kMaxDevices = 64;
  static size_t smem_attr[kMaxDevices][4] = {};
  int dev = 0;
  cudaError_t ed = cudaGetDevice(&dev);
  if (ed != cudaSuccess) return ed;
  size_t* have = (dev >= 0 && dev < kMaxDevices) ? &smem_attr[dev][inst] : nullptr;
  if (!have || *have < smem) {
    cudaError_t ea = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (ea != cudaSuccess) return ea;
    if (have) *have = smem;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.max_chunks, a.nkv, a.tiles);
  cfg.blockDim = dim3(32 * kAttnWarps);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  cudaError_t e = cudaLaunchKernelEx(&cfg, kern, qtile, M, a.nq, a.nkv, a.group, a.tiles,
                                     a.chunk, kv, kvmap, layer, tree_mask, tree_base, part, status, (int)a.early,
                                     ring_s);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg2 = {};
  cfg2.gridDim = dim3(a.nq * 128 / 256, 16);
  cfg2.blockDim = dim3(256);
  cfg2.dynamicSmemBytes = sizeof(float) * 2 * (size_t)a.max_chunks;
  cfg2.stream = st;
  cfg2.attrs = attr;
  cfg2.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg2, attn_merge_kernel, (const float*)part, M, a.nq, a.max_chunks,
                            a.chunk, (const int32_t*)kv.seq_len, out, act, status,
                            ring_s >= 0 ? kv.swa_window : 0);
}

}  // namespace spec
