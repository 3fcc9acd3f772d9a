// gemm.cu — skinny Q4_K x Q8 GEMM for 1..16 rows on sm_103a tensor cores.
//
// The integer-dot anchor (Muser book Ch. 32 "Precision across the handoff",
// §32.7) asks for exact integer sub-block dot products; the verify step streams
// k-quant weights with k+1 = 16 rows per weight read (Ch. 33 §33.1, Ch. 8 §8.1)
// and the weights are consumed in their k-quant form (Ch. 8 §8.5).
//
// How the integers stay exact on the tensor cores (tcgen05.mma):
//   * a 4-bit weight code q, kept as the byte q (0..15), is the e4m3 number
//     q * 2^-9: codes 0..7 are the subnormals m * 2^-9 and codes 8..15 the
//     first normal binade (8 + m) * 2^-9.  Masking the code bytes with
//     0x0F0F0F0F (and shifting by 4 for the high nibbles) is the whole unpack;
//   * an 8-bit activation code is split as 16*h + l (both exact e4m3 values),
//     and the two MMAs A*B_hi and A*B_lo (kind::f8f6f4, K = 32 = one
//     sub-block) chain into one f32 accumulator: D_j = 2^-9 * S_j exactly,
//     |S_j| <= 32*15*127 = 60960;
//   * the sub-block scales are applied in the combine step in f32:
//     sum_j sc_j D_j over sub-blocks 0-3 and 4-7 separately are exact
//     (each below 2^24 units of 2^-9), and their sum rounds once, giving
//     (float)ISc * 2^-9; the factor 2^9 is folded into the superblock scale d
//     (exact), so d*ISc rounds exactly as in the plain formula;
//   * the min term IMn = sum_j m_j A_j is one more MMA per superblock
//     (kind::f16) with the activation sums split as A_j = 64*hi_j + lo_j.
// The per-superblock combination d_a*(d*ISc - dmin*IMn) rounds each
// operation on its own, and the superblock values accumulate in f32 in
// superblock order.  Packed f32x2 multiplies feeding an add or sub get fused
// into one fma by the compiler (d*ISc - dmin*IMn then rounds once), so every
// product is an fma whose addend is -0, passed in as a kernel argument the
// compiler cannot fold: RN(a*b + -0) = RN(a*b) for all a, b (a zero product
// keeps its sign), and an fma is never fused into its consumer.
//
// Work split: one CTA per SM owns 128 weight columns at a time.  Four
// unpack warps (one thread per column) turn a column's 144-byte superblock
// into e4m3 code bytes and store them into TMEM lane c (the MMA's A operand,
// M = 128 rows = columns of W); the 16 activation rows are the MMA's N = 16
// columns, read from shared memory (B operand).  Two warps share the 17
// MMAs of a superblock; each runs converged and lets one elected lane issue,
// which keeps the MMA operands in uniform registers (a lone lane issuing
// MMAs manages about one per 100 cycles, a converged warp about one per 35).
// One warp was 12 % slower on the 35840 x 6656 shape, three and four 0.2 %
// and 6 % slower than two.
// Four warps read the results back and combine them (one thread per column,
// all 16 rows in two batches of 8), and one warp issues the bulk copies that stage
// weights and activations.  A is triple-buffered and D double-buffered in
// TMEM, so unpacking, MMAs and combining of consecutive superblocks overlap.
//
// Row i's result depends only on row i's codes and on the fixed (K, N)
// work plan, so it is identical for every M (batch-height invariance, "The
// Two-Fifteen That Wasn't", section "The stream that was load-bearing").
#include <cstdio>

#include "common.cuh"
#include "internal.h"

namespace spec {

// ---------------------------------------------------------------------------
// Tiled layout: superblocks are regrouped so that the 128 columns of a tile
// are contiguous per superblock; bytes inside a superblock are unchanged.
// Tile T (columns 128T .. 128T+cols(T)-1, cols(T) = min(128, N-128T)),
// superblock b, column c: byte offset 128*T*nb*144 + (b*cols(T) + c)*144.
// ---------------------------------------------------------------------------
__host__ __device__ __forceinline__ size_t tiled_offset(int N, int nb, int col, int b) {
  const int T = col / kGemmCols, c = col % kGemmCols;
  const int cols = min(kGemmCols, N - kGemmCols * T);
  return ((size_t)kGemmCols * T * nb + (size_t)b * cols + c) * kSB;
}

__global__ void repack_kernel(const uint4* __restrict__ src, uint4* __restrict__ dst, int N, int nb) {
  const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;   // 16-byte chunk
  const long long total = (long long)N * nb * (kSB / 16);
  if (i >= total) return;
  const long long sbi = i / (kSB / 16);
  const int part = (int)(i - sbi * (kSB / 16));
  const int col = (int)(sbi / nb), b = (int)(sbi % nb);
  dst[tiled_offset(N, nb, col, b) / 16 + part] = src[i];
}

cudaError_t launch_repack(const void* src, void* dst, int N, int K, cudaStream_t st) {
  const int nb = K / 256;
  const long long total = (long long)N * nb * (kSB / 16);
  if (total == 0) return cudaSuccess;
  repack_kernel<<<(unsigned)((total + 255) / 256), 256, 0, st>>>(static_cast<const uint4*>(src),
                                                                  static_cast<uint4*>(dst), N, nb);
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// plan
// ---------------------------------------------------------------------------
__host__ __device__ __forceinline__ int cta_of_unit(long long x, long long U, int G) {
  return (int)(((x + 1) * (long long)G - 1) / U);
}

int plan_slots_of_group(const GemmPlan& p, int gr) {
  long long first = (long long)gr * p.nb, last = first + p.nb - 1;
  return cta_of_unit(last, p.U, p.G) - cta_of_unit(first, p.U, p.G) + 1;
}

GemmPlan make_gemm_plan(int N, int K, int num_sms) {
  GemmPlan p;
  p.N = N;
  p.K = K;
  p.nb = K / 256;
  p.ntiles = N / 16;
  p.ngroups = (p.ntiles + kTilesPerGroup - 1) / kTilesPerGroup;
  p.U = (long long)p.ngroups * p.nb;
  long long G = (long long)num_sms * kGemmCtasPerSm;
  if (G > p.U) G = p.U;
  // at most kMaxSlots CTAs may share a group: each CTA then owns >= nb/6 units
  const long long cap = (6 * p.U) / (p.nb > 0 ? p.nb : 1);
  if (G > cap) G = cap;
  if (G < 1) G = 1;
  for (;;) {
    p.G = (int)G;
    int mx = 1;
    for (int gr = 0; gr < p.ngroups; ++gr) {
      int s = plan_slots_of_group(p, gr);
      if (s > mx) mx = s;
    }
    p.max_slots = mx;
    if (mx <= kMaxSlots || G == 1) break;
    --G;
  }
  return p;
}

constexpr int kStageWeightBytes = kGemmCols * kSB;            // 18432
constexpr int kStageBytes = kStageWeightBytes + kActSBBytes;   // 27200
constexpr int kTmemCols = 512;
// TMEM columns: A buffer b = 0, 1, 2 at 72*b: sub-block j's 32 code bytes in
// columns 8j .. 8j+7 (four codes per column, lowest k in the low byte), the
// min-term A' (f16, K = 16) in columns 64 .. 71.  D buffer b = 0, 1 at
// 224 + 144*b: sub-block j's 16 rows in columns 16j .. 16j+15, the min term
// in 128 .. 143.
constexpr int kABufs = 3;
constexpr int kTmemA = 0, kTmemAStride = 72, kTmemAm = 64, kTmemD0 = 224, kTmemDStride = 144,
              kTmemDm = 128;
static_assert(kTmemD0 >= kABufs * kTmemAStride && kTmemD0 + 2 * kTmemDStride <= kTmemCols, "TMEM layout");

size_t gemm_smem_bytes() { return (size_t)kGemmStages * kStageBytes; }

// four code words of one sub-block (16 bytes, element r < 16 in the low nibble
// of byte r, element 16 + r in its high nibble) -> 8 TMEM columns of e4m3 code
// bytes in natural order: column t = elements 4t .. 4t+3
__device__ __forceinline__ void unpack_sub(const uint4& c, uint32_t* r) {
  const uint32_t w[4] = {c.x, c.y, c.z, c.w};
#pragma unroll
  for (int t = 0; t < 4; ++t) {
    r[t] = w[t] & 0x0F0F0F0Fu;
    r[4 + t] = (w[t] >> 4) & 0x0F0F0F0Fu;
  }
}

__device__ __forceinline__ uint32_t sub_scale(uint32_t f0, uint32_t f1, uint32_t f2, int j) {
  const int pos = 6 * j;                       // compile-time after unrolling
  return __funnelshift_r(pos < 32 ? f0 : f1, pos < 32 ? f1 : f2, pos & 31) & 63u;
}

SPEC_DEV void tmem_ld8(uint32_t taddr, uint32_t (&r)[8]) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];\n"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
                 "=r"(r[7])
               : "r"(taddr));
}

// Roles and hand-offs of one CTA.  Unit i = (group, superblock) number i of
// this CTA's range; it lives in stage slot s = i % kGemmStages, TMEM A buffer
// i % 3 and D buffer i % 2.  Every wait is bounded in wall time (kWaitNs); a
// thread that gives up sets SPEC_ST_DEVICE_WAIT and leaves its loop, and the
// threads that depend on it give up in turn.
//   producer warp, lane 0: wait empty[s] (unit i-S combined) -> expect the
//     unit's bytes on full[s] -> bulk-copy its 128 weight superblocks and its
//     activation block into slot s.
//   unpack warps, unit i: wait full[s] and a_free[i%3] (the MMAs of unit i-3
//     are complete) -> unpack into A[i%3] -> arrive a_full[i%3].
//   MMA warps, unit i: wait a_full[i%3] and d_free[i%2] (unit i-2 read out)
//     -> the elected lane issues the warp's share of the MMAs into D[i%2] and
//     commits to mma_done[i%2] and a_free[i%3] (one arrival per MMA warp).
//   combine warps, unit i: wait mma_done[i%2] -> start reading D, read the
//     unit's scales from its slot, arrive empty[s] -> read D (rows 0-7, then
//     8-15), arrive d_free[i%2] -> combine.
constexpr uint64_t kWaitNs = 2000000000ull;
constexpr int kWarpCombine0 = kGemmUnpackWarps;
constexpr int kWarpProducer = kWarpCombine0 + kGemmCombineThreads / 32;
constexpr int kWarpMma0 = kWarpProducer + 1;
constexpr int kGemmWarps = kWarpMma0 + kGemmMmaWarps;
static_assert(kGemmWarps * 32 == kGemmThreads, "warp roles");
// registers: each of the 4 schedulers holds the registers of its warps (16K)
constexpr int kGemmMaxRegs = kGemmWarps <= 12 ? 168 : (kGemmWarps <= 16 ? 128 : 96);
static_assert(((kGemmWarps + 3) / 4) * 32 * kGemmMaxRegs <= 16384, "register budget");

// MMA share of warp q: sub-blocks mma_j0(q) .. mma_j0(q+1)-1 (two MMAs each);
// the last warp also issues the min term
__host__ __device__ constexpr int mma_j0(int q) { return (8 * q + kGemmMmaWarps - 1) / kGemmMmaWarps; }

template <bool SUMS>
__global__ void __maxnreg__(kGemmMaxRegs)
gemm_q4k_kernel(const uint8_t* __restrict__ wt, const uint8_t* __restrict__ act,
                float* __restrict__ pieces, int N, int nb, int U, int G,
                int32_t* __restrict__ isc_out, int32_t* __restrict__ imn_out, int m_sums,
                int pre_stages, int withhold, int32_t* status, float neg_zero) {
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ uint32_t tmem_slot;
  __shared__ __align__(8) uint64_t full[kGemmStages], empty[kGemmStages];
  __shared__ __align__(8) uint64_t a_full[kABufs], a_free[kABufs], mma_done[2], d_free[2];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int lg = warp & 3;                          // TMEM lane group of this warp
  const int col_local = 32 * lg + lane;             // weight column inside the tile
  const int u0 = (int)((long long)blockIdx.x * U / G);
  const int u1 = (int)((long long)(blockIdx.x + 1) * U / G);
  const int nunits = u1 - u0;

  if (warp == 0) tmem_alloc(&tmem_slot, kTmemCols);
  if (tid == 0) {
    for (int b = 0; b < kGemmStages; ++b) {
      mbar_init(&full[b], 1);
      mbar_init(&empty[b], kGemmCombineThreads);
    }
    for (int b = 0; b < kABufs; ++b) {
      mbar_init(&a_full[b], kGemmUnpackThreads);
      mbar_init(&a_free[b], kGemmMmaWarps);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&mma_done[b], kGemmMmaWarps);
      mbar_init(&d_free[b], kGemmCombineThreads);
    }
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_slot;

  if (warp == kWarpProducer) {
    // ------------------------------------------------------------- producer
    if (lane == 0) {
      const uint64_t pol_w = l2_policy_evict_first(), pol_a = l2_policy_evict_last();
      bool ok = true;
      int issued = 0;
      int g = u0 / nb, b = u0 - (u0 / nb) * nb;
      auto weights_of = [&](int gg, int bb, uint32_t& bytes) {
        const int cols = min(kGemmCols, N - kGemmCols * gg);
        bytes = (uint32_t)(cols * kSB);
        return wt + ((size_t)kGemmCols * gg * nb + (size_t)bb * cols) * kSB;
      };
      // Weights of the first pre_stages stages do not depend on the previous
      // kernel and are fetched before the wait.  Not all 6: this prefetch runs
      // while the previous (latency-bound) kernel reads its inputs from L2,
      // and 152 CTAs x 6 stages of 18 KB queued in front of those reads slowed
      // them (the plan sets the depth per GEMM).
      // withhold (the self-test of the bounded waits): no copy is issued, so
      // every consumer wait gives up with nothing in flight
      const int nissue = withhold ? 0 : nunits;
      const int pre = min(nissue, min(max(pre_stages, 0), kGemmStages));
      {
        int gg = g, bb = b;
        for (int i = 0; i < pre; ++i) {
          uint32_t wb;
          const uint8_t* src = weights_of(gg, bb, wb);
          mbar_arrive_expect_tx(&full[i], wb + (uint32_t)kActSBBytes);
          bulk_g2s(smem + i * kStageBytes, src, wb, &full[i], pol_w);
          if (++bb == nb) { bb = 0; ++gg; }
        }
      }
      pdl_trigger();
      pdl_wait();
      for (int i = 0; i < nissue; ++i) {
        const int s = i % kGemmStages;
        if (i >= kGemmStages && !mbar_wait_ns(&empty[s], ((i / kGemmStages) - 1) & 1, kWaitNs)) {
          ok = false;
          break;
        }
        if (i >= pre) {
          uint32_t wb;
          const uint8_t* src = weights_of(g, b, wb);
          mbar_arrive_expect_tx(&full[s], wb + (uint32_t)kActSBBytes);
          bulk_g2s(smem + s * kStageBytes, src, wb, &full[s], pol_w);
        }
        bulk_g2s(smem + s * kStageBytes + kStageWeightBytes, act + (size_t)b * kActSBBytes,
                 (uint32_t)kActSBBytes, &full[s], pol_a);
        issued = i + 1;
        if (++b == nb) { b = 0; ++g; }
      }
      if (!ok) atomicOr(status, SPEC_ST_DEVICE_WAIT);
      // no copy may still be writing shared memory when the CTA exits
      for (int u = max(0, issued - kGemmStages); u < issued; ++u)
        mbar_wait_ns(&full[u % kGemmStages], (u / kGemmStages) & 1, kWaitNs);
    }
  } else if (warp >= kWarpMma0) {
    // ------------------------------------------------------------------ MMA
    pdl_trigger();
    pdl_wait();
    // warp-uniform values (the whole warp runs this loop; one lane issues)
    const int q = __shfl_sync(0xffffffffu, warp - kWarpMma0, 0);
    const uint32_t tm = __shfl_sync(0xffffffffu, tmem, 0);
    const uint32_t sbase = __shfl_sync(0xffffffffu, smem_u32(smem), 0);
    const int j0 = mma_j0(q), j1 = mma_j0(q + 1);
    // D f32, A and B e4m3 (kind::f8f6f4) or f16 (kind::f16): both format codes 0
    constexpr uint32_t kIdesc = (1u << 4) | ((16u >> 3) << 17) | ((128u >> 4) << 24);
    bool ok = true;
    int last = -1;
    for (int i = 0; i < nunits; ++i) {
      const int s = i % kGemmStages, ab = i % kABufs;
      ok = __all_sync(0xffffffffu,
                      mbar_wait_ns(&a_full[ab], (i / kABufs) & 1, kWaitNs) &&
                          (i < 2 || mbar_wait_ns(&d_free[i & 1], ((i - 2) >> 1) & 1, kWaitNs)));
      if (!ok) break;
      tc_fence_after();
      const uint32_t d = tm + (uint32_t)(kTmemD0 + (i & 1) * kTmemDStride);
      const uint32_t a = tm + (uint32_t)(kTmemA + ab * kTmemAStride);
      // B blocks: hi of sub-block j at 1024*j, lo at +512 (descriptor units of 16 B)
      const uint64_t desc0 = smem_desc(sbase + (uint32_t)(s * kStageBytes + kStageWeightBytes), 128, 256);
      if (elect_one()) {
#pragma unroll
        for (int jj = 0; jj < (8 + kGemmMmaWarps - 1) / kGemmMmaWarps; ++jj) {
          const int j = j0 + jj;
          if (j < j1) {
            mma_f8_ts(d + 16 * j, a + 8 * j, desc0 + 64ull * j, kIdesc, 0);
            mma_f8_ts(d + 16 * j, a + 8 * j, desc0 + 64ull * j + 32, kIdesc, 1);
          }
        }
        if (q == kGemmMmaWarps - 1) mma_f16_ts(d + kTmemDm, a + kTmemAm, desc0 + 32ull * 16, kIdesc, 0);
        mma_commit(&mma_done[i & 1]);
        mma_commit(&a_free[ab]);
      }
      __syncwarp();
      last = i;
    }
    if (!ok && lane == 0) atomicOr(status, SPEC_ST_DEVICE_WAIT);
    // TMEM is released at the end: the MMAs of this warp must have finished
    if (last >= 0) mbar_wait_ns(&a_free[last % kABufs], (last / kABufs) & 1, kWaitNs);
  } else if (warp < kWarpCombine0) {
    // --------------------------------------------------------------- unpack
    const uint32_t lane_base = (uint32_t)(32 * lg) << 16;
    bool ok = true;
    int cg = u0 / nb;
    int cb = u0 - cg * nb;
    for (int i = 0; i < nunits; ++i) {
      const int s = i % kGemmStages, ab = i % kABufs;
      // warp-uniform decisions: the TMEM stores below are warp-collective
      ok = __all_sync(0xffffffffu,
                      mbar_wait_ns(&full[s], (i / kGemmStages) & 1, kWaitNs) &&
                          (i < kABufs || mbar_wait_ns(&a_free[ab], ((i - kABufs) / kABufs) & 1, kWaitNs)));
      if (!ok) break;
      tc_fence_after();
      const uint8_t* stg = smem + s * kStageBytes;
      const int cols = min(kGemmCols, N - kGemmCols * cg);
      const bool valid = col_local < cols;
      const uint4* sbp = reinterpret_cast<const uint4*>(stg + col_local * kSB);
      const uint32_t abase = tmem + lane_base + (uint32_t)(kTmemA + ab * kTmemAStride);
#pragma unroll
      for (int hq = 0; hq < 2; ++hq) {             // sub-blocks 4hq .. 4hq+3 per TMEM store
        uint32_t r[32];
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) {
          uint4 c = make_uint4(0, 0, 0, 0);
          if (valid) c = sbp[1 + 4 * hq + jj];
          unpack_sub(c, r + 8 * jj);
        }
        tmem_st32(abase + (uint32_t)(32 * hq), r);
      }
      {
        // min-term operand: k = j -> m_j, k = 8 + j -> m_j (f16 pairs)
        uint4 hdr = make_uint4(0, 0, 0, 0);
        if (valid) hdr = sbp[0];
        const uint32_t f1 = hdr.z, f2 = hdr.w;
        uint32_t mp[4];
#pragma unroll
        for (int qq = 0; qq < 4; ++qq) {
          const int p0 = 48 + 12 * qq;             // bits of m_2qq, m_2qq+1
          const uint32_t m12 = __funnelshift_r(p0 < 64 ? f1 : f2, p0 < 64 ? f2 : 0u, p0 & 31);
          mp[qq] = hadd2_u32(((m12 & 63u) | (((m12 >> 6) & 63u) << 16)) + 0x64006400u, 0xE400E400u);
        }
        tmem_st4(abase + (uint32_t)kTmemAm, mp[0], mp[1], mp[2], mp[3]);
        tmem_st4(abase + (uint32_t)(kTmemAm + 4), mp[0], mp[1], mp[2], mp[3]);
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(&a_full[ab]);
      if (++cb == nb) {
        cb = 0;
        ++cg;
      }
    }
    if (!ok && lane == 0) atomicOr(status, SPEC_ST_DEVICE_WAIT);
  } else {
    // -------------------------------------------------------------- combine
    pdl_trigger();
    pdl_wait();
    const uint32_t lane_base = (uint32_t)(32 * lg) << 16;
    bool ok = true;
    float y[16];
#pragma unroll
    for (int n = 0; n < 16; ++n) y[n] = 0.f;
    int ug = u0 / nb;
    int ub = u0 - ug * nb;
    for (int u = 0; u < nunits; ++u) {
      // warp-uniform decision: the TMEM loads below are warp-collective
      ok = __all_sync(0xffffffffu, mbar_wait_ns(&mma_done[u & 1], (u >> 1) & 1, kWaitNs));
      if (!ok) break;
      tc_fence_after();
      const int pslot = u % kGemmStages;
      const uint8_t* stg = smem + pslot * kStageBytes;
      const int cols = min(kGemmCols, N - kGemmCols * ug);
      const bool valid = col_local < cols;
      const int col = kGemmCols * ug + col_local;
      const uint32_t dbase = tmem + lane_base + (uint32_t)(kTmemD0 + (u & 1) * kTmemDStride);
      // rows 0..7 of every accumulator: start the TMEM loads
      uint32_t dj[8][8], rm[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) tmem_ld8(dbase + 16 * j, dj[j]);
      tmem_ld8(dbase + kTmemDm, rm);
      // the stage was filled before the MMAs of this unit were issued, and the
      // MMAs are done with it: read the scales and free the slot
      uint4 hdr = make_uint4(0, 0, 0, 0);
      if (valid) hdr = *reinterpret_cast<const uint4*>(stg + col_local * kSB);
      float da[16];
      {
        const float4* dap = reinterpret_cast<const float4*>(stg + kStageWeightBytes + kActSlots * 512);
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) {
          const float4 v4 = dap[q4];
          da[4 * q4] = v4.x; da[4 * q4 + 1] = v4.y; da[4 * q4 + 2] = v4.z; da[4 * q4 + 3] = v4.w;
        }
      }
      mbar_arrive(&empty[pslot]);
      // 6-bit scales as exact floats: 2^23 + sc with the 2^23 subtracted
      float scf[8];
#pragma unroll
      for (int j = 0; j < 8; ++j)
        scf[j] = __uint_as_float(0x4B000000u | sub_scale(hdr.y, hdr.z, hdr.w, j)) - 8388608.f;
      // d * 2^9 (exact): the D values are 2^-9 * integer sums
      const float d = __half2float(__ushort_as_half((unsigned short)(hdr.x & 0xffff))) * 512.f;
      const float dm = __half2float(__ushort_as_half((unsigned short)(hdr.x >> 16)));
      const unsigned long long D2 = f2pack(d, d), M2 = f2pack(dm, dm), NZ = f2pack(neg_zero, neg_zero);
#pragma unroll
      for (int rb = 0; rb < 2; ++rb) {             // rows 8rb .. 8rb+7
        if (rb == 1) {
#pragma unroll
          for (int j = 0; j < 8; ++j) tmem_ld8(dbase + 16 * j + 8, dj[j]);
          tmem_ld8(dbase + kTmemDm + 8, rm);
        }
        tmem_wait_ld();
        if (rb == 1) {
          tc_fence_before();
          mbar_arrive(&d_free[u & 1]);
        }
#pragma unroll
        for (int n = 0; n < 8; n += 2) {
          unsigned long long lo = 0ull, hi = 0ull;   // sub-blocks 0-3 and 4-7: sum_j sc_j S_j * 2^-9
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const unsigned long long sc2 = f2pack(scf[j], scf[j]);
            const unsigned long long sj = f2pack(__uint_as_float(dj[j][n]), __uint_as_float(dj[j][n + 1]));
            if (j < 4) lo = j == 0 ? f2mul(sc2, sj) : f2fma(sc2, sj, lo);
            else hi = j == 4 ? f2mul(sc2, sj) : f2fma(sc2, sj, hi);
          }
          const int r = 8 * rb + n;
          const unsigned long long isc = f2add(lo, hi);   // exact: ISc * 2^-9
          const unsigned long long imn = f2pack(__uint_as_float(rm[n]), __uint_as_float(rm[n + 1]));
          const unsigned long long t = f2sub(f2fma(D2, isc, NZ), f2fma(M2, imn, NZ));
          const unsigned long long v = f2fma(f2pack(da[r], da[r + 1]), t, NZ);
          f2unpack(f2add(f2pack(y[r], y[r + 1]), v), y[r], y[r + 1]);
          if (SUMS && valid) {
            float l0, l1, h0, h1;
            f2unpack(lo, l0, l1);
            f2unpack(hi, h0, h1);
#pragma unroll
            for (int e = 0; e < 2; ++e) {
              if (r + e < m_sums) {
                const size_t o = ((size_t)(r + e) * N + col) * nb + ub;
                isc_out[o] = (int)((e ? l1 : l0) * 512.f) + (int)((e ? h1 : h0) * 512.f);
                imn_out[o] = (int)__uint_as_float(rm[n + e]);
              }
            }
          }
        }
      }
      // end of this CTA's run over the group: write the piece
      if (u0 + u + 1 == u1 || ub + 1 == nb) {
        const int slot_id = (int)blockIdx.x - cta_of_unit((long long)ug * nb, U, G);
        if (valid) {
          float* base = pieces + (size_t)slot_id * 16 * N + col;
#pragma unroll
          for (int n = 0; n < 16; ++n) base[(size_t)n * N] = y[n];
        }
#pragma unroll
        for (int n = 0; n < 16; ++n) y[n] = 0.f;
      }
      if (++ub == nb) {
        ub = 0;
        ++ug;
      }
    }
    if (!ok && lane == 0) atomicOr(status, SPEC_ST_DEVICE_WAIT);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// The kernel's dynamic shared memory exceeds the default limit; the limit is
// a per-device attribute, raised on every device that runs the GEMM (by
// spec_verify_init for a ctx, and on a device's first allocation-free call).
cudaError_t gemm_init_attributes() {
  const int smem = (int)gemm_smem_bytes();
  cudaError_t e = cudaFuncSetAttribute(gemm_q4k_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(gemm_q4k_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
}

cudaError_t launch_gemm(const GemmPlan& p, const void* w_tiled, const uint8_t* act, float* pieces,
                        int32_t* isc, int32_t* imn, int m_sums, int32_t* status, cudaStream_t st,
                        bool pdl, bool withhold) {
  const size_t smem = gemm_smem_bytes();
  const bool sums = isc != nullptr;
  auto kern = sums ? gemm_q4k_kernel<true> : gemm_q4k_kernel<false>;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.G);
  cfg.blockDim = dim3(kGemmThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, static_cast<const uint8_t*>(w_tiled), act, pieces, p.N, p.nb,
                            (int)p.U, p.G, isc, imn, m_sums, p.pre_stages, (int)withhold, status, -0.0f);
}

// y[m][n] = sum over the group's slots, in slot order
__global__ void sum_pieces_kernel(const float* __restrict__ pieces, float* __restrict__ y, int N,
                                  int M, int nb, long long U, int G) {
  pdl_trigger();
  pdl_wait();
  const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= (long long)M * N) return;
  const int m = (int)(i / N), n = (int)(i % N);
  const int gr = (n / 16) / kTilesPerGroup;
  const int c0 = cta_of_unit((long long)gr * nb, U, G);
  const int ns = cta_of_unit((long long)gr * nb + nb - 1, U, G) - c0 + 1;
  float v[kMaxSlots];
#pragma unroll
  for (int k = 0; k < kMaxSlots; ++k) v[k] = k < ns ? pieces[((size_t)k * 16 + m) * N + n] : 0.f;
  float s = v[0];
#pragma unroll
  for (int k = 1; k < kMaxSlots; ++k)
    if (k < ns) s += v[k];
  y[(size_t)m * N + n] = s;
}

cudaError_t launch_sum_pieces(const GemmPlan& p, const float* pieces, float* y, int M,
                              cudaStream_t st, bool pdl) {
  const long long n = (long long)M * p.N;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)((n + 255) / 256));
  cfg.blockDim = dim3(256);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, sum_pieces_kernel, pieces, y, p.N, M, p.nb, p.U, p.G);
}

}  // namespace spec
