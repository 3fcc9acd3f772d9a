// gemm.cu — skinny Q4_K x Q8 GEMM for 1..16 rows on sm_103a tensor cores.
//
// The integer-dot anchor (Muser book Ch. 32 "Precision across the handoff",
// §32.7) asks for exact integer sub-block dot products; the verify step streams
// k-quant weights with k+1 = 16 rows per weight read (Ch. 33 §33.1, Ch. 8 §8.1)
// and the weights are consumed in their k-quant form (Ch. 8 §8.5).
//
// How the integers stay exact on f16 tensor cores:
//   * a weight code q (0..15) times its 6-bit sub-scale sc is at most 945 and
//     an activation code is in [-127, 127]: both are exact f16 integers;
//   * the f16 weight operand sc*q is built as fma(1024+q, sc, -1024*sc): the
//     LOP3 "magic" 0x6400|q is the f16 number 1024+q, and a fused multiply-add
//     rounds the exact result sc*q once, i.e. not at all;
//   * products accumulate in f32; four sub-blocks contribute at most
//     4*32*945*127 < 2^24, so the two half-superblock accumulators are exact
//     integers and their f32 sum is the exact ISc rounded once, as (float)ISc;
//   * the min term IMn = sum_j m_j A_j is one more MMA per superblock with the
//     activation sums split as A_j = 64*hi_j + lo_j (both exact in f16).
// The per-superblock combination d_a*(d*ISc - dmin*IMn) uses packed f32x2
// operations, each rounded on its own (no contraction), and the superblock
// values accumulate in f32 in superblock order.
//
// Row i's result depends only on row i's codes and on the fixed (K, N)
// work plan, so it is identical for every M (batch-height invariance, "The
// Two-Fifteen That Wasn't", section "The stream that was load-bearing").
#include <cstdio>

#include "common.cuh"
#include "internal.h"

namespace spec {

// ---------------------------------------------------------------------------
// k-slot permutation.  An m16n8k16 step s (0..15) of superblock b covers 16
// k-slots; lane quad position t (0..3) owns slots {2t, 2t+1} ("pair A") and
// {2t+8, 2t+9} ("pair B") of every step.  Slots are mapped to superblock
// elements so that lane t only ever meets sub-blocks 2t and 2t+1:
//   pair A, slot 2t+u   -> element 64t + 2s + u        (sub-block 2t)
//   pair B, slot 2t+8+u -> element 64t + 32 + 2s + u   (sub-block 2t+1)
// The activation fragments use the same map, so the dot product is unchanged;
// each lane then needs the sub-scales of 2 sub-blocks instead of 8.
//
// Tiled layout of one (tile of 16 columns, superblock) block of 2304 bytes:
//   [0, 2048)    codes: chunk q (0..3) at 512q; lane L = 4g+t owns 16 bytes at
//                512q + 16L = words { W(g,A,q), W(g+8,A,q), W(g,B,q), W(g+8,B,q) }.
//                W(c, P, q) holds, for steps s = 4q+p (p = 0..3), the codes of
//                column c at the pair-P elements of step s: the even element in
//                bits 4p..4p+3, the odd one in bits 16+4p..16+4p+3.
//   [2048, 2112) column c: (d, dmin) binary16 pair at 2048 + 4c
//   [2112, 2304) column c: the 12-byte 6-bit scale/min field at 2112 + 12c
// ---------------------------------------------------------------------------

__device__ __forceinline__ int canon_code(const uint8_t* sb, int e) {
  int j = e >> 5, r = e & 31;
  uint8_t byte = sb[16 + 16 * j + (r & 15)];
  return r < 16 ? (byte & 15) : (byte >> 4);
}

__global__ void repack_kernel(const uint8_t* __restrict__ src, uint8_t* __restrict__ dst, int nb,
                              long long nblocks) {
  long long blk = blockIdx.x;
  if (blk >= nblocks) return;
  int tile = (int)(blk / nb), b = (int)(blk % nb);
  uint8_t* out = dst + blk * kTileSB;
  for (int w = threadIdx.x; w < kTileSB / 4; w += blockDim.x) {
    uint32_t word = 0;
    if (w < 512) {
      const int q = w >> 7, L = (w >> 2) & 31, sl = w & 3;
      const int g = L >> 2, t = L & 3;
      const int c = g + 8 * (sl & 1);
      const int pairB = sl >> 1;
      const uint8_t* sb = src + ((size_t)(tile * 16 + c) * nb + b) * kSB;
#pragma unroll
      for (int p = 0; p < 4; ++p) {
        const int s = 4 * q + p;
        const int e = 64 * t + 32 * pairB + 2 * s;
        word |= (uint32_t)canon_code(sb, e) << (4 * p);
        word |= (uint32_t)canon_code(sb, e + 1) << (16 + 4 * p);
      }
    } else if (w < 528) {
      int c = w - 512;
      const uint8_t* sb = src + ((size_t)(tile * 16 + c) * nb + b) * kSB;
      word = sb[0] | (sb[1] << 8) | (sb[2] << 16) | ((uint32_t)sb[3] << 24);
    } else {
      int i = w - 528;            // 48 words of scales: column i/3, word i%3
      int c = i / 3, wi = i % 3;
      const uint8_t* sb = src + ((size_t)(tile * 16 + c) * nb + b) * kSB + 4 + 4 * wi;
      word = sb[0] | (sb[1] << 8) | (sb[2] << 16) | ((uint32_t)sb[3] << 24);
    }
    reinterpret_cast<uint32_t*>(out)[w] = word;
  }
}

cudaError_t launch_repack(const void* src, void* dst, int N, int K, cudaStream_t st) {
  int nb = K / 256;
  long long nblocks = (long long)(N / 16) * nb;
  if (nblocks == 0) return cudaSuccess;
  repack_kernel<<<(unsigned)nblocks, 192, 0, st>>>(static_cast<const uint8_t*>(src),
                                                   static_cast<uint8_t*>(dst), nb, nblocks);
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// plan
// ---------------------------------------------------------------------------
__host__ __device__ __forceinline__ int cta_of_unit(long long x, long long U, int G) {
  return (int)(((x + 1) * (long long)G - 1) / U);
}

GemmPlan make_gemm_plan(int N, int K, int num_sms) {
  GemmPlan p;
  p.N = N;
  p.K = K;
  p.nb = K / 256;
  p.ntiles = N / 16;
  p.ngroups = (p.ntiles + kTilesPerGroup - 1) / kTilesPerGroup;
  p.U = (long long)p.ngroups * p.nb;
  long long G = num_sms;
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

int plan_slots_of_group(const GemmPlan& p, int gr) {
  long long first = (long long)gr * p.nb, last = first + p.nb - 1;
  return cta_of_unit(last, p.U, p.G) - cta_of_unit(first, p.U, p.G) + 1;
}

constexpr int kStageWeightBytes = kTilesPerGroup * kTileSB;
constexpr int kStageBytes = kStageWeightBytes + kActSBBytes;

size_t gemm_smem_bytes() { return (size_t)kGemmStages * kStageBytes; }

// ---------------------------------------------------------------------------
// the GEMM kernel
// ---------------------------------------------------------------------------
__device__ __forceinline__ void mma16816_zc(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                            uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%10,%10,%10,%10};\n"
      : "=f"(c[0]), "=f"(c[1]), "=f"(c[2]), "=f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1), "f"(0.0f));
}

// f16x2 constants for one (column, sub-block) with 6-bit scale sc:
//   S = {sc, sc}, O = {-1024 sc, ...} for codes held as 1024+q (mask 0x000F);
//   S16 = {sc/16, ...}, O16 = {-64 sc, ...} for codes held as 1024+16q (mask 0x00F0).
// Every value is an exact f16 (sc <= 63), so fma(x, S, O) = sc*q exactly.
struct ScaleC {
  uint32_t S, O, S16, O16;
};
__device__ __forceinline__ ScaleC scale_consts(uint32_t sc) {
  ScaleC r;
  const uint32_t v = sc * 0x00010001u + 0x64006400u;   // {1024+sc, 1024+sc}
  r.S = hadd2_u32(v, 0xE400E400u);                      // - 1024
  r.O = hmul2_u32(r.S, 0xE400E400u);                    // * -1024
  r.S16 = hmul2_u32(r.S, 0x2C002C00u);                  // * 1/16
  r.O16 = hmul2_u32(r.S, 0xD400D400u);                  // * -64
  return r;
}

// codes at bits (0,16) of x -> {sc*q_lo, sc*q_hi}
__device__ __forceinline__ uint32_t unpack_lo(uint32_t x, const ScaleC& c) {
  return hfma2_u32(lop3_and_or(x, 0x000F000Fu, 0x64006400u), c.S, c.O);
}
// codes at bits (4,20) of x -> {sc*q_lo, sc*q_hi}
__device__ __forceinline__ uint32_t unpack_hi(uint32_t x, const ScaleC& c) {
  return hfma2_u32(lop3_and_or(x, 0x00F000F0u, 0x64006400u), c.S16, c.O16);
}

template <bool SUMS>
__global__ void __launch_bounds__(kGemmWarps * 32, 1)
gemm_q4k_kernel(const uint8_t* __restrict__ wt, const uint8_t* __restrict__ act,
                float* __restrict__ pieces, int N, int nb, int ntiles, int U, int G,
                int32_t* __restrict__ isc_out, int32_t* __restrict__ imn_out, int m_sums) {
  extern __shared__ __align__(128) uint8_t smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, t = lane & 3;
  const int u0 = (int)((long long)blockIdx.x * U / G);
  const int u1 = (int)((long long)(blockIdx.x + 1) * U / G);

  // lane constants: bit positions of (sc_2t, sc_2t+1) and (m_2t, m_2t+1) in the field
  const int ws = (12 * t) >> 5, sh_s = (12 * t) & 31;
  const int wm = (48 + 12 * t) >> 5, sh_m = (48 + 12 * t) & 31;

  // copy cursor (unit being issued) and its (group, superblock)
  int iu = u0, ig = u0 / nb, ib = u0 - (u0 / nb) * nb;
  auto issue_weights = [&](int slot) {
    uint8_t* dst = smem + slot * kStageBytes + warp * kGemmTilesPerWarp * kTileSB;
    const int tile0 = ig * kTilesPerGroup + warp * kGemmTilesPerWarp;
    const uint8_t* src0 = wt + ((size_t)tile0 * nb + ib) * kTileSB;
    const uint8_t* src1 = src0 + (size_t)nb * kTileSB;
    const bool ok0 = tile0 < ntiles, ok1 = tile0 + 1 < ntiles;
#pragma unroll
    for (int i = 0; i < 2 * kTileSB / 16 / 32; ++i) {
      const int c = lane + 32 * i;
      if (c < kTileSB / 16) {
        if (ok0) cp_async16(dst + c * 16, src0 + c * 16);
      } else {
        if (ok1) cp_async16(dst + c * 16, src1 + (c - kTileSB / 16) * 16);
      }
    }
  };
  auto issue_act = [&](int slot) {
    uint8_t* dst = smem + slot * kStageBytes + kStageWeightBytes;
    const uint8_t* src = act + (size_t)ib * kActSBBytes;
    for (int c = threadIdx.x; c < kActSBBytes / 16; c += kGemmWarps * 32) cp_async16(dst + c * 16, src + c * 16);
  };
  auto advance = [&]() {
    ++iu;
    if (++ib == nb) {
      ib = 0;
      ++ig;
    }
  };

  // Weights do not depend on the previous kernel: stream them first, then wait
  // for the producer of the activations.
  {
    const int su = iu, sg = ig, sb = ib;
    for (int s = 0; s < kGemmStages - 1; ++s) {
      if (iu < u1) issue_weights(s);
      advance();
    }
    iu = su;
    ig = sg;
    ib = sb;
    pdl_wait();
    pdl_trigger();
    for (int s = 0; s < kGemmStages - 1; ++s) {
      if (iu < u1) issue_act(s);
      cp_async_commit();
      advance();
    }
  }

  // output accumulators as packed f32 pairs: [tile][h*2 + column half]
  unsigned long long yacc[kGemmTilesPerWarp][4];
#pragma unroll
  for (int tt = 0; tt < kGemmTilesPerWarp; ++tt)
#pragma unroll
    for (int i = 0; i < 4; ++i) yacc[tt][i] = 0ull;

  int cgrp = u0 / nb, cb = u0 - (u0 / nb) * nb;   // compute cursor
  int slot = 0, islot = kGemmStages - 1;
  for (int u = u0; u < u1; ++u) {
    cp_async_wait<kGemmStages - 2>();
    __syncthreads();
    if (iu < u1) {
      issue_weights(islot);
      issue_act(islot);
    }
    cp_async_commit();
    advance();
    islot = (islot + 1 == kGemmStages) ? 0 : islot + 1;

    const uint8_t* stg = smem + slot * kStageBytes;
    const uint8_t* ast = stg + kStageWeightBytes;
    slot = (slot + 1 == kGemmStages) ? 0 : slot + 1;

    uint4 nib[kGemmTilesPerWarp][4];
    ScaleC sc[kGemmTilesPerWarp][2][2];     // [tile][column g, g+8][pair A, B]
    uint32_t mfrag[kGemmTilesPerWarp][2];
    uint32_t ddw[kGemmTilesPerWarp][2];
#pragma unroll
    for (int tt = 0; tt < kGemmTilesPerWarp; ++tt) {
      const uint8_t* wtile = stg + (warp * kGemmTilesPerWarp + tt) * kTileSB;
#pragma unroll
      for (int q = 0; q < 4; ++q) nib[tt][q] = *reinterpret_cast<const uint4*>(wtile + 512 * q + 16 * lane);
#pragma unroll
      for (int cc = 0; cc < 2; ++cc) {
        const uint32_t* f = reinterpret_cast<const uint32_t*>(wtile + 2112 + 12 * (g + 8 * cc));
        const uint32_t s12 = __funnelshift_r(f[ws], f[ws + 1], sh_s);
        const uint32_t m12 = __funnelshift_r(f[wm], wm < 2 ? f[wm + 1] : 0u, sh_m);
        sc[tt][cc][0] = scale_consts(s12 & 63u);
        sc[tt][cc][1] = scale_consts((s12 >> 6) & 63u);
        mfrag[tt][cc] = hadd2_u32(((m12 & 63u) | (((m12 >> 6) & 63u) << 16)) + 0x64006400u, 0xE400E400u);
        ddw[tt][cc] = *reinterpret_cast<const uint32_t*>(wtile + 2048 + 4 * (g + 8 * cc));
      }
    }

    float acc[kGemmTilesPerWarp][2][2][4];   // [tile][steps 0-7 | 8-15][row half][4]
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      uint4 xs[kGemmTilesPerWarp];
#pragma unroll
      for (int tt = 0; tt < kGemmTilesPerWarp; ++tt)
        xs[tt] = make_uint4(nib[tt][q].x >> 8, nib[tt][q].y >> 8, nib[tt][q].z >> 8, nib[tt][q].w >> 8);
#pragma unroll
      for (int p = 0; p < 4; ++p) {
        const int s = 4 * q + p;
        const int half = s >> 3;
        const uint4 av = *reinterpret_cast<const uint4*>(ast + s * 512 + 16 * lane);
#pragma unroll
        for (int tt = 0; tt < kGemmTilesPerWarp; ++tt) {
          const uint4 x = (p < 2) ? nib[tt][q] : xs[tt];
          uint32_t a0, a1, a2, a3;
          if ((p & 1) == 0) {
            a0 = unpack_lo(x.x, sc[tt][0][0]);
            a1 = unpack_lo(x.y, sc[tt][1][0]);
            a2 = unpack_lo(x.z, sc[tt][0][1]);
            a3 = unpack_lo(x.w, sc[tt][1][1]);
          } else {
            a0 = unpack_hi(x.x, sc[tt][0][0]);
            a1 = unpack_hi(x.y, sc[tt][1][0]);
            a2 = unpack_hi(x.z, sc[tt][0][1]);
            a3 = unpack_hi(x.w, sc[tt][1][1]);
          }
          if ((s & 7) == 0) {
            mma16816_zc(acc[tt][half][0], a0, a1, a2, a3, av.x, av.y);
            mma16816_zc(acc[tt][half][1], a0, a1, a2, a3, av.z, av.w);
          } else {
            mma16816(acc[tt][half][0], a0, a1, a2, a3, av.x, av.y);
            mma16816(acc[tt][half][1], a0, a1, a2, a3, av.z, av.w);
          }
        }
      }
    }

    // min term, d/dmin/d_a combination, accumulation
    const uint4 am = *reinterpret_cast<const uint4*>(ast + 16 * 512 + 16 * lane);
    const float2 da0 = *reinterpret_cast<const float2*>(ast + kActSlots * 512 + 4 * (2 * t));
    const float2 da1 = *reinterpret_cast<const float2*>(ast + kActSlots * 512 + 4 * (8 + 2 * t));
#pragma unroll
    for (int tt = 0; tt < kGemmTilesPerWarp; ++tt) {
      float imn[2][4];
      mma16816_zc(imn[0], mfrag[tt][0], mfrag[tt][1], mfrag[tt][0], mfrag[tt][1], am.x, am.y);
      mma16816_zc(imn[1], mfrag[tt][0], mfrag[tt][1], mfrag[tt][0], mfrag[tt][1], am.z, am.w);
      const uint32_t dd0 = ddw[tt][0], dd1 = ddw[tt][1];
      const float d0 = __half2float(__ushort_as_half((unsigned short)(dd0 & 0xffff)));
      const float m0f = __half2float(__ushort_as_half((unsigned short)(dd0 >> 16)));
      const float d1 = __half2float(__ushort_as_half((unsigned short)(dd1 & 0xffff)));
      const float m1f = __half2float(__ushort_as_half((unsigned short)(dd1 >> 16)));
      const unsigned long long D0 = f2pack(d0, d0), M0 = f2pack(m0f, m0f);
      const unsigned long long D1 = f2pack(d1, d1), M1 = f2pack(m1f, m1f);
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const unsigned long long DA = h == 0 ? f2pack(da0.x, da0.y) : f2pack(da1.x, da1.y);
        // exact ISc (rounded once to f32) from the two exact half sums
        const unsigned long long isc01 =
            f2add(f2pack(acc[tt][0][h][0], acc[tt][0][h][1]), f2pack(acc[tt][1][h][0], acc[tt][1][h][1]));
        const unsigned long long isc23 =
            f2add(f2pack(acc[tt][0][h][2], acc[tt][0][h][3]), f2pack(acc[tt][1][h][2], acc[tt][1][h][3]));
        // column g (c0, c1 of the fragment), column g+8 (c2, c3)
        const unsigned long long v01 =
            f2mul(DA, f2sub(f2mul(D0, isc01), f2mul(M0, f2pack(imn[h][0], imn[h][1]))));
        const unsigned long long v23 =
            f2mul(DA, f2sub(f2mul(D1, isc23), f2mul(M1, f2pack(imn[h][2], imn[h][3]))));
        yacc[tt][2 * h + 0] = f2add(yacc[tt][2 * h + 0], v01);
        yacc[tt][2 * h + 1] = f2add(yacc[tt][2 * h + 1], v23);
        if (SUMS) {
          const int tile = cgrp * kTilesPerGroup + warp * kGemmTilesPerWarp + tt;
          if (tile < ntiles) {
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const int row = 8 * h + 2 * t + (e & 1);
              const int col = tile * 16 + g + 8 * (e >> 1);
              if (row < m_sums) {
                const size_t o = ((size_t)row * N + col) * nb + cb;
                isc_out[o] = (int)acc[tt][0][h][e] + (int)acc[tt][1][h][e];
                imn_out[o] = (int)imn[h][e];
              }
            }
          }
        }
      }
    }

    // end of this CTA's run over the group: write the piece
    const bool last_of_group = (cb + 1 == nb);
    if (u + 1 == u1 || last_of_group) {
      const int slot_id = (int)blockIdx.x - cta_of_unit((long long)cgrp * nb, U, G);
      float* base = pieces + (size_t)slot_id * 16 * N;
#pragma unroll
      for (int tt = 0; tt < kGemmTilesPerWarp; ++tt) {
        const int tile = cgrp * kTilesPerGroup + warp * kGemmTilesPerWarp + tt;
        if (tile < ntiles) {
#pragma unroll
          for (int h = 0; h < 2; ++h)
#pragma unroll
            for (int cc = 0; cc < 2; ++cc) {
              float lo, hi;
              f2unpack(yacc[tt][2 * h + cc], lo, hi);
              const int row = 8 * h + 2 * t;
              const int col = tile * 16 + g + 8 * cc;
              base[(size_t)row * N + col] = lo;
              base[(size_t)(row + 1) * N + col] = hi;
            }
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) yacc[tt][i] = 0ull;
      }
    }
    if (++cb == nb) {
      cb = 0;
      ++cgrp;
    }
  }
  cp_async_wait<0>();
}

static bool g_gemm_attr_set[2] = {false, false};

cudaError_t gemm_init_attributes() {
  const int smem = (int)gemm_smem_bytes();
  cudaError_t e = cudaFuncSetAttribute(gemm_q4k_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(gemm_q4k_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  g_gemm_attr_set[0] = g_gemm_attr_set[1] = true;
  return cudaSuccess;
}

cudaError_t launch_gemm(const GemmPlan& p, const void* w_tiled, const uint8_t* act, float* pieces,
                        int32_t* isc, int32_t* imn, int m_sums, cudaStream_t st, bool pdl) {
  const size_t smem = gemm_smem_bytes();
  const bool sums = isc != nullptr;
  auto kern = sums ? gemm_q4k_kernel<true> : gemm_q4k_kernel<false>;
  if (!g_gemm_attr_set[sums]) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    g_gemm_attr_set[sums] = true;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.G);
  cfg.blockDim = dim3(kGemmWarps * 32);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, static_cast<const uint8_t*>(w_tiled), act, pieces, p.N,
                            p.nb, p.ntiles, (int)p.U, p.G, isc, imn, m_sums);
}

// y[m][n] = sum over the group's slots, in slot order
__global__ void sum_pieces_kernel(const float* __restrict__ pieces, float* __restrict__ y, int N,
                                  int M, int nb, long long U, int G) {
  pdl_wait();
  pdl_trigger();
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
