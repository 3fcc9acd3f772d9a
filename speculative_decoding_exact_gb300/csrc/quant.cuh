// quant.cuh — per-row, per-256-block activation quantisation into the
// MMA-operand-ordered activation buffer read by the Q4_K GEMM.
//   d_a = amax/127 (IEEE fp32 division), q = clamp(rint(x/d_a), -127, 127)
//   with round-half-even, all-zero block -> d_a = 0, q = 0; A_j = sum of the
//   32 codes of sub-block j.
#pragma once
#include "common.cuh"

namespace spec {

// ---------------------------------------------------------------------------
// Activation buffer of one superblock (kActSBBytes bytes), read by the GEMM's
// tensor-core MMAs as their B operand.  An 8-bit code q in [-127, 127] is
// split as q = 16*h + l with l = q & 15 in [0, 15] and h = q >> 4 in [-8, 7];
// both 16*h and l are exact e4m3 numbers.
//   at 1024*j (sub-block j = 0..7): the e4m3 values 16*h of the 16 rows x 32
//     codes of sub-block j; at 1024*j + 512 the values l.  Each 512-byte block
//     is in the canonical K-major core-matrix layout of an MMA with N = 16,
//     K = 32: code k of row n at (n/8)*256 + (k/16)*128 + (n%8)*16 + k%16;
//   block 16 (at 8192): the min-term operand, f16, K = 16: k = j (0..7) ->
//     64*hi_j, k = 8+j -> lo_j, where A_j = 64*hi_j + lo_j; value (n, k) at
//     (n/8)*256 + (k/8)*128 + (n%8)*16 + (k%8)*2;
//   at 512*17: d_a of the 16 rows (fp32).
// Codes keep their natural order inside a sub-block: the GEMM stores weight
// code k of sub-block j at the same k of its A operand.
// ---------------------------------------------------------------------------
SPEC_DEV int act_off(int n, int s, int k) {
  return 512 * s + (n >> 3) * 256 + (k >> 3) * 128 + (n & 7) * 16 + (k & 7) * 2;
}
SPEC_DEV int act_off8(int n, int j, int part, int k) {
  return 1024 * j + 512 * part + (n >> 3) * 256 + (k >> 4) * 128 + (n & 7) * 16 + (k & 15);
}
// e4m3 bytes of two exact e4m3 values: lo in bits 0-7, hi in bits 8-15
SPEC_DEV uint32_t e4m3x2(float lo, float hi) {
  unsigned short r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

// Quantisation of one 256-block of one row, executed by one warp.  Lane l owns
// elements 8l..8l+7 (sub-block l/4).
//
// q = rint(x/d_a) needs the IEEE quotient only where it decides the integer.
// With r = RN(1/d_a) and y = RN(x*r), |y - x/d_a| <= 2^-23 |x/d_a| and
// |RN(x/d_a) - x/d_a| <= 2^-24 |x/d_a|; for |x/d_a| <= 128 the two differ by
// less than 2^-15.  So when y lies more than 2^-12 away from every
// half-integer, rint(y) = rint(RN(x/d_a)); a lane with an element closer than
// that (or a block with a non-finite element, or d_a outside
// [2^-125, FLT_MAX]) takes the IEEE division for all its elements.  Codes,
// their 16h + l split and the sub-block sums are carried as exact floats.
__device__ __forceinline__ void quant_block_warp(const float (&v)[8], int row, int b, int K, uint8_t* act,
                                                 int8_t* q_dbg, float* da_dbg, int32_t* A_dbg,
                                                 int32_t* status) {
  const int lane = threadIdx.x & 31;
  float amax = 0.f;
  bool ok = true;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    ok = ok && fabsf(v[i]) <= 3.40282347e38f;          // false for inf and NaN
    amax = fmaxf(amax, fabsf(v[i]));
  }
  if (!ok) atomicOr(status, SPEC_ST_NONFINITE);
  const bool all_ok = __all_sync(0xffffffffu, ok);
  amax = warp_max(amax);
  const float d = amax / 127.0f;
  const bool exact = !all_ok || !(d == 0.f || (d >= 0x1p-125f && d <= 3.40282347e38f));
  const float r = (exact || d == 0.f) ? 0.f : __frcp_rn(d);
  float q[8];
  bool near = exact;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const float y = v[i] * r;
    q[i] = rintf(y);
    near = near || fabsf(fabsf(y - q[i]) - 0.5f) < 0x1p-12f;
  }
  if (near) {
#pragma unroll
    for (int i = 0; i < 8; ++i) q[i] = (d != 0.f && fabsf(v[i]) <= 3.40282347e38f) ? rintf(v[i] / d) : 0.f;
  }
  float part = 0.f;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    q[i] = fminf(fmaxf(q[i], -127.f), 127.f) + 0.f;     // + 0 turns -0 into +0
    part += q[i];
  }
  part += __shfl_xor_sync(0xffffffffu, part, 1);
  part += __shfl_xor_sync(0xffffffffu, part, 2);   // A_j for j = lane/4 (all 4 lanes of the quad)

  uint8_t* sb = act + (size_t)b * kActSBBytes;
  // codes: elements 8*lane + i = code k = 8*(lane%4) + i of sub-block lane/4;
  // q = 16h + l with h = floor(q/16)
  const int j = lane >> 2, q4 = lane & 3;
  float hv[8], lv[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    hv[i] = 16.f * floorf(q[i] * 0.0625f);
    lv[i] = q[i] - hv[i];
  }
  uint32_t hw[2], lw[2];
#pragma unroll
  for (int w = 0; w < 2; ++w) {
    hw[w] = e4m3x2(hv[4 * w], hv[4 * w + 1]) | (e4m3x2(hv[4 * w + 2], hv[4 * w + 3]) << 16);
    lw[w] = e4m3x2(lv[4 * w], lv[4 * w + 1]) | (e4m3x2(lv[4 * w + 2], lv[4 * w + 3]) << 16);
  }
  *reinterpret_cast<uint2*>(sb + act_off8(row, j, 0, 8 * q4)) = make_uint2(hw[0], hw[1]);
  *reinterpret_cast<uint2*>(sb + act_off8(row, j, 1, 8 * q4)) = make_uint2(lw[0], lw[1]);
  // min-term block: lane 4j writes 64*hi_j and lo_j of sub-block j
  if (q4 == 0) {
    const float hh = 64.f * floorf(part * 0.015625f), ll = part - hh;
    *reinterpret_cast<unsigned short*>(sb + act_off(row, 16, j)) = __half_as_ushort(__float2half_rn(hh));
    *reinterpret_cast<unsigned short*>(sb + act_off(row, 16, 8 + j)) = __half_as_ushort(__float2half_rn(ll));
  }
  if (lane == 0) reinterpret_cast<float*>(sb + kActSlots * 512)[row] = d;
  if (q_dbg) {
#pragma unroll
    for (int i = 0; i < 8; ++i) q_dbg[(size_t)row * K + 256 * b + 8 * lane + i] = (int8_t)(int)q[i];
    if ((lane & 3) == 0) A_dbg[(size_t)row * (K / 32) + 8 * b + (lane >> 2)] = (int)part;
    if (lane == 0) da_dbg[(size_t)row * (K / 256) + b] = d;
  }
}

// zero entries of a row >= M (codes 0, sums 0, d_a 0); in each of the 17
// blocks a row owns two 16-byte chunks, at k-halves 0 and 1
__device__ __forceinline__ void zero_block_warp(int row, int b, uint8_t* act) {
  const int lane = threadIdx.x & 31;
  uint8_t* sb = act + (size_t)b * kActSBBytes;
  for (int i = lane; i < kActSlots * 2; i += 32)      // 17 blocks x 2 k-halves x 16 bytes
    *reinterpret_cast<uint4*>(sb + act_off(row, i >> 1, 8 * (i & 1))) = make_uint4(0, 0, 0, 0);
  if (lane == 0) reinterpret_cast<float*>(sb + kActSlots * 512)[row] = 0.f;
}

}  // namespace spec
