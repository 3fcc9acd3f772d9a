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
// e4m3 bits of an integer v with |v| <= 240 and at most 4 significant bits
// (sign, 4-bit exponent with bias 7, 3-bit mantissa), read off its fp32 bits
SPEC_DEV uint32_t e4m3_of_int(int v) {
  if (v == 0) return 0u;
  const uint32_t b = __float_as_uint((float)v);
  const uint32_t e = ((b >> 23) & 255u) - 127u + 7u;
  return ((b >> 24) & 0x80u) | (e << 3) | ((b >> 20) & 7u);
}

// Quantisation of one 256-block of one row, executed by one warp.  Lane l owns
// elements 8l..8l+7 (sub-block l/4).
__device__ __forceinline__ void quant_block_warp(const float (&v)[8], int row, int b, int K, uint8_t* act,
                                                 int8_t* q_dbg, float* da_dbg, int32_t* A_dbg,
                                                 int32_t* status) {
  const int lane = threadIdx.x & 31;
  float amax = 0.f;
  bool bad = false;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    bad |= !isfinite(v[i]);
    amax = fmaxf(amax, fabsf(v[i]));
  }
  amax = warp_max(amax);
  if (bad) atomicOr(status, SPEC_ST_NONFINITE);
  const float d = amax / 127.0f;
  int q[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    int c = 0;
    if (d != 0.f && isfinite(v[i])) {
      float r = rintf(v[i] / d);
      r = fminf(fmaxf(r, -127.f), 127.f);
      c = (int)r;
    }
    q[i] = c;
  }
  int part = 0;
#pragma unroll
  for (int i = 0; i < 8; ++i) part += q[i];
  part += __shfl_xor_sync(0xffffffffu, part, 1);
  part += __shfl_xor_sync(0xffffffffu, part, 2);   // A_j for j = lane/4 (all 4 lanes of the quad)

  uint8_t* sb = act + (size_t)b * kActSBBytes;
  // codes: elements 8*lane + i = code k = 8*(lane%4) + i of sub-block lane/4
  const int j = lane >> 2, q4 = lane & 3;
  uint32_t hw[2] = {0u, 0u}, lw[2] = {0u, 0u};
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int l = q[i] & 15, h = q[i] >> 4;     // q = 16h + l (arithmetic shift: floor)
    hw[i >> 2] |= e4m3_of_int(16 * h) << (8 * (i & 3));
    lw[i >> 2] |= e4m3_of_int(l) << (8 * (i & 3));
  }
  *reinterpret_cast<uint2*>(sb + act_off8(row, j, 0, 8 * q4)) = make_uint2(hw[0], hw[1]);
  *reinterpret_cast<uint2*>(sb + act_off8(row, j, 1, 8 * q4)) = make_uint2(lw[0], lw[1]);
  // min-term block: lane 4j writes 64*hi_j and lo_j of sub-block j
  if (q4 == 0) {
    const int hh = part >> 6, ll = part & 63;
    *reinterpret_cast<unsigned short*>(sb + act_off(row, 16, j)) = __half_as_ushort(__int2half_rn(64 * hh));
    *reinterpret_cast<unsigned short*>(sb + act_off(row, 16, 8 + j)) = __half_as_ushort(__int2half_rn(ll));
  }
  if (lane == 0) reinterpret_cast<float*>(sb + kActSlots * 512)[row] = d;
  if (q_dbg) {
#pragma unroll
    for (int i = 0; i < 8; ++i) q_dbg[(size_t)row * K + 256 * b + 8 * lane + i] = (int8_t)q[i];
    if ((lane & 3) == 0) A_dbg[(size_t)row * (K / 32) + 8 * b + (lane >> 2)] = part;
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
