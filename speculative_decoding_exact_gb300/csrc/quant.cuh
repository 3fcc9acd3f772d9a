// quant.cuh — per-row, per-256-block activation quantisation into the
// fragment-ordered activation buffer read by the Q4_K GEMM.
//   d_a = amax/127 (IEEE fp32 division), q = clamp(rint(x/d_a), -127, 127)
//   with round-half-even, all-zero block -> d_a = 0, q = 0; A_j = sum of the
//   32 codes of sub-block j.
#pragma once
#include "common.cuh"

namespace spec {

// ---------------------------------------------------------------------------
// Quantisation of one 256-block of one row, executed by one warp.  Lane l owns
// elements 8l..8l+7 (sub-block l/4).  Writes the block's entries of the
// activation buffer for this row:
//   slot s (k-step), lane (g = row%8, t), word (row<8 ? 0 : 2) + P:
//   f16 pair of codes at elements 64t + 32P + 2s + {0, 1} (P = 0, 1)
//   slot 16 words {64*hi_2t, 64*hi_2t+1} and {lo_2t, lo_2t+1}, A_j = 64 hi + lo
//   slot 17: d_a (fp32) at 4*row
// ---------------------------------------------------------------------------
__device__ __forceinline__ void quant_block_warp(const float (&v)[8], int row, int b, int K, uint8_t* act,
                                 int8_t* q_dbg, float* da_dbg, int32_t* A_dbg, int32_t* status) {
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
  const int g = row & 7, rw = row >> 3;
  // codes: element e = 8*lane + i, pairs (e, e+1); k-slot map of the GEMM:
  // e = 64t + 32P + 2s + u -> step s, lane (g, t), word 2*rw + P, half u
#pragma unroll
  for (int i = 0; i < 8; i += 2) {
    const int e = 8 * lane + i;
    const int t = e >> 6, within = e & 63;
    const int s = (within & 31) >> 1;
    const int word = 2 * rw + (within >> 5);
    const uint32_t lo = __half_as_ushort(__int2half_rn(q[i]));
    const uint32_t hi = __half_as_ushort(__int2half_rn(q[i + 1]));
    reinterpret_cast<uint32_t*>(sb + s * 512 + (4 * g + t) * 16)[word] = lo | (hi << 16);
  }
  // min-term slot: lane 4j holds A_j; lanes t = 0..3 write pairs (2t, 2t+1)
  const int A_even = __shfl_sync(0xffffffffu, part, (8 * (lane & 3)) & 31);
  const int A_odd = __shfl_sync(0xffffffffu, part, (8 * (lane & 3) + 4) & 31);
  if (lane < 4) {
    const int t = lane;
    const int he = A_even >> 6, le = A_even & 63;
    const int ho = A_odd >> 6, lo = A_odd & 63;
    uint32_t* w = reinterpret_cast<uint32_t*>(sb + 16 * 512 + (4 * g + t) * 16);
    w[2 * rw] = (uint32_t)__half_as_ushort(__int2half_rn(64 * he)) |
                ((uint32_t)__half_as_ushort(__int2half_rn(64 * ho)) << 16);
    w[2 * rw + 1] = (uint32_t)__half_as_ushort(__int2half_rn(le)) |
                    ((uint32_t)__half_as_ushort(__int2half_rn(lo)) << 16);
  }
  if (lane == 0) reinterpret_cast<float*>(sb + kActSlots * 512)[row] = d;
  if (q_dbg) {
#pragma unroll
    for (int i = 0; i < 8; ++i) q_dbg[(size_t)row * K + 256 * b + 8 * lane + i] = (int8_t)q[i];
    if ((lane & 3) == 0) A_dbg[(size_t)row * (K / 32) + 8 * b + (lane >> 2)] = part;
    if (lane == 0) da_dbg[(size_t)row * (K / 256) + b] = d;
  }
}

// zero entries of a row >= M (codes 0, sums 0, d_a 0)
__device__ __forceinline__ void zero_block_warp(int row, int b, uint8_t* act) {
  const int lane = threadIdx.x & 31;
  uint8_t* sb = act + (size_t)b * kActSBBytes;
  const int g = row & 7, rw = row >> 3;
  // 17 slots x 4 t x 2 words
  for (int i = lane; i < 17 * 4 * 2; i += 32) {
    const int s = i >> 3, t = (i >> 1) & 3, wd = 2 * rw + (i & 1);
    reinterpret_cast<uint32_t*>(sb + s * 512 + (4 * g + t) * 16)[wd] = 0u;
  }
  if (lane == 0) reinterpret_cast<float*>(sb + kActSlots * 512)[row] = 0.f;
}

}  // namespace spec
