// common.cuh — device helpers shared by the verify-step kernels (sm_103a).
//
// Everything here is hand-written inline PTX or CUDA built-ins: the legacy
// warp-level tensor-core MMA (m16n8k16, f16 inputs, f32 accumulate), 16-byte
// cp.async global->shared copies, LOP3 bit selection, packed f16x2 FMA and the
// packed f32x2 arithmetic introduced with sm_100.
#pragma once
#include <cstdint>
#include <cuda_fp16.h>
#include <cuda_bf16.h>

#include "../../include/spec_verify.h"

#define SPEC_DEV __device__ __forceinline__

namespace spec {

constexpr int kSB = 144;            // bytes per Q4_K superblock
constexpr int kTileSB = 16 * kSB;   // bytes per tiled (16 columns x 1 superblock) block
constexpr int kActSlots = 17;       // 16 k-steps + 1 min-term slot per superblock
constexpr int kActSBBytes = kActSlots * 512 + 64;   // + 16 fp32 d_a
constexpr int kPage = 16;

// ---- tensor core: D += A(16x16 f16, row) * B(16x8 f16, col), f32 accumulate
SPEC_DEV void mma16816(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                       uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};\n"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// bf16 variant (attention)
SPEC_DEV void mma16816_bf16(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                            uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};\n"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// ---- async copies
SPEC_DEV uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
SPEC_DEV void cp_async16(void* smem, const void* gmem) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(smem_u32(smem)), "l"(gmem));
}
SPEC_DEV void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::); }
template <int N>
SPEC_DEV void cp_async_wait() { asm volatile("cp.async.wait_group %0;\n" ::"n"(N)); }

// ---- bit tricks
// (a & b) | c
SPEC_DEV uint32_t lop3_and_or(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t d;
  asm("lop3.b32 %0, %1, %2, %3, 0xEA;\n" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}
SPEC_DEV uint32_t hfma2_u32(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t d;
  asm("fma.rn.f16x2 %0, %1, %2, %3;\n" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}
SPEC_DEV uint32_t hadd2_u32(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("add.rn.f16x2 %0, %1, %2;\n" : "=r"(d) : "r"(a), "r"(b));
  return d;
}
SPEC_DEV uint32_t hmul2_u32(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("mul.rn.f16x2 %0, %1, %2;\n" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

// ---- packed fp32 pairs (sm_100+): each lane of the pair rounds on its own
SPEC_DEV unsigned long long f2pack(float lo, float hi) {
  unsigned long long r;
  asm("mov.b64 %0, {%1,%2};\n" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
SPEC_DEV void f2unpack(unsigned long long v, float& lo, float& hi) {
  asm("mov.b64 {%0,%1}, %2;\n" : "=f"(lo), "=f"(hi) : "l"(v));
}
SPEC_DEV unsigned long long f2mul(unsigned long long a, unsigned long long b) {
  unsigned long long r;
  asm("mul.rn.f32x2 %0, %1, %2;\n" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
SPEC_DEV unsigned long long f2sub(unsigned long long a, unsigned long long b) {
  unsigned long long r;
  asm("sub.rn.f32x2 %0, %1, %2;\n" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
SPEC_DEV unsigned long long f2add(unsigned long long a, unsigned long long b) {
  unsigned long long r;
  asm("add.rn.f32x2 %0, %1, %2;\n" : "=l"(r) : "l"(a), "l"(b));
  return r;
}

SPEC_DEV float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
SPEC_DEV float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// Programmatic dependent launch: let the next kernel in the stream start its
// independent prologue (weight prefetch) early, and wait for the previous
// kernel's results before touching them.
SPEC_DEV void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;\n" ::); }
SPEC_DEV void pdl_wait() { asm volatile("griddepcontrol.wait;\n" ::: "memory"); }

// Query fragments for the attention MMAs: per head, 8 k-steps of 16 dims, a
// bf16 hi part and a bf16 lo part (x - hi), 32 lanes x 16 bytes in the
// m16n8k16 A-fragment order (row = query row of the block).
SPEC_DEV void write_qfrag(uint8_t* qf, int row, int head, int d, float v) {
  const int kk = d >> 4, within = d & 15;
  const int t = (within & 7) >> 1, u = within & 1;
  const int reg = (row >> 3) + ((within >> 3) << 1);
  const int lane = 4 * (row & 7) + t;
  const __nv_bfloat16 hi = __float2bfloat16_rn(v);
  const __nv_bfloat16 lo = __float2bfloat16_rn(v - __bfloat162float(hi));
  const size_t base = ((size_t)(head * 8 + kk) * 2) * 32 * 16 + (size_t)lane * 16 + reg * 4 + u * 2;
  *reinterpret_cast<unsigned short*>(qf + base) = __bfloat16_as_ushort(hi);
  *reinterpret_cast<unsigned short*>(qf + base + 32 * 16) = __bfloat16_as_ushort(lo);
}

}  // namespace spec
