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
constexpr int kActSlots = 17;       // 16 k-steps + 1 min-term slot per superblock
constexpr int kActSBBytes = kActSlots * 512 + 64;   // + 16 fp32 d_a
constexpr int kTreeMax = 64;        // nodes of a token tree (passes of up to 16 rows)

// ---- shared-memory addresses
SPEC_DEV uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
// ---- packed f16 arithmetic
SPEC_DEV uint32_t hadd2_u32(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("add.rn.f16x2 %0, %1, %2;\n" : "=r"(d) : "r"(a), "r"(b));
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
SPEC_DEV unsigned long long f2fma(unsigned long long a, unsigned long long b, unsigned long long c) {
  unsigned long long r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;\n" : "=l"(r) : "l"(a), "l"(b), "l"(c));
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

// Thread-block cluster: this CTA's rank, a store into a peer CTA's shared
// memory, and the cluster-wide barrier (release on arrive, acquire on wait).
SPEC_DEV uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;\n" : "=r"(r));
  return r;
}
SPEC_DEV void st_cluster_f32(const float* local, uint32_t rank, float v) {
  uint32_t remote;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;\n" : "=r"(remote) : "r"(smem_u32(local)), "r"(rank));
  asm volatile("st.shared::cluster.f32 [%0], %1;\n" ::"r"(remote), "f"(v) : "memory");
}
SPEC_DEV void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n" ::: "memory");
  asm volatile("barrier.cluster.wait.acquire.aligned;\n" ::: "memory");
}

// status bits after which a step does no work on the block (nothing was
// reserved in the KV)
constexpr int32_t kStepAbort = SPEC_ST_TOKEN_RANGE | SPEC_ST_POOL_EMPTY | SPEC_ST_CTX_FULL | SPEC_ST_BAD_TREE;

// Programmatic dependent launch: let the next kernel in the stream start its
// independent prologue (weight prefetch) early, and wait for the previous
// kernel's results before touching them.
SPEC_DEV void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;\n" ::); }
SPEC_DEV void pdl_wait() { asm volatile("griddepcontrol.wait;\n" ::: "memory"); }

// ---- 5th-generation tensor core (tcgen05) and mbarriers
SPEC_DEV void tmem_alloc(uint32_t* slot, int ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;\n" ::"r"(smem_u32(slot)),
               "r"(ncols));
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;\n" ::);
}
SPEC_DEV void tmem_dealloc(uint32_t taddr, int ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;\n" ::"r"(taddr), "r"(ncols));
}
// make this thread's completed generic-proxy shared-memory writes (including
// cp.async) visible to the async proxy that the tensor core reads through
SPEC_DEV void fence_proxy_async() { asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory"); }
SPEC_DEV void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;\n" ::: "memory"); }
SPEC_DEV void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;\n" ::: "memory"); }
SPEC_DEV void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;\n" ::: "memory"); }
SPEC_DEV void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;\n" ::: "memory"); }
// this warp's 32 lanes, 32 consecutive 32-bit columns
SPEC_DEV void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};\n" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
      "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]),
      "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]),
      "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31]));
}
SPEC_DEV void tmem_st4(uint32_t taddr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x4.b32 [%0], {%1,%2,%3,%4};\n" ::"r"(taddr), "r"(a), "r"(b),
               "r"(c), "r"(d));
}
// D[tmem] (+)= A[tmem] * B[smem]^T, kind::f16 (f16 inputs, f32 accumulate), issued by one thread
SPEC_DEV void mma_f16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.u32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}\n" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate));
}
// D[tmem] (+)= A[tmem] * B[smem]^T, kind::f8f6f4 (8-bit float inputs, types in
// idesc; f32 accumulate), K = 32 per instruction, issued by one thread
SPEC_DEV void mma_f8_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.u32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], [%1], %2, %3, p;\n}\n" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate));
}
SPEC_DEV void mma_commit(uint64_t* mbar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n" ::"r"(
      smem_u32(mbar)));
}
SPEC_DEV void mbar_init(uint64_t* mbar, int count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;\n" ::"r"(smem_u32(mbar)), "r"(count));
}
SPEC_DEV uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;\n" : "=l"(t));
  return t;
}
// one try_wait on the phase with the given parity; the thread may be suspended
// for up to ~0.5 ms while the phase is incomplete (woken early when it completes)
SPEC_DEV bool mbar_try(uint64_t* mbar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(done)
      : "r"(smem_u32(mbar)), "r"(parity), "r"(500000u)
      : "memory");
  return done != 0;
}
// wait for the phase with the given parity, giving up after limit_ns of wall
// time (the bound holds whatever the hardware does with the suspend hint; the
// clock is read once per 32 tries to keep the loop short)
SPEC_DEV bool mbar_wait_ns(uint64_t* mbar, uint32_t parity, uint64_t limit_ns) {
  if (mbar_try(mbar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (;;) {
#pragma unroll 1
    for (int k = 0; k < 32; ++k)
      if (mbar_try(mbar, parity)) return true;
    if (globaltimer_ns() - t0 > limit_ns) return false;
  }
}
// arrive once and add tx_bytes to the bytes the current phase waits for
SPEC_DEV void mbar_arrive_expect_tx(uint64_t* mbar, uint32_t tx_bytes) {
  asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;\n" ::"r"(smem_u32(mbar)),
               "r"(tx_bytes)
               : "memory");
}
// bulk (non-tensor) copy global -> shared, completion counted on mbar in bytes;
// both addresses 16-byte aligned, bytes a multiple of 16
SPEC_DEV void bulk_g2s(void* dst_smem, const void* src, uint32_t bytes, uint64_t* mbar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;\n" ::"r"(
          smem_u32(dst_smem)),
      "l"(src), "r"(bytes), "r"(smem_u32(mbar)), "l"(policy)
      : "memory");
}
// the same without an L2 cache hint
SPEC_DEV void bulk_g2s(void* dst_smem, const void* src, uint32_t bytes, uint64_t* mbar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];\n" ::"r"(
                   smem_u32(dst_smem)),
               "l"(src), "r"(bytes), "r"(smem_u32(mbar))
               : "memory");
}
SPEC_DEV void fence_mbarrier_init() { asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory"); }
SPEC_DEV uint64_t l2_policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;\n" : "=l"(p));
  return p;
}
SPEC_DEV uint64_t l2_policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;\n" : "=l"(p));
  return p;
}
// true in exactly one lane of the converged warp (tcgen05 issue from a
// converged warp keeps the operands in uniform registers)
SPEC_DEV bool elect_one() {
  uint32_t p;
  asm volatile("{\n .reg .pred e;\n elect.sync _|e, 0xffffffff;\n selp.u32 %0, 1, 0, e;\n}\n" : "=r"(p));
  return p != 0;
}
SPEC_DEV void mbar_arrive(uint64_t* mbar) {
  asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];\n" ::"r"(smem_u32(mbar)) : "memory");
}
// named barrier over `count` threads with an AND reduction of `pred`
SPEC_DEV bool named_bar_and(int id, int count, bool pred) {
  uint32_t r;
  asm volatile(
      "{\n .reg .pred p, q;\n setp.ne.u32 p, %1, 0;\n bar.red.and.pred q, %2, %3, p;\n"
      " selp.u32 %0, 1, 0, q;\n}\n"
      : "=r"(r)
      : "r"((uint32_t)pred), "r"(id), "r"(count)
      : "memory");
  return r != 0;
}
// shared-memory matrix descriptor: canonical K-major layout without swizzle;
// lbo = byte stride between core matrices along K, sbo = along M/N
SPEC_DEV uint64_t smem_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = (uint64_t)((saddr & 0x3FFFFu) >> 4);
  d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
  d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
  d |= (uint64_t)1 << 46;   // descriptor version of the sm_100 family
  return d;
}

// Query tiles of the attention MMAs: per (kv head, tile of 8 query heads) a
// 64 KB block: the bf16 hi parts, then the lo parts (x - hi), each as two d
// halves of [128 rows][128 B], row = 16 * (head % 8) + block row, with the
// 16-byte chunk j of row r at j ^ (r % 8) (the 128-byte swizzle of the MMA
// operand).
SPEC_DEV void write_qtile(uint8_t* qt, int row, int head, int d, float v, int group, int tiles) {
  const int kvh = head / group, hl = head - kvh * group;
  const int r = ((hl & 7) << 4) + row;
  const int half = d >> 6, j = (d & 63) >> 3, e = d & 7;
  const size_t base = (size_t)(kvh * tiles + (hl >> 3)) * 65536 + (size_t)half * 16384 + (size_t)r * 128 +
                      (size_t)((j ^ (r & 7)) << 4) + 2 * e;
  const __nv_bfloat16 hi = __float2bfloat16_rn(v);
  const __nv_bfloat16 lo = __float2bfloat16_rn(v - __bfloat162float(hi));
  *reinterpret_cast<unsigned short*>(qt + base) = __bfloat16_as_ushort(hi);
  *reinterpret_cast<unsigned short*>(qt + base + 32768) = __bfloat16_as_ushort(lo);
}

}  // namespace spec
