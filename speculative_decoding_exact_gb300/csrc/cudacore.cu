// cudacore.cu — the skinny Q4_K x Q8 GEMM on CUDA cores (dp4a), the baseline
// against which the tensor-core kernel (gemm.cu) was chosen.
//
// The integer sums are the same exact quantities as the tensor-core path's
// (Muser book Ch. 32 "Precision across the handoff" §32.7, the integer-dot
// anchor): S_j = sum of 32 products q_w * q_a, eight 4-way byte dot products
// (dp4a) per sub-block and row; ISc = sum_j sc_j S_j and IMn = sum_j m_j A_j
// in int32; v_b = d_a * (d * ISc - dmin * IMn) in fp32, each operation
// rounded on its own.  Only the sum of the v_b over superblocks differs from
// gemm.cu: the superblock ranges of a column are split over CTAs and the
// ranges' sums are added with atomics, so the result is within rounding of
// the tensor-core path, not bit-identical to it.
//
// CTA (128 columns, range of superblocks), one thread per column: per
// superblock the CTA stages the 16 rows' int8 codes (4 KB) in shared memory;
// each thread reads its column's 144-byte superblock (the tiled layout keeps
// the 128 columns of a superblock contiguous), masks the nibbles into bytes
// and runs 1,024 dp4a for the 16 rows.
#include "common.cuh"
#include "internal.h"

namespace spec {

constexpr int kCcCols = 128;

__global__ void __launch_bounds__(kCcCols)
gemm_q4k_dp4a_kernel(const uint8_t* __restrict__ wt, const int8_t* __restrict__ q, const float* __restrict__ da,
                     const int32_t* __restrict__ A, int M, int N, int nb, int sb_per_cta, float* __restrict__ y) {
  __shared__ __align__(16) int32_t qa_s[16][64];     // 16 rows x 256 codes, 4 per word
  __shared__ int32_t a_s[16][8];
  __shared__ float da_s[16];
  const int T = blockIdx.x, c = threadIdx.x;
  const int col = kCcCols * T + c;
  const int cols = min(kCcCols, N - kCcCols * T);
  const int b0 = blockIdx.y * sb_per_cta, b1 = min(nb, b0 + sb_per_cta);
  float acc[16];
#pragma unroll
  for (int m = 0; m < 16; ++m) acc[m] = 0.f;
  for (int b = b0; b < b1; ++b) {
    __syncthreads();
    for (int i = c; i < 16 * 64; i += kCcCols) {
      const int m = i >> 6, w = i & 63;
      qa_s[m][w] = m < M ? reinterpret_cast<const int32_t*>(q + (size_t)m * nb * 256 + (size_t)b * 256)[w] : 0;
    }
    if (c < 128) {
      const int m = c >> 3, j = c & 7;
      a_s[m][j] = m < M ? A[(size_t)m * nb * 8 + (size_t)b * 8 + j] : 0;
    }
    if (c < 16) da_s[c] = c < M ? da[(size_t)c * nb + b] : 0.f;
    __syncthreads();
    if (c >= cols) continue;
    const uint4* sb = reinterpret_cast<const uint4*>(wt + ((size_t)kCcCols * T * nb + (size_t)b * cols + c) * kSB);
    const uint4 hdr = sb[0];
    const float d = __half2float(__ushort_as_half((unsigned short)(hdr.x & 0xffff)));
    const float dm = __half2float(__ushort_as_half((unsigned short)(hdr.x >> 16)));
    int sc[8], mn[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int p = 6 * j, r = 48 + 6 * j;
      sc[j] = (int)(__funnelshift_r(p < 32 ? hdr.y : hdr.z, p < 32 ? hdr.z : hdr.w, p & 31) & 63u);
      mn[j] = (int)(__funnelshift_r(r < 64 ? hdr.z : hdr.w, r < 64 ? hdr.w : 0u, r & 31) & 63u);
    }
    int isc[16];
#pragma unroll
    for (int m = 0; m < 16; ++m) isc[m] = 0;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const uint4 cw = sb[1 + j];
      const uint32_t w4[4] = {cw.x, cw.y, cw.z, cw.w};
      int lo[4], hi[4];                              // elements 4t..4t+3 and 16+4t..
#pragma unroll
      for (int t = 0; t < 4; ++t) {
        lo[t] = (int)(w4[t] & 0x0F0F0F0Fu);
        hi[t] = (int)((w4[t] >> 4) & 0x0F0F0F0Fu);
      }
#pragma unroll
      for (int m = 0; m < 16; ++m) {
        const int4 a0 = *reinterpret_cast<const int4*>(&qa_s[m][8 * j]);
        const int4 a1 = *reinterpret_cast<const int4*>(&qa_s[m][8 * j + 4]);
        int s = 0;
        s = __dp4a(lo[0], a0.x, s);
        s = __dp4a(lo[1], a0.y, s);
        s = __dp4a(lo[2], a0.z, s);
        s = __dp4a(lo[3], a0.w, s);
        s = __dp4a(hi[0], a1.x, s);
        s = __dp4a(hi[1], a1.y, s);
        s = __dp4a(hi[2], a1.z, s);
        s = __dp4a(hi[3], a1.w, s);
        isc[m] += sc[j] * s;
      }
    }
#pragma unroll
    for (int m = 0; m < 16; ++m) {
      int imn = 0;
#pragma unroll
      for (int j = 0; j < 8; ++j) imn += mn[j] * a_s[m][j];
      const float v = __fmul_rn(da_s[m], __fsub_rn(__fmul_rn(d, (float)isc[m]), __fmul_rn(dm, (float)imn)));
      acc[m] = __fadd_rn(acc[m], v);
    }
  }
  if (c < cols)
    for (int m = 0; m < M; ++m) atomicAdd(y + (size_t)m * N + col, acc[m]);
}

cudaError_t launch_gemm_dp4a(const void* w_tiled, const int8_t* q, const float* da, const int32_t* A, int M,
                             int N, int K, float* y, int num_sms, cudaStream_t st) {
  const int nb = K / 256, tiles = (N + kCcCols - 1) / kCcCols;
  // about four CTAs per SM in all
  int splits = (4 * num_sms + tiles - 1) / tiles;
  if (splits > nb) splits = nb;
  if (splits < 1) splits = 1;
  const int per = (nb + splits - 1) / splits;
  splits = (nb + per - 1) / per;
  cudaError_t e = cudaMemsetAsync(y, 0, sizeof(float) * (size_t)M * N, st);
  if (e != cudaSuccess) return e;
  gemm_q4k_dp4a_kernel<<<dim3(tiles, splits), kCcCols, 0, st>>>(static_cast<const uint8_t*>(w_tiled), q, da, A,
                                                                 M, N, nb, per, y);
  return cudaGetLastError();
}

}  // namespace spec
