// gemm_plan.h — the work plan and the warp layout of the skinny Q4_K GEMM
// (gemm.cu), shared with the host-side code that sizes its workspaces.
#pragma once
#include <cstddef>
#include <cuda_runtime.h>

namespace spec {

// Work plan of one skinny Q4_K GEMM.  Columns are cut into 16-wide tiles and
// the tiles into groups of kTilesPerGroup; a work unit is (group, superblock).
// Units are numbered group-major and CTA i of G owns units
// [floor(i*U/G), floor((i+1)*U/G)).  Every (CTA, group) run writes one fp32
// partial "piece" of the group's 16 x (16*kTilesPerGroup) outputs into slot
// (i - first CTA of that group); the consumer adds the slots in order.  The
// plan depends only on (N, K, number of SMs), never on the row count M.
struct GemmPlan {
  int N = 0, K = 0, nb = 0, ntiles = 0, ngroups = 0, G = 0, max_slots = 0;
  long long U = 0;
  int pre_stages = 3;   // stages whose weights are fetched before the dependency wait (<= 6)
};

// tcgen05 GEMM: one CTA per SM owns 128 weight columns (one per TMEM lane).
// Warp roles: 4 unpack warps and 4 combine warps (one thread per column each),
// one warp that issues the bulk copies, and kGemmMmaWarps warps that share the
// 17 MMAs of a superblock.
constexpr int kGemmUnpackWarps = 4;
constexpr int kGemmUnpackThreads = 32 * kGemmUnpackWarps;
constexpr int kGemmCombineThreads = 128;
constexpr int kGemmMmaWarps = 2;
constexpr int kGemmThreads = kGemmUnpackThreads + kGemmCombineThreads + 32 + 32 * kGemmMmaWarps;
constexpr int kTilesPerGroup = 8;          // 16-column tiles per group = 128 columns
constexpr int kGemmCols = 16 * kTilesPerGroup;
constexpr int kGemmStages = 6;
constexpr int kGemmCtasPerSm = 1;
constexpr int kMaxSlots = 8;      // pieces per group, guaranteed by make_gemm_plan

GemmPlan make_gemm_plan(int N, int K, int num_sms);
cudaError_t gemm_init_attributes();   // once per device, before any launch or capture
size_t gemm_smem_bytes();
// slots of group gr, and the CTA owning a unit (host mirror of the device math)
int plan_slots_of_group(const GemmPlan& p, int gr);

}  // namespace spec
