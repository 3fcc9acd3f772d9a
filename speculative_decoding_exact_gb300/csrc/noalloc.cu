// noalloc.cu — a Q4_K GEMM entry point that never allocates device memory.
//
// Some callers cannot call cudaMalloc: code that runs where an allocation
// could block or fail at the wrong moment (a real-time decode loop that must
// not take the allocator's lock, a process whose memory was reserved up front
// by another runtime, an embedding host that forbids the CUDA allocator).
// spec_gemm_q4k needs a spec_ctx, whose workspace is allocated by
// spec_verify_init.  This file gives those callers spec_gemm_q4k_noalloc: the
// same kernels (activation quantiser, skinny GEMM, ordered sum of the
// partial pieces) with their scratch taken from one fixed array that the
// library reserves as a file-scope __device__ variable when it is loaded.
//
// Properties a caller must know:
//   * the scratch is kNoAllocScratchBytes (8 MiB) on every device that loads
//     the library, held until the process exits;
//   * a request whose activations plus partial pieces do not fit is rejected
//     with SPEC_ECAPACITY before anything is enqueued;
//   * every call on a device uses the same array: two calls whose work
//     overlaps on the GPU (different streams, no ordering between them) race
//     and corrupt each other's results; calls ordered on one stream are safe;
//   * the first call on a device looks up the array's device address with
//     cudaGetSymbolAddress while that device is current, and raises the GEMM
//     kernel's shared-memory limit on that device; make that first call before
//     capturing any stream into a CUDA graph;
//   * device-detected conditions (a non-finite activation, a bounded device
//     wait that gave up, after which y is incomplete) are OR-ed into a status
//     word at the start of the array, cleared by every call;
//     spec_gemm_q4k_noalloc_status reads it back without allocating.
#include <mutex>

#include "../../include/spec_verify.h"
#include "common.cuh"
#include "internal.h"

namespace {

constexpr size_t kNoAllocScratchBytes = size_t(8) << 20;
constexpr int kMaxDevices = 64;

// Scratch: [status word, padded to 256 B][activation buffer][partial pieces]
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

struct DeviceSlot {
  bool ready = false;
  unsigned char* scratch = nullptr;   // device address of g_noalloc_scratch
  int num_sms = 0;
};
DeviceSlot g_slots[kMaxDevices];
std::mutex g_slots_mu;

int device_slot(DeviceSlot** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return SPEC_ENODEV;
  std::lock_guard<std::mutex> lock(g_slots_mu);
  DeviceSlot& s = g_slots[dev];
  if (!s.ready) {
    int major = 0, minor = 0, sms = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return SPEC_ECUDA;
    if (major != 10 || minor != 3) return SPEC_ENODEV;
    void* p = nullptr;
    // the host-side symbol is only a stand-in: the kernels need the device address
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) return SPEC_ECUDA;
    // the shared-memory limit is a per-device attribute
    if (spec::gemm_init_attributes() != cudaSuccess) return SPEC_ECUDA;
    s.scratch = static_cast<unsigned char*>(p);
    s.num_sms = sms;
    s.ready = true;
  }
  *out = &s;
  return SPEC_OK;
}

}  // namespace

extern "C" SPEC_API int spec_gemm_q4k_noalloc(const void* w_tiled, int N, int K, const float* x,
                                              int M, float* y, void* cuda_stream) {
  using namespace spec;
  if (!w_tiled || !x || !y) return SPEC_ENULL;
  if (M < 1 || M > 16 || N <= 0 || K <= 0 || N % 16 || K % 256) return SPEC_EINVAL;
  if ((reinterpret_cast<uintptr_t>(w_tiled) | reinterpret_cast<uintptr_t>(x)) % 16) return SPEC_EALIGN;
  DeviceSlot* slot = nullptr;
  int rc = device_slot(&slot);
  if (rc) return rc;
  const GemmPlan p = make_gemm_plan(N, K, slot->num_sms);
  const size_t status_bytes = 256;
  const size_t act_bytes = (size_t)(K / 256) * kActSBBytes;
  const size_t act_off = status_bytes;
  const size_t pieces_off = (act_off + act_bytes + 255) / 256 * 256;
  const size_t pieces_bytes = (size_t)p.max_slots * 16 * p.N * sizeof(float);
  if (pieces_off + pieces_bytes > kNoAllocScratchBytes) return SPEC_ECAPACITY;

  cudaStream_t st = static_cast<cudaStream_t>(cuda_stream);
  int32_t* status = reinterpret_cast<int32_t*>(slot->scratch);
  uint8_t* act = slot->scratch + act_off;
  float* pieces = reinterpret_cast<float*>(slot->scratch + pieces_off);
  // the status word is the only scratch that must start at zero: the quantiser
  // rewrites every activation entry (rows beyond M as zeros) and the GEMM
  // rewrites every piece slot before it is summed
  if (cudaMemsetAsync(status, 0, sizeof(int32_t), st) != cudaSuccess) return SPEC_ECUDA;
  if (launch_quantize(x, M, K, act, nullptr, nullptr, nullptr, status, st, false) != cudaSuccess)
    return SPEC_ECUDA;
  if (launch_gemm(p, w_tiled, act, pieces, nullptr, nullptr, 0, status, st, true) != cudaSuccess)
    return SPEC_ECUDA;
  if (launch_sum_pieces(p, pieces, y, M, st, true) != cudaSuccess) return SPEC_ECUDA;
  return SPEC_OK;
}

extern "C" SPEC_API int spec_gemm_q4k_noalloc_status(void* cuda_stream) {
  DeviceSlot* slot = nullptr;
  int rc = device_slot(&slot);
  if (rc) return rc;
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(cuda_stream)) != cudaSuccess) return SPEC_ECUDA;
  int32_t word = 0;
  if (cudaMemcpy(&word, slot->scratch, sizeof(word), cudaMemcpyDeviceToHost) != cudaSuccess) return SPEC_ECUDA;
  return word;
}
