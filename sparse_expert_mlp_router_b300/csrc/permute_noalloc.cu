// moe_permute_noalloc: the grouping stage without a caller-provided workspace.
//
// Some callers cannot call cudaMalloc: code that enqueues work while a CUDA
// stream is being captured into a graph (allocation is not allowed there),
// plug-ins whose host framework owns every byte of device memory and hands out
// only the tensors of the call, and real-time loops that must not touch the
// allocator after start-up. For them this entry point keeps the one piece of
// scratch the grouping kernels need -- the per-chunk expert histogram, which
// the scan turns into per-chunk rank bases -- in a fixed array in the
// library's own device memory, so the call needs nothing beyond its inputs
// and outputs.
//
// Limits and sharing:
//   * the array holds kNoAllocScratchInts int32 (256 KiB); a configuration
//     needs ceil(T/128) * E of them, so e.g. T <= 32768 at E = 256 or
//     T <= 65536 at E = 128. Larger configurations are refused with
//     MOE_ERR_WORKSPACE before anything is enqueued.
//   * every GPU that loads libmoe.so holds the array until the process exits.
//   * every call on a device uses the same array and leaves its contents
//     behind; the kernels overwrite every entry they read, so nothing has to
//     start at zero. Two calls that overlap on the GPU (different streams
//     without ordering between them) race on the array and give wrong results.
//   * the device address of the array is looked up once per device, by the
//     first call made while that device is current (cudaGetSymbolAddress).
//     Make that first call before any stream capture begins.
#include <mutex>

#include "internal.cuh"

namespace moe {
namespace {

constexpr int64_t kNoAllocScratchInts = 65536;
constexpr int kMaxDevices = 64;

// Host code must not use this name as a device address; see scratch_address().
static __device__ __align__(256) int32_t g_group_scratch[kNoAllocScratchInts];

std::mutex g_mu;
int32_t* g_addr[kMaxDevices] = {nullptr};

// Device address of g_group_scratch on the current device (looked up once per device).
cudaError_t scratch_address(int32_t** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_mu);
  if (g_addr[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_group_scratch);
    if (e != cudaSuccess) return e;
    g_addr[dev] = static_cast<int32_t*>(p);
  }
  *out = g_addr[dev];
  return cudaSuccess;
}

}  // namespace
}  // namespace moe

extern "C" moe_status_t moe_permute_noalloc(const moe_config_t* cfg, const int32_t* topk_idx, const void* x,
                                            int32_t* counts, int32_t* offsets, int32_t* dest_row,
                                            int32_t* src_token, void* x_perm, int32_t* status,
                                            cudaStream_t stream) {
  using namespace moe;
  moe_status_t rc = moe_check_config(cfg);
  if (rc != MOE_OK) return rc;
  if (!topk_idx || !x || !counts || !offsets || !dest_row || !src_token || !x_perm) return MOE_ERR_INVALID_ARG;
  auto al = [](const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; };
  if (!al(topk_idx, 4) || !al(x, 16) || !al(counts, 4) || !al(offsets, 4) || !al(dest_row, 4) ||
      !al(src_token, 4) || !al(x_perm, 16) || (status && !al(status, 4)))
    return MOE_ERR_INVALID_ARG;
  const Shape s = make_shape(*cfg);
  if ((int64_t)s.nchunks * s.E > kNoAllocScratchInts) return MOE_ERR_WORKSPACE;
  int32_t* scratch = nullptr;
  if (scratch_address(&scratch) != cudaSuccess) return MOE_ERR_CUDA;
  if (launch_group_hist(s, topk_idx, scratch, status, stream) != cudaSuccess) return MOE_ERR_CUDA;
  if (launch_group_scan(s, scratch, counts, offsets, nullptr, stream) != cudaSuccess) return MOE_ERR_CUDA;
  if (launch_group_scatter(s, topk_idx, scratch, offsets, dest_row, src_token, stream) != cudaSuccess)
    return MOE_ERR_CUDA;
  if (launch_gather_rows(s, x, src_token, offsets, x_perm, stream) != cudaSuccess) return MOE_ERR_CUDA;
  return MOE_OK;
}
