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
//   * a batch of at most 128 tokens (one chunk: decode-sized batches) is grouped
//     in one launch whose blocks each keep the histogram in their own shared
//     memory; such calls never touch the array below and cannot race with other
//     calls;
//   * larger batches use the array: kNoAllocScratchInts int32 (256 KiB); a
//     configuration needs ceil(T/128) * E of them, so e.g. T <= 32768 at E = 256
//     or T <= 65536 at E = 128. Larger configurations are refused with
//     MOE_ERR_WORKSPACE before anything is enqueued.
//   * every GPU that loads libmoe.so holds the array until the process exits.
//   * every call on a device uses the same array and leaves its contents
//     behind; the kernels overwrite every entry they read, so nothing has to
//     start at zero. Two calls that overlap on the GPU (different streams
//     without ordering between them) race on the array and give wrong results.
//   * the device address of the array is looked up (cudaGetSymbolAddress) by the
//     first multi-chunk call made while a given CUDA context is current on a
//     device, and reused while that context stays current; a new context on the
//     device (after cudaDeviceReset, or a driver context made current by the
//     caller) gets its own lookup on its first call. Make that first call before
//     any stream capture begins.
#include <mutex>

#include <cuda.h>

#include "internal.cuh"

namespace moe {
namespace {

constexpr int64_t kNoAllocScratchInts = 65536;
constexpr int kMaxDevices = 64;

// Host code must not use this name as a device address; see scratch_address().
static __device__ __align__(256) int32_t g_group_scratch[kNoAllocScratchInts];

using CtxGetCurrentFn = CUresult (*)(CUcontext*);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long*);

struct Entry {
  unsigned long long ctx_id = 0;   // context the address was looked up in (ids are never reused)
  int32_t* addr = nullptr;
};

std::mutex g_mu;
Entry g_entry[kMaxDevices];
CtxGetCurrentFn g_ctx_current = nullptr;
CtxGetIdFn g_ctx_id = nullptr;

// The driver's unique id of the context current on this thread (0 if none can be had).
cudaError_t current_ctx_id(unsigned long long* id) {
  *id = 0;
  if (g_ctx_current == nullptr || g_ctx_id == nullptr) {
    void* a = nullptr;
    void* b = nullptr;
    cudaDriverEntryPointQueryResult qa, qb;
    cudaError_t e = cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &a, 4000, cudaEnableDefault, &qa);
    if (e != cudaSuccess || qa != cudaDriverEntryPointSuccess) return e != cudaSuccess ? e : cudaErrorNotSupported;
    e = cudaGetDriverEntryPointByVersion("cuCtxGetId", &b, 12000, cudaEnableDefault, &qb);
    if (e != cudaSuccess || qb != cudaDriverEntryPointSuccess) return e != cudaSuccess ? e : cudaErrorNotSupported;
    g_ctx_current = reinterpret_cast<CtxGetCurrentFn>(a);
    g_ctx_id = reinterpret_cast<CtxGetIdFn>(b);
  }
  CUcontext ctx = nullptr;
  if (g_ctx_current(&ctx) != CUDA_SUCCESS || ctx == nullptr) return cudaErrorDeviceUninitialized;
  if (g_ctx_id(ctx, id) != CUDA_SUCCESS) return cudaErrorDeviceUninitialized;
  return cudaSuccess;
}

// Device address of g_group_scratch in the context current on this thread: looked up once per
// device and context, with that device current.
cudaError_t scratch_address(int32_t** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_mu);
  Entry& en = g_entry[dev];
  unsigned long long id = 0;
  if (current_ctx_id(&id) == cudaSuccess && en.addr != nullptr && en.ctx_id == id) {
    *out = en.addr;
    return cudaSuccess;
  }
  // the lookup also binds the device's primary context to this thread if none was current
  void* p = nullptr;
  if ((e = cudaGetSymbolAddress(&p, g_group_scratch)) != cudaSuccess) return e;
  if ((e = current_ctx_id(&id)) != cudaSuccess) return e;
  en.addr = static_cast<int32_t*>(p);
  en.ctx_id = id;
  *out = en.addr;
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
  if (s.nchunks == 1) {
    // one chunk of tokens: histogram, scan, scatter and the row copy in one launch, each block
    // grouping in its own shared memory
    if (launch_group_gather_single_chunk(s, topk_idx, counts, offsets, dest_row, src_token, nullptr, status, x,
                                         x_perm, stream) != cudaSuccess)
      return MOE_ERR_CUDA;
    return MOE_OK;
  }
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
