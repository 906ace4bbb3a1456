// Routing telemetry of one batch, computed on the device from the per-expert counts.
//
// shubhamtatvamasi.com/llm-inference/moe "Mixture of Experts", section "Load
// imbalance": experts receive uneven loads; a capacity limit drops the
// overflow, and dropless serving waits for the busiest expert, so the useful
// share of expert compute is the mean load over the maximum load. Section
// "Memory vs compute, quantified": the experts a batch touches are the ones
// whose weights are read.
#include "internal.cuh"

namespace moe {
namespace {

constexpr int kStatThreads = 256;   // one thread per expert (E <= 256)

__global__ void __launch_bounds__(kStatThreads)
routing_stats_kernel(const int32_t* __restrict__ counts, int E, int T, int cap, moe_routing_stats_t* out) {
  __shared__ int s_sum[kStatThreads / 32], s_kept[kStatThreads / 32], s_touched[kStatThreads / 32],
      s_max[kStatThreads / 32];
  const int e = threadIdx.x, lane = e & 31, warp = e >> 5;
  int c = 0;
  if (e < E) c = counts[e] > 0 ? counts[e] : 0;
  const int kept = c < cap ? c : cap;
  int sum = c, ksum = kept, touched = kept > 0 ? 1 : 0, mx = kept;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    sum += __shfl_xor_sync(0xffffffffu, sum, o);
    ksum += __shfl_xor_sync(0xffffffffu, ksum, o);
    touched += __shfl_xor_sync(0xffffffffu, touched, o);
    mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  }
  if (lane == 0) {
    s_sum[warp] = sum;
    s_kept[warp] = ksum;
    s_touched[warp] = touched;
    s_max[warp] = mx;
  }
  __syncthreads();
  if (e == 0) {
    int P = 0, K = 0, U = 0, M = 0;
    for (int w = 0; w < kStatThreads / 32; ++w) {
      P += s_sum[w];
      K += s_kept[w];
      U += s_touched[w];
      M = max(M, s_max[w]);
    }
    moe_routing_stats_t r;
    r.tokens = T;
    r.pairs = P;
    r.kept = K;
    r.dropped = P - K;
    r.experts_touched = U;
    r.max_load = M;
    r.capacity = cap;
    r.mean_load = __fdiv_rn((float)K, (float)E);
    r.efficiency = M > 0 ? __fdiv_rn(r.mean_load, (float)M) : 1.0f;
    *out = r;
  }
}

}  // namespace
}  // namespace moe

extern "C" moe_status_t moe_routing_stats(const moe_config_t* cfg, const int32_t* counts, moe_routing_stats_t* stats,
                                          cudaStream_t stream) {
  using namespace moe;
  moe_status_t rc = moe_check_config(cfg);
  if (rc != MOE_OK) return rc;
  if (!counts || !stats) return MOE_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(counts) & 3u) || (reinterpret_cast<uintptr_t>(stats) & 3u))
    return MOE_ERR_INVALID_ARG;
  const Shape s = make_shape(*cfg);
  routing_stats_kernel<<<1, kStatThreads, 0, stream>>>(counts, s.E, s.T, s.cap, stats);
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}
