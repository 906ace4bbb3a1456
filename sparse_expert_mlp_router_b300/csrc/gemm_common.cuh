// Device helpers shared by the grouped-GEMM kernels (bf16 and FP8 weights).
#pragma once

#include "internal.cuh"
#include "tc_ptx.cuh"

namespace moe {
namespace gemm {

constexpr uint64_t kWaitLimitNs = 4000000000ull;     // 4 s: far beyond any legitimate wait
constexpr uint64_t kDrainLimitNs = 100000000ull;     // 100 ms for draining after an abort

// Tiles ordered (group, n-tile, m-tile) from a prefix of m-tiles per group.
__device__ __forceinline__ void decode_tile(int L, const int32_t* tile_start, int G, int nt, int& g, int& m,
                                            int& n) {
  int lo = 0, hi = G;
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (tile_start[mid] * nt <= L) lo = mid; else hi = mid;
  }
  g = lo;
  const int mt = tile_start[g + 1] - tile_start[g];
  const int local = L - tile_start[g] * nt;
  n = local / mt;
  m = local - n * mt;
}

__device__ __forceinline__ float silu_f(float z) { return __fdividef(z, 1.0f + __expf(-z)); }

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&v);
}

// After an abort: the most recent fill of each of the `issued` slots before (stage, phase)
// lands before the shared memory is left. A fill whose phase already completed passes at once.
__device__ __forceinline__ void drain_fills(uint64_t* full, int n_stages, int stage, uint32_t phase, int issued) {
  for (int j = 0; j < issued; ++j) {
    if (stage == 0) {
      stage = n_stages - 1;
      phase ^= 1u;
    } else {
      --stage;
    }
    ptx::mbar_wait_bounded(ptx::smem_u32(&full[stage]), phase, nullptr, kDrainLimitNs);
  }
}

}  // namespace gemm
}  // namespace moe
