// The group schedule of the grouped expert MLPs, built by one warp from the
// kept-pair offsets of the grouping stage: for each group (the routed experts,
// then the shared expert) its first input row, first output row, row count
// and the prefix sum of its 128-row M tiles (layout: SchedView in internal.cuh).
#pragma once

#include "internal.cuh"

namespace moe {

constexpr int kSchedTileRows = 128;

// One full warp. `offsets` (E+1 entries, shared or global memory) must already be
// checked; `bad` makes every routed group empty. Groups are taken 32 at a time
// with a warp prefix sum over their tile counts.
__device__ __forceinline__ void build_schedule_warp(const int32_t* offsets, bool bad, int E, int S, int T,
                                                    int64_t R, int32_t* __restrict__ sched) {
  const int G = E + S;
  int32_t* tile_start = sched;
  int32_t* a_row = sched + (G + 1);
  int32_t* out_row = a_row + G;
  int32_t* rows = out_row + G;
  const int lane = threadIdx.x & 31;
  int carry = 0;
  for (int base = 0; base < G; base += 32) {
    const int g = base + lane;
    int ar = 0, orow = 0, nr = 0;
    if (g < E) {
      ar = bad ? 0 : offsets[g];
      orow = ar;
      nr = bad ? 0 : offsets[g + 1] - offsets[g];
    } else if (g < G) {
      ar = 0;
      orow = (int)(R + (int64_t)(g - E) * T);
      nr = T;
    }
    const int tiles = (nr + kSchedTileRows - 1) / kSchedTileRows;
    int incl = tiles;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += v;
    }
    if (g < G) {
      tile_start[g] = carry + incl - tiles;
      a_row[g] = ar;
      out_row[g] = orow;
      rows[g] = nr;
    }
    carry += __shfl_sync(0xffffffffu, incl, 31);
  }
  if (lane == 0) tile_start[G] = carry;
}

}  // namespace moe
