// The grouping of a single chunk of tokens (T <= 128, decode) as a device function for one
// block of 256 threads (one per expert): membership masks, per-expert counts, capacity clamp and
// scan, the group schedule, and the scatter of row indices, with the ranks of the multi-chunk
// kernels (klaylearn.com/glossary/mixture-of-experts "Mixture of Experts", definition;
// shubhamtatvamasi.com/llm-inference/moe, section "Load imbalance": within one expert rows
// follow ascending token index, and the tokens past the capacity are the highest-index ones).
//
// The kernels that also copy (or quantise) the grouped rows run it in every block of their
// grid: each block rebuilds the grouping in its own shared memory (T k <= 1024 pairs: a few
// microseconds), block 0 alone writes it out, and each block then takes its share of the rows,
// so the grouping and the row copy are one launch with no block waiting on another.
#pragma once

#include "internal.cuh"
#include "sched.cuh"

namespace moe {

constexpr int kSingleThreads = 256;        // one thread per expert (E <= kMaxExperts)
constexpr int kSingleWords = kChunk / 32;  // mask words per expert

struct SingleChunkSmem {
  uint32_t mask[kMaxExperts * kSingleWords];
  bool dup[kChunk * kMaxTopK];
  int32_t warp_tot[kSingleThreads / 32];
  int32_t off[kMaxExperts + 1];            // kept-pair offsets, off[E] = kept pairs
  int32_t src[kChunk * kMaxTopK];          // token of each kept row (rows < off[E])
};

// Every thread of the block (blockDim.x == kSingleThreads) calls it. write: this block stores
// counts, offsets, dest_row, src_token and the schedule (sched may be NULL) and reports bad or
// repeated ids in `status`; every block leaves offsets and src_token in `sm`.
__device__ __forceinline__ void single_chunk_group(const int32_t* __restrict__ idx, int T, int k, int E, int cap,
                                                   bool write, int32_t* __restrict__ counts,
                                                   int32_t* __restrict__ offsets, int32_t* __restrict__ dest_row,
                                                   int32_t* __restrict__ src_token, int32_t* __restrict__ sched,
                                                   int S, int64_t R, int32_t* status, SingleChunkSmem& sm) {
  for (int w = threadIdx.x; w < E * kSingleWords; w += blockDim.x) sm.mask[w] = 0u;
  __syncthreads();
  for (int p = threadIdx.x; p < T * k; p += blockDim.x) {
    const int tl = p / k;
    const int e = idx[p];
    bool dup = false;
    if (e < 0 || e >= E) {
      if (write) set_status(status, MOE_ERR_DEVICE_INDEX);
      dup = true;
    } else {
      const uint32_t bit = 1u << (tl & 31);
      const uint32_t old = atomicOr(&sm.mask[e * kSingleWords + (tl >> 5)], bit);
      if (old & bit) {
        if (write) set_status(status, MOE_ERR_DEVICE_INDEX);
        dup = true;
      }
    }
    sm.dup[p] = dup;
  }
  __syncthreads();
  const int e = threadIdx.x;
  int n = 0;
  if (e < E) {
#pragma unroll
    for (int w = 0; w < kSingleWords; ++w) n += __popc(sm.mask[e * kSingleWords + w]);
    if (write) counts[e] = n;
  }
  const int kv = (e < E) ? min(n, cap) : 0;
  const int lane = e & 31, warp = e >> 5;
  int incl = kv;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += v;
  }
  if (lane == 31) sm.warp_tot[warp] = incl;
  __syncthreads();
  int base = 0;
  for (int w = 0; w < warp; ++w) base += sm.warp_tot[w];
  if (e < E) {
    sm.off[e] = base + incl - kv;
    if (write) offsets[e] = base + incl - kv;
  }
  if (e == kSingleThreads - 1) {
    sm.off[E] = base + incl;
    if (write) offsets[E] = base + incl;
  }
  __syncthreads();
  if (write && sched != nullptr && warp == 0) build_schedule_warp(sm.off, false, E, S, T, R, sched);
  for (int p = threadIdx.x; p < T * k; p += blockDim.x) {
    const int t = p / k;
    const int ex = idx[p];
    int row = -1;
    if (!sm.dup[p]) {
      const uint32_t* m = sm.mask + ex * kSingleWords;
      int r = 0;
      for (int w = 0; w < (t >> 5); ++w) r += __popc(m[w]);
      r += __popc(m[t >> 5] & ((1u << (t & 31)) - 1u));
      const int lo = sm.off[ex], hi = sm.off[ex + 1];
      if (r < hi - lo) {
        row = lo + r;
        sm.src[row] = t;
        if (write) src_token[row] = t;
      }
    }
    if (write) dest_row[p] = row;
  }
  __syncthreads();
}

}  // namespace moe
