// Grouping of (token, slot) pairs by destination expert: histogram, prefix sum,
// capacity, scatter of row indices, and the 16-byte row gather of x.
//
// Follows klaylearn.com/glossary/mixture-of-experts "Mixture of Experts" (its
// definition: tokens are sorted by the expert they go to before the grouped GEMMs,
// and put back in order after) and shubhamtatvamasi.com/llm-inference/moe "Mixture
// of Experts", section "Load imbalance" (each expert accepts at most the capacity
// factor times its even share of the tokens, the overflow skips that expert; or
// dropless) and its Q&A on capacity factor (the even share is T·k/E).
//
// Determinism: within one expert, rows follow ascending token index, and the
// tokens past the capacity are the highest-index ones. The kernels reach this
// without sorting: tokens are cut into chunks of 128; inside a chunk each
// expert owns a 128-bit membership mask built with atomicOr (order-free), so a
// pair's rank inside the chunk is a popcount of the mask bits below its token;
// a per-expert prefix over chunks then gives the global rank.
#include "group_single.cuh"
#include "internal.cuh"
#include "sched.cuh"

namespace moe {
namespace {

constexpr int kWords = kChunk / 32;     // mask words per expert per chunk

// Build the chunk's masks. Returns nothing; flags ids outside [0, E) and repeated
// (token, expert) pairs. `dup` (optional) receives, per pair, whether its bit was
// already set by another slot of the same token.
__device__ __forceinline__ void build_masks(uint32_t* mask, const int32_t* __restrict__ idx, int t0, int nt,
                                            int k, int E, int32_t* status, bool* dup_flags) {
  for (int w = threadIdx.x; w < E * kWords; w += blockDim.x) mask[w] = 0u;
  __syncthreads();
  for (int p = threadIdx.x; p < nt * k; p += blockDim.x) {
    const int tl = p / k;
    const int e = idx[(size_t)t0 * k + p];
    bool dup = false;
    if (e < 0 || e >= E) {
      set_status(status, MOE_ERR_DEVICE_INDEX);
      dup = true;
    } else {
      const uint32_t bit = 1u << (tl & 31);
      const uint32_t old = atomicOr(&mask[e * kWords + (tl >> 5)], bit);
      if (old & bit) {
        set_status(status, MOE_ERR_DEVICE_INDEX);
        dup = true;
      }
    }
    if (dup_flags) dup_flags[p] = dup;
  }
  __syncthreads();
}

__global__ void group_hist_kernel(const int32_t* __restrict__ idx, int T, int k, int E,
                                  int32_t* __restrict__ chunk_counts, int32_t* status) {
  __shared__ uint32_t mask[kMaxExperts * kWords];
  const int c = blockIdx.x;
  const int t0 = c * kChunk;
  const int nt = min(kChunk, T - t0);
  build_masks(mask, idx, t0, nt, k, E, status, nullptr);
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    int n = 0;
#pragma unroll
    for (int w = 0; w < kWords; ++w) n += __popc(mask[e * kWords + w]);
    chunk_counts[(size_t)c * E + e] = n;
  }
}

// One CTA of 256 threads (one per expert): per expert, exclusive prefix over chunks
// (in place: counts -> rank base), total counts, capacity clamp, exclusive scan of
// the kept counts over experts; optionally the group schedule of the grouped GEMMs.
// Chunk counts are staged through shared memory 32 chunks at a time, so the loads
// of a tile are all in flight together.
constexpr int kScanThreads = 256;
constexpr int kScanTile = 32;

__global__ void __launch_bounds__(kScanThreads)
group_scan_kernel(int32_t* __restrict__ chunk_counts, int nchunks, int E, int cap, int32_t* __restrict__ counts,
                  int32_t* __restrict__ offsets, int32_t* __restrict__ sched, int S, int T, int64_t R) {
  __shared__ int32_t tile[kScanTile * kMaxExperts];
  __shared__ int32_t warp_tot[kScanThreads / 32];
  __shared__ int32_t s_off[kMaxExperts + 1];
  const int e = threadIdx.x;
  int run = 0;
  for (int c0 = 0; c0 < nchunks; c0 += kScanTile) {
    const int nc = min(kScanTile, nchunks - c0);
    int32_t* g = chunk_counts + (size_t)c0 * E;
    for (int i = threadIdx.x; i < nc * E; i += kScanThreads) tile[i] = g[i];
    __syncthreads();
    if (e < E)
      for (int c = 0; c < nc; ++c) {
        const int v = tile[c * E + e];
        tile[c * E + e] = run;
        run += v;
      }
    __syncthreads();
    for (int i = threadIdx.x; i < nc * E; i += kScanThreads) g[i] = tile[i];
    __syncthreads();
  }
  if (e < E) counts[e] = run;
  const int kv = (e < E) ? min(run, cap) : 0;
  // block-wide exclusive scan of kv over the experts
  const int lane = e & 31, warp = e >> 5;
  int incl = kv;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += v;
  }
  if (lane == 31) warp_tot[warp] = incl;
  __syncthreads();
  int base = 0;
  for (int w = 0; w < warp; ++w) base += warp_tot[w];
  if (e < E) {
    offsets[e] = base + incl - kv;
    s_off[e] = base + incl - kv;
  }
  if (e == kScanThreads - 1) {
    offsets[E] = base + incl;
    s_off[E] = base + incl;
  }
  if (sched != nullptr) {
    __syncthreads();
    if (warp == 0) build_schedule_warp(s_off, false, E, S, T, R, sched);
  }
}

__global__ void group_scatter_kernel(const int32_t* __restrict__ idx, int T, int k, int E,
                                     const int32_t* __restrict__ chunk_base, const int32_t* __restrict__ offsets,
                                     int32_t* __restrict__ dest_row, int32_t* __restrict__ src_token) {
  __shared__ uint32_t mask[kMaxExperts * kWords];
  __shared__ bool dup[kChunk * kMaxTopK];
  const int c = blockIdx.x;
  const int t0 = c * kChunk;
  const int nt = min(kChunk, T - t0);
  build_masks(mask, idx, t0, nt, k, E, nullptr, dup);
  for (int p = threadIdx.x; p < nt * k; p += blockDim.x) {
    const int tl = p / k;
    const int t = t0 + tl;
    const int e = idx[(size_t)t0 * k + p];
    int row = -1;
    if (!dup[p]) {
      const uint32_t* m = mask + e * kWords;
      int r = 0;
      for (int w = 0; w < (tl >> 5); ++w) r += __popc(m[w]);
      r += __popc(m[tl >> 5] & ((1u << (tl & 31)) - 1u));
      const int rank = chunk_base[(size_t)c * E + e] + r;
      const int lo = offsets[e], hi = offsets[e + 1];
      if (rank < hi - lo) {
        row = lo + rank;
        src_token[row] = t;
      }
    }
    dest_row[(size_t)t * k + (p % k)] = row;
  }
}

// The three steps above in one CTA when the batch is a single chunk (T <= 128, decode): the
// chunk's masks once, per-expert counts, capacity clamp and scan, the group schedule, then
// the scatter, with the same ranks as the three-kernel path (chunk base 0).
__global__ void __launch_bounds__(kSingleThreads)
group_single_chunk_kernel(const int32_t* __restrict__ idx, int T, int k, int E, int cap,
                          int32_t* __restrict__ counts, int32_t* __restrict__ offsets,
                          int32_t* __restrict__ dest_row, int32_t* __restrict__ src_token,
                          int32_t* __restrict__ sched, int S, int64_t R, int32_t* status) {
  __shared__ SingleChunkSmem sm;
  single_chunk_group(idx, T, k, E, cap, true, counts, offsets, dest_row, src_token, sched, S, R, status, sm);
}

// One warp copies grouped row r = token t's row of x: 16-byte vectors, four loads in flight per
// lane before their stores.
__device__ __forceinline__ void copy_row(const uint4* __restrict__ x, int64_t t, uint4* __restrict__ dst,
                                         int vec_per_row, int lane) {
  const uint4* src = x + (size_t)t * vec_per_row;
  int v = lane;
  for (; v + 96 < vec_per_row; v += 128) {
    const uint4 a = __ldg(src + v), b = __ldg(src + v + 32), c = __ldg(src + v + 64), e = __ldg(src + v + 96);
    dst[v] = a;
    dst[v + 32] = b;
    dst[v + 64] = c;
    dst[v + 96] = e;
  }
  for (; v < vec_per_row; v += 32) dst[v] = __ldg(src + v);
}

// The single-chunk grouping and the grouped copy of x in one launch: every block rebuilds the
// grouping in shared memory (block 0 writes it out), then copies its rows, one warp per row.
__global__ void __launch_bounds__(kSingleThreads)
group_gather_single_chunk_kernel(const int32_t* __restrict__ idx, int T, int k, int E, int cap,
                                 int32_t* __restrict__ counts, int32_t* __restrict__ offsets,
                                 int32_t* __restrict__ dest_row, int32_t* __restrict__ src_token,
                                 int32_t* __restrict__ sched, int S, int64_t R, int32_t* status,
                                 const uint4* __restrict__ x, int vec_per_row, uint4* __restrict__ x_perm) {
  __shared__ SingleChunkSmem sm;
  single_chunk_group(idx, T, k, E, cap, blockIdx.x == 0, counts, offsets, dest_row, src_token, sched, S, R, status,
                     sm);
  const int64_t n_rows = min((int64_t)sm.off[E], R);
  const int lane = threadIdx.x & 31;
  const int64_t warps = (int64_t)gridDim.x * (blockDim.x >> 5);
  for (int64_t r = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); r < n_rows; r += warps)
    copy_row(x, sm.src[r], x_perm + (size_t)r * vec_per_row, vec_per_row, lane);
}

// x_perm[r] = x[src_token[r]] for r < offsets[E]; one warp per row, 16-byte vectors.
__global__ void gather_rows_kernel(const uint4* __restrict__ x, const int32_t* __restrict__ src_token,
                                   const int32_t* __restrict__ offsets, int E, int vec_per_row, int64_t R,
                                   uint4* __restrict__ x_perm) {
  const int64_t n_rows = min((int64_t)offsets[E], R);
  const int lane = threadIdx.x & 31;
  const int64_t warps = (int64_t)gridDim.x * (blockDim.x >> 5);
  for (int64_t r = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); r < n_rows; r += warps)
    copy_row(x, src_token[r], x_perm + (size_t)r * vec_per_row, vec_per_row, lane);
}

}  // namespace

cudaError_t launch_group_hist(const Shape& s, const int32_t* idx, int32_t* chunk_counts,
                              int32_t* status, cudaStream_t st) {
  group_hist_kernel<<<s.nchunks, 256, 0, st>>>(idx, s.T, s.k, s.E, chunk_counts, status);
  return cudaGetLastError();
}

cudaError_t launch_group_scan(const Shape& s, int32_t* chunk_counts, int32_t* counts, int32_t* offsets,
                              void* sched, cudaStream_t st) {
  group_scan_kernel<<<1, kScanThreads, 0, st>>>(chunk_counts, s.nchunks, s.E, s.cap, counts, offsets,
                                                static_cast<int32_t*>(sched), s.S, s.T, s.R);
  return cudaGetLastError();
}

cudaError_t launch_group_scatter(const Shape& s, const int32_t* idx, const int32_t* chunk_base,
                                 const int32_t* offsets, int32_t* dest_row, int32_t* src_token,
                                 cudaStream_t st) {
  group_scatter_kernel<<<s.nchunks, 256, 0, st>>>(idx, s.T, s.k, s.E, chunk_base, offsets, dest_row, src_token);
  return cudaGetLastError();
}

cudaError_t launch_group_single_chunk(const Shape& s, const int32_t* idx, int32_t* counts, int32_t* offsets,
                                      int32_t* dest_row, int32_t* src_token, void* sched, int32_t* status,
                                      cudaStream_t st) {
  if (s.nchunks != 1) return cudaErrorInvalidValue;
  group_single_chunk_kernel<<<1, kSingleThreads, 0, st>>>(idx, s.T, s.k, s.E, s.cap, counts, offsets, dest_row,
                                                        src_token, static_cast<int32_t*>(sched), s.S, s.R, status);
  return cudaGetLastError();
}

cudaError_t launch_gather_rows(const Shape& s, const void* x, const int32_t* src_token,
                               const int32_t* offsets, void* x_perm, cudaStream_t st) {
  const int vec_per_row = (int)((size_t)s.d * s.esize / 16);
  const int threads = 256;
  int64_t blocks = (s.R + 7) / 8;
  const int64_t cap = (int64_t)num_sms() * 16;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  gather_rows_kernel<<<(unsigned)blocks, threads, 0, st>>>(static_cast<const uint4*>(x), src_token, offsets, s.E,
                                                            vec_per_row, s.R, static_cast<uint4*>(x_perm));
  return cudaGetLastError();
}

cudaError_t launch_group_gather_single_chunk(const Shape& s, const int32_t* idx, int32_t* counts, int32_t* offsets,
                                             int32_t* dest_row, int32_t* src_token, void* sched, int32_t* status,
                                             const void* x, void* x_perm, cudaStream_t st) {
  if (s.nchunks != 1) return cudaErrorInvalidValue;
  const int vec_per_row = (int)((size_t)s.d * s.esize / 16);
  int64_t blocks = (s.R + 7) / 8;       // one warp per row, as the separate copy
  const int64_t cap = (int64_t)num_sms() * 16;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  group_gather_single_chunk_kernel<<<(unsigned)blocks, kSingleThreads, 0, st>>>(
      idx, s.T, s.k, s.E, s.cap, counts, offsets, dest_row, src_token, static_cast<int32_t*>(sched), s.S, s.R, status,
      static_cast<const uint4*>(x), vec_per_row, static_cast<uint4*>(x_perm));
  return cudaGetLastError();
}

}  // namespace moe
