// Group schedule of the grouped expert MLPs, and the float32 CUDA-core path of
// those MLPs.
//
// The schedule turns the kept-pair offsets of the grouping stage into the
// per-group row ranges and 128-row tile counts the grouped GEMMs walk (one
// group per routed expert, then one per shared expert, which all tokens pass
// through: shubhamtatvamasi.com/llm-inference/moe "Mixture of Experts", section
// "The router"). It also checks the offsets: a grouping
// that is not monotone or overruns the row capacity is recorded as
// MOE_ERR_DEVICE_INDEX and replaced by an empty one, so no kernel reads out of
// bounds.
//
// The float32 path computes the same SwiGLU expert MLP as the tensor-core
// path, y = W_down (silu(W_gate a) * (W_up a)), one output element per thread
// with float32 FMAs; tensor cores have no float32 mode precise enough for
// float32 layers. It serves layers stored in float32.
#include "internal.cuh"
#include "sched.cuh"

namespace moe {
namespace {

// One warp: checks offsets supplied by the caller (offsets[0] == 0, non-decreasing,
// offsets[E] <= R), then builds the schedule.
__global__ void group_schedule_kernel(const int32_t* __restrict__ offsets, int E, int S, int T, int64_t R,
                                      int32_t* __restrict__ sched, int32_t* status) {
  const int lane = threadIdx.x;
  bool bad = false;
  for (int g = lane; g < E; g += 32) {
    const int lo = offsets[g], hi = offsets[g + 1];
    if (lo > hi || (g == 0 && lo != 0) || hi > R) bad = true;
  }
  bad = __any_sync(0xffffffffu, bad);
  if (bad && lane == 0) set_status(status, MOE_ERR_DEVICE_INDEX);
  build_schedule_warp(offsets, bad, E, S, T, R, sched);
}

__device__ __forceinline__ float silu_precise(float z) { return z / (1.0f + expf(-z)); }

// Which group a grouped row belongs to; -1 when the row holds no pair.
__device__ __forceinline__ int row_group(const int32_t* sched, int G, int64_t r, int& local) {
  const int32_t* out_row = sched + (G + 1) + G;
  const int32_t* rows = out_row + G;
  for (int g = 0; g < G; ++g) {
    const int64_t lo = out_row[g];
    if (r >= lo && r < lo + rows[g]) {
      local = (int)(r - lo);
      return g;
    }
  }
  return -1;
}

template <typename TE>
__global__ void ffn_gateup_fma_kernel(const TE* __restrict__ x_perm, const TE* __restrict__ x,
                                      const TE* __restrict__ wg, const TE* __restrict__ wu,
                                      const int32_t* __restrict__ sched, int G, int E, int d, int F,
                                      int64_t n_rows, TE* __restrict__ h) {
  const int64_t total = n_rows * F;
  for (int64_t o = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; o < total; o += (int64_t)gridDim.x * blockDim.x) {
    const int64_t r = o / F;
    const int f = (int)(o % F);
    int local = 0;
    const int g = row_group(sched, G, r, local);
    if (g < 0) continue;
    const int32_t* a_row = sched + (G + 1);
    const TE* a = (g >= E) ? x + (size_t)(a_row[g] + local) * d : x_perm + (size_t)(a_row[g] + local) * d;
    const TE* wgr = wg + ((size_t)g * F + f) * d;
    const TE* wur = wu + ((size_t)g * F + f) * d;
    float sg = 0.f, su = 0.f;
    for (int i = 0; i < d; ++i) {
      const float av = to_f32(a[i]);
      sg = fmaf(av, to_f32(wgr[i]), sg);
      su = fmaf(av, to_f32(wur[i]), su);
    }
    h[(size_t)r * F + f] = from_f32<TE>(silu_precise(sg) * su);
  }
}

template <typename TE>
__global__ void ffn_down_fma_kernel(const TE* __restrict__ h, const TE* __restrict__ wd,
                                    const int32_t* __restrict__ sched, int G, int d, int F, int64_t n_rows,
                                    TE* __restrict__ y) {
  const int64_t total = n_rows * d;
  for (int64_t o = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; o < total; o += (int64_t)gridDim.x * blockDim.x) {
    const int64_t r = o / d;
    const int c = (int)(o % d);
    int local = 0;
    const int g = row_group(sched, G, r, local);
    if (g < 0) continue;
    const TE* hr = h + (size_t)r * F;
    const TE* wr = wd + ((size_t)g * d + c) * F;
    float acc = 0.f;
    for (int f = 0; f < F; ++f) acc = fmaf(to_f32(hr[f]), to_f32(wr[f]), acc);
    y[(size_t)r * d + c] = from_f32<TE>(acc);
  }
}

}  // namespace

cudaError_t launch_group_schedule(const Shape& s, const int32_t* offsets, void* sched, int32_t* status,
                                  cudaStream_t st) {
  group_schedule_kernel<<<1, 32, 0, st>>>(offsets, s.E, s.S, s.T, s.R, static_cast<int32_t*>(sched), status);
  return cudaGetLastError();
}

// The two float32 MLP kernels; mid_event (nullable) is recorded between them.
cudaError_t launch_ffn_fma(const Shape& s, const void* x_perm, const void* x, const void* w_gate, const void* w_up,
                           const void* w_down, const void* sched, void* h, void* y, cudaStream_t st,
                           cudaEvent_t mid_event) {
  const int64_t n_rows = s.R + (int64_t)s.S * s.T;
  const int threads = 256;
  const int64_t cap = (int64_t)num_sms() * 32;
  int64_t b1 = (n_rows * s.F + threads - 1) / threads;
  int64_t b2 = (n_rows * s.d + threads - 1) / threads;
  b1 = b1 < cap ? (b1 < 1 ? 1 : b1) : cap;
  b2 = b2 < cap ? (b2 < 1 ? 1 : b2) : cap;
  const int32_t* sc = static_cast<const int32_t*>(sched);
  // float32 layers only; bf16 layers run on the tensor cores
  ffn_gateup_fma_kernel<float><<<(unsigned)b1, threads, 0, st>>>(
      static_cast<const float*>(x_perm), static_cast<const float*>(x), static_cast<const float*>(w_gate),
      static_cast<const float*>(w_up), sc, s.G, s.E, s.d, s.F, n_rows, static_cast<float*>(h));
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  if (mid_event && (e = record_event(mid_event, st)) != cudaSuccess) return e;
  ffn_down_fma_kernel<float><<<(unsigned)b2, threads, 0, st>>>(
      static_cast<const float*>(h), static_cast<const float*>(w_down), sc, s.G, s.d, s.F, n_rows,
      static_cast<float*>(y));
  return cudaGetLastError();
}

}  // namespace moe
