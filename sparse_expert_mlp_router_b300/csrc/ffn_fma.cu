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
// path, y = W_down (silu(W_gate a) * (W_up a)), one output element per four
// lanes with float32 FMAs; tensor cores have no float32 mode precise enough
// for float32 layers. It serves layers stored in float32.
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

// Four lanes share one output element: lane part p of the quad takes the float4 vectors
// v = p, p + 4, p + 8, ... of the reduction, so the quad's loads of a weight row are contiguous
// (64 bytes per step) and a thread's chain of dependent FMAs is a quarter of the reduction; the
// quad's partial sums are then added with two shuffles.
constexpr int kQuad = 4;

__device__ __forceinline__ float quad_sum(float v) {
  v += __shfl_xor_sync(0xffffffffu, v, 1);
  v += __shfl_xor_sync(0xffffffffu, v, 2);
  return v;
}

// A routed group's rows are read from x_perm, or (src_token non-NULL: the whole-layer call,
// which then skips the grouped copy) from x through src_token: the same values.
__global__ void ffn_gateup_fma_kernel(const float* __restrict__ x_perm, const float* __restrict__ x,
                                      const int32_t* __restrict__ src_token, const float* __restrict__ wg,
                                      const float* __restrict__ wu, const int32_t* __restrict__ sched, int G, int E,
                                      int d, int F, int64_t n_rows, float* __restrict__ h) {
  const int p = threadIdx.x & (kQuad - 1);
  const int64_t total = n_rows * F;
  const int64_t stride = (int64_t)gridDim.x * (blockDim.x / kQuad);
  const int nv = d / 4;
  // every lane runs the same number of iterations, so the quad's shuffles see all four lanes
  for (int64_t o0 = (int64_t)blockIdx.x * (blockDim.x / kQuad); o0 < total; o0 += stride) {
    const int64_t o = o0 + (threadIdx.x / kQuad);
    float sg = 0.f, su = 0.f;
    int64_t r = 0;
    int f = 0;
    int g = -1;
    if (o < total) {
      r = o / F;
      f = (int)(o % F);
      int local = 0;
      g = row_group(sched, G, r, local);
      if (g >= 0) {
        const int32_t* a_row = sched + (G + 1);
        const int arow = a_row[g] + local;
        const float* base = (g >= E) ? x + (size_t)arow * d
                            : src_token ? x + (size_t)src_token[arow] * d
                                        : x_perm + (size_t)arow * d;
        const float4* a = reinterpret_cast<const float4*>(base);
        const float4* wgr = reinterpret_cast<const float4*>(wg + ((size_t)g * F + f) * d);
        const float4* wur = reinterpret_cast<const float4*>(wu + ((size_t)g * F + f) * d);
        for (int v = p; v < nv; v += kQuad) {
          const float4 av = __ldg(a + v), gv = __ldg(wgr + v), uv = __ldg(wur + v);
          sg = fmaf(av.x, gv.x, sg); sg = fmaf(av.y, gv.y, sg); sg = fmaf(av.z, gv.z, sg); sg = fmaf(av.w, gv.w, sg);
          su = fmaf(av.x, uv.x, su); su = fmaf(av.y, uv.y, su); su = fmaf(av.z, uv.z, su); su = fmaf(av.w, uv.w, su);
        }
      }
    }
    sg = quad_sum(sg);
    su = quad_sum(su);
    if (o < total && g >= 0 && p == 0) h[(size_t)r * F + f] = silu_precise(sg) * su;
  }
}

__global__ void ffn_down_fma_kernel(const float* __restrict__ h, const float* __restrict__ wd,
                                    const int32_t* __restrict__ sched, int G, int d, int F, int64_t n_rows,
                                    float* __restrict__ y) {
  const int p = threadIdx.x & (kQuad - 1);
  const int64_t total = n_rows * d;
  const int64_t stride = (int64_t)gridDim.x * (blockDim.x / kQuad);
  const int nv = F / 4;
  for (int64_t o0 = (int64_t)blockIdx.x * (blockDim.x / kQuad); o0 < total; o0 += stride) {
    const int64_t o = o0 + (threadIdx.x / kQuad);
    float acc = 0.f;
    int64_t r = 0;
    int c = 0;
    int g = -1;
    if (o < total) {
      r = o / d;
      c = (int)(o % d);
      int local = 0;
      g = row_group(sched, G, r, local);
      if (g >= 0) {
        const float4* hr = reinterpret_cast<const float4*>(h + (size_t)r * F);
        const float4* wr = reinterpret_cast<const float4*>(wd + ((size_t)g * d + c) * F);
        for (int v = p; v < nv; v += kQuad) {
          const float4 hv = __ldg(hr + v), wv = __ldg(wr + v);
          acc = fmaf(hv.x, wv.x, acc); acc = fmaf(hv.y, wv.y, acc); acc = fmaf(hv.z, wv.z, acc);
          acc = fmaf(hv.w, wv.w, acc);
        }
      }
    }
    acc = quad_sum(acc);
    if (o < total && g >= 0 && p == 0) y[(size_t)r * d + c] = acc;
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
                           cudaEvent_t mid_event, const int32_t* src_token) {
  const int64_t n_rows = s.R + (int64_t)s.S * s.T;
  const int threads = 256;                      // 64 output elements per block (four lanes each)
  const int64_t per_block = threads / 4;
  const int64_t cap = (int64_t)num_sms() * 32;
  int64_t b1 = (n_rows * s.F + per_block - 1) / per_block;
  int64_t b2 = (n_rows * s.d + per_block - 1) / per_block;
  b1 = b1 < cap ? (b1 < 1 ? 1 : b1) : cap;
  b2 = b2 < cap ? (b2 < 1 ? 1 : b2) : cap;
  const int32_t* sc = static_cast<const int32_t*>(sched);
  // float32 layers only; bf16 layers run on the tensor cores
  ffn_gateup_fma_kernel<<<(unsigned)b1, threads, 0, st>>>(
      static_cast<const float*>(x_perm), static_cast<const float*>(x), src_token, static_cast<const float*>(w_gate),
      static_cast<const float*>(w_up), sc, s.G, s.E, s.d, s.F, n_rows, static_cast<float*>(h));
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  if (mid_event && (e = record_event(mid_event, st)) != cudaSuccess) return e;
  ffn_down_fma_kernel<<<(unsigned)b2, threads, 0, st>>>(
      static_cast<const float*>(h), static_cast<const float*>(w_down), sc, s.G, s.d, s.F, n_rows,
      static_cast<float*>(y));
  return cudaGetLastError();
}

}  // namespace moe
