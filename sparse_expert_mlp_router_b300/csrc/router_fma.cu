// Router on CUDA cores: logits = x W_r^T (+ b), softmax or sigmoid scores,
// top-k by warp-level selection, gate renormalisation.
//
// Follows shubhamtatvamasi.com/llm-inference/moe "Mixture of Experts", section
// "The router" (one small linear layer scoring every expert, softmax or the
// sigmoid variant, keep the top-k, renormalise the chosen gates to sum to one)
// and its Q&A "How does a top-k router work?".
//
// This kernel serves float32 layers and any layer the tensor-core router does
// not take. One CTA computes the logits of TOK tokens (32, or 8 when 32-token
// CTAs would not fill the GPU) against all E experts with float32 FMAs from
// shared-memory tiles, then each warp selects the top-k of its tokens: every lane
// holds E/32 scores, and k rounds of a warp-wide arg-max (ties to the lower
// expert id) pick the experts in rank order. The selection is a chain of
// dependent shuffles and divisions, so small batches spread it over more CTAs.
#include <cfloat>
#include <cmath>

#include "internal.cuh"
#include "select.cuh"

namespace moe {
namespace {

constexpr int kDc = 32;       // d_model chunk staged per iteration
constexpr int kPad = 4;       // row padding (floats) keeping 16-byte rows conflict-free
constexpr int kThreads = 256;

template <typename TIn>
__device__ __forceinline__ float4 load4(const TIn* p);
template <>
__device__ __forceinline__ float4 load4<float>(const float* p) {
  return *reinterpret_cast<const float4*>(p);
}
template <>
__device__ __forceinline__ float4 load4<__nv_bfloat16>(const __nv_bfloat16* p) {
  const uint2 u = *reinterpret_cast<const uint2*>(p);
  return make_float4(__uint_as_float(u.x << 16), __uint_as_float(u.x & 0xFFFF0000u),
                     __uint_as_float(u.y << 16), __uint_as_float(u.y & 0xFFFF0000u));
}

template <typename TIn, int TOK>
__global__ void __launch_bounds__(kThreads)
router_fma_kernel(const TIn* __restrict__ x, const TIn* __restrict__ w, const float* __restrict__ bias,
                  int T, int d, int E, int k, int score, int renorm,
                  int32_t* __restrict__ idx_out, float* __restrict__ gate_out, float* __restrict__ scores_out) {
  extern __shared__ __align__(16) float smem[];
  float* xs = smem;                              // [TOK][kDc + kPad]
  float* wsm = xs + TOK * (kDc + kPad);          // [E][kDc + kPad]
  float* logit = wsm + E * (kDc + kPad);         // [TOK][E + 1]

  const int tid = threadIdx.x;
  const int t0 = blockIdx.x * TOK;
  const int n_out = TOK * E;
  constexpr int kMaxPerThread = TOK * kMaxExperts / kThreads;    // 32 or 8

  float acc[kMaxPerThread];
#pragma unroll
  for (int i = 0; i < kMaxPerThread; ++i) acc[i] = 0.f;

  for (int c0 = 0; c0 < d; c0 += kDc) {
    // stage x[t0 .. t0+kTok, c0 .. c0+kDc) and W_r[:, c0 .. c0+kDc) as float32 (d % 4 == 0)
    for (int q = tid; q < TOK * (kDc / 4); q += kThreads) {
      const int r = q / (kDc / 4), c = (q % (kDc / 4)) * 4;
      float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
      if (t0 + r < T && c0 + c < d) v = load4<TIn>(x + (size_t)(t0 + r) * d + c0 + c);
      *reinterpret_cast<float4*>(xs + r * (kDc + kPad) + c) = v;
    }
    for (int q = tid; q < E * (kDc / 4); q += kThreads) {
      const int r = q / (kDc / 4), c = (q % (kDc / 4)) * 4;
      float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
      if (c0 + c < d) v = load4<TIn>(w + (size_t)r * d + c0 + c);
      *reinterpret_cast<float4*>(wsm + r * (kDc + kPad) + c) = v;
    }
    __syncthreads();
#pragma unroll
    for (int i = 0; i < kMaxPerThread; ++i) {
      const int o = tid + i * kThreads;
      if (o < n_out) {
        const float* xr = xs + (o / E) * (kDc + kPad);
        const float* wr = wsm + (o % E) * (kDc + kPad);
        float a = acc[i];
#pragma unroll
        for (int c = 0; c < kDc; c += 4) {
          const float4 xv = *reinterpret_cast<const float4*>(xr + c);
          const float4 wv = *reinterpret_cast<const float4*>(wr + c);
          a = fmaf(xv.x, wv.x, a);
          a = fmaf(xv.y, wv.y, a);
          a = fmaf(xv.z, wv.z, a);
          a = fmaf(xv.w, wv.w, a);
        }
        acc[i] = a;
      }
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < kMaxPerThread; ++i) {
    const int o = tid + i * kThreads;
    if (o < n_out) {
      const int e = o % E;
      logit[(o / E) * (E + 1) + e] = acc[i] + (bias ? bias[e] : 0.f);
    }
  }
  __syncthreads();

  const int warp = tid / 32, lane = tid % 32;
  for (int r = warp; r < TOK; r += kThreads / 32) {
    const int t = t0 + r;
    if (t >= T) break;
    select_topk_warp(logit + r * (E + 1), E, k, score, renorm, lane,
                     idx_out + (size_t)t * k, gate_out + (size_t)t * k,
                     scores_out ? scores_out + (size_t)t * E : nullptr);
  }
}

template <typename TIn, int TOK>
cudaError_t launch_tok(const Shape& s, const void* x, const void* w, const float* bias, int32_t* idx, float* gate,
                       float* scores, cudaStream_t st) {
  const size_t smem = sizeof(float) * ((size_t)TOK * (kDc + kPad) + (size_t)s.E * (kDc + kPad) +
                                       (size_t)TOK * (s.E + 1));
  auto kern = router_fma_kernel<TIn, TOK>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  kern<<<(s.T + TOK - 1) / TOK, kThreads, smem, st>>>(static_cast<const TIn*>(x), static_cast<const TIn*>(w), bias,
                                                      s.T, s.d, s.E, s.k, s.score, s.renorm, idx, gate, scores);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_router_fma(const Shape& s, const void* x, const void* w, const float* bias,
                              int32_t* idx, float* gate, float* scores, cudaStream_t st) {
  const bool small = (s.T + 31) / 32 < num_sms();     // 32-token CTAs would leave SMs idle
  if (s.dtype == MOE_BF16)
    return small ? launch_tok<__nv_bfloat16, 8>(s, x, w, bias, idx, gate, scores, st)
                 : launch_tok<__nv_bfloat16, 32>(s, x, w, bias, idx, gate, scores, st);
  return small ? launch_tok<float, 8>(s, x, w, bias, idx, gate, scores, st)
               : launch_tok<float, 32>(s, x, w, bias, idx, gate, scores, st);
}

}  // namespace moe
