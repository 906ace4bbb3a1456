// Gate-weighted combine back in token order, and the bounded-wait self-test.
//
// out[t] = sum over the token's kept slots j of gate[t,j] * y[dest_row[t,j]],
// plus the shared expert's row with weight one. Follows
// shubhamtatvamasi.com/llm-inference/moe "Mixture of Experts", Q&A "How does
// a top-k router work?" (the output is the gate-weighted sum of the selected
// experts' outputs) and section "The router" (shared experts every token
// visits), and klaylearn.com/glossary/mixture-of-experts (undo the
// permutation). A dropped slot (dest_row = -1) contributes nothing: for that
// expert the token only goes on through the residual connection (same page, "Load
// imbalance"); the residual add itself is outside this layer.
//
// One CTA per token; each thread owns 16 bytes of the row and accumulates its
// slots in float32 in slot order, the shared row last. All loads and stores are
// coalesced 16-byte vectors. A thread issues the loads of all its slots (kept as
// raw 16-byte words, KM of them: k rounded up to 2, 4 or 8) before the first
// multiply-add, so a token's k rows are in flight together.
#include "internal.cuh"
#include "tc_ptx.cuh"

namespace moe {
namespace {

template <typename TE>
struct Vec;
template <>
struct Vec<__nv_bfloat16> {
  static constexpr int kN = 8;
  __device__ static void unpack(const uint4 u, float (&v)[8]) {
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      v[2 * i] = __uint_as_float(w[i] << 16);
      v[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
    }
  }
  __device__ static void store(__nv_bfloat16* p, const float (&v)[8]) {
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const __nv_bfloat162 b = __floats2bfloat162_rn(v[2 * i], v[2 * i + 1]);
      w[i] = *reinterpret_cast<const uint32_t*>(&b);
    }
    *reinterpret_cast<uint4*>(p) = make_uint4(w[0], w[1], w[2], w[3]);
  }
};
template <>
struct Vec<float> {
  static constexpr int kN = 4;
  __device__ static void unpack(const uint4 u, float (&v)[4]) {
    v[0] = __uint_as_float(u.x); v[1] = __uint_as_float(u.y); v[2] = __uint_as_float(u.z); v[3] = __uint_as_float(u.w);
  }
  __device__ static void store(float* p, const float (&v)[4]) {
    *reinterpret_cast<float4*>(p) = make_float4(v[0], v[1], v[2], v[3]);
  }
};

template <typename TE, int KM>
__global__ void combine_kernel(const TE* __restrict__ y, const int32_t* __restrict__ dest_row,
                               const float* __restrict__ gate, TE* __restrict__ out, int d, int k, int S, int T,
                               int64_t R, int32_t* status) {
  constexpr int V = Vec<TE>::kN;
  const int t = blockIdx.x;
  __shared__ int32_t s_row[kMaxTopK];
  __shared__ float s_gate[kMaxTopK];
  if (threadIdx.x < k) {
    int r = dest_row[(size_t)t * k + threadIdx.x];
    if (r >= R) {
      set_status(status, MOE_ERR_DEVICE_INDEX);
      r = -1;
    }
    s_row[threadIdx.x] = r < 0 ? -1 : r;
    s_gate[threadIdx.x] = gate[(size_t)t * k + threadIdx.x];
  }
  __syncthreads();
  for (int c = threadIdx.x * V; c < d; c += blockDim.x * V) {
    uint4 raw[KM];
#pragma unroll
    for (int j = 0; j < KM; ++j) {
      const int r = j < k ? s_row[j] : -1;
      raw[j] = r >= 0 ? __ldg(reinterpret_cast<const uint4*>(y + (size_t)r * d + c)) : make_uint4(0, 0, 0, 0);
    }
    uint4 shared_raw = make_uint4(0, 0, 0, 0);
    if (S > 0) shared_raw = __ldg(reinterpret_cast<const uint4*>(y + (size_t)(R + t) * d + c));
    float acc[V];
#pragma unroll
    for (int i = 0; i < V; ++i) acc[i] = 0.f;
#pragma unroll
    for (int j = 0; j < KM; ++j) {
      if (j >= k || s_row[j] < 0) continue;
      float v[V];
      Vec<TE>::unpack(raw[j], v);
      const float g = s_gate[j];
#pragma unroll
      for (int i = 0; i < V; ++i) acc[i] = fmaf(g, v[i], acc[i]);
    }
    if (S > 0) {
      float v[V];
      Vec<TE>::unpack(shared_raw, v);
#pragma unroll
      for (int i = 0; i < V; ++i) acc[i] += v[i];
    }
    Vec<TE>::store(out + (size_t)t * d + c, acc);
  }
}

// One CTA waits on an mbarrier that no one arrives on; the bounded wait gives up.
__global__ void wait_selftest_kernel(int32_t* status, uint64_t limit_ns) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    ptx::mbar_init(ptx::smem_u32(&bar), 1);
    abort_flag = 0;
    ptx::fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    if (!ptx::mbar_wait_bounded(ptx::smem_u32(&bar), 0, &abort_flag, limit_ns))
      set_status(status, MOE_ERR_TIMEOUT);
  }
}

// out = bf16(acc), eight elements (32 bytes in, 16 out) per thread step.
__global__ void combine_finalize_kernel(const float4* __restrict__ acc, uint4* __restrict__ out, int64_t n8) {
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n8; i += (int64_t)gridDim.x * blockDim.x) {
    const float4 a = acc[2 * i], b = acc[2 * i + 1];
    const __nv_bfloat162 p0 = __floats2bfloat162_rn(a.x, a.y), p1 = __floats2bfloat162_rn(a.z, a.w);
    const __nv_bfloat162 p2 = __floats2bfloat162_rn(b.x, b.y), p3 = __floats2bfloat162_rn(b.z, b.w);
    out[i] = make_uint4(*reinterpret_cast<const uint32_t*>(&p0), *reinterpret_cast<const uint32_t*>(&p1),
                        *reinterpret_cast<const uint32_t*>(&p2), *reinterpret_cast<const uint32_t*>(&p3));
  }
}

}  // namespace

cudaError_t launch_combine_finalize(const Shape& s, const float* acc, void* out, cudaStream_t st) {
  const int64_t n8 = (int64_t)s.T * s.d / 8;          // d is a multiple of 128 for bf16 layers
  int64_t blocks = (n8 + 255) / 256;
  const int64_t cap = (int64_t)num_sms() * 8;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  combine_finalize_kernel<<<(unsigned)blocks, 256, 0, st>>>(reinterpret_cast<const float4*>(acc),
                                                              static_cast<uint4*>(out), n8);
  return cudaGetLastError();
}

cudaError_t launch_combine(const Shape& s, const void* y, const int32_t* dest_row, const float* gate, void* out,
                           int32_t* status, cudaStream_t st) {
  const int V = (s.dtype == MOE_BF16) ? 8 : 4;
  int threads = (s.d / V + 31) / 32 * 32;
  if (threads > 256) threads = 256;
  if (threads < 32) threads = 32;
  if (s.dtype == MOE_BF16) {
    const __nv_bfloat16* yb = static_cast<const __nv_bfloat16*>(y);
    __nv_bfloat16* ob = static_cast<__nv_bfloat16*>(out);
    if (s.k <= 2)
      combine_kernel<__nv_bfloat16, 2><<<s.T, threads, 0, st>>>(yb, dest_row, gate, ob, s.d, s.k, s.S, s.T, s.R, status);
    else if (s.k <= 4)
      combine_kernel<__nv_bfloat16, 4><<<s.T, threads, 0, st>>>(yb, dest_row, gate, ob, s.d, s.k, s.S, s.T, s.R, status);
    else
      combine_kernel<__nv_bfloat16, 8><<<s.T, threads, 0, st>>>(yb, dest_row, gate, ob, s.d, s.k, s.S, s.T, s.R, status);
  } else {
    const float* yf = static_cast<const float*>(y);
    float* of = static_cast<float*>(out);
    if (s.k <= 2)
      combine_kernel<float, 2><<<s.T, threads, 0, st>>>(yf, dest_row, gate, of, s.d, s.k, s.S, s.T, s.R, status);
    else if (s.k <= 4)
      combine_kernel<float, 4><<<s.T, threads, 0, st>>>(yf, dest_row, gate, of, s.d, s.k, s.S, s.T, s.R, status);
    else
      combine_kernel<float, 8><<<s.T, threads, 0, st>>>(yf, dest_row, gate, of, s.d, s.k, s.S, s.T, s.R, status);
  }
  return cudaGetLastError();
}

cudaError_t launch_wait_selftest(int32_t* status, uint64_t limit_ns, cudaStream_t st) {
  wait_selftest_kernel<<<1, 32, 0, st>>>(status, limit_ns);
  return cudaGetLastError();
}

}  // namespace moe
