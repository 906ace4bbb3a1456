// Seeded synthetic input generator, device side.
//
// Test and benchmark infrastructure: fills device buffers with the same
// values synth/gen_host.c produces on the host, bit for bit, so that
// multi-gigabyte expert weights never cross PCIe. It holds none of the MoE
// layer's arithmetic. The definition (SplitMix64 counter stream -> Irwin-Hall(4)
// centred sum -> one binary32 multiply -> optional bf16 round-to-nearest-even)
// is written out in synth/gen_host.c; the two files must agree exactly.
#include <cstdint>
#include <cuda_runtime.h>

namespace {

__device__ __forceinline__ uint64_t mix64(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
  return z ^ (z >> 31);
}

__device__ __forceinline__ float synth_value(uint64_t key, uint64_t i, float scale) {
  uint64_t b = mix64(key + (i + 1ULL) * 0x9E3779B97F4A7C15ULL);
  uint32_t s = (uint32_t)(b & 0xFFFFu) + (uint32_t)((b >> 16) & 0xFFFFu) +
               (uint32_t)((b >> 32) & 0xFFFFu) + (uint32_t)((b >> 48) & 0xFFFFu);
  int32_t c = 2 * (int32_t)s - 262140;
  return __fmul_rn((float)c, scale);  // |c| < 2^24: the conversion is exact
}

__device__ __forceinline__ uint16_t bf16_rne_bits(float v) {
  uint32_t u = __float_as_uint(v);
  u += 0x7FFFu + ((u >> 16) & 1u);
  return (uint16_t)(u >> 16);
}

__global__ void fill_bf16_kernel(uint64_t key, uint64_t start, uint64_t n, float scale,
                                 uint16_t* __restrict__ out) {
  // Eight elements per thread, one 16-byte store when the run is whole.
  uint64_t base = ((uint64_t)blockIdx.x * blockDim.x + threadIdx.x) * 8ULL;
  const uint64_t stride = (uint64_t)gridDim.x * blockDim.x * 8ULL;
  for (; base < n; base += stride) {
    if (base + 8 <= n && ((reinterpret_cast<uintptr_t>(out + base) & 15u) == 0)) {
      uint32_t w[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        uint32_t lo = bf16_rne_bits(synth_value(key, start + base + 2 * q, scale));
        uint32_t hi = bf16_rne_bits(synth_value(key, start + base + 2 * q + 1, scale));
        w[q] = lo | (hi << 16);
      }
      *reinterpret_cast<uint4*>(out + base) = make_uint4(w[0], w[1], w[2], w[3]);
    } else {
      for (uint64_t j = base; j < n && j < base + 8; ++j)
        out[j] = bf16_rne_bits(synth_value(key, start + j, scale));
    }
  }
}

__global__ void fill_f32_kernel(uint64_t key, uint64_t start, uint64_t n, float scale,
                                float* __restrict__ out) {
  uint64_t j = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const uint64_t stride = (uint64_t)gridDim.x * blockDim.x;
  for (; j < n; j += stride) out[j] = synth_value(key, start + j, scale);
}

uint64_t host_mix64(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
  return z ^ (z >> 31);
}

}  // namespace

extern "C" {

// Fills out[0..n) (device memory) with elements start..start+n of the stream
// (seed, tensor_id). dtype 0 = float32, 1 = bfloat16 bit patterns. Returns the
// cudaError_t of the launch (0 on success). Asynchronous on `stream`.
int synth_fill_device(void* out, uint64_t n, uint64_t seed, uint64_t tensor_id,
                      uint64_t start, float scale, int dtype, cudaStream_t stream) {
  if (n == 0) return 0;
  if (out == nullptr) return (int)cudaErrorInvalidValue;
  const uint64_t key = host_mix64(seed * 0x9E3779B97F4A7C15ULL + tensor_id * 0xD1B54A32D192ED03ULL);
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int threads = 256;
  const uint64_t per_block = (dtype == 1 ? 8ULL : 1ULL) * threads;
  uint64_t want = (n + per_block - 1) / per_block;
  uint64_t cap = (uint64_t)sms * 16ULL;
  unsigned blocks = (unsigned)(want < cap ? want : cap);
  if (dtype == 1)
    fill_bf16_kernel<<<blocks, threads, 0, stream>>>(key, start, n, scale, static_cast<uint16_t*>(out));
  else
    fill_f32_kernel<<<blocks, threads, 0, stream>>>(key, start, n, scale, static_cast<float*>(out));
  return (int)cudaGetLastError();
}

}  // extern "C"
