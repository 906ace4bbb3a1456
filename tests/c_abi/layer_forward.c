/*
 * A plain C client of libmoe.so: one bf16 MoE layer forward through the C ABI of
 * include/moe.h, with no Python and no torch. Inputs come from a fixed integer hash (the
 * same values the Python test builds), device memory from cudaMalloc; the output, the top-k
 * ids and the per-expert counts are written raw to the file named by argv[1].
 *
 * Layer: T = 64 tokens, d_model = 256, 8 experts, top-2, d_ff = 256, softmax with
 * renormalised gates, dropless, no bias, no shared expert.
 *
 * Exit status: 0 on success, 1 on a usage or CUDA error, 2 when a moe_* call fails.
 */
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cuda_runtime.h>

#include "moe.h"

enum { T = 64, D = 256, E = 8, K = 2, F = 256 };

/* value i of stream `seed`: uniform on [-1, 1) in steps of 2^-23, times 2^-scale_log2 */
static float hash_value(uint32_t seed, uint32_t i, int scale_log2) {
  uint32_t h = i * 2654435761u ^ seed;
  h ^= h >> 15;
  h *= 0x2c1b3c6du;
  h ^= h >> 12;
  h *= 0x297a2d39u;
  h ^= h >> 15;
  const float u = (float)(h >> 8) * (1.0f / 16777216.0f);   /* [0, 1), exact */
  const float v = u * 2.0f - 1.0f;                          /* exact */
  return v / (float)(1u << scale_log2);                      /* exact: a power of two */
}

/* float32 -> bf16, round to nearest even (finite values) */
static uint16_t to_bf16(float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  u += 0x7FFFu + ((u >> 16) & 1u);
  return (uint16_t)(u >> 16);
}

static int cuda_ok(cudaError_t e, const char* what) {
  if (e == cudaSuccess) return 1;
  fprintf(stderr, "%s: %s\n", what, cudaGetErrorString(e));
  return 0;
}

/* a device bf16 tensor of n values of stream `seed` */
static void* device_tensor(uint32_t seed, size_t n, int scale_log2) {
  uint16_t* h = (uint16_t*)malloc(n * sizeof(uint16_t));
  void* d = NULL;
  if (h == NULL) return NULL;
  for (size_t i = 0; i < n; ++i) h[i] = to_bf16(hash_value(seed, (uint32_t)i, scale_log2));
  if (!cuda_ok(cudaMalloc(&d, n * sizeof(uint16_t)), "cudaMalloc") ||
      !cuda_ok(cudaMemcpy(d, h, n * sizeof(uint16_t), cudaMemcpyHostToDevice), "cudaMemcpy")) {
    free(h);
    return NULL;
  }
  free(h);
  return d;
}

int main(int argc, char** argv) {
  if (argc != 2) {
    fprintf(stderr, "usage: %s OUTPUT_FILE\n", argv[0]);
    return 1;
  }
  moe_config_t cfg;
  memset(&cfg, 0, sizeof(cfg));
  cfg.T = T;
  cfg.d_model = D;
  cfg.n_experts = E;
  cfg.top_k = K;
  cfg.d_ff = F;
  cfg.n_shared = 0;
  cfg.score = MOE_SOFTMAX;
  cfg.renormalize = 1;
  cfg.capacity_factor = 0.0f;
  cfg.dtype = MOE_BF16;
  moe_status_t rc = moe_check_config(&cfg);
  if (rc != MOE_OK) {
    fprintf(stderr, "moe_check_config: %s\n", moe_status_string(rc));
    return 2;
  }

  void* x = device_tensor(1u, (size_t)T * D, 0);
  void* w_router = device_tensor(2u, (size_t)E * D, 4);
  void* w_gate = device_tensor(3u, (size_t)E * F * D, 4);
  void* w_up = device_tensor(4u, (size_t)E * F * D, 4);
  void* w_down = device_tensor(5u, (size_t)E * D * F, 4);
  if (!x || !w_router || !w_gate || !w_up || !w_down) return 1;
  void *out = NULL, *ws = NULL;
  int32_t *idx = NULL, *counts = NULL;
  const size_t ws_bytes = moe_workspace_size(&cfg);
  if (ws_bytes == 0) return 2;
  if (!cuda_ok(cudaMalloc(&out, (size_t)T * D * 2), "cudaMalloc") ||
      !cuda_ok(cudaMalloc((void**)&idx, (size_t)T * K * 4), "cudaMalloc") ||
      !cuda_ok(cudaMalloc((void**)&counts, (size_t)E * 4), "cudaMalloc") ||
      !cuda_ok(cudaMalloc(&ws, ws_bytes), "cudaMalloc"))
    return 1;

  cudaStream_t stream;
  if (!cuda_ok(cudaStreamCreate(&stream), "cudaStreamCreate")) return 1;
  if ((rc = moe_workspace_init(ws, ws_bytes, stream)) != MOE_OK ||
      (rc = moe_layer_forward(&cfg, x, w_router, NULL, w_gate, w_up, w_down, out, idx, counts, ws, ws_bytes,
                              stream)) != MOE_OK ||
      (rc = moe_get_device_error(ws, stream)) != MOE_OK) {
    fprintf(stderr, "moe_layer_forward: %s\n", moe_status_string(rc));
    return 2;
  }

  uint16_t h_out[T * D];
  int32_t h_idx[T * K], h_counts[E];
  if (!cuda_ok(cudaMemcpy(h_out, out, sizeof(h_out), cudaMemcpyDeviceToHost), "cudaMemcpy") ||
      !cuda_ok(cudaMemcpy(h_idx, idx, sizeof(h_idx), cudaMemcpyDeviceToHost), "cudaMemcpy") ||
      !cuda_ok(cudaMemcpy(h_counts, counts, sizeof(h_counts), cudaMemcpyDeviceToHost), "cudaMemcpy"))
    return 1;
  FILE* f = fopen(argv[1], "wb");
  if (f == NULL) {
    perror(argv[1]);
    return 1;
  }
  const int ok = fwrite(h_out, sizeof(h_out), 1, f) == 1 && fwrite(h_idx, sizeof(h_idx), 1, f) == 1 &&
                 fwrite(h_counts, sizeof(h_counts), 1, f) == 1;
  fclose(f);
  cudaStreamDestroy(stream);
  cudaFree(x);
  cudaFree(w_router);
  cudaFree(w_gate);
  cudaFree(w_up);
  cudaFree(w_down);
  cudaFree(out);
  cudaFree(idx);
  cudaFree(counts);
  cudaFree(ws);
  return ok ? 0 : 1;
}
