// Internal declarations shared by the kernels of libmoe.so.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>
#include <cuda_bf16.h>

#include "../../include/moe.h"

namespace moe {

// ---------------------------------------------------------------- limits ---
constexpr int kMaxExperts = 256;
constexpr int kMaxTopK = 8;
constexpr int kChunk = 128;          // tokens per chunk of the grouping kernels

// ------------------------------------------------------ workspace layout ---
// Byte offsets inside the caller's workspace; every segment is 256-byte aligned.
struct WsLayout {
  size_t status;        // int32 status word (+ padding)
  size_t topk_idx;      // [T*k] int32
  size_t topk_gate;     // [T*k] float
  size_t chunk_counts;  // [nchunks*E] int32: per-chunk histogram, then per-chunk rank base
  size_t counts;        // [E] int32
  size_t offsets;       // [E+1] int32
  size_t sched;         // [4*(G+1)] int32: group schedule of the grouped GEMMs
  size_t dest_row;      // [T*k] int32
  size_t src_token;     // [R] int32
  size_t x_perm;        // [R*d] elements (at least (R+S*T)*d bytes: the W8A8 grouped row codes)
  size_t h;             // [(R+S*T)*F] elements: silu(gate) * up
  size_t y;             // [(R+S*T)*d] elements: expert outputs; with the fused combine, the
                        // [T*d] float32 output accumulator instead (the region holds either);
                        // in the W8A8 layer first the E4M3 codes of the expert inputs [(R+S*T)*d]
  size_t a8_scale;      // [R+S*T] float: W8A8 per-row scales of the expert inputs
  size_t xq_scale;      // [T] float: W8A8 per-token scales (the per-token codes use the y region)
  size_t h8;            // [(R+S*T)*F] bytes: W8A8 E4M3 codes of h
  size_t h8_scale;      // [R+S*T] float: their per-row scales
  size_t mlp_ready;     // [2 * m-tiles] int32: the one-launch expert MLP's per-m-tile counters
  size_t total;
};

struct Shape {
  int T, d, E, k, F, S, G;
  int score, renorm, dtype;
  int cap;            // per-expert capacity (T when dropless)
  int64_t R;          // rows of the grouped buffer for routed pairs
  int nchunks;
  size_t esize;       // bytes per activation / weight element
};

Shape make_shape(const moe_config_t& c);
WsLayout make_layout(const Shape& s);

// Group schedule (device, int32), G groups:
//   tile_start[G+1]  prefix sum of 128-row M tiles per group
//   a_row[G]         first A row of the group (x_perm row, or x row 0 for the shared group)
//   out_row[G]       first output row of the group in h / y
//   rows[G]          rows of the group
struct SchedView {
  int32_t* tile_start;
  int32_t* a_row;
  int32_t* out_row;
  int32_t* rows;
};
inline SchedView sched_view(void* base, int G) {
  int32_t* p = static_cast<int32_t*>(base);
  return SchedView{p, p + (G + 1), p + (G + 1) + G, p + (G + 1) + 2 * G};
}

// ------------------------------------------------------- device helpers ---
__device__ __forceinline__ void set_status(int32_t* status, int code) {
  if (status) atomicCAS(status, 0, code);
}

__device__ __forceinline__ float bf16_to_f32(__nv_bfloat16 v) { return __bfloat162float(v); }

template <typename T> __device__ __forceinline__ float to_f32(T v);
template <> __device__ __forceinline__ float to_f32<float>(float v) { return v; }
template <> __device__ __forceinline__ float to_f32<__nv_bfloat16>(__nv_bfloat16 v) { return __bfloat162float(v); }

template <typename T> __device__ __forceinline__ T from_f32(float v);
template <> __device__ __forceinline__ float from_f32<float>(float v) { return v; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float v) { return __float2bfloat16_rn(v); }

// ------------------------------------------------------------- launchers ---
// Each returns cudaGetLastError() after enqueueing.
cudaError_t launch_router_fma(const Shape& s, const void* x, const void* w, const float* bias,
                              int32_t* idx, float* gate, float* scores, cudaStream_t st);
bool router_tc_supported(const Shape& s);
cudaError_t launch_router_tc(const Shape& s, const void* x, const void* w, const float* bias,
                             int32_t* idx, float* gate, float* scores, int32_t* status, cudaStream_t st);

cudaError_t launch_group_hist(const Shape& s, const int32_t* idx, int32_t* chunk_counts,
                              int32_t* status, cudaStream_t st);
// sched: NULL, or the workspace group schedule to build from the new offsets
cudaError_t launch_group_scan(const Shape& s, int32_t* chunk_counts, int32_t* counts,
                              int32_t* offsets, void* sched, cudaStream_t st);
cudaError_t launch_group_scatter(const Shape& s, const int32_t* idx, const int32_t* chunk_base,
                                 const int32_t* offsets, int32_t* dest_row, int32_t* src_token,
                                 cudaStream_t st);
// hist + scan (+ schedule) + scatter in one CTA; only for a single chunk (T <= kChunk).
cudaError_t launch_group_single_chunk(const Shape& s, const int32_t* idx, int32_t* counts, int32_t* offsets,
                                      int32_t* dest_row, int32_t* src_token, void* sched, int32_t* status,
                                      cudaStream_t st);
cudaError_t launch_gather_rows(const Shape& s, const void* x, const int32_t* src_token,
                               const int32_t* offsets, void* x_perm, cudaStream_t st);
// The single-chunk grouping and the grouped copy of x in one launch (every block groups in its
// own shared memory, block 0 writes the grouping out, each block copies its rows).
cudaError_t launch_group_gather_single_chunk(const Shape& s, const int32_t* idx, int32_t* counts, int32_t* offsets,
                                             int32_t* dest_row, int32_t* src_token, void* sched, int32_t* status,
                                             const void* x, void* x_perm, cudaStream_t st);

cudaError_t launch_group_schedule(const Shape& s, const int32_t* offsets, void* sched,
                                  int32_t* status, cudaStream_t st);
// The float32 MLP (two kernels); mid_event (nullable) is recorded between them. src_token
// (nullable): routed rows are read from x through it instead of from x_perm.
cudaError_t launch_ffn_fma(const Shape& s, const void* x_perm, const void* x, const void* w_gate,
                           const void* w_up, const void* w_down, const void* sched, void* h, void* y,
                           cudaStream_t st, cudaEvent_t mid_event, const int32_t* src_token = nullptr);

// A timing event: recorded as an external event node when the stream is being captured
// into a CUDA graph, so that replays record it (a plain record would only order nodes).
inline cudaError_t record_event(cudaEvent_t ev, cudaStream_t st) {
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  cudaError_t e = cudaStreamIsCapturing(st, &cs);
  if (e != cudaSuccess) return e;
  if (cs == cudaStreamCaptureStatusActive) return cudaEventRecordWithFlags(ev, st, cudaEventRecordExternal);
  return cudaEventRecord(ev, st);
}
cudaError_t launch_gemm_gateup_tc(const Shape& s, const void* x_perm, const void* x,
                                  const void* w_gate, const void* w_up, const void* sched, void* h,
                                  int32_t* status, cudaStream_t st);
cudaError_t launch_gemm_down_tc(const Shape& s, const void* h, const void* w_down,
                                const void* sched, void* y, int32_t* status, cudaStream_t st);
// The down projection with the combine in its epilogue: each row's output times its gate
// (one for the shared expert) is added in float32 into acc_out [T, d] (zeroed beforehand).
cudaError_t launch_gemm_down_combine_tc(const Shape& s, const void* h, const void* w_down, const void* sched,
                                        const int32_t* src_token, const int32_t* dest_row, const float* gate,
                                        float* acc_out, int32_t* status, cudaStream_t st);
// out [T, d] bf16 = acc [T, d] float32, rounded once.
cudaError_t launch_combine_finalize(const Shape& s, const float* acc, void* out, cudaStream_t st);

// FP8 (E4M3) expert weights with per-row float32 scales (gemm_fp8w.cu).
bool fp8w_supported(const Shape& s);
cudaError_t launch_quantize_fp8_rows(const void* w, int64_t rows, int cols, uint8_t* wq, float* scale,
                                     cudaStream_t st);
cudaError_t launch_gemm_gateup_fp8w(const Shape& s, const void* x_perm, const void* x, const uint8_t* wg_q,
                                    const float* wg_s, const uint8_t* wu_q, const float* wu_s, const void* sched,
                                    void* h, int32_t* status, cudaStream_t st);
cudaError_t launch_gemm_down_fp8w(const Shape& s, const void* h, const uint8_t* wd_q, const float* wd_s,
                                  const void* sched, void* y, int32_t* status, cudaStream_t st);

// Both contractions of the bf16 expert MLP in one persistent launch (gemm_fused.cu); `ready`
// holds fused_mlp_ready_ints(s) int32 (zeroed by the launcher). out non-NULL: the down tiles
// also combine (each token's output row by the tile that completes it; src_token, dest_row
// and gate of the grouping and router), with the separate combine's bits.
bool fused_mlp_supported(const Shape& s);
int64_t fused_mlp_ready_ints(const Shape& s);
cudaError_t launch_mlp_fused_tc(const Shape& s, const void* x_perm, const void* x, const void* w_gate,
                                const void* w_up, const void* w_down, const void* sched, void* h, void* y,
                                int32_t* ready, int32_t* status, cudaStream_t st, const int32_t* src_token = nullptr,
                                const int32_t* dest_row = nullptr, const float* gate = nullptr, void* out = nullptr);

// The W8A8 expert MLP in one persistent launch (gemm_w8a8_fused.cu); `counters` holds
// 2 * fused_mlp_ready_ints(s) int32 (zeroed by the launcher).
cudaError_t launch_mlp_w8a8_fused(const Shape& s, const uint8_t* x8, const float* x8_scale, const uint8_t* wg_q,
                                  const float* wg_s, const uint8_t* wu_q, const float* wu_s, const uint8_t* wd_q,
                                  const float* wd_s, const void* sched, void* h, uint8_t* h8, float* h8_scale,
                                  void* y, int32_t* counters, int32_t* status, cudaStream_t st);

// W8A8 (E4M3 weights and activations, gemm_w8a8.cu).
bool w8a8_supported(const Shape& s);
// Activation rows to E4M3 codes + per-row scales: rows [0, min(*n_a, max_a)) of src_a to the
// same rows of dst, rows [0, n_b) of src_b (may be NULL when n_b = 0) to rows [R, R + n_b).
cudaError_t launch_quantize_act_rows(const Shape& s, const void* src_a, const int32_t* n_a, int64_t max_a,
                                     const void* src_b, int64_t n_b, int cols, uint8_t* dst, float* scale,
                                     cudaStream_t st);
// x rows of the grouping (src_token order; the shared expert's tokens after row R) -> E4M3
// codes and per-row scales, in place of the bf16 row copy, for batches of more than one chunk.
// xq [T, d] bytes and xq_scale [T]: scratch for the per-token codes.
cudaError_t launch_gather_quant_rows(const Shape& s, const void* x, const int32_t* src_token, const int32_t* offsets,
                                     uint8_t* x8, float* x8_scale, uint8_t* xq, float* xq_scale, cudaStream_t st);
// W8A8, a single chunk: the grouping and the grouped rows as E4M3 codes in one launch (as
// launch_group_gather_single_chunk, each block quantising its rows; the shared expert's after R).
cudaError_t launch_group_quant_single_chunk(const Shape& s, const int32_t* idx, int32_t* counts, int32_t* offsets,
                                            int32_t* dest_row, int32_t* src_token, void* sched, int32_t* status,
                                            const void* x, uint8_t* x8, float* x8_scale, cudaStream_t st);
cudaError_t launch_gemm_gateup_w8a8(const Shape& s, const uint8_t* x8, const float* x8_scale, const uint8_t* wg_q,
                                    const float* wg_s, const uint8_t* wu_q, const float* wu_s, const void* sched,
                                    void* h, int32_t* status, cudaStream_t st);
cudaError_t launch_gemm_down_w8a8(const Shape& s, const uint8_t* h8, const float* h8_scale, const uint8_t* wd_q,
                                  const float* wd_s, const void* sched, void* y, int32_t* status, cudaStream_t st);

cudaError_t launch_combine(const Shape& s, const void* y, const int32_t* dest_row,
                           const float* gate, void* out, int32_t* status, cudaStream_t st);

cudaError_t launch_wait_selftest(int32_t* status, uint64_t limit_ns, cudaStream_t st);

int num_sms();

}  // namespace moe
