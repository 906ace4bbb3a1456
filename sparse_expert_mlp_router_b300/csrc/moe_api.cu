// The C ABI of libmoe.so: host-side validation, workspace layout and the
// enqueueing of the stage kernels. Declarations and their documentation are in
// include/moe.h.
#include <atomic>
#include <cmath>
#include <cstdlib>
#include <cstring>

#include <nvtx3/nvToolsExt.h>

#include "internal.cuh"

namespace moe {

// SM count of the current device, cached per device (threads may race to fill an entry; they
// store the same value).
int num_sms() {
  static std::atomic<int> cached[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return 148;
  if (dev < 64) {
    const int c = cached[dev].load(std::memory_order_relaxed);
    if (c > 0) return c;
  }
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 148;
  if (dev < 64) cached[dev].store(n, std::memory_order_relaxed);
  return n;
}

namespace {

constexpr size_t kAlign = 256;
inline size_t align_up(size_t v) { return (v + kAlign - 1) / kAlign * kAlign; }

// Exact ceil(cf * T * k / E) on the binary32 value of cf, clamped to [1, T].
// cf = m * 2^e with m a 24-bit integer; the quotient is evaluated in 128-bit integers.
int exact_capacity(float cf, int T, int k, int E) {
  if (!(cf > 0.0f)) return T;
  int ex = 0;
  const float fr = std::frexp(cf, &ex);                    // cf = fr * 2^ex, fr in [0.5, 1)
  const unsigned __int128 m = (unsigned __int128)(uint64_t)std::ldexp(fr, 24);   // exact
  const int e = ex - 24;
  unsigned __int128 num = m * (unsigned __int128)T * (unsigned __int128)k;
  unsigned __int128 den = (unsigned __int128)E;
  if (e >= 0) {
    if (e > 40) return T;
    num <<= e;
  } else {
    if (-e > 100) return 1;
    den <<= -e;
  }
  const unsigned __int128 q = (num + den - 1) / den;
  if (q >= (unsigned __int128)T) return T;
  return q < 1 ? 1 : (int)q;
}

moe_status_t check_cfg(const moe_config_t* c) {
  if (c == nullptr) return MOE_ERR_INVALID_ARG;
  if (c->T < 1 || c->d_model < 1 || c->n_experts < 1 || c->top_k < 1 || c->d_ff < 1) return MOE_ERR_INVALID_ARG;
  if (c->top_k > c->n_experts) return MOE_ERR_INVALID_ARG;
  if (c->n_shared < 0 || (c->score != MOE_SOFTMAX && c->score != MOE_SIGMOID)) return MOE_ERR_INVALID_ARG;
  if (c->renormalize != 0 && c->renormalize != 1) return MOE_ERR_INVALID_ARG;
  if (c->dtype != MOE_F32 && c->dtype != MOE_BF16) return MOE_ERR_INVALID_ARG;
  if (std::isnan(c->capacity_factor)) return MOE_ERR_INVALID_ARG;
  if (c->T > (1 << 20) || c->n_experts > kMaxExperts || c->top_k > kMaxTopK || c->n_shared > 1)
    return MOE_ERR_UNSUPPORTED;
  if (c->dtype == MOE_BF16) {
    if (c->d_model % 128 != 0 || c->d_ff % 128 != 0) return MOE_ERR_UNSUPPORTED;
  } else {
    if (c->d_model % 4 != 0 || c->d_ff % 4 != 0) return MOE_ERR_UNSUPPORTED;
  }
  if ((int64_t)c->d_model * c->d_ff * (c->n_experts + c->n_shared) > (int64_t)1 << 40) return MOE_ERR_UNSUPPORTED;
  return MOE_OK;
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

}  // namespace

Shape make_shape(const moe_config_t& c) {
  Shape s{};
  s.T = c.T;
  s.d = c.d_model;
  s.E = c.n_experts;
  s.k = c.top_k;
  s.F = c.d_ff;
  s.S = c.n_shared;
  s.G = s.E + s.S;
  s.score = c.score;
  s.renorm = c.renormalize;
  s.dtype = c.dtype;
  s.cap = exact_capacity(c.capacity_factor, s.T, s.k, s.E);
  const int64_t tk = (int64_t)s.T * s.k, ec = (int64_t)s.E * s.cap;
  s.R = tk < ec ? tk : ec;
  s.nchunks = (s.T + kChunk - 1) / kChunk;
  s.esize = (c.dtype == MOE_BF16) ? 2 : 4;
  return s;
}

WsLayout make_layout(const Shape& s) {
  WsLayout L{};
  size_t o = 0;
  auto take = [&](size_t bytes) {
    const size_t at = o;
    o = align_up(o + bytes);
    return at;
  };
  const size_t pairs = (size_t)s.T * s.k;
  const size_t grouped = (size_t)s.R + (size_t)s.S * s.T;
  L.status = take(kAlign);
  L.topk_idx = take(pairs * 4);
  L.topk_gate = take(pairs * 4);
  L.chunk_counts = take((size_t)s.nchunks * s.E * 4);
  L.counts = take((size_t)s.E * 4);
  L.offsets = take((size_t)(s.E + 1) * 4);
  L.sched = take((size_t)4 * (s.G + 1) * 4);
  L.dest_row = take(pairs * 4);
  L.src_token = take((size_t)s.R * 4);
  // x_perm holds the W8A8 layer's grouped E4M3 rows [R + S*T, d] (bytes) instead of the bf16
  // rows: nothing in the expert stage writes it, so the one-launch MLP's gate/up tiles can read
  // the codes while its down tiles already write y
  size_t xp_bytes = (size_t)s.R * s.d * s.esize;
  if (s.dtype == MOE_BF16 && xp_bytes < grouped * s.d) xp_bytes = grouped * s.d;
  L.x_perm = take(xp_bytes);
  L.h = take(grouped * s.F * s.esize);
  // y also holds the fused combine's float32 sums [T, d] and, during the grouping stage of a
  // multi-chunk W8A8 layer, the per-token E4M3 codes [T, d] (bytes)
  size_t y_bytes = grouped * s.d * s.esize;
  if (s.dtype == MOE_BF16 && y_bytes < (size_t)s.T * s.d * 4) y_bytes = (size_t)s.T * s.d * 4;
  L.y = take(y_bytes);
  if (s.dtype == MOE_BF16) {
    L.a8_scale = take(grouped * 4);
    L.xq_scale = take((size_t)s.T * 4);
    L.h8 = take(grouped * s.F);
    L.h8_scale = take(grouped * 4);
    L.mlp_ready = take((size_t)2 * fused_mlp_ready_ints(s) * 4);
  }
  L.total = o;
  return L;
}

}  // namespace moe

using namespace moe;

namespace {

// NVTX range over a scope (host-side; a profiler shows the kernels each stage enqueues under
// its name, e.g. ncu --nvtx --nvtx-include "moe_layer/experts/"). Without a tool attached the
// calls return at once.
struct NvtxRange {
  explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
  ~NvtxRange() { nvtxRangePop(); }
  NvtxRange(const NvtxRange&) = delete;
  NvtxRange& operator=(const NvtxRange&) = delete;
};

template <typename T>
T* at(void* ws, size_t off) {
  return reinterpret_cast<T*>(static_cast<char*>(ws) + off);
}

moe_status_t check_ws(const Shape& s, const void* ws, size_t ws_bytes) {
  if (ws == nullptr || !aligned(ws, 256)) return MOE_ERR_INVALID_ARG;
  if (ws_bytes < make_layout(s).total) return MOE_ERR_WORKSPACE;
  return MOE_OK;
}

inline moe_status_t cuda_status(cudaError_t e) { return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA; }

// The stage bodies, shared by the stage entry points and the whole-layer call.
cudaError_t run_router(const Shape& s, const void* x, const void* w_router, const float* bias, int32_t* idx,
                       float* gate, float* scores, int32_t* status, cudaStream_t st) {
  if (router_tc_supported(s)) return launch_router_tc(s, x, w_router, bias, idx, gate, scores, status, st);
  return launch_router_fma(s, x, w_router, bias, idx, gate, scores, st);
}

// with_schedule: the scan also builds the group schedule of the grouped GEMMs (the
// whole-layer call); the permute stage call leaves it to moe_grouped_ffn.
// x8 / x8s (W8A8 layer): when set, the grouped rows are written as E4M3 codes with per-row
// scales (the shared expert's tokens after row R) instead of the bf16 copy in x_perm.
cudaError_t run_permute(const Shape& s, const WsLayout& L, void* ws, const int32_t* idx, const void* x,
                        int32_t* counts, int32_t* offsets, int32_t* dest_row, int32_t* src_token, void* x_perm,
                        bool with_schedule, cudaStream_t st, uint8_t* x8 = nullptr, float* x8s = nullptr,
                        bool copy_rows = true) {
  int32_t* status = at<int32_t>(ws, L.status);
  int32_t* cc = at<int32_t>(ws, L.chunk_counts);
  cudaError_t e;
  if (s.nchunks == 1) {
    // one chunk of tokens (decode): the three grouping steps and the row copy (or quantising
    // copy) in one launch, each block grouping in its own shared memory
    void* sched = with_schedule ? at<void>(ws, L.sched) : nullptr;
    if (x8 != nullptr)
      return launch_group_quant_single_chunk(s, idx, counts, offsets, dest_row, src_token, sched, status, x, x8, x8s,
                                             st);
    if (copy_rows)
      return launch_group_gather_single_chunk(s, idx, counts, offsets, dest_row, src_token, sched, status, x, x_perm,
                                              st);
    return launch_group_single_chunk(s, idx, counts, offsets, dest_row, src_token, sched, status, st);
  } else {
    if ((e = launch_group_hist(s, idx, cc, status, st)) != cudaSuccess) return e;
    if ((e = launch_group_scan(s, cc, counts, offsets, with_schedule ? at<void>(ws, L.sched) : nullptr, st)) !=
        cudaSuccess)
      return e;
    if ((e = launch_group_scatter(s, idx, cc, offsets, dest_row, src_token, st)) != cudaSuccess) return e;
  }
  if (x8 != nullptr)   // per-token codes (multi-chunk batches) go to the y region, free until the down projection
    return launch_gather_quant_rows(s, x, src_token, offsets, x8, x8s, at<uint8_t>(ws, L.y),
                                    at<float>(ws, L.xq_scale), st);
  if (!copy_rows) return cudaSuccess;
  return launch_gather_rows(s, x, src_token, offsets, x_perm, st);
}

// Group schedule from the offsets (one small kernel), then the two contractions.
cudaError_t run_schedule(const Shape& s, const WsLayout& L, void* ws, const int32_t* offsets, cudaStream_t st) {
  return launch_group_schedule(s, offsets, at<void>(ws, L.sched), at<int32_t>(ws, L.status), st);
}

// Whether the bf16 expert MLP runs as one persistent launch of both contractions instead of
// two launches: by default for batches of one 128-token chunk (decode), where the down tiles of
// the first experts fill the gate/up launch's last round of tiles and the gap between the
// launches (decode layer 0.192 -> 0.187 ms); on the prefill layers, which run at the power
// limit, it measured the same as two launches. MOE_FUSED_MLP=1 / 0 in the environment (read
// at every call) forces it on / off.
bool fused_mlp(const Shape& s) {
  if (!fused_mlp_supported(s)) return false;
  const char* v = getenv("MOE_FUSED_MLP");
  if (v != nullptr && (v[0] == '0' || v[0] == '1')) return v[0] == '1';
  return s.nchunks == 1;
}

// The W8A8 expert MLP as one launch (gate/up, h's quantisation by the tile that completes each
// m-tile, down) only when MOE_FUSED_MLP=1: it measured slower than the three launches on every
// shape (decode 0.137 vs 0.132 ms, Qwen3-shaped 1.61 vs 0.48, DeepSeek-shaped 2.95 vs 2.27).
bool fused_mlp_w8a8(const Shape& s) {
  if (!fused_mlp_supported(s)) return false;
  const char* v = getenv("MOE_FUSED_MLP");
  return v != nullptr && v[0] == '1';
}

// Whether the one-launch bf16 expert MLP also combines (each token's output row summed by the
// down tile that completes the token, in slot order: the separate combine's bits) instead of a
// combine launch after it: only with MOE_MLP_COMBINE=1 in the environment (read at every
// call), since on the decode batch it measured slower (0.203 vs 0.186 ms: the per-tile barriers
// of the epilogue warps and the per-token acquire-release counts slow the whole pipeline by
// more than the 6.6 us combine launch it saves).
bool mlp_combine(const Shape& s) {
  if (!fused_mlp(s)) return false;
  const char* v = getenv("MOE_MLP_COMBINE");
  return v != nullptr && v[0] == '1';
}

// Expert weights of a call: bf16 / float32 tensors, or FP8 codes with per-row scales.
struct ExpertWeights {
  const void* g;
  const void* u;
  const void* d;
  const float* gs = nullptr;
  const float* us = nullptr;
  const float* ds = nullptr;
  bool fp8 = false;
  bool a8 = false;       // W8A8: the activations entering each contraction quantised to E4M3 too
};

// src_token (nullable, float32 layers): the routed rows are read from x through it, x_perm unused.
cudaError_t run_ffn(const Shape& s, const WsLayout& L, void* ws, const void* x_perm, const void* x,
                    const ExpertWeights& w, void* y, cudaStream_t st, cudaEvent_t mid_event,
                    const int32_t* src_token = nullptr) {
  int32_t* status = at<int32_t>(ws, L.status);
  void* sched = at<void>(ws, L.sched);
  void* h = at<void>(ws, L.h);
  cudaError_t e;
  if (w.fp8) {
    if ((e = launch_gemm_gateup_fp8w(s, x_perm, x, static_cast<const uint8_t*>(w.g), w.gs,
                                     static_cast<const uint8_t*>(w.u), w.us, sched, h, status, st)) != cudaSuccess)
      return e;
    if (mid_event && (e = record_event(mid_event, st)) != cudaSuccess) return e;
    return launch_gemm_down_fp8w(s, h, static_cast<const uint8_t*>(w.d), w.ds, sched, y, status, st);
  }
  if (s.dtype == MOE_BF16 && fused_mlp(s)) {
    // one launch for both contractions: the stage boundary event falls before it
    if (mid_event && (e = record_event(mid_event, st)) != cudaSuccess) return e;
    return launch_mlp_fused_tc(s, x_perm, x, w.g, w.u, w.d, sched, h, y, at<int32_t>(ws, L.mlp_ready), status, st);
  }
  if (s.dtype == MOE_BF16) {
    if ((e = launch_gemm_gateup_tc(s, x_perm, x, w.g, w.u, sched, h, status, st)) != cudaSuccess) return e;
    if (mid_event && (e = record_event(mid_event, st)) != cudaSuccess) return e;
    return launch_gemm_down_tc(s, h, w.d, sched, y, status, st);
  }
  return launch_ffn_fma(s, x_perm, x, w.g, w.u, w.d, sched, h, y, st, mid_event, src_token);
}

// FP8 weights: bf16 layers whose shapes the FP8 kernels take, aligned codes and scales.
moe_status_t check_fp8_weights(const Shape& s, const uint8_t* wg_q, const float* wg_s, const uint8_t* wu_q,
                               const float* wu_s, const uint8_t* wd_q, const float* wd_s) {
  if (!wg_q || !wg_s || !wu_q || !wu_s || !wd_q || !wd_s) return MOE_ERR_INVALID_ARG;
  if (!aligned(wg_q, 16) || !aligned(wu_q, 16) || !aligned(wd_q, 16) || !aligned(wg_s, 4) || !aligned(wu_s, 4) ||
      !aligned(wd_s, 4))
    return MOE_ERR_INVALID_ARG;
  if (!fp8w_supported(s)) return MOE_ERR_UNSUPPORTED;
  return MOE_OK;
}

// Whether the whole-layer call runs the down projection with the combine in its epilogue
// (float32 reductions into an output accumulator, then one rounding pass) instead of writing
// the grouped expert outputs and combining them in a separate kernel. bf16 layers with bf16
// weights only; selected by MOE_FUSED_COMBINE=1 in the environment, read at every call. The
// order of the float32 additions then depends on scheduling, so the output is not
// bit-reproducible from run to run (the separate combine's is).
bool fused_combine(const Shape& s, const ExpertWeights& w) {
  if (s.dtype != MOE_BF16 || w.fp8) return false;
  const char* v = getenv("MOE_FUSED_COMBINE");
  return v != nullptr && v[0] == '1';
}

// Kernel launches one layer call enqueues; weights: 0 bf16 / float32, 1 FP8 codes with bf16
// activations, 2 W8A8. Memset nodes are not counted.
int layer_launches(const Shape& s, int weights) {
  // grouping: hist, scan (+ group schedule), scatter, row copy (W8A8: per-token quantiser and
  // code-row copy); one launch of all of it when the batch is a single chunk of tokens
  int grouping = s.nchunks == 1 ? 1 : 4;
  if (weights == 2 && s.nchunks != 1) grouping += 1;
  if (s.dtype == MOE_F32 && s.nchunks != 1) grouping -= 1;            // no grouped copy of x
  int mlp = 2;
  ExpertWeights w{nullptr, nullptr, nullptr};
  w.fp8 = weights != 0;
  if (weights == 2) mlp = fused_mlp_w8a8(s) ? 1 : 3;                 // + the quantiser of h
  else if (weights == 0 && s.dtype == MOE_BF16 && !fused_combine(s, w) && fused_mlp(s)) mlp = 1;
  const int combine = (mlp == 1 && weights == 0 && mlp_combine(s)) ? 0 : 1;   // in the one-launch MLP
  return 1 /*router*/ + grouping + mlp + combine;
}

moe_status_t layer_forward(const moe_config_t* cfg, const void* x, const void* w_router, const float* bias,
                           const ExpertWeights& w, void* out, int32_t* topk_idx_out, int32_t* counts_out, void* ws,
                           size_t ws_bytes, void* const* events, int n_events, cudaStream_t st) {
  moe_status_t rc = check_cfg(cfg);
  if (rc != MOE_OK) return rc;
  if (!x || !w_router || !w.g || !w.u || !w.d || !out) return MOE_ERR_INVALID_ARG;
  if (!aligned(x, 16) || !aligned(w_router, 16) || !aligned(w.g, 16) || !aligned(w.u, 16) ||
      !aligned(w.d, 16) || !aligned(out, 16) || (bias && !aligned(bias, 4)) ||
      (topk_idx_out && !aligned(topk_idx_out, 4)) || (counts_out && !aligned(counts_out, 4)))
    return MOE_ERR_INVALID_ARG;
  if (n_events < 0 || n_events > 6 || (n_events > 0 && events == nullptr)) return MOE_ERR_INVALID_ARG;
  const Shape s = make_shape(*cfg);
  if (w.fp8 && (rc = check_fp8_weights(s, static_cast<const uint8_t*>(w.g), w.gs, static_cast<const uint8_t*>(w.u),
                                       w.us, static_cast<const uint8_t*>(w.d), w.ds)) != MOE_OK)
    return rc;
  if (w.a8 && !w8a8_supported(s)) return MOE_ERR_UNSUPPORTED;
  if ((rc = check_ws(s, ws, ws_bytes)) != MOE_OK) return rc;
  const WsLayout L = make_layout(s);
  cudaEvent_t ev[6] = {nullptr, nullptr, nullptr, nullptr, nullptr, nullptr};
  for (int i = 0; i < n_events; ++i) ev[i] = static_cast<cudaEvent_t>(events[i]);

  int32_t* status = at<int32_t>(ws, L.status);
  int32_t* idx = topk_idx_out ? topk_idx_out : at<int32_t>(ws, L.topk_idx);
  float* gate = at<float>(ws, L.topk_gate);
  int32_t* counts = counts_out ? counts_out : at<int32_t>(ws, L.counts);
  int32_t* offsets = at<int32_t>(ws, L.offsets);
  int32_t* dest_row = at<int32_t>(ws, L.dest_row);
  int32_t* src_token = at<int32_t>(ws, L.src_token);
  void* x_perm = at<void>(ws, L.x_perm);
  void* y = at<void>(ws, L.y);

  auto mark = [&](int i) { return ev[i] == nullptr || record_event(ev[i], st) == cudaSuccess; };
  const NvtxRange layer_range("moe_layer");
  if (!mark(0)) return MOE_ERR_CUDA;
  {
    const NvtxRange r("moe_layer/router");
    if (run_router(s, x, w_router, bias, idx, gate, nullptr, status, st) != cudaSuccess) return MOE_ERR_CUDA;
  }
  if (!mark(1)) return MOE_ERR_CUDA;
  {
    const NvtxRange r("moe_layer/grouping");
    // W8A8: the grouped x rows go straight to E4M3 codes in the x_perm region
    uint8_t* x8 = w.a8 ? at<uint8_t>(ws, L.x_perm) : nullptr;
    float* x8s = w.a8 ? at<float>(ws, L.a8_scale) : nullptr;
    // float32 layers: the MLP reads the routed rows from x through src_token, no grouped copy
    const bool f32 = s.dtype == MOE_F32;
    if (run_permute(s, L, ws, idx, x, counts, offsets, dest_row, src_token, x_perm, true, st, x8, x8s, !f32) !=
        cudaSuccess)
      return MOE_ERR_CUDA;
  }
  if (!mark(2)) return MOE_ERR_CUDA;
  const bool fused = fused_combine(s, w);
  // the one-launch bf16 MLP with the combine in its down tiles
  const bool mlp_comb = !w.fp8 && !fused && s.dtype == MOE_BF16 && mlp_combine(s);
  float* acc = at<float>(ws, L.y);
  {
    const NvtxRange r("moe_layer/experts");
    if (w.a8) {
      // gate/up on the codes of the grouping stage, h -> codes, down on codes
      void* sched = at<void>(ws, L.sched);
      void* h = at<void>(ws, L.h);
      uint8_t* x8 = at<uint8_t>(ws, L.x_perm);
      float* x8s = at<float>(ws, L.a8_scale);
      uint8_t* h8 = at<uint8_t>(ws, L.h8);
      float* h8s = at<float>(ws, L.h8_scale);
      const int64_t n_sh = (int64_t)s.S * s.T;
      if (fused_mlp_w8a8(s)) {
        // both contractions and h's quantisation in one launch; the stage boundary event falls before it
        if (!mark(3)) return MOE_ERR_CUDA;
        if (launch_mlp_w8a8_fused(s, x8, x8s, static_cast<const uint8_t*>(w.g), w.gs, static_cast<const uint8_t*>(w.u),
                                  w.us, static_cast<const uint8_t*>(w.d), w.ds, sched, h, h8, h8s, y,
                                  at<int32_t>(ws, L.mlp_ready), status, st) != cudaSuccess)
          return MOE_ERR_CUDA;
      } else {
        if (launch_gemm_gateup_w8a8(s, x8, x8s, static_cast<const uint8_t*>(w.g), w.gs,
                                    static_cast<const uint8_t*>(w.u), w.us, sched, h, status, st) != cudaSuccess)
          return MOE_ERR_CUDA;
        if (!mark(3)) return MOE_ERR_CUDA;
        const void* h_shared = n_sh ? static_cast<const void*>(static_cast<const char*>(h) + (size_t)s.R * s.F * 2)
                                    : nullptr;
        if (launch_quantize_act_rows(s, h, offsets + s.E, s.R, h_shared, n_sh, s.F, h8, h8s, st) != cudaSuccess)
          return MOE_ERR_CUDA;
        if (launch_gemm_down_w8a8(s, h8, h8s, static_cast<const uint8_t*>(w.d), w.ds, sched, y, status, st) !=
            cudaSuccess)
          return MOE_ERR_CUDA;
      }
    } else if (fused) {
      void* sched = at<void>(ws, L.sched);
      void* h = at<void>(ws, L.h);
      if (launch_gemm_gateup_tc(s, x_perm, x, w.g, w.u, sched, h, status, st) != cudaSuccess) return MOE_ERR_CUDA;
      if (!mark(3)) return MOE_ERR_CUDA;
      if (cudaMemsetAsync(acc, 0, (size_t)s.T * s.d * sizeof(float), st) != cudaSuccess) return MOE_ERR_CUDA;
      if (launch_gemm_down_combine_tc(s, h, w.d, sched, src_token, dest_row, gate, acc, status, st) != cudaSuccess)
        return MOE_ERR_CUDA;
    } else if (mlp_comb) {
      // both contractions and the combine in one launch: the stage boundary events fall before it
      if (!mark(3)) return MOE_ERR_CUDA;
      if (launch_mlp_fused_tc(s, x_perm, x, w.g, w.u, w.d, at<void>(ws, L.sched), at<void>(ws, L.h), y,
                              at<int32_t>(ws, L.mlp_ready), status, st, src_token, dest_row, gate, out) != cudaSuccess)
        return MOE_ERR_CUDA;
    } else if (run_ffn(s, L, ws, x_perm, x, w, y, st, ev[3], s.dtype == MOE_F32 ? src_token : nullptr) !=
               cudaSuccess) {
      return MOE_ERR_CUDA;
    }
  }
  if (!mark(4)) return MOE_ERR_CUDA;
  if (!mlp_comb) {
    const NvtxRange r("moe_layer/combine");
    if (fused ? launch_combine_finalize(s, acc, out, st) != cudaSuccess
              : launch_combine(s, y, dest_row, gate, out, status, st) != cudaSuccess)
      return MOE_ERR_CUDA;
  }
  if (!mark(5)) return MOE_ERR_CUDA;
  return MOE_OK;
}

}  // namespace

extern "C" {

const char* moe_status_string(moe_status_t status) {
  switch (status) {
    case MOE_OK: return "MOE_OK";
    case MOE_ERR_INVALID_ARG: return "MOE_ERR_INVALID_ARG: invalid argument";
    case MOE_ERR_UNSUPPORTED: return "MOE_ERR_UNSUPPORTED: configuration outside what the kernels handle";
    case MOE_ERR_WORKSPACE: return "MOE_ERR_WORKSPACE: workspace too small";
    case MOE_ERR_CUDA: return "MOE_ERR_CUDA: CUDA runtime or launch failure";
    case MOE_ERR_TIMEOUT: return "MOE_ERR_TIMEOUT: a bounded wait inside a kernel ran out";
    case MOE_ERR_DEVICE_INDEX: return "MOE_ERR_DEVICE_INDEX: an out-of-range index or offset was skipped";
  }
  return "unknown moe_status_t";
}

moe_status_t moe_check_config(const moe_config_t* cfg) { return check_cfg(cfg); }

int32_t moe_capacity(const moe_config_t* cfg) {
  if (check_cfg(cfg) != MOE_OK) return -1;
  return make_shape(*cfg).cap;
}

int64_t moe_rows_capacity(const moe_config_t* cfg) {
  if (check_cfg(cfg) != MOE_OK) return -1;
  return make_shape(*cfg).R;
}

int64_t moe_grouped_rows(const moe_config_t* cfg) {
  if (check_cfg(cfg) != MOE_OK) return -1;
  const Shape s = make_shape(*cfg);
  return s.R + (int64_t)s.S * s.T;
}

size_t moe_workspace_size(const moe_config_t* cfg) {
  if (check_cfg(cfg) != MOE_OK) return 0;
  return make_layout(make_shape(*cfg)).total;
}

moe_status_t moe_workspace_init(void* ws, size_t ws_bytes, cudaStream_t stream) {
  if (ws == nullptr || !aligned(ws, 256) || ws_bytes < 256) return MOE_ERR_INVALID_ARG;
  return cuda_status(cudaMemsetAsync(ws, 0, 256, stream));
}

moe_status_t moe_clear_device_error(void* ws, cudaStream_t stream) {
  if (ws == nullptr || !aligned(ws, 256)) return MOE_ERR_INVALID_ARG;
  return cuda_status(cudaMemsetAsync(ws, 0, sizeof(int32_t), stream));
}

moe_status_t moe_get_device_error(const void* ws, cudaStream_t stream) {
  if (ws == nullptr || !aligned(ws, 256)) return MOE_ERR_INVALID_ARG;
  if (cudaStreamSynchronize(stream) != cudaSuccess) return MOE_ERR_CUDA;
  int32_t v = 0;
  if (cudaMemcpy(&v, ws, sizeof(v), cudaMemcpyDeviceToHost) != cudaSuccess) return MOE_ERR_CUDA;
  return static_cast<moe_status_t>(v);
}

moe_status_t moe_router_topk(const moe_config_t* cfg, const void* x, const void* w_router, const float* bias,
                             int32_t* topk_idx, float* topk_gate, float* scores, cudaStream_t stream) {
  moe_status_t rc = check_cfg(cfg);
  if (rc != MOE_OK) return rc;
  if (!x || !w_router || !topk_idx || !topk_gate) return MOE_ERR_INVALID_ARG;
  if (!aligned(x, 16) || !aligned(w_router, 16) || (bias && !aligned(bias, 4)) || !aligned(topk_idx, 4) ||
      !aligned(topk_gate, 4) || (scores && !aligned(scores, 4)))
    return MOE_ERR_INVALID_ARG;
  const Shape s = make_shape(*cfg);
  return cuda_status(run_router(s, x, w_router, bias, topk_idx, topk_gate, scores, nullptr, stream));
}

moe_status_t moe_permute(const moe_config_t* cfg, const int32_t* topk_idx, const void* x, int32_t* counts,
                         int32_t* offsets, int32_t* dest_row, int32_t* src_token, void* x_perm, void* ws,
                         size_t ws_bytes, cudaStream_t stream) {
  moe_status_t rc = check_cfg(cfg);
  if (rc != MOE_OK) return rc;
  if (!topk_idx || !x || !counts || !offsets || !dest_row || !src_token || !x_perm) return MOE_ERR_INVALID_ARG;
  if (!aligned(topk_idx, 4) || !aligned(x, 16) || !aligned(counts, 4) || !aligned(offsets, 4) ||
      !aligned(dest_row, 4) || !aligned(src_token, 4) || !aligned(x_perm, 16))
    return MOE_ERR_INVALID_ARG;
  const Shape s = make_shape(*cfg);
  if ((rc = check_ws(s, ws, ws_bytes)) != MOE_OK) return rc;
  return cuda_status(run_permute(s, make_layout(s), ws, topk_idx, x, counts, offsets, dest_row, src_token, x_perm,
                                 false, stream));
}

moe_status_t moe_grouped_ffn(const moe_config_t* cfg, const void* x_perm, const int32_t* offsets, const void* x,
                             const void* w_gate, const void* w_up, const void* w_down, void* y_perm, void* ws,
                             size_t ws_bytes, cudaStream_t stream) {
  moe_status_t rc = check_cfg(cfg);
  if (rc != MOE_OK) return rc;
  if (!x_perm || !offsets || !w_gate || !w_up || !w_down || !y_perm) return MOE_ERR_INVALID_ARG;
  if (cfg->n_shared > 0 && !x) return MOE_ERR_INVALID_ARG;
  if (!aligned(x_perm, 16) || !aligned(offsets, 4) || (x && !aligned(x, 16)) || !aligned(w_gate, 16) ||
      !aligned(w_up, 16) || !aligned(w_down, 16) || !aligned(y_perm, 16))
    return MOE_ERR_INVALID_ARG;
  const Shape s = make_shape(*cfg);
  if ((rc = check_ws(s, ws, ws_bytes)) != MOE_OK) return rc;
  const WsLayout L = make_layout(s);
  cudaError_t e = run_schedule(s, L, ws, offsets, stream);
  if (e != cudaSuccess) return MOE_ERR_CUDA;
  return cuda_status(run_ffn(s, L, ws, x_perm, x ? x : x_perm, ExpertWeights{w_gate, w_up, w_down}, y_perm, stream,
                             nullptr));
}

moe_status_t moe_combine(const moe_config_t* cfg, const void* y_perm, const int32_t* dest_row,
                         const float* topk_gate, void* out, void* ws, size_t ws_bytes, cudaStream_t stream) {
  moe_status_t rc = check_cfg(cfg);
  if (rc != MOE_OK) return rc;
  if (!y_perm || !dest_row || !topk_gate || !out) return MOE_ERR_INVALID_ARG;
  if (!aligned(y_perm, 16) || !aligned(dest_row, 4) || !aligned(topk_gate, 4) || !aligned(out, 16))
    return MOE_ERR_INVALID_ARG;
  const Shape s = make_shape(*cfg);
  if ((rc = check_ws(s, ws, ws_bytes)) != MOE_OK) return rc;
  return cuda_status(launch_combine(s, y_perm, dest_row, topk_gate, out, at<int32_t>(ws, make_layout(s).status),
                                    stream));
}

moe_status_t moe_layer_forward(const moe_config_t* cfg, const void* x, const void* w_router, const float* bias,
                               const void* w_gate, const void* w_up, const void* w_down, void* out,
                               int32_t* topk_idx_out, int32_t* counts_out, void* ws, size_t ws_bytes,
                               cudaStream_t stream) {
  return layer_forward(cfg, x, w_router, bias, ExpertWeights{w_gate, w_up, w_down}, out, topk_idx_out, counts_out,
                       ws, ws_bytes, nullptr, 0, stream);
}

moe_status_t moe_layer_forward_fp8(const moe_config_t* cfg, const void* x, const void* w_router, const float* bias,
                                   const uint8_t* wg_q, const float* wg_s, const uint8_t* wu_q, const float* wu_s,
                                   const uint8_t* wd_q, const float* wd_s, void* out, int32_t* topk_idx_out,
                                   int32_t* counts_out, void* ws, size_t ws_bytes, cudaStream_t stream) {
  return layer_forward(cfg, x, w_router, bias, ExpertWeights{wg_q, wu_q, wd_q, wg_s, wu_s, wd_s, true}, out,
                       topk_idx_out, counts_out, ws, ws_bytes, nullptr, 0, stream);
}

moe_status_t moe_layer_forward_fp8_timed(const moe_config_t* cfg, const void* x, const void* w_router,
                                         const float* bias, const uint8_t* wg_q, const float* wg_s,
                                         const uint8_t* wu_q, const float* wu_s, const uint8_t* wd_q,
                                         const float* wd_s, void* out, int32_t* topk_idx_out, int32_t* counts_out,
                                         void* ws, size_t ws_bytes, void* const* events, int32_t n_events,
                                         cudaStream_t stream) {
  return layer_forward(cfg, x, w_router, bias, ExpertWeights{wg_q, wu_q, wd_q, wg_s, wu_s, wd_s, true}, out,
                       topk_idx_out, counts_out, ws, ws_bytes, events, n_events, stream);
}

moe_status_t moe_layer_forward_w8a8(const moe_config_t* cfg, const void* x, const void* w_router, const float* bias,
                                    const uint8_t* wg_q, const float* wg_s, const uint8_t* wu_q, const float* wu_s,
                                    const uint8_t* wd_q, const float* wd_s, void* out, int32_t* topk_idx_out,
                                    int32_t* counts_out, void* ws, size_t ws_bytes, cudaStream_t stream) {
  return layer_forward(cfg, x, w_router, bias, ExpertWeights{wg_q, wu_q, wd_q, wg_s, wu_s, wd_s, true, true}, out,
                       topk_idx_out, counts_out, ws, ws_bytes, nullptr, 0, stream);
}

moe_status_t moe_layer_forward_w8a8_timed(const moe_config_t* cfg, const void* x, const void* w_router,
                                          const float* bias, const uint8_t* wg_q, const float* wg_s,
                                          const uint8_t* wu_q, const float* wu_s, const uint8_t* wd_q,
                                          const float* wd_s, void* out, int32_t* topk_idx_out, int32_t* counts_out,
                                          void* ws, size_t ws_bytes, void* const* events, int32_t n_events,
                                          cudaStream_t stream) {
  return layer_forward(cfg, x, w_router, bias, ExpertWeights{wg_q, wu_q, wd_q, wg_s, wu_s, wd_s, true, true}, out,
                       topk_idx_out, counts_out, ws, ws_bytes, events, n_events, stream);
}

moe_status_t moe_grouped_ffn_fp8(const moe_config_t* cfg, const void* x_perm, const int32_t* offsets, const void* x,
                                 const uint8_t* wg_q, const float* wg_s, const uint8_t* wu_q, const float* wu_s,
                                 const uint8_t* wd_q, const float* wd_s, void* y_perm, void* ws, size_t ws_bytes,
                                 cudaStream_t stream) {
  moe_status_t rc = check_cfg(cfg);
  if (rc != MOE_OK) return rc;
  if (!x_perm || !offsets || !y_perm) return MOE_ERR_INVALID_ARG;
  if (cfg->n_shared > 0 && !x) return MOE_ERR_INVALID_ARG;
  if (!aligned(x_perm, 16) || !aligned(offsets, 4) || (x && !aligned(x, 16)) || !aligned(y_perm, 16))
    return MOE_ERR_INVALID_ARG;
  const Shape s = make_shape(*cfg);
  if ((rc = check_fp8_weights(s, wg_q, wg_s, wu_q, wu_s, wd_q, wd_s)) != MOE_OK) return rc;
  if ((rc = check_ws(s, ws, ws_bytes)) != MOE_OK) return rc;
  const WsLayout L = make_layout(s);
  if (run_schedule(s, L, ws, offsets, stream) != cudaSuccess) return MOE_ERR_CUDA;
  return cuda_status(run_ffn(s, L, ws, x_perm, x ? x : x_perm,
                             ExpertWeights{wg_q, wu_q, wd_q, wg_s, wu_s, wd_s, true}, y_perm, stream, nullptr));
}

moe_status_t moe_quantize_fp8_rows(const void* w, int64_t rows, int32_t cols, uint8_t* wq, float* scale,
                                   cudaStream_t stream) {
  if (!w || !wq || !scale || rows < 1 || cols < 16 || cols % 16 != 0) return MOE_ERR_INVALID_ARG;
  if (!aligned(w, 16) || !aligned(wq, 16) || !aligned(scale, 4)) return MOE_ERR_INVALID_ARG;
  return cuda_status(launch_quantize_fp8_rows(w, rows, cols, wq, scale, stream));
}

moe_status_t moe_layer_forward_timed(const moe_config_t* cfg, const void* x, const void* w_router,
                                     const float* bias, const void* w_gate, const void* w_up, const void* w_down,
                                     void* out, int32_t* topk_idx_out, int32_t* counts_out, void* ws,
                                     size_t ws_bytes, void* const* events, int32_t n_events, cudaStream_t stream) {
  return layer_forward(cfg, x, w_router, bias, ExpertWeights{w_gate, w_up, w_down}, out, topk_idx_out, counts_out,
                       ws, ws_bytes, events, n_events, stream);
}

int32_t moe_layer_launch_count(const moe_config_t* cfg) {
  if (check_cfg(cfg) != MOE_OK) return -1;
  return layer_launches(make_shape(*cfg), 0);
}

int32_t moe_layer_launch_count_weights(const moe_config_t* cfg, int32_t weights) {
  if (check_cfg(cfg) != MOE_OK || weights < 0 || weights > 2) return -1;
  const Shape s = make_shape(*cfg);
  if (weights != 0 && !fp8w_supported(s)) return -1;
  return layer_launches(s, weights);
}

int32_t moe_layer_mlp_fused(const moe_config_t* cfg) {
  if (check_cfg(cfg) != MOE_OK) return -1;
  const Shape s = make_shape(*cfg);
  return (s.dtype == MOE_BF16 && fused_mlp(s)) ? 1 : 0;
}

int32_t moe_layer_mlp_fused_weights(const moe_config_t* cfg, int32_t weights) {
  if (check_cfg(cfg) != MOE_OK || weights < 0 || weights > 2) return -1;
  const Shape s = make_shape(*cfg);
  if (weights != 0 && !fp8w_supported(s)) return -1;
  if (weights == 1 || s.dtype != MOE_BF16) return 0;
  return (weights == 2 ? fused_mlp_w8a8(s) : fused_mlp(s)) ? 1 : 0;
}

moe_status_t moe_selftest_bounded_wait(void* ws, size_t ws_bytes, uint64_t limit_ns, cudaStream_t stream) {
  if (ws == nullptr || !aligned(ws, 256) || ws_bytes < 256) return MOE_ERR_INVALID_ARG;
  if (limit_ns > 10000000000ull) return MOE_ERR_INVALID_ARG;
  return cuda_status(launch_wait_selftest(static_cast<int32_t*>(ws), limit_ns, stream));
}

}  // extern "C"
