/*
 * moe.h -- C ABI of the B300 (sm_103a) Mixture-of-Experts FFN layer forward.
 *
 * One MoE layer, one GPU: router logits -> softmax or sigmoid scores -> top-k
 * with renormalised gates -> grouping of tokens by destination expert
 * (histogram, prefix sum, scatter; dropless or capacity-limited) -> grouped
 * SwiGLU expert MLPs (plus an optional always-on shared expert) -> gate-weighted
 * combine back in token order. Every stage is a CUDA kernel of libmoe.so.
 *
 * Source pages the operations follow (cited by these short names below):
 *   [ST] shubhamtatvamasi.com/llm-inference/moe, "Mixture of Experts"
 *   [KG] klaylearn.com/glossary/mixture-of-experts, "Mixture of Experts"
 *   [TB] techbonafide.com, "Mixture of Experts (MoE) explained"
 *   [SA] shipai.vats.cc/learn/advanced-concepts/mixture-of-experts, "Mixture of Experts (MoE)"
 *
 * Conventions shared by every call:
 *   - All tensors are row-major and contiguous. Pointers marked "device" are
 *     device memory the CALLER allocated and owns; the library never allocates,
 *     frees or synchronises (except moe_get_device_error, which synchronises
 *     the stream it is given).
 *   - Device pointers to activations and weights must be 16-byte aligned; the
 *     workspace must be 256-byte aligned.
 *   - Element type of x, weights, x_perm, y_perm and out is cfg->dtype
 *     (MOE_BF16 or MOE_F32); router scores, gates and the bias are float32;
 *     indices are int32. bf16 paths accumulate in float32.
 *   - Calls are asynchronous on `stream`. Arguments are validated on the host
 *     first; a bad argument returns an error before anything is enqueued.
 *     A failed launch returns MOE_ERR_CUDA. Problems found on the device
 *     (an expert index out of range, offsets that are not a valid grouping, a
 *     bounded wait that ran out) are recorded in the workspace status word
 *     and read with moe_get_device_error. Nothing aborts or traps.
 *   - G = n_experts + n_shared groups. Weight tensors hold the routed experts
 *     first and the shared expert (if any) last:
 *       w_gate, w_up : [G, d_ff, d_model]     w_down : [G, d_model, d_ff]
 *   - R = moe_rows_capacity(cfg) = min(T*k, E*cap) rows hold the kept
 *     (token, expert) pairs grouped by expert; the shared expert's T rows
 *     follow at rows R .. R+T-1 of the grouped outputs.
 *
 * Environment switches (each selects among kernel paths that compute the same layer; the
 * defaults are the paths measured fastest on a B300):
 *   MOE_FUSED_MLP=0|1    the bf16 expert MLP as one persistent launch of both contractions
 *                        (default: batches of at most 128 tokens) or two launches; for W8A8
 *                        layers, =1 selects the one-launch kernel (default: three launches).
 *                        Same bits either way. Read at every call.
 *   MOE_MLP_COMBINE=1    with the one-launch bf16 MLP, the combine in its down tiles (per-token
 *                        counts, the last arrival sums the rows in slot order: the separate
 *                        combine's bits) instead of a combine launch. Default off. Every call.
 *   MOE_FUSED_COMBINE=1  bf16 layers: the down projection adds its rows into a float32 output
 *                        accumulator (red.global.add), then one rounding pass, instead of the
 *                        combine kernel; the order of the float32 additions depends on
 *                        scheduling, so the output is not bit-reproducible. Default off. Every call.
 *   MOE_GEMM_PAIRS=1     the bf16 grouped GEMMs as 2-SM (cta_group::2) pair kernels with 256-row
 *                        tiles. Default off. Read once per process.
 */
#ifndef MOE_H
#define MOE_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = 1,   /* null or misaligned pointer, non-positive size, k > E, ... */
  MOE_ERR_UNSUPPORTED = 2,   /* valid but outside what the kernels handle (see moe_config_t) */
  MOE_ERR_WORKSPACE = 3,     /* ws_bytes < moe_workspace_size(cfg) */
  MOE_ERR_CUDA = 4,          /* a CUDA runtime call or kernel launch failed */
  MOE_ERR_TIMEOUT = 5,       /* device: a bounded wait inside a kernel ran out */
  MOE_ERR_DEVICE_INDEX = 6   /* device: an index or offset out of range was seen and skipped */
} moe_status_t;

typedef enum { MOE_F32 = 0, MOE_BF16 = 1 } moe_dtype_t;
typedef enum { MOE_SOFTMAX = 0, MOE_SIGMOID = 1 } moe_score_t;

/*
 * Layer shape and policy.
 *   T               tokens in the batch (1 .. 1048576; an empty batch is MOE_ERR_INVALID_ARG: there
 *                   is nothing to enqueue, so a caller skips the call)
 *   d_model         hidden size d;   bf16: multiple of 128;  f32: multiple of 4
 *   n_experts       routed experts E (1 .. 256)
 *   top_k           experts per token k (1 .. min(E, 8))
 *   d_ff            expert hidden size F;  bf16: multiple of 128;  f32: multiple of 4
 *   n_shared        always-on shared experts S (0 or 1), same d_ff as the routed ones [ST "The router"]
 *   score           MOE_SOFTMAX over all E logits, or MOE_SIGMOID per expert [ST "The router"]
 *   renormalize     1: gates = selected scores / their sum [ST "The router"]; 0: gates = raw scores
 *   capacity_factor <= 0: dropless; > 0: each expert keeps at most
 *                   cap = ceil(capacity_factor * T * k / E) tokens, evaluated exactly on this binary32
 *                   value, admitting tokens in ascending token index; the overflow pairs contribute
 *                   nothing: the token misses that expert and only goes on through the residual
 *                   connection [ST "Load imbalance"]
 *   dtype           MOE_BF16 or MOE_F32 (activations and weights)
 */
typedef struct moe_config {
  int32_t T;
  int32_t d_model;
  int32_t n_experts;
  int32_t top_k;
  int32_t d_ff;
  int32_t n_shared;
  int32_t score;          /* moe_score_t */
  int32_t renormalize;
  float capacity_factor;
  int32_t dtype;          /* moe_dtype_t */
} moe_config_t;

/* Human-readable name of a status code (static string, never NULL). */
const char* moe_status_string(moe_status_t status);

/* Host-side validation of a configuration: MOE_OK, MOE_ERR_INVALID_ARG or MOE_ERR_UNSUPPORTED. */
moe_status_t moe_check_config(const moe_config_t* cfg);

/* Per-expert capacity cap (T when dropless); -1 for an invalid configuration. */
int32_t moe_capacity(const moe_config_t* cfg);

/* R = min(T*k, E*cap): rows of x_perm and src_token. -1 for an invalid configuration. */
int64_t moe_rows_capacity(const moe_config_t* cfg);

/* R + S*T: rows of y_perm (the shared expert's rows follow the routed ones). -1 if invalid. */
int64_t moe_grouped_rows(const moe_config_t* cfg);

/* Bytes of device workspace every call below needs (0 for an invalid configuration). */
size_t moe_workspace_size(const moe_config_t* cfg);

/* Zero the workspace status word (asynchronous). Call once after allocating a workspace. */
moe_status_t moe_workspace_init(void* ws, size_t ws_bytes, cudaStream_t stream);

/*
 * Router: logits = x W_r^T (+ bias), scores, top-k, gates.
 * [ST "The router" and Q&A "How does a top-k router work?"; SA "How routing works (intuition)"]
 *   x         device [T, d_model]             w_router device [E, d_model]
 *   bias      device [E] float32 or NULL; added to the logits before the score function
 *   topk_idx  device [T, k] int32 out: expert ids in rank order (highest score first, equal
 *             scores to the lower id); always k distinct ids in [0, E)
 *   topk_gate device [T, k] float32 out: gates (sum to one when renormalize)
 *   scores    device [T, E] float32 out, or NULL: the full softmax / sigmoid scores
 */
moe_status_t moe_router_topk(const moe_config_t* cfg, const void* x, const void* w_router,
                             const float* bias, int32_t* topk_idx, float* topk_gate, float* scores,
                             cudaStream_t stream);

/*
 * Grouping by destination expert [KG "Mixture of Experts" definition: permute tokens by
 * destination expert; ST "Load imbalance": capacity limit or dropless].
 *   topk_idx  device [T, k] int32 in (ids outside [0, E) are skipped and flagged)
 *   x         device [T, d_model] in
 *   counts    device [E] int32 out: pairs routed to each expert, before capacity
 *   offsets   device [E+1] int32 out: exclusive scan of the kept counts; offsets[E] = P' kept pairs
 *   dest_row  device [T, k] int32 out: row of pair (t, j) in x_perm, or -1 when dropped
 *   src_token device [R] int32 out: token of each grouped row (rows >= P' untouched)
 *   x_perm    device [R, d_model] out: x[src_token[r]] for r < P' (rows >= P' untouched)
 * Rows of one expert are in ascending token order, so the result is deterministic.
 */
moe_status_t moe_permute(const moe_config_t* cfg, const int32_t* topk_idx, const void* x,
                         int32_t* counts, int32_t* offsets, int32_t* dest_row, int32_t* src_token,
                         void* x_perm, void* ws, size_t ws_bytes, cudaStream_t stream);

/*
 * moe_permute for callers that cannot allocate device memory: code that enqueues work while
 * a stream is being captured into a CUDA graph, a plug-in whose host framework owns all
 * device memory and passes in only the call's tensors, a real-time loop that must not touch
 * the allocator. The source pages have no counterpart; this is an interface of this library.
 *   Same arguments and results as moe_permute, without ws / ws_bytes, plus
 *   status  device int32 or NULL: a device-side problem (an id outside [0, E), or an expert
 *           repeated within a token) is recorded here with an atomic compare-and-swap from 0,
 *           so zero it before the call. With status == NULL such problems go unreported: the
 *           pair is still skipped (dest_row = -1) but nothing records that it happened.
 * Batches of at most 128 tokens are grouped in the shared memory of each block of one launch
 * (which also copies the rows) and touch no shared state. Larger batches keep the per-chunk expert histogram in a fixed 256 KiB array in
 * libmoe.so's own device memory, held by every GPU that loads the library until the process
 * exits. It fits ceil(T/128) * E <= 65536 (T <= 32768 at E = 256); larger configurations
 * return MOE_ERR_WORKSPACE before anything is enqueued. Nothing is allocated or freed. The
 * first such call in a CUDA context looks up the array's device address (again after a
 * cudaDeviceReset or under another context): make it before any stream capture. All these
 * calls share the array and leave their contents in it; calls that overlap on the GPU
 * (unordered streams) race and give wrong results.
 */
moe_status_t moe_permute_noalloc(const moe_config_t* cfg, const int32_t* topk_idx, const void* x,
                                 int32_t* counts, int32_t* offsets, int32_t* dest_row,
                                 int32_t* src_token, void* x_perm, int32_t* status,
                                 cudaStream_t stream);

/*
 * Grouped expert MLPs [KG definition: one grouped GEMM pass over every expert's batch of rows;
 * TB "Experts as Specialized Subnetworks"]: for every routed expert e and kept row r in
 * [offsets[e], offsets[e+1]) and, for the shared expert, every token t:
 *     y = W_down (silu(W_gate a) * (W_up a)),  silu(z) = z * sigmoid(z)
 * with a = x_perm[r] (routed) or x[t] (shared). bf16: the intermediate silu(.)*(.) is
 * rounded to bf16 once before the down projection, y is rounded to bf16 from the
 * float32 accumulator.
 *   x_perm  device [R, d_model] in        offsets device [E+1] int32 in (validated on the device)
 *   x       device [T, d_model] in (read only when n_shared > 0; may be NULL otherwise)
 *   w_gate, w_up device [G, d_ff, d_model]; w_down device [G, d_model, d_ff]
 *   y_perm  device [R + S*T, d_model] out: routed rows r < P', then the shared rows R + t
 */
moe_status_t moe_grouped_ffn(const moe_config_t* cfg, const void* x_perm, const int32_t* offsets,
                             const void* x, const void* w_gate, const void* w_up, const void* w_down,
                             void* y_perm, void* ws, size_t ws_bytes, cudaStream_t stream);

/*
 * FP8 expert weights [ST "Memory vs compute, quantified": the 671B model's weights are about
 * 671 GB in FP8 instead of 1.3 TB in BF16; small-batch decode streams the touched experts'
 * weights, so their bytes set the step time]. A weight matrix is stored as E4M3 codes with one
 * float32 scale per output row:  W[r][c] = scale[r] * e4m3(wq[r][c]).  For w_gate / w_up the
 * rows are the d_ff outputs of each group ([G, d_ff, d_model] codes, [G, d_ff] scales); for
 * w_down the d_model outputs ([G, d_model, d_ff] codes, [G, d_model] scales). Activations stay
 * bf16; the kernels widen the codes to bf16 (exactly) in shared memory and apply the scales to
 * the float32 accumulators, so a layer with FP8 weights computes exactly what the bf16 layer
 * computes with the dequantized weights.
 *
 * Quantisation of a bf16 matrix [rows, cols] (cols a multiple of 16):
 *   scale[r] = max_c |w[r][c]| / 448 (float32; 0 for an all-zero row)
 *   wq[r][c] = E4M3 code of float32(w[r][c]) / scale[r], rounded to nearest even and saturated
 *              to +-448 (0 when scale[r] = 0)
 *   w   device [rows, cols] bf16 in;  wq device [rows, cols] uint8 out;  scale device [rows] float32 out
 */
moe_status_t moe_quantize_fp8_rows(const void* w, int64_t rows, int32_t cols, uint8_t* wq, float* scale,
                                   cudaStream_t stream);

/*
 * moe_grouped_ffn with FP8 expert weights: the same rows and outputs as moe_grouped_ffn for the
 * dequantized weights. bf16 layers with d_model a multiple of 256 only; MOE_ERR_UNSUPPORTED
 * otherwise (float32 activations, or d_model = 128 mod 256).
 *   wg_q, wu_q  device [G, d_ff, d_model] uint8     wg_s, wu_s device [G, d_ff] float32
 *   wd_q        device [G, d_model, d_ff] uint8     wd_s       device [G, d_model] float32
 */
moe_status_t moe_grouped_ffn_fp8(const moe_config_t* cfg, const void* x_perm, const int32_t* offsets,
                                 const void* x, const uint8_t* wg_q, const float* wg_s, const uint8_t* wu_q,
                                 const float* wu_s, const uint8_t* wd_q, const float* wd_s, void* y_perm,
                                 void* ws, size_t ws_bytes, cudaStream_t stream);

/*
 * Combine [ST Q&A "How does a top-k router work?": gate-weighted sum of the selected experts;
 * ST "The router": shared experts every token visits; KG definition: undo the permutation]:
 *     out[t] = sum_{j: dest_row[t,j] >= 0} gate[t,j] * y_perm[dest_row[t,j]]  (+ y_perm[R + t] if S = 1)
 * accumulated in float32 in slot order, shared part last. No residual add.
 *   y_perm device [R + S*T, d_model] in; dest_row device [T, k] int32; topk_gate device [T, k] float32
 *   out    device [T, d_model] out
 *   ws, ws_bytes  the workspace (moe_workspace_size bytes, 256-byte aligned): only its status
 *          word is used, to record a dest_row entry at or past R (the entry is then skipped).
 * The per-expert offsets of the grouping are not an argument: dest_row already names each
 * pair's grouped row (or -1), and the shared expert's rows follow the R routed rows.
 */
moe_status_t moe_combine(const moe_config_t* cfg, const void* y_perm, const int32_t* dest_row,
                         const float* topk_gate, void* out, void* ws, size_t ws_bytes,
                         cudaStream_t stream);

/*
 * The whole layer: router -> permute -> grouped MLPs -> combine, enqueued on `stream`
 * with no host synchronisation (capturable in a CUDA graph). A float32 layer's expert MLP
 * reads the routed rows from x through src_token, so its permute writes no x_perm copy (the
 * same values as the stage calls).
 *   out            device [T, d_model] out: the MoE FFN output (no residual add)
 *   topk_idx_out   device [T, k] int32 out or NULL (routing is then kept in the workspace)
 *   counts_out     device [E] int32 out or NULL (per-expert load before capacity)
 */
moe_status_t moe_layer_forward(const moe_config_t* cfg, const void* x, const void* w_router,
                               const float* bias, const void* w_gate, const void* w_up,
                               const void* w_down, void* out, int32_t* topk_idx_out,
                               int32_t* counts_out, void* ws, size_t ws_bytes, cudaStream_t stream);

/*
 * moe_layer_forward that also records CUDA events between its stages, for timing:
 * events[0] before the router, [1] after the router, [2] after the grouping (histogram,
 * scan, scatter, row gather, group schedule), [3] after the gate/up GEMM, [4] after the down GEMM,
 * [5] after the combine. `events` holds n_events cudaEvent_t handles (n_events <= 6;
 * the first n_events boundaries are recorded).
 */
moe_status_t moe_layer_forward_timed(const moe_config_t* cfg, const void* x, const void* w_router,
                                     const float* bias, const void* w_gate, const void* w_up,
                                     const void* w_down, void* out, int32_t* topk_idx_out,
                                     int32_t* counts_out, void* ws, size_t ws_bytes,
                                     void* const* events, int32_t n_events, cudaStream_t stream);

/*
 * Routing telemetry of one batch [ST "Load imbalance": per-expert load, drops under a capacity
 * limit, and for dropless serving the share of expert compute that is useful while every
 * expert waits for the busiest one; ST "Memory vs compute, quantified": experts touched].
 * Computed on the device from the per-expert counts of moe_permute / moe_layer_forward, so it
 * needs no host synchronisation.
 *   counts  device [E] int32 in: pairs routed to each expert before capacity
 *   stats   device moe_routing_stats_t out
 * kept[e] = min(counts[e], cap); mean_load = sum(kept) / E (float32); efficiency = mean_load /
 * max_load (1 when no pair is kept). Negative counts are treated as 0 and flagged nowhere.
 */
typedef struct moe_routing_stats {
  int32_t tokens;           /* T */
  int32_t pairs;            /* sum of counts: routed (token, expert) pairs, T*k for valid routing */
  int32_t kept;             /* sum of kept[e] */
  int32_t dropped;          /* pairs - kept */
  int32_t experts_touched;  /* experts with kept[e] > 0 */
  int32_t max_load;         /* max over e of kept[e] */
  int32_t capacity;         /* per-expert cap (T when dropless) */
  float mean_load;          /* kept / E */
  float efficiency;         /* mean_load / max_load */
} moe_routing_stats_t;

moe_status_t moe_routing_stats(const moe_config_t* cfg, const int32_t* counts, moe_routing_stats_t* stats,
                               cudaStream_t stream);

/*
 * moe_layer_forward and moe_layer_forward_timed with FP8 expert weights (bf16 layers only; the
 * weight arguments as for moe_grouped_ffn_fp8).
 */
moe_status_t moe_layer_forward_fp8(const moe_config_t* cfg, const void* x, const void* w_router,
                                   const float* bias, const uint8_t* wg_q, const float* wg_s,
                                   const uint8_t* wu_q, const float* wu_s, const uint8_t* wd_q,
                                   const float* wd_s, void* out, int32_t* topk_idx_out, int32_t* counts_out,
                                   void* ws, size_t ws_bytes, cudaStream_t stream);
moe_status_t moe_layer_forward_fp8_timed(const moe_config_t* cfg, const void* x, const void* w_router,
                                         const float* bias, const uint8_t* wg_q, const float* wg_s,
                                         const uint8_t* wu_q, const float* wu_s, const uint8_t* wd_q,
                                         const float* wd_s, void* out, int32_t* topk_idx_out,
                                         int32_t* counts_out, void* ws, size_t ws_bytes,
                                         void* const* events, int32_t n_events, cudaStream_t stream);

/*
 * The layer with FP8 (E4M3) expert weights AND E4M3 activations (W8A8). The source pages put
 * the model's weights in FP8 (shubhamtatvamasi.com "Mixture of Experts", "Memory vs compute,
 * quantified"); quantising the activations as well is this library's reading beyond them: the
 * rows entering each expert contraction -- the grouped x rows before gate/up, and
 * h = silu(g) * u (stored in bf16) before down -- are quantised per row exactly as the weights
 * are (one float32 scale = max|row| / 448 per row, codes rounded to nearest even, saturated),
 * and the contractions run on the 8-bit tensor-core path (tcgen05.mma kind::f8f6f4) with
 * float32 accumulation; the row scales of both operands are applied to the accumulator. The
 * results therefore differ from moe_layer_forward_fp8's by the activations' quantisation error
 * (at most 2^-4 of an element). Arguments, layouts and errors as for moe_layer_forward_fp8;
 * bf16 layers with d_model a multiple of 256 only (MOE_ERR_UNSUPPORTED otherwise). The
 * grouping stage writes the grouped x rows as codes (no bf16 copy); one more kernel than
 * moe_layer_forward enqueues (the quantiser of h).
 */
moe_status_t moe_layer_forward_w8a8(const moe_config_t* cfg, const void* x, const void* w_router,
                                    const float* bias, const uint8_t* wg_q, const float* wg_s,
                                    const uint8_t* wu_q, const float* wu_s, const uint8_t* wd_q,
                                    const float* wd_s, void* out, int32_t* topk_idx_out, int32_t* counts_out,
                                    void* ws, size_t ws_bytes, cudaStream_t stream);
moe_status_t moe_layer_forward_w8a8_timed(const moe_config_t* cfg, const void* x, const void* w_router,
                                          const float* bias, const uint8_t* wg_q, const float* wg_s,
                                          const uint8_t* wu_q, const float* wu_s, const uint8_t* wd_q,
                                          const float* wd_s, void* out, int32_t* topk_idx_out,
                                          int32_t* counts_out, void* ws, size_t ws_bytes,
                                          void* const* events, int32_t n_events, cudaStream_t stream);

/* Number of kernel launches one moe_layer_forward call (bf16 or float32 weights) enqueues for this
 * configuration (-1 if invalid). Memset nodes are not counted. */
int32_t moe_layer_launch_count(const moe_config_t* cfg);

/* The same for the layer call with the given weights: 0 bf16 / float32 (moe_layer_forward),
 * 1 FP8 codes with bf16 activations (moe_layer_forward_fp8), 2 W8A8 (moe_layer_forward_w8a8);
 * -1 if the configuration is invalid or the FP8 kernels do not take it. */
int32_t moe_layer_launch_count_weights(const moe_config_t* cfg, int32_t weights);

/*
 * 1 if moe_layer_forward and moe_layer_forward_w8a8 run the expert MLP's two contractions
 * (gate/up + SwiGLU, then down; in W8A8 with h's quantisation between them) as one persistent
 * launch for this configuration, 0 if as separate launches, -1 if the configuration is invalid.
 * One launch is the default for bf16 layers whose batch is a single chunk of at most 128 tokens
 * (decode): each CTA takes its gate/up tiles, then its down tiles, and a down tile waits
 * (bounded) until every gate/up tile of its 128-row block has published its rows of h through a
 * counter in the workspace (in W8A8 the tile that completes a block quantises its rows first).
 * The results are bit-identical to the separate launches.
 * MOE_FUSED_MLP=1 or 0 in the environment forces one or two launches for every bf16 layer
 * whose d_model is a multiple of 256 (read at every call). The one launch needs all of its
 * CTAs (one per SM) resident at once: a GPU shared with other work that holds SMs for long can
 * make its waits run out (MOE_ERR_TIMEOUT in the status word) instead of hanging.
 */
int32_t moe_layer_mlp_fused(const moe_config_t* cfg);

/*
 * moe_layer_mlp_fused per weight format (`weights` as in moe_layer_launch_count_weights): 1 if
 * the expert MLP runs as one launch, 0 if not, -1 for an invalid config or a format the shape
 * does not take. FP8 weights with bf16 activations: always two launches. W8A8: one launch (the
 * tile that completes an m-tile's gate/up quantises its h rows, then its down tiles start) only
 * with MOE_FUSED_MLP=1, since it measured slower than gate/up, quantiser and down as three
 * launches.
 */
int32_t moe_layer_mlp_fused_weights(const moe_config_t* cfg, int32_t weights);

/*
 * Synchronise `stream`, then return the first device-side status recorded in the workspace
 * since the last moe_workspace_init / moe_clear_device_error (MOE_OK if none).
 */
moe_status_t moe_get_device_error(const void* ws, cudaStream_t stream);

/* Reset the workspace status word to MOE_OK (asynchronous). */
moe_status_t moe_clear_device_error(void* ws, cudaStream_t stream);

/*
 * Self-test of the bounded wait used by the pipelined kernels: one CTA waits on an
 * mbarrier that nothing completes, gives up after about `limit_ns` nanoseconds, records
 * MOE_ERR_TIMEOUT in the workspace status word and returns normally. Lets a caller check,
 * without hanging the GPU, that a stalled pipeline surfaces as a status.
 */
moe_status_t moe_selftest_bounded_wait(void* ws, size_t ws_bytes, uint64_t limit_ns,
                                       cudaStream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* MOE_H */
