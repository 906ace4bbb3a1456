// Router on the 5th-generation tensor cores (bf16 layers): logits = x W_r^T
// (+ b) accumulated in tensor memory, then score function, top-k and gate
// renormalisation fused into the same kernel.
//
// Follows shubhamtatvamasi.com/llm-inference/moe "Mixture of Experts", section
// "The router" (one small linear layer scores every expert; softmax, or the
// sigmoid variant; keep the top-k; renormalise the chosen gates to sum to one)
// and its Q&A "How does a top-k router work?"; klaylearn.com's glossary names
// this "fused routing" as one of the kernels an MoE layer needs.
//
// Work split. A tile is 128 tokens x all E experts: one tcgen05 accumulator of
// 128 TMEM lanes (one per token) x N columns, N = E rounded up to a multiple
// of 16 (the tcgen05 M=128 shape; columns past E come from W_r rows the TMA
// load zero-fills). The reduction over d_model is split across the C CTAs of
// a thread-block cluster (C = 1, 2, 4 or 8, chosen so that tiles x C fills
// about one wave of the GPU): each CTA accumulates d_model / C of the sum,
// copies its partial accumulator to its own shared memory, and after a
// cluster barrier CTA c adds the C partials of rows [c*128/C, (c+1)*128/C) in
// rank order through distributed shared memory (a fixed order, so the result
// is deterministic) and selects the top-k of those rows.
//
// Roles inside a CTA (576 threads):
//   warp 0      TMA producer: x tile 128 x 64 and W_r tile N x 64 per k-step
//   warp 1      TMEM allocation and the tcgen05.mma issuer (M=128, N, K=16)
//   warps 2-17  epilogue: TMEM -> shared copy (four warps per 32-lane TMEM
//               quarter, 32-column slices), then selection with P = 512 / rows
//               threads per token: thread p of a token scans experts p, p+P,
//               ... keeping a sorted partial top-k in registers, and the P
//               lists are merged by a butterfly of bitonic merges (shuffles)
// The products of two bf16 values are exact in float32; the tensor core adds
// them in float32.
//
// Selection is done on the logits (plus bias). Softmax and the sigmoid are
// monotone, so this is the order of the exact scores; a float32 score could
// tie where the logits differ. Equal logits go to the lower expert id, NaN
// logits rank below every number, and the k ids are always distinct.
// Gates: softmax with renormalisation is exp(l_j - l_1) / sum over the chosen
// of exp(l_i - l_1), l_1 the top logit (the full softmax denominator cancels,
// so it is not computed); without renormalisation the full softmax score,
// whose denominator sum_e exp(l_e - l_1) takes one more pass; sigmoid gates
// are sigma(l_j), divided by their sum when renormalising.
//
// Every wait is bounded. A stall records MOE_ERR_TIMEOUT in the status word
// (when the caller gave one) and the tokens of the cluster get expert id -1,
// which the grouping stage skips and reports. Every CTA passes both cluster
// barriers on every path, and the TMEM is freed on every path.
#include <cfloat>
#include <mutex>

#include "internal.cuh"
#include "tc_ptx.cuh"
#include "tmap.cuh"

namespace moe {
namespace {

constexpr int kBM = 128;
constexpr int kBK = 64;
constexpr int kEpiWarps = 16;
constexpr int kEpiThreads = 32 * kEpiWarps;             // 512
constexpr int kThreads = 64 + kEpiThreads;              // producer warp, MMA warp, epilogue
constexpr uint32_t kABytes = kBM * kBK * 2;             // 16 KB
constexpr size_t kSmemBudget = 200 * 1024;
constexpr int kMaxCluster = 8;
constexpr uint64_t kWaitLimitNs = 4000000000ull;
constexpr uint64_t kDrainLimitNs = 100000000ull;
constexpr int kNoExpert = 0x7fffffff;

struct RouterArgs {
  int T, E, N, k, k_steps, stages, score, renorm;
  int csplit;             // CTAs per cluster splitting d_model
  int sel_p;              // selection threads per token (a power of two, >= 32 / rows)
  int np;                 // floats per row of the shared partial / logit buffer (N + 4)
  uint32_t tmem_cols;
  size_t region;          // bytes of the stage / partial region
  const float* bias;
  int32_t* idx;
  float* gate;
  float* scores;
  int32_t* status;
};

__device__ __forceinline__ bool ranks_before(float a, int ea, float b, int eb) {
  return a > b || (a == b && ea < eb);
}

__device__ __forceinline__ float sigmoid_f(float z) { return 1.0f / (1.0f + expf(-z)); }

// Insert (key, e) into the sorted list v/id (best first). A thread offers its
// experts in ascending id, so an equal key goes after the ones already there
// (lower id first) and is dropped when the list is full of keys >= it.
// Branch-free shift: every slot is computed from the old list at once.
template <int KS>
__device__ __forceinline__ void topk_insert(float key, int e, float (&v)[KS], int (&id)[KS]) {
  bool gt[KS];
#pragma unroll
  for (int j = 0; j < KS; ++j) gt[j] = key > v[j];
#pragma unroll
  for (int j = KS - 1; j >= 0; --j) {
    const bool above = (j > 0) && gt[j > 0 ? j - 1 : 0];
    const float vp = v[j > 0 ? j - 1 : 0];
    const int ip = id[j > 0 ? j - 1 : 0];
    v[j] = above ? vp : (gt[j] ? key : v[j]);
    id[j] = above ? ip : (gt[j] ? e : id[j]);
  }
}

// Compare-exchange (selects, no branch): the better of slots i and j ends in i.
template <int KS>
__device__ __forceinline__ void cas_desc(float (&v)[KS], int (&id)[KS], int i, int j) {
  const bool sw = ranks_before(v[j], id[j], v[i], id[i]);
  const float vi = v[i], vj = v[j];
  const int ii = id[i], ij = id[j];
  v[i] = sw ? vj : vi;
  v[j] = sw ? vi : vj;
  id[i] = sw ? ij : ii;
  id[j] = sw ? ii : ij;
}

// Merge the sorted list of the lane `offset` away (xor) into this lane's: the
// better of v[j] and the partner's [KS-1-j] form a bitonic sequence holding the
// top KS of both lists, which a bitonic network sorts. Both lanes end with the
// same list.
template <int KS>
__device__ __forceinline__ void merge_with_lane(float (&v)[KS], int (&id)[KS], int offset) {
  float w[KS];
  int wid[KS];
#pragma unroll
  for (int j = 0; j < KS; ++j) {
    w[j] = __shfl_xor_sync(0xffffffffu, v[j], offset);
    wid[j] = __shfl_xor_sync(0xffffffffu, id[j], offset);
  }
#pragma unroll
  for (int j = 0; j < KS; ++j) {
    const bool take = ranks_before(w[KS - 1 - j], wid[KS - 1 - j], v[j], id[j]);
    v[j] = take ? w[KS - 1 - j] : v[j];
    id[j] = take ? wid[KS - 1 - j] : id[j];
  }
#pragma unroll
  for (int s = KS / 2; s >= 1; s >>= 1) {
#pragma unroll
    for (int i = 0; i < KS; ++i)
      if ((i & s) == 0) cas_desc<KS>(v, id, i, i + s);
  }
}

template <int KS>
__global__ void __launch_bounds__(kThreads, 1)
router_tc_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmW,
                 const RouterArgs a) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_u32 = ptx::smem_u32(smem_raw);
  uint8_t* smem = smem_raw + ((1024u - (raw_u32 & 1023u)) & 1023u);
  const uint32_t stage_bytes = kABytes + (uint32_t)a.N * kBK * 2;
  // region: the pipeline stages; once this CTA's accumulator is complete, its partial
  // sums [128][np] float32 (rows of this CTA's selection are summed in place)
  float* part = reinterpret_cast<float*>(smem);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + a.region);
  uint64_t* empty = full + a.stages;
  uint64_t* tfull = empty + a.stages;
  uint64_t* drain = tfull + 1;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);
  float* s_bias = reinterpret_cast<float*>(tmem_holder + 4);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int C = a.csplit;
  const int crank = (int)ptx::cluster_ctarank();
  const int tile = blockIdx.x / C;
  const int m0 = tile * kBM;
  const int kb0 = crank * a.k_steps / C;
  const int kb1 = (crank + 1) * a.k_steps / C;

  for (int e = threadIdx.x; e < a.E; e += kThreads) s_bias[e] = a.bias ? a.bias[e] : 0.0f;
  if (threadIdx.x == 0) {
    for (int s = 0; s < a.stages; ++s) {
      ptx::mbar_init(ptx::smem_u32(&full[s]), 1);
      ptx::mbar_init(ptx::smem_u32(&empty[s]), 1);
    }
    ptx::mbar_init(ptx::smem_u32(tfull), 1);
    ptx::mbar_init(ptx::smem_u32(drain), 1);
    *abort_flag = 0;
    ptx::fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    ptx::prefetch_tmap(&tmX);
    ptx::prefetch_tmap(&tmW);
  }
  if (warp == 1) {
    ptx::tmem_alloc(ptx::smem_u32(tmem_holder), a.tmem_cols);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem_base = *tmem_holder;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      const uint32_t full0 = ptx::smem_u32(full), empty0 = ptx::smem_u32(empty), stage0 = ptx::smem_u32(smem);
      int issued = 0;
      bool ok = true;
      int stage = 0;
      uint32_t phase = 0;
      for (int kb = kb0; kb < kb1; ++kb) {
        if (!ptx::mbar_wait_bounded(empty0 + 8u * stage, phase ^ 1u, abort_flag, kWaitLimitNs)) {
          ok = false;
          break;
        }
        const uint32_t fb = full0 + 8u * stage;
        const uint32_t sa = stage0 + (uint32_t)stage * stage_bytes;
        ptx::mbar_arrive_expect_tx(fb, stage_bytes);
        ptx::tma_load_2d(sa, &tmX, kb * kBK, m0, fb);
        ptx::tma_load_2d(sa + kABytes, &tmW, kb * kBK, 0, fb);
        if (issued < a.stages) ++issued;
        if (++stage == a.stages) {
          stage = 0;
          phase ^= 1u;
        }
      }
      if (!ok) {
        set_status(a.status, MOE_ERR_TIMEOUT);
        *abort_flag = 1;
        // the latest fill of each slot lands before the shared memory is reused
        // (walking back from the slot that was not filled)
        for (int j = 0; j < issued; ++j) {
          if (stage == 0) {
            stage = a.stages - 1;
            phase ^= 1u;
          } else {
            --stage;
          }
          ptx::mbar_wait_bounded(full0 + 8u * stage, phase, nullptr, kDrainLimitNs);
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t idesc = ptx::idesc_bf16_f32(kBM, a.N);
      const uint32_t full0 = ptx::smem_u32(full), empty0 = ptx::smem_u32(empty), stage0 = ptx::smem_u32(smem);
      bool ok = true;
      int stage = 0;
      uint32_t phase = 0;
      for (int kb = kb0; kb < kb1; ++kb) {
        if (!ptx::mbar_wait_bounded(full0 + 8u * stage, phase, abort_flag, kWaitLimitNs)) {
          ok = false;
          break;
        }
        ptx::tc_fence_after();
        const uint32_t sa = stage0 + (uint32_t)stage * stage_bytes;
        const uint64_t a_desc = ptx::sw128_kmajor_desc(sa);
        const uint64_t b_desc = ptx::sw128_kmajor_desc(sa + kABytes);
#pragma unroll
        for (int kk = 0; kk < kBK / 16; ++kk)
          ptx::mma_bf16(tmem_base, a_desc + (uint64_t)(2 * kk), b_desc + (uint64_t)(2 * kk), idesc,
                        (kb != kb0 || kk != 0) ? 1u : 0u);
        ptx::mma_commit(empty0 + 8u * stage);
        if (++stage == a.stages) {
          stage = 0;
          phase ^= 1u;
        }
      }
      if (ok) {
        ptx::mma_commit(ptx::smem_u32(tfull));
      } else {
        set_status(a.status, MOE_ERR_TIMEOUT);
        *abort_flag = 1;
      }
      ptx::mma_commit(ptx::smem_u32(drain));
      ptx::mbar_wait_bounded(ptx::smem_u32(drain), 0, nullptr, kDrainLimitNs);
    }
  } else {
    // ------------------------------------- epilogue part 1: TMEM -> shared partials
    const int quarter = warp & 3;                     // the TMEM lanes this warp may read
    const int slice0 = (warp - 2) >> 2;               // first 32-column slice of this warp
    const int r = quarter * 32 + lane;                // row of the tile = TMEM lane
    if (!ptx::mbar_wait_bounded(ptx::smem_u32(tfull), 0, abort_flag, kWaitLimitNs)) {
      set_status(a.status, MOE_ERR_TIMEOUT);
      *abort_flag = 1;
    }
    const bool ok = __all_sync(0xffffffffu, *abort_flag == 0);
    if (ok) {
      ptx::tc_fence_after();
      const uint32_t trow = tmem_base + ((uint32_t)(quarter * 32) << 16);
      for (int sl = slice0; sl * 32 < a.N; sl += 4) {
        uint32_t v[32];
        ptx::tmem_ld32(trow + (uint32_t)(sl * 32), v);
        ptx::tmem_ld_wait();
        float4* dst = reinterpret_cast<float4*>(part + (size_t)r * a.np + sl * 32);
#pragma unroll
        for (int q = 0; q < 8; ++q)
          if (sl * 32 + 4 * q < a.N)
            dst[q] = make_float4(__uint_as_float(v[4 * q]), __uint_as_float(v[4 * q + 1]),
                                 __uint_as_float(v[4 * q + 2]), __uint_as_float(v[4 * q + 3]));
      }
    }
  }
  __syncwarp();
  ptx::tc_fence_before();
  ptx::cluster_sync_all();                            // partials of every CTA are complete

  // ------------------------------------------- reduction over the cluster (all threads)
  const int R = kBM / C;                              // rows this CTA selects
  const int row0 = crank * R;
  int my_flag = 0;
  if (threadIdx.x < C)
    my_flag = (int)ptx::ld_shared_cluster_u32(
        ptx::map_shared_rank(ptx::smem_u32((const void*)abort_flag), (uint32_t)threadIdx.x));
  const bool any_abort = __syncthreads_or(my_flag) != 0;
  if (!any_abort) {
    const int n4 = a.N / 4;
    const uint32_t part_u32 = ptx::smem_u32(part);
    for (int i = threadIdx.x; i < R * n4; i += kThreads) {
      const int rr = row0 + i / n4;
      const int c4 = i - (i / n4) * n4;
      const uint32_t off = (uint32_t)(((size_t)rr * a.np + 4 * c4) * 4);
      // all C loads in flight first, then the sum in rank order
      float4 pv[kMaxCluster];
#pragma unroll
      for (int c = 0; c < kMaxCluster; ++c)
        if (c < C) pv[c] = ptx::ld_shared_cluster_v4(ptx::map_shared_rank(part_u32 + off, (uint32_t)c));
      float4 acc = pv[0];
#pragma unroll
      for (int c = 1; c < kMaxCluster; ++c) {
        if (c < C) {
          acc.x += pv[c].x;
          acc.y += pv[c].y;
          acc.z += pv[c].z;
          acc.w += pv[c].w;
        }
      }
      const int e = 4 * c4;
      acc.x += e < a.E ? s_bias[e] : 0.0f;
      acc.y += e + 1 < a.E ? s_bias[e + 1] : 0.0f;
      acc.z += e + 2 < a.E ? s_bias[e + 2] : 0.0f;
      acc.w += e + 3 < a.E ? s_bias[e + 3] : 0.0f;
      // rows [row0, row0 + R) of this CTA's buffer are read by no other CTA
      *reinterpret_cast<float4*>(part + (size_t)rr * a.np + 4 * c4) = acc;
    }
  }
  __syncthreads();

  // --------------------------------------------------- selection (epilogue threads)
  const int P = a.sel_p;                              // threads per token
  if (warp >= 2 && (warp - 2) * 32 < R * P) {
    const int et = threadIdx.x - 64;
    const int rl = et / P;                            // row among this CTA's R rows
    const int p = et - rl * P;
    const int t = m0 + row0 + rl;
    const float* lrow = part + (size_t)(row0 + rl) * a.np;
    const bool softmax = (a.score == MOE_SOFTMAX);
    if (any_abort) {
      if (t < a.T)
        for (int j = p; j < a.k; j += P) {
          a.idx[(size_t)t * a.k + j] = -1;
          a.gate[(size_t)t * a.k + j] = 0.0f;
        }
    } else {
      float best[KS];
      int best_e[KS];
#pragma unroll
      for (int j = 0; j < KS; ++j) {
        best[j] = -INFINITY;
        best_e[j] = kNoExpert;
      }
      // eight logits per batch: the shared loads are issued together, then inserted
      for (int e0 = p; e0 < a.E; e0 += 8 * P) {
        float lv[8];
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          const int e = e0 + q * P;
          lv[q] = e < a.E ? lrow[e] : -INFINITY;
        }
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          const int e = e0 + q * P;
          topk_insert<KS>(isnan(lv[q]) ? -INFINITY : lv[q], e < a.E ? e : kNoExpert, best, best_e);
        }
      }
      for (int o = 1; o < P; o <<= 1) merge_with_lane<KS>(best, best_e, o);
      // fewer than k ranked entries (NaN logits): the lowest unused ids fill the rest
#pragma unroll
      for (int j = 0; j < KS; ++j) {
        if (j < a.k && best_e[j] == kNoExpert) {
          for (int e = 0; e < a.E; ++e) {
            bool used = false;
#pragma unroll
            for (int i = 0; i < KS; ++i) used |= (i < j && best_e[i] == e);
            if (!used) {
              best_e[j] = e;
              break;
            }
          }
        }
      }
      const float mx = best[0];
      float denom = 1.0f;
      if (softmax && (!a.renorm || a.scores != nullptr)) {
        float ps = 0.0f;
        for (int e = p; e < a.E; e += P) ps += expf(lrow[e] - mx);
        for (int o = 1; o < P; o <<= 1) ps += __shfl_xor_sync(0xffffffffu, ps, o);
        denom = ps;
      }
      // thread p of the token owns slots p, p+P, ...: their scores, then the sum of the
      // k selected over the token's threads
      float mine[KS];
      float part_sum = 0.0f;
#pragma unroll
      for (int j = 0; j < KS; ++j) {
        mine[j] = 0.0f;
        if (j < a.k && (j & (P - 1)) == p) {
          mine[j] = softmax ? expf(best[j] - mx) : sigmoid_f(best[j]);
          part_sum += mine[j];
        }
      }
      float total = part_sum;
      for (int o = 1; o < P; o <<= 1) total += __shfl_xor_sync(0xffffffffu, total, o);
      if (t < a.T) {
#pragma unroll
        for (int j = 0; j < KS; ++j) {
          if (j < a.k && (j & (P - 1)) == p) {
            const float g =
                a.renorm ? __fdiv_rn(mine[j], total) : (softmax ? __fdiv_rn(mine[j], denom) : mine[j]);
            a.idx[(size_t)t * a.k + j] = best_e[j];
            a.gate[(size_t)t * a.k + j] = g;
          }
        }
        if (a.scores != nullptr)
          for (int e = p; e < a.E; e += P)
            a.scores[(size_t)t * a.E + e] = softmax ? __fdiv_rn(expf(lrow[e] - mx), denom) : sigmoid_f(lrow[e]);
      }
    }
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem_base, a.tmem_cols);
  }
  __syncwarp();
  ptx::cluster_sync_all();                            // no CTA leaves while others read its partials
}

// Instruction-count model of the selection: a warp scans E / P experts (one insertion
// each) and runs log2(P) list merges; warps = rows x P / 32 share four schedulers.
int pick_sel_p(int rows, int E, int ks) {
  const int c_ins = ks == 8 ? 50 : ks == 4 ? 25 : 12;
  const int c_merge = ks == 8 ? 170 : ks == 4 ? 80 : 40;
  int best_p = 0;
  long best_cost = 0;
  for (int P = 1; P <= 32; P <<= 1) {
    if (rows * P < 32 || rows * P > kEpiThreads) continue;
    int lg = 0;
    while ((1 << lg) < P) ++lg;
    const long per_warp = (long)((E + P - 1) / P) * c_ins + (long)lg * c_merge;
    const long cost = (long)((rows * P + 127) / 128) * per_warp;
    if (best_p == 0 || cost < best_cost) {
      best_p = P;
      best_cost = cost;
    }
  }
  return best_p;
}

// cudaOccupancyMaxActiveClusters answers, cached per (list size, split, shared memory).
struct ClusterFit {
  int ks, csplit;
  size_t smem;
  bool fits;
};
std::mutex g_fit_mu;
ClusterFit g_fit[64];
int g_nfit = 0;

template <int KS>
bool cluster_fits(const cudaLaunchConfig_t& cfg, int csplit) {
  {
    std::lock_guard<std::mutex> lock(g_fit_mu);
    for (int i = 0; i < g_nfit; ++i)
      if (g_fit[i].ks == KS && g_fit[i].csplit == csplit && g_fit[i].smem == cfg.dynamicSmemBytes)
        return g_fit[i].fits;
  }
  int n = 0;
  const bool fits = cudaOccupancyMaxActiveClusters(&n, router_tc_kernel<KS>, &cfg) == cudaSuccess && n > 0;
  cudaGetLastError();
  std::lock_guard<std::mutex> lock(g_fit_mu);
  if (g_nfit < 64) g_fit[g_nfit++] = ClusterFit{KS, csplit, cfg.dynamicSmemBytes, fits};
  return fits;
}

template <int KS>
cudaError_t launch_ks(const CUtensorMap& tx, const CUtensorMap& tw, RouterArgs a, int tiles, cudaStream_t st) {
  auto kern = router_tc_kernel<KS>;
  // alignment slack, stage / partial region, barriers (2 per stage + 2), TMEM address +
  // abort flag + padding, bias
  const size_t smem = 1024 + a.region + (size_t)(2 * a.stages + 2) * 8 + 16 + (size_t)a.E * 4;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  // the largest split whose clusters can be resident (the query needs the smem size set)
  for (; a.csplit > 1; a.csplit >>= 1) {
    attr[0].val.clusterDim.x = (unsigned)a.csplit;
    cfg.gridDim = dim3((unsigned)(tiles * a.csplit));
    if (cluster_fits<KS>(cfg, a.csplit)) break;
  }
  a.sel_p = pick_sel_p(kBM / a.csplit, a.E, KS);
  attr[0].val.clusterDim.x = (unsigned)a.csplit;
  cfg.gridDim = dim3((unsigned)(tiles * a.csplit));
  e = cudaLaunchKernelEx(&cfg, kern, tx, tw, a);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace

bool router_tc_supported(const Shape& s) {
  return s.dtype == MOE_BF16 && s.d % kBK == 0 && s.E >= 1 && s.E <= 256 && s.k <= 8;
}

cudaError_t launch_router_tc(const Shape& s, const void* x, const void* w, const float* bias, int32_t* idx,
                             float* gate, float* scores, int32_t* status, cudaStream_t st) {
  if (!router_tc_supported(s)) return cudaErrorInvalidValue;
  RouterArgs a{};
  a.T = s.T;
  a.E = s.E;
  a.N = (s.E + 15) / 16 * 16;
  a.np = a.N + 4;
  a.k = s.k;
  a.k_steps = s.d / kBK;
  a.score = s.score;
  a.renorm = s.renorm;
  a.tmem_cols = 32;
  while ((int)a.tmem_cols < a.N) a.tmem_cols <<= 1;
  const size_t stage_bytes = kABytes + (size_t)a.N * kBK * 2;
  int stages = (int)(kSmemBudget / stage_bytes);
  if (stages > 8) stages = 8;
  if (stages > a.k_steps) stages = a.k_steps;
  if (stages < 1) stages = 1;
  a.stages = stages;
  const size_t part_bytes = (size_t)kBM * a.np * 4;
  const size_t main_bytes = (size_t)stages * stage_bytes;
  a.region = ((main_bytes > part_bytes ? main_bytes : part_bytes) + 1023) / 1024 * 1024;
  const int tiles = (s.T + kBM - 1) / kBM;
  // split d_model over up to 8 CTAs while tiles x split stays within one wave
  int c = 1;
  while (c < kMaxCluster && (int64_t)tiles * c * 2 <= num_sms() && c * 2 <= a.k_steps) c *= 2;
  a.csplit = c;
  a.bias = bias;
  a.idx = idx;
  a.gate = gate;
  a.scores = scores;
  a.status = status;
  CUtensorMap tx, tw;
  if (!make_tmap_bf16(&tx, x, (uint64_t)s.d, (uint64_t)s.T, kBM)) return cudaErrorInvalidValue;
  if (!make_tmap_bf16(&tw, w, (uint64_t)s.d, (uint64_t)s.E, (uint32_t)a.N)) return cudaErrorInvalidValue;
  if (s.k <= 2) return launch_ks<2>(tx, tw, a, tiles, st);
  if (s.k <= 4) return launch_ks<4>(tx, tw, a, tiles, st);
  return launch_ks<8>(tx, tw, a, tiles, st);
}

}  // namespace moe
