// The expert MLP's two grouped contractions in ONE persistent launch (bf16): gate/up + SwiGLU
// tiles, then down-projection tiles, each CTA walking its share of both lists in order.
//
// The separate launches of gemm_tc.cu hand out tiles round-robin, so a launch whose tile count
// is just past a multiple of the SM count ends with a round on a few SMs (the Mixtral-shaped
// down projection: 1088 tiles over 148 SMs, 7.35 rounds; the decode batch: 672 gate/up and 896
// down tiles), and the down projection cannot start before the last gate/up tile has finished.
// Here the down tiles of an expert's m-tile start as soon as that m-tile's h rows are complete:
// every gate/up tile publishes, per epilogue warp, one count on a per-m-tile counter in global
// memory (release), and a down tile's producer waits (acquire, bounded) until the counter holds
// all gate/up n-tiles of its m-tile before its first TMA load of h. A CTA reaches its own down
// tiles only after all of its gate/up tiles, so every gate/up tile is finished by a CTA that
// never waits before it, and with one resident CTA per SM the waits end.
//
// Tiles, stages and roles are those of gemm_tc.cu's single-CTA kernel: warp 0 TMA producer
// (128 x 64 A and 256 x 64 B tiles, 4 stages of 48 KB), warp 1 MMA issuer (tcgen05 kind::f16,
// M=128, N=256, two TMEM accumulators), warps 2-9 epilogue (staged whole-sector stores). h is
// written by generic stores and read by TMA in other CTAs: the writers fence the generic proxy
// against the async proxy before publishing, the reader fences again after acquiring.
//
// With COMBINE the down tiles also produce the layer output (the deterministic gather-reduce
// of the combine, klaylearn.com/glossary/mixture-of-experts: restore token order): once a down
// tile's rows are stored, one thread per row fences and adds one (acquire-release) to its
// token's counter; the add that reaches the token's total (down n-tiles x its kept rows and
// shared row) queues the token, and the tile's 256 epilogue threads sum its rows in slot order
// with the separate combine kernel's arithmetic, so the output has the same bits. No thread
// waits for another: the last arrival does the work.
#include "epilogue.cuh"
#include "gemm_common.cuh"
#include "internal.cuh"
#include "tc_ptx.cuh"
#include "tmap.cuh"

namespace moe {
namespace {

using gemm::decode_tile;
using gemm::drain_fills;
using gemm::kDrainLimitNs;
using gemm::kWaitLimitNs;

constexpr int kBM = 128;
constexpr int kBK = 64;
constexpr int kEpiWarps = 8;
constexpr int kThreads = 64 + 32 * kEpiWarps;
constexpr int kABytes = kBM * kBK * 2;             // 16 KB
constexpr int kBBytes = 256 * kBK * 2;             // 32 KB
constexpr int kStageBytes = kABytes + kBBytes;
constexpr int kStages = 4;
constexpr int kTmemCols = 512;
constexpr int kSchedInts = 4 * (kMaxExperts + 2);
constexpr size_t kStgOff = (size_t)kStages * kStageBytes + 256 + (((size_t)kSchedInts * 4 + 127) / 128) * 128;
constexpr size_t kListOff = kStgOff + (size_t)kEpiWarps * epi::kStageOutBytes;
constexpr size_t kSmem = 1024 + kListOff + (size_t)kBM * 4;     // + the tokens a down tile completes
constexpr int kEpiThreads = 32 * kEpiWarps;

struct FusedArgs {
  int K1, K2;             // reductions: d (gate/up), d_ff (down)
  int nt1, nt2;           // n-tiles per group: d_ff / 128 (gate/up), d / 256 (down)
  int G, E;               // groups; groups >= E (shared expert) read x itself in gate/up
  int F, d;
  const int32_t* sched;   // device group schedule
  __nv_bfloat16* h;       // [rows, d_ff]
  __nv_bfloat16* y;       // [rows, d]
  int32_t* ready;         // [m-tiles]: published epilogue-warp counts of finished gate/up tiles
  int32_t* status;
  // the combine in the down tiles (COMBINE): out[t] = sum over t's kept slots j in slot order of
  // gate[t, j] * y[dest_row[t, j]] (+ y[R + t] with a shared expert), by the tile that completes t
  const int32_t* src_token;
  const int32_t* dest_row;
  const float* gate;
  __nv_bfloat16* out;
  int32_t* tok_done;      // [T]: finished (row, down n-tile) pieces of each token
  int k, T, S;
  int64_t R;
};

__device__ __forceinline__ void fence_proxy_async_global() {
  asm volatile("fence.proxy.async.global;" ::: "memory");
}
__device__ __forceinline__ void red_release_add(int32_t* p, int v) {
  asm volatile("red.release.gpu.global.add.s32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ int ld_acquire(const int32_t* p) {
  int v;
  asm volatile("ld.acquire.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ int atom_acq_rel_add(int32_t* p, int v) {
  int old;
  asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}
// the eight epilogue warps (threads 64 .. 319)
__device__ __forceinline__ void epi_bar() { asm volatile("bar.sync 1, %0;" ::"r"(kEpiThreads) : "memory"); }

// Rows of token t the down tiles write: its kept slots (dest_row in [0, R)) and the shared
// expert's row.
__device__ __forceinline__ int token_rows(const FusedArgs& a, int t) {
  int n = a.S;
  for (int j = 0; j < a.k; ++j) {
    const int r = __ldg(a.dest_row + (int64_t)t * a.k + j);
    n += (r >= 0 && r < a.R) ? 1 : 0;
  }
  return n;
}

// Token t's output row by the 256 epilogue threads (et = 0 .. 255), 8 columns per thread and
// pass: the arithmetic of the separate combine kernel (float32, slot order, the shared row
// last), so the same bits. y rows were written by other CTAs in this launch: coherent loads.
__device__ __forceinline__ void combine_token(const FusedArgs& a, int t, int et) {
  for (int c = et * 8; c < a.d; c += kEpiThreads * 8) {
    float acc[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i] = 0.f;
    for (int j = 0; j < a.k; ++j) {
      int r = __ldg(a.dest_row + (int64_t)t * a.k + j);
      if (r >= a.R) {
        set_status(a.status, MOE_ERR_DEVICE_INDEX);
        r = -1;
      }
      if (r < 0) continue;
      const uint4 u = __ldcg(reinterpret_cast<const uint4*>(a.y + (int64_t)r * a.d + c));
      const float g = __ldg(a.gate + (int64_t)t * a.k + j);
      const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        acc[2 * i] = fmaf(g, __uint_as_float(w[i] << 16), acc[2 * i]);
        acc[2 * i + 1] = fmaf(g, __uint_as_float(w[i] & 0xFFFF0000u), acc[2 * i + 1]);
      }
    }
    if (a.S > 0) {
      const uint4 u = __ldcg(reinterpret_cast<const uint4*>(a.y + (a.R + t) * a.d + c));
      const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        acc[2 * i] += __uint_as_float(w[i] << 16);
        acc[2 * i + 1] += __uint_as_float(w[i] & 0xFFFF0000u);
      }
    }
    uint32_t o[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const __nv_bfloat162 b = __floats2bfloat162_rn(acc[2 * i], acc[2 * i + 1]);
      o[i] = *reinterpret_cast<const uint32_t*>(&b);
    }
    *reinterpret_cast<uint4*>(a.out + (int64_t)t * a.d + c) = make_uint4(o[0], o[1], o[2], o[3]);
  }
}

// Wait until *p >= target, giving up after limit_ns or when *abort is set. True on success.
__device__ __forceinline__ bool wait_count(const int32_t* p, int target, volatile int* abort, uint64_t limit_ns) {
  if (ld_acquire(p) >= target) return true;
  const uint64_t t0 = ptx::globaltimer_ns();
#pragma unroll 1
  while (true) {
    for (int i = 0; i < 32; ++i) {
      __nanosleep(64);
      if (ld_acquire(p) >= target) return true;
    }
    if (*abort) return false;
    if (ptx::globaltimer_ns() - t0 > limit_ns) return false;
  }
}

template <bool COMBINE>
__global__ void __launch_bounds__(kThreads, 1)
grouped_mlp_fused_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmXs,
                         const __grid_constant__ CUtensorMap tmWg, const __grid_constant__ CUtensorMap tmWu,
                         const __grid_constant__ CUtensorMap tmH, const __grid_constant__ CUtensorMap tmWd,
                         const FusedArgs args) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_u32 = ptx::smem_u32(smem_raw);
  uint8_t* smem = smem_raw + ((1024u - (raw_u32 & 1023u)) & 1023u);   // 1024-byte aligned
  uint8_t* stage_base = smem;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + (size_t)kStages * kStageBytes);
  uint64_t* full = bars;                       // [kStages]
  uint64_t* empty = bars + kStages;            // [kStages]
  uint64_t* tfull = bars + 2 * kStages;        // [2]
  uint64_t* tempty = tfull + 2;                // [2]
  uint64_t* drain = tempty + 2;                // [1]
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);
  volatile int* s_stop = abort_flag + 1;       // COMBINE: the epilogue's snapshot of the abort flag
  int32_t* s_ncomb = reinterpret_cast<int32_t*>(tmem_holder + 4);   // COMBINE: tokens the down tile completed
  int32_t* s_list = reinterpret_cast<int32_t*>(smem + kListOff);
  int32_t* s_tile_start = reinterpret_cast<int32_t*>(smem + (size_t)kStages * kStageBytes + 256);
  int32_t* s_a_row = s_tile_start + (args.G + 1);
  int32_t* s_out_row = s_a_row + args.G;
  int32_t* s_rows = s_out_row + args.G;
  const uint32_t stg_base = ptx::smem_u32(smem + kStgOff);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  for (int i = threadIdx.x; i < 4 * args.G + 1; i += kThreads) s_tile_start[i] = args.sched[i];
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      ptx::mbar_init(ptx::smem_u32(&full[s]), 1);
      ptx::mbar_init(ptx::smem_u32(&empty[s]), 1);
    }
    for (int a = 0; a < 2; ++a) {
      ptx::mbar_init(ptx::smem_u32(&tfull[a]), 1);
      ptx::mbar_init(ptx::smem_u32(&tempty[a]), kEpiWarps * 32);
    }
    ptx::mbar_init(ptx::smem_u32(drain), 1);
    *abort_flag = 0;
    ptx::fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    ptx::prefetch_tmap(&tmX);
    ptx::prefetch_tmap(&tmXs);
    ptx::prefetch_tmap(&tmWg);
    ptx::prefetch_tmap(&tmWu);
    ptx::prefetch_tmap(&tmH);
    ptx::prefetch_tmap(&tmWd);
  }
  if (warp == 1) {
    ptx::tmem_alloc(ptx::smem_u32(tmem_holder), kTmemCols);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem_base = *tmem_holder;

  const int m_tiles = s_tile_start[args.G];
  const int n1 = m_tiles * args.nt1;                 // gate/up tiles come first
  const int total = n1 + m_tiles * args.nt2;
  const int ready_target = args.nt1 * kEpiWarps;     // every epilogue warp of every gate/up n-tile

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      int stage = 0, issued = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int L = blockIdx.x; L < total && ok; L += gridDim.x) {
        const bool up = L < n1;
        int g, m, n;
        decode_tile(up ? L : L - n1, s_tile_start, args.G, up ? args.nt1 : args.nt2, g, m, n);
        const void* map_a;
        const void* map_b;
        int a_row, b_row, k_steps;
        if (up) {
          map_a = (g >= args.E) ? (const void*)&tmXs : (const void*)&tmX;
          map_b = &tmWg;
          a_row = s_a_row[g] + m * kBM;
          b_row = g * args.F + n * 128;
          k_steps = args.K1 / kBK;
        } else {
          // h rows of this m-tile: complete once all gate/up n-tiles of it have been published
          if (!wait_count(args.ready + s_tile_start[g] + m, ready_target, abort_flag, kWaitLimitNs)) {
            ok = false;
            break;
          }
          fence_proxy_async_global();
          map_a = &tmH;
          map_b = &tmWd;
          a_row = s_out_row[g] + m * kBM;
          b_row = g * args.d + n * 256;
          k_steps = args.K2 / kBK;
        }
        for (int kb = 0; kb < k_steps; ++kb) {
          if (!ptx::mbar_wait_bounded(ptx::smem_u32(&empty[stage]), phase ^ 1u, abort_flag, kWaitLimitNs)) {
            ok = false;
            break;
          }
          const uint32_t fb = ptx::smem_u32(&full[stage]);
          const uint32_t sa = ptx::smem_u32(stage_base + (size_t)stage * kStageBytes);
          const uint32_t sb = sa + kABytes;
          ptx::mbar_arrive_expect_tx(fb, kStageBytes);
          ptx::tma_load_2d(sa, map_a, kb * kBK, a_row, fb);
          ptx::tma_load_2d(sb, map_b, kb * kBK, b_row, fb);
          if (up) ptx::tma_load_2d(sb + 128 * 128, &tmWu, kb * kBK, b_row, fb);
          if (issued < kStages) ++issued;
          if (++stage == kStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (!ok) {
        set_status(args.status, MOE_ERR_TIMEOUT);
        *abort_flag = 1;
        drain_fills(full, kStages, stage, phase, issued);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc = ptx::idesc_bf16_f32(kBM, 256);
      int stage = 0, it = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int L = blockIdx.x; L < total && ok; L += gridDim.x, ++it) {
        const int k_steps = (L < n1 ? args.K1 : args.K2) / kBK;
        const int acc = it & 1;
        const uint32_t acc_phase = (uint32_t)(it >> 1) & 1u;
        if (!ptx::mbar_wait_bounded(ptx::smem_u32(&tempty[acc]), acc_phase ^ 1u, abort_flag, kWaitLimitNs)) {
          ok = false;
          break;
        }
        ptx::tc_fence_after();
        const uint32_t d_tmem = tmem_base + (uint32_t)(acc * 256);
        for (int kb = 0; kb < k_steps; ++kb) {
          if (!ptx::mbar_wait_bounded(ptx::smem_u32(&full[stage]), phase, abort_flag, kWaitLimitNs)) {
            ok = false;
            break;
          }
          ptx::tc_fence_after();
          const uint32_t sa = ptx::smem_u32(stage_base + (size_t)stage * kStageBytes);
          const uint64_t a_desc = ptx::sw128_kmajor_desc(sa);
          const uint64_t b_desc = ptx::sw128_kmajor_desc(sa + kABytes);
#pragma unroll
          for (int kk = 0; kk < kBK / 16; ++kk)
            ptx::mma_bf16(d_tmem, a_desc + (uint64_t)(2 * kk), b_desc + (uint64_t)(2 * kk), idesc,
                          (kb | kk) != 0 ? 1u : 0u);
          ptx::mma_commit(ptx::smem_u32(&empty[stage]));
          if (++stage == kStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        ptx::mma_commit(ptx::smem_u32(&tfull[acc]));
      }
      if (!ok) {
        set_status(args.status, MOE_ERR_TIMEOUT);
        *abort_flag = 1;
      }
      ptx::mma_commit(ptx::smem_u32(drain));
      ptx::mbar_wait_bounded(ptx::smem_u32(drain), 0, nullptr, kDrainLimitNs);
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int quarter = warp & 3;
    const int half = (warp - 2) >> 2;
    const int et = threadIdx.x - 64;                 // 0 .. 255
    const uint32_t stg = stg_base + (uint32_t)(warp - 2) * epi::kStageOutBytes;
    if constexpr (COMBINE) {
      // tokens no row reaches (every slot dropped, no shared expert) get a zero output row here
      for (int t = (int)blockIdx.x * kEpiThreads + et; t < args.T; t += (int)gridDim.x * kEpiThreads)
        if (token_rows(args, t) == 0)
          for (int c = 0; c < args.d; c += 8)
            *reinterpret_cast<uint4*>(args.out + (int64_t)t * args.d + c) = make_uint4(0, 0, 0, 0);
    }
    int it = 0;
    for (int L = blockIdx.x; L < total; L += gridDim.x, ++it) {
      const bool up = L < n1;
      int g, m, n;
      decode_tile(up ? L : L - n1, s_tile_start, args.G, up ? args.nt1 : args.nt2, g, m, n);
      const int acc = it & 1;
      const uint32_t acc_phase = (uint32_t)(it >> 1) & 1u;
      if (!ptx::mbar_wait_bounded(ptx::smem_u32(&tfull[acc]), acc_phase, abort_flag, kWaitLimitNs)) {
        set_status(args.status, MOE_ERR_TIMEOUT);
        *abort_flag = 1;
        if (!COMBINE) break;
      }
      if constexpr (COMBINE) {
        // the epilogue warps meet at named barriers: all eight leave on the same snapshot
        epi_bar();
        if (et == 0) *s_stop = *abort_flag;
        epi_bar();
        if (*s_stop != 0) break;
      }
      ptx::tc_fence_after();
      const int row0 = m * kBM + quarter * 32;
      const int64_t orow = (int64_t)s_out_row[g] + row0;
      const uint32_t t_row = tmem_base + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(acc * 256);
      if (up) {
        epi::store_tile<true, 128>(t_row, s_rows[g] - row0, args.h + orow * args.F + (int64_t)n * 128, args.F, half,
                                   stg, lane);
        // publish this warp's part of the m-tile's h rows: its stores, ordered against the async
        // proxy that reads h, then one release count
        fence_proxy_async_global();
        __syncwarp();
        if (lane == 0) red_release_add(args.ready + s_tile_start[g] + m, 1);
      } else {
        epi::store_tile<false, 256>(t_row, s_rows[g] - row0, args.y + orow * args.d + (int64_t)n * 256, args.d, half,
                                    stg, lane);
      }
      // the accumulator is free: the combine below reads y, not TMEM
      ptx::tc_fence_before();
      ptx::mbar_arrive(ptx::smem_u32(&tempty[acc]));
      if (!up) {
        if constexpr (COMBINE) {
          // count this tile's rows on their tokens: the barrier orders all eight warps' stores
          // before each counting thread's gpu-scope release; the count that completes a token
          // queues it, and the warps combine it
          if (et == 0) *s_ncomb = 0;
          epi_bar();
          const int rows_here = min(kBM, s_rows[g] - m * kBM);
          if (et < rows_here) {
            const int lr = m * kBM + et;
            const int t = (g >= args.E) ? lr : __ldg(args.src_token + s_out_row[g] + lr);
            const int target = token_rows(args, t) * args.nt2;
            if (atom_acq_rel_add(args.tok_done + t, 1) + 1 == target) s_list[atomicAdd(s_ncomb, 1)] = t;
          }
          epi_bar();
          const int nc = *s_ncomb;
          for (int i = 0; i < nc; ++i) combine_token(args, s_list[i], et);
          epi_bar();
        }
      }
    }
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem_base, kTmemCols);
  }
}

int64_t max_m_tiles(const Shape& s) {
  return (s.R + kBM - 1) / kBM + s.E + (int64_t)s.S * ((s.T + kBM - 1) / kBM);
}

}  // namespace

bool fused_mlp_supported(const Shape& s) { return s.dtype == MOE_BF16 && s.d % 256 == 0 && s.F % 128 == 0; }

int64_t fused_mlp_ready_ints(const Shape& s) { return max_m_tiles(s) + s.T; }

cudaError_t launch_mlp_fused_tc(const Shape& s, const void* x_perm, const void* x, const void* w_gate,
                                const void* w_up, const void* w_down, const void* sched, void* h, void* y,
                                int32_t* ready, int32_t* status, cudaStream_t st, const int32_t* src_token,
                                const int32_t* dest_row, const float* gate, void* out) {
  CUtensorMap tx, txs, twg, twu, th, twd;
  const uint64_t R = (uint64_t)(s.R > 0 ? s.R : 1);
  const uint64_t rows = (uint64_t)s.R + (uint64_t)s.S * s.T;
  if (!make_tmap_bf16(&tx, x_perm, s.d, R, kBM)) return cudaErrorInvalidValue;
  if (!make_tmap_bf16(&txs, s.S > 0 ? x : x_perm, s.d, s.S > 0 ? (uint64_t)s.T : R, kBM)) return cudaErrorInvalidValue;
  if (!make_tmap_bf16(&twg, w_gate, s.d, (uint64_t)s.G * s.F, 128)) return cudaErrorInvalidValue;
  if (!make_tmap_bf16(&twu, w_up, s.d, (uint64_t)s.G * s.F, 128)) return cudaErrorInvalidValue;
  if (!make_tmap_bf16(&th, h, s.F, rows > 0 ? rows : 1, kBM)) return cudaErrorInvalidValue;
  if (!make_tmap_bf16(&twd, w_down, s.F, (uint64_t)s.G * s.d, 256)) return cudaErrorInvalidValue;
  FusedArgs args{};
  args.K1 = s.d;
  args.K2 = s.F;
  args.nt1 = s.F / 128;
  args.nt2 = s.d / 256;
  args.G = s.G;
  args.E = s.E;
  args.F = s.F;
  args.d = s.d;
  args.sched = static_cast<const int32_t*>(sched);
  args.h = static_cast<__nv_bfloat16*>(h);
  args.y = static_cast<__nv_bfloat16*>(y);
  args.ready = ready;
  args.status = status;
  const bool combine = out != nullptr;
  if (combine && (src_token == nullptr || dest_row == nullptr || gate == nullptr)) return cudaErrorInvalidValue;
  args.src_token = src_token;
  args.dest_row = dest_row;
  args.gate = gate;
  args.out = static_cast<__nv_bfloat16*>(out);
  args.tok_done = ready + max_m_tiles(s);
  args.k = s.k;
  args.T = s.T;
  args.S = s.S;
  args.R = s.R;
  cudaError_t e = cudaMemsetAsync(ready, 0, (size_t)(max_m_tiles(s) + (combine ? s.T : 0)) * sizeof(int32_t), st);
  if (e != cudaSuccess) return e;
  auto kern = combine ? grouped_mlp_fused_kernel<true> : grouped_mlp_fused_kernel<false>;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmem);
  if (e != cudaSuccess) return e;
  int64_t grid = num_sms();
  const int64_t max_tiles = max_m_tiles(s) * (args.nt1 + args.nt2);
  if (max_tiles < grid) grid = max_tiles;
  if (grid < 1) grid = 1;
  kern<<<(unsigned)grid, kThreads, kSmem, st>>>(tx, txs, twg, twu, th, twd, args);
  return cudaGetLastError();
}

}  // namespace moe
