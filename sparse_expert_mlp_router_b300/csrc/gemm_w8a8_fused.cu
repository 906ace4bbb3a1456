// The W8A8 expert MLP in ONE persistent launch: gate/up tiles (E4M3 x codes, E4M3 weights,
// SwiGLU, bf16 h), h quantised to E4M3 per row, then down tiles (E4M3 h codes, E4M3 weights).
//
// As in gemm_fused.cu, every CTA walks its gate/up tiles, then its down tiles, and a down tile
// of an m-tile (128 grouped rows) waits for that m-tile's h. W8A8 adds one step between: h is
// quantised per row, and a row's scale needs all d_ff of its columns, which the m-tile's
// gate/up tiles (one per 128 columns) produce on different CTAs. So each gate/up tile, once its
// eight epilogue warps have stored their h rows, counts itself on the m-tile's first counter
// (acquire-release); the tile that completes the count quantises the m-tile's rows (one warp
// per row: its max, scale = max / 448, E4M3 codes; the quantiser of the weights) and then
// publishes the m-tile's second counter (release), on which the down tiles' producer waits
// (acquire, bounded) before its first TMA load of the codes. A CTA reaches its own down tiles
// only after all of its gate/up tiles, so every gate/up tile belongs to a CTA that never waits
// before it, and with one resident CTA per SM the waits end.
//
// Tiles, stages and roles are those of gemm_w8a8.cu: warp 0 TMA producer (A 128 rows x 128
// codes, B 256 rows x 128 codes, 4 stages of 48 KB), warp 1 MMA issuer (tcgen05.mma
// kind::f8f6f4, M=128, N=256, K=32), warps 2-9 epilogue (row and column scales on the float32
// accumulator, staged whole-sector bf16 stores). The epilogue warps meet at named barriers, so
// they all take one snapshot of the abort flag at the start of every tile and leave together.
#include "epilogue.cuh"
#include "fp8_quant.cuh"
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
using gemm::pack_bf16;
using gemm::silu_f;

constexpr int kBM = 128;
constexpr int kBK = 128;                          // codes per k-step: one 128-byte swizzle atom
constexpr int kEpiWarps = 8;
constexpr int kEpiThreads = 32 * kEpiWarps;
constexpr int kThreads = 64 + kEpiThreads;
constexpr int kABytes = kBM * kBK;                // 16 KB
constexpr int kBBytes = 256 * kBK;                // 32 KB
constexpr int kStageBytes = kABytes + kBBytes;
constexpr int kStages = 4;
constexpr int kTmemCols = 512;
constexpr int kSchedInts = 4 * (kMaxExperts + 2);
constexpr size_t kStgOff = (size_t)kStages * kStageBytes + 256 + (((size_t)kSchedInts * 4 + 127) / 128) * 128;
constexpr size_t kSmem = 1024 + kStgOff + (size_t)kEpiWarps * epi::kStageOutBytes;

__host__ __device__ constexpr uint32_t idesc_e4m3_f32(int M, int N) {
  return (1u << 4) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ void mma_e4m3(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                         uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

__device__ __forceinline__ void fence_proxy_async_global() { asm volatile("fence.proxy.async.global;" ::: "memory"); }
__device__ __forceinline__ void red_release_add(int32_t* p, int v) {
  asm volatile("red.release.gpu.global.add.s32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ int atom_acq_rel_add(int32_t* p, int v) {
  int old;
  asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}
__device__ __forceinline__ int ld_acquire(const int32_t* p) {
  int v;
  asm volatile("ld.acquire.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
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
// the eight epilogue warps (threads 64 .. 319)
__device__ __forceinline__ void epi_bar() { asm volatile("bar.sync 1, %0;" ::"r"(kEpiThreads) : "memory"); }

struct W8FusedArgs {
  int K1, K2;             // reductions: d (gate/up), d_ff (down)
  int nt1, nt2;           // n-tiles per group: d_ff / 128, d / 256
  int G, F, d;
  const int32_t* sched;
  const float* x8_scale;  // [rows] scales of the x codes
  const float* wg_s;      // [G, F]
  const float* wu_s;      // [G, F]
  const float* wd_s;      // [G, d]
  __nv_bfloat16* h;       // [rows, F] bf16 h
  uint8_t* h8;            // [rows, F] its codes
  float* h8_scale;        // [rows]
  __nv_bfloat16* y;       // [rows, d]
  int32_t* done;          // [m-tiles] gate/up tiles finished
  int32_t* quant;         // [m-tiles] 1 once the m-tile's h rows are quantised
  int32_t* status;
};

__global__ void __launch_bounds__(kThreads, 1)
grouped_mlp_w8a8_fused_kernel(const __grid_constant__ CUtensorMap tmX8, const __grid_constant__ CUtensorMap tmWg,
                              const __grid_constant__ CUtensorMap tmWu, const __grid_constant__ CUtensorMap tmH8,
                              const __grid_constant__ CUtensorMap tmWd, const W8FusedArgs args) {
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
  volatile int* s_stop = abort_flag + 1;       // the epilogue's snapshot of the abort flag
  volatile int* s_last = abort_flag + 2;       // this gate/up tile completed its m-tile
  int32_t* s_tile_start = reinterpret_cast<int32_t*>(smem + (size_t)kStages * kStageBytes + 256);
  int32_t* s_out_row = s_tile_start + (args.G + 1) + args.G;
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
      ptx::mbar_init(ptx::smem_u32(&tempty[a]), kEpiThreads);
    }
    ptx::mbar_init(ptx::smem_u32(drain), 1);
    *abort_flag = 0;
    ptx::fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    ptx::prefetch_tmap(&tmX8);
    ptx::prefetch_tmap(&tmWg);
    ptx::prefetch_tmap(&tmWu);
    ptx::prefetch_tmap(&tmH8);
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
        const int a_row = s_out_row[g] + m * kBM;   // x codes and h codes sit at the output rows
        int b_row, k_steps;
        const void* map_a;
        const void* map_b;
        if (up) {
          map_a = &tmX8;
          map_b = &tmWg;
          b_row = g * args.F + n * 128;
          k_steps = args.K1 / kBK;
        } else {
          if (!wait_count(args.quant + s_tile_start[g] + m, 1, abort_flag, kWaitLimitNs)) {
            ok = false;
            break;
          }
          fence_proxy_async_global();
          map_a = &tmH8;
          map_b = &tmWd;
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
          if (up) ptx::tma_load_2d(sb + 128 * kBK, &tmWu, kb * kBK, b_row, fb);
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
      constexpr uint32_t idesc = idesc_e4m3_f32(kBM, 256);
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
          for (int kk = 0; kk < kBK / 32; ++kk)
            mma_e4m3(d_tmem, a_desc + (uint64_t)(2 * kk), b_desc + (uint64_t)(2 * kk), idesc, (kb | kk) != 0 ? 1u : 0u);
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
    const int et = threadIdx.x - 64;                 // 0 .. 255
    const int ew = warp - 2;                         // 0 .. 7
    const int quarter = warp & 3;
    const int half = ew >> 2;
    const uint32_t stg = stg_base + (uint32_t)ew * epi::kStageOutBytes;
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
      }
      // all eight warps leave on the same snapshot of the abort flag
      epi_bar();
      if (et == 0) *s_stop = *abort_flag;
      epi_bar();
      if (*s_stop != 0) break;
      ptx::tc_fence_after();
      const int mt = s_tile_start[g] + m;
      const int row0 = m * kBM + quarter * 32;
      const int nvalid = s_rows[g] - row0;
      const int64_t orow = (int64_t)s_out_row[g] + row0;
      const uint32_t t_row = tmem_base + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(acc * 256);
      if (up) {
        if (nvalid > 0) {
          const float sa = (lane < nvalid) ? args.x8_scale[orow + lane] : 0.0f;
          __nv_bfloat16* orow0 = args.h + orow * args.F + (int64_t)n * 128;
#pragma unroll 1
          for (int c = half * 64; c < half * 64 + 64; c += 32) {
            const float* sg = args.wg_s + (int64_t)g * args.F + n * 128 + c;
            const float* su = args.wu_s + (int64_t)g * args.F + n * 128 + c;
            uint32_t gv[32], uv[32];
            ptx::tmem_ld32(t_row + c, gv);
            ptx::tmem_ld32(t_row + 128 + c, uv);
            ptx::tmem_ld_wait();
            uint32_t packed[16];
#pragma unroll
            for (int q = 0; q < 16; ++q) {
              const float g0 = __uint_as_float(gv[2 * q]) * (sa * __ldg(sg + 2 * q));
              const float g1 = __uint_as_float(gv[2 * q + 1]) * (sa * __ldg(sg + 2 * q + 1));
              const float u0 = __uint_as_float(uv[2 * q]) * (sa * __ldg(su + 2 * q));
              const float u1 = __uint_as_float(uv[2 * q + 1]) * (sa * __ldg(su + 2 * q + 1));
              packed[q] = pack_bf16(silu_f(g0) * u0, silu_f(g1) * u1);
            }
            epi::store_chunk(packed, nvalid, orow0, args.F, c, stg, lane);
          }
        }
        // count this tile on its m-tile; the tile that completes the count quantises the m-tile
        __threadfence();
        ptx::tc_fence_before();
        epi_bar();
        if (et == 0) *s_last = (atom_acq_rel_add(args.done + mt, 1) == args.nt1 - 1) ? 1 : 0;
        epi_bar();
        if (*s_last) {
          const int rows = min(kBM, s_rows[g] - m * kBM);
          const int64_t base = (int64_t)s_out_row[g] + m * kBM;
          for (int r = ew; r < rows; r += kEpiWarps)
            quantize_row_e4m3_warp<true>(args.h + (base + r) * args.F, args.F, args.h8 + (base + r) * args.F,
                                         args.h8_scale + base + r, lane);
          // the codes are read by TMA (async proxy), the scales by generic loads
          fence_proxy_async_global();
          __threadfence();
          epi_bar();
          if (et == 0) red_release_add(args.quant + mt, 1);
        }
      } else {
        if (nvalid > 0) {
          // the m-tile's scales were written by the CTA that quantised it
          if (lane == 0) (void)ld_acquire(args.quant + mt);
          __syncwarp();
          const float sa = (lane < nvalid) ? __ldcg(args.h8_scale + orow + lane) : 0.0f;
          __nv_bfloat16* orow0 = args.y + orow * args.d + (int64_t)n * 256;
#pragma unroll 1
          for (int c = half * 128; c < half * 128 + 128; c += 32) {
            const float* sd = args.wd_s + (int64_t)g * args.d + n * 256 + c;
            uint32_t v[32];
            ptx::tmem_ld32(t_row + c, v);
            ptx::tmem_ld_wait();
            uint32_t packed[16];
#pragma unroll
            for (int q = 0; q < 16; ++q)
              packed[q] = pack_bf16(__uint_as_float(v[2 * q]) * (sa * __ldg(sd + 2 * q)),
                                    __uint_as_float(v[2 * q + 1]) * (sa * __ldg(sd + 2 * q + 1)));
            epi::store_chunk(packed, nvalid, orow0, args.d, c, stg, lane);
          }
        }
      }
      ptx::tc_fence_before();
      ptx::mbar_arrive(ptx::smem_u32(&tempty[acc]));
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

cudaError_t launch_mlp_w8a8_fused(const Shape& s, const uint8_t* x8, const float* x8_scale, const uint8_t* wg_q,
                                  const float* wg_s, const uint8_t* wu_q, const float* wu_s, const uint8_t* wd_q,
                                  const float* wd_s, const void* sched, void* h, uint8_t* h8, float* h8_scale,
                                  void* y, int32_t* counters, int32_t* status, cudaStream_t st) {
  CUtensorMap tx, twg, twu, th, twd;
  const uint64_t rows = (uint64_t)s.R + (uint64_t)s.S * s.T;
  if (!make_tmap_u8_sw128(&tx, x8, s.d, rows > 0 ? rows : 1, kBM)) return cudaErrorInvalidValue;
  if (!make_tmap_u8_sw128(&twg, wg_q, s.d, (uint64_t)s.G * s.F, 128)) return cudaErrorInvalidValue;
  if (!make_tmap_u8_sw128(&twu, wu_q, s.d, (uint64_t)s.G * s.F, 128)) return cudaErrorInvalidValue;
  if (!make_tmap_u8_sw128(&th, h8, s.F, rows > 0 ? rows : 1, kBM)) return cudaErrorInvalidValue;
  if (!make_tmap_u8_sw128(&twd, wd_q, s.F, (uint64_t)s.G * s.d, 256)) return cudaErrorInvalidValue;
  const int64_t mtiles = max_m_tiles(s);
  W8FusedArgs args{};
  args.K1 = s.d;
  args.K2 = s.F;
  args.nt1 = s.F / 128;
  args.nt2 = s.d / 256;
  args.G = s.G;
  args.F = s.F;
  args.d = s.d;
  args.sched = static_cast<const int32_t*>(sched);
  args.x8_scale = x8_scale;
  args.wg_s = wg_s;
  args.wu_s = wu_s;
  args.wd_s = wd_s;
  args.h = static_cast<__nv_bfloat16*>(h);
  args.h8 = h8;
  args.h8_scale = h8_scale;
  args.y = static_cast<__nv_bfloat16*>(y);
  args.done = counters;
  args.quant = counters + mtiles;
  args.status = status;
  cudaError_t e = cudaMemsetAsync(counters, 0, (size_t)2 * mtiles * sizeof(int32_t), st);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(grouped_mlp_w8a8_fused_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmem);
  if (e != cudaSuccess) return e;
  int64_t grid = num_sms();
  const int64_t max_tiles = mtiles * (args.nt1 + args.nt2);
  if (max_tiles < grid) grid = max_tiles;
  if (grid < 1) grid = 1;
  grouped_mlp_w8a8_fused_kernel<<<(unsigned)grid, kThreads, kSmem, st>>>(tx, twg, twu, th, twd, args);
  return cudaGetLastError();
}

}  // namespace moe
