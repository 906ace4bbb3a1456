// Grouped expert GEMMs on the 5th-generation tensor cores (tcgen05 + TMEM),
// fed by TMA over a per-expert tile schedule.
//
// The MoE layer sorts tokens by the expert they go to, multiplies each expert's
// batch in grouped GEMMs and restores token order afterwards (klaylearn.com/glossary/
// mixture-of-experts, "Mixture of Experts", definition). The expert is a SwiGLU
// MLP y = W_down (silu(W_gate a) * (W_up a)); this file holds its two
// contractions:
//   gate/up : per group g, h[rows_g, F] = silu(A_g W_gate[g]^T) * (A_g W_up[g]^T)
//             (A_g = the group's x_perm rows; the shared expert reads x itself)
//   down    : per group g, y[rows_g, d] = h_g W_down[g]^T
//
// Two kernels share one structure (persistent, 320 threads, warp-specialised):
//   warp 0      TMA producer into a ring of shared-memory stages (bf16, K-major,
//               128-byte swizzle, 64 elements of K per stage)
//   warp 1      MMA issuer: tcgen05.mma kind::f16, K=16 (x4 per stage) into one of
//               two TMEM accumulators of 256 float32 columns
//   warps 2-9   epilogue: tcgen05.ld the accumulator (one row per thread; two
//               warps per 32-lane TMEM quarter, each storing half of the tile's
//               output columns), SwiGLU or plain convert, bf16 stores of the
//               valid rows
// For gate/up the B operand is the 128 W_gate rows and the 128 W_up rows of the
// same output columns, so one N=256 MMA yields both projections side by side in
// TMEM and the SwiGLU is fused into the epilogue. The two TMEM accumulators let
// the epilogue of tile i overlap the MMAs of tile i+1.
//
// Pair kernel (selected with MOE_GEMM_PAIRS=1). CTAs run in clusters of two on a pair of SMs and
// compute 256-row tiles with the 2-SM MMA (tcgen05 .cta_group::2, M=256, N=256):
// each CTA loads its own 128 rows of A and its half of B (gate/up: rank 0 the
// W_gate rows, rank 1 the W_up rows; down: 128 of the 256 W_down rows), and the
// MMA issued by rank 0 reads both CTAs' shared memory and writes each CTA's 128
// accumulator rows into that CTA's TMEM. A stage is 32 KB per SM instead of the
// 48 KB a single-CTA 128x256 tile needs, and the MMA instructions per FLOP halve.
// The loads of both
// CTAs complete on rank 0's stage barrier; rank 0's MMA thread releases each
// stage and each finished accumulator to both CTAs with multicast commits, and
// the epilogue threads of both CTAs release an accumulator on rank 0's barrier.
// A group's rows are covered by 256-row tiles; rows past the group's end are
// computed and discarded.
//
// Single-CTA kernel (the default): 128 x 256 tiles (down with d not a multiple of
// 256: 128 x 128) and cta_group::1; also the fallback where clusters of two cannot
// be scheduled.
//
// Tiles are ordered (group, n-tile, m-tile): neighbouring CTAs share the same
// weight columns, so each expert's weights stream from HBM about once while its
// activation rows are re-read from L2.
//
// Every wait is bounded: a stall records MOE_ERR_TIMEOUT, all roles leave their
// loops, in-flight copies and MMAs are drained with bounded waits, and the TMEM
// is freed before the CTA exits. Pair CTAs meet at a cluster barrier before
// freeing TMEM (collectively) and leaving, so neither leaves while the other may
// still use its shared memory or barriers.
#include <cstdlib>
#include <mutex>

#include "internal.cuh"
#include "tc_ptx.cuh"
#include "tmap.cuh"
#include "gemm_common.cuh"
#include "epilogue.cuh"

namespace moe {
namespace {

constexpr int kBM = 128;
constexpr int kBK = 64;              // one 128-byte swizzle atom of bf16
constexpr int kEpiWarps = 8;         // two per 32-lane TMEM quarter
constexpr int kThreads = 64 + 32 * kEpiWarps;
using gemm::kWaitLimitNs;
using gemm::kDrainLimitNs;
using gemm::decode_tile;
using gemm::silu_f;
using gemm::pack_bf16;
using gemm::drain_fills;
constexpr int kSchedInts = 5 * (kMaxExperts + 2);    // schedule + a tile prefix, in shared memory

struct GemmArgs {
  int K;                // reduction length
  int n_tiles;          // N tiles per group
  int G;                // groups
  int shared_from;      // groups >= shared_from read A from the second A map (gate/up only)
  int b_rows;           // rows of B per group (F for gate/up, d for down)
  const int32_t* sched; // device group schedule
  __nv_bfloat16* out;
  int64_t ldo;          // elements per output row
  int32_t* status;
  // MODE 2 (down projection with the combine in its epilogue) only:
  const int32_t* src_token;   // [R] token of each routed row
  const int32_t* dest_row;    // [T, k] grouped row of each (token, slot), -1 if dropped
  const float* gate;          // [T, k] gates
  float* acc_out;             // [T, d] float32 output accumulator, zeroed before the launch
  int k;                      // slots per token
  int routed_groups;          // E: groups >= E are the shared expert (weight one, row = token)
};

using epi::kStageOutBytes;
using epi::ld_shared_v4;
using epi::st_shared_v4;

__device__ __forceinline__ void red_add_v4(float* p, float a, float b, float c, float d) {
  asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(p), "f"(a), "f"(b), "f"(c), "f"(d)
               : "memory");
}

// Epilogue of MODE 2: the warp's 32 accumulator rows (this thread holds row `lane`; each row
// is one (token, slot) pair, or one token of the shared expert) times their gates, added into
// the tokens' float32 output rows. `arow` is this thread's row pointer (already offset to the
// tile's first column), `ok` whether its row is added at all. Columns [half * COLS/2, ...).
// As in store_tile, each 16-column piece goes through the warp's 2 KB staging buffer so that
// one reduction instruction covers 8 rows x 64 contiguous bytes (whole sectors) instead of
// 32 rows x 16 bytes; the row pointers and flags of other lanes come by shuffle.
template <int COLS>
__device__ __forceinline__ void combine_tile(uint32_t t_row, bool ok, float* arow, float gw, int half, uint32_t stg,
                                             int lane) {
  if (!__any_sync(0xffffffffu, ok)) return;
  const int c0 = half * (COLS / 2), c1 = c0 + COLS / 2;
  const uint32_t my_row = stg + (uint32_t)lane * 64u;
  const uint32_t sw = (uint32_t)((lane >> 1) & 3);
  const int j = lane & 3;
#pragma unroll 1
  for (int c = c0; c < c1; c += 32) {
    uint32_t v[32];
    ptx::tmem_ld32(t_row + c, v);
    ptx::tmem_ld_wait();
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
#pragma unroll
      for (int p = 0; p < 4; ++p)
        st_shared_v4(my_row + ((p ^ sw) << 4), __float_as_uint(gw * __uint_as_float(v[16 * hh + 4 * p])),
                     __float_as_uint(gw * __uint_as_float(v[16 * hh + 4 * p + 1])),
                     __float_as_uint(gw * __uint_as_float(v[16 * hh + 4 * p + 2])),
                     __float_as_uint(gw * __uint_as_float(v[16 * hh + 4 * p + 3])));
      __syncwarp();
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int r = 8 * q + (lane >> 2);
        const uint4 u = ld_shared_v4(stg + (uint32_t)r * 64u + ((uint32_t)(j ^ ((r >> 1) & 3)) << 4));
        float* dst = reinterpret_cast<float*>(__shfl_sync(0xffffffffu, reinterpret_cast<uintptr_t>(arow), r));
        const bool rok = __shfl_sync(0xffffffffu, ok ? 1 : 0, r) != 0;
        if (rok)
          red_add_v4(dst + c + 16 * hh + 4 * j, __uint_as_float(u.x), __uint_as_float(u.y), __uint_as_float(u.z),
                     __uint_as_float(u.w));
      }
      __syncwarp();
    }
  }
}

// =====================================================================================
// Single-CTA kernel
// =====================================================================================
template <int MODE, int BN>
struct Cfg {
  static constexpr int kNmma = (MODE == 0) ? 256 : BN;            // MMA N
  static constexpr int kOutCols = (MODE == 0) ? 128 : BN;         // output columns per tile
  static constexpr int kABytes = kBM * kBK * 2;                    // 16 KB
  static constexpr int kBBytes = kNmma * kBK * 2;
  static constexpr int kStageBytes = kABytes + kBBytes;
  static constexpr int kStages = (kStageBytes <= 32768) ? 6 : 4;
  static constexpr int kTmemCols = 2 * kNmma;                      // two accumulators
  static constexpr size_t kStgOff = (size_t)kStages * kStageBytes + 256 + (((size_t)kSchedInts * 4 + 127) / 128) * 128;
  static constexpr size_t kSmem = 1024 /*alignment slack*/ + kStgOff + (size_t)kEpiWarps * kStageOutBytes;
};

template <int MODE, int BN>
__global__ void __launch_bounds__(kThreads, 1)
grouped_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmA2,
                    const __grid_constant__ CUtensorMap tmB, const __grid_constant__ CUtensorMap tmB2,
                    const GemmArgs args) {
  using C = Cfg<MODE, BN>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_u32 = ptx::smem_u32(smem_raw);
  uint8_t* smem = smem_raw + ((1024u - (raw_u32 & 1023u)) & 1023u);   // 1024-byte aligned
  uint8_t* stage_base = smem;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + (size_t)C::kStages * C::kStageBytes);
  uint64_t* full = bars;                       // [kStages]
  uint64_t* empty = bars + C::kStages;         // [kStages]
  uint64_t* tfull = bars + 2 * C::kStages;     // [2]
  uint64_t* tempty = tfull + 2;                // [2]
  uint64_t* drain = tempty + 2;                // [1]
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);
  int32_t* s_tile_start = reinterpret_cast<int32_t*>(smem + (size_t)C::kStages * C::kStageBytes + 256);
  int32_t* s_a_row = s_tile_start + (args.G + 1);
  int32_t* s_out_row = s_a_row + args.G;
  int32_t* s_rows = s_out_row + args.G;
  const uint32_t stg_base = ptx::smem_u32(smem + C::kStgOff);   // epilogue staging, 2 KB per warp

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  // schedule -> shared memory
  for (int i = threadIdx.x; i < 4 * args.G + 1; i += kThreads) s_tile_start[i] = args.sched[i];
  if (threadIdx.x == 0) {
    for (int s = 0; s < C::kStages; ++s) {
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
    ptx::prefetch_tmap(&tmA);
    ptx::prefetch_tmap(&tmB);
    if (MODE == 0) {
      ptx::prefetch_tmap(&tmA2);
      ptx::prefetch_tmap(&tmB2);
    }
  }
  if (warp == 1) {
    ptx::tmem_alloc(ptx::smem_u32(tmem_holder), C::kTmemCols);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem_base = *tmem_holder;

  const int total_tiles = s_tile_start[args.G] * args.n_tiles;
  const int k_steps = args.K / kBK;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      int issued = 0;              // loads issued (saturating at kStages)
      bool ok = true;
      for (int L = blockIdx.x; L < total_tiles && ok; L += gridDim.x) {
        int g, m, n;
        decode_tile(L, s_tile_start, args.G, args.n_tiles, g, m, n);
        const bool use_a2 = (MODE == 0) && (g >= args.shared_from);
        const int a_row = ((MODE == 0) ? s_a_row[g] : s_out_row[g]) + m * kBM;
        const int b_row = g * args.b_rows + n * ((MODE == 0) ? 128 : BN);
        for (int kb = 0; kb < k_steps; ++kb) {
          if (!ptx::mbar_wait_bounded(ptx::smem_u32(&empty[stage]), phase ^ 1u, abort_flag, kWaitLimitNs)) {
            ok = false;
            break;
          }
          const uint32_t fb = ptx::smem_u32(&full[stage]);
          const uint32_t sa = ptx::smem_u32(stage_base + (size_t)stage * C::kStageBytes);
          const uint32_t sb = sa + C::kABytes;
          ptx::mbar_arrive_expect_tx(fb, C::kStageBytes);
          ptx::tma_load_2d(sa, use_a2 ? (const void*)&tmA2 : (const void*)&tmA, kb * kBK, a_row, fb);
          ptx::tma_load_2d(sb, &tmB, kb * kBK, b_row, fb);
          if (MODE == 0) ptx::tma_load_2d(sb + 128 * 128, &tmB2, kb * kBK, b_row, fb);
          if (issued < C::kStages) ++issued;
          if (++stage == C::kStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (!ok) {
        set_status(args.status, MOE_ERR_TIMEOUT);
        *abort_flag = 1;
        drain_fills(full, C::kStages, stage, phase, issued);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc = ptx::idesc_bf16_f32(kBM, C::kNmma);
      int stage = 0;
      uint32_t phase = 0;
      int it = 0;
      bool ok = true;
      for (int L = blockIdx.x; L < total_tiles && ok; L += gridDim.x, ++it) {
        const int acc = it & 1;
        const uint32_t acc_phase = (uint32_t)(it >> 1) & 1u;
        if (!ptx::mbar_wait_bounded(ptx::smem_u32(&tempty[acc]), acc_phase ^ 1u, abort_flag, kWaitLimitNs)) {
          ok = false;
          break;
        }
        ptx::tc_fence_after();
        const uint32_t d_tmem = tmem_base + (uint32_t)(acc * C::kNmma);
        for (int kb = 0; kb < k_steps; ++kb) {
          if (!ptx::mbar_wait_bounded(ptx::smem_u32(&full[stage]), phase, abort_flag, kWaitLimitNs)) {
            ok = false;
            break;
          }
          ptx::tc_fence_after();
          const uint32_t sa = ptx::smem_u32(stage_base + (size_t)stage * C::kStageBytes);
          const uint64_t a_desc = ptx::sw128_kmajor_desc(sa);
          const uint64_t b_desc = ptx::sw128_kmajor_desc(sa + C::kABytes);
#pragma unroll
          for (int kk = 0; kk < kBK / 16; ++kk) {
            // advance 16 bf16 = 32 bytes along K inside the swizzle atom
            ptx::mma_bf16(d_tmem, a_desc + (uint64_t)(2 * kk), b_desc + (uint64_t)(2 * kk), idesc,
                          (kb | kk) != 0 ? 1u : 0u);
          }
          ptx::mma_commit(ptx::smem_u32(&empty[stage]));
          if (++stage == C::kStages) {
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
      // all MMAs issued by this thread complete before TMEM is released
      ptx::mma_commit(ptx::smem_u32(drain));
      ptx::mbar_wait_bounded(ptx::smem_u32(drain), 0, nullptr, kDrainLimitNs);
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int quarter = warp & 3;            // TMEM lanes this warp may access
    const int half = (warp - 2) >> 2;        // which half of the output columns
    const int r_local = quarter * 32 + lane; // accumulator row == TMEM lane
    int it = 0;
    for (int L = blockIdx.x; L < total_tiles; L += gridDim.x, ++it) {
      int g, m, n;
      decode_tile(L, s_tile_start, args.G, args.n_tiles, g, m, n);
      const int acc = it & 1;
      const uint32_t acc_phase = (uint32_t)(it >> 1) & 1u;
      if (!ptx::mbar_wait_bounded(ptx::smem_u32(&tfull[acc]), acc_phase, abort_flag, kWaitLimitNs)) {
        set_status(args.status, MOE_ERR_TIMEOUT);
        *abort_flag = 1;
        break;
      }
      ptx::tc_fence_after();
      const bool valid = (m * kBM + r_local) < s_rows[g];
      const int64_t out_row = (int64_t)s_out_row[g] + m * kBM + r_local;
      const uint32_t t_row = tmem_base + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(acc * C::kNmma);
      if constexpr (MODE == 2) {
        // the pair's token and gate: the slot of the token whose dest_row names this row
        int tok = 0;
        float gw = 0.0f;
        bool ok_row = valid;
        if (valid) {
          if (g >= args.routed_groups) {
            tok = m * kBM + r_local;
            gw = 1.0f;
          } else {
            tok = args.src_token[out_row];
            ok_row = false;
            for (int j = 0; j < args.k; ++j)
              if (args.dest_row[(int64_t)tok * args.k + j] == (int32_t)out_row) {
                gw = args.gate[(int64_t)tok * args.k + j];
                ok_row = true;
              }
            if (!ok_row) set_status(args.status, MOE_ERR_DEVICE_INDEX);
          }
        }
        combine_tile<C::kOutCols>(t_row, ok_row, args.acc_out + (int64_t)tok * args.ldo + (int64_t)n * C::kOutCols,
                                  gw, half, stg_base + (uint32_t)(warp - 2) * kStageOutBytes, lane);
      } else {
        const int row0 = m * kBM + quarter * 32;                // the warp's first row in the group
        __nv_bfloat16* orow0 = args.out + ((int64_t)s_out_row[g] + row0) * args.ldo + (int64_t)n * C::kOutCols;
        epi::store_tile<MODE == 0, C::kOutCols>(t_row, s_rows[g] - row0, orow0, args.ldo, half,
                                                stg_base + (uint32_t)(warp - 2) * kStageOutBytes, lane);
      }
      ptx::tc_fence_before();
      ptx::mbar_arrive(ptx::smem_u32(&tempty[acc]));
    }
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem_base, C::kTmemCols);
  }
}

// =====================================================================================
// Pair kernel (2-SM MMA)
// =====================================================================================
template <int MODE>
struct PairCfg {
  static constexpr int kN = 256;                                   // MMA N of the pair
  static constexpr int kOutCols = (MODE == 0) ? 128 : 256;         // output columns per tile
  static constexpr int kABytes = kBM * kBK * 2;                    // this CTA's 128 A rows: 16 KB
  static constexpr int kBBytes = 128 * kBK * 2;                    // this CTA's half of B: 16 KB
  static constexpr int kStageBytes = kABytes + kBBytes;            // 32 KB
  static constexpr int kStages = 6;
  static constexpr int kTmemCols = 2 * kN;                         // two accumulators (512)
  static constexpr size_t kStgOff = (size_t)kStages * kStageBytes + 256 + (((size_t)kSchedInts * 4 + 127) / 128) * 128;
  static constexpr size_t kSmem = 1024 + kStgOff + (size_t)kEpiWarps * kStageOutBytes;
};

template <int MODE>
__global__ void __launch_bounds__(kThreads, 1)
grouped_gemm_pair_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmA2,
                         const __grid_constant__ CUtensorMap tmB, const __grid_constant__ CUtensorMap tmB2,
                         const GemmArgs args) {
  using C = PairCfg<MODE>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_u32 = ptx::smem_u32(smem_raw);
  uint8_t* smem = smem_raw + ((1024u - (raw_u32 & 1023u)) & 1023u);   // 1024-byte aligned
  uint8_t* stage_base = smem;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + (size_t)C::kStages * C::kStageBytes);
  uint64_t* full = bars;                       // [kStages]  rank 0's count both CTAs' loads
  uint64_t* empty = bars + C::kStages;         // [kStages]  released by rank 0's MMA thread
  uint64_t* tfull = bars + 2 * C::kStages;     // [2]        accumulator ready (both CTAs)
  uint64_t* tempty = tfull + 2;                // [2]        rank 0's: both CTAs' epilogues done
  uint64_t* drain = tempty + 2;                // [1]
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);
  int32_t* s_tile_start = reinterpret_cast<int32_t*>(smem + (size_t)C::kStages * C::kStageBytes + 256);
  int32_t* s_a_row = s_tile_start + (args.G + 1);
  int32_t* s_out_row = s_a_row + args.G;
  int32_t* s_rows = s_out_row + args.G;
  int32_t* s_pair_start = s_rows + args.G;     // [G+1] prefix of 256-row tiles per group
  const uint32_t stg_base = ptx::smem_u32(smem + C::kStgOff);   // epilogue staging, 2 KB per warp

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int rank = (int)ptx::cluster_ctarank();
  const bool leader = (rank == 0);
  const int unit0 = blockIdx.x >> 1;
  const int unit_step = gridDim.x >> 1;
  constexpr uint16_t kBoth = 0x3;

  for (int i = threadIdx.x; i < 4 * args.G + 1; i += kThreads) s_tile_start[i] = args.sched[i];
  if (threadIdx.x == 0) {
    for (int s = 0; s < C::kStages; ++s) {
      ptx::mbar_init(ptx::smem_u32(&full[s]), 1);
      ptx::mbar_init(ptx::smem_u32(&empty[s]), 1);
    }
    for (int a = 0; a < 2; ++a) {
      ptx::mbar_init(ptx::smem_u32(&tfull[a]), 1);
      ptx::mbar_init(ptx::smem_u32(&tempty[a]), 2 * kEpiWarps * 32);
    }
    ptx::mbar_init(ptx::smem_u32(drain), 1);
    *abort_flag = 0;
    ptx::fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    ptx::prefetch_tmap(&tmA);
    ptx::prefetch_tmap(&tmB);
    if (MODE == 0) {
      ptx::prefetch_tmap(&tmA2);
      ptx::prefetch_tmap(&tmB2);
    }
  }
  if (warp == 1) {
    // collective with the peer CTA's warp 1: both get the same TMEM columns
    ptx::tmem_alloc_pair(ptx::smem_u32(tmem_holder), C::kTmemCols);
    ptx::tmem_relinquish_pair();
  }
  __syncthreads();
  if (warp == 2) {
    // 256-row tiles per group, prefix-summed 32 groups at a time
    int carry = 0;
    for (int base = 0; base < args.G; base += 32) {
      const int g = base + lane;
      int pt = 0;
      if (g < args.G) pt = (s_tile_start[g + 1] - s_tile_start[g] + 1) >> 1;
      int incl = pt;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
      }
      if (g < args.G) s_pair_start[g] = carry + incl - pt;
      carry += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (lane == 0) s_pair_start[args.G] = carry;
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::cluster_sync_all();                     // both CTAs' barriers exist before any remote use
  ptx::tc_fence_after();
  const uint32_t tmem_base = *tmem_holder;

  const int total_tiles = s_pair_start[args.G] * args.n_tiles;
  const int k_steps = args.K / kBK;

  if (warp == 0) {
    // ------------------------------------------------------------ producer (both CTAs)
    if (lane == 0) {
      const uint32_t full0 = ptx::smem_u32(full);
      const uint32_t full0_leader = ptx::map_shared_rank(full0, 0);
      int stage = 0;
      uint32_t phase = 0;
      int issued = 0;
      bool ok = true;
      for (int L = unit0; L < total_tiles && ok; L += unit_step) {
        int g, p, n;
        decode_tile(L, s_pair_start, args.G, args.n_tiles, g, p, n);
        const int m = 2 * p + rank;            // this CTA's 128-row half of the 256-row tile
        const bool use_a2 = (MODE == 0) && (g >= args.shared_from);
        const int a_row = ((MODE == 0) ? s_a_row[g] : s_out_row[g]) + m * kBM;
        const int b_row = (MODE == 0) ? g * args.b_rows + n * 128 : g * args.b_rows + n * 256 + 128 * rank;
        const void* map_a = use_a2 ? (const void*)&tmA2 : (const void*)&tmA;
        const void* map_b = (MODE == 0 && rank == 1) ? (const void*)&tmB2 : (const void*)&tmB;
        for (int kb = 0; kb < k_steps; ++kb) {
          if (!ptx::mbar_wait_bounded(ptx::smem_u32(&empty[stage]), phase ^ 1u, abort_flag, kWaitLimitNs)) {
            ok = false;
            break;
          }
          const uint32_t sa = ptx::smem_u32(stage_base + (size_t)stage * C::kStageBytes);
          const uint32_t bar = full0_leader + 8u * stage;
          // rank 0's barrier expects the stage bytes of both CTAs
          if (leader) ptx::mbar_arrive_expect_tx(full0 + 8u * stage, 2 * C::kStageBytes);
          ptx::tma_load_2d_pair(sa, map_a, kb * kBK, a_row, bar);
          ptx::tma_load_2d_pair(sa + C::kABytes, map_b, kb * kBK, b_row, bar);
          if (issued < C::kStages) ++issued;
          if (++stage == C::kStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (!ok) {
        set_status(args.status, MOE_ERR_TIMEOUT);
        *abort_flag = 1;
        // rank 0's barriers count both CTAs' fills; rank 1's fills are covered by rank 0's
        // drain before the closing cluster barrier
        if (leader) drain_fills(full, C::kStages, stage, phase, issued);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer (rank 0)
    if (lane == 0 && leader) {
      constexpr uint32_t idesc = ptx::idesc_bf16_f32(2 * kBM, C::kN);
      int stage = 0;
      uint32_t phase = 0;
      int it = 0;
      bool ok = true;
      for (int L = unit0; L < total_tiles && ok; L += unit_step, ++it) {
        const int acc = it & 1;
        const uint32_t acc_phase = (uint32_t)(it >> 1) & 1u;
        if (!ptx::mbar_wait_bounded(ptx::smem_u32(&tempty[acc]), acc_phase ^ 1u, abort_flag, kWaitLimitNs)) {
          ok = false;
          break;
        }
        ptx::tc_fence_after();
        const uint32_t d_tmem = tmem_base + (uint32_t)(acc * C::kN);
        for (int kb = 0; kb < k_steps; ++kb) {
          if (!ptx::mbar_wait_bounded(ptx::smem_u32(&full[stage]), phase, abort_flag, kWaitLimitNs)) {
            ok = false;
            break;
          }
          ptx::tc_fence_after();
          const uint32_t sa = ptx::smem_u32(stage_base + (size_t)stage * C::kStageBytes);
          const uint64_t a_desc = ptx::sw128_kmajor_desc(sa);
          const uint64_t b_desc = ptx::sw128_kmajor_desc(sa + C::kABytes);
#pragma unroll
          for (int kk = 0; kk < kBK / 16; ++kk)
            ptx::mma_bf16_pair(d_tmem, a_desc + (uint64_t)(2 * kk), b_desc + (uint64_t)(2 * kk), idesc,
                               (kb | kk) != 0 ? 1u : 0u);
          // both CTAs' slots are free once these MMAs have read them
          ptx::mma_commit_pair_multicast(ptx::smem_u32(&empty[stage]), kBoth);
          if (++stage == C::kStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        ptx::mma_commit_pair_multicast(ptx::smem_u32(&tfull[acc]), kBoth);
      }
      if (!ok) {
        set_status(args.status, MOE_ERR_TIMEOUT);
        *abort_flag = 1;
      }
      ptx::mma_commit_pair(ptx::smem_u32(drain));
      ptx::mbar_wait_bounded(ptx::smem_u32(drain), 0, nullptr, kDrainLimitNs);
    }
  } else {
    // ------------------------------------------------------------ epilogue (both CTAs)
    const int quarter = warp & 3;
    const int half = (warp - 2) >> 2;
    const uint32_t tempty_leader = ptx::map_shared_rank(ptx::smem_u32(tempty), 0);
    int it = 0;
    for (int L = unit0; L < total_tiles; L += unit_step, ++it) {
      int g, p, n;
      decode_tile(L, s_pair_start, args.G, args.n_tiles, g, p, n);
      const int m = 2 * p + rank;
      const int acc = it & 1;
      const uint32_t acc_phase = (uint32_t)(it >> 1) & 1u;
      if (!ptx::mbar_wait_bounded(ptx::smem_u32(&tfull[acc]), acc_phase, abort_flag, kWaitLimitNs)) {
        set_status(args.status, MOE_ERR_TIMEOUT);
        *abort_flag = 1;
        break;
      }
      ptx::tc_fence_after();
      const int row0 = m * kBM + quarter * 32;
      __nv_bfloat16* orow0 = args.out + ((int64_t)s_out_row[g] + row0) * args.ldo + (int64_t)n * C::kOutCols;
      const uint32_t t_row = tmem_base + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(acc * C::kN);
      epi::store_tile<MODE == 0, C::kOutCols>(t_row, s_rows[g] - row0, orow0, args.ldo, half,
                                              stg_base + (uint32_t)(warp - 2) * kStageOutBytes, lane);
      ptx::tc_fence_before();
      ptx::mbar_arrive_cluster(tempty_leader + 8u * acc);
    }
  }

  ptx::tc_fence_before();
  __syncthreads();
  ptx::cluster_sync_all();                     // the peer is done with this CTA's memory and TMEM
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc_pair(tmem_base, C::kTmemCols);
  }
}

// ------------------------------------------------------------------ host ---
std::mutex g_pair_mu;
int g_pair_fit[2] = {-1, -1};   // [MODE]: 1 if clusters of two fit, 0 if not, -1 unknown

template <int MODE>
bool pairs_fit(const cudaLaunchConfig_t& cfg) {
  std::lock_guard<std::mutex> lock(g_pair_mu);
  int& f = g_pair_fit[MODE];
  if (f < 0) {
    int n = 0;
    f = (cudaOccupancyMaxActiveClusters(&n, grouped_gemm_pair_kernel<MODE>, &cfg) == cudaSuccess && n > 0) ? 1 : 0;
    cudaGetLastError();
  }
  return f == 1;
}

// Which kernel: the single-CTA kernel unless MOE_GEMM_PAIRS=1 (read once per process)
// selects the pair kernel. Measured back to back on one B300, the pair kernel was within a
// few percent of the single-CTA kernel on the tensor-bound layers (all of them run at the
// power limit) and slower where experts have few rows (decode, capacity-limited layers),
// where a 256-row tile doubles the wasted MMA work.
bool want_pairs(const Shape& s) {
  (void)s;
  static const bool forced = [] {
    const char* v = getenv("MOE_GEMM_PAIRS");
    return v != nullptr && v[0] == '1';
  }();
  return forced;
}

int64_t max_m_tiles(const Shape& s) {
  // routed rows R spread over E groups (each may add one partial tile) + shared rows
  return (s.R + kBM - 1) / kBM + s.E + (int64_t)s.S * ((s.T + kBM - 1) / kBM);
}

int64_t grid_for(int64_t max_units) {
  int64_t grid = num_sms();
  if (max_units < grid) grid = max_units;
  return grid < 1 ? 1 : grid;
}

// Pair kernel when clusters of two can be scheduled; returns cudaErrorNotSupported otherwise.
template <int MODE>
cudaError_t launch_pair(const CUtensorMap& a, const CUtensorMap& a2, const CUtensorMap& b, const CUtensorMap& b2,
                        const GemmArgs& args, int64_t max_pair_tiles, cudaStream_t st) {
  using C = PairCfg<MODE>;
  auto kern = grouped_gemm_pair_kernel<MODE>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)C::kSmem);
  if (e != cudaSuccess) return e;
  int64_t grid = grid_for(2 * max_pair_tiles) / 2 * 2;
  if (grid < 2) grid = 2;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = C::kSmem;
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (!pairs_fit<MODE>(cfg)) return cudaErrorNotSupported;
  e = cudaLaunchKernelEx(&cfg, kern, a, a2, b, b2, args);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

template <int MODE, int BN>
cudaError_t launch_single(const CUtensorMap& a, const CUtensorMap& a2, const CUtensorMap& b, const CUtensorMap& b2,
                          const GemmArgs& args, int64_t max_tiles, cudaStream_t st) {
  using C = Cfg<MODE, BN>;
  auto kern = grouped_gemm_kernel<MODE, BN>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)C::kSmem);
  if (e != cudaSuccess) return e;
  kern<<<(unsigned)grid_for(max_tiles), kThreads, C::kSmem, st>>>(a, a2, b, b2, args);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_gemm_gateup_tc(const Shape& s, const void* x_perm, const void* x, const void* w_gate,
                                  const void* w_up, const void* sched, void* h, int32_t* status, cudaStream_t st) {
  CUtensorMap a, a2, b, b2;
  const uint64_t R = (uint64_t)(s.R > 0 ? s.R : 1);
  if (!make_tmap_bf16(&a, x_perm, s.d, R, kBM)) return cudaErrorInvalidValue;
  if (!make_tmap_bf16(&a2, s.S > 0 ? x : x_perm, s.d, s.S > 0 ? (uint64_t)s.T : R, kBM)) return cudaErrorInvalidValue;
  if (!make_tmap_bf16(&b, w_gate, s.d, (uint64_t)s.G * s.F, 128)) return cudaErrorInvalidValue;
  if (!make_tmap_bf16(&b2, w_up, s.d, (uint64_t)s.G * s.F, 128)) return cudaErrorInvalidValue;
  GemmArgs args{};
  args.K = s.d;
  args.n_tiles = s.F / 128;
  args.G = s.G;
  args.shared_from = s.E;
  args.b_rows = s.F;
  args.sched = static_cast<const int32_t*>(sched);
  args.out = static_cast<__nv_bfloat16*>(h);
  args.ldo = s.F;
  args.status = status;
  const int64_t max_tiles = max_m_tiles(s) * args.n_tiles;
  if (want_pairs(s)) {
    cudaError_t e = launch_pair<0>(a, a2, b, b2, args, max_tiles, st);
    if (e != cudaErrorNotSupported) return e;
  }
  return launch_single<0, 128>(a, a2, b, b2, args, max_tiles, st);
}

cudaError_t launch_gemm_down_tc(const Shape& s, const void* h, const void* w_down, const void* sched, void* y,
                                int32_t* status, cudaStream_t st) {
  CUtensorMap a, b;
  const uint64_t rows = (uint64_t)s.R + (uint64_t)s.S * s.T;
  GemmArgs args{};
  args.K = s.F;
  args.G = s.G;
  args.shared_from = s.G;
  args.b_rows = s.d;
  args.sched = static_cast<const int32_t*>(sched);
  args.out = static_cast<__nv_bfloat16*>(y);
  args.ldo = s.d;
  args.status = status;
  if (!make_tmap_bf16(&a, h, s.F, rows > 0 ? rows : 1, kBM)) return cudaErrorInvalidValue;
  if (s.d % 256 == 0) {
    args.n_tiles = s.d / 256;
    const int64_t max_tiles = max_m_tiles(s) * args.n_tiles;
    // pair kernel: each CTA loads 128 of a tile's 256 W_down rows
    if (want_pairs(s)) {
      if (!make_tmap_bf16(&b, w_down, s.F, (uint64_t)s.G * s.d, 128)) return cudaErrorInvalidValue;
      cudaError_t e = launch_pair<1>(a, a, b, b, args, max_tiles, st);
      if (e != cudaErrorNotSupported) return e;
    }
    if (!make_tmap_bf16(&b, w_down, s.F, (uint64_t)s.G * s.d, 256)) return cudaErrorInvalidValue;
    return launch_single<1, 256>(a, a, b, b, args, max_tiles, st);
  }
  args.n_tiles = s.d / 128;
  if (!make_tmap_bf16(&b, w_down, s.F, (uint64_t)s.G * s.d, 128)) return cudaErrorInvalidValue;
  return launch_single<1, 128>(a, a, b, b, args, max_m_tiles(s) * args.n_tiles, st);
}

cudaError_t launch_gemm_down_combine_tc(const Shape& s, const void* h, const void* w_down, const void* sched,
                                        const int32_t* src_token, const int32_t* dest_row, const float* gate,
                                        float* acc_out, int32_t* status, cudaStream_t st) {
  CUtensorMap a, b;
  const uint64_t rows = (uint64_t)s.R + (uint64_t)s.S * s.T;
  GemmArgs args{};
  args.K = s.F;
  args.G = s.G;
  args.shared_from = s.G;
  args.b_rows = s.d;
  args.sched = static_cast<const int32_t*>(sched);
  args.out = nullptr;
  args.ldo = s.d;
  args.status = status;
  args.src_token = src_token;
  args.dest_row = dest_row;
  args.gate = gate;
  args.acc_out = acc_out;
  args.k = s.k;
  args.routed_groups = s.E;
  if (!make_tmap_bf16(&a, h, s.F, rows > 0 ? rows : 1, kBM)) return cudaErrorInvalidValue;
  if (s.d % 256 == 0) {
    args.n_tiles = s.d / 256;
    if (!make_tmap_bf16(&b, w_down, s.F, (uint64_t)s.G * s.d, 256)) return cudaErrorInvalidValue;
    return launch_single<2, 256>(a, a, b, b, args, max_m_tiles(s) * args.n_tiles, st);
  }
  args.n_tiles = s.d / 128;
  if (!make_tmap_bf16(&b, w_down, s.F, (uint64_t)s.G * s.d, 128)) return cudaErrorInvalidValue;
  return launch_single<2, 128>(a, a, b, b, args, max_m_tiles(s) * args.n_tiles, st);
}

}  // namespace moe
