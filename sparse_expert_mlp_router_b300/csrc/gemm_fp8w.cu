// Grouped expert GEMMs with FP8 (E4M3) expert weights and bf16 activations,
// and the per-row quantiser that produces such weights.
//
// shubhamtatvamasi.com/llm-inference/moe "Mixture of Experts", section
// "Memory vs compute, quantified": the weights of the 671B model are about
// 671 GB in FP8 against 1.3 TB in BF16, and a decode step streams the touched
// experts' weights, so halving their bytes halves the memory-bound part of the
// step. The contraction is the one of gemm_tc.cu (the SwiGLU expert of
// klaylearn.com's "Mixture of Experts" grouped GEMMs) with each weight row
// scaled: W[r][:] = scale[r] * e4m3(wq[r][:]).
//
// Every E4M3 value is exactly a bf16 value, and a per-output-row scale factors
// out of the dot product, so the tensor cores run kind::f16 on bf16 operands:
//   warp 0       TMA producer of the bf16 A tiles (128 x 64) into a 3-stage ring
//   warp 1       MMA issuer (tcgen05 M=128, N=256, K=16), two TMEM accumulators
//   warp 2       TMA producer of the weight codes (256 rows x 64 bytes per k-step)
//                into a 4-slot staging ring, so more DRAM bytes are in flight
//                than the bf16 stages alone would allow
//   warps 3-6    epilogue: per-column scales applied to the float32 accumulator
//                (before the SwiGLU for gate/up), bf16 stores of the valid rows
//   warps 7-22   widen the codes to bf16 into the stage's B region in the
//                128-byte-swizzled K-major layout the MMA reads (the pattern a
//                TMA SWIZZLE_128B load writes: 16-byte chunk c of row r at chunk
//                c ^ (r mod 8)), then a proxy fence and an arrive hand the tile
//                to the tensor cores. Two groups of eight warps take alternate
//                k-steps: a k-step's widening is a chain of waits, shared loads,
//                conversions, stores and a fence that one group cannot shorten,
//                so two chains run at once
// Tiles and bounded waits are those of the bf16 single-CTA kernel.
//
// Decode-shaped layers (at most 8 pairs per expert on average, reduction <= 2048) run a
// resident-token variant: tiles of 8 token rows whose A operand for the whole reduction
// (K/64 boxes of 8 rows x 64 bf16, 1 KB each) is loaded once per tile into its own buffer,
// and the M=128 MMA reads it through a descriptor whose 8-row group stride is 0, so rows
// 8..127 repeat rows 0..7 and are masked in the epilogue. The stages then hold only the
// widened weights, the per-k-step token tile (which otherwise waits behind the SM's code
// reads) disappears, and the freed memory deepens the code ring.
#include <cuda_fp8.h>

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
constexpr int kBK = 64;
constexpr int kStages = 3;                       // (A +) widened B per stage
constexpr int kMaxQSlots = 8;                    // weight-code slots (4 with per-k-step A tiles)
constexpr int kResRows = 8;                      // token rows of a resident-token tile
constexpr int kABytes = kBM * kBK * 2;           // 16 KB
constexpr int kBRows = 256;                      // gate/up: 128 W_gate + 128 W_up rows; down: 256 W_down rows
constexpr int kBBytes = kBRows * kBK * 2;        // 32 KB of bf16
constexpr int kQBytes = kBRows * kBK;            // 16 KB of codes
constexpr int kResBoxBytes = kResRows * kBK * 2; // 1 KB: 8 token rows of one k-step

template <bool RES>
struct FCfg {
  static constexpr int kStageBytes = RES ? kBBytes : kABytes + kBBytes;
  static constexpr int kBOff = RES ? 0 : kABytes;   // B within a stage
  static constexpr int kRows = RES ? kResRows : kBM;  // token rows of a tile
};
constexpr int kEpiWarps = 4;
constexpr int kConvGroups = 2;                   // converter groups, alternate k-steps
constexpr int kConvThreads = 256;                // threads of one converter group
constexpr int kConvWarps = kConvGroups * kConvThreads / 32;
constexpr int kFirstEpiWarp = 3;
constexpr int kFirstConvWarp = kFirstEpiWarp + kEpiWarps;
constexpr int kThreads = 32 * (kFirstConvWarp + kConvWarps);   // 736
constexpr int kSchedInts = 4 * (kMaxExperts + 2);
constexpr size_t kSmemFixed = 1024 /*alignment*/ + 512 /*barriers*/ + 256 * 4 /*column scales*/ +
                              (size_t)kSchedInts * 4;
constexpr size_t kSmemMax = 232448;

struct Fp8Args {
  int K;                 // reduction length
  int n_tiles;           // N tiles per group
  int G;                 // groups
  int shared_from;       // groups >= shared_from read A from the second A map (gate/up only)
  int b_rows;            // weight rows per group (F for gate/up, d for down)
  const int32_t* sched;  // device group schedule
  int qslots;            // weight-code slots (<= kMaxQSlots)
  int res_bytes;         // resident-token buffer (K/64 KB) when tiles are 8 rows, else 0
  const float* scale;    // gate/up: W_gate row scales [G, F]; down: W_down row scales [G, d]
  const float* scale2;   // gate/up: W_up row scales [G, F]
  __nv_bfloat16* out;
  int64_t ldo;
  int32_t* status;
};

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void epi_bar() { asm volatile("bar.sync 1, %0;" ::"r"(32 * kEpiWarps) : "memory"); }

// Two E4M3 codes (low byte first) -> bf16x2 (exact).
__device__ __forceinline__ uint32_t widen2(uint32_t pair) {
  const __half2_raw hr = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(pair & 0xFFFFu), __NV_E4M3);
  const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&hr));
  const __nv_bfloat162 b = __float22bfloat162_rn(f);
  return *reinterpret_cast<const uint32_t*>(&b);
}

// A 128-row tile (not a resident-token tile) whose group has at most 64 rows left: M=64 MMAs,
// half the tensor work; its accumulator rows 16 q .. 16 q + 15 sit in TMEM lanes 32 q .. 32 q + 15.
template <bool RES>
__device__ __forceinline__ bool half_tile(int rows, int m) {
  return !RES && rows - m * kBM <= 64;
}

template <int MODE, bool RES>
__global__ void __launch_bounds__(kThreads, 1)
grouped_gemm_fp8w_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmA2,
                         const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmQ2,
                         const Fp8Args args) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_u32 = ptx::smem_u32(smem_raw);
  uint8_t* smem = smem_raw + ((1024u - (raw_u32 & 1023u)) & 1023u);   // 1024-byte aligned
  using C = FCfg<RES>;
  const int kQStages = args.qslots;
  uint8_t* stage_base = smem;
  uint8_t* code_base = smem + (size_t)kStages * C::kStageBytes;
  uint8_t* a_res = code_base + (size_t)kQStages * kQBytes;            // resident-token tile (RES)
  uint64_t* bars = reinterpret_cast<uint64_t*>(a_res + args.res_bytes);
  uint64_t* full = bars;                       // [kStages] A landed (per-k-step A tiles)
  uint64_t* conv = full + kStages;             // [kStages] B widened
  uint64_t* empty = conv + kStages;            // [kStages] stage read by the MMAs
  uint64_t* qfull = empty + kStages;           // [qslots] codes landed
  uint64_t* qempty = qfull + kMaxQSlots;       // [qslots] codes read by the converters
  uint64_t* tfull = qempty + kMaxQSlots;       // [2]
  uint64_t* tempty = tfull + 2;                // [2]
  uint64_t* drain = tempty + 2;                // [1]
  uint64_t* afull = drain + 1;                 // [1] resident-token tile landed (RES)
  uint64_t* aempty = afull + 1;                // [1] resident-token tile read by the MMAs (RES)
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(aempty + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);
  volatile int* s_stop = reinterpret_cast<volatile int*>(tmem_holder + 2);   // epilogue's snapshot
  float* s_scale = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(bars) + 512);   // [256]
  int32_t* s_tile_start = reinterpret_cast<int32_t*>(s_scale + 256);
  int32_t* s_a_row = s_tile_start + (args.G + 1);
  int32_t* s_out_row = s_a_row + args.G;
  int32_t* s_rows = s_out_row + args.G;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  // The schedule's rows, and a prefix of this kernel's m-tiles (C::kRows token rows each).
  for (int i = args.G + 1 + threadIdx.x; i < 4 * args.G + 1; i += kThreads) s_tile_start[i] = args.sched[i];
  if (warp == 0) {
    const int32_t* n_rows = args.sched + (args.G + 1) + 2 * args.G;
    int carry = 0;
    for (int base = 0; base < args.G; base += 32) {
      const int g = base + lane;
      const int r = g < args.G ? n_rows[g] : 0;
      const int tiles = (r + C::kRows - 1) / C::kRows;
      int incl = tiles;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
      }
      if (g < args.G) s_tile_start[g] = carry + incl - tiles;
      carry += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (lane == 0) s_tile_start[args.G] = carry;
  }
  if (threadIdx.x == 0) {
    ptx::mbar_init(ptx::smem_u32(afull), 1);
    ptx::mbar_init(ptx::smem_u32(aempty), 1);
    for (int s = 0; s < kStages; ++s) {
      ptx::mbar_init(ptx::smem_u32(&full[s]), 1);
      ptx::mbar_init(ptx::smem_u32(&conv[s]), kConvThreads / 32);      // one arrive per converter warp
      ptx::mbar_init(ptx::smem_u32(&empty[s]), 1);
    }
    for (int q = 0; q < kQStages; ++q) {
      ptx::mbar_init(ptx::smem_u32(&qfull[q]), 1);
      ptx::mbar_init(ptx::smem_u32(&qempty[q]), kConvThreads / 32);
    }
    for (int a = 0; a < 2; ++a) {
      ptx::mbar_init(ptx::smem_u32(&tfull[a]), 1);
      ptx::mbar_init(ptx::smem_u32(&tempty[a]), 32 * kEpiWarps);
    }
    ptx::mbar_init(ptx::smem_u32(drain), 1);
    *abort_flag = 0;
    ptx::fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    ptx::prefetch_tmap(&tmA);
    if (MODE == 0) ptx::prefetch_tmap(&tmA2);
  }
  if (warp == 2 && lane == 0) {
    ptx::prefetch_tmap(&tmQ);
    if (MODE == 0) ptx::prefetch_tmap(&tmQ2);
  }
  if (warp == 1) {
    ptx::tmem_alloc(ptx::smem_u32(tmem_holder), 512);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem_base = *tmem_holder;

  const int total_tiles = s_tile_start[args.G] * args.n_tiles;
  const int k_steps = args.K / kBK;

  if (warp == 0) {
    // ------------------------------------------------------------ A producer
    if (lane == 0 && RES) {
      // one resident-token tile per tile: K/64 boxes of 8 rows into the resident buffer
      int it = 0;
      bool ok = true;
      for (int L = blockIdx.x; L < total_tiles; L += gridDim.x, ++it) {
        int g, m, n;
        decode_tile(L, s_tile_start, args.G, args.n_tiles, g, m, n);
        const bool use_a2 = (MODE == 0) && (g >= args.shared_from);
        const int a_row = ((MODE == 0) ? s_a_row[g] : s_out_row[g]) + m * kResRows;
        if (!ptx::mbar_wait_bounded(ptx::smem_u32(aempty), (uint32_t)(it & 1) ^ 1u, abort_flag, kWaitLimitNs)) {
          ok = false;
          break;
        }
        const uint32_t fb = ptx::smem_u32(afull);
        ptx::mbar_arrive_expect_tx(fb, (uint32_t)(k_steps * kResBoxBytes));
        for (int kb = 0; kb < k_steps; ++kb)
          ptx::tma_load_2d(ptx::smem_u32(a_res + (size_t)kb * kResBoxBytes),
                           use_a2 ? (const void*)&tmA2 : (const void*)&tmA, kb * kBK, a_row, fb);
      }
      if (!ok) {
        set_status(args.status, MOE_ERR_TIMEOUT);
        *abort_flag = 1;
      }
      // the last resident tile issued lands before the shared memory is left
      if (it > 0) ptx::mbar_wait_bounded(ptx::smem_u32(afull), (uint32_t)((it - 1) & 1), nullptr, kDrainLimitNs);
    } else if (lane == 0) {
      int stage = 0, issued = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int L = blockIdx.x; L < total_tiles && ok; L += gridDim.x) {
        int g, m, n;
        decode_tile(L, s_tile_start, args.G, args.n_tiles, g, m, n);
        const bool use_a2 = (MODE == 0) && (g >= args.shared_from);
        const int a_row = ((MODE == 0) ? s_a_row[g] : s_out_row[g]) + m * kBM;
        for (int kb = 0; kb < k_steps; ++kb) {
          if (!ptx::mbar_wait_bounded(ptx::smem_u32(&empty[stage]), phase ^ 1u, abort_flag, kWaitLimitNs)) {
            ok = false;
            break;
          }
          const uint32_t fb = ptx::smem_u32(&full[stage]);
          ptx::mbar_arrive_expect_tx(fb, kABytes);
          ptx::tma_load_2d(ptx::smem_u32(stage_base + (size_t)stage * C::kStageBytes),
                           use_a2 ? (const void*)&tmA2 : (const void*)&tmA, kb * kBK, a_row, fb);
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
  } else if (warp == 2) {
    // ------------------------------------------------------------ weight-code producer
    if (lane == 0) {
      int slot = 0, issued = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int L = blockIdx.x; L < total_tiles && ok; L += gridDim.x) {
        int g, m, n;
        decode_tile(L, s_tile_start, args.G, args.n_tiles, g, m, n);
        const int b_row = g * args.b_rows + n * ((MODE == 0) ? 128 : 256);
        for (int kb = 0; kb < k_steps; ++kb) {
          if (!ptx::mbar_wait_bounded(ptx::smem_u32(&qempty[slot]), phase ^ 1u, abort_flag, kWaitLimitNs)) {
            ok = false;
            break;
          }
          const uint32_t fb = ptx::smem_u32(&qfull[slot]);
          const uint32_t dst = ptx::smem_u32(code_base + (size_t)slot * kQBytes);
          ptx::mbar_arrive_expect_tx(fb, kQBytes);
          if (MODE == 0) {
            ptx::tma_load_2d(dst, &tmQ, kb * kBK, b_row, fb);              // W_gate codes
            ptx::tma_load_2d(dst + 128 * kBK, &tmQ2, kb * kBK, b_row, fb); // W_up codes
          } else {
            ptx::tma_load_2d(dst, &tmQ, kb * kBK, b_row, fb);
            ptx::tma_load_2d(dst + 128 * kBK, &tmQ, kb * kBK, b_row + 128, fb);
          }
          if (issued < kQStages) ++issued;
          if (++slot == kQStages) {
            slot = 0;
            phase ^= 1u;
          }
        }
      }
      if (!ok) {
        set_status(args.status, MOE_ERR_TIMEOUT);
        *abort_flag = 1;
        drain_fills(qfull, kQStages, slot, phase, issued);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      // resident-token tiles hold at most 8 rows: an M=64 MMA (rows 0-15 in TMEM lanes 0-15);
      // a 128-row tile whose group has at most 64 rows left runs M=64 MMAs too (half_tile)
      constexpr uint32_t idesc128 = ptx::idesc_bf16_f32(RES ? 64 : kBM, 256);
      constexpr uint32_t idesc64 = ptx::idesc_bf16_f32(64, 256);
      int stage = 0, it = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int L = blockIdx.x; L < total_tiles && ok; L += gridDim.x, ++it) {
        int g, m, n;
        decode_tile(L, s_tile_start, args.G, args.n_tiles, g, m, n);
        const uint32_t idesc = half_tile<RES>(s_rows[g], m) ? idesc64 : idesc128;
        const int acc = it & 1;
        const uint32_t acc_phase = (uint32_t)(it >> 1) & 1u;
        if (!ptx::mbar_wait_bounded(ptx::smem_u32(&tempty[acc]), acc_phase ^ 1u, abort_flag, kWaitLimitNs)) {
          ok = false;
          break;
        }
        if (RES && !ptx::mbar_wait_bounded(ptx::smem_u32(afull), (uint32_t)(it & 1), abort_flag, kWaitLimitNs)) {
          ok = false;
          break;
        }
        ptx::tc_fence_after();
        const uint32_t d_tmem = tmem_base + (uint32_t)(acc * 256);
        for (int kb = 0; kb < k_steps; ++kb) {
          if ((!RES && !ptx::mbar_wait_bounded(ptx::smem_u32(&full[stage]), phase, abort_flag, kWaitLimitNs)) ||
              !ptx::mbar_wait_bounded(ptx::smem_u32(&conv[stage]), phase, abort_flag, kWaitLimitNs)) {
            ok = false;
            break;
          }
          ptx::tc_fence_after();
          const uint32_t sa = ptx::smem_u32(stage_base + (size_t)stage * C::kStageBytes);
          const uint64_t a_desc = RES ? ptx::sw128_kmajor_desc_rows8(ptx::smem_u32(a_res + (size_t)kb * kResBoxBytes))
                                      : ptx::sw128_kmajor_desc(sa);
          const uint64_t b_desc = ptx::sw128_kmajor_desc(sa + C::kBOff);
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
        if (RES) ptx::mma_commit(ptx::smem_u32(aempty));     // the tile's MMAs are done with its tokens
        ptx::mma_commit(ptx::smem_u32(&tfull[acc]));
      }
      if (!ok) {
        set_status(args.status, MOE_ERR_TIMEOUT);
        *abort_flag = 1;
      }
      ptx::mma_commit(ptx::smem_u32(drain));
      ptx::mbar_wait_bounded(ptx::smem_u32(drain), 0, nullptr, kDrainLimitNs);
    }
  } else if (warp < kFirstConvWarp) {
    // ------------------------------------------------------------ epilogue
    const int et = threadIdx.x - 32 * kFirstEpiWarp;        // 0..127
    const int quarter = warp & 3;
    const int r_local = quarter * 32 + lane;
    int it = 0;
    for (int L = blockIdx.x; L < total_tiles; L += gridDim.x, ++it) {
      int g, m, n;
      decode_tile(L, s_tile_start, args.G, args.n_tiles, g, m, n);
      const int acc = it & 1;
      const uint32_t acc_phase = (uint32_t)(it >> 1) & 1u;
      if (!ptx::mbar_wait_bounded(ptx::smem_u32(&tfull[acc]), acc_phase, abort_flag, kWaitLimitNs)) {
        set_status(args.status, MOE_ERR_TIMEOUT);
        *abort_flag = 1;
      }
      // The tile's column scales, shared by the four warps. Every epilogue thread passes both
      // barriers, and all of them leave on the same snapshot of the abort flag (taken between
      // the barriers), so no warp is left waiting at a barrier the others have left.
      epi_bar();
      if (et == 0) *s_stop = *abort_flag;
      if (MODE == 0) {
        s_scale[et] = args.scale[(size_t)g * args.b_rows + n * 128 + et];
        s_scale[128 + et] = args.scale2[(size_t)g * args.b_rows + n * 128 + et];
      } else {
        s_scale[et] = args.scale[(size_t)g * args.b_rows + n * 256 + et];
        s_scale[128 + et] = args.scale[(size_t)g * args.b_rows + n * 256 + 128 + et];
      }
      epi_bar();
      if (*s_stop != 0) break;
      ptx::tc_fence_after();
      // an M=64 tile's row 16 q + i sits in lane i of quarter q (i < 16)
      const bool m64 = half_tile<RES>(s_rows[g], m);
      const int r_row = m64 ? (lane < 16 ? quarter * 16 + lane : C::kRows) : r_local;
      const bool valid = r_row < C::kRows && (m * C::kRows + r_row) < s_rows[g];
      const int64_t out_row = (int64_t)s_out_row[g] + m * C::kRows + r_row;
      const uint32_t t_row = tmem_base + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(acc * 256);
      if (MODE == 0) {
        __nv_bfloat16* orow = args.out + out_row * args.ldo + (int64_t)n * 128;
#pragma unroll 1
        for (int c = 0; c < 128; c += 16) {
          uint32_t gv[16], uv[16];
          ptx::tmem_ld16(t_row + c, gv);
          ptx::tmem_ld16(t_row + 128 + c, uv);
          ptx::tmem_ld_wait();
          if (valid) {
            uint32_t packed[8];
#pragma unroll
            for (int q = 0; q < 8; ++q) {
              const float g0 = __uint_as_float(gv[2 * q]) * s_scale[c + 2 * q];
              const float g1 = __uint_as_float(gv[2 * q + 1]) * s_scale[c + 2 * q + 1];
              const float u0 = __uint_as_float(uv[2 * q]) * s_scale[128 + c + 2 * q];
              const float u1 = __uint_as_float(uv[2 * q + 1]) * s_scale[128 + c + 2 * q + 1];
              packed[q] = pack_bf16(silu_f(g0) * u0, silu_f(g1) * u1);
            }
            uint4* dst = reinterpret_cast<uint4*>(orow + c);
#pragma unroll
            for (int q = 0; q < 2; ++q)
              dst[q] = make_uint4(packed[4 * q], packed[4 * q + 1], packed[4 * q + 2], packed[4 * q + 3]);
          }
        }
      } else {
        __nv_bfloat16* orow = args.out + out_row * args.ldo + (int64_t)n * 256;
#pragma unroll 1
        for (int c = 0; c < 256; c += 16) {
          uint32_t v[16];
          ptx::tmem_ld16(t_row + c, v);
          ptx::tmem_ld_wait();
          if (valid) {
            uint32_t packed[8];
#pragma unroll
            for (int q = 0; q < 8; ++q)
              packed[q] = pack_bf16(__uint_as_float(v[2 * q]) * s_scale[c + 2 * q],
                                    __uint_as_float(v[2 * q + 1]) * s_scale[c + 2 * q + 1]);
            uint4* dst = reinterpret_cast<uint4*>(orow + c);
#pragma unroll
            for (int q = 0; q < 2; ++q)
              dst[q] = make_uint4(packed[4 * q], packed[4 * q + 1], packed[4 * q + 2], packed[4 * q + 3]);
          }
        }
      }
      ptx::tc_fence_before();
      ptx::mbar_arrive(ptx::smem_u32(&tempty[acc]));
    }
  } else {
    // ------------------------------------------------------------ code widening
    const int cidx = threadIdx.x - 32 * kFirstConvWarp;
    const int group = cidx / kConvThreads;                   // takes the k-steps j with j % 2 == group
    const int ct = cidx - group * kConvThreads;              // 0..255
    int stage = 0, slot = 0, j = 0;
    uint32_t phase = 0, qphase = 0;
    for (int L = blockIdx.x; L < total_tiles; L += gridDim.x) {
      bool ok = true;
      for (int kb = 0; kb < k_steps; ++kb, ++j) {
        if ((j % kConvGroups) != group) {                    // the other group's k-step
          if (++stage == kStages) {
            stage = 0;
            phase ^= 1u;
          }
          if (++slot == kQStages) {
            slot = 0;
            qphase ^= 1u;
          }
          continue;
        }
        if (!ptx::mbar_wait_bounded(ptx::smem_u32(&qfull[slot]), qphase, abort_flag, kWaitLimitNs) ||
            !ptx::mbar_wait_bounded(ptx::smem_u32(&empty[stage]), phase ^ 1u, abort_flag, kWaitLimitNs)) {
          ok = false;
          break;
        }
        const uint8_t* codes = code_base + (size_t)slot * kQBytes;
        uint8_t* bdst = stage_base + (size_t)stage * C::kStageBytes + C::kBOff;
#pragma unroll
        for (int u = 0; u < (kBRows * 4) / kConvThreads; ++u) {
          const int t = ct + u * kConvThreads;
          const int r = t >> 2, j = t & 3;                    // row, 16-code group
          const uint4 raw = *reinterpret_cast<const uint4*>(codes + r * kBK + j * 16);
          const uint4 lo = make_uint4(widen2(raw.x), widen2(raw.x >> 16), widen2(raw.y), widen2(raw.y >> 16));
          const uint4 hi = make_uint4(widen2(raw.z), widen2(raw.z >> 16), widen2(raw.w), widen2(raw.w >> 16));
          uint8_t* rowp = bdst + (r >> 3) * 1024 + (r & 7) * 128;
          *reinterpret_cast<uint4*>(rowp + (((2 * j) ^ (r & 7)) << 4)) = lo;
          *reinterpret_cast<uint4*>(rowp + (((2 * j + 1) ^ (r & 7)) << 4)) = hi;
        }
        // Each thread's widened stores are made visible to the async proxy, then one lane per
        // warp hands the warp's part to the MMA and frees its codes (8 arrives, not 256 that
        // would serialise on the barrier).
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          ptx::mbar_arrive(ptx::smem_u32(&conv[stage]));
          ptx::mbar_arrive(ptx::smem_u32(&qempty[slot]));
        }
        if (++stage == kStages) {
          stage = 0;
          phase ^= 1u;
        }
        if (++slot == kQStages) {
          slot = 0;
          qphase ^= 1u;
        }
      }
      if (!ok) {
        set_status(args.status, MOE_ERR_TIMEOUT);
        *abort_flag = 1;
        break;
      }
    }
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem_base, 512);
  }
}

// One warp per row: the row's absolute maximum, its scale, then the codes, 16 per lane step.
__global__ void quantize_fp8_rows_kernel(const __nv_bfloat16* __restrict__ w, int64_t rows, int cols,
                                         uint8_t* __restrict__ wq, float* __restrict__ scale) {
  const int lane = threadIdx.x & 31;
  const int64_t warps = (int64_t)gridDim.x * (blockDim.x >> 5);
  for (int64_t r = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); r < rows; r += warps)
    quantize_row_e4m3_warp(w + r * cols, cols, wq + r * cols, scale + r, lane);
}

// Resident-token tiles where the average expert holds at most 8 pairs (decode) and the tile's
// tokens for the whole reduction (K/64 KB) leave at least four code slots.
bool use_resident(const Shape& s, int K) {
  return (int64_t)s.T * s.k <= (int64_t)kResRows * s.E && K <= 2048;
}

// Upper bound on a launch's m-tiles of `rows` token rows: the routed rows spread over E groups
// (each may add one partial tile) plus the shared groups' rows.
int64_t max_m_tiles(const Shape& s, int rows) {
  return (s.R + rows - 1) / rows + s.E + (int64_t)s.S * ((s.T + rows - 1) / rows);
}

template <int MODE, bool RES>
cudaError_t launch_fp8w(const CUtensorMap& a, const CUtensorMap& a2, const CUtensorMap& q, const CUtensorMap& q2,
                        Fp8Args args, const Shape& s, cudaStream_t st) {
  using C = FCfg<RES>;
  args.res_bytes = RES ? (args.K / kBK) * kResBoxBytes : 0;
  const size_t base = kSmemFixed + (size_t)kStages * C::kStageBytes + (size_t)args.res_bytes;
  int q_slots = RES ? (int)((kSmemMax - base) / kQBytes) : 4;
  if (q_slots > kMaxQSlots) q_slots = kMaxQSlots;
  if (q_slots < 2) return cudaErrorInvalidValue;
  args.qslots = q_slots;
  const size_t smem = base + (size_t)q_slots * kQBytes;
  auto kern = grouped_gemm_fp8w_kernel<MODE, RES>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  const int64_t max_tiles = max_m_tiles(s, C::kRows) * args.n_tiles;
  int64_t grid = num_sms();
  if (max_tiles < grid) grid = max_tiles;
  if (grid < 1) grid = 1;
  kern<<<(unsigned)grid, kThreads, smem, st>>>(a, a2, q, q2, args);
  return cudaGetLastError();
}

}  // namespace

bool fp8w_supported(const Shape& s) { return s.dtype == MOE_BF16 && s.d % 256 == 0 && s.F % 128 == 0; }

cudaError_t launch_quantize_fp8_rows(const void* w, int64_t rows, int cols, uint8_t* wq, float* scale,
                                     cudaStream_t st) {
  int64_t blocks = (rows + 7) / 8;
  const int64_t cap = (int64_t)num_sms() * 16;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  quantize_fp8_rows_kernel<<<(unsigned)blocks, 256, 0, st>>>(static_cast<const __nv_bfloat16*>(w), rows, cols, wq,
                                                             scale);
  return cudaGetLastError();
}

cudaError_t launch_gemm_gateup_fp8w(const Shape& s, const void* x_perm, const void* x, const uint8_t* wg_q,
                                    const float* wg_s, const uint8_t* wu_q, const float* wu_s, const void* sched,
                                    void* h, int32_t* status, cudaStream_t st) {
  CUtensorMap a, a2, q, q2;
  const uint64_t R = (uint64_t)(s.R > 0 ? s.R : 1);
  const bool res = use_resident(s, s.d);
  const uint32_t box = res ? kResRows : kBM;
  if (!make_tmap_bf16(&a, x_perm, s.d, R, box)) return cudaErrorInvalidValue;
  if (!make_tmap_bf16(&a2, s.S > 0 ? x : x_perm, s.d, s.S > 0 ? (uint64_t)s.T : R, box)) return cudaErrorInvalidValue;
  if (!make_tmap_u8(&q, wg_q, s.d, (uint64_t)s.G * s.F, 128)) return cudaErrorInvalidValue;
  if (!make_tmap_u8(&q2, wu_q, s.d, (uint64_t)s.G * s.F, 128)) return cudaErrorInvalidValue;
  Fp8Args args{};
  args.K = s.d;
  args.n_tiles = s.F / 128;
  args.G = s.G;
  args.shared_from = s.E;
  args.b_rows = s.F;
  args.sched = static_cast<const int32_t*>(sched);
  args.scale = wg_s;
  args.scale2 = wu_s;
  args.out = static_cast<__nv_bfloat16*>(h);
  args.ldo = s.F;
  args.status = status;
  return res ? launch_fp8w<0, true>(a, a2, q, q2, args, s, st) : launch_fp8w<0, false>(a, a2, q, q2, args, s, st);
}

cudaError_t launch_gemm_down_fp8w(const Shape& s, const void* h, const uint8_t* wd_q, const float* wd_s,
                                  const void* sched, void* y, int32_t* status, cudaStream_t st) {
  CUtensorMap a, q;
  const uint64_t rows = (uint64_t)s.R + (uint64_t)s.S * s.T;
  const bool res = use_resident(s, s.F);
  if (!make_tmap_bf16(&a, h, s.F, rows > 0 ? rows : 1, res ? kResRows : kBM)) return cudaErrorInvalidValue;
  if (!make_tmap_u8(&q, wd_q, s.F, (uint64_t)s.G * s.d, 128)) return cudaErrorInvalidValue;
  Fp8Args args{};
  args.K = s.F;
  args.n_tiles = s.d / 256;
  args.G = s.G;
  args.shared_from = s.G;
  args.b_rows = s.d;
  args.sched = static_cast<const int32_t*>(sched);
  args.scale = wd_s;
  args.scale2 = wd_s;
  args.out = static_cast<__nv_bfloat16*>(y);
  args.ldo = s.d;
  args.status = status;
  return res ? launch_fp8w<1, true>(a, a, q, q, args, s, st) : launch_fp8w<1, false>(a, a, q, q, args, s, st);
}

}  // namespace moe
