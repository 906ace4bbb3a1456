// Grouped expert GEMMs on the 5th-generation tensor cores (tcgen05 + TMEM),
// fed by TMA over a per-expert tile schedule.
//
// "Permuting tokens by destination expert, running grouped GEMMs on each
// expert's batch, then undoing the permutation" (klaylearn.com/glossary/
// mixture-of-experts, "Mixture of Experts", definition). The expert is a SwiGLU
// MLP y = W_down (silu(W_gate a) * (W_up a)); this file holds its two
// contractions:
//   gate/up : per group g, h[rows_g, F] = silu(A_g W_gate[g]^T) * (A_g W_up[g]^T)
//             (A_g = the group's x_perm rows; the shared expert reads x itself)
//   down    : per group g, y[rows_g, d] = h_g W_down[g]^T
//
// Design (one persistent CTA per SM, 192 threads, warp-specialised):
//   warp 0      TMA producer: A tile 128 x 64 and B tile(s) N x 64 (bf16, K-major,
//               128-byte swizzle) per k-step into a 4-stage shared-memory ring
//   warp 1      MMA issuer: tcgen05.mma kind::f16 M=128, N=256, K=16 (x4 per
//               stage) into one of two TMEM accumulators of 256 float32 columns
//   warps 2-5   epilogue: tcgen05.ld the accumulator (one row per thread),
//               SwiGLU or plain convert, bf16 stores of the valid rows
// For gate/up the B stage holds the 128 W_gate rows followed by the 128 W_up rows
// of the same output columns, so one N=256 MMA yields both projections side by
// side in TMEM and the SwiGLU is fused into the epilogue. The two TMEM
// accumulators let the epilogue of tile i overlap the MMAs of tile i+1.
//
// Tiles are ordered (group, n-tile, m-tile): neighbouring CTAs share the same
// weight columns, so each expert's weights stream from HBM about once while
// its activation rows are re-read from L2. A group's last m-tile may run past
// its rows into the next group's rows; those rows are computed and discarded.
//
// Every wait is bounded: a stall records MOE_ERR_TIMEOUT, all roles leave
// their loops, in-flight copies and MMAs are drained with bounded waits, and
// the TMEM is freed before the CTA exits.
#include "internal.cuh"
#include "tc_ptx.cuh"
#include "tmap.cuh"

namespace moe {
namespace {

constexpr int kBM = 128;
constexpr int kBK = 64;              // one 128-byte swizzle atom of bf16
constexpr int kThreads = 192;
constexpr uint64_t kWaitLimitNs = 4000000000ull;     // 4 s: far beyond any legitimate wait
constexpr uint64_t kDrainLimitNs = 100000000ull;     // 100 ms for draining after an abort

template <int MODE, int BN>
struct Cfg {
  static constexpr int kNmma = (MODE == 0) ? 256 : BN;            // MMA N
  static constexpr int kOutCols = (MODE == 0) ? 128 : BN;         // output columns per tile
  static constexpr int kABytes = kBM * kBK * 2;                    // 16 KB
  static constexpr int kBBytes = kNmma * kBK * 2;
  static constexpr int kStageBytes = kABytes + kBBytes;
  static constexpr int kStages = (kStageBytes <= 32768) ? 6 : 4;
  static constexpr int kTmemCols = 2 * kNmma;                      // two accumulators
  static constexpr int kSchedInts = 4 * (kMaxExperts + 2);
  static constexpr size_t kSmem = 1024 /*alignment slack*/ + (size_t)kStages * kStageBytes + 256 /*barriers*/ +
                                  (size_t)kSchedInts * 4;
};

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
};

__device__ __forceinline__ void decode_tile(int L, const int32_t* tile_start, int G, int nt, int& g, int& m,
                                            int& n) {
  int lo = 0, hi = G;
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (tile_start[mid] * nt <= L) lo = mid; else hi = mid;
  }
  g = lo;
  const int mt = tile_start[g + 1] - tile_start[g];
  const int local = L - tile_start[g] * nt;
  n = local / mt;
  m = local - n * mt;
}

__device__ __forceinline__ float silu_f(float z) { return __fdividef(z, 1.0f + __expf(-z)); }

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&v);
}

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
      ptx::mbar_init(ptx::smem_u32(&tempty[a]), 4 * 32);
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
          if (MODE == 0) {
            ptx::tma_load_2d(sb, &tmB, kb * kBK, b_row, fb);
            ptx::tma_load_2d(sb + 128 * 128, &tmB2, kb * kBK, b_row, fb);
          } else {
            ptx::tma_load_2d(sb, &tmB, kb * kBK, b_row, fb);
          }
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
        // Drain after an abort: the most recent fill of each slot must land before the
        // CTA exits. A fill whose phase already completed passes at once.
        int s = stage;
        uint32_t ph = phase;
        for (int j = 0; j < issued; ++j) {
          if (s == 0) {
            s = C::kStages - 1;
            ph ^= 1u;
          } else {
            --s;
          }
          ptx::mbar_wait_bounded(ptx::smem_u32(&full[s]), ph, nullptr, kDrainLimitNs);
        }
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
      __nv_bfloat16* orow = args.out + out_row * args.ldo + (int64_t)n * C::kOutCols;
      const uint32_t t_row = tmem_base + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(acc * C::kNmma);
      if (MODE == 0) {
#pragma unroll 1
        for (int c = 0; c < 128; c += 32) {
          uint32_t gv[32], uv[32];
          ptx::tmem_ld32(t_row + c, gv);
          ptx::tmem_ld32(t_row + 128 + c, uv);
          ptx::tmem_ld_wait();
          if (valid) {
            uint32_t packed[16];
#pragma unroll
            for (int q = 0; q < 16; ++q) {
              const float h0 = silu_f(__uint_as_float(gv[2 * q])) * __uint_as_float(uv[2 * q]);
              const float h1 = silu_f(__uint_as_float(gv[2 * q + 1])) * __uint_as_float(uv[2 * q + 1]);
              packed[q] = pack_bf16(h0, h1);
            }
            uint4* dst = reinterpret_cast<uint4*>(orow + c);
#pragma unroll
            for (int q = 0; q < 4; ++q)
              dst[q] = make_uint4(packed[4 * q], packed[4 * q + 1], packed[4 * q + 2], packed[4 * q + 3]);
          }
        }
      } else {
#pragma unroll 1
        for (int c = 0; c < C::kOutCols; c += 32) {
          uint32_t v[32];
          ptx::tmem_ld32(t_row + c, v);
          ptx::tmem_ld_wait();
          if (valid) {
            uint32_t packed[16];
#pragma unroll
            for (int q = 0; q < 16; ++q) packed[q] = pack_bf16(__uint_as_float(v[2 * q]), __uint_as_float(v[2 * q + 1]));
            uint4* dst = reinterpret_cast<uint4*>(orow + c);
#pragma unroll
            for (int q = 0; q < 4; ++q)
              dst[q] = make_uint4(packed[4 * q], packed[4 * q + 1], packed[4 * q + 2], packed[4 * q + 3]);
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
    ptx::tmem_dealloc(tmem_base, C::kTmemCols);
  }
}

// ------------------------------------------------------------------ host ---
template <int MODE, int BN>
cudaError_t launch_grouped(const CUtensorMap& a, const CUtensorMap& a2, const CUtensorMap& b, const CUtensorMap& b2,
                           const GemmArgs& args, int64_t max_tiles, cudaStream_t st) {
  using C = Cfg<MODE, BN>;
  auto kern = grouped_gemm_kernel<MODE, BN>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)C::kSmem);
  if (e != cudaSuccess) return e;
  int64_t grid = num_sms();
  if (max_tiles < grid) grid = max_tiles;
  if (grid < 1) grid = 1;
  kern<<<(unsigned)grid, kThreads, C::kSmem, st>>>(a, a2, b, b2, args);
  return cudaGetLastError();
}

int64_t max_m_tiles(const Shape& s) {
  // routed rows R spread over E groups (each may add one partial tile) + shared rows
  return (s.R + kBM - 1) / kBM + s.E + (int64_t)s.S * ((s.T + kBM - 1) / kBM);
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
  return launch_grouped<0, 128>(a, a2, b, b2, args, max_m_tiles(s) * args.n_tiles, st);
}

cudaError_t launch_gemm_down_tc(const Shape& s, const void* h, const void* w_down, const void* sched, void* y,
                                int32_t* status, cudaStream_t st) {
  CUtensorMap a, b;
  const uint64_t rows = (uint64_t)s.R + (uint64_t)s.S * s.T;
  const int bn = (s.d % 256 == 0) ? 256 : 128;
  if (!make_tmap_bf16(&a, h, s.F, rows > 0 ? rows : 1, kBM)) return cudaErrorInvalidValue;
  if (!make_tmap_bf16(&b, w_down, s.F, (uint64_t)s.G * s.d, (uint32_t)bn)) return cudaErrorInvalidValue;
  GemmArgs args{};
  args.K = s.F;
  args.n_tiles = s.d / bn;
  args.G = s.G;
  args.shared_from = s.G;
  args.b_rows = s.d;
  args.sched = static_cast<const int32_t*>(sched);
  args.out = static_cast<__nv_bfloat16*>(y);
  args.ldo = s.d;
  args.status = status;
  if (bn == 256) return launch_grouped<1, 256>(a, a, b, b, args, max_m_tiles(s) * args.n_tiles, st);
  return launch_grouped<1, 128>(a, a, b, b, args, max_m_tiles(s) * args.n_tiles, st);
}

}  // namespace moe
