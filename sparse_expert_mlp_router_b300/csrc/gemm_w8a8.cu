// Grouped expert GEMMs with E4M3 weights AND E4M3 activations (W8A8), on the 8-bit
// tensor-core path (tcgen05.mma kind::f8f6f4), and the per-row quantiser of the activation
// rows that feed them.
//
// The source pages put an FP8 model at about half the bytes of its BF16 copy
// (shubhamtatvamasi.com/llm-inference/moe "Mixture of Experts", section "Memory vs compute,
// quantified") and say nothing about the activations. The FP8-weight kernels of gemm_fp8w.cu
// keep bf16 activations and widen the weight codes to bf16 in shared memory for a kind::f16
// MMA; there the widening and four N=256 MMAs per 16 KB of codes hold the kernel near 0.6 of
// HBM bandwidth on memory-bound layers. This mode quantises the activation rows too, per row
// like the weights (scale = max|row| / 448, E4M3 codes), so both operands go from TMA straight
// to the 8-bit MMA: a k-step is 128 codes (one 128-byte swizzle atom), four K=32 MMAs per
// 32 KB of weight codes, no widening. Numerically it is the oracle's expert_mlp_w8a8 reading,
// not the bf16-activation layer.
//
// Kernel structure (one CTA per SM, persistent, 320 threads), as in gemm_tc.cu:
//   warp 0      TMA producer: A = 128 activation rows x 128 codes (16 KB), B = 256 weight
//               rows x 128 codes (32 KB; gate/up: 128 W_gate + 128 W_up rows), 4 stages
//   warp 1      MMA issuer: tcgen05.mma kind::f8f6f4, M=128, N=256, K=32 (x4 per stage), two
//               TMEM accumulators of 256 float32 columns
//   warps 2-9   epilogue: accumulator x activation-row scale x weight-row scale, SwiGLU for
//               gate/up, bf16 rows staged in shared memory and stored 8 rows x 64 bytes per
//               instruction
// Tiles are ordered (group, n-tile, m-tile) over the schedule of the grouping stage. Every wait
// is bounded (a stall records MOE_ERR_TIMEOUT, the roles leave, TMEM is freed).
#include "epilogue.cuh"
#include "fp8_quant.cuh"
#include "gemm_common.cuh"
#include "group_single.cuh"
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
constexpr int kThreads = 64 + 32 * kEpiWarps;
constexpr int kABytes = kBM * kBK;                // 16 KB
constexpr int kBBytes = 256 * kBK;                // 32 KB
constexpr int kStageBytes = kABytes + kBBytes;    // 48 KB
constexpr int kStages = 4;
constexpr int kTmemCols = 512;                    // two accumulators of 256 columns
constexpr int kSchedInts = 4 * (kMaxExperts + 2);
using epi::kStageOutBytes;
constexpr size_t kStgOff = (size_t)kStages * kStageBytes + 256 + (((size_t)kSchedInts * 4 + 127) / 128) * 128;
constexpr size_t kSmem = 1024 + kStgOff + (size_t)kEpiWarps * kStageOutBytes;

// Instruction descriptor of tcgen05.mma kind::f8f6f4 with E4M3 A and B (format code 0 in both
// fields), float32 D, both operands K-major, shape M x N.
__host__ __device__ constexpr uint32_t idesc_e4m3_f32(int M, int N) {
  return (1u << 4)                       // D format: f32
         | ((uint32_t)(N >> 3) << 17)    // N / 8
         | ((uint32_t)(M >> 4) << 24);   // M / 16
}

// D[tmem] (+)= A[smem desc] * B[smem desc]^T on E4M3 operands (K = 32 per instruction).
__device__ __forceinline__ void mma_e4m3(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                         uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

struct W8Args {
  int K;                  // reduction length (codes)
  int n_tiles;            // N tiles per group
  int G;                  // groups
  int b_rows;             // weight rows per group (F for gate/up, d for down)
  const int32_t* sched;   // device group schedule
  const float* a_scale;   // per activation row (indexed like the rows of the output)
  const float* scale;     // gate/up: W_gate row scales [G, F]; down: W_down row scales [G, d]
  const float* scale2;    // gate/up: W_up row scales [G, F]
  __nv_bfloat16* out;
  int64_t ldo;
  int32_t* status;
};

template <int MODE>
__global__ void __launch_bounds__(kThreads, 1)
grouped_gemm_w8a8_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                         const __grid_constant__ CUtensorMap tmB2, const W8Args args) {
  constexpr int kOutCols = (MODE == 0) ? 128 : 256;
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
      ptx::mbar_init(ptx::smem_u32(&tempty[a]), kEpiWarps * 32);
    }
    ptx::mbar_init(ptx::smem_u32(drain), 1);
    *abort_flag = 0;
    ptx::fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    ptx::prefetch_tmap(&tmA);
    ptx::prefetch_tmap(&tmB);
    if (MODE == 0) ptx::prefetch_tmap(&tmB2);
  }
  if (warp == 1) {
    ptx::tmem_alloc(ptx::smem_u32(tmem_holder), kTmemCols);
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
      int stage = 0, issued = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int L = blockIdx.x; L < total_tiles && ok; L += gridDim.x) {
        int g, m, n;
        decode_tile(L, s_tile_start, args.G, args.n_tiles, g, m, n);
        // activation rows are stored at the output rows (routed rows, then the shared expert's)
        const int a_row = s_out_row[g] + m * kBM;
        const int b_row = g * args.b_rows + n * ((MODE == 0) ? 128 : 256);
        for (int kb = 0; kb < k_steps; ++kb) {
          if (!ptx::mbar_wait_bounded(ptx::smem_u32(&empty[stage]), phase ^ 1u, abort_flag, kWaitLimitNs)) {
            ok = false;
            break;
          }
          const uint32_t fb = ptx::smem_u32(&full[stage]);
          const uint32_t sa = ptx::smem_u32(stage_base + (size_t)stage * kStageBytes);
          const uint32_t sb = sa + kABytes;
          ptx::mbar_arrive_expect_tx(fb, kStageBytes);
          ptx::tma_load_2d(sa, &tmA, kb * kBK, a_row, fb);
          if (MODE == 0) {
            ptx::tma_load_2d(sb, &tmB, kb * kBK, b_row, fb);                   // W_gate rows
            ptx::tma_load_2d(sb + 128 * kBK, &tmB2, kb * kBK, b_row, fb);      // W_up rows
          } else {
            ptx::tma_load_2d(sb, &tmB, kb * kBK, b_row, fb);
          }
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
      for (int L = blockIdx.x; L < total_tiles && ok; L += gridDim.x, ++it) {
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
            // advance 32 codes = 32 bytes along K inside the swizzle atom
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
    const int quarter = warp & 3;            // TMEM lanes this warp may access
    const int half = (warp - 2) >> 2;        // which half of the output columns
    const uint32_t stg = stg_base + (uint32_t)(warp - 2) * kStageOutBytes;
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
      const int row0 = m * kBM + quarter * 32;                      // the warp's first row in the group
      const int nvalid = s_rows[g] - row0;
      const int64_t my_out = (int64_t)s_out_row[g] + row0 + lane;
      const float sa = (lane < nvalid) ? args.a_scale[my_out] : 0.0f;
      __nv_bfloat16* orow0 = args.out + ((int64_t)s_out_row[g] + row0) * args.ldo + (int64_t)n * kOutCols;
      const uint32_t t_row = tmem_base + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(acc * 256);
      if (nvalid > 0) {
        const int c0 = half * (kOutCols / 2), c1 = c0 + kOutCols / 2;
#pragma unroll 1
        for (int c = c0; c < c1; c += 32) {
          uint32_t packed[16];
          if (MODE == 0) {
            const float* sg = args.scale + (int64_t)g * args.b_rows + n * 128 + c;
            const float* su = args.scale2 + (int64_t)g * args.b_rows + n * 128 + c;
            uint32_t gv[32], uv[32];
            ptx::tmem_ld32(t_row + c, gv);
            ptx::tmem_ld32(t_row + 128 + c, uv);
            ptx::tmem_ld_wait();
#pragma unroll
            for (int q = 0; q < 16; ++q) {
              const float g0 = __uint_as_float(gv[2 * q]) * (sa * __ldg(sg + 2 * q));
              const float g1 = __uint_as_float(gv[2 * q + 1]) * (sa * __ldg(sg + 2 * q + 1));
              const float u0 = __uint_as_float(uv[2 * q]) * (sa * __ldg(su + 2 * q));
              const float u1 = __uint_as_float(uv[2 * q + 1]) * (sa * __ldg(su + 2 * q + 1));
              packed[q] = pack_bf16(silu_f(g0) * u0, silu_f(g1) * u1);
            }
          } else {
            const float* sd = args.scale + (int64_t)g * args.b_rows + n * 256 + c;
            uint32_t v[32];
            ptx::tmem_ld32(t_row + c, v);
            ptx::tmem_ld_wait();
#pragma unroll
            for (int q = 0; q < 16; ++q)
              packed[q] = pack_bf16(__uint_as_float(v[2 * q]) * (sa * __ldg(sd + 2 * q)),
                                    __uint_as_float(v[2 * q + 1]) * (sa * __ldg(sd + 2 * q + 1)));
          }
          epi::store_chunk(packed, nvalid, orow0, args.ldo, c, stg, lane);
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

// Activation rows -> E4M3 codes and per-row scales, one warp per row. Segment a: rows
// [0, min(*n_a, max_a)) of src_a (the grouped rows actually filled, a count on the device) to
// the same rows of dst; segment b: rows [0, n_b) of src_b to rows [b0, b0 + n_b) of dst.
__global__ void quantize_act_rows_kernel(const __nv_bfloat16* __restrict__ src_a, const int32_t* __restrict__ n_a,
                                         int64_t max_a, const __nv_bfloat16* __restrict__ src_b, int64_t n_b,
                                         int64_t b0, int cols, uint8_t* __restrict__ dst, float* __restrict__ scale) {
  const int lane = threadIdx.x & 31;
  int64_t na = *n_a;
  if (na > max_a) na = max_a;
  if (na < 0) na = 0;
  const int64_t total = max_a + n_b;
  const int64_t warps = (int64_t)gridDim.x * (blockDim.x >> 5);
  for (int64_t v = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); v < total; v += warps) {
    if (v < max_a) {
      if (v >= na) continue;
      quantize_row_e4m3_warp(src_a + v * cols, cols, dst + v * cols, scale + v, lane);
    } else {
      const int64_t r = v - max_a;
      quantize_row_e4m3_warp(src_b + r * cols, cols, dst + (b0 + r) * cols, scale + b0 + r, lane);
    }
  }
}

// Rows [0, rows) of a bf16 tensor to E4M3 codes and per-row scales, one warp per row.
__global__ void quantize_fp8_rows_kernel_act(const __nv_bfloat16* __restrict__ w, int64_t rows, int cols,
                                             uint8_t* __restrict__ wq, float* __restrict__ scale) {
  const int lane = threadIdx.x & 31;
  const int64_t warps = (int64_t)gridDim.x * (blockDim.x >> 5);
  for (int64_t r = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); r < rows; r += warps)
    quantize_row_e4m3_warp(w + r * cols, cols, wq + r * cols, scale + r, lane);
}

// One chunk of tokens: the grouping (every block in its own shared memory, block 0 writing it
// out) and the grouped rows quantised as they are copied, one warp per row; the shared expert's
// rows R .. R+T-1 are the tokens in order.
__global__ void __launch_bounds__(kSingleThreads)
group_quant_single_chunk_kernel(const int32_t* __restrict__ idx, int T, int k, int E, int cap,
                                int32_t* __restrict__ counts, int32_t* __restrict__ offsets,
                                int32_t* __restrict__ dest_row, int32_t* __restrict__ src_token,
                                int32_t* __restrict__ sched, int S, int64_t R, int32_t* status,
                                const __nv_bfloat16* __restrict__ x, int d, uint8_t* __restrict__ dst,
                                float* __restrict__ scale) {
  __shared__ SingleChunkSmem sm;
  single_chunk_group(idx, T, k, E, cap, blockIdx.x == 0, counts, offsets, dest_row, src_token, sched, S, R, status,
                     sm);
  const int lane = threadIdx.x & 31;
  const int64_t n = min((int64_t)sm.off[E], R);
  const int64_t total = R + (int64_t)S * T;
  const int64_t warps = (int64_t)gridDim.x * (blockDim.x >> 5);
  for (int64_t v = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); v < total; v += warps) {
    int64_t t;
    if (v < R) {
      if (v >= n) continue;
      t = sm.src[v];
    } else {
      t = v - R;
    }
    quantize_row_e4m3_warp(x + t * d, d, dst + v * d, scale + v, lane);
  }
}

// Grouped rows as copies of per-token codes: row r < offsets[E] gets token src_token[r]'s codes
// and scale from xq / xq_scale (x quantised once per token), the shared expert's rows R .. R+T-1
// the tokens in order. One warp per row, 16-byte vectors (d is a multiple of 256).
__global__ void gather_code_rows_kernel(const uint4* __restrict__ xq, const float* __restrict__ xq_scale,
                                        const int32_t* __restrict__ src_token, const int32_t* __restrict__ offsets,
                                        int E, int64_t R, int64_t n_shared_rows, int vec_per_row,
                                        uint4* __restrict__ dst, float* __restrict__ scale) {
  const int lane = threadIdx.x & 31;
  int64_t n = offsets[E];
  if (n > R) n = R;
  const int64_t total = R + n_shared_rows;
  const int64_t warps = (int64_t)gridDim.x * (blockDim.x >> 5);
  for (int64_t v = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); v < total; v += warps) {
    int64_t t;
    if (v < R) {
      if (v >= n) continue;
      t = src_token[v];
    } else {
      t = v - R;
    }
    const uint4* src = xq + t * vec_per_row;
    uint4* out = dst + v * vec_per_row;
    for (int c = lane; c < vec_per_row; c += 32) out[c] = __ldg(src + c);
    if (lane == 0) scale[v] = xq_scale[t];
  }
}

int64_t max_m_tiles(const Shape& s) {
  return (s.R + kBM - 1) / kBM + s.E + (int64_t)s.S * ((s.T + kBM - 1) / kBM);
}

template <int MODE>
cudaError_t launch_w8a8(const CUtensorMap& a, const CUtensorMap& b, const CUtensorMap& b2, const W8Args& args,
                        const Shape& s, cudaStream_t st) {
  auto kern = grouped_gemm_w8a8_kernel<MODE>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmem);
  if (e != cudaSuccess) return e;
  int64_t grid = num_sms();
  const int64_t max_tiles = max_m_tiles(s) * args.n_tiles;
  if (max_tiles < grid) grid = max_tiles;
  if (grid < 1) grid = 1;
  kern<<<(unsigned)grid, kThreads, kSmem, st>>>(a, b, b2, args);
  return cudaGetLastError();
}

}  // namespace

bool w8a8_supported(const Shape& s) { return s.dtype == MOE_BF16 && s.d % 256 == 0 && s.F % 128 == 0; }

cudaError_t launch_quantize_act_rows(const Shape& s, const void* src_a, const int32_t* n_a, int64_t max_a,
                                     const void* src_b, int64_t n_b, int cols, uint8_t* dst, float* scale,
                                     cudaStream_t st) {
  const int64_t rows = max_a + n_b;
  int64_t blocks = (rows + 7) / 8;
  const int64_t cap = (int64_t)num_sms() * 16;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  quantize_act_rows_kernel<<<(unsigned)blocks, 256, 0, st>>>(
      static_cast<const __nv_bfloat16*>(src_a), n_a, max_a, static_cast<const __nv_bfloat16*>(src_b), n_b, s.R,
      cols, dst, scale);
  return cudaGetLastError();
}

cudaError_t launch_group_quant_single_chunk(const Shape& s, const int32_t* idx, int32_t* counts, int32_t* offsets,
                                            int32_t* dest_row, int32_t* src_token, void* sched, int32_t* status,
                                            const void* x, uint8_t* x8, float* x8_scale, cudaStream_t st) {
  if (s.nchunks != 1) return cudaErrorInvalidValue;
  const int64_t rows = s.R + (int64_t)s.S * s.T;
  const int64_t cap = (int64_t)num_sms() * 16;
  int64_t blocks = (rows + 7) / 8;      // one warp per row, as the separate quantising copy
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  group_quant_single_chunk_kernel<<<(unsigned)blocks, kSingleThreads, 0, st>>>(
      idx, s.T, s.k, s.E, s.cap, counts, offsets, dest_row, src_token, static_cast<int32_t*>(sched), s.S, s.R, status,
      static_cast<const __nv_bfloat16*>(x), s.d, x8, x8_scale);
  return cudaGetLastError();
}

// Batches of more than one chunk, where every token appears k times among the grouped rows:
// quantise the T tokens once into xq (codes, T x d bytes) and xq_scale, then copy code rows
// (half the bytes of bf16 rows). A single chunk takes launch_group_quant_single_chunk.
cudaError_t launch_gather_quant_rows(const Shape& s, const void* x, const int32_t* src_token, const int32_t* offsets,
                                     uint8_t* x8, float* x8_scale, uint8_t* xq, float* xq_scale, cudaStream_t st) {
  const int64_t n_sh = (int64_t)s.S * s.T;
  const int64_t rows = s.R + n_sh;
  const int64_t cap = (int64_t)num_sms() * 16;
  int64_t blocks = (rows + 7) / 8;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  if (s.nchunks == 1) return cudaErrorInvalidValue;
  int64_t qblocks = ((int64_t)s.T + 7) / 8;
  if (qblocks > cap) qblocks = cap;
  quantize_fp8_rows_kernel_act<<<(unsigned)qblocks, 256, 0, st>>>(static_cast<const __nv_bfloat16*>(x), s.T, s.d,
                                                                  xq, xq_scale);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  gather_code_rows_kernel<<<(unsigned)blocks, 256, 0, st>>>(reinterpret_cast<const uint4*>(xq), xq_scale, src_token,
                                                            offsets, s.E, s.R, n_sh, s.d / 16,
                                                            reinterpret_cast<uint4*>(x8), x8_scale);
  return cudaGetLastError();
}

cudaError_t launch_gemm_gateup_w8a8(const Shape& s, const uint8_t* x8, const float* x8_scale, const uint8_t* wg_q,
                                    const float* wg_s, const uint8_t* wu_q, const float* wu_s, const void* sched,
                                    void* h, int32_t* status, cudaStream_t st) {
  CUtensorMap a, b, b2;
  const uint64_t rows = (uint64_t)s.R + (uint64_t)s.S * s.T;
  if (!make_tmap_u8_sw128(&a, x8, s.d, rows > 0 ? rows : 1, kBM)) return cudaErrorInvalidValue;
  if (!make_tmap_u8_sw128(&b, wg_q, s.d, (uint64_t)s.G * s.F, 128)) return cudaErrorInvalidValue;
  if (!make_tmap_u8_sw128(&b2, wu_q, s.d, (uint64_t)s.G * s.F, 128)) return cudaErrorInvalidValue;
  W8Args args{};
  args.K = s.d;
  args.n_tiles = s.F / 128;
  args.G = s.G;
  args.b_rows = s.F;
  args.sched = static_cast<const int32_t*>(sched);
  args.a_scale = x8_scale;
  args.scale = wg_s;
  args.scale2 = wu_s;
  args.out = static_cast<__nv_bfloat16*>(h);
  args.ldo = s.F;
  args.status = status;
  return launch_w8a8<0>(a, b, b2, args, s, st);
}

cudaError_t launch_gemm_down_w8a8(const Shape& s, const uint8_t* h8, const float* h8_scale, const uint8_t* wd_q,
                                  const float* wd_s, const void* sched, void* y, int32_t* status, cudaStream_t st) {
  CUtensorMap a, b;
  const uint64_t rows = (uint64_t)s.R + (uint64_t)s.S * s.T;
  if (!make_tmap_u8_sw128(&a, h8, s.F, rows > 0 ? rows : 1, kBM)) return cudaErrorInvalidValue;
  if (!make_tmap_u8_sw128(&b, wd_q, s.F, (uint64_t)s.G * s.d, 256)) return cudaErrorInvalidValue;
  W8Args args{};
  args.K = s.F;
  args.n_tiles = s.d / 256;
  args.G = s.G;
  args.b_rows = s.d;
  args.sched = static_cast<const int32_t*>(sched);
  args.a_scale = h8_scale;
  args.scale = wd_s;
  args.scale2 = wd_s;
  args.out = static_cast<__nv_bfloat16*>(y);
  args.ldo = s.d;
  args.status = status;
  return launch_w8a8<1>(a, b, b, args, s, st);
}

}  // namespace moe
