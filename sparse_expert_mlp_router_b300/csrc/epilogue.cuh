// Epilogue helpers shared by the persistent expert-MLP kernels: bf16 rows of a warp's 32
// accumulator lanes staged in shared memory and stored as whole sectors.
#pragma once

#include "gemm_common.cuh"
#include "tc_ptx.cuh"

namespace moe {
namespace epi {

constexpr int kStageOutBytes = 32 * 64;   // one epilogue warp's staging: 32 rows x 32 bf16

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}
__device__ __forceinline__ uint4 ld_shared_v4(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr)
               : "memory");
  return v;
}

// One warp's 32 rows of a 32-column chunk: this thread's row as 16 packed bf16 pairs, staged in
// the warp's 2 KB buffer `stg` (row r's 16-byte piece j at r * 64 + 16 * (j ^ ((r >> 1) & 3)):
// free of bank conflicts both row-wise and column-wise) and stored 8 rows x 64 contiguous bytes
// per instruction, rows >= nvalid skipped. Columns [c, c + 32) of rows orow0 + r * ldo.
__device__ __forceinline__ void store_chunk(const uint32_t (&packed)[16], int nvalid, __nv_bfloat16* orow0,
                                            int64_t ldo, int c, uint32_t stg, int lane) {
  const uint32_t my_row = stg + (uint32_t)lane * 64u;
  const uint32_t sw = (uint32_t)((lane >> 1) & 3);
#pragma unroll
  for (int j = 0; j < 4; ++j)
    st_shared_v4(my_row + ((j ^ sw) << 4), packed[4 * j], packed[4 * j + 1], packed[4 * j + 2], packed[4 * j + 3]);
  __syncwarp();
  const int j = lane & 3;
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const int r = 8 * q + (lane >> 2);
    const uint4 v = ld_shared_v4(stg + (uint32_t)r * 64u + ((uint32_t)(j ^ ((r >> 1) & 3)) << 4));
    if (r < nvalid) *reinterpret_cast<uint4*>(orow0 + (int64_t)r * ldo + c + 8 * j) = v;
  }
  __syncwarp();
}

// Accumulator columns of this warp's TMEM lanes -> bf16 rows. GATEUP: columns [0,128) are gate,
// [128,256) up, COLS = 128 outputs of silu(gate) * up; else COLS plain outputs. Output columns
// [half * COLS/2, (half + 1) * COLS/2).
template <bool GATEUP, int COLS>
__device__ __forceinline__ void store_tile(uint32_t t_row, int nvalid, __nv_bfloat16* orow0, int64_t ldo, int half,
                                           uint32_t stg, int lane) {
  if (nvalid <= 0) return;                      // warp-uniform: no row of this warp is valid
  const int c0 = half * (COLS / 2), c1 = c0 + COLS / 2;
#pragma unroll 1
  for (int c = c0; c < c1; c += 32) {
    uint32_t packed[16];
    if (GATEUP) {
      uint32_t gv[32], uv[32];
      ptx::tmem_ld32(t_row + c, gv);
      ptx::tmem_ld32(t_row + 128 + c, uv);
      ptx::tmem_ld_wait();
#pragma unroll
      for (int q = 0; q < 16; ++q) {
        const float h0 = gemm::silu_f(__uint_as_float(gv[2 * q])) * __uint_as_float(uv[2 * q]);
        const float h1 = gemm::silu_f(__uint_as_float(gv[2 * q + 1])) * __uint_as_float(uv[2 * q + 1]);
        packed[q] = gemm::pack_bf16(h0, h1);
      }
    } else {
      uint32_t v[32];
      ptx::tmem_ld32(t_row + c, v);
      ptx::tmem_ld_wait();
#pragma unroll
      for (int q = 0; q < 16; ++q)
        packed[q] = gemm::pack_bf16(__uint_as_float(v[2 * q]), __uint_as_float(v[2 * q + 1]));
    }
    store_chunk(packed, nvalid, orow0, ldo, c, stg, lane);
  }
}

}  // namespace epi
}  // namespace moe
