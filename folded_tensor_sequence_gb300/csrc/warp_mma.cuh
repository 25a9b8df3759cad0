// Warp-level tensor-core helpers (ldmatrix, mma.sync m16n8k16 bf16, cp.async)
// and the swizzled [rows][128] bf16 shared-memory tile layout used by the
// attention kernels.
#pragma once

#include "common.cuh"

namespace tsp {
namespace wm {

constexpr int DH = 128;         // head dim of the bf16 attention kernels
constexpr int CHUNKS = DH / 8;  // 16-byte chunks per row

__host__ __device__ __forceinline__ int64_t min64(int64_t a, int64_t b) { return a < b ? a : b; }

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Swizzled element offset of (row, col) in a [rows][DH] bf16 tile.
__device__ __forceinline__ int swz(int row, int col) {
  return row * DH + ((((col >> 3) ^ (row & 7))) << 3) + (col & 7);
}

__device__ __forceinline__ void cp_async16(uint32_t saddr, const void* g, bool valid) {
  const int n = valid ? 16 : 0;
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(saddr), "l"(g), "r"(n) : "memory");
}
__device__ __forceinline__ void cp_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_wait_all() { asm volatile("cp.async.wait_group 0;" ::: "memory"); }

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Loads `rows` rows of a [*][DH] bf16 matrix (row stride `ld` elements; only
// the first `valid` rows exist) into a swizzled smem tile with cp.async;
// missing rows are zero-filled without touching global memory.
template <int NT>
__device__ __forceinline__ void load_tile_async(__nv_bfloat16* sm, const __nv_bfloat16* g, int64_t ld, int rows,
                                                int valid) {
  const uint32_t base = smem_u32(sm);
  for (int i = threadIdx.x; i < rows * CHUNKS; i += NT) {
    const int r = i / CHUNKS, c = i % CHUNKS;
    const bool ok = r < valid;
    const __nv_bfloat16* src = g + (ok ? (int64_t)r * ld + c * 8 : 0);
    cp_async16(base + swz(r, c * 8) * 2, src, ok);
  }
}

}  // namespace wm
}  // namespace tsp
