// Persistent bf16 GEMM on the 5th-generation tensor cores (tcgen05 + TMEM).
//
// C[M][N] = sum_k A[m][k] * B[n][k], both operands K-major bf16, fp32
// accumulation in tensor memory, fused epilogues for the TSP layer:
//   - QKV projection over all weight shards at once (N = h + 2*Hk*dh): the epilogue
//     writes Q in zigzag token order and scatters K/V straight into gathered
//     natural order per head, which is the zigzag K/V all-gather of the TSP
//     attention schedule done for free (ai-trends.today TSP article, "How to
//     Fold a Book");
//   - output projection and down projection, whose K loop walks every weight
//     shard in turn: the row-sharded partial products X_s W_s are summed in
//     the TMEM accumulator, never leaving the SM (the per-rank accumulation of
//     partial outputs that replaces the all-reduce; row split XW = X1W1 + X2W2,
//     r007 chapter "Распределенное обучение", section "Тензорный параллелизм"),
//     plus the residual add;
//   - gate/up projection with SiLU(gate) * up computed from one TMEM tile that
//     holds matching gate and up columns.
//
// Tile 128 x 256 x 64, 4-stage TMA ring (128-byte swizzle).  The grid has one
// CTA per tile; the CTAs that start (one per SM) take over the tiles of those
// that have not started by cancelling their launch (cluster launch control),
// in tile order, so each SM runs one CTA over many tiles.  Warp roles: warp 0
// = TMA producer, warp 1 = MMA issuer (and TMEM owner), warps 2..5 =
// epilogue (one TMEM lane quadrant each).
// Two 256-column accumulators (all 512 TMEM columns) let the epilogue of one
// tile overlap the main loop of the next.
//
// CTA-pair form (CG = 2): a cluster of two CTAs computes a 256 x 256 tile
// with M = 256 MMAs issued by the first CTA.  Each CTA loads
// its own 128 rows of A and 128 of the tile's 256 rows of B (the tensor cores
// of the pair exchange the B halves), so a CTA's stage is 32 KB instead of
// 48 KB and the ring holds 6 stages; each CTA's epilogue reads its own 128
// accumulator rows.  The pair's copies complete on the first CTA's "full"
// barriers, the MMA completions arrive on both CTAs' "empty" and
// "accumulator full" barriers, and both CTAs' epilogue warps release an
// accumulator on the first CTA's "accumulator empty" barrier.
#include <cuda.h>

#include "common.cuh"
#include "internal.h"

namespace tsp {

namespace {

constexpr int BM = 128;
constexpr int BN = 256;
constexpr int BK = 64;
constexpr int THREADS = 192;
constexpr uint32_t A_STAGE_BYTES = BM * BK * 2;  // 16 KB
// Ring of CG-CTA tiles: B rows held per CTA BN / CG (32 or 16 KB a stage).
template <int CG>
__host__ __device__ constexpr int ring_stages() { return CG == 2 ? 6 : 4; }
template <int CG>
__host__ __device__ constexpr uint32_t b_stage_bytes() { return (BN / CG) * BK * 2; }
template <int CG>
__host__ __device__ constexpr uint32_t ring_stage_bytes() { return A_STAGE_BYTES + b_stage_bytes<CG>(); }
// Alignment slack, the ring, and its barriers (and the tile-request ring).
template <int CG>
__host__ __device__ constexpr size_t ring_smem_bytes() { return 1024 + ring_stages<CG>() * ring_stage_bytes<CG>() + 512; }
// Tile requests in flight (slots of the response ring).
constexpr int kResp = 4;
// Epilogue staging in shared memory behind the stage ring (1 KB of barriers
// between them), 32 rows x 32 columns of bf16 (64-byte rows) per matrix:
//   SwiGLU derivative: G and U of a chunk, two chunks per epilogue warp;
//   residual: the chunk's residual (the sum written over it), two chunks per warp;
//   SwiGLU: the chunk's G, U (kept for the backward) and SiLU(G)*U outputs;
//   QKV: the chunk's Q, K or V (V^T: transposed) block, one buffer per warp.
constexpr uint32_t MAT_BYTES = 32 * 64;
template <int EPI>
__host__ __device__ constexpr uint32_t chunk_bytes() {  // one staged chunk of the streamed (loaded) epilogues
  return EPI == EPI_DSWIGLU ? 2 * MAT_BYTES : EPI == EPI_RESID ? MAT_BYTES : 0;
}
// Epilogues that stream loaded chunks through the staging buffers (and own
// the 8 staging barriers).
template <int EPI>
__host__ __device__ constexpr bool streamed_epi() { return chunk_bytes<EPI>() != 0; }
constexpr uint32_t SWG_WARP_BYTES = 3 * MAT_BYTES;
template <int EPI>
__host__ __device__ constexpr size_t stage_bytes() {
  return EPI == EPI_SWIGLU ? 4 * SWG_WARP_BYTES : EPI == EPI_QKV ? 4 * MAT_BYTES : 4 * 2 * chunk_bytes<EPI>();
}
template <int EPI, int CG>
__host__ __device__ constexpr size_t smem_bytes() {
  return ring_smem_bytes<CG>() + (stage_bytes<EPI>() ? 1024 + stage_bytes<EPI>() : 0);
}
static_assert(smem_bytes<EPI_DSWIGLU, 1>() <= 227 * 1024 && smem_bytes<EPI_SWIGLU, 1>() <= 227 * 1024 &&
                  smem_bytes<EPI_RESID, 1>() <= 227 * 1024 && smem_bytes<EPI_QKV, 1>() <= 227 * 1024 &&
                  smem_bytes<EPI_DSWIGLU, 2>() <= 227 * 1024 && smem_bytes<EPI_SWIGLU, 2>() <= 227 * 1024 &&
                  smem_bytes<EPI_RESID, 2>() <= 227 * 1024 && smem_bytes<EPI_QKV, 2>() <= 227 * 1024,
              "shared memory");
// Raster: tiles are visited in bands of group_m m-tiles (all n-tiles of a band
// before the next band), group_m chosen so one band of A is ~32 MB and stays
// in L2 while the B operand streams past it; or, when B is the smaller
// operand (N < M), in bands of group_n n-tiles (kBBandTiles, at most
// kBBandBytes of B) that stay in L2 while A streams past them.
constexpr size_t kBandBytes = size_t(32) << 20;
constexpr size_t kBBandBytes = size_t(64) << 20;
constexpr int kBBandTiles = 16;  // 12 and 24 measured: equal and 3 % slower (headline layer)
constexpr uint32_t TMEM_COLS = 512;
#ifndef TSP_GEMM_PAIRS
#define TSP_GEMM_PAIRS 1
#endif
// CTA-pair tiles for GEMMs of more than 128 rows (0 at build time: one-CTA tiles only).
constexpr bool kGemmPairs = TSP_GEMM_PAIRS != 0;

struct GemmShape {
  int M, N, K;
  int num_m, num_n, num_tiles, kblocks;
  int group_m;  // > 0: bands of group_m m-tiles (A resident, B streams)
  int group_n;  // > 0: bands of group_n n-tiles (B resident, A streams)
};

__device__ __forceinline__ void tile_coords(int t, const GemmShape& s, int& mt, int& nt) {
  if (s.group_n > 0) {
    const int per_group = s.group_n * s.num_m;
    const int group = t / per_group;
    const int first_n = group * s.group_n;
    const int gsz = min(s.num_n - first_n, s.group_n);
    const int in_g = t - group * per_group;
    nt = first_n + in_g % gsz;
    mt = in_g / gsz;
    return;
  }
  const int per_group = s.group_m * s.num_n;
  const int group = t / per_group;
  const int first_m = group * s.group_m;
  const int gsz = min(s.num_m - first_m, s.group_m);
  const int in_g = t - group * per_group;
  mt = first_m + in_g % gsz;
  nt = in_g / gsz;
}

__device__ __forceinline__ void store32_bf16(void* dst, const float (&v)[32]) {
  uint4* d = reinterpret_cast<uint4*>(dst);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    d[i] = make_uint4(pack_bf16x2(v[8 * i + 0], v[8 * i + 1]), pack_bf16x2(v[8 * i + 2], v[8 * i + 3]),
                      pack_bf16x2(v[8 * i + 4], v[8 * i + 5]), pack_bf16x2(v[8 * i + 6], v[8 * i + 7]));
  }
}

__device__ __forceinline__ float silu_f(float z) { return z / (1.0f + __expf(-z)); }

// TMA tensor store shared -> global (bulk-group completion).  c0 * 2 bytes
// must be a multiple of 16; rows beyond the tensor are not written.
__device__ __forceinline__ void tma_store_2d(const CUtensorMap* tm, int c0, int c1, const void* src) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%1, %2}], [%3];" ::"l"(
                   reinterpret_cast<uint64_t>(tm)),
               "r"(c0), "r"(c1), "r"(smem_u32(src))
               : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// Until every committed bulk store of this thread has read its shared memory.
__device__ __forceinline__ void bulk_wait_read_all() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
// Until every committed bulk store of this thread has completed.
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
__device__ __forceinline__ void fence_proxy_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// Packed gate_up column of dM column n: 128-column gate blocks interleaved
// with their up blocks (the up column is this + 128).
__device__ __forceinline__ int gu_col(int n) { return (n / 128) * 256 + n % 128; }

// Zigzag row m of [D][B][2C] -> natural row b*S + pos.
__device__ __forceinline__ int64_t zigzag_row_to_natural(int64_t m, const EpiParams& ep) {
  const int64_t twoC = 2 * (int64_t)ep.C;
  const int64_t per_rank = (int64_t)ep.B * twoC;
  const int64_t r = m / per_rank;
  const int64_t rem = m - r * per_rank;
  const int64_t b = rem / twoC;
  const int64_t k = rem - b * twoC;
  const int64_t p = (k < ep.C) ? r * ep.C + k : (2 * ep.D - 1 - r) * ep.C + (k - ep.C);
  return b * ep.S + p;
}

// Zigzag row m of [D][B][2C] -> (batch b, natural position p).
__device__ __forceinline__ void zigzag_row_to_pos(int64_t m, const EpiParams& ep, int& b, int64_t& p) {
  const int64_t twoC = 2 * (int64_t)ep.C;
  const int64_t per_rank = (int64_t)ep.B * twoC;
  const int r = (int)(m / per_rank);
  const int64_t rem = m - (int64_t)r * per_rank;
  b = (int)(rem / twoC);
  const int64_t k = rem - (int64_t)b * twoC;
  p = (k < ep.C) ? (int64_t)r * ep.C + k : (int64_t)(2 * ep.D - 1 - r) * ep.C + (k - ep.C);
}

// AMN / BMN: the operand is MN-major (global [K][M] / [K][N], M / N
// contiguous), loaded as 64-wide boxes of [64 K rows][64 elements] into 8 KB
// chunks and described with the MN-major 128-byte-swizzle descriptor.
// tmE0 / tmE1: epilogue tensor maps (32 x 32 boxes, 64-byte swizzle):
//   EPI_DSWIGLU: saved G|U (read) / dG|dU (written);
//   EPI_RESID:   the residual (read) / the sum (written);
//   EPI_SWIGLU:  the G|U copy kept for the backward / SiLU(G)*U;
//   EPI_QKV:     Q [T][h] / K [B*Hk*S][dh] / tmE2: V, [B*Hk*S][dh] or V^T
//                [B*Hk*dh][S] (only when the chunk length is a multiple of 32).
template <int EPI, bool AMN, bool BMN, int CG>
__global__ void __launch_bounds__(THREADS, 1)
    gemm_bf16_tc_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                        const __grid_constant__ CUtensorMap tmE0, const __grid_constant__ CUtensorMap tmE1,
                        const __grid_constant__ CUtensorMap tmE2,
                        const GemmShape shape, const EpiParams ep) {
  constexpr int STAGES = ring_stages<CG>();
  constexpr uint32_t B_STAGE_BYTES = b_stage_bytes<CG>();
  constexpr uint32_t STAGE_BYTES = ring_stage_bytes<CG>();
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* smA = smem;
  uint8_t* smB = smem + STAGES * A_STAGE_BYTES;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + STAGES * STAGE_BYTES);
  uint64_t* empty = full + STAGES;
  uint64_t* tfull = empty + STAGES;
  uint64_t* tempty = tfull + 2;
  uint64_t* drain = tempty + 2;
  uint64_t* gbar = drain + 1;  // [4 warps][2] staging buffers of the streamed epilogues
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(gbar + 8);
  uint8_t* gstage = smem + STAGES * STAGE_BYTES + 1024;  // epilogue staging (all but EPI_STORE)
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  // Tile-request responses (kResp x 16 bytes, 16-byte aligned) and their barriers
  uint64_t* resp_full = reinterpret_cast<uint64_t*>(tmem_slot + 2);
  uint64_t* resp_empty = resp_full + kResp;
  uint8_t* resp = reinterpret_cast<uint8_t*>(resp_empty + kResp);

  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  // Tiles of TM rows: this CTA's rows of tile mt start at mt * TM + roff.
  // The pair walks its tiles together, starting with tile t0.
  constexpr int TM = BM * CG;
  const uint32_t crank = CG == 2 ? cluster_ctarank() : 0;
  const int roff = (int)crank * BM;
  const int t0 = CG == 2 ? (int)blockIdx.x / 2 : (int)blockIdx.x;
  const bool leader = crank == 0;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tfull[a], 1);
      // CTA pairs: one arrival per epilogue warp of both CTAs
      mbar_init(&tempty[a], CG == 2 ? 8 : 128);
    }
    mbar_init(drain, 1);
    for (int r = 0; r < kResp; ++r) {
      mbar_init(&resp_full[r], 1);
      // readers: the (first) CTA's producer, MMA thread and 4 epilogue warps,
      // and a pair's second CTA's producer and 4 epilogue warps
      mbar_init(&resp_empty[r], CG == 2 ? 11 : 6);
    }
    if constexpr (streamed_epi<EPI>())
      for (int i = 0; i < 8; ++i) mbar_init(&gbar[i], 1);
    *abort_flag = 0;
    fence_mbarrier_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
    if constexpr (EPI == EPI_DSWIGLU || EPI == EPI_SWIGLU || EPI == EPI_RESID) {
      if (EPI != EPI_SWIGLU || ep.aux) tma_prefetch_desc(&tmE0);  // the SwiGLU map exists only with aux
      tma_prefetch_desc(&tmE1);
    }
    if constexpr (EPI == EPI_QKV) {
      if (ep.C % 32 == 0) {  // the maps exist only then
        tma_prefetch_desc(&tmE0);
        tma_prefetch_desc(&tmE1);
        tma_prefetch_desc(&tmE2);
      }
    }
  }
  if (warp == 1) {
    if constexpr (CG == 2) {
      tmem_alloc_pair(tmem_slot, TMEM_COLS);
      tmem_relinquish_pair();
    } else {
      tmem_alloc(tmem_slot, TMEM_COLS);
      tmem_relinquish();
    }
  }
  tc_fence_before();
  if constexpr (CG == 2)
    cluster_sync_all();  // both CTAs' barriers initialised before any copy or commit reaches them
  else
    __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  // Tile sequence.  The grid has one CTA (pair: one cluster) per tile, and
  // step 0 is the CTA's (pair's) own tile.  At the start of step j the
  // (first CTA's) producer asks for the tile of step j + 1 by cancelling the
  // launch of a CTA (cluster) that has not started, whose tile is then done
  // here: the tiles in flight stay a window of consecutive tiles however
  // the CTAs' speeds differ, and the operands they share meet in L2.  (With
  // a fixed tile stride the CTAs drift apart over many waves: the CTA-pair
  // down projection at 2 x 16K tokens read 9.55 GB from DRAM that way, 4.02
  // GB in this order.)  The response lands in ring slot j % kResp (of both
  // CTAs of a pair); every role reads its own copy and releases the slot on
  // the (first) CTA's barrier.
  // next_tile: (one thread) the tile of step s >= 1, or -1 when none is left.
  auto next_tile = [&](uint32_t s, unsigned int code) -> int {
    const uint32_t slot = (s - 1) % kResp;
    if (!mbar_wait<CG == 2>(&resp_full[slot], ((s - 1) / kResp) & 1, abort_flag, ep.err, code)) return -1;
    const int x = clc_cancelled_x(resp + slot * 16);
    if (leader)
      mbar_arrive(&resp_empty[slot]);
    else
      mbar_arrive_cluster(cluster_smem_addr(&resp_empty[slot], 0));
    return x < 0 ? -1 : x / CG;
  };

  if (warp == 0) {
    // ---------------- TMA producer ----------------
    if (lane == 0) {
      uint32_t it = 0, step = 0;
      bool ok = true;
      for (int t = t0; t >= 0 && ok; t = next_tile(++step, (KID_GEMM_TC << 8) | 10)) {
        {
          // ask for the tile of the next step (no request follows one that found none)
          const uint32_t slot = step % kResp;
          if (leader) {
            if (!mbar_wait<CG == 2>(&resp_empty[slot], ((step / kResp) & 1) ^ 1, abort_flag, ep.err,
                                    (KID_GEMM_TC << 8) | 9)) {
              ok = false;
              break;
            }
            mbar_arrive_expect_tx(&resp_full[slot], 16);
            if constexpr (CG == 2)
              clc_try_cancel_all(resp + slot * 16, &resp_full[slot]);
            else
              clc_try_cancel(resp + slot * 16, &resp_full[slot]);
          } else {
            mbar_arrive_expect_tx(&resp_full[slot], 16);
          }
        }
        int mt, nt;
        tile_coords(t, shape, mt, nt);
        // (the second CTA's rows of a pair's last tile may lie past M: zeros)
        const int64_t r_a = (int64_t)mt * TM + roff;
        const int arow = (ep.a_natural && r_a < shape.M) ? (int)zigzag_row_to_natural(r_a, ep) : (int)r_a;
        for (int kb = 0; kb < shape.kblocks; ++kb, ++it) {
          const int s = it % STAGES;
          const uint32_t ph = (it / STAGES) & 1;
          if (!mbar_wait(&empty[s], ph ^ 1, abort_flag, ep.err, (KID_GEMM_TC << 8) | 1)) {
            ok = false;
            break;
          }
          if constexpr (CG == 2) {
            // The first CTA's barrier counts both CTAs' bytes; the second CTA's
            // copies complete on it (possibly before this arrival: the
            // transaction count may go negative within a phase).  MN-major
            // operands come as 64-wide boxes of this CTA's 128 rows of A / of B.
            const int b0 = nt * BN + (int)crank * (BN / 2);
            if (leader) {
              mbar_arrive_expect_tx(&full[s], 2 * STAGE_BYTES);
              if constexpr (AMN) {
#pragma unroll
                for (int c = 0; c < BM / 64; ++c)
                  tma_load_2d(smA + s * A_STAGE_BYTES + c * 8192, &tmA, (int)r_a + c * 64, kb * BK, &full[s]);
              } else {
                tma_load_2d(smA + s * A_STAGE_BYTES, &tmA, kb * BK, arow, &full[s]);
              }
              if constexpr (BMN) {
#pragma unroll
                for (int c = 0; c < BN / 2 / 64; ++c)
                  tma_load_2d(smB + s * B_STAGE_BYTES + c * 8192, &tmB, b0 + c * 64, kb * BK, &full[s]);
              } else {
                tma_load_2d(smB + s * B_STAGE_BYTES, &tmB, kb * BK, b0, &full[s]);
              }
            } else {
              const uint32_t fb = cluster_smem_addr(&full[s], 0);
              if constexpr (AMN) {
#pragma unroll
                for (int c = 0; c < BM / 64; ++c)
                  tma_load_2d_pair(smA + s * A_STAGE_BYTES + c * 8192, &tmA, (int)r_a + c * 64, kb * BK, fb);
              } else {
                tma_load_2d_pair(smA + s * A_STAGE_BYTES, &tmA, kb * BK, arow, fb);
              }
              if constexpr (BMN) {
#pragma unroll
                for (int c = 0; c < BN / 2 / 64; ++c)
                  tma_load_2d_pair(smB + s * B_STAGE_BYTES + c * 8192, &tmB, b0 + c * 64, kb * BK, fb);
              } else {
                tma_load_2d_pair(smB + s * B_STAGE_BYTES, &tmB, kb * BK, b0, fb);
              }
            }
            continue;
          }
          mbar_arrive_expect_tx(&full[s], STAGE_BYTES);
          if constexpr (AMN) {
#pragma unroll
            for (int c = 0; c < BM / 64; ++c)
              tma_load_2d(smA + s * A_STAGE_BYTES + c * 8192, &tmA, mt * BM + c * 64, kb * BK, &full[s]);
          } else {
            tma_load_2d(smA + s * A_STAGE_BYTES, &tmA, kb * BK, arow, &full[s]);
          }
          if constexpr (BMN) {
#pragma unroll
            for (int c = 0; c < BN / 64; ++c)
              tma_load_2d(smB + s * B_STAGE_BYTES + c * 8192, &tmB, nt * BN + c * 64, kb * BK, &full[s]);
          } else {
            tma_load_2d(smB + s * B_STAGE_BYTES, &tmB, kb * BK, nt * BN, &full[s]);
          }
        }
      }
      // Before leaving, make sure every copy this thread issued has landed
      // (always true on the normal path, bounded on the abort path).  The
      // second CTA of a pair cannot wait on the first CTA's barriers; its
      // copies have landed once the first CTA's MMAs have consumed them, which
      // the closing cluster barrier orders before either CTA exits.
      const uint32_t issued = it;
      const uint32_t first = issued > (uint32_t)STAGES ? issued - STAGES : 0;
      for (uint32_t j = first; j < issued && leader; ++j) {
        volatile int dummy = 0;
        mbar_wait(&full[j % STAGES], (j / STAGES) & 1, &dummy, ep.err, (KID_GEMM_TC << 8) | 2);
      }
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer ----------------
    if (lane == 0 && leader) {
      constexpr uint32_t idesc = idesc_bf16_f32(TM, BN, AMN, BMN);
      uint32_t it = 0, tl = 0;
      bool ok = true;
      for (int t = t0; t >= 0 && ok; t = next_tile(tl + 1, (KID_GEMM_TC << 8) | 11), ++tl) {
        const int acc = tl & 1;
        const uint32_t aph = (tl >> 1) & 1;
        if (!mbar_wait<CG == 2>(&tempty[acc], aph ^ 1, abort_flag, ep.err, (KID_GEMM_TC << 8) | 3)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + acc * BN;
        for (int kb = 0; kb < shape.kblocks; ++kb, ++it) {
          const int s = it % STAGES;
          const uint32_t ph = (it / STAGES) & 1;
          if (!mbar_wait(&full[s], ph, abort_flag, ep.err, (KID_GEMM_TC << 8) | 4)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sa = smem_u32(smA + s * A_STAGE_BYTES), sb = smem_u32(smB + s * B_STAGE_BYTES);
#pragma unroll
          for (int k = 0; k < BK / 16; ++k) {
            // K-major: +32 bytes along K inside the 128-byte swizzle atom (+2 in the >>4 field);
            // MN-major: +16 K rows = +2048 bytes.
            const uint64_t adesc = AMN ? sdesc_mn_sw128(sa + 2048 * k, 8192) : sdesc_kmajor_sw128(sa) + 2 * k;
            const uint64_t bdesc = BMN ? sdesc_mn_sw128(sb + 2048 * k, 8192) : sdesc_kmajor_sw128(sb) + 2 * k;
            if constexpr (CG == 2)
              umma_bf16_pair(d_tmem, adesc, bdesc, idesc, (kb | k) != 0);
            else
              umma_bf16(d_tmem, adesc, bdesc, idesc, (kb | k) != 0);
          }
          if constexpr (CG == 2)
            umma_commit_pair_mc(&empty[s], 0x3);  // both CTAs' stage s is free
          else
            umma_commit(&empty[s]);
        }
        if (!ok) break;
        if constexpr (CG == 2)
          umma_commit_pair_mc(&tfull[acc], 0x3);
        else
          umma_commit(&tfull[acc]);
      }
      // Drain: wait until every MMA issued above has completed before TMEM is freed.
      if constexpr (CG == 2)
        umma_commit_pair(drain);
      else
        umma_commit(drain);
      volatile int dummy = 0;
      mbar_wait(drain, 0, &dummy, ep.err, (KID_GEMM_TC << 8) | 5);
    }
  } else {
    // ---------------- epilogue: warps 2..5 ----------------
    const int quad = warp & 3;  // TMEM lanes this warp may access: 32*quad .. 32*quad+31
    const int row = quad * 32 + lane;
    // Streamed epilogues (SwiGLU derivative: the warp's 32 rows x 32 columns
    // of G and of U; residual: of the residual) pass each chunk through two
    // staging buffers; chunk q (counted over all of the CTA's tiles) uses
    // buffer q & 1.  Lane 0 issues the TMA loads two chunks ahead and the TMA
    // stores of the results, which the threads write over the loaded data.
    constexpr uint32_t CH = chunk_bytes<EPI>();
    uint8_t* gbuf = gstage + quad * 2 * CH;
    uint64_t* gb_full = gbar + quad * 2;
    uint32_t q_issued = 0, q_done = 0;
    auto issue_chunk = [&](int tt, int c) {  // lane 0: the loaded data of chunk c of tile tt
      int mq, nq;
      tile_coords(tt, shape, mq, nq);
      const int b = q_issued & 1;
      uint8_t* dst = gbuf + b * CH;
      const int r0 = mq * TM + roff + quad * 32;
      mbar_arrive_expect_tx(&gb_full[b], CH);
      if constexpr (EPI == EPI_DSWIGLU) {
        const int gcol = gu_col(nq * BN + c * 32);
        tma_load_2d(dst, &tmE0, gcol, r0, &gb_full[b]);
        tma_load_2d(dst + MAT_BYTES, &tmE0, gcol + 128, r0, &gb_full[b]);
      } else {
        // 32 zigzag rows of a chunk of 128-row multiples are 32 consecutive natural rows
        const int rr = (ep.resid_natural && r0 < shape.M) ? (int)zigzag_row_to_natural(r0, ep) : r0;
        tma_load_2d(dst, &tmE0, nq * BN + c * 32, rr, &gb_full[b]);
      }
      ++q_issued;
    };
    constexpr bool streamed = streamed_epi<EPI>();
    if constexpr (streamed) {
      if (lane == 0) {
        issue_chunk(t0, 0);
        issue_chunk(t0, 1);
      }
    }
    bool epi_ok = true;
    uint32_t tl = 0;
    for (int t = t0, tn = -1; t >= 0 && epi_ok; t = tn, ++tl) {
      int mt, nt;
      tile_coords(t, shape, mt, nt);
      const int acc = tl & 1;
      const uint32_t aph = (tl >> 1) & 1;
      // Warp-uniform decision: tcgen05.ld below needs every lane of the warp.
      const bool got = mbar_wait(&tfull[acc], aph, abort_flag, ep.err, (KID_GEMM_TC << 8) | 6);
      if (!__all_sync(0xffffffffu, got)) break;
      // the tile after this one (lane 0 reads it, the warp shares it)
      tn = lane == 0 ? next_tile(tl + 1, (KID_GEMM_TC << 8) | 12) : 0;
      tn = __shfl_sync(0xffffffffu, tn, 0);
      tc_fence_after();
      const int64_t m = (int64_t)mt * TM + roff + row;
      const bool valid = m < shape.M;
      const uint32_t tbase = tmem_base + (static_cast<uint32_t>(quad * 32) << 16) + acc * BN;
      if constexpr (EPI == EPI_SWIGLU) {
        // The tile's 256 columns are a 128-column gate block and its up block.
        // Per 32-column chunk the warp stages its 32 rows of SiLU(G)*U (and, for
        // the backward, of G and U) in shared memory (64-byte rows, 64-byte
        // swizzle: 16-byte unit j of row r at unit j ^ ((r >> 1) & 3)) and one
        // lane stores them by TMA; rows past M are not written.
        uint8_t* sg = gstage + quad * SWG_WARP_BYTES;
        uint8_t* su = sg + 2048;
        uint8_t* so = sg + 4096;
        const bool keep = ep.aux != nullptr;
        const int r0 = mt * TM + roff + quad * 32;
#pragma unroll 1
        for (int c = 0; c < 4; ++c) {
          float g[32], u[32];
          tmem_ld32(tbase + c * 32, g);
          tmem_ld32(tbase + 128 + c * 32, u);
          float o[32];
#pragma unroll
          for (int i = 0; i < 32; ++i) o[i] = silu_f(g[i]) * u[i];
          if (lane == 0) bulk_wait_read_all();  // the previous chunk's stores have read the buffer
          __syncwarp();
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const uint32_t off = lane * 64 + ((j ^ ((lane >> 1) & 3)) << 4);
            if (keep) {
              *reinterpret_cast<uint4*>(sg + off) =
                  make_uint4(pack_bf16x2(g[8 * j + 0], g[8 * j + 1]), pack_bf16x2(g[8 * j + 2], g[8 * j + 3]),
                             pack_bf16x2(g[8 * j + 4], g[8 * j + 5]), pack_bf16x2(g[8 * j + 6], g[8 * j + 7]));
              *reinterpret_cast<uint4*>(su + off) =
                  make_uint4(pack_bf16x2(u[8 * j + 0], u[8 * j + 1]), pack_bf16x2(u[8 * j + 2], u[8 * j + 3]),
                             pack_bf16x2(u[8 * j + 4], u[8 * j + 5]), pack_bf16x2(u[8 * j + 6], u[8 * j + 7]));
            }
            *reinterpret_cast<uint4*>(so + off) =
                make_uint4(pack_bf16x2(o[8 * j + 0], o[8 * j + 1]), pack_bf16x2(o[8 * j + 2], o[8 * j + 3]),
                           pack_bf16x2(o[8 * j + 4], o[8 * j + 5]), pack_bf16x2(o[8 * j + 6], o[8 * j + 7]));
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0 && r0 < shape.M) {
            if (keep) {
              tma_store_2d(&tmE0, nt * BN + c * 32, r0, sg);
              tma_store_2d(&tmE0, nt * BN + 128 + c * 32, r0, su);
            }
            tma_store_2d(&tmE1, nt * (BN / 2) + c * 32, r0, so);
            bulk_commit();
          }
        }
      } else if constexpr (EPI == EPI_DSWIGLU) {
        // acc = dM[m][f]; dG = dM * u * s * (1 + g (1 - s)), dU = dM * g * s with
        // s = sigmoid(g), in the packed gate_up order.  The thread's row of G and
        // U is read from the staging buffer (64-byte rows, 64-byte swizzle: 16-byte
        // unit j of row r sits at unit j ^ ((r >> 1) & 3)), dG and dU are written
        // over it, and the buffer goes back to global memory by TMA.  Rows past
        // M load as zeros and are not stored.
#pragma unroll 1
        for (int c = 0; c < BN / 32; ++c, ++q_done) {
          float v[32];
          tmem_ld32(tbase + c * 32, v);
          const int gb = q_done & 1;
          const bool landed =
              mbar_wait(&gb_full[gb], (q_done >> 1) & 1, abort_flag, ep.err, (KID_GEMM_TC << 8) | 7);
          if (!__all_sync(0xffffffffu, landed)) {
            epi_ok = false;
            break;
          }
          uint8_t* gs = gbuf + gb * CH;
          uint8_t* us = gs + MAT_BYTES;
          uint32_t off[4];
          uint4 g4[4], u4[4];
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            off[j] = lane * 64 + ((j ^ ((lane >> 1) & 3)) << 4);
            g4[j] = *reinterpret_cast<const uint4*>(gs + off[j]);
            u4[j] = *reinterpret_cast<const uint4*>(us + off[j]);
          }
          float dg[32], du[32];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const uint32_t gw[4] = {g4[i].x, g4[i].y, g4[i].z, g4[i].w};
            const uint32_t uw[4] = {u4[i].x, u4[i].y, u4[i].z, u4[i].w};
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              const float2 g2 = unpack_bf16x2(gw[j]), u2 = unpack_bf16x2(uw[j]);
              const float gg[2] = {g2.x, g2.y}, uu[2] = {u2.x, u2.y};
#pragma unroll
              for (int e = 0; e < 2; ++e) {
                const int k = 8 * i + 2 * j + e;
                const float sg = 1.0f / (1.0f + __expf(-gg[e]));
                du[k] = v[k] * gg[e] * sg;
                dg[k] = v[k] * uu[e] * sg * (1.0f + gg[e] * (1.0f - sg));
              }
            }
          }
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            *reinterpret_cast<uint4*>(gs + off[j]) =
                make_uint4(pack_bf16x2(dg[8 * j + 0], dg[8 * j + 1]), pack_bf16x2(dg[8 * j + 2], dg[8 * j + 3]),
                           pack_bf16x2(dg[8 * j + 4], dg[8 * j + 5]), pack_bf16x2(dg[8 * j + 6], dg[8 * j + 7]));
            *reinterpret_cast<uint4*>(us + off[j]) =
                make_uint4(pack_bf16x2(du[8 * j + 0], du[8 * j + 1]), pack_bf16x2(du[8 * j + 2], du[8 * j + 3]),
                           pack_bf16x2(du[8 * j + 4], du[8 * j + 5]), pack_bf16x2(du[8 * j + 6], du[8 * j + 7]));
          }
          fence_proxy_async_smem();  // the stores below read what the threads wrote
          __syncwarp();
          if (lane == 0) {
            const int gcol = gu_col(nt * BN + c * 32), r0 = mt * TM + roff + quad * 32;
            if (r0 < shape.M) {  // a box starting past the last row has nothing to store
              tma_store_2d(&tmE1, gcol, r0, gs);
              tma_store_2d(&tmE1, gcol + 128, r0, us);
              bulk_commit();
            }
            bulk_wait_read_all();  // the buffer is free once the stores have read it
            if (c + 2 < BN / 32)
              issue_chunk(t, c + 2);
            else if (tn >= 0)
              issue_chunk(tn, c + 2 - BN / 32);
          }
          __syncwarp();
        }
        if (!epi_ok) break;
      } else if constexpr (EPI == EPI_RESID) {
        // out = resid + acc: the chunk's residual arrives by TMA in the staging
        // buffer (64-byte swizzle), the sum is written over it and stored by
        // TMA.  Residual and output rows follow the natural order when asked
        // (32 zigzag rows of a chunk of 128-row multiples are 32 consecutive
        // natural rows); rows past M are not stored.
        const int r0 = mt * TM + roff + quad * 32;
        const int orow = (ep.out_natural && r0 < shape.M) ? (int)zigzag_row_to_natural(r0, ep) : r0;
#pragma unroll 1
        for (int c = 0; c < BN / 32; ++c, ++q_done) {
          float v[32];
          tmem_ld32(tbase + c * 32, v);
          const int gb = q_done & 1;
          const bool landed =
              mbar_wait(&gb_full[gb], (q_done >> 1) & 1, abort_flag, ep.err, (KID_GEMM_TC << 8) | 7);
          if (!__all_sync(0xffffffffu, landed)) {
            epi_ok = false;
            break;
          }
          uint8_t* rs = gbuf + gb * CH;
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            uint4* cell = reinterpret_cast<uint4*>(rs + lane * 64 + ((j ^ ((lane >> 1) & 3)) << 4));
            const uint4 w = *cell;
            const float2 a = unpack_bf16x2(w.x), bb = unpack_bf16x2(w.y), cc = unpack_bf16x2(w.z),
                         dd = unpack_bf16x2(w.w);
            *cell = make_uint4(pack_bf16x2(v[8 * j + 0] + a.x, v[8 * j + 1] + a.y),
                               pack_bf16x2(v[8 * j + 2] + bb.x, v[8 * j + 3] + bb.y),
                               pack_bf16x2(v[8 * j + 4] + cc.x, v[8 * j + 5] + cc.y),
                               pack_bf16x2(v[8 * j + 6] + dd.x, v[8 * j + 7] + dd.y));
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            if (r0 < shape.M) {
              tma_store_2d(&tmE1, nt * BN + c * 32, orow, rs);
              bulk_commit();
            }
            bulk_wait_read_all();
            if (c + 2 < BN / 32)
              issue_chunk(t, c + 2);
            else if (tn >= 0)
              issue_chunk(tn, c + 2 - BN / 32);
          }
          __syncwarp();
        }
        if (!epi_ok) break;
      } else if (EPI == EPI_QKV && ep.C % 32 == 0) {
        // Q|K|V scatter by TMA.  A 32-column chunk lies in one head of one of Q,
        // K, V (a shard's Q, K and V blocks are multiples of 128 columns), and
        // the warp's 32 zigzag rows lie in one chunk of the sequence, i.e. are 32
        // consecutive positions p0.. of one sequence b.  The warp stages the
        // 32 x 32 block (64-byte rows, 64-byte swizzle; V^T transposed: rows are
        // head dims, columns positions) and one lane stores it as one box.
        uint8_t* sb = gstage + quad * MAT_BYTES;
        const int r0 = mt * TM + roff + quad * 32;
        int b0 = 0;
        int64_t p0 = 0;
        if (r0 < shape.M) zigzag_row_to_pos(r0, ep, b0, p0);
#pragma unroll 1
        for (int c = 0; c < BN / 32; ++c) {
          float v[32];
          tmem_ld32(tbase + c * 32, v);
          const int n = nt * BN + c * 32;
          const int hs = ep.h / ep.D, ks = ep.Hk * ep.dh / ep.D;
          const int sh = n / (hs + 2 * ks);
          const int within = n - sh * (hs + 2 * ks);
          const int which = within < hs ? 0 : (within < hs + ks ? 1 : 2);
          const int cin = within - (which == 0 ? 0 : hs + (which - 1) * ks);
          const int head = sh * ((which == 0 ? ep.H : ep.Hk) / ep.D) + cin / ep.dh;
          const int d0 = cin % ep.dh;
          const bool vt = which == 2 && ep.v_transposed;
          if (lane == 0) bulk_wait_read_all();  // the previous chunk's store has read the buffer
          __syncwarp();
          if (vt) {
            // element (head dim i, position lane): row i, 16-byte unit lane / 8
#pragma unroll
            for (int i = 0; i < 32; ++i) {
              __nv_bfloat16* e = reinterpret_cast<__nv_bfloat16*>(
                  sb + i * 64 + (((lane >> 3) ^ ((i >> 1) & 3)) << 4) + (lane & 7) * 2);
              *e = __float2bfloat16_rn(v[i]);
            }
          } else {
#pragma unroll
            for (int j = 0; j < 4; ++j)
              *reinterpret_cast<uint4*>(sb + lane * 64 + ((j ^ ((lane >> 1) & 3)) << 4)) =
                  make_uint4(pack_bf16x2(v[8 * j + 0], v[8 * j + 1]), pack_bf16x2(v[8 * j + 2], v[8 * j + 3]),
                             pack_bf16x2(v[8 * j + 4], v[8 * j + 5]), pack_bf16x2(v[8 * j + 6], v[8 * j + 7]));
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0 && r0 < shape.M) {
            const int kvrow = ((int)b0 * ep.Hk + head) * ep.S + (int)p0;  // K / V row of position p0
            if (which == 0)
              tma_store_2d(&tmE0, head * ep.dh + d0, r0, sb);
            else if (which == 1)
              tma_store_2d(&tmE1, d0, kvrow, sb);
            else if (!vt)
              tma_store_2d(&tmE2, d0, kvrow, sb);
            else
              tma_store_2d(&tmE2, (int)p0, ((int)b0 * ep.Hk + head) * ep.dh + d0, sb);
            bulk_commit();
          }
        }
      } else {
        int b = 0;
        int64_t p = 0;
        if constexpr (EPI == EPI_QKV) {
          if (valid) zigzag_row_to_pos(m, ep, b, p);
        }
#pragma unroll 1
        for (int c = 0; c < BN / 32; ++c) {
          float v[32];
          tmem_ld32(tbase + c * 32, v);
          if (!valid) continue;
          const int64_t n = (int64_t)nt * BN + c * 32;
          if constexpr (EPI == EPI_STORE) {
            if (ep.split_col > 0 && n >= ep.split_col)
              store32_bf16(reinterpret_cast<__nv_bfloat16*>(ep.aux) + m * ep.ldx + (n - ep.split_col), v);
            else
              store32_bf16(reinterpret_cast<__nv_bfloat16*>(ep.out) + m * ep.ldo + n, v);
          } else if constexpr (EPI == EPI_QKV) {
            // packed column n -> (shard s, which of q/k/v, head, d); a shard's
            // columns are Q (h/D) | K (Hk*dh/D) | V (Hk*dh/D)
            const int hs = ep.h / ep.D, ks = ep.Hk * ep.dh / ep.D;
            const int s = (int)(n / (hs + 2 * ks));
            const int within = (int)(n - (int64_t)s * (hs + 2 * ks));
            const int which = within < hs ? 0 : (within < hs + ks ? 1 : 2);
            const int cin = within - (which == 0 ? 0 : hs + (which - 1) * ks);
            const int head = s * ((which == 0 ? ep.H : ep.Hk) / ep.D) + cin / ep.dh;
            const int d = cin % ep.dh;
            if (which == 0) {
              store32_bf16(reinterpret_cast<__nv_bfloat16*>(ep.q) + m * ep.h + head * ep.dh + d, v);
            } else if (which == 1 || !ep.v_transposed) {
              __nv_bfloat16* dst = reinterpret_cast<__nv_bfloat16*>(which == 1 ? ep.k : ep.v);
              store32_bf16(dst + (((int64_t)b * ep.Hk + head) * ep.S + p) * ep.dh + d, v);
            } else {
              // V^T [B][Hk][dh][S]: lanes hold consecutive positions, so each store is coalesced
              __nv_bfloat16* dst = reinterpret_cast<__nv_bfloat16*>(ep.v) +
                                   (((int64_t)b * ep.Hk + head) * ep.dh + d) * ep.S + p;
#pragma unroll
              for (int i = 0; i < 32; ++i) dst[(int64_t)i * ep.S] = __float2bfloat16_rn(v[i]);
            }
          }
        }
      }
      tc_fence_before();
      if constexpr (CG == 2) {
        // one arrival per warp on the first CTA's barrier (the warp's TMEM
        // loads have all completed: tcgen05.ld waits inside each load)
        __syncwarp();
        if (lane == 0) {
          if (leader)
            mbar_arrive(&tempty[acc]);
          else
            mbar_arrive_cluster(cluster_smem_addr(&tempty[acc], 0));
        }
      } else {
        mbar_arrive(&tempty[acc]);
      }
    }
    if constexpr (EPI == EPI_SWIGLU || EPI == EPI_QKV) {
      if (lane == 0) bulk_wait_all();  // every staged store complete before leaving (none on the per-row path)
      __syncwarp();
    }
    if constexpr (streamed) {
      // Before leaving: every staged store complete, and (on the abort path)
      // every load still in flight landed (bounded).
      if (lane == 0) {
        bulk_wait_all();
        volatile int dummy = 0;
        for (uint32_t q = q_done; q < q_issued; ++q)
          mbar_wait(&gb_full[q & 1], (q >> 1) & 1, &dummy, ep.err, (KID_GEMM_TC << 8) | 8);
      }
      __syncwarp();
    }
  }

  tc_fence_before();
  if constexpr (CG == 2) {
    // Neither CTA leaves (or frees TMEM) while the other may still signal its
    // barriers or the first CTA's MMAs may still write its TMEM.
    __syncwarp();
    cluster_sync_all();
  } else {
    __syncthreads();
  }
  if (warp == 1) {
    tc_fence_after();
    if constexpr (CG == 2)
      tmem_dealloc_pair(tmem_base, TMEM_COLS);
    else
      tmem_dealloc(tmem_base, TMEM_COLS);
  }
}

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// Looked up once (a function-local static is initialised exactly once, even
// when several host threads call in together); nullptr if unavailable.
EncodeTiledFn get_encode_fn() {
  static const EncodeTiledFn fn = []() -> EncodeTiledFn {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      return reinterpret_cast<EncodeTiledFn>(p);
    return nullptr;
  }();
  return fn;
}

}  // namespace

// 2-D bf16 tensor map over a row-major [rows][cols] matrix with row stride
// `ld` elements; box = 64 columns x box_rows rows, 128-byte swizzle.
bool make_tma_2d_bf16(CUtensorMap* m, const void* base, int64_t rows, int64_t cols, int64_t ld, int box_rows) {
  EncodeTiledFn enc = get_encode_fn();
  if (!enc) return false;
  cuuint64_t gdim[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  cuuint64_t gstride[1] = {(cuuint64_t)(ld * 2)};
  cuuint32_t box[2] = {(cuuint32_t)BK, (cuuint32_t)box_rows};
  cuuint32_t estride[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), gdim, gstride, box, estride,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

namespace {

// 2-D bf16 map of the SwiGLU-derivative epilogue's G|U / dG|dU matrices
// ([rows][cols], row stride ld elements): box 32 columns x 32 rows, 64-byte
// swizzle.
bool make_tma_epi(CUtensorMap* m, const void* base, int64_t rows, int64_t cols, int64_t ld) {
  EncodeTiledFn enc = get_encode_fn();
  if (!enc) return false;
  cuuint64_t gdim[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  cuuint64_t gstride[1] = {(cuuint64_t)(ld * 2)};
  cuuint32_t box[2] = {32, 32};
  cuuint32_t estride[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), gdim, gstride, box, estride,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int EPI, bool AMN, bool BMN>
cudaError_t launch_epi(const CUtensorMap& ta, const CUtensorMap& tb, const CUtensorMap& tg, const CUtensorMap& tdg,
                       const CUtensorMap& te2, const GemmShape& s, const EpiParams& ep, cudaStream_t stream) {
  static std::atomic<unsigned long long> configured{0};  // devices set up for this instantiation
  if (needs_setup(configured)) {
    cudaError_t e = cudaFuncSetAttribute(gemm_bf16_tc_kernel<EPI, AMN, BMN, 1>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem_bytes<EPI, 1>());
    if (e != cudaSuccess) return e;
    mark_setup_done(configured);
  }
  // one CTA per tile: the CTAs that start cancel the launch of the others and do their tiles
  gemm_bf16_tc_kernel<EPI, AMN, BMN, 1><<<s.num_tiles, THREADS, smem_bytes<EPI, 1>(), stream>>>(ta, tb, tg, tdg, te2,
                                                                                            s, ep);
  return cudaGetLastError();
}

// CTA-pair kernels: launched as clusters of two, one cluster per tile; the
// clusters that start cancel the launch of the others and do their tiles.
template <int EPI>
cudaLaunchConfig_t pair_config(cudaLaunchAttribute* attr, int pairs, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * pairs, 1, 1);
  cfg.blockDim = dim3(THREADS, 1, 1);
  cfg.dynamicSmemBytes = smem_bytes<EPI, 2>();
  cfg.stream = stream;
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cfg;
}

// Clusters of two the pair kernel can keep resident on the current device
// (queried once per device), 0 if none.
template <int EPI>
int pair_slots() {
  static std::atomic<int> slots[64];
  static std::atomic<unsigned long long> configured{0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  if (needs_setup(configured)) {
    int n = 0;
    cudaError_t e = cudaFuncSetAttribute(gemm_bf16_tc_kernel<EPI, false, false, 2>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem_bytes<EPI, 2>());
    if (e == cudaSuccess) {
      cudaLaunchAttribute attr[1];
      const cudaLaunchConfig_t cfg = pair_config<EPI>(attr, num_sms() / 2, nullptr);
      e = cudaOccupancyMaxActiveClusters(&n, gemm_bf16_tc_kernel<EPI, false, false, 2>, &cfg);
    }
    if (e != cudaSuccess) {
      n = 0;
      (void)cudaGetLastError();  // this query's own error: the one-CTA kernel stays in use
    }
    slots[dev].store(n < 0 ? 0 : n);
    mark_setup_done(configured);
  }
  return slots[dev].load();
}

template <int EPI, bool AMN, bool BMN>
cudaError_t launch_pair(const CUtensorMap& ta, const CUtensorMap& tb, const CUtensorMap& tg, const CUtensorMap& tdg,
                        const CUtensorMap& te2, const GemmShape& s, const EpiParams& ep, cudaStream_t stream) {
  static std::atomic<unsigned long long> configured{0};  // devices set up for this instantiation
  if (needs_setup(configured)) {
    cudaError_t e = cudaFuncSetAttribute(gemm_bf16_tc_kernel<EPI, AMN, BMN, 2>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem_bytes<EPI, 2>());
    if (e != cudaSuccess) return e;
    mark_setup_done(configured);
  }
  cudaLaunchAttribute attr[1];
  const cudaLaunchConfig_t cfg = pair_config<EPI>(attr, s.num_tiles, stream);
  return cudaLaunchKernelEx(&cfg, gemm_bf16_tc_kernel<EPI, AMN, BMN, 2>, ta, tb, tg, tdg, te2, s, ep);
}

// Pair slots for the K-major instantiation of `epi` (0: use one-CTA tiles).
int pair_slots_for(EpiKind epi) {
  switch (epi) {
    case EPI_STORE: return pair_slots<EPI_STORE>();
    case EPI_RESID: return pair_slots<EPI_RESID>();
    case EPI_QKV: return pair_slots<EPI_QKV>();
    case EPI_SWIGLU: return pair_slots<EPI_SWIGLU>();
    case EPI_DSWIGLU: return pair_slots<EPI_DSWIGLU>();
    default: return 0;
  }
}

}  // namespace

tsp_status gemm_bf16_tc(const void* A, int64_t lda, const void* B, int64_t ldb, int M, int N, int K, EpiKind epi,
                        const EpiParams& ep, cudaStream_t stream, bool a_mn, bool b_mn) {
  if (M <= 0 || N <= 0 || K <= 0) return TSP_OK;
  if (N % BN || K % BK || lda % 8 || ldb % 8) return TSP_ERR_UNSUPPORTED;
  if (a_mn && M % 64) return TSP_ERR_UNSUPPORTED;
  if ((reinterpret_cast<uintptr_t>(A) | reinterpret_cast<uintptr_t>(B)) & 15) return TSP_ERR_INVALID_ARG;
  // CTA pairs (256 x 256 tiles) when A has more than one 128-row block and
  // the device can keep pairs resident.  Measured
  // at 2 x 16K tokens, h = 4096, under ncu: QKV 1.70 -> 1.69 ms, output
  // projection 0.588 -> 0.585, gate/up 4.12 -> 3.91, down 2.18 -> 2.01;
  // forward step (same box, interleaved) 12.17-12.19 -> 11.88-11.92 ms.
  const bool pair_shape = M > BM;
  const int slots = (kGemmPairs && pair_shape) ? pair_slots_for(epi) : 0;
  const int CG = slots > 0 ? 2 : 1;
  CUtensorMap ta, tb;
  const bool ok_a = a_mn ? make_tma_2d_bf16(&ta, A, K, M, lda, 64) : make_tma_2d_bf16(&ta, A, M, K, lda, BM);
  const bool ok_b = b_mn ? make_tma_2d_bf16(&tb, B, K, N, ldb, 64) : make_tma_2d_bf16(&tb, B, N, K, ldb, BN / CG);
  if (!ok_a || !ok_b) return TSP_ERR_CUDA;
  // Epilogue tensor maps: G|U in and dG|dU out of the SwiGLU-derivative
  // epilogue; the G|U copy and SiLU(G)*U out of the SwiGLU epilogue.
  CUtensorMap tg{}, tdg{}, te2{};
  if (epi == EPI_QKV && ep.C % 32 == 0) {
    // Q [M][h] (zigzag rows), K [B*Hk*S][dh], V likewise or V^T [B*Hk*dh][S]
    const int64_t kv_rows = (int64_t)ep.B * ep.Hk * ep.S;
    if (!ep.q || !ep.k || !ep.v ||
        ((reinterpret_cast<uintptr_t>(ep.q) | reinterpret_cast<uintptr_t>(ep.k) | reinterpret_cast<uintptr_t>(ep.v)) &
         15) ||
        ep.dh % 32 || ep.h % 32 || ep.S % 32 || kv_rows * (ep.v_transposed ? ep.dh : 1) > INT32_MAX)
      return TSP_ERR_INVALID_ARG;
    const bool ok = make_tma_epi(&tg, ep.q, M, ep.h, ep.h) && make_tma_epi(&tdg, ep.k, kv_rows, ep.dh, ep.dh) &&
                    (ep.v_transposed ? make_tma_epi(&te2, ep.v, (int64_t)ep.B * ep.Hk * ep.dh, ep.S, ep.S)
                                     : make_tma_epi(&te2, ep.v, kv_rows, ep.dh, ep.dh));
    if (!ok) return TSP_ERR_CUDA;
  }
  if (epi == EPI_SWIGLU) {
    if (!ep.out || (reinterpret_cast<uintptr_t>(ep.out) & 15) || ep.ldo % 8 || ep.ldo < N / 2 ||
        (ep.aux && ((reinterpret_cast<uintptr_t>(ep.aux) & 15) || ep.ldx % 8 || ep.ldx < (int64_t)N)))
      return TSP_ERR_INVALID_ARG;
    if ((ep.aux && !make_tma_epi(&tg, ep.aux, M, N, ep.ldx)) || !make_tma_epi(&tdg, ep.out, M, N / 2, ep.ldo))
      return TSP_ERR_CUDA;
  }
  if (epi == EPI_RESID) {
    if (!ep.resid || !ep.out || ((reinterpret_cast<uintptr_t>(ep.resid) | reinterpret_cast<uintptr_t>(ep.out)) & 15) ||
        ep.ldr % 8 || ep.ldo % 8 || ep.ldr < (int64_t)N || ep.ldo < (int64_t)N)
      return TSP_ERR_INVALID_ARG;
    if (!make_tma_epi(&tg, ep.resid, M, N, ep.ldr) || !make_tma_epi(&tdg, ep.out, M, N, ep.ldo)) return TSP_ERR_CUDA;
  }
  if (epi == EPI_DSWIGLU) {
    if (!ep.resid || !ep.out || ((reinterpret_cast<uintptr_t>(ep.resid) | reinterpret_cast<uintptr_t>(ep.out)) & 15) ||
        ep.ldr % 8 || ep.ldo % 8 || ep.ldr < 2 * (int64_t)N || ep.ldo < 2 * (int64_t)N)
      return TSP_ERR_INVALID_ARG;
    if (!make_tma_epi(&tg, ep.resid, M, 2 * (int64_t)N, ep.ldr) || !make_tma_epi(&tdg, ep.out, M, 2 * (int64_t)N, ep.ldo))
      return TSP_ERR_CUDA;
  }
  GemmShape s;
  s.M = M;
  s.N = N;
  s.K = K;
  s.num_m = (M + BM * CG - 1) / (BM * CG);
  s.num_n = N / BN;
  s.num_tiles = s.num_m * s.num_n;
  s.kblocks = K / BK;
  {
    const size_t band_rows = kBandBytes / ((size_t)K * 2);
    int gm = (int)(band_rows / (BM * CG));
    s.group_m = gm < 1 ? 1 : (gm > s.num_m ? s.num_m : gm);
    s.group_n = 0;
    if (N < M) {
      // B is the smaller operand: bands of 16 of B's n-tiles (at most 64 MB)
      // stay in L2 while A streams past them.  Measured at 2 x 16K tokens:
      // gate/up, QKV and output projection 2-4 % faster than with A bands,
      // and the down projection (K = 14336, 8 n-tiles per band) reads 3.9 GB
      // from DRAM instead of 5.2 (its 117 MB weight was re-read every wave).
      // Larger B bands (64, 96 MB of gate/up's B) and L2 eviction hints on
      // the streaming operand were slower.
      const size_t band_cols = kBBandBytes / ((size_t)K * 2);
      int gn = (int)(band_cols / BN);
      gn = gn > kBBandTiles ? kBBandTiles : gn;
      s.group_n = gn < 1 ? 1 : (gn > s.num_n ? s.num_n : gn);
    }
  }
  cudaError_t e;
  const int mode = (a_mn ? 2 : 0) | (b_mn ? 1 : 0);
  if (CG == 2) {
    switch (epi * 4 + mode) {
      case EPI_STORE * 4 + 0: e = launch_pair<EPI_STORE, false, false>(ta, tb, tg, tdg, te2, s, ep, stream); break;
      case EPI_STORE * 4 + 1: e = launch_pair<EPI_STORE, false, true>(ta, tb, tg, tdg, te2, s, ep, stream); break;
      case EPI_STORE * 4 + 3: e = launch_pair<EPI_STORE, true, true>(ta, tb, tg, tdg, te2, s, ep, stream); break;
      case EPI_RESID * 4 + 0: e = launch_pair<EPI_RESID, false, false>(ta, tb, tg, tdg, te2, s, ep, stream); break;
      case EPI_RESID * 4 + 1: e = launch_pair<EPI_RESID, false, true>(ta, tb, tg, tdg, te2, s, ep, stream); break;
      case EPI_QKV * 4 + 0: e = launch_pair<EPI_QKV, false, false>(ta, tb, tg, tdg, te2, s, ep, stream); break;
      case EPI_SWIGLU * 4 + 0: e = launch_pair<EPI_SWIGLU, false, false>(ta, tb, tg, tdg, te2, s, ep, stream); break;
      case EPI_DSWIGLU * 4 + 0:
        e = launch_pair<EPI_DSWIGLU, false, false>(ta, tb, tg, tdg, te2, s, ep, stream);
        break;
      case EPI_DSWIGLU * 4 + 1: e = launch_pair<EPI_DSWIGLU, false, true>(ta, tb, tg, tdg, te2, s, ep, stream); break;
      default: return TSP_ERR_UNSUPPORTED;
    }
    return e == cudaSuccess ? TSP_OK : TSP_ERR_CUDA;
  }
  switch (epi * 4 + mode) {
    case EPI_STORE * 4 + 0: e = launch_epi<EPI_STORE, false, false>(ta, tb, tg, tdg, te2, s, ep, stream); break;
    case EPI_STORE * 4 + 1: e = launch_epi<EPI_STORE, false, true>(ta, tb, tg, tdg, te2, s, ep, stream); break;
    case EPI_STORE * 4 + 3: e = launch_epi<EPI_STORE, true, true>(ta, tb, tg, tdg, te2, s, ep, stream); break;
    case EPI_RESID * 4 + 0: e = launch_epi<EPI_RESID, false, false>(ta, tb, tg, tdg, te2, s, ep, stream); break;
    case EPI_RESID * 4 + 1: e = launch_epi<EPI_RESID, false, true>(ta, tb, tg, tdg, te2, s, ep, stream); break;
    case EPI_QKV * 4 + 0: e = launch_epi<EPI_QKV, false, false>(ta, tb, tg, tdg, te2, s, ep, stream); break;
    case EPI_SWIGLU * 4 + 0: e = launch_epi<EPI_SWIGLU, false, false>(ta, tb, tg, tdg, te2, s, ep, stream); break;
    case EPI_DSWIGLU * 4 + 0: e = launch_epi<EPI_DSWIGLU, false, false>(ta, tb, tg, tdg, te2, s, ep, stream); break;
    case EPI_DSWIGLU * 4 + 1: e = launch_epi<EPI_DSWIGLU, false, true>(ta, tb, tg, tdg, te2, s, ep, stream); break;
    default: return TSP_ERR_UNSUPPORTED;
  }
  return e == cudaSuccess ? TSP_OK : TSP_ERR_CUDA;
}

}  // namespace tsp
