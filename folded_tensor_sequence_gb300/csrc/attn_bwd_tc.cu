// Causal flash-attention backward on the 5th-generation tensor cores
// (tcgen05 + TMEM), head_dim 128, bf16 in, fp32 accumulation.
//
// Exact gradient of the forward (the TSP posts do not describe a backward):
//   P = exp(S/sqrt(dh) - lse),  dP = dO V^T,  dS = P * (dP - rowsum(dO * O)),
//   dV = P^T dO,  dK = dS^T Q / sqrt(dh),  dQ = dS K / sqrt(dh).
// Two kernels, no atomics; every tensor-core operand arrives by TMA:
//   dK/dV: one CTA per mirror pair of 128-key tiles (j, nk-1-j: together they
//     see a constant number of query blocks) of one K/V head.  K and V of the
//     tile stay in shared memory; 128-query blocks of Q and dO (of every query
//     head reading the K/V head) stream through a 2-stage ring, read K-major by
//     S^T = K Q^T, dP^T = V dO^T and MN-major by dV += P^T dO, dK += dS^T Q.
//     TMEM: S^T, dP^T (single-buffered), dV and dK accumulators.
//   dQ: one CTA per mirror pair of 128-query tiles (the forward's zigzag
//     pairing: both tiles on the same rank).  Q and dO stay in shared memory;
//     key blocks of 64 stream K and V (4-stage ring) for S = Q K^T,
//     dP = dO V^T, with the K tile read again as the MN-major operand of
//     dQ += dS K.  TMEM: S and dP double-buffered, dQ accumulator.
// In both, warps 0-7 turn scores into P and dS (a TMEM lane = a row, split
// over two threads) and write them back into tensor memory as packed bf16,
// where the accumulating MMAs read them as their A operand; lse and dsum of
// each query block come in with the stage by bulk copy (dK/dV) or are read
// once per tile (dQ).  Warp 8 issues TMA, warp 9 issues tcgen05.mma from one
// thread, warp 10 relays landed stages to warp 9.
#include <type_traits>

#include "common.cuh"
#include "internal.h"

namespace tsp {

namespace {

constexpr int HD = 128;
constexpr int THREADS = 352;  // warps 0-7 elementwise (two per TMEM lane quadrant), 8 TMA, 9 MMA, 10 relay
// Named barriers into the MMA warp (which never waits on an mbarrier inside a
// tile): the relay warp announces each landed stage on kBarStage + (n % 4)
// (64 threads: relay + MMA), the elementwise warps hand back dS of block i
// on kBarDS + (i % 2) in the dQ kernel, P and dS on kBarP2 / kBarDS2 in the
// dK/dV kernel (256 + 32 threads).  A warp arrives without blocking
// only while the data it hands over keeps it in step with the MMA warp; the
// relay, and any warp that has given up waiting, uses the blocking form, so
// no warp can run ahead and complete a barrier phase in the MMA warp's place.
constexpr int kBarStage = 1, kBarDS = 5;
constexpr int kStageThreads = 64, kDSThreads = 256 + 32;
constexpr uint32_t SUB64 = 64 * 64 * 2;     // [64 rows][64 cols] bf16, 8 KB
constexpr uint32_t SUB128 = 128 * 64 * 2;   // [128 rows][64 cols] bf16, 16 KB
constexpr float kLog2e = 1.4426950408889634f;
constexpr unsigned CODE_DKDV = KID_ATTN_BWD << 8;
constexpr unsigned CODE_DQ = (KID_ATTN_BWD << 8) | 0x80;
constexpr unsigned CODE_FUSED = (KID_ATTN_BWD << 8) | 0x40;

struct BwdTcParams {
  int B, H, D;
  int Hk;  // K/V heads; query head `head` reads K/V head head / (H / Hk)
  int64_t S, C;
  int h;
  const float* lse;   // [B][H][S], natural log
  const float* dsum;  // [B][H][S]
  float* dq_acc;      // [B][H][S][dh] fp32, unscaled dS K sums
  __nv_bfloat16* dk;  // [B][H][S][dh]
  __nv_bfloat16* dv;
  unsigned int* err;
};

__device__ __forceinline__ float ex2f(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ int64_t zz_row(int64_t pos, int64_t C, int D, int B, int b) {
  const int64_t c = pos / C, off = pos - c * C;
  const int64_t r = c < D ? c : 2 * D - 1 - c;
  return (r * B + b) * 2 * C + (c < D ? off : C + off);
}

// ===========================================================================
// dK, dV with 128-query blocks
// ===========================================================================
// Every MMA is 128 x 128 x 16 (full rate) and a block needs 32 of them for
// 128 queries, against 48 for two 64-query blocks; the hand-offs per query
// halve.  TMEM holds S^T, dP^T (128 columns each, single-buffered), dV and
// dK.  The elementwise warps work in two phases per block -- P^T (feeds
// dV += P^T dO) and then dS^T (feeds dK += dS^T Q) -- and the MMA order
//   S(n), dP(n), [P(n)] dV(n), S(n+1), [dS(n)] dK(n), dP(n+1), ...
// keeps the tensor core on the next block's scores while they work.
constexpr int QB2 = 128;
constexpr int QSTG2 = 2;
constexpr uint32_t STG2_DATA = 4 * SUB128;            // Q (2 sub-tiles [128][64]), dO (2)
constexpr uint32_t STG2_BYTES = STG2_DATA + 1024;     // + lse, dsum of the block (512 B each)
constexpr size_t DKDV2_SMEM = 1024 + 4 * (size_t)SUB128 + QSTG2 * (size_t)STG2_BYTES + 256;
constexpr int kBarP2 = 5, kBarDS2 = 6;                 // P and dS hand-offs (256 + 32 threads)

__global__ void __launch_bounds__(THREADS, 1)
    attn_dkdv128_tc_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                           const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmdO,
                           const BwdTcParams p, int nk) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* Ks = smem;                    // 2 x SUB128
  uint8_t* Vs = smem + 2 * SUB128;       // 2 x SUB128
  uint8_t* stg = smem + 4 * SUB128;      // [QSTG2] stages
  uint64_t* bars = reinterpret_cast<uint64_t*>(stg + QSTG2 * STG2_BYTES);
  uint64_t* kv_full = bars + 0;
  uint64_t* kv_free = bars + 1;
  uint64_t* q_full = bars + 2;   // [QSTG2]
  uint64_t* q_free = bars + 4;   // [QSTG2]
  uint64_t* s_full = bars + 6;   // S^T of the current block is in TMEM
  uint64_t* dp_full = bars + 7;  // dP^T of the current block is in TMEM
  uint64_t* o_done = bars + 8;
  uint64_t* drain = bars + 9;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 10);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  // blockIdx.y is a K/V head; the `grp` query heads that read it stream through
  // one after another (their dK, dV contributions add up in tensor memory)
  const int kvh = blockIdx.y, b = blockIdx.z;
  const int grp = p.H / p.Hk;
  const int64_t bkv = (int64_t)b * p.Hk + kvh;
  auto tile_of = [&](int t) { return t == 0 ? (int)blockIdx.x : nk - 1 - (int)blockIdx.x; };
  const int ntile = (nk - 1 - (int)blockIdx.x == (int)blockIdx.x) ? 1 : 2;

  if (threadIdx.x == 0) {
    mbar_init(kv_full, 1);
    mbar_init(kv_free, 1);
    for (int s = 0; s < QSTG2; ++s) {
      mbar_init(&q_full[s], 1);
      mbar_init(&q_free[s], 1);
    }
    mbar_init(s_full, 1);
    mbar_init(dp_full, 1);
    mbar_init(o_done, 1);
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbarrier_init();
  }
  if (warp == 8 && lane == 0) {
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
    tma_prefetch_desc(&tmQ);
    tma_prefetch_desc(&tmdO);
  }
  if (warp == 9) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  // TMEM columns: S^T at 0, dP^T at 128, dV at 256, dK at 384.  P^T (bf16
  // pairs) goes over the first 32 columns of each 64-column half of S^T (the
  // half whose scores the writing thread read), dS^T likewise over dP^T.

  if (warp == 8) {
    // ---------------- TMA producer ----------------
    if (lane == 0) {
      uint32_t qi = 0;
      int kv_armed = 0;
      bool ok = true;
      for (int t = 0; t < ntile && ok; ++t) {
        const int64_t k0 = (int64_t)tile_of(t) * 128;
        if (!mbar_wait(kv_free, (t & 1) ^ 1, abort_flag, p.err, CODE_DKDV | 1)) break;
        mbar_arrive_expect_tx(kv_full, 4 * SUB128);
        ++kv_armed;
        for (int c = 0; c < 2; ++c) {
          tma_load_2d(Ks + c * SUB128, &tmK, c * 64, (int)(bkv * p.S + k0), kv_full);
          tma_load_2d(Vs + c * SUB128, &tmV, c * 64, (int)(bkv * p.S + k0), kv_full);
        }
        const int nq = (int)((p.S - k0) / QB2);
        for (int u = 0; u < grp * nq; ++u, ++qi) {
          const int i = u % nq;
          const int head = kvh * grp + u / nq;
          const int64_t bh = (int64_t)b * p.H + head;
          const int s = qi % QSTG2;
          if (!mbar_wait(&q_free[s], ((qi / QSTG2) & 1) ^ 1, abort_flag, p.err, CODE_DKDV | 2)) {
            ok = false;
            break;
          }
          const int64_t q0 = k0 + (int64_t)i * QB2;
          const int64_t zr = zz_row(q0, p.C, p.D, p.B, b);  // a 128-query block never crosses a chunk
          uint8_t* st = stg + s * STG2_BYTES;
          mbar_arrive_expect_tx(&q_full[s], STG2_DATA + 2 * QB2 * 4);
          for (int c = 0; c < 2; ++c) {
            tma_load_2d(st + c * SUB128, &tmQ, head * HD + c * 64, (int)zr, &q_full[s]);
            tma_load_2d(st + 2 * SUB128 + c * SUB128, &tmdO, head * HD + c * 64, (int)zr, &q_full[s]);
          }
          bulk_load(st + STG2_DATA, p.lse + bh * p.S + q0, QB2 * 4, &q_full[s]);
          bulk_load(st + STG2_DATA + QB2 * 4, p.dsum + bh * p.S + q0, QB2 * 4, &q_full[s]);
        }
      }
      volatile int dummy = 0;
      const uint32_t first = qi > QSTG2 ? qi - QSTG2 : 0;
      for (uint32_t n = first; n < qi; ++n) mbar_wait(&q_full[n % QSTG2], (n / QSTG2) & 1, &dummy, p.err, CODE_DKDV | 3);
      if (kv_armed) mbar_wait(kv_full, (kv_armed - 1) & 1, &dummy, p.err, CODE_DKDV | 3);
    }
  } else if (warp == 9) {
    // ---------------- MMA issuer (whole warp walks the schedule and issues; one elected lane) ----------------
    constexpr uint32_t id_s = idesc_bf16_f32(128, QB2);              // M = keys, N = queries
    constexpr uint32_t id_o = idesc_bf16_f32(128, HD, false, true);  // M = keys, N = head dim (B MN-major)
    uint32_t qi = 0;
    bool ok = true;  // warp-uniform
    auto stage = [&](uint32_t n) { return stg + (n % QSTG2) * STG2_BYTES; };
    auto scores = [&](uint32_t n) {  // S^T = K Q^T
      uint8_t* st = stage(n);
#pragma unroll
      for (int k = 0; k < HD / 16; ++k) {
        const uint64_t ak = sdesc_kmajor_sw128(smem_u32(Ks + (k / 4) * SUB128)) + 2 * (k % 4);
        const uint64_t bq = sdesc_kmajor_sw128(smem_u32(st + (k / 4) * SUB128)) + 2 * (k % 4);
        umma_bf16_warp(tmem_base, ak, bq, id_s, k > 0);
      }
      umma_commit_warp(s_full);
    };
    auto dpscores = [&](uint32_t n) {  // dP^T = V dO^T
      uint8_t* st = stage(n);
#pragma unroll
      for (int k = 0; k < HD / 16; ++k) {
        const uint64_t av = sdesc_kmajor_sw128(smem_u32(Vs + (k / 4) * SUB128)) + 2 * (k % 4);
        const uint64_t bo = sdesc_kmajor_sw128(smem_u32(st + 2 * SUB128 + (k / 4) * SUB128)) + 2 * (k % 4);
        umma_bf16_warp(tmem_base + 128, av, bo, id_s, k > 0);
      }
      umma_commit_warp(dp_full);
    };
    // dV += P^T dO and dK += dS^T Q: the stage's dO / Q tiles as MN-major B
    // operands (rows = queries = K dimension; 64-column chunks SUB128 apart)
    auto accum_v = [&](uint32_t n, bool acc) {
      uint8_t* st = stage(n);
#pragma unroll
      for (int k = 0; k < QB2 / 16; ++k) {
        const uint64_t bo = sdesc_mn_sw128(smem_u32(st + 2 * SUB128) + 2048 * k, SUB128);
        umma_bf16_ts_warp(tmem_base + 256, tmem_base + 64 * (k / 4) + 8 * (k % 4), bo, id_o, (acc || k > 0) ? 1u : 0u);
      }
    };
    auto accum_k = [&](uint32_t n, bool acc) {
      uint8_t* st = stage(n);
#pragma unroll
      for (int k = 0; k < QB2 / 16; ++k) {
        const uint64_t bq = sdesc_mn_sw128(smem_u32(st) + 2048 * k, SUB128);
        umma_bf16_ts_warp(tmem_base + 384, tmem_base + 128 + 64 * (k / 4) + 8 * (k % 4), bq, id_o,
                     (acc || k > 0) ? 1u : 0u);
      }
      umma_commit_warp(&q_free[n % QSTG2]);
    };
    auto sync_on = [&](int id, int count) {
      __syncwarp();
      named_bar_sync(id, count);
      tc_fence_after();
    };
    for (int t = 0; t < ntile; ++t) {
      const int64_t k0 = (int64_t)tile_of(t) * 128;
      const int nq = grp * (int)((p.S - k0) / QB2);  // query blocks of all the group's heads
      if (ok) {
        bool w = true;
        if (lane == 0) w = mbar_wait(kv_full, t & 1, abort_flag, p.err, CODE_DKDV | 4);
        ok = __shfl_sync(0xffffffffu, w ? 1 : 0, 0) != 0;
      }
      sync_on(kBarStage + (qi & 3), kStageThreads);
      if (ok) {
        scores(qi);
        dpscores(qi);
      }
      for (int i = 0; i < nq; ++i) {
        const uint32_t n = qi + i;
        sync_on(kBarP2, kDSThreads);  // P^T(n) in TMEM
        if (ok) accum_v(n, i > 0);
        if (i + 1 < nq) {
          sync_on(kBarStage + ((n + 1) & 3), kStageThreads);
          if (ok) scores(n + 1);
        }
        sync_on(kBarDS2, kDSThreads);  // dS^T(n) in TMEM
        if (ok) {
          accum_k(n, i > 0);
          if (i + 1 < nq) dpscores(n + 1);
        }
      }
      if (ok) {
        umma_commit_warp(o_done);
        umma_commit_warp(kv_free);
      }
      qi += nq;
    }
    umma_commit_warp(drain);
    if (lane == 0) {
      volatile int dummy = 0;
      mbar_wait(drain, 0, &dummy, p.err, CODE_DKDV | 7);
    }
    __syncwarp();
  } else if (warp == 10) {
    // ---------------- relay: announces each landed stage to the MMA warp ----------------
    uint32_t n = 0;
    for (int t = 0; t < ntile; ++t) {
      const int nq = grp * (int)((p.S - (int64_t)tile_of(t) * 128) / QB2);
      for (int i = 0; i < nq; ++i, ++n) {
        if (lane == 0) mbar_wait(&q_full[n % QSTG2], (n / QSTG2) & 1, abort_flag, p.err, CODE_DKDV | 9);
        __syncwarp();
        named_bar_sync(kBarStage + (n & 3), kStageThreads);
      }
    }
  } else {
    // ------- elementwise warps 0-7: one key row, 64 of the 128 query columns per thread -------
    const int quad = warp & 3, half = warp >> 2;
    const int row = quad * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(quad * 32) << 16;
    const float sl2 = kLog2e * rsqrtf((float)HD);
    const float scale = rsqrtf((float)HD);
    uint32_t cnt = 0;  // blocks processed (phase of s_full / dp_full; stage = cnt % QSTG2)
    bool alive = true;  // warp-uniform; once false the warp only keeps the hand-off count
    const uint32_t cS = tmem_base + lane_off + 64 * half;
    const uint32_t cdP = tmem_base + lane_off + 128 + 64 * half;
    for (int t = 0; t < ntile; ++t) {
      const int64_t k0 = (int64_t)tile_of(t) * 128;
      const int nqh = (int)((p.S - k0) / QB2);
      const int64_t key = k0 + row;
      for (int u = 0; u < grp * nqh; ++u, ++cnt) {
        const int i = u % nqh;  // query block within the head
        // ---- P phase ----
        bool got = alive && mbar_wait(s_full, cnt & 1, abort_flag, p.err, CODE_DKDV | 8);
        alive = __all_sync(0xffffffffu, got);
        if (!alive) {
          named_bar_sync(kBarP2, kDSThreads);
          named_bar_sync(kBarDS2, kDSThreads);
          continue;
        }
        tc_fence_after();
        uint32_t sa[32], sb[32];
        tmem_ld32_issue(cS, sa);
        tmem_ld32_issue(cS + 32, sb);
        const float4* lse4 = reinterpret_cast<const float4*>(stg + (cnt % QSTG2) * STG2_BYTES + STG2_DATA) + 16 * half;
        const float4* ds4 = lse4 + QB2 / 4;
        const int64_t q0 = k0 + (int64_t)i * QB2 + 64 * half;  // query of this thread's first column
        const bool diag = i == 0;
        float pv[64];
        tmem_wait_ld32(sa);
        tmem_wait_ld32(sb);
#pragma unroll
        for (int c4 = 0; c4 < 16; ++c4) {
          const float4 l4 = lse4[c4];
          const float lv[4] = {l4.x * kLog2e, l4.y * kLog2e, l4.z * kLog2e, l4.w * kLog2e};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int c = c4 * 4 + e;
            const float sc = __uint_as_float(c < 32 ? sa[c] : sb[c - 32]);
            float pe = ex2f(fmaf(sc, sl2, -lv[e]));
            if (diag && q0 + c < key) pe = 0.f;
            pv[c] = pe;
          }
        }
        uint32_t pk[32];
#pragma unroll
        for (int c = 0; c < 32; ++c) pk[c] = pack_bf16x2(pv[2 * c], pv[2 * c + 1]);
        tmem_st32_nowait(cS, pk);  // P^T over the start of this thread's S^T columns
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        named_bar_arrive(kBarP2, kDSThreads);
        // ---- dS phase ----
        got = mbar_wait(dp_full, cnt & 1, abort_flag, p.err, CODE_DKDV | 11);
        alive = __all_sync(0xffffffffu, got);
        if (!alive) {
          named_bar_sync(kBarDS2, kDSThreads);
          continue;
        }
        tc_fence_after();
        tmem_ld32_issue(cdP, sa);
        tmem_ld32_issue(cdP + 32, sb);
        tmem_wait_ld32(sa);
        tmem_wait_ld32(sb);
#pragma unroll
        for (int c4 = 0; c4 < 16; ++c4) {
          const float4 d4 = ds4[c4];
          const float dv[4] = {d4.x, d4.y, d4.z, d4.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int c = c4 * 4 + e;
            const float dp = __uint_as_float(c < 32 ? sa[c] : sb[c - 32]);
            pv[c] = pv[c] * (dp - dv[e]);
          }
        }
#pragma unroll
        for (int c = 0; c < 32; ++c) pk[c] = pack_bf16x2(pv[2 * c], pv[2 * c + 1]);
        tmem_st32_nowait(cdP, pk);  // dS^T over the start of this thread's dP^T columns
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        named_bar_arrive(kBarDS2, kDSThreads);
      }
      if (!alive) continue;
      const bool got = mbar_wait(o_done, t & 1, abort_flag, p.err, CODE_DKDV | 10);
      alive = __all_sync(0xffffffffu, got);
      if (!alive) continue;
      tc_fence_after();
      uint4* dvrow = reinterpret_cast<uint4*>(p.dv + (bkv * p.S + key) * HD) + 8 * half;
      uint4* dkrow = reinterpret_cast<uint4*>(p.dk + (bkv * p.S + key) * HD) + 8 * half;
#pragma unroll 1
      for (int c32 = 0; c32 < 2; ++c32) {
        float a[32], d[32];
        tmem_ld32(tmem_base + lane_off + 256 + 64 * half + 32 * c32, a);
        tmem_ld32(tmem_base + lane_off + 384 + 64 * half + 32 * c32, d);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          dvrow[c32 * 4 + q] = make_uint4(pack_bf16x2(a[q * 8 + 0], a[q * 8 + 1]), pack_bf16x2(a[q * 8 + 2], a[q * 8 + 3]),
                                          pack_bf16x2(a[q * 8 + 4], a[q * 8 + 5]), pack_bf16x2(a[q * 8 + 6], a[q * 8 + 7]));
          dkrow[c32 * 4 + q] = make_uint4(
              pack_bf16x2(d[q * 8 + 0] * scale, d[q * 8 + 1] * scale), pack_bf16x2(d[q * 8 + 2] * scale, d[q * 8 + 3] * scale),
              pack_bf16x2(d[q * 8 + 4] * scale, d[q * 8 + 5] * scale), pack_bf16x2(d[q * 8 + 6] * scale, d[q * 8 + 7] * scale));
        }
      }
      tc_fence_before();
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 9) {
    tc_fence_after();
    tmem_dealloc(tmem_base, 512);
  }
}

// ===========================================================================
// Fused dK, dV and dQ with 64-query blocks
// ===========================================================================
// Five MMA groups per block instead of the seven of the two kernels above
// (scores and dP are not recomputed for dQ) and one exponential per score:
//   S^T = K Q^T, dP^T = V dO^T            (M = 128 keys, N = 64 queries)
//   dV += P^T dO, dK += dS^T Q            (P^T, dS^T from TMEM; N = head dim)
//   dQ^T = K^T dS^T                       (M = head dim, N = 64 queries; K tile
//                                          and dS^T both read MN-major from
//                                          shared memory)
// The dQ^T of a block is a partial sum over this CTA's 128 keys: the
// elementwise warps read it out of TMEM and add it into an fp32 accumulator
// [B][H][S][dh] with L2 reductions (zeroed beforehand; scaled by 1/sqrt(dh)
// when it is assembled), so the summation order, and the last bit of dQ,
// varies from run to run.  TMEM: S^T at 0 (P^T over its start), dP^T at 64,
// dQ^T at 128, dS^T at 192, dV at 256, dK at 384.  MMA order per block
//   [P(n)] dV(n), S(n+1), [dS(n)] dP(n+1), dK(n), dQ(n)
// puts the next block's dP right behind the dS hand-off, so the elementwise
// warps compute dS(n+1) while dK(n) and dQ(n) run; before they overwrite
// dS^T (TMEM and shared memory) and read dQ^T(n) out they wait for the
// commit that follows dQ(n), and they hand dS(n+1) over before adding
// dQ^T(n) into memory.  The MMA warp is then limited by its own issue rate.
constexpr int QBF = 64;
constexpr int NSTGF = 4;
constexpr uint32_t STGF_BYTES = 4 * SUB64;   // Q (2 sub-tiles [64][64]), dO (2)
constexpr uint32_t LDF_BYTES = 2 * QBF * 4;  // lse, dsum of the block
constexpr size_t FUSED_SMEM =
    1024 + 4 * (size_t)SUB128 + NSTGF * (size_t)STGF_BYTES + SUB128 + NSTGF * (size_t)LDF_BYTES + 256;
constexpr int kBarPF = 5, kBarDSF = 6;  // P and dS hand-offs (256 + 32 threads)

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void red_add_f32(float* addr, float v) {
  asm volatile("red.global.add.f32 [%0], %1;" ::"l"(addr), "f"(v) : "memory");
}

__global__ void __launch_bounds__(THREADS, 1)
    attn_bwd_fused_tc_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                             const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmdO,
                             const BwdTcParams p, int nk, int paired) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* Ks = smem;                          // 2 x SUB128
  uint8_t* Vs = smem + 2 * SUB128;             // 2 x SUB128
  uint8_t* stg = smem + 4 * SUB128;            // [NSTGF] stages
  uint8_t* dSs = stg + NSTGF * STGF_BYTES;     // dS^T [128 keys][64 queries], 128-byte swizzle
  uint8_t* ldr = dSs + SUB128;                 // [NSTGF] lse, dsum
  uint64_t* bars = reinterpret_cast<uint64_t*>(ldr + NSTGF * LDF_BYTES);
  uint64_t* kv_full = bars + 0;
  uint64_t* kv_free = bars + 1;
  uint64_t* q_full = bars + 2;   // [NSTGF]
  uint64_t* q_free = bars + 6;   // [NSTGF]
  uint64_t* s_full = bars + 10;  // S^T of the current block is in TMEM
  uint64_t* dp_full = bars + 11; // dP^T of the current block is in TMEM
  uint64_t* dq_full = bars + 12; // dQ^T of a block is in TMEM (and every earlier MMA is done)
  uint64_t* drain = bars + 13;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 14);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  // paired: grid (mirror pair, K/V head, batch), two key tiles of equal total
  // work per CTA; otherwise grid (K/V head, batch, key tile), one tile per
  // CTA, heaviest tiles (the earliest keys see the most queries) launched first
  const int kvh = paired ? (int)blockIdx.y : (int)blockIdx.x;
  const int b = paired ? (int)blockIdx.z : (int)blockIdx.y;
  const int grp = p.H / p.Hk;
  const int64_t bkv = (int64_t)b * p.Hk + kvh;
  auto tile_of = [&](int t) {
    return paired ? (t == 0 ? (int)blockIdx.x : nk - 1 - (int)blockIdx.x) : (int)blockIdx.z;
  };
  const int ntile = paired ? ((nk - 1 - (int)blockIdx.x == (int)blockIdx.x) ? 1 : 2) : 1;

  if (threadIdx.x == 0) {
    mbar_init(kv_full, 1);
    mbar_init(kv_free, 1);
    for (int s = 0; s < NSTGF; ++s) {
      mbar_init(&q_full[s], 1);
      mbar_init(&q_free[s], 1);
    }
    mbar_init(s_full, 1);
    mbar_init(dp_full, 1);
    mbar_init(dq_full, 1);
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbarrier_init();
  }
  if (warp == 8 && lane == 0) {
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
    tma_prefetch_desc(&tmQ);
    tma_prefetch_desc(&tmdO);
  }
  if (warp == 9) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 8) {
    // ---------------- TMA producer ----------------
    if (lane == 0) {
      uint32_t qi = 0;
      int kv_armed = 0;
      bool ok = true;
      for (int t = 0; t < ntile && ok; ++t) {
        const int64_t k0 = (int64_t)tile_of(t) * 128;
        if (!mbar_wait(kv_free, (t & 1) ^ 1, abort_flag, p.err, CODE_FUSED | 1)) break;
        mbar_arrive_expect_tx(kv_full, 4 * SUB128);
        ++kv_armed;
        for (int c = 0; c < 2; ++c) {
          tma_load_2d(Ks + c * SUB128, &tmK, c * 64, (int)(bkv * p.S + k0), kv_full);
          tma_load_2d(Vs + c * SUB128, &tmV, c * 64, (int)(bkv * p.S + k0), kv_full);
        }
        const int nq = (int)((p.S - k0) / QBF);
        for (int u = 0; u < grp * nq; ++u, ++qi) {
          const int i = u % nq;
          const int head = kvh * grp + u / nq;
          const int64_t bh = (int64_t)b * p.H + head;
          const int s = qi % NSTGF;
          if (!mbar_wait(&q_free[s], ((qi / NSTGF) & 1) ^ 1, abort_flag, p.err, CODE_FUSED | 2)) {
            ok = false;
            break;
          }
          const int64_t q0 = k0 + (int64_t)i * QBF;
          const int64_t zr = zz_row(q0, p.C, p.D, p.B, b);  // a 64-query block never crosses a chunk
          uint8_t* st = stg + s * STGF_BYTES;
          uint8_t* ld = ldr + s * LDF_BYTES;
          mbar_arrive_expect_tx(&q_full[s], STGF_BYTES + LDF_BYTES);
          for (int c = 0; c < 2; ++c) {
            tma_load_2d(st + c * SUB64, &tmQ, head * HD + c * 64, (int)zr, &q_full[s]);
            tma_load_2d(st + 2 * SUB64 + c * SUB64, &tmdO, head * HD + c * 64, (int)zr, &q_full[s]);
          }
          bulk_load(ld, p.lse + bh * p.S + q0, QBF * 4, &q_full[s]);
          bulk_load(ld + QBF * 4, p.dsum + bh * p.S + q0, QBF * 4, &q_full[s]);
        }
      }
      volatile int dummy = 0;
      const uint32_t first = qi > NSTGF ? qi - NSTGF : 0;
      for (uint32_t n = first; n < qi; ++n)
        mbar_wait(&q_full[n % NSTGF], (n / NSTGF) & 1, &dummy, p.err, CODE_FUSED | 3);
      if (kv_armed) mbar_wait(kv_full, (kv_armed - 1) & 1, &dummy, p.err, CODE_FUSED | 3);
    }
  } else if (warp == 9) {
    // ---------------- MMA issuer (whole warp walks the schedule and issues; one elected lane) ----------------
    constexpr uint32_t id_s = idesc_bf16_f32(128, QBF);                // M = keys, N = queries
    constexpr uint32_t id_o = idesc_bf16_f32(128, HD, false, true);    // M = keys, N = head dim (B MN-major)
    constexpr uint32_t id_q = idesc_bf16_f32(HD, QBF, true, true);     // M = head dim, N = queries (A, B MN-major)
    uint32_t qi = 0;
    bool ok = true;  // warp-uniform
    // Descriptor low words computed once (the issuing stream stays short;
    // the elementwise warps' instructions on this sub-partition delay every
    // MMA issue): K-major tiles for S^T and dP^T, MN-major for dV, dK, dQ^T.
    // A stage adds s * (STGF_BYTES >> 4); K step k of a K-major [rows][128]
    // tile in two 64-column sub-tiles adds (k / 4) * (sub-tile >> 4) + 2 (k % 4),
    // of an MN-major tile 2048 k >> 4 = 128 k.
    const uint32_t k_lo = sdesc_lo(smem_u32(Ks)), v_lo = sdesc_lo(smem_u32(Vs));
    const uint32_t stg_lo = sdesc_lo(smem_u32(stg)), stg_mn = sdesc_mn_lo(smem_u32(stg), SUB64);
    const uint32_t k_mn = sdesc_mn_lo(smem_u32(Ks), SUB128), ds_mn = sdesc_mn_lo(smem_u32(dSs), SUB128);
    const uint32_t s_full_at = smem_u32(s_full), dp_full_at = smem_u32(dp_full), dq_full_at = smem_u32(dq_full);
    const uint32_t q_free_at = smem_u32(q_free);  // stage s: + 8 s
    auto stage_off = [](uint32_t n) { return (n % NSTGF) * (STGF_BYTES >> 4); };
    auto kstep128 = [](int k) { return (uint32_t)((k / 4) * (SUB128 >> 4) + 2 * (k % 4)); };
    auto kstep64 = [](int k) { return (uint32_t)((k / 4) * (SUB64 >> 4) + 2 * (k % 4)); };
    auto scores = [&](uint32_t n) {  // S^T = K Q^T
      const uint32_t q = stg_lo + stage_off(n);
#pragma unroll
      for (int k = 0; k < HD / 16; ++k) mma_ss_lo(tmem_base, k_lo + kstep128(k), q + kstep64(k), id_s, k > 0);
      commit_to(s_full_at);
    };
    auto dpscores = [&](uint32_t n) {  // dP^T = V dO^T
      const uint32_t o = stg_lo + stage_off(n) + ((2 * SUB64) >> 4);
#pragma unroll
      for (int k = 0; k < HD / 16; ++k) mma_ss_lo(tmem_base + 64, v_lo + kstep128(k), o + kstep64(k), id_s, k > 0);
      commit_to(dp_full_at);
    };
    // dV += P^T dO and dK += dS^T Q: the stage's dO / Q tiles as MN-major B
    // operands (rows = queries = K dimension; 64-column chunks SUB64 apart).
    // P^T of queries 32x..32x+31 sits in columns 32x..32x+15 of the S^T region;
    // dS^T is packed contiguously (queries 2c, 2c+1 in column 192 + c).
    auto accum_v = [&](uint32_t n, bool acc) {
      const uint32_t o = stg_mn + stage_off(n) + ((2 * SUB64) >> 4);
#pragma unroll
      for (int k = 0; k < QBF / 16; ++k)
        mma_ts_lo(tmem_base + 256, tmem_base + 32 * (k / 2) + 8 * (k % 2), o + 128 * k, id_o, (acc || k > 0) ? 1u : 0u);
    };
    auto accum_kq = [&](uint32_t n, bool acc) {
      const uint32_t q = stg_mn + stage_off(n);
#pragma unroll
      for (int k = 0; k < QBF / 16; ++k)
        mma_ts_lo(tmem_base + 384, tmem_base + 192 + 8 * k, q + 128 * k, id_o, (acc || k > 0) ? 1u : 0u);
      // dQ^T = K^T dS^T: the K tile (rows = keys, head-dim chunks SUB128 apart) as
      // the MN-major A operand, dS^T (rows = keys, 64 queries) as the MN-major B
#pragma unroll
      for (int k = 0; k < 128 / 16; ++k) mma_ss_lo(tmem_base + 128, k_mn + 128 * k, ds_mn + 128 * k, id_q, k > 0);
      commit_to(dq_full_at);
      commit_to(q_free_at + 8 * (n % NSTGF));
    };
    auto sync_on = [&](int id, int count) {
      __syncwarp();
      named_bar_sync(id, count);
      tc_fence_after();
    };
    for (int t = 0; t < ntile; ++t) {
      const int64_t k0 = (int64_t)tile_of(t) * 128;
      const int nq = grp * (int)((p.S - k0) / QBF);  // query blocks of all the group's heads
      if (ok) {
        bool w = true;
        if (lane == 0) w = mbar_wait(kv_full, t & 1, abort_flag, p.err, CODE_FUSED | 4);
        ok = __shfl_sync(0xffffffffu, w ? 1 : 0, 0) != 0;
      }
      sync_on(kBarStage + (qi & 3), kStageThreads);
      if (ok) {
        scores(qi);
        dpscores(qi);
      }
      for (int i = 0; i < nq; ++i) {
        const uint32_t n = qi + i;
        sync_on(kBarPF, kDSThreads);  // P^T(n) in TMEM
        if (ok) accum_v(n, i > 0);
        if (i + 1 < nq) {
          sync_on(kBarStage + ((n + 1) & 3), kStageThreads);
          if (ok) scores(n + 1);
        }
        sync_on(kBarDSF, kDSThreads);  // dS^T(n) in TMEM and shared memory, dQ^T(n-1) read out
        if (ok) {
          if (i + 1 < nq) dpscores(n + 1);
          accum_kq(n, i > 0);
        }
      }
      if (ok) umma_commit_warp(kv_free);
      qi += nq;
    }
    umma_commit_warp(drain);
    if (lane == 0) {
      volatile int dummy = 0;
      mbar_wait(drain, 0, &dummy, p.err, CODE_FUSED | 7);
    }
    __syncwarp();
  } else if (warp == 10) {
    // ---------------- relay: announces each landed stage to the MMA warp ----------------
    uint32_t n = 0;
    for (int t = 0; t < ntile; ++t) {
      const int nq = grp * (int)((p.S - (int64_t)tile_of(t) * 128) / QBF);
      for (int i = 0; i < nq; ++i, ++n) {
        if (lane == 0) mbar_wait(&q_full[n % NSTGF], (n / NSTGF) & 1, abort_flag, p.err, CODE_FUSED | 9);
        __syncwarp();
        named_bar_sync(kBarStage + (n & 3), kStageThreads);
      }
    }
  } else {
    // ------- elementwise warps 0-7: one key row, 32 of the 64 query columns per thread -------
    // (for dQ^T the TMEM lane is a head-dim index instead: the thread adds
    // column d = its row of the 32 queries it covers)
    const int quad = warp & 3, half = warp >> 2;
    const int row = quad * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(quad * 32) << 16;
    const uint32_t cS = tmem_base + lane_off + 32 * half;
    const uint32_t cdP = tmem_base + lane_off + 64 + 32 * half;
    const uint32_t cdQ = tmem_base + lane_off + 128 + 32 * half;
    const uint32_t cdS = tmem_base + lane_off + 192 + 16 * half;
    const float sl2 = kLog2e * rsqrtf((float)HD);
    const uint64_t sl2x2 = f2pack(sl2, sl2), nlog2e2 = f2pack(-kLog2e, -kLog2e);
    const float scale = rsqrtf((float)HD);
    uint8_t* ds_row = dSs + row * 128;
    uint32_t cnt = 0;   // blocks processed (phase of s_full / dp_full; ring slot = cnt % NSTGF)
    bool alive = true;  // warp-uniform; once false the warp only keeps the hand-off count
    auto add_dq = [&](float* dst, const float (&a)[32]) {  // a block's dQ^T column -> fp32 accumulator
#pragma unroll
      for (int c = 0; c < 32; ++c) red_add_f32(dst + (int64_t)c * HD, a[c]);
    };
    for (int t = 0; t < ntile; ++t) {
      const int64_t k0 = (int64_t)tile_of(t) * 128;
      const int nqh = (int)((p.S - k0) / QBF);
      const int64_t key = k0 + row;
      float* dq_prev = nullptr;  // accumulator column of the previous block of this tile
      for (int u = 0; u < grp * nqh; ++u, ++cnt) {
        const int i = u % nqh;  // query block within the head
        const int head = kvh * grp + u / nqh;
        const int64_t q0 = k0 + (int64_t)i * QBF + 32 * half;  // query of this thread's first column
        // ---- P phase ----
        bool got = alive && mbar_wait(s_full, cnt & 1, abort_flag, p.err, CODE_FUSED | 8);
        alive = __all_sync(0xffffffffu, got);
        if (!alive) {
          named_bar_sync(kBarPF, kDSThreads);
          named_bar_sync(kBarDSF, kDSThreads);
          continue;
        }
        tc_fence_after();
        uint32_t sa[32];
        tmem_ld32_issue(cS, sa);
        const float4* lse4 = reinterpret_cast<const float4*>(ldr + (cnt % NSTGF) * LDF_BYTES) + 8 * half;
        const float4* ds4 = lse4 + QBF / 4;
        const bool diag = i < 2;  // the two blocks that overlap the key tile
        // P = 2^(s sl2 - lse log2e) in packed pairs (one f32x2 multiply and
        // one f32x2 FMA per two scores)
        uint64_t pv2[16];
        uint32_t pk[16];
        tmem_wait_ld32(sa);
        // The causal mask only touches the two blocks that overlap the key
        // tile; the others take the loop without the per-score test (a
        // warp-uniform branch, so it is not turned into selects).
        auto p_phase = [&](auto masked) {
#pragma unroll
          for (int c4 = 0; c4 < 8; ++c4) {
            const float4 l4 = lse4[c4];
            float a[4];
            f2unpack(f2fma(f2pack(__uint_as_float(sa[4 * c4]), __uint_as_float(sa[4 * c4 + 1])), sl2x2,
                           f2mul(f2pack(l4.x, l4.y), nlog2e2)),
                     a[0], a[1]);
            f2unpack(f2fma(f2pack(__uint_as_float(sa[4 * c4 + 2]), __uint_as_float(sa[4 * c4 + 3])), sl2x2,
                           f2mul(f2pack(l4.z, l4.w), nlog2e2)),
                     a[2], a[3]);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              a[e] = ex2f(a[e]);
              if constexpr (decltype(masked)::value)
                if (q0 + 4 * c4 + e < key) a[e] = 0.f;
            }
            pv2[2 * c4] = f2pack(a[0], a[1]);
            pv2[2 * c4 + 1] = f2pack(a[2], a[3]);
            pk[2 * c4] = pack_bf16x2(a[0], a[1]);
            pk[2 * c4 + 1] = pack_bf16x2(a[2], a[3]);
          }
        };
        if (diag)
          p_phase(std::true_type{});
        else
          p_phase(std::false_type{});
        tmem_st16_nowait(cS, pk);  // P^T over the start of this thread's S^T columns
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        named_bar_arrive(kBarPF, kDSThreads);
        // ---- dS phase ----
        got = mbar_wait(dp_full, cnt & 1, abort_flag, p.err, CODE_FUSED | 11);
        alive = __all_sync(0xffffffffu, got);
        if (!alive) {
          named_bar_sync(kBarDSF, kDSThreads);
          continue;
        }
        tc_fence_after();
        tmem_ld32_issue(cdP, sa);
        tmem_wait_ld32(sa);
        // dS = P (dP - dsum) in packed pairs
#pragma unroll
        for (int c4 = 0; c4 < 8; ++c4) {
          const float4 d4 = ds4[c4];
          float g[4];
          f2unpack(f2mul(pv2[2 * c4], f2sub(f2pack(__uint_as_float(sa[4 * c4]), __uint_as_float(sa[4 * c4 + 1])),
                                            f2pack(d4.x, d4.y))),
                   g[0], g[1]);
          f2unpack(f2mul(pv2[2 * c4 + 1], f2sub(f2pack(__uint_as_float(sa[4 * c4 + 2]), __uint_as_float(sa[4 * c4 + 3])),
                                                f2pack(d4.z, d4.w))),
                   g[2], g[3]);
          pk[2 * c4] = pack_bf16x2(g[0], g[1]);
          pk[2 * c4 + 1] = pack_bf16x2(g[2], g[3]);
        }
        // dK(n-1) and dQ(n-1) must be done with dS^T(n-1) before it is overwritten
        float qa[32];
        if (dq_prev != nullptr) {
          got = mbar_wait(dq_full, (cnt - 1) & 1, abort_flag, p.err, CODE_FUSED | 12);
          alive = __all_sync(0xffffffffu, got);
          if (!alive) {
            named_bar_sync(kBarDSF, kDSThreads);
            continue;
          }
          tc_fence_after();
          tmem_ld32(cdQ, qa);  // dQ^T(n-1), added to memory after the hand-off
        }
        tmem_st16_nowait(cdS, pk);
        // dS^T row for the dQ MMA: 16-byte chunks 4*half..4*half+3 of the
        // key's 128-byte row, XOR-swizzled by the row within its 8-row group
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int chunk = 4 * half + j;
          *reinterpret_cast<uint4*>(ds_row + ((chunk ^ (row & 7)) << 4)) =
              make_uint4(pk[4 * j], pk[4 * j + 1], pk[4 * j + 2], pk[4 * j + 3]);
        }
        fence_proxy_async_smem();
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        named_bar_arrive(kBarDSF, kDSThreads);
        if (dq_prev != nullptr) add_dq(dq_prev, qa);
        dq_prev = p.dq_acc + (((int64_t)b * p.H + head) * p.S + q0) * HD + row;
      }
      if (!alive) continue;
      // the tile's last dQ (its commit also covers the last dK, dV)
      const bool got = mbar_wait(dq_full, (cnt - 1) & 1, abort_flag, p.err, CODE_FUSED | 10);
      alive = __all_sync(0xffffffffu, got);
      if (!alive) continue;
      tc_fence_after();
      {
        float qa[32];
        tmem_ld32(cdQ, qa);
        add_dq(dq_prev, qa);
      }
      uint4* dvrow = reinterpret_cast<uint4*>(p.dv + (bkv * p.S + key) * HD) + 8 * half;
      uint4* dkrow = reinterpret_cast<uint4*>(p.dk + (bkv * p.S + key) * HD) + 8 * half;
#pragma unroll 1
      for (int c32 = 0; c32 < 2; ++c32) {
        float a[32], d[32];
        tmem_ld32(tmem_base + lane_off + 256 + 64 * half + 32 * c32, a);
        tmem_ld32(tmem_base + lane_off + 384 + 64 * half + 32 * c32, d);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          dvrow[c32 * 4 + q] = make_uint4(pack_bf16x2(a[q * 8 + 0], a[q * 8 + 1]), pack_bf16x2(a[q * 8 + 2], a[q * 8 + 3]),
                                          pack_bf16x2(a[q * 8 + 4], a[q * 8 + 5]), pack_bf16x2(a[q * 8 + 6], a[q * 8 + 7]));
          dkrow[c32 * 4 + q] = make_uint4(
              pack_bf16x2(d[q * 8 + 0] * scale, d[q * 8 + 1] * scale), pack_bf16x2(d[q * 8 + 2] * scale, d[q * 8 + 3] * scale),
              pack_bf16x2(d[q * 8 + 4] * scale, d[q * 8 + 5] * scale), pack_bf16x2(d[q * 8 + 6] * scale, d[q * 8 + 7] * scale));
        }
      }
      tc_fence_before();
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 9) {
    tc_fence_after();
    tmem_dealloc(tmem_base, 512);
  }
}

// ===========================================================================
// dQ
// ===========================================================================
constexpr int DQ_KB = 64;  // keys per block
constexpr int KSTG = 4;
constexpr uint32_t DQ_STAGE_BYTES = 4 * SUB64;  // K, V (2 sub-tiles each)
constexpr size_t DQ_SMEM = 1024 + 4 * (size_t)SUB128 + KSTG * (size_t)DQ_STAGE_BYTES + 256;

__global__ void __launch_bounds__(THREADS, 1)
    attn_dq_tc_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmdO,
                      const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                      const BwdTcParams p, int n_tiles) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* Qs = smem;                  // 2 x SUB128
  uint8_t* dOs = smem + 2 * SUB128;    // 2 x SUB128
  uint8_t* stg = smem + 4 * SUB128;    // [KSTG] stages
  uint64_t* bars = reinterpret_cast<uint64_t*>(stg + KSTG * DQ_STAGE_BYTES);
  uint64_t* q_full = bars + 0;
  uint64_t* q_free = bars + 1;
  uint64_t* k_full = bars + 2;   // [KSTG]
  uint64_t* k_free = bars + 6;   // [KSTG]
  uint64_t* s_full = bars + 10;  // [2]
  uint64_t* o_done = bars + 14;
  uint64_t* drain = bars + 15;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 16);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int head = blockIdx.y, b = blockIdx.z;
  const int64_t bh = (int64_t)b * p.H + head;
  const int64_t bkv = (int64_t)b * p.Hk + head / (p.H / p.Hk);  // the K/V head this query head reads
  const int total_tiles = 2 * p.D * n_tiles;
  auto tile_of = [&](int t) { return t == 0 ? total_tiles - 1 - (int)blockIdx.x : (int)blockIdx.x; };
  auto geo = [&](int g, int64_t& zrow0, int64_t& p0) {
    const int c = g / n_tiles, i = g % n_tiles;
    const int64_t r = c < p.D ? c : 2 * p.D - 1 - c;
    const int64_t off = (int64_t)i * 128;
    zrow0 = (r * p.B + b) * 2 * p.C + (c < p.D ? off : p.C + off);
    p0 = (int64_t)c * p.C + off;
  };

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    mbar_init(q_free, 1);
    for (int s = 0; s < KSTG; ++s) {
      mbar_init(&k_full[s], 1);
      mbar_init(&k_free[s], 1);
    }
    mbar_init(&s_full[0], 1);
    mbar_init(&s_full[1], 1);
    mbar_init(o_done, 1);
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbarrier_init();
  }
  if (warp == 8 && lane == 0) {
    tma_prefetch_desc(&tmQ);
    tma_prefetch_desc(&tmdO);
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
  }
  if (warp == 9) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  // TMEM columns: S[x] at 64x, dP[x] at 128 + 64x, dQ at 256.  dS (bf16
  // pairs) is written over the first 32 columns of S[x] and read from there by
  // the dQ MMA; MMAs of one CTA execute in issue order.

  if (warp == 8) {
    if (lane == 0) {
      uint32_t ki = 0;
      int q_armed = 0;
      bool ok = true;
      for (int t = 0; t < 2 && ok; ++t) {
        int64_t zrow0, p0;
        geo(tile_of(t), zrow0, p0);
        if (!mbar_wait(q_free, (t & 1) ^ 1, abort_flag, p.err, CODE_DQ | 1)) break;
        mbar_arrive_expect_tx(q_full, 4 * SUB128);
        ++q_armed;
        for (int c = 0; c < 2; ++c) {
          tma_load_2d(Qs + c * SUB128, &tmQ, head * HD + c * 64, (int)zrow0, q_full);
          tma_load_2d(dOs + c * SUB128, &tmdO, head * HD + c * 64, (int)zrow0, q_full);
        }
        const int nkb = (int)((p0 + 128) / DQ_KB);
        for (int j = 0; j < nkb; ++j, ++ki) {
          const int s = ki % KSTG;
          if (!mbar_wait(&k_free[s], ((ki / KSTG) & 1) ^ 1, abort_flag, p.err, CODE_DQ | 2)) {
            ok = false;
            break;
          }
          uint8_t* st = stg + s * DQ_STAGE_BYTES;
          mbar_arrive_expect_tx(&k_full[s], DQ_STAGE_BYTES);
          const int krow = (int)(bkv * p.S + (int64_t)j * DQ_KB);
          for (int c = 0; c < 2; ++c) {
            tma_load_2d(st + c * SUB64, &tmK, c * 64, krow, &k_full[s]);
            tma_load_2d(st + 2 * SUB64 + c * SUB64, &tmV, c * 64, krow, &k_full[s]);
          }
        }
      }
      volatile int dummy = 0;
      const uint32_t first = ki > KSTG ? ki - KSTG : 0;
      for (uint32_t n = first; n < ki; ++n) mbar_wait(&k_full[n % KSTG], (n / KSTG) & 1, &dummy, p.err, CODE_DQ | 3);
      if (q_armed) mbar_wait(q_full, (q_armed - 1) & 1, &dummy, p.err, CODE_DQ | 3);
    }
  } else if (warp == 9) {
    // ---------------- MMA issuer (whole warp walks the schedule and issues; one elected lane) ----------------
    constexpr uint32_t id_s = idesc_bf16_f32(128, DQ_KB);
    constexpr uint32_t id_o = idesc_bf16_f32(128, HD, false, true);  // B (K tile) MN-major
    uint32_t ki = 0;
    bool ok = true;  // warp-uniform
    auto scores = [&](uint32_t n, int x) {  // S = Q K^T, dP = dO V^T for key block n
      uint8_t* st = stg + (n % KSTG) * DQ_STAGE_BYTES;
#pragma unroll
      for (int k = 0; k < HD / 16; ++k) {
        const uint64_t aq = sdesc_kmajor_sw128(smem_u32(Qs + (k / 4) * SUB128)) + 2 * (k % 4);
        const uint64_t bk = sdesc_kmajor_sw128(smem_u32(st + (k / 4) * SUB64)) + 2 * (k % 4);
        umma_bf16_warp(tmem_base + 64 * x, aq, bk, id_s, k > 0);
      }
#pragma unroll
      for (int k = 0; k < HD / 16; ++k) {
        const uint64_t ao = sdesc_kmajor_sw128(smem_u32(dOs + (k / 4) * SUB128)) + 2 * (k % 4);
        const uint64_t bv = sdesc_kmajor_sw128(smem_u32(st + 2 * SUB64 + (k / 4) * SUB64)) + 2 * (k % 4);
        umma_bf16_warp(tmem_base + 128 + 64 * x, ao, bv, id_s, k > 0);
      }
      umma_commit_warp(&s_full[x]);
    };
    auto accumulate = [&](uint32_t n, int x, bool acc) {  // dQ += dS K for key block n (K tile as MN-major B)
      uint8_t* st = stg + (n % KSTG) * DQ_STAGE_BYTES;
#pragma unroll
      for (int k = 0; k < DQ_KB / 16; ++k) {
        const uint64_t bk = sdesc_mn_sw128(smem_u32(st) + 2048 * k, SUB64);
        umma_bf16_ts_warp(tmem_base + 256, tmem_base + 64 * x + 32 * (k / 2) + 8 * (k % 2), bk, id_o,
                     (acc || k > 0) ? 1u : 0u);
      }
      umma_commit_warp(&k_free[n % KSTG]);
    };
    auto sync_ds = [&](int j) {  // elementwise results of key block j of the tile are in TMEM
      __syncwarp();
      named_bar_sync(kBarDS + (j & 1), kDSThreads);
      tc_fence_after();
    };
    for (int t = 0; t < 2; ++t) {
      int64_t zrow0, p0;
      geo(tile_of(t), zrow0, p0);
      const int nkb = (int)((p0 + 128) / DQ_KB);
      if (ok) {
        bool w = true;
        if (lane == 0) w = mbar_wait(q_full, t & 1, abort_flag, p.err, CODE_DQ | 4);
        ok = __shfl_sync(0xffffffffu, w ? 1 : 0, 0) != 0;
      }
      for (int j = 0; j < nkb; ++j) {
        const uint32_t n = ki + j;
        __syncwarp();
        named_bar_sync(kBarStage + (n & 3), kStageThreads);  // stage n has landed
        tc_fence_after();
        if (ok) scores(n, j & 1);
        if (j > 0) {
          sync_ds(j - 1);
          if (ok) accumulate(n - 1, (j - 1) & 1, j - 1 > 0);
        }
      }
      sync_ds(nkb - 1);
      if (ok) {
        accumulate(ki + nkb - 1, (nkb - 1) & 1, nkb - 1 > 0);
        umma_commit_warp(o_done);
        umma_commit_warp(q_free);
      }
      ki += nkb;
    }
    umma_commit_warp(drain);
    if (lane == 0) {
      volatile int dummy = 0;
      mbar_wait(drain, 0, &dummy, p.err, CODE_DQ | 7);
    }
    __syncwarp();
  } else if (warp == 10) {
    // ---------------- relay: announces each landed stage to the MMA warp ----------------
    uint32_t n = 0;
    for (int t = 0; t < 2; ++t) {
      int64_t zrow0, p0;
      geo(tile_of(t), zrow0, p0);
      const int nkb = (int)((p0 + 128) / DQ_KB);
      for (int j = 0; j < nkb; ++j, ++n) {
        if (lane == 0) mbar_wait(&k_full[n % KSTG], (n / KSTG) & 1, abort_flag, p.err, CODE_DQ | 9);
        __syncwarp();
        named_bar_sync(kBarStage + (n & 3), kStageThreads);
      }
    }
  } else {
    // ------- elementwise warps 0-7: one query row, 32 of the 64 key columns per thread -------
    const int quad = warp & 3, half = warp >> 2;
    const int row = quad * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(quad * 32) << 16;
    const float sl2 = kLog2e * rsqrtf((float)HD);
    uint32_t scnt[2] = {0, 0};
    bool alive = true;  // warp-uniform; once false the warp only keeps the hand-off count
    for (int t = 0; t < 2; ++t) {
      int64_t zrow0, p0;
      geo(tile_of(t), zrow0, p0);
      const int nkb = (int)((p0 + 128) / DQ_KB);
      const int64_t qpos = p0 + row;
      const float l2 = p.lse[bh * p.S + qpos] * kLog2e;
      const float dsr = p.dsum[bh * p.S + qpos];
      for (int j = 0; j < nkb; ++j) {
        const int x = j & 1;
        const bool got = alive && mbar_wait(&s_full[x], scnt[x] & 1, abort_flag, p.err, CODE_DQ | 8);
        ++scnt[x];
        alive = __all_sync(0xffffffffu, got);
        if (!alive) {
          named_bar_sync(kBarDS + (j & 1), kDSThreads);
          continue;
        }
        tc_fence_after();
        const uint32_t cS = tmem_base + lane_off + 64 * x + 32 * half;
        float sv[32], dp[32];
        tmem_ld32(cS, sv);
        tmem_ld32(tmem_base + lane_off + 128 + 64 * x + 32 * half, dp);
        const int64_t key0 = (int64_t)j * DQ_KB + 32 * half;
        const bool diag = key0 + 31 > p0;
        uint32_t dsk[16];
#pragma unroll
        for (int c = 0; c < 32; c += 2) {
          float pv0 = ex2f(fmaf(sv[c], sl2, -l2));
          float pv1 = ex2f(fmaf(sv[c + 1], sl2, -l2));
          if (diag && key0 + c > qpos) pv0 = 0.f;
          if (diag && key0 + c + 1 > qpos) pv1 = 0.f;
          dsk[c / 2] = pack_bf16x2(pv0 * (dp[c] - dsr), pv1 * (dp[c + 1] - dsr));
        }
        tmem_st16_nowait(cS, dsk);  // dS over the start of this thread's S columns
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        named_bar_arrive(kBarDS + (j & 1), kDSThreads);
      }
      if (!alive) continue;
      const bool got = mbar_wait(o_done, t & 1, abort_flag, p.err, CODE_DQ | 10);
      alive = __all_sync(0xffffffffu, got);
      if (!alive) continue;
      tc_fence_after();
      float4* dst = reinterpret_cast<float4*>(p.dq_acc + (bh * p.S + qpos) * HD + 64 * half);
#pragma unroll 1
      for (int c32 = 0; c32 < 2; ++c32) {
        float a[32];
        tmem_ld32(tmem_base + lane_off + 256 + 64 * half + 32 * c32, a);
#pragma unroll
        for (int q = 0; q < 8; ++q) dst[c32 * 8 + q] = make_float4(a[4 * q], a[4 * q + 1], a[4 * q + 2], a[4 * q + 3]);
      }
      tc_fence_before();
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 9) {
    tc_fence_after();
    tmem_dealloc(tmem_base, 512);
  }
}

}  // namespace

bool attn_bwd_tc_supported(int head_dim, int64_t chunk) { return head_dim == HD && chunk % 128 == 0; }

tsp_status attn_bwd_bf16_tc(const AttnBwdTcArgs& a, cudaStream_t stream, int which) {
  if (!attn_bwd_tc_supported(a.dh, a.C)) return TSP_ERR_UNSUPPORTED;
  if ((int64_t)a.B * a.S == 0) return TSP_OK;
  const int64_t T = (int64_t)a.B * a.S;
  const int h = a.H * HD;
  const int64_t kv_rows = (int64_t)a.B * a.Hk * a.S;
  CUtensorMap mK128, mV128, mQ64, mdO64, mQ128, mdO128, mK64, mV64;
  if (!make_tma_2d_bf16(&mK128, a.k, kv_rows, HD, HD, 128) || !make_tma_2d_bf16(&mV128, a.v, kv_rows, HD, HD, 128) ||
      !make_tma_2d_bf16(&mQ64, a.q, T, h, h, 64) || !make_tma_2d_bf16(&mdO64, a.dO, T, h, h, 64) ||
      !make_tma_2d_bf16(&mQ128, a.q, T, h, h, 128) || !make_tma_2d_bf16(&mdO128, a.dO, T, h, h, 128) ||
      !make_tma_2d_bf16(&mK64, a.k, kv_rows, HD, HD, 64) || !make_tma_2d_bf16(&mV64, a.v, kv_rows, HD, HD, 64))
    return TSP_ERR_CUDA;
  static std::atomic<unsigned long long> configured{0};  // devices set up
  if (needs_setup(configured)) {
    if (cudaFuncSetAttribute(attn_dkdv128_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)DKDV2_SMEM) != cudaSuccess ||
        cudaFuncSetAttribute(attn_dq_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)DQ_SMEM) !=
            cudaSuccess ||
        cudaFuncSetAttribute(attn_bwd_fused_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)FUSED_SMEM) != cudaSuccess)
      return TSP_ERR_CUDA;
    mark_setup_done(configured);
  }
  BwdTcParams p;
  p.B = a.B;
  p.H = a.H;
  p.Hk = a.Hk;
  p.D = a.D;
  p.S = a.S;
  p.C = a.C;
  p.h = h;
  p.lse = a.lse;
  p.dsum = a.dsum;
  p.dq_acc = a.dq_acc;
  p.dk = static_cast<__nv_bfloat16*>(a.dk);
  p.dv = static_cast<__nv_bfloat16*>(a.dv);
  p.err = dev_error_word();
  const int nk = (int)(a.S / 128);
  dim3 g1((nk + 1) / 2, a.Hk, a.B);
  if (which & 4) {
    // Mirror pairs give every CTA the same work; when their count leaves the
    // last wave on the SMs mostly empty (few K/V heads, short sequences),
    // single tiles in decreasing order of work balance better.
    const int64_t pairs = (int64_t)g1.x * g1.y * g1.z;
    const int64_t sms = num_sms();
    const double pair_eff = (double)pairs / (double)(((pairs + sms - 1) / sms) * sms);
    if (pair_eff >= 0.9) {
      attn_bwd_fused_tc_kernel<<<g1, THREADS, FUSED_SMEM, stream>>>(mK128, mV128, mQ64, mdO64, p, nk, 1);
    } else {
      attn_bwd_fused_tc_kernel<<<dim3(a.Hk, a.B, nk), THREADS, FUSED_SMEM, stream>>>(mK128, mV128, mQ64, mdO64, p,
                                                                                     nk, 0);
    }
    if (cudaGetLastError() != cudaSuccess) return TSP_ERR_CUDA;
  }
  if (which & 1) {
    attn_dkdv128_tc_kernel<<<g1, THREADS, DKDV2_SMEM, stream>>>(mK128, mV128, mQ128, mdO128, p, nk);
    if (cudaGetLastError() != cudaSuccess) return TSP_ERR_CUDA;
  }
  if (!(which & 2)) return TSP_OK;
  const int n_tiles = (int)(a.C / 128);
  dim3 g2(a.D * n_tiles, a.H, a.B);
  attn_dq_tc_kernel<<<g2, THREADS, DQ_SMEM, stream>>>(mQ128, mdO128, mK64, mV64, p, n_tiles);
  return cudaGetLastError() == cudaSuccess ? TSP_OK : TSP_ERR_CUDA;
}

}  // namespace tsp
