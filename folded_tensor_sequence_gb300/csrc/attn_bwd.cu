// Causal flash-attention backward on the zigzag token layout (bf16, dh 128).
//
// The TSP posts do not describe the backward; this is the exact gradient of
// the forward, recomputing the probabilities from the saved log-sum-exp:
//   P = exp(S / sqrt(dh) - lse),  dV = P^T dO,  dP = dO V^T,
//   dS = P * (dP - rowsum(dO * O)),  dQ = dS K / sqrt(dh),  dK = dS^T Q / sqrt(dh).
// Three kernels, no atomics:
//   1. dsum[b][head][p] = rowsum(dO * O)
//   2. dK, dV: one CTA per mirror pair of 64-key tiles (tiles j and nk-1-j
//      together see a constant number of query blocks), looping over the
//      query blocks at or after the diagonal;
//   3. dQ: one CTA per mirror pair of 64-query tiles (the forward's zigzag
//      pairing), looping over the key tiles up to the diagonal.
// Queries, dO and dQ live in zigzag rows; K, V, dK, dV in gathered natural
// order per head.
#include "common.cuh"
#include "internal.h"
#include "warp_mma.cuh"

namespace tsp {

namespace {

using namespace wm;

constexpr int BT = 128;  // threads: 4 warps
constexpr int KT = 64;   // keys per dK/dV CTA tile (16 per warp)
constexpr int QB = 32;   // query rows per step of the dK/dV loop
constexpr int QT = 64;   // query rows per dQ CTA tile (16 per warp)

__device__ __forceinline__ int64_t zz_row(int64_t pos, int64_t C, int D, int B, int b) {
  const int64_t c = pos / C, off = pos - c * C;
  const int64_t r = c < D ? c : 2 * D - 1 - c;
  const int64_t k = c < D ? off : C + off;
  return (r * B + b) * 2 * C + k;
}

// rows [pos0, pos0+rows) of the zigzag [T][h] tensor, head slice -> swizzled smem
__device__ __forceinline__ void load_zz_rows(__nv_bfloat16* sm, const __nv_bfloat16* g, int64_t pos0, int rows,
                                             int64_t S, int64_t C, int D, int B, int b, int h, int head) {
  const uint32_t base = smem_u32(sm);
  for (int i = threadIdx.x; i < rows * CHUNKS; i += BT) {
    const int r = i / CHUNKS, c = i % CHUNKS;
    const int64_t pos = pos0 + r;
    const bool ok = pos < S;
    const __nv_bfloat16* src = g + (ok ? zz_row(pos, C, D, B, b) * h + head * DH + c * 8 : 0);
    cp_async16(base + swz(r, c * 8) * 2, src, ok);
  }
}

__global__ void dsum_kernel(const __nv_bfloat16* __restrict__ o, const __nv_bfloat16* __restrict__ dO,
                            float* __restrict__ dsum, int D, int B, int H, int64_t S, int64_t C,
                            float* __restrict__ dq_zero) {
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int64_t w = (int64_t)blockIdx.x * (blockDim.x / 32) + warp;  // over (b, head, pos)
  if (w >= (int64_t)B * H * S) return;
  const int64_t pos = w % S;
  const int64_t bh = w / S;
  const int head = (int)(bh % H), b = (int)(bh / H);
  const int h = H * DH;
  const int64_t row = zz_row(pos, C, D, B, b);
  const uint2 a = reinterpret_cast<const uint2*>(o + row * h + head * DH)[lane];
  const uint2 c = reinterpret_cast<const uint2*>(dO + row * h + head * DH)[lane];
  float2 a0 = unpack_bf16x2(a.x), a1 = unpack_bf16x2(a.y), c0 = unpack_bf16x2(c.x), c1 = unpack_bf16x2(c.y);
  float s = a0.x * c0.x + a0.y * c0.y + a1.x * c1.x + a1.y * c1.y;
  for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
  if (lane == 0) dsum[w] = s;
  // the same (b, head, pos) row of the fp32 dQ accumulator, 128 floats
  if (dq_zero != nullptr) reinterpret_cast<float4*>(dq_zero + w * DH)[lane] = make_float4(0.f, 0.f, 0.f, 0.f);
}

// ---------------------------------------------------------------------------
// dK, dV
// ---------------------------------------------------------------------------
constexpr size_t DKV_SMEM = (size_t)(2 * KT + 4 * QB) * DH * 2 + 4 * QB * sizeof(float);

__global__ void __launch_bounds__(BT) attn_dkdv_kernel(AttnBwdParams p, int nk) {
  extern __shared__ __align__(128) uint8_t sm[];
  __nv_bfloat16* Ks = reinterpret_cast<__nv_bfloat16*>(sm);
  __nv_bfloat16* Vs = Ks + KT * DH;
  __nv_bfloat16* Qs = Vs + KT * DH;      // [2][QB][DH]
  __nv_bfloat16* dOs = Qs + 2 * QB * DH;  // [2][QB][DH]
  float* lse2s = reinterpret_cast<float*>(dOs + 2 * QB * DH);  // [2][QB]
  float* dsums = lse2s + 2 * QB;                               // [2][QB]
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int g = lane / 4, t = lane % 4;
  const int head = blockIdx.y, b = blockIdx.z;
  const int D = p.D, B = p.B, H = p.H, h = H * DH;
  const int64_t S = p.S, C = p.C;
  const float scale = rsqrtf((float)DH);
  const float sl2 = kLog2e * scale;
  const int64_t bh = (int64_t)b * H + head;
  const __nv_bfloat16* Kg = static_cast<const __nv_bfloat16*>(p.k) + bh * S * DH;
  const __nv_bfloat16* Vg = static_cast<const __nv_bfloat16*>(p.v) + bh * S * DH;
  const __nv_bfloat16* Qg = static_cast<const __nv_bfloat16*>(p.q);
  const __nv_bfloat16* dOg = static_cast<const __nv_bfloat16*>(p.dO);
  const float* lseg = p.lse + bh * S;
  const float* dsg = p.dsum + bh * S;

  for (int which = 0; which < 2; ++which) {
    const int kt = which == 0 ? (int)blockIdx.x : nk - 1 - (int)blockIdx.x;
    if (which == 1 && kt == (int)blockIdx.x) break;  // middle tile of an odd count
    const int64_t k0 = (int64_t)kt * KT;
    const int nkeys = (int)min64(KT, S - k0);
    __syncthreads();
    load_tile_async<BT>(Ks, Kg + k0 * DH, DH, KT, nkeys);
    load_tile_async<BT>(Vs, Vg + k0 * DH, DH, KT, nkeys);
    const int64_t qb_first = k0 / QB;
    const int64_t nqb = (S + QB - 1) / QB;
    // first query block
    {
      const int64_t q0 = qb_first * QB;
      load_zz_rows(Qs, Qg, q0, QB, S, C, D, B, b, h, head);
      load_zz_rows(dOs, dOg, q0, QB, S, C, D, B, b, h, head);
      if (threadIdx.x < QB) {
        const int64_t q = q0 + threadIdx.x;
        lse2s[threadIdx.x] = q < S ? lseg[q] * kLog2e : INFINITY;
        dsums[threadIdx.x] = q < S ? dsg[q] : 0.f;
      }
    }
    cp_commit();
    cp_wait_all();
    __syncthreads();

    float dk[DH / 8][4], dv[DH / 8][4];
#pragma unroll
    for (int j = 0; j < DH / 8; ++j)
#pragma unroll
      for (int e = 0; e < 4; ++e) dk[j][e] = dv[j][e] = 0.f;
    const int64_t key_r0 = k0 + warp * 16 + g;  // this thread's key rows: key_r0, key_r0 + 8
    const uint32_t kbase = smem_u32(Ks), vbase = smem_u32(Vs);

    for (int64_t qb = qb_first; qb < nqb; ++qb) {
      const int buf = (int)((qb - qb_first) & 1);
      if (qb + 1 < nqb) {
        const int64_t q0n = (qb + 1) * QB;
        load_zz_rows(Qs + (buf ^ 1) * QB * DH, Qg, q0n, QB, S, C, D, B, b, h, head);
        load_zz_rows(dOs + (buf ^ 1) * QB * DH, dOg, q0n, QB, S, C, D, B, b, h, head);
        if (threadIdx.x < QB) {
          const int64_t q = q0n + threadIdx.x;
          lse2s[(buf ^ 1) * QB + threadIdx.x] = q < S ? lseg[q] * kLog2e : INFINITY;
          dsums[(buf ^ 1) * QB + threadIdx.x] = q < S ? dsg[q] : 0.f;
        }
      }
      cp_commit();
      const uint32_t qbase = smem_u32(Qs + buf * QB * DH), obase = smem_u32(dOs + buf * QB * DH);
      const float* l2 = lse2s + buf * QB;
      const float* ds = dsums + buf * QB;
      const int64_t q0 = qb * QB;

      // S^T = K_w Q^T and dP^T = V_w dO^T, 16 keys x QB queries
      float st[QB / 8][4], dpt[QB / 8][4];
#pragma unroll
      for (int j = 0; j < QB / 8; ++j)
#pragma unroll
        for (int e = 0; e < 4; ++e) st[j][e] = dpt[j][e] = 0.f;
#pragma unroll
      for (int kk = 0; kk < DH / 16; ++kk) {
        uint32_t ak[4], av[4];
        const int arow = warp * 16 + (lane % 16);
        const int acol = (2 * kk + lane / 16) * 8;
        ldsm_x4(kbase + swz(arow, acol) * 2, ak[0], ak[1], ak[2], ak[3]);
        ldsm_x4(vbase + swz(arow, acol) * 2, av[0], av[1], av[2], av[3]);
#pragma unroll
        for (int jp = 0; jp < QB / 16; ++jp) {
          const int brow = jp * 16 + (lane % 8) + (lane / 16) * 8;
          const int bcol = (2 * kk + (lane / 8) % 2) * 8;
          uint32_t b0, b1, b2, b3;
          ldsm_x4(qbase + swz(brow, bcol) * 2, b0, b1, b2, b3);
          mma16816(st[2 * jp], ak, b0, b1);
          mma16816(st[2 * jp + 1], ak, b2, b3);
          ldsm_x4(obase + swz(brow, bcol) * 2, b0, b1, b2, b3);
          mma16816(dpt[2 * jp], av, b0, b1);
          mma16816(dpt[2 * jp + 1], av, b2, b3);
        }
      }
      // P^T and dS^T
#pragma unroll
      for (int j = 0; j < QB / 8; ++j) {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int qi = j * 8 + 2 * t + (e & 1);
          const int64_t key = key_r0 + ((e >= 2) ? 8 : 0);
          const int64_t q = q0 + qi;
          float pv = ex2(st[j][e] * sl2 - l2[qi]);
          if (q < key) pv = 0.f;
          st[j][e] = pv;
          dpt[j][e] = pv * (dpt[j][e] - ds[qi]);
        }
      }
      // dV += P^T dO,  dK += dS^T Q   (k = queries)
#pragma unroll
      for (int kk2 = 0; kk2 < QB / 16; ++kk2) {
        uint32_t ap[4], as[4];
        ap[0] = pack_bf16x2(st[2 * kk2][0], st[2 * kk2][1]);
        ap[1] = pack_bf16x2(st[2 * kk2][2], st[2 * kk2][3]);
        ap[2] = pack_bf16x2(st[2 * kk2 + 1][0], st[2 * kk2 + 1][1]);
        ap[3] = pack_bf16x2(st[2 * kk2 + 1][2], st[2 * kk2 + 1][3]);
        as[0] = pack_bf16x2(dpt[2 * kk2][0], dpt[2 * kk2][1]);
        as[1] = pack_bf16x2(dpt[2 * kk2][2], dpt[2 * kk2][3]);
        as[2] = pack_bf16x2(dpt[2 * kk2 + 1][0], dpt[2 * kk2 + 1][1]);
        as[3] = pack_bf16x2(dpt[2 * kk2 + 1][2], dpt[2 * kk2 + 1][3]);
#pragma unroll
        for (int jd = 0; jd < DH / 16; ++jd) {
          const int brow = kk2 * 16 + (lane % 8) + ((lane / 8) % 2) * 8;
          const int bcol = (2 * jd + lane / 16) * 8;
          uint32_t b0, b1, b2, b3;
          ldsm_x4_t(obase + swz(brow, bcol) * 2, b0, b1, b2, b3);
          mma16816(dv[2 * jd], ap, b0, b1);
          mma16816(dv[2 * jd + 1], ap, b2, b3);
          ldsm_x4_t(qbase + swz(brow, bcol) * 2, b0, b1, b2, b3);
          mma16816(dk[2 * jd], as, b0, b1);
          mma16816(dk[2 * jd + 1], as, b2, b3);
        }
      }
      cp_wait_all();
      __syncthreads();
    }
    // store dK (scaled), dV
    __nv_bfloat16* dKg = static_cast<__nv_bfloat16*>(p.dk) + bh * S * DH;
    __nv_bfloat16* dVg = static_cast<__nv_bfloat16*>(p.dv) + bh * S * DH;
#pragma unroll
    for (int hr = 0; hr < 2; ++hr) {
      const int64_t key = key_r0 + 8 * hr;
      if (key - k0 < nkeys) {
#pragma unroll
        for (int j = 0; j < DH / 8; ++j) {
          const int64_t off = key * DH + j * 8 + 2 * t;
          *reinterpret_cast<uint32_t*>(dKg + off) = pack_bf16x2(dk[j][2 * hr] * scale, dk[j][2 * hr + 1] * scale);
          *reinterpret_cast<uint32_t*>(dVg + off) = pack_bf16x2(dv[j][2 * hr], dv[j][2 * hr + 1]);
        }
      }
    }
  }
}

// ---------------------------------------------------------------------------
// dQ
// ---------------------------------------------------------------------------
constexpr size_t DQ_SMEM = (size_t)(2 * QT + 4 * KT) * DH * 2;

__global__ void __launch_bounds__(BT) attn_dq_kernel(AttnBwdParams p, int n_tiles) {
  extern __shared__ __align__(128) uint8_t sm[];
  __nv_bfloat16* Qs = reinterpret_cast<__nv_bfloat16*>(sm);
  __nv_bfloat16* dOs = Qs + QT * DH;
  __nv_bfloat16* Ks = dOs + QT * DH;  // [2][KT][DH]
  __nv_bfloat16* Vs = Ks + 2 * KT * DH;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int g = lane / 4, t = lane % 4;
  const int head = blockIdx.y, b = blockIdx.z;
  const int D = p.D, B = p.B, H = p.H, h = H * DH;
  const int64_t S = p.S, C = p.C;
  const float scale = rsqrtf((float)DH);
  const float sl2 = kLog2e * scale;
  const int64_t bh = (int64_t)b * H + head;
  const __nv_bfloat16* Kg = static_cast<const __nv_bfloat16*>(p.k) + bh * S * DH;
  const __nv_bfloat16* Vg = static_cast<const __nv_bfloat16*>(p.v) + bh * S * DH;
  const int total_tiles = 2 * D * n_tiles;

  for (int which = 0; which < 2; ++which) {
    const int gt = which == 0 ? total_tiles - 1 - (int)blockIdx.x : (int)blockIdx.x;
    const int c = gt / n_tiles, i = gt % n_tiles;
    const int64_t off = (int64_t)i * QT;
    const int nrows = (int)min64(QT, C - off);
    const int64_t r = c < D ? c : 2 * D - 1 - c;
    const int64_t kz0 = c < D ? off : C + off;
    const int64_t zrow0 = (r * B + b) * 2 * C + kz0;
    const int64_t p0 = (int64_t)c * C + off;
    const int64_t qlast = p0 + nrows - 1;
    const int nkt = (int)(qlast / KT) + 1;

    __syncthreads();
    load_tile_async<BT>(Qs, static_cast<const __nv_bfloat16*>(p.q) + zrow0 * h + head * DH, h, QT, nrows);
    load_tile_async<BT>(dOs, static_cast<const __nv_bfloat16*>(p.dO) + zrow0 * h + head * DH, h, QT, nrows);
    load_tile_async<BT>(Ks, Kg, DH, KT, (int)min64(KT, S));
    load_tile_async<BT>(Vs, Vg, DH, KT, (int)min64(KT, S));
    cp_commit();
    cp_wait_all();
    __syncthreads();

    const int lr0 = warp * 16 + g;
    const int64_t qpos0 = p0 + lr0, qpos1 = qpos0 + 8;
    float l2[2], dsr[2];
    l2[0] = lr0 < nrows ? p.lse[bh * S + qpos0] * kLog2e : 0.f;
    l2[1] = lr0 + 8 < nrows ? p.lse[bh * S + qpos1] * kLog2e : 0.f;
    dsr[0] = lr0 < nrows ? p.dsum[bh * S + qpos0] : 0.f;
    dsr[1] = lr0 + 8 < nrows ? p.dsum[bh * S + qpos1] : 0.f;

    float dq[DH / 8][4];
#pragma unroll
    for (int j = 0; j < DH / 8; ++j) dq[j][0] = dq[j][1] = dq[j][2] = dq[j][3] = 0.f;
    const uint32_t qbase = smem_u32(Qs), obase = smem_u32(dOs);

    for (int kt = 0; kt < nkt; ++kt) {
      const int buf = kt & 1;
      if (kt + 1 < nkt) {
        const int64_t key0 = (int64_t)(kt + 1) * KT;
        const int valid = (int)min64(KT, S - key0);
        load_tile_async<BT>(Ks + (buf ^ 1) * KT * DH, Kg + key0 * DH, DH, KT, valid);
        load_tile_async<BT>(Vs + (buf ^ 1) * KT * DH, Vg + key0 * DH, DH, KT, valid);
      }
      cp_commit();
      const uint32_t kbase = smem_u32(Ks + buf * KT * DH), vbase = smem_u32(Vs + buf * KT * DH);
      float s[KT / 8][4], dp[KT / 8][4];
#pragma unroll
      for (int j = 0; j < KT / 8; ++j)
#pragma unroll
        for (int e = 0; e < 4; ++e) s[j][e] = dp[j][e] = 0.f;
#pragma unroll
      for (int kk = 0; kk < DH / 16; ++kk) {
        uint32_t aq[4], ao[4];
        const int arow = warp * 16 + (lane % 16);
        const int acol = (2 * kk + lane / 16) * 8;
        ldsm_x4(qbase + swz(arow, acol) * 2, aq[0], aq[1], aq[2], aq[3]);
        ldsm_x4(obase + swz(arow, acol) * 2, ao[0], ao[1], ao[2], ao[3]);
#pragma unroll
        for (int jp = 0; jp < KT / 16; ++jp) {
          const int brow = jp * 16 + (lane % 8) + (lane / 16) * 8;
          const int bcol = (2 * kk + (lane / 8) % 2) * 8;
          uint32_t b0, b1, b2, b3;
          ldsm_x4(kbase + swz(brow, bcol) * 2, b0, b1, b2, b3);
          mma16816(s[2 * jp], aq, b0, b1);
          mma16816(s[2 * jp + 1], aq, b2, b3);
          ldsm_x4(vbase + swz(brow, bcol) * 2, b0, b1, b2, b3);
          mma16816(dp[2 * jp], ao, b0, b1);
          mma16816(dp[2 * jp + 1], ao, b2, b3);
        }
      }
      const int64_t key_base = (int64_t)kt * KT;
#pragma unroll
      for (int j = 0; j < KT / 8; ++j) {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int hr = e >> 1;
          const int64_t key = key_base + j * 8 + 2 * t + (e & 1);
          const int64_t qp = hr ? qpos1 : qpos0;
          float pv = ex2(s[j][e] * sl2 - l2[hr]);
          if (key > qp) pv = 0.f;
          s[j][e] = pv * (dp[j][e] - dsr[hr]);  // dS
        }
      }
      // dQ += dS K
#pragma unroll
      for (int kk2 = 0; kk2 < KT / 16; ++kk2) {
        uint32_t a[4];
        a[0] = pack_bf16x2(s[2 * kk2][0], s[2 * kk2][1]);
        a[1] = pack_bf16x2(s[2 * kk2][2], s[2 * kk2][3]);
        a[2] = pack_bf16x2(s[2 * kk2 + 1][0], s[2 * kk2 + 1][1]);
        a[3] = pack_bf16x2(s[2 * kk2 + 1][2], s[2 * kk2 + 1][3]);
#pragma unroll
        for (int jd = 0; jd < DH / 16; ++jd) {
          const int brow = kk2 * 16 + (lane % 8) + ((lane / 8) % 2) * 8;
          const int bcol = (2 * jd + lane / 16) * 8;
          uint32_t b0, b1, b2, b3;
          ldsm_x4_t(kbase + swz(brow, bcol) * 2, b0, b1, b2, b3);
          mma16816(dq[2 * jd], a, b0, b1);
          mma16816(dq[2 * jd + 1], a, b2, b3);
        }
      }
      cp_wait_all();
      __syncthreads();
    }
    __nv_bfloat16* dQg = static_cast<__nv_bfloat16*>(p.dq);
#pragma unroll
    for (int hr = 0; hr < 2; ++hr) {
      const int lr = lr0 + 8 * hr;
      if (lr < nrows) {
        __nv_bfloat16* row = dQg + (zrow0 + lr) * h + head * DH;
#pragma unroll
        for (int j = 0; j < DH / 8; ++j)
          *reinterpret_cast<uint32_t*>(row + j * 8 + 2 * t) =
              pack_bf16x2(dq[j][2 * hr] * scale, dq[j][2 * hr + 1] * scale);
      }
    }
  }
}

}  // namespace

cudaError_t launch_attn_dsum(const void* o, const void* dO, float* dsum, int D, int B, int H, int64_t S, int64_t C,
                             cudaStream_t stream, float* dq_zero) {
  const int64_t rows = (int64_t)B * H * S;
  if (rows == 0) return cudaSuccess;
  dsum_kernel<<<(unsigned)((rows + 7) / 8), 256, 0, stream>>>(static_cast<const __nv_bfloat16*>(o),
                                                              static_cast<const __nv_bfloat16*>(dO), dsum, D, B, H,
                                                              S, C, dq_zero);
  return cudaGetLastError();
}

tsp_status attn_bwd_bf16(const AttnBwdParams& p, cudaStream_t stream) {
  if (p.dh != DH) return TSP_ERR_UNSUPPORTED;
  if (p.B * p.S == 0) return TSP_OK;
  static std::atomic<unsigned long long> configured{0};  // devices set up
  if (needs_setup(configured)) {
    if (cudaFuncSetAttribute(attn_dkdv_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)DKV_SMEM) !=
            cudaSuccess ||
        cudaFuncSetAttribute(attn_dq_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)DQ_SMEM) !=
            cudaSuccess)
      return TSP_ERR_CUDA;
    mark_setup_done(configured);
  }
  const int64_t rows = (int64_t)p.B * p.H * p.S;
  dsum_kernel<<<(unsigned)((rows + 7) / 8), 256, 0, stream>>>(static_cast<const __nv_bfloat16*>(p.o),
                                                              static_cast<const __nv_bfloat16*>(p.dO), p.dsum, p.D,
                                                              p.B, p.H, p.S, p.C, nullptr);
  const int nk = (int)((p.S + KT - 1) / KT);
  dim3 g1((nk + 1) / 2, p.H, p.B);
  attn_dkdv_kernel<<<g1, BT, DKV_SMEM, stream>>>(p, nk);
  const int n_tiles = (int)((p.C + QT - 1) / QT);
  dim3 g2(p.D * n_tiles, p.H, p.B);
  attn_dq_kernel<<<g2, BT, DQ_SMEM, stream>>>(p, n_tiles);
  return cudaGetLastError() == cudaSuccess ? TSP_OK : TSP_ERR_CUDA;
}

}  // namespace tsp
