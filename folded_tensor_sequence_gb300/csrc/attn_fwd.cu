// Causal flash attention on the zigzag token layout.
//
// Queries come from the zigzag rows of the rank that owns them; keys and
// values come from the gathered, natural-order per-head tensors (the K/V
// all-gather of the TSP attention schedule, ai-trends.today TSP article,
// "How to Fold a Book").  Key j is visible to query i iff pos(j) <= pos(i) in
// global sequence positions.  Online softmax as in FlashAttention / ring
// attention (r007 chapter, "Параллелизм по контексту: Ring Attention против
// Ulysses").
//
// Schedule.  A chunk of C queries is split into n = ceil(C/128) query tiles;
// tile g (global, over the 2D chunks) needs g+1 key tiles of 128.  Each CTA
// takes the mirror pair (g, 2Dn-1-g), which lie in chunks c and 2D-1-c of the
// SAME rank, so every CTA -- and every rank -- does 2Dn+1 key tiles: the
// zigzag balance carried down to the tile schedule.  Fully masked key tiles
// are never visited; only tiles crossing the diagonal apply the element mask.
#include "common.cuh"
#include "internal.h"
#include "warp_mma.cuh"

namespace tsp {

namespace {

using namespace wm;

// ===========================================================================
// fp32 path: one warp per (query row, head); exact fp32 arithmetic.
// ===========================================================================
__global__ void attn_fwd_f32_kernel(AttnParams p) {
  extern __shared__ float qs_all[];
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int64_t twoC = 2 * p.C, per_rank = (int64_t)p.B * twoC;
  const int64_t T = p.rank < 0 ? (int64_t)p.B * p.S : per_rank;  // rows of q and o
  const int64_t w = (int64_t)blockIdx.x * (blockDim.x / 32) + warp;
  if (w >= T * p.H) return;
  const int64_t zrow = w / p.H;  // row of q and o
  const int head = (int)(w % p.H);
  const int64_t r = p.rank < 0 ? zrow / per_rank : p.rank, rem = p.rank < 0 ? zrow % per_rank : zrow;
  const int64_t b = rem / twoC, kk = rem % twoC;
  const int64_t qpos = kk < p.C ? r * p.C + kk : (2 * p.D - 1 - r) * p.C + (kk - p.C);
  const int dh = p.dh, h = p.H * dh;
  float* qs = qs_all + warp * dh;
  const float* q = static_cast<const float*>(p.q) + zrow * h + head * dh;
  for (int d = lane; d < dh; d += 32) qs[d] = q[d];
  __syncwarp();
  const float scale = 1.0f / sqrtf((float)dh);
  const int kvh = head / (p.H / p.Hk);  // K/V head read by this query head
  const float* K = static_cast<const float*>(p.k) + ((b * p.Hk + kvh) * p.S) * dh;
  const float* V = static_cast<const float*>(p.v) + ((b * p.Hk + kvh) * p.S) * dh;
  float m = -INFINITY, l = 0.0f;
  float o[4] = {0.f, 0.f, 0.f, 0.f};  // dims lane + 32 i
  for (int64_t j0 = 0; j0 <= qpos; j0 += 32) {
    const int64_t j = j0 + lane;
    float s = -INFINITY;
    if (j <= qpos) {
      const float* kr = K + j * dh;
      float dot = 0.f;
      for (int d = 0; d < dh; ++d) dot = fmaf(qs[d], kr[d], dot);
      s = dot * scale;
    }
    float mx = s;
    for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
    const float m_new = fmaxf(m, mx);
    const float corr = expf(m - m_new);
    const float e = (j <= qpos) ? expf(s - m_new) : 0.f;
    float sum = e;
    for (int off = 16; off > 0; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
    l = l * corr + sum;
    for (int i = 0; i < 4; ++i) o[i] *= corr;
    const int64_t jmax = qpos - j0 < 31 ? qpos - j0 : 31;
    for (int jj = 0; jj <= jmax; ++jj) {
      const float pj = __shfl_sync(0xffffffffu, e, jj);
      const float* vr = V + (j0 + jj) * dh;
      for (int i = 0; i < 4; ++i) {
        const int d = lane + 32 * i;
        if (d < dh) o[i] = fmaf(pj, vr[d], o[i]);
      }
    }
    m = m_new;
  }
  float* out = static_cast<float*>(p.o) + zrow * h + head * dh;
  const float inv = 1.0f / l;
  for (int i = 0; i < 4; ++i) {
    const int d = lane + 32 * i;
    if (d < dh) out[d] = o[i] * inv;
  }
  if (p.lse && lane == 0) p.lse[(b * p.H + head) * p.S + qpos] = m + logf(l);
}

// ===========================================================================
// bf16 path: warp-level tensor-core MMA (m16n8k16), 128 queries x 64 keys per
// step, K/V double-buffered through shared memory with cp.async.
// ===========================================================================
constexpr int BQ = 128;
constexpr int BKV = 64;
constexpr int ATT_THREADS = 256;
constexpr size_t ATT_SMEM = (size_t)(BQ + 4 * BKV) * DH * 2;

__global__ void __launch_bounds__(ATT_THREADS) attn_fwd_bf16_kernel(AttnParams p, int n_tiles) {
  extern __shared__ __align__(128) uint8_t att_smem[];
  __nv_bfloat16* Qs = reinterpret_cast<__nv_bfloat16*>(att_smem);
  __nv_bfloat16* Ks = Qs + BQ * DH;       // [2][BKV][DH]
  __nv_bfloat16* Vs = Ks + 2 * BKV * DH;  // [2][BKV][DH]
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int g = lane / 4, t = lane % 4;
  const int head = blockIdx.y, b = blockIdx.z;
  const int D = p.D;
  const int64_t C = p.C, S = p.S;
  const int h = p.H * DH;
  const float sl2 = kLog2e / sqrtf((float)DH);
  const int kvh = head / (p.H / p.Hk);  // K/V head read by this query head
  const __nv_bfloat16* Kg = static_cast<const __nv_bfloat16*>(p.k) + ((int64_t)b * p.Hk + kvh) * S * DH;
  const __nv_bfloat16* Vg = static_cast<const __nv_bfloat16*>(p.v) + ((int64_t)b * p.Hk + kvh) * S * DH;
  const int total_tiles = 2 * D * n_tiles;

  // one rank's queries: that rank's light tiles only, q and o holding its rows alone
  const int light = (p.rank < 0 ? 0 : p.rank * n_tiles) + (int)blockIdx.x;
  const int64_t row_off = p.rank < 0 ? 0 : (int64_t)p.rank * p.B * 2 * C;
  for (int which = 0; which < 2; ++which) {
    // heavy tile of the mirror pair first
    const int gt = which == 0 ? total_tiles - 1 - light : light;
    const int c = gt / n_tiles, i = gt % n_tiles;
    const int64_t off = (int64_t)i * BQ;
    const int nrows = (int)min64(BQ, C - off);
    const int64_t r = c < D ? c : 2 * D - 1 - c;
    const int64_t k0 = c < D ? off : C + off;
    const int64_t zrow0 = (r * p.B + b) * 2 * C + k0 - row_off;
    const int64_t p0 = (int64_t)c * C + off;  // global position of the tile's first query
    const int64_t qlast = p0 + nrows - 1;
    const int nkt = (int)(qlast / BKV) + 1;

    __syncthreads();  // previous tile's smem readers are done
    load_tile_async<ATT_THREADS>(Qs, static_cast<const __nv_bfloat16*>(p.q) + zrow0 * h + head * DH, h, BQ, nrows);
    load_tile_async<ATT_THREADS>(Ks, Kg, DH, BKV, (int)min64(BKV, S));
    load_tile_async<ATT_THREADS>(Vs, Vg, DH, BKV, (int)min64(BKV, S));
    cp_commit();
    cp_wait_all();
    __syncthreads();

    uint32_t qf[DH / 16][4];
    {
      const uint32_t qbase = smem_u32(Qs);
#pragma unroll
      for (int kk = 0; kk < DH / 16; ++kk) {
        const int row = warp * 16 + (lane % 16);
        const int col = (2 * kk + lane / 16) * 8;
        ldsm_x4(qbase + swz(row, col) * 2, qf[kk][0], qf[kk][1], qf[kk][2], qf[kk][3]);
      }
    }
    float oacc[DH / 8][4];
#pragma unroll
    for (int j = 0; j < DH / 8; ++j) oacc[j][0] = oacc[j][1] = oacc[j][2] = oacc[j][3] = 0.f;
    float mrow[2] = {-INFINITY, -INFINITY}, lrow[2] = {0.f, 0.f};
    const int64_t qpos0 = p0 + warp * 16 + g;
    const int64_t qpos1 = qpos0 + 8;

    for (int kt = 0; kt < nkt; ++kt) {
      const int buf = kt & 1;
      if (kt + 1 < nkt) {
        const int64_t key0 = (int64_t)(kt + 1) * BKV;
        const int valid = (int)min64(BKV, S - key0);
        load_tile_async<ATT_THREADS>(Ks + (buf ^ 1) * BKV * DH, Kg + key0 * DH, DH, BKV, valid);
        load_tile_async<ATT_THREADS>(Vs + (buf ^ 1) * BKV * DH, Vg + key0 * DH, DH, BKV, valid);
      }
      cp_commit();
      const uint32_t kbase = smem_u32(Ks + buf * BKV * DH);
      const uint32_t vbase = smem_u32(Vs + buf * BKV * DH);

      float s[BKV / 8][4];
#pragma unroll
      for (int j = 0; j < BKV / 8; ++j) s[j][0] = s[j][1] = s[j][2] = s[j][3] = 0.f;
#pragma unroll
      for (int kk = 0; kk < DH / 16; ++kk) {
#pragma unroll
        for (int jp = 0; jp < BKV / 16; ++jp) {
          const int key = jp * 16 + (lane % 8) + (lane / 16) * 8;
          const int col = (2 * kk + (lane / 8) % 2) * 8;
          uint32_t b0, b1, b2, b3;
          ldsm_x4(kbase + swz(key, col) * 2, b0, b1, b2, b3);
          mma16816(s[2 * jp], qf[kk], b0, b1);
          mma16816(s[2 * jp + 1], qf[kk], b2, b3);
        }
      }
      // scale to log2 units and mask keys beyond the diagonal
      const int64_t key_base = (int64_t)kt * BKV;
      const bool diag = key_base + BKV - 1 > p0;
#pragma unroll
      for (int j = 0; j < BKV / 8; ++j) {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          float v = s[j][e] * sl2;
          if (diag) {
            const int64_t key = key_base + j * 8 + 2 * t + (e & 1);
            const int64_t qp = (e < 2) ? qpos0 : qpos1;
            if (key > qp) v = -INFINITY;
          }
          s[j][e] = v;
        }
      }
      // online softmax, rows g (e = 0,1) and g+8 (e = 2,3)
#pragma unroll
      for (int hr = 0; hr < 2; ++hr) {
        float mx = -INFINITY;
#pragma unroll
        for (int j = 0; j < BKV / 8; ++j) mx = fmaxf(mx, fmaxf(s[j][2 * hr], s[j][2 * hr + 1]));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
        const float m_new = fmaxf(mrow[hr], mx);
        const float corr = ex2(mrow[hr] - m_new);
        float sum = 0.f;
#pragma unroll
        for (int j = 0; j < BKV / 8; ++j) {
          const float e0 = ex2(s[j][2 * hr] - m_new);
          const float e1 = ex2(s[j][2 * hr + 1] - m_new);
          s[j][2 * hr] = e0;
          s[j][2 * hr + 1] = e1;
          sum += e0 + e1;
        }
        lrow[hr] = lrow[hr] * corr + sum;  // per-thread partial; reduced at the end
        mrow[hr] = m_new;
#pragma unroll
        for (int j = 0; j < DH / 8; ++j) {
          oacc[j][2 * hr] *= corr;
          oacc[j][2 * hr + 1] *= corr;
        }
      }
      // O += P V
#pragma unroll
      for (int kk2 = 0; kk2 < BKV / 16; ++kk2) {
        uint32_t a[4];
        a[0] = pack_bf16x2(s[2 * kk2][0], s[2 * kk2][1]);
        a[1] = pack_bf16x2(s[2 * kk2][2], s[2 * kk2][3]);
        a[2] = pack_bf16x2(s[2 * kk2 + 1][0], s[2 * kk2 + 1][1]);
        a[3] = pack_bf16x2(s[2 * kk2 + 1][2], s[2 * kk2 + 1][3]);
#pragma unroll
        for (int jd = 0; jd < DH / 16; ++jd) {
          const int key = kk2 * 16 + (lane % 8) + ((lane / 8) % 2) * 8;
          const int col = (2 * jd + lane / 16) * 8;
          uint32_t b0, b1, b2, b3;
          ldsm_x4_t(vbase + swz(key, col) * 2, b0, b1, b2, b3);
          mma16816(oacc[2 * jd], a, b0, b1);
          mma16816(oacc[2 * jd + 1], a, b2, b3);
        }
      }
      cp_wait_all();
      __syncthreads();
    }
    // finalize: full row sums across the quad, normalize, store
#pragma unroll
    for (int hr = 0; hr < 2; ++hr) {
      float l = lrow[hr];
      l += __shfl_xor_sync(0xffffffffu, l, 1);
      l += __shfl_xor_sync(0xffffffffu, l, 2);
      lrow[hr] = l;
    }
    __nv_bfloat16* Og = static_cast<__nv_bfloat16*>(p.o);
#pragma unroll
    for (int hr = 0; hr < 2; ++hr) {
      const int lr = warp * 16 + g + 8 * hr;
      if (lr < nrows) {
        const float inv = 1.0f / lrow[hr];
        __nv_bfloat16* orow = Og + (zrow0 + lr) * h + head * DH;
#pragma unroll
        for (int j = 0; j < DH / 8; ++j) {
          *reinterpret_cast<uint32_t*>(orow + j * 8 + 2 * t) =
              pack_bf16x2(oacc[j][2 * hr] * inv, oacc[j][2 * hr + 1] * inv);
        }
        if (p.lse && t == 0) p.lse[((int64_t)b * p.H + head) * S + p0 + lr] = (mrow[hr] + __log2f(lrow[hr])) * kLn2;
      }
    }
  }
}

}  // namespace

tsp_status attn_fwd_f32(const AttnParams& p, cudaStream_t stream) {
  const int64_t warps = (p.rank < 0 ? (int64_t)p.B * p.S : (int64_t)p.B * 2 * p.C) * p.H;
  if (warps == 0) return TSP_OK;
  if (p.dh > 128) return TSP_ERR_UNSUPPORTED;
  const int wpb = 8;
  const int64_t blocks = (warps + wpb - 1) / wpb;
  attn_fwd_f32_kernel<<<(unsigned)blocks, wpb * 32, wpb * p.dh * sizeof(float), stream>>>(p);
  return cudaGetLastError() == cudaSuccess ? TSP_OK : TSP_ERR_CUDA;
}

tsp_status attn_fwd_bf16(const AttnParams& p, cudaStream_t stream) {
  if (p.dh != DH) return TSP_ERR_UNSUPPORTED;
  if (p.B * p.S == 0) return TSP_OK;
  static std::atomic<unsigned long long> configured{0};  // devices set up
  if (needs_setup(configured)) {
    if (cudaFuncSetAttribute(attn_fwd_bf16_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)ATT_SMEM) !=
        cudaSuccess)
      return TSP_ERR_CUDA;
    mark_setup_done(configured);
  }
  const int n_tiles = (int)((p.C + BQ - 1) / BQ);
  dim3 grid(p.rank < 0 ? p.D * n_tiles : n_tiles, p.H, p.B);
  attn_fwd_bf16_kernel<<<grid, ATT_THREADS, ATT_SMEM, stream>>>(p, n_tiles);
  return cudaGetLastError() == cudaSuccess ? TSP_OK : TSP_ERR_CUDA;
}

}  // namespace tsp
