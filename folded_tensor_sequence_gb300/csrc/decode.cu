// One decode step of the TSP layer: B sequences each append one token at
// position `pos` of a key/value cache.
//
// The TSP posts present the scheme for inference as well as training
// (ai-trends.today TSP article, introduction; its 7B reference model is "for
// decoding", "Memory and Processing Results").  Reading used here: the cache
// of the plan's seq positions is sharded over the D virtual ranks by the
// zigzag rule (rank r owns positions of chunks r and 2D-1-r); each rank
// computes a partial softmax (running max, sum, unnormalised output) of the
// new query against its own cached keys, and the partials are merged with
// the log-sum-exp rule -- the reduction the ranks would perform.  The
// projections stream every weight shard once (on one GPU the shard
// broadcast / ring is a loop over the packed weight).
//
// With a handful of tokens per step every projection is a matrix-vector
// product bound by streaming the weights from HBM, and the attention is
// bound by streaming the cache; so these kernels are written for HBM
// bandwidth (16-byte coalesced loads, many loads in flight, grids of many
// CTAs), not for the tensor cores.
#include <cuda_bf16.h>
#include <math.h>

#include "common.cuh"
#include "internal.h"
#include "warp_mma.cuh"

namespace tsp {

namespace {

constexpr int GV_WARPS = 4;   // warps per GEMV CTA
constexpr int DA_THREADS = 256;
constexpr int HD = 128;
constexpr float kLog2e = 1.4426950408889634f;

// Streaming 16-byte load that does not keep the line in L1 (weights and cache
// are read once per step).
__device__ __forceinline__ uint4 ld_stream16(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

__device__ __forceinline__ float bf_lo(uint32_t u) { return __uint_as_float(u << 16); }
__device__ __forceinline__ float bf_hi(uint32_t u) { return __uint_as_float(u & 0xffff0000u); }

__device__ __forceinline__ float dot8(const uint4& a, const uint4& b) {
  float s = bf_lo(a.x) * bf_lo(b.x);
  s = fmaf(bf_hi(a.x), bf_hi(b.x), s);
  s = fmaf(bf_lo(a.y), bf_lo(b.y), s);
  s = fmaf(bf_hi(a.y), bf_hi(b.y), s);
  s = fmaf(bf_lo(a.z), bf_lo(b.z), s);
  s = fmaf(bf_hi(a.z), bf_hi(b.z), s);
  s = fmaf(bf_lo(a.w), bf_lo(b.w), s);
  s = fmaf(bf_hi(a.w), bf_hi(b.w), s);
  return s;
}

__device__ __forceinline__ float silu_f(float z) { return z / (1.0f + __expf(-z)); }

__device__ __forceinline__ float ex2f(float x) {  // 2^x; 2^-inf = 0
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

enum GemvKind : int { GV_RESID = 0, GV_QKV = 1, GV_SWIGLU = 2 };

struct GemvParams {
  const __nv_bfloat16* x;  // [B][K]
  const __nv_bfloat16* w;  // packed weight, rows of K elements
  int B, K;
  int rows;                // weight rows (outputs, or 2F for the gate/up weight)
  __nv_bfloat16* out;      // GV_RESID: [B][rows]; GV_SWIGLU: [B][rows / 2]
  const __nv_bfloat16* resid;
  // GV_QKV: packed columns of shard s are Q (h/D) | K (hk/D) | V (hk/D)
  __nv_bfloat16* q;        // [B][h]
  __nv_bfloat16* kc;       // [B][Hk][S][dh]
  __nv_bfloat16* vc;
  int D, H, Hk, dh, h;
  int64_t S, pos;
};

// out[b][n] = sum_k x[b][k] w[n][k] with an epilogue.  Each warp owns R
// weight rows (for SwiGLU R = 4: two gate rows and the matching two up rows of
// the packed gate/up layout) and streams them once for all B tokens, U
// 256-element chunks of every row in flight per step.  Bytes in flight over
// the whole GPU are about rows x U x 512 B, so small weights take U = 4 and
// one row per warp (more warps) to keep HBM busy.
template <int KIND, int NB, int R, int U>
__global__ void __launch_bounds__(GV_WARPS * 32) gemv_bf16_kernel(const GemvParams p) {
  constexpr int GV_ROWS = R;
  static_assert(KIND != GV_SWIGLU || R == 4, "SwiGLU pairs two gate rows with two up rows");
  const int lane = threadIdx.x & 31;
  const int64_t wg = (int64_t)blockIdx.x * GV_WARPS + (threadIdx.x >> 5);
  int64_t row[GV_ROWS];
  bool valid[GV_ROWS];
  if constexpr (KIND == GV_SWIGLU) {
    const int64_t f0 = wg * 2;  // outputs f0, f0 + 1
    const int64_t blk = f0 / 128, i = f0 % 128;
    row[0] = blk * 256 + i;
    row[1] = row[0] + 1;
    row[2] = row[0] + 128;
    row[3] = row[1] + 128;
    for (int r = 0; r < GV_ROWS; ++r) valid[r] = f0 < p.rows / 2;
  } else {
    for (int r = 0; r < GV_ROWS; ++r) {
      row[r] = wg * GV_ROWS + r;
      valid[r] = row[r] < p.rows;
    }
  }
  if (!valid[0]) return;
  float acc[GV_ROWS][NB];
#pragma unroll
  for (int r = 0; r < GV_ROWS; ++r)
#pragma unroll
    for (int b = 0; b < NB; ++b) acc[r][b] = 0.f;
  const int64_t K = p.K;
  for (int64_t k0 = lane * 8; k0 < K; k0 += 256 * U) {
    uint4 wv[U][GV_ROWS];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      if (k0 + 256 * u >= K) break;
#pragma unroll
      for (int r = 0; r < GV_ROWS; ++r) {
        const int64_t rr = valid[r] ? row[r] : row[0];
        wv[u][r] = ld_stream16(p.w + rr * K + k0 + 256 * u);
      }
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      if (k0 + 256 * u >= K) break;
#pragma unroll
      for (int b = 0; b < NB; ++b) {
        if (b >= p.B) break;
        const uint4 xv = __ldg(reinterpret_cast<const uint4*>(p.x + (int64_t)b * K + k0 + 256 * u));
#pragma unroll
        for (int r = 0; r < GV_ROWS; ++r) acc[r][b] += dot8(wv[u][r], xv);
      }
    }
  }
#pragma unroll
  for (int r = 0; r < GV_ROWS; ++r)
#pragma unroll
    for (int b = 0; b < NB; ++b)
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) acc[r][b] += __shfl_xor_sync(0xffffffffu, acc[r][b], off);
  // every lane now holds every sum; lane r * NB + b writes output (r, b)
#pragma unroll
  for (int r = 0; r < GV_ROWS; ++r) {
#pragma unroll
    for (int b = 0; b < NB; ++b) {
      if (lane != r * NB + b || b >= p.B || !valid[r]) continue;
      const float v = acc[r][b];
      const int64_t n = row[r];
      if constexpr (KIND == GV_RESID) {
        const float res = p.resid ? __bfloat162float(p.resid[(int64_t)b * p.rows + n]) : 0.f;
        p.out[(int64_t)b * p.rows + n] = __float2bfloat16_rn(v + res);
      } else if constexpr (KIND == GV_SWIGLU) {
        if (r < 2) {
          const int64_t f = wg * 2 + r;
          p.out[(int64_t)b * (p.rows / 2) + f] = __float2bfloat16_rn(silu_f(v) * acc[(r + 2) % R][b]);
        }
      } else {  // GV_QKV
        const int hs = p.h / p.D, ks = p.Hk * p.dh / p.D;
        const int s = (int)(n / (hs + 2 * ks));
        const int within = (int)(n - (int64_t)s * (hs + 2 * ks));
        const int which = within < hs ? 0 : (within < hs + ks ? 1 : 2);
        const int cin = within - (which == 0 ? 0 : hs + (which - 1) * ks);
        const int head = s * ((which == 0 ? p.H : p.Hk) / p.D) + cin / p.dh;
        const int d = cin % p.dh;
        const __nv_bfloat16 o = __float2bfloat16_rn(v);
        if (which == 0)
          p.q[(int64_t)b * p.h + head * p.dh + d] = o;
        else
          (which == 1 ? p.kc : p.vc)[(((int64_t)b * p.Hk + head) * p.S + p.pos) * p.dh + d] = o;
      }
    }
  }
}

// The same products on the warp tensor cores, for several tokens: a CTA owns
// 16 weight rows (the MMA's M; for SwiGLU 8 gate rows and their 8 up rows)
// and its GM_KS warps split K; the tokens are the MMA's N (padded to 8).  A
// lane's 16-byte load of 8 consecutive weights of one row feeds two k-steps
// -- the order in which K is summed does not matter as long as the tokens'
// fragments use the same lane -> k mapping -- so every weight byte is loaded
// once, coalesced, and the per-token dot products that bound the scalar
// kernel at B > 1 become MMAs.  Partial sums meet in shared memory.
constexpr int GM_KS = 8;  // warps (K slices) per CTA
constexpr int GM_U = 4;   // 32-element k blocks in flight per warp

template <int KIND>
__global__ void __launch_bounds__(GM_KS * 32) gemv_mma_kernel(const GemvParams p) {
  __shared__ float part[GM_KS][16][9];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, t = lane & 3;
  // the CTA's 16 weight rows; lane g loads rows g and g + 8
  int64_t rows[2];
  int64_t f0 = 0;
  if constexpr (KIND == GV_SWIGLU) {
    f0 = (int64_t)blockIdx.x * 8;  // outputs f0 .. f0 + 7
    const int64_t blk = f0 / 128, i0 = f0 % 128;
    rows[0] = blk * 256 + i0 + g;        // gate
    rows[1] = blk * 256 + 128 + i0 + g;  // up
  } else {
    rows[0] = (int64_t)blockIdx.x * 16 + g;
    rows[1] = rows[0] + 8;
  }
  const int64_t r0 = rows[0] < p.rows ? rows[0] : 0, r1 = rows[1] < p.rows ? rows[1] : 0;
  const int64_t K = p.K, kslice = K / GM_KS;
  const int64_t kb0 = warp * kslice, kb1 = kb0 + kslice;
  const __nv_bfloat16* w0 = p.w + r0 * K + 8 * t;
  const __nv_bfloat16* w1 = p.w + r1 * K + 8 * t;
  const bool tok = g < p.B;
  const __nv_bfloat16* xr = p.x + (int64_t)(tok ? g : 0) * K + 8 * t;
  float c[4] = {0.f, 0.f, 0.f, 0.f};
  for (int64_t kb = kb0; kb < kb1; kb += 32 * GM_U) {
    uint4 a0[GM_U], a1[GM_U], xv[GM_U];
#pragma unroll
    for (int u = 0; u < GM_U; ++u) {
      if (kb + 32 * u < kb1) {
        a0[u] = ld_stream16(w0 + kb + 32 * u);
        a1[u] = ld_stream16(w1 + kb + 32 * u);
        xv[u] = tok ? __ldg(reinterpret_cast<const uint4*>(xr + kb + 32 * u)) : make_uint4(0, 0, 0, 0);
      }
    }
#pragma unroll
    for (int u = 0; u < GM_U; ++u) {
      if (kb + 32 * u < kb1) {
        const uint32_t fa[4] = {a0[u].x, a1[u].x, a0[u].y, a1[u].y};
        wm::mma16816(c, fa, xv[u].x, xv[u].y);
        const uint32_t fb[4] = {a0[u].z, a1[u].z, a0[u].w, a1[u].w};
        wm::mma16816(c, fb, xv[u].z, xv[u].w);
      }
    }
  }
  // c: (row g, token 2t), (row g, token 2t+1), (row g+8, token 2t), (row g+8, token 2t+1)
  part[warp][g][2 * t] = c[0];
  part[warp][g][2 * t + 1] = c[1];
  part[warp][g + 8][2 * t] = c[2];
  part[warp][g + 8][2 * t + 1] = c[3];
  __syncthreads();
  if (threadIdx.x >= 128) return;
  const int r = threadIdx.x / 8, b = threadIdx.x % 8;  // local row, token
  if (b >= p.B) return;
  float v = 0.f;
#pragma unroll
  for (int w = 0; w < GM_KS; ++w) v += part[w][r][b];
  if constexpr (KIND == GV_SWIGLU) {
    if (r >= 8) return;
    float u = 0.f;
#pragma unroll
    for (int w = 0; w < GM_KS; ++w) u += part[w][r + 8][b];
    const int64_t f = f0 + r;
    if (f < p.rows / 2) p.out[(int64_t)b * (p.rows / 2) + f] = __float2bfloat16_rn(silu_f(v) * u);
    return;
  } else {
    const int64_t n = (int64_t)blockIdx.x * 16 + r;
    if (n >= p.rows) return;
    if constexpr (KIND == GV_RESID) {
      const float res = p.resid ? __bfloat162float(p.resid[(int64_t)b * p.rows + n]) : 0.f;
      p.out[(int64_t)b * p.rows + n] = __float2bfloat16_rn(v + res);
    } else {  // GV_QKV
      const int hs = p.h / p.D, ks = p.Hk * p.dh / p.D;
      const int s = (int)(n / (hs + 2 * ks));
      const int within = (int)(n - (int64_t)s * (hs + 2 * ks));
      const int which = within < hs ? 0 : (within < hs + ks ? 1 : 2);
      const int cin = within - (which == 0 ? 0 : hs + (which - 1) * ks);
      const int head = s * ((which == 0 ? p.H : p.Hk) / p.D) + cin / p.dh;
      const int d = cin % p.dh;
      const __nv_bfloat16 o = __float2bfloat16_rn(v);
      if (which == 0)
        p.q[(int64_t)b * p.h + head * p.dh + d] = o;
      else
        (which == 1 ? p.kc : p.vc)[(((int64_t)b * p.Hk + head) * p.S + p.pos) * p.dh + d] = o;
    }
  }
}

struct DecAttnParams {
  const __nv_bfloat16* q;   // [B][h]
  const __nv_bfloat16* kc;  // [B][Hk][S][dh]
  const __nv_bfloat16* vc;
  float* part_o;            // [B][H][P][dh], unnormalised, relative to part_m
  float* part_ml;           // [B][H][P][2]: running max (log2 units) and sum
  int B, H, Hk, D, split;
  int64_t S, C, pos;
};

// Partial attention of the new queries of the G query heads that read K/V
// head blockIdx.y, over piece blockIdx.x % split of rank blockIdx.x / split's
// cached keys (its chunks r and 2D-1-r, positions <= pos).  Half-warps take
// keys in turn (16 lanes x 8 dims per key), keep an online softmax per query
// head, and the CTA merges its 16 half-warp states at the end.  Used for one
// query head per K/V head; with several, the per-key scalar arithmetic
// grows with G and decode_attn_mma_kernel takes over.
template <int G>
__global__ void __launch_bounds__(DA_THREADS) decode_attn_partial_kernel(const DecAttnParams p) {
  extern __shared__ float sm[];  // [16 half-warps][G][HD + 2]
  const int tid = threadIdx.x, hw = tid >> 4, l16 = tid & 15;
  const int kvh = blockIdx.y, b = blockIdx.z;
  const int r = blockIdx.x / p.split, piece = blockIdx.x % p.split;
  const int64_t twoC = 2 * p.C;
  const int64_t k_lo = twoC * piece / p.split, k_hi = twoC * (piece + 1) / p.split;
  const float sl2 = rsqrtf((float)HD) * kLog2e;
  float qv[G][8], o[G][8], m[G], l[G];
#pragma unroll
  for (int j = 0; j < G; ++j) {
    const uint4 u = *reinterpret_cast<const uint4*>(p.q + (int64_t)b * p.H * HD + (kvh * G + j) * HD + l16 * 8);
    qv[j][0] = bf_lo(u.x) * sl2; qv[j][1] = bf_hi(u.x) * sl2;
    qv[j][2] = bf_lo(u.y) * sl2; qv[j][3] = bf_hi(u.y) * sl2;
    qv[j][4] = bf_lo(u.z) * sl2; qv[j][5] = bf_hi(u.z) * sl2;
    qv[j][6] = bf_lo(u.w) * sl2; qv[j][7] = bf_hi(u.w) * sl2;
    m[j] = -INFINITY;
    l[j] = 0.f;
#pragma unroll
    for (int d = 0; d < 8; ++d) o[j][d] = 0.f;
  }
  const __nv_bfloat16* kbase = p.kc + ((int64_t)b * p.Hk + kvh) * p.S * HD + l16 * 8;
  const __nv_bfloat16* vbase = p.vc + ((int64_t)b * p.Hk + kvh) * p.S * HD + l16 * 8;
  auto position = [&](int64_t k) { return k < p.C ? r * p.C + k : (2 * p.D - 1 - r) * p.C + (k - p.C); };
  // Half-warp hw takes keys k_lo + hw + 16 * (U * t + u).  Each warp walks its
  // own block loop from k_lo + 2 * (its warp index), so both halves of a warp
  // always run the same iterations, as the full-warp shuffles need.  Many
  // CTAs per SM (few registers) hide the load latency.
  constexpr int U = 4;
  uint4 kv[U], vv[U];
  bool use[U];
  auto fetch = [&](int64_t kb, uint4 (&kd)[U], uint4 (&vd)[U], bool (&ud)[U]) {
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int64_t k = kb + 16 * u + (hw & 1);
      const int64_t pp = k < k_hi ? position(k) : 0;
      ud[u] = k < k_hi && pp <= p.pos;
      kd[u] = make_uint4(0, 0, 0, 0);
      vd[u] = make_uint4(0, 0, 0, 0);
      if (ud[u]) {
        kd[u] = ld_stream16(kbase + pp * HD);
        vd[u] = ld_stream16(vbase + pp * HD);
      }
    }
  };
  const int64_t kw = k_lo + (hw & ~1);  // this warp's first key
  for (int64_t kb = kw; kb < k_hi; kb += 16 * U) {
    fetch(kb, kv, vv, use);
#pragma unroll
    for (int u = 0; u < U; ++u) {
      // the two half-warps may differ in `use[u]`: the whole warp computes and
      // shuffles, and only lanes whose key is in range update their state
      float kf[8], vf[8];
      kf[0] = bf_lo(kv[u].x); kf[1] = bf_hi(kv[u].x); kf[2] = bf_lo(kv[u].y); kf[3] = bf_hi(kv[u].y);
      kf[4] = bf_lo(kv[u].z); kf[5] = bf_hi(kv[u].z); kf[6] = bf_lo(kv[u].w); kf[7] = bf_hi(kv[u].w);
      vf[0] = bf_lo(vv[u].x); vf[1] = bf_hi(vv[u].x); vf[2] = bf_lo(vv[u].y); vf[3] = bf_hi(vv[u].y);
      vf[4] = bf_lo(vv[u].z); vf[5] = bf_hi(vv[u].z); vf[6] = bf_lo(vv[u].w); vf[7] = bf_hi(vv[u].w);
#pragma unroll
      for (int j = 0; j < G; ++j) {
        float s = 0.f;
#pragma unroll
        for (int d = 0; d < 8; ++d) s = fmaf(qv[j][d], kf[d], s);
        s += __shfl_xor_sync(0xffffffffu, s, 8);
        s += __shfl_xor_sync(0xffffffffu, s, 4);
        s += __shfl_xor_sync(0xffffffffu, s, 2);
        s += __shfl_xor_sync(0xffffffffu, s, 1);
        if (use[u]) {
          const float mn = fmaxf(m[j], s);
          const float corr = ex2f(m[j] - mn), e = ex2f(s - mn);
          m[j] = mn;
          l[j] = l[j] * corr + e;
#pragma unroll
          for (int d = 0; d < 8; ++d) o[j][d] = fmaf(o[j][d], corr, e * vf[d]);
        }
      }
    }
  }
  // CTA merge of the 16 half-warp states
  constexpr int ST = HD + 2;
#pragma unroll
  for (int j = 0; j < G; ++j) {
    float* s = sm + (hw * G + j) * ST;
#pragma unroll
    for (int d = 0; d < 8; ++d) s[l16 * 8 + d] = o[j][d];
    if (l16 == 0) {
      s[HD] = m[j];
      s[HD + 1] = l[j];
    }
  }
  __syncthreads();
  const int P = p.D * p.split;
  for (int idx = tid; idx < G * HD; idx += DA_THREADS) {
    const int j = idx / HD, d = idx % HD;
    float M = -INFINITY;
    for (int w = 0; w < 16; ++w) M = fmaxf(M, sm[(w * G + j) * ST + HD]);
    float L = 0.f, O = 0.f;
    if (M != -INFINITY) {
      for (int w = 0; w < 16; ++w) {
        const float* s = sm + (w * G + j) * ST;
        if (s[HD + 1] == 0.f) continue;
        const float c = exp2f(s[HD] - M);
        L = fmaf(s[HD + 1], c, L);
        O = fmaf(s[d], c, O);
      }
    }
    const int head = kvh * G + j;
    const int64_t slot = ((int64_t)b * p.H + head) * P + blockIdx.x;
    p.part_o[slot * HD + d] = O;
    if (d == 0) {
      p.part_ml[slot * 2] = M;
      p.part_ml[slot * 2 + 1] = L;
    }
  }
}

// Partial attention for G = 2, 4 or 8 query heads per K/V head, on the warp
// tensor cores.  The same split and output as decode_attn_partial_kernel,
// but the G query rows (padded to 16) are multiplied against 16 keys per
// warp and step: S = Q K^T and O += P V with mma.sync m16n8k16 (the score
// accumulators become P's A fragments in registers), K and V arriving in
// 64-key blocks through a 3-stage cp.async ring of swizzled shared-memory
// tiles.  Each warp keeps an online softmax over its 16 keys of every block;
// the CTA merges the four warps at the end.  Still bound by streaming the
// cache: the tensor cores only remove the per-key scalar arithmetic that
// limits the half-warp kernel once several query heads share a key.
constexpr int DM_THREADS = 128;
constexpr int DM_KB = 64;      // keys per block (16 per warp)
constexpr int DM_STAGES = 3;
constexpr size_t DM_STAGE_ELEMS = 2 * (size_t)DM_KB * HD;  // K tile then V tile
constexpr size_t DM_SMEM = DM_STAGES * DM_STAGE_ELEMS * 2;

template <int G>
__global__ void __launch_bounds__(DM_THREADS) decode_attn_mma_kernel(const DecAttnParams p) {
  extern __shared__ __align__(128) uint8_t dm_smem[];
  __nv_bfloat16* tiles = reinterpret_cast<__nv_bfloat16*>(dm_smem);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, t = lane & 3;  // fragment row / column pair
  const int kvh = blockIdx.y, b = blockIdx.z;
  const int r = blockIdx.x / p.split, piece = blockIdx.x % p.split;
  const int64_t twoC = 2 * p.C;
  const int64_t k_lo = twoC * piece / p.split, k_hi = twoC * (piece + 1) / p.split;
  const int nblk = (int)((k_hi - k_lo + DM_KB - 1) / DM_KB);
  const float sl2 = rsqrtf((float)HD) * kLog2e;
  const __nv_bfloat16* kbase = p.kc + ((int64_t)b * p.Hk + kvh) * p.S * HD;
  const __nv_bfloat16* vbase = p.vc + ((int64_t)b * p.Hk + kvh) * p.S * HD;
  auto position = [&](int64_t k) { return k < p.C ? r * p.C + k : (2 * p.D - 1 - r) * p.C + (k - p.C); };
  auto key_ok = [&](int64_t k) { return k < k_hi && position(k) <= p.pos; };

  // K and V rows of block j -> stage j % DM_STAGES (missing rows zero-filled)
  auto load_block = [&](int j) {
    __nv_bfloat16* kt = tiles + (size_t)(j % DM_STAGES) * DM_STAGE_ELEMS;
    __nv_bfloat16* vt = kt + (size_t)DM_KB * HD;
    const uint32_t ks = smem_u32(kt), vs = smem_u32(vt);
    for (int i = tid; i < DM_KB * wm::CHUNKS; i += DM_THREADS) {
      const int row = i / wm::CHUNKS, c = i % wm::CHUNKS;
      const int64_t k = k_lo + (int64_t)j * DM_KB + row;
      const bool ok = key_ok(k);
      const int64_t off = ok ? position(k) * HD + c * 8 : 0;
      wm::cp_async16(ks + wm::swz(row, c * 8) * 2, kbase + off, ok);
      wm::cp_async16(vs + wm::swz(row, c * 8) * 2, vbase + off, ok);
    }
  };

  // Q rows g < G as A fragments (rows 8..15 and G..7 are zero)
  uint32_t qa[HD / 16][2];
  {
    const uint32_t* qrow =
        reinterpret_cast<const uint32_t*>(p.q + ((int64_t)b * p.H + (int64_t)kvh * G + (g < G ? g : 0)) * HD);
#pragma unroll
    for (int kk = 0; kk < HD / 16; ++kk) {
      qa[kk][0] = g < G ? qrow[(16 * kk + 2 * t) / 2] : 0u;
      qa[kk][1] = g < G ? qrow[(16 * kk + 8 + 2 * t) / 2] : 0u;
    }
  }
  float o[HD / 8][2];  // row g, head dims 8*dt + 2t, +1
#pragma unroll
  for (int dt = 0; dt < HD / 8; ++dt) o[dt][0] = o[dt][1] = 0.f;
  float m_run = -INFINITY, l_part = 0.f;  // l_part: this thread's columns only

  for (int j = 0; j < DM_STAGES - 1 && j < nblk; ++j) {
    load_block(j);
    wm::cp_commit();
  }
  for (int j = 0; j < nblk; ++j) {
    if (j + 1 < nblk)
      asm volatile("cp.async.wait_group 1;" ::: "memory");
    else
      wm::cp_wait_all();
    __syncthreads();  // block j landed for every thread; stage (j + 2) % 3 is free
    if (j + DM_STAGES - 1 < nblk) {
      load_block(j + DM_STAGES - 1);
      wm::cp_commit();
    }
    const __nv_bfloat16* kt = tiles + (size_t)(j % DM_STAGES) * DM_STAGE_ELEMS;
    const __nv_bfloat16* vt = kt + (size_t)DM_KB * HD;
    const uint32_t ks = smem_u32(kt), vs = smem_u32(vt);
    // S = Q K^T for this warp's keys 16*warp .. +15 (two n-tiles of 8)
    float s[2][4];
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
      s[nt][0] = s[nt][1] = s[nt][2] = s[nt][3] = 0.f;
      const int krow = 16 * warp + 8 * nt + (lane & 7);
#pragma unroll
      for (int kp = 0; kp < HD / 32; ++kp) {  // pairs of 16-wide k steps
        uint32_t b0, b1, b2, b3;
        wm::ldsm_x4(ks + wm::swz(krow, (4 * kp + (lane >> 3)) * 8) * 2, b0, b1, b2, b3);
        const uint32_t a0[4] = {qa[2 * kp][0], 0u, qa[2 * kp][1], 0u};
        const uint32_t a1[4] = {qa[2 * kp + 1][0], 0u, qa[2 * kp + 1][1], 0u};
        wm::mma16816(s[nt], a0, b0, b1);
        wm::mma16816(s[nt], a1, b2, b3);
      }
    }
    // online softmax of row g over the 16 keys (c0, c1 of each n-tile; rows g + 8 are padding)
    const int64_t kbase_blk = k_lo + (int64_t)j * DM_KB + 16 * warp;
    float x[4];
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int64_t k = kbase_blk + 8 * nt + 2 * t + e;
        x[2 * nt + e] = key_ok(k) ? s[nt][e] * sl2 : -INFINITY;
      }
    float mb = fmaxf(fmaxf(x[0], x[1]), fmaxf(x[2], x[3]));
    mb = fmaxf(mb, __shfl_xor_sync(0xffffffffu, mb, 1));
    mb = fmaxf(mb, __shfl_xor_sync(0xffffffffu, mb, 2));
    const float m_new = fmaxf(m_run, mb);
    if (m_new == -INFINITY) continue;  // nothing visible yet in this warp's keys (uniform per row group)
    const float corr = ex2f(m_run - m_new);
    m_run = m_new;
    float pv[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) pv[i] = ex2f(x[i] - m_new);
    l_part = l_part * corr + (pv[0] + pv[1]) + (pv[2] + pv[3]);
#pragma unroll
    for (int dt = 0; dt < HD / 8; ++dt) {
      o[dt][0] *= corr;
      o[dt][1] *= corr;
    }
    const uint32_t pa[4] = {pack_bf16x2(pv[0], pv[1]), 0u, pack_bf16x2(pv[2], pv[3]), 0u};
    // O += P V: V rows = this warp's keys, two head-dim n-tiles per ldmatrix
    const int vrow = 16 * warp + ((lane >> 3) & 1) * 8 + (lane & 7);
#pragma unroll
    for (int dp = 0; dp < HD / 16; ++dp) {
      uint32_t b0, b1, b2, b3;
      wm::ldsm_x4_t(vs + wm::swz(vrow, (2 * dp + (lane >> 4)) * 8) * 2, b0, b1, b2, b3);
      float acc0[4] = {o[2 * dp][0], o[2 * dp][1], 0.f, 0.f};
      float acc1[4] = {o[2 * dp + 1][0], o[2 * dp + 1][1], 0.f, 0.f};
      wm::mma16816(acc0, pa, b0, b1);
      wm::mma16816(acc1, pa, b2, b3);
      o[2 * dp][0] = acc0[0];
      o[2 * dp][1] = acc0[1];
      o[2 * dp + 1][0] = acc1[0];
      o[2 * dp + 1][1] = acc1[1];
    }
  }
  // row sums over the four lanes of a row, then the CTA merge of the four warps
  float l_row = l_part + __shfl_xor_sync(0xffffffffu, l_part, 1);
  l_row += __shfl_xor_sync(0xffffffffu, l_row, 2);
  __syncthreads();  // every warp is done with the stage tiles
  constexpr int ST = HD + 2;
  float* ms = reinterpret_cast<float*>(dm_smem);  // [4 warps][G][ST]
  if (g < G) {
    float* row = ms + (warp * G + g) * ST;
#pragma unroll
    for (int dt = 0; dt < HD / 8; ++dt) {
      row[8 * dt + 2 * t] = o[dt][0];
      row[8 * dt + 2 * t + 1] = o[dt][1];
    }
    if (t == 0) {
      row[HD] = m_run;
      row[HD + 1] = l_row;
    }
  }
  __syncthreads();
  const int P = p.D * p.split;
  for (int idx = tid; idx < G * HD; idx += DM_THREADS) {
    const int jh = idx / HD, d = idx % HD;
    float M = -INFINITY;
    for (int w = 0; w < 4; ++w) M = fmaxf(M, ms[(w * G + jh) * ST + HD]);
    float L = 0.f, O = 0.f;
    if (M != -INFINITY) {
      for (int w = 0; w < 4; ++w) {
        const float* row = ms + (w * G + jh) * ST;
        if (row[HD + 1] == 0.f) continue;
        const float c = exp2f(row[HD] - M);
        L = fmaf(row[HD + 1], c, L);
        O = fmaf(row[d], c, O);
      }
    }
    const int64_t slot = ((int64_t)b * p.H + (int64_t)kvh * G + jh) * P + blockIdx.x;
    p.part_o[slot * HD + d] = O;
    if (d == 0) {
      p.part_ml[slot * 2] = M;
      p.part_ml[slot * 2 + 1] = L;
    }
  }
}

// out[b][head*dh + d] = merge of the P partial softmax results (log-sum-exp rule).
__global__ void decode_attn_combine_kernel(const float* __restrict__ part_o, const float* __restrict__ part_ml,
                                           __nv_bfloat16* __restrict__ out, int H, int P) {
  const int head = blockIdx.x, b = blockIdx.y, d = threadIdx.x;
  const int64_t base = ((int64_t)b * H + head) * P;
  float M = -INFINITY;
  for (int i = 0; i < P; ++i)
    if (part_ml[(base + i) * 2 + 1] > 0.f) M = fmaxf(M, part_ml[(base + i) * 2]);
  float L = 0.f, O = 0.f;
  for (int i = 0; i < P; ++i) {
    const float li = part_ml[(base + i) * 2 + 1];
    if (li == 0.f) continue;
    const float c = exp2f(part_ml[(base + i) * 2] - M);
    L = fmaf(li, c, L);
    O = fmaf(part_o[(base + i) * HD + d], c, O);
  }
  out[((int64_t)b * H + head) * HD + d] = __float2bfloat16_rn(O / L);
}

template <int KIND, int R, int U>
cudaError_t launch_gemv_ru(const GemvParams& p, cudaStream_t st) {
  const int64_t warps = KIND == GV_SWIGLU ? (p.rows / 2 + 1) / 2 : (p.rows + R - 1) / R;
  const unsigned grid = (unsigned)((warps + GV_WARPS - 1) / GV_WARPS);
  switch (p.B) {
    case 1: gemv_bf16_kernel<KIND, 1, R, U><<<grid, GV_WARPS * 32, 0, st>>>(p); break;
    case 2: gemv_bf16_kernel<KIND, 2, R, U><<<grid, GV_WARPS * 32, 0, st>>>(p); break;
    case 3:
    case 4: gemv_bf16_kernel<KIND, 4, R, U><<<grid, GV_WARPS * 32, 0, st>>>(p); break;
    default: gemv_bf16_kernel<KIND, 8, R, U><<<grid, GV_WARPS * 32, 0, st>>>(p); break;
  }
  return cudaGetLastError();
}

template <int KIND>
cudaError_t launch_gemv(const GemvParams& p, cudaStream_t st) {
  // Tensor-core GEMV (16 weight rows per CTA, K split over its warps), except
  // for the single-token gate/up product, which the scalar kernel already
  // streams at HBM speed (measured: 39 against 43 us at h = 4096).
  if (p.K % (32 * GM_KS) == 0 && (p.B > 1 || KIND != GV_SWIGLU)) {
    const int64_t ctas = KIND == GV_SWIGLU ? (p.rows / 2 + 7) / 8 : (p.rows + 15) / 16;
    gemv_mma_kernel<KIND><<<(unsigned)ctas, GM_KS * 32, 0, st>>>(p);
    return cudaGetLastError();
  }
  if constexpr (KIND == GV_SWIGLU)
    return launch_gemv_ru<KIND, 4, 2>(p, st);
  else
    return launch_gemv_ru<KIND, 1, 4>(p, st);
}

}  // namespace

int decode_split(int D, int H, int Hk, int B, int64_t C) {
  const int64_t base = (int64_t)D * Hk * B;  // CTAs per piece of every rank
  const int64_t max_split = (2 * C) / 64 > 0 ? (2 * C) / 64 : 1;  // pieces of >= 64 keys
  if (H / Hk == 1) {
    // half-warp kernel: enough CTAs to keep every SM streaming (about 4 per SM)
    const int64_t target = 4LL * num_sms();
    int64_t split = (target + base - 1) / base;
    if (split > max_split) split = max_split;
    return split < 1 ? 1 : (int)split;
  }
  // tensor-core kernel: two CTAs per SM and equal pieces, so whole waves
  // matter; take the smallest split that fills one wave and leaves the last
  // wave at least 95 % full (else the fullest within eight times that)
  const int64_t slots = 2LL * num_sms();
  int64_t first = (slots + base - 1) / base;
  if (first > max_split) first = max_split;
  if (first < 1) first = 1;
  int64_t best = first;
  double best_eff = 0.0;
  for (int64_t split = first; split <= max_split && split <= 8 * first; ++split) {
    const int64_t n = base * split;
    const int64_t waves = (n + slots - 1) / slots;
    const double eff = (double)n / (double)(waves * slots);
    if (eff >= 0.95) return (int)split;
    if (eff > best_eff) {
      best_eff = eff;
      best = split;
    }
  }
  return (int)best;
}

size_t decode_ws_bytes(const tsp_plan* p, int batch) {
  const size_t B = batch, h = p->hidden, F = p->ffn, H = p->heads;
  const size_t P = (size_t)p->D * decode_split(p->D, p->heads, p->kv_heads, batch, p->chunk);
  auto a = [](size_t x) { return (x + 255) & ~size_t(255); };
  return a(B * h * 2) * 3 + a(B * F * 2) + a(B * H * P * HD * 4) + a(B * H * P * 2 * 4);
}

tsp_status decode_step_bf16(const tsp_plan* pl, int batch, int64_t pos, const void* x_new, const tsp_weights* w,
                            void* k_cache, void* v_cache, void* y_new, void* ws, cudaStream_t st) {
  const int B = batch, h = pl->hidden, F = pl->ffn, H = pl->heads, Hk = pl->kv_heads, D = pl->D;
  const int hk = Hk * pl->head_dim;
  const int split = decode_split(D, H, Hk, B, pl->chunk);
  const int P = D * split;
  auto a = [](size_t x) { return (x + 255) & ~size_t(255); };
  char* base = static_cast<char*>(ws);
  __nv_bfloat16* q = reinterpret_cast<__nv_bfloat16*>(base);
  __nv_bfloat16* o = reinterpret_cast<__nv_bfloat16*>(base + a((size_t)B * h * 2));
  __nv_bfloat16* hb = reinterpret_cast<__nv_bfloat16*>(base + 2 * a((size_t)B * h * 2));
  __nv_bfloat16* mb = reinterpret_cast<__nv_bfloat16*>(base + 3 * a((size_t)B * h * 2));
  float* part_o = reinterpret_cast<float*>(base + 3 * a((size_t)B * h * 2) + a((size_t)B * F * 2));
  float* part_ml = reinterpret_cast<float*>(reinterpret_cast<char*>(part_o) + a((size_t)B * H * P * HD * 4));
  cudaError_t e;
  // 1. Q/K/V of the new tokens; K and V land in the cache at `pos`
  GemvParams g{};
  g.x = static_cast<const __nv_bfloat16*>(x_new);
  g.w = static_cast<const __nv_bfloat16*>(w->qkv);
  g.B = B;
  g.K = h;
  g.rows = h + 2 * hk;
  g.q = q;
  g.kc = static_cast<__nv_bfloat16*>(k_cache);
  g.vc = static_cast<__nv_bfloat16*>(v_cache);
  g.D = D;
  g.H = H;
  g.Hk = Hk;
  g.dh = pl->head_dim;
  g.h = h;
  g.S = pl->seq;
  g.pos = pos;
  prof_begin("decode QKV projection", st);
  e = launch_gemv<GV_QKV>(g, st);
  prof_end(st);
  if (e != cudaSuccess) return TSP_ERR_CUDA;
  // 2. per-rank partial attention over the zigzag-sharded cache, then the merge
  DecAttnParams ap;
  ap.q = q;
  ap.kc = g.kc;
  ap.vc = g.vc;
  ap.part_o = part_o;
  ap.part_ml = part_ml;
  ap.B = B;
  ap.H = H;
  ap.Hk = Hk;
  ap.D = D;
  ap.split = split;
  ap.S = pl->seq;
  ap.C = pl->chunk;
  ap.pos = pos;
  const int G = H / Hk;
  const dim3 grid(P, Hk, B);
  prof_begin("decode attention", st);
  if (G == 1) {
    decode_attn_partial_kernel<1><<<grid, DA_THREADS, (size_t)16 * (HD + 2) * 4, st>>>(ap);
  } else if (G == 2 || G == 4 || G == 8) {
    // several query heads per cached key: tensor-core partials
    static std::atomic<unsigned long long> configured{0};  // devices set up
    if (needs_setup(configured)) {
      if (cudaFuncSetAttribute(decode_attn_mma_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               (int)DM_SMEM) != cudaSuccess ||
          cudaFuncSetAttribute(decode_attn_mma_kernel<4>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               (int)DM_SMEM) != cudaSuccess ||
          cudaFuncSetAttribute(decode_attn_mma_kernel<8>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               (int)DM_SMEM) != cudaSuccess) {
        prof_end(st);
        return TSP_ERR_CUDA;
      }
      mark_setup_done(configured);
    }
    if (G == 2)
      decode_attn_mma_kernel<2><<<grid, DM_THREADS, DM_SMEM, st>>>(ap);
    else if (G == 4)
      decode_attn_mma_kernel<4><<<grid, DM_THREADS, DM_SMEM, st>>>(ap);
    else
      decode_attn_mma_kernel<8><<<grid, DM_THREADS, DM_SMEM, st>>>(ap);
  } else {
    prof_end(st);
    return TSP_ERR_UNSUPPORTED;
  }
  e = cudaGetLastError();
  if (e == cudaSuccess) {
    decode_attn_combine_kernel<<<dim3(H, B), HD, 0, st>>>(part_o, part_ml, o, H, P);
    e = cudaGetLastError();
  }
  prof_end(st);
  if (e != cudaSuccess) return TSP_ERR_CUDA;
  // 3. H = x + O Wo
  GemvParams go{};
  go.x = o;
  go.w = static_cast<const __nv_bfloat16*>(w->o);
  go.B = B;
  go.K = h;
  go.rows = h;
  go.out = hb;
  go.resid = static_cast<const __nv_bfloat16*>(x_new);
  prof_begin("decode output projection", st);
  e = launch_gemv<GV_RESID>(go, st);
  prof_end(st);
  if (e != cudaSuccess) return TSP_ERR_CUDA;
  // 4. M = SiLU(H Wg) * (H Wu)
  GemvParams gg{};
  gg.x = hb;
  gg.w = static_cast<const __nv_bfloat16*>(w->gate_up);
  gg.B = B;
  gg.K = h;
  gg.rows = 2 * F;
  gg.out = mb;
  prof_begin("decode gate/up projection", st);
  e = launch_gemv<GV_SWIGLU>(gg, st);
  prof_end(st);
  if (e != cudaSuccess) return TSP_ERR_CUDA;
  // 5. y = H + M Wd
  GemvParams gd{};
  gd.x = mb;
  gd.w = static_cast<const __nv_bfloat16*>(w->down);
  gd.B = B;
  gd.K = F;
  gd.rows = h;
  gd.out = static_cast<__nv_bfloat16*>(y_new);
  gd.resid = hb;
  prof_begin("decode down projection", st);
  e = launch_gemv<GV_RESID>(gd, st);
  prof_end(st);
  return e == cudaSuccess ? TSP_OK : TSP_ERR_CUDA;
}

}  // namespace tsp
