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

namespace tsp {

namespace {

constexpr int GV_WARPS = 4;   // warps per GEMV CTA
constexpr int GV_ROWS = 4;    // weight rows per warp
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

// out[b][n] = sum_k x[b][k] w[n][k] with an epilogue.  Each warp owns four
// weight rows (for SwiGLU: two gate rows and the matching two up rows of the
// packed gate/up layout) and streams them once for all B tokens.
template <int KIND, int NB>
__global__ void __launch_bounds__(GV_WARPS * 32) gemv_bf16_kernel(const GemvParams p) {
  const int lane = threadIdx.x & 31;
  const int64_t wg = (int64_t)blockIdx.x * GV_WARPS + (threadIdx.x >> 5);
  int64_t row[GV_ROWS];
  bool valid[GV_ROWS];
  if (KIND == GV_SWIGLU) {
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
  for (int64_t k0 = lane * 8; k0 < K; k0 += 512) {
    uint4 wv[2][GV_ROWS];
    const bool second = k0 + 256 < K;
#pragma unroll
    for (int r = 0; r < GV_ROWS; ++r) {
      const int64_t rr = valid[r] ? row[r] : row[0];
      wv[0][r] = ld_stream16(p.w + rr * K + k0);
      if (second) wv[1][r] = ld_stream16(p.w + rr * K + k0 + 256);
    }
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      if (u == 1 && !second) break;
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
      if (KIND == GV_RESID) {
        const float res = p.resid ? __bfloat162float(p.resid[(int64_t)b * p.rows + n]) : 0.f;
        p.out[(int64_t)b * p.rows + n] = __float2bfloat16_rn(v + res);
      } else if (KIND == GV_SWIGLU) {
        if (r < 2) {
          const int64_t f = wg * 2 + r;
          p.out[(int64_t)b * (p.rows / 2) + f] = __float2bfloat16_rn(silu_f(v) * acc[r + 2][b]);
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
// head, and the CTA merges its 16 half-warp states at the end.
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
  // always run the same iterations, as the full-warp shuffles need.  With several query
  // heads per key (G >= 4) the per-key arithmetic is long enough that the
  // next block's loads are issued before the current block is consumed; with
  // one or two, more CTAs per SM (fewer registers) hide the latency better.
  constexpr int U = G >= 4 ? 2 : 4;
  constexpr bool kPrefetch = G >= 4;
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
  if (kPrefetch) fetch(kw, kv, vv, use);
  for (int64_t kb = kw; kb < k_hi; kb += 16 * U) {
    uint4 kn[U], vn[U];
    bool un[U];
    if (kPrefetch)
      fetch(kb + 16 * U, kn, vn, un);
    else
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
    if (kPrefetch) {
#pragma unroll
      for (int u = 0; u < U; ++u) {
        kv[u] = kn[u];
        vv[u] = vn[u];
        use[u] = un[u];
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

template <int KIND>
cudaError_t launch_gemv(const GemvParams& p, cudaStream_t st) {
  const int64_t warps = KIND == GV_SWIGLU ? (p.rows / 2 + 1) / 2 : (p.rows + GV_ROWS - 1) / GV_ROWS;
  const unsigned grid = (unsigned)((warps + GV_WARPS - 1) / GV_WARPS);
  switch (p.B) {
    case 1: gemv_bf16_kernel<KIND, 1><<<grid, GV_WARPS * 32, 0, st>>>(p); break;
    case 2: gemv_bf16_kernel<KIND, 2><<<grid, GV_WARPS * 32, 0, st>>>(p); break;
    case 3:
    case 4: gemv_bf16_kernel<KIND, 4><<<grid, GV_WARPS * 32, 0, st>>>(p); break;
    default: gemv_bf16_kernel<KIND, 8><<<grid, GV_WARPS * 32, 0, st>>>(p); break;
  }
  return cudaGetLastError();
}

}  // namespace

int decode_split(int D, int Hk, int B, int64_t C) {
  // enough CTAs to keep every SM streaming (about 4 per SM), pieces of >= 64 keys
  const int64_t target = 4LL * num_sms();
  int64_t split = (target + (int64_t)D * Hk * B - 1) / ((int64_t)D * Hk * B);
  const int64_t max_split = (2 * C) / 64 > 0 ? (2 * C) / 64 : 1;
  if (split > max_split) split = max_split;
  return split < 1 ? 1 : (int)split;
}

size_t decode_ws_bytes(const tsp_plan* p, int batch) {
  const size_t B = batch, h = p->hidden, F = p->ffn, H = p->heads;
  const size_t P = (size_t)p->D * decode_split(p->D, p->kv_heads, batch, p->chunk);
  auto a = [](size_t x) { return (x + 255) & ~size_t(255); };
  return a(B * h * 2) * 3 + a(B * F * 2) + a(B * H * P * HD * 4) + a(B * H * P * 2 * 4);
}

tsp_status decode_step_bf16(const tsp_plan* pl, int batch, int64_t pos, const void* x_new, const tsp_weights* w,
                            void* k_cache, void* v_cache, void* y_new, void* ws, cudaStream_t st) {
  const int B = batch, h = pl->hidden, F = pl->ffn, H = pl->heads, Hk = pl->kv_heads, D = pl->D;
  const int hk = Hk * pl->head_dim;
  const int split = decode_split(D, Hk, B, pl->chunk);
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
  const size_t smem = (size_t)16 * G * (HD + 2) * 4;
  prof_begin("decode attention", st);
  switch (G) {
    case 1: decode_attn_partial_kernel<1><<<grid, DA_THREADS, smem, st>>>(ap); break;
    case 2: decode_attn_partial_kernel<2><<<grid, DA_THREADS, smem, st>>>(ap); break;
    case 4: decode_attn_partial_kernel<4><<<grid, DA_THREADS, smem, st>>>(ap); break;
    case 8: {
      static std::atomic<unsigned long long> configured{0};  // devices set up
      if (needs_setup(configured)) {
        if (cudaFuncSetAttribute(decode_attn_partial_kernel<8>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)((size_t)16 * 8 * (HD + 2) * 4)) != cudaSuccess) {
          prof_end(st);
          return TSP_ERR_CUDA;
        }
        mark_setup_done(configured);
      }
      decode_attn_partial_kernel<8><<<grid, DA_THREADS, smem, st>>>(ap);
      break;
    }
    default: prof_end(st); return TSP_ERR_UNSUPPORTED;
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
