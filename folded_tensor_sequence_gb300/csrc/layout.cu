// Memory-bound layout kernels: zigzag token permutation, the K/V all-gather
// into natural order, weight packing, transposes and small elementwise steps.
//
// Zigzag partition (ai-trends.today TSP article, "How to Fold a Book": K/V
// are reordered with a zigzag scheme so causal attention work is balanced):
// the sequence is cut into 2D chunks of C tokens; virtual rank r holds chunk r
// then chunk 2D-1-r.  Zigzag row (r*B + b)*2C + k holds natural position
// pos(r,k) = r*C + k (k < C) or (2D-1-r)*C + (k-C) (k >= C).
//
// All copies move 16-byte vectors, consecutive threads touching consecutive
// vectors, over a grid of at most (SM count x 8) CTAs striding the work.
#include "common.cuh"
#include "internal.h"

namespace tsp {

namespace {

__device__ __forceinline__ int64_t zigzag_pos(int64_t r, int64_t k, int64_t C, int D) {
  return k < C ? r * C + k : (2 * D - 1 - r) * C + (k - C);
}

// Vectors each thread keeps in flight in the copy kernels below (loads issued
// back to back, then the stores): 2048 threads x 4 x 16 B = 128 KB per SM,
// well above what HBM latency times bandwidth per SM asks for.
constexpr int kCopyUnroll = 4;
constexpr int kCopyThreads = 256;

// Copies `nvec` 16-byte vectors src[i] -> dst[i], i in [first, nvec), the
// calling CTA taking every `stride`-th group of kCopyThreads*kCopyUnroll.
__device__ __forceinline__ void copy_span(const uint4* __restrict__ src, uint4* __restrict__ dst, int64_t nvec,
                                          int64_t first, int64_t stride) {
  for (int64_t v0 = first + threadIdx.x; v0 < nvec; v0 += stride) {
    uint4 t[kCopyUnroll];
#pragma unroll
    for (int u = 0; u < kCopyUnroll; ++u) {
      const int64_t i = v0 + (int64_t)u * kCopyThreads;
      if (i < nvec) t[u] = __ldcs(src + i);
    }
#pragma unroll
    for (int u = 0; u < kCopyUnroll; ++u) {
      const int64_t i = v0 + (int64_t)u * kCopyThreads;
      if (i < nvec) __stcs(dst + i, t[u]);
    }
  }
}

// Zigzag permute / unpermute.  Each of the 2*D*B chunk copies is contiguous on
// both sides: half e of rank r's rows of sequence b (C zigzag rows from
// (r*B + b)*2C + e*C) is natural chunk c = r (e = 0) or 2D-1-r (e = 1) of that
// sequence (C rows from b*S + c*C).  Work item w = (chunk copy, part): `parts`
// CTAs share one chunk copy, so the grid needs no per-vector index arithmetic.
__global__ void __launch_bounds__(kCopyThreads) zigzag_rows_kernel(const uint4* __restrict__ src,
                                                                   uint4* __restrict__ dst, int64_t vecs_per_row,
                                                                   int D, int B, int64_t S, int parts,
                                                                   bool to_zigzag) {
  const int64_t C = S / (2 * D);
  const int64_t seg_vecs = C * vecs_per_row;
  const int items = 2 * D * B * parts;
  for (int w = blockIdx.x; w < items; w += gridDim.x) {
    const int seg = w / parts, part = w - seg * parts;
    const int e = seg & 1, rb = seg >> 1;  // rb = r*B + b
    const int r = rb / B, b = rb - r * B;
    const int64_t c = e == 0 ? r : 2 * D - 1 - r;
    const int64_t zrow0 = (int64_t)rb * 2 * C + e * C;
    const int64_t nrow0 = (int64_t)b * S + c * C;
    const uint4* s0 = src + (to_zigzag ? nrow0 : zrow0) * vecs_per_row;
    uint4* d0 = dst + (to_zigzag ? zrow0 : nrow0) * vecs_per_row;
    copy_span(s0, d0, seg_vecs, (int64_t)part * kCopyThreads * kCopyUnroll,
              (int64_t)parts * kCopyThreads * kCopyUnroll);
  }
}

// K/V all-gather into natural order: gathered [B][Hk][S][dh] <- zigzag
// [T][Hk*dh] (source rows `vec_per_row` vectors apart).  Work item = (tensor
// K or V, sequence b, K/V head, chunk c): natural positions c*C .. c*C+C-1 of
// that head are C consecutive rows of dh*e bytes in the destination, read
// from C consecutive zigzag rows of rank r(c) at the head's column offset.
// vph = vectors per head row, a power of two (dh * elem_bytes / 16 with dh in
// {32, 64, 128}).
__global__ void __launch_bounds__(kCopyThreads) kv_gather_kernel(const uint4* __restrict__ kz,
                                                                 const uint4* __restrict__ vz, uint4* __restrict__ k,
                                                                 uint4* __restrict__ v, int lg_vph, int D, int B,
                                                                 int64_t S, int H, int64_t vec_per_row, int ntens) {
  const int64_t C = S / (2 * D);
  const int vph = 1 << lg_vph;
  const int64_t seg_vecs = C << lg_vph;
  const int64_t items = (int64_t)ntens * B * H * 2 * D;  // ntens 1: K only
  for (int64_t w = blockIdx.x; w < items; w += gridDim.x) {
    const int c = (int)(w % (2 * D));
    int64_t rest = w / (2 * D);
    const int head = (int)(rest % H);
    rest /= H;
    const int b = (int)(rest % B);
    const int tensor = (int)(rest / B);
    const int64_t r = c < D ? c : 2 * D - 1 - c;
    const int64_t zrow0 = (r * B + b) * 2 * C + (c < D ? 0 : C);
    const uint4* src = (tensor == 0 ? kz : vz) + zrow0 * vec_per_row + (int64_t)head * vph;
    uint4* dst = (tensor == 0 ? k : v) + (((int64_t)b * H + head) * S + (int64_t)c * C) * vph;
    for (int64_t v0 = threadIdx.x; v0 < seg_vecs; v0 += kCopyThreads * kCopyUnroll) {
      uint4 t[kCopyUnroll];
#pragma unroll
      for (int u = 0; u < kCopyUnroll; ++u) {
        const int64_t i = v0 + u * kCopyThreads;
        if (i < seg_vecs) t[u] = __ldcs(src + (i >> lg_vph) * vec_per_row + (i & (vph - 1)));
      }
#pragma unroll
      for (int u = 0; u < kCopyUnroll; ++u) {
        const int64_t i = v0 + u * kCopyThreads;
        if (i < seg_vecs) __stcs(dst + i, t[u]);
      }
    }
  }
}

// 2-D copy: `rows` rows of `row_vecs` 16-byte vectors, source rows
// `src_pitch` vectors apart, destination rows `dst_pitch` vectors apart.
__global__ void __launch_bounds__(kCopyThreads) copy_rows_kernel(const uint4* __restrict__ src, int64_t src_pitch,
                                                                 uint4* __restrict__ dst, int64_t dst_pitch,
                                                                 int64_t rows, int64_t row_vecs) {
  const int64_t total = rows * row_vecs;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t r = i / row_vecs, c = i - r * row_vecs;
    dst[r * dst_pitch + c] = __ldg(&src[r * src_pitch + c]);
  }
}

// V of the all-gathered rows straight into the transposed natural layout the
// tcgen05 attention reads: vt [B][H][dh][S] <- src zigzag rows [T][ld] (V of
// head e in columns v_col0 + e*dh ..).  One CTA per 64 positions x 64 head
// dims: the 64 positions lie in one chunk (C % 64 == 0), i.e. 64 consecutive
// zigzag rows of one rank; through a 64 x 64 shared tile whose 16-byte chunk c
// of row r sits at c ^ ((r / 8) % 8), as in transpose_b16_kernel.
__global__ void __launch_bounds__(256) kv_gather_vt_kernel(const uint16_t* __restrict__ src, int64_t ld,
                                                           int64_t v_col0, uint16_t* __restrict__ vt, int D, int B,
                                                           int64_t S, int H, int dh) {
  __shared__ __align__(16) uint16_t tile[64 * 64];
  const int64_t C = S / (2 * D);
  const int64_t ptiles = S / 64, dtiles = dh / 64;
  const int64_t ntiles = (int64_t)B * H * ptiles * dtiles;
  for (int64_t t = blockIdx.x; t < ntiles; t += gridDim.x) {
    const int64_t dt = t % dtiles;
    int64_t rest = t / dtiles;
    const int64_t pt = rest % ptiles;
    rest /= ptiles;
    const int head = (int)(rest % H);
    const int b = (int)(rest / H);
    const int64_t p0 = pt * 64, d0 = dt * 64;
    const int64_t c = p0 / C, off = p0 - c * C;
    const int64_t r = c < D ? c : 2 * D - 1 - c;
    const int64_t zrow0 = (r * B + b) * 2 * C + (c < D ? 0 : C) + off;
    const uint16_t* s0 = src + zrow0 * ld + v_col0 + (int64_t)head * dh + d0;
#pragma unroll
    for (int it = 0; it < 2; ++it) {
      const int idx = threadIdx.x + it * 256;  // 64 positions x 8 chunks of 8 dims
      const int rr = idx / 8, cv = idx % 8;
      const uint4 val = __ldg(reinterpret_cast<const uint4*>(s0 + (int64_t)rr * ld + cv * 8));
      *reinterpret_cast<uint4*>(&tile[rr * 64 + ((cv ^ ((rr / 8) & 7)) * 8)]) = val;
    }
    __syncthreads();
    uint16_t* d0p = vt + (((int64_t)b * H + head) * dh + d0) * S + p0;
#pragma unroll
    for (int it = 0; it < 2; ++it) {
      const int idx = threadIdx.x + it * 256;  // 64 dims x 8 chunks of 8 positions
      const int cc = idx / 8, rv = idx % 8;    // head dim d0 + cc, positions rv*8 .. rv*8+7
      const int pos = (((cc / 8) ^ rv) * 8) + (cc % 8);
      uint16_t e[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) e[k] = tile[(rv * 8 + k) * 64 + pos];
      uint4 val;
      val.x = e[0] | (uint32_t(e[1]) << 16);
      val.y = e[2] | (uint32_t(e[3]) << 16);
      val.z = e[4] | (uint32_t(e[5]) << 16);
      val.w = e[6] | (uint32_t(e[7]) << 16);
      *reinterpret_cast<uint4*>(d0p + (int64_t)cc * S + rv * 8) = val;
    }
    __syncthreads();
  }
}

// dqkv [T][h + 2hk] in packed column order <- dq zigzag [T][h], dk/dv gathered
// [B][Hk][S][dh] (hk = Hk*dh; a shard's columns are Q h/D | K hk/D | V hk/D).
// One CTA per zigzag row: the row's (rank, batch, position) is decoded once.
__global__ void assemble_dqkv_kernel(const uint4* __restrict__ dq, const uint4* __restrict__ dk,
                                     const uint4* __restrict__ dv, uint4* __restrict__ out, int vec_per_head, int D,
                                     int B, int64_t S, int H, int Hk) {
  const int64_t C = S / (2 * D);
  const int64_t twoC = 2 * C;
  const int64_t zrow = blockIdx.x;
  const int64_t r = zrow / (B * twoC);
  const int64_t rem = zrow - r * (B * twoC);
  const int64_t b = rem / twoC;
  const int64_t kk = rem - b * twoC;
  const int64_t p = zigzag_pos(r, kk, C, D);
  const int qs = (H / D) * vec_per_head;       // Q vectors of one shard
  const int ks = (Hk / D) * vec_per_head;      // K (and V) vectors of one shard
  const int row_vecs = (H + 2 * Hk) * vec_per_head;
  const uint4* dq_row = dq + zrow * (int64_t)H * vec_per_head;
  uint4* out_row = out + zrow * (int64_t)row_vecs;
  for (int cv = threadIdx.x; cv < row_vecs; cv += blockDim.x) {
    const int s = cv / (qs + 2 * ks);
    const int within = cv - s * (qs + 2 * ks);
    const int which = within < qs ? 0 : (within < qs + ks ? 1 : 2);
    const int cin = within - (which == 0 ? 0 : qs + (which - 1) * ks);
    const int d = cin % vec_per_head;
    uint4 v;
    if (which == 0) {
      v = __ldg(&dq_row[(s * (H / D) + cin / vec_per_head) * vec_per_head + d]);
    } else {
      const int head = s * (Hk / D) + cin / vec_per_head;
      const int64_t g = ((b * Hk + head) * S + p) * vec_per_head + d;
      v = __ldg(which == 1 ? &dk[g] : &dv[g]);
    }
    out_row[cv] = v;
  }
}

// As above with dQ read from an fp32 [B][H][S][dh] accumulator and scaled.
__global__ void assemble_dqkv_f32q_kernel(const float4* __restrict__ dq, float scale, const uint4* __restrict__ dk,
                                          const uint4* __restrict__ dv, uint4* __restrict__ out, int vec_per_head,
                                          int D, int B, int64_t S, int H, int Hk) {
  const int64_t C = S / (2 * D);
  const int64_t twoC = 2 * C;
  const int64_t zrow = blockIdx.x;
  const int64_t r = zrow / (B * twoC);
  const int64_t rem = zrow - r * (B * twoC);
  const int64_t b = rem / twoC;
  const int64_t kk = rem - b * twoC;
  const int64_t p = zigzag_pos(r, kk, C, D);
  const int qs = (H / D) * vec_per_head;
  const int ks = (Hk / D) * vec_per_head;
  const int row_vecs = (H + 2 * Hk) * vec_per_head;
  uint4* out_row = out + zrow * (int64_t)row_vecs;
  for (int cv = threadIdx.x; cv < row_vecs; cv += blockDim.x) {
    const int s = cv / (qs + 2 * ks);
    const int within = cv - s * (qs + 2 * ks);
    const int which = within < qs ? 0 : (within < qs + ks ? 1 : 2);
    const int cin = within - (which == 0 ? 0 : qs + (which - 1) * ks);
    const int d = cin % vec_per_head;
    uint4 v;
    if (which == 0) {
      const int head = s * (H / D) + cin / vec_per_head;
      const float4* src = dq + (((b * H + head) * S + p) * vec_per_head + d) * 2;  // 8 floats per vector
      const float4 lo = __ldg(src), hi = __ldg(src + 1);
      v = make_uint4(pack_bf16x2(lo.x * scale, lo.y * scale), pack_bf16x2(lo.z * scale, lo.w * scale),
                     pack_bf16x2(hi.x * scale, hi.y * scale), pack_bf16x2(hi.z * scale, hi.w * scale));
    } else {
      const int head = s * (Hk / D) + cin / vec_per_head;
      const int64_t g = ((b * Hk + head) * S + p) * vec_per_head + d;
      v = __ldg(which == 1 ? &dk[g] : &dv[g]);
    }
    out_row[cv] = v;
  }
}

// 32x32 tiles through shared memory, element type T (used for 4-byte elements).
template <typename T>
__global__ void transpose_kernel(const T* __restrict__ src, T* __restrict__ dst, int64_t rows, int64_t cols) {
  __shared__ T tile[32][33];
  src += (int64_t)blockIdx.y * rows * cols;  // batch of matrices along grid y
  dst += (int64_t)blockIdx.y * rows * cols;
  const int64_t tiles_c = (cols + 31) / 32;
  const int64_t tiles_r = (rows + 31) / 32;
  for (int64_t t = blockIdx.x; t < tiles_r * tiles_c; t += gridDim.x) {
    const int64_t r0 = (t / tiles_c) * 32, c0 = (t % tiles_c) * 32;
    for (int j = threadIdx.y; j < 32; j += blockDim.y) {
      const int64_t r = r0 + j, c = c0 + threadIdx.x;
      if (r < rows && c < cols) tile[j][threadIdx.x] = src[r * cols + c];
    }
    __syncthreads();
    for (int j = threadIdx.y; j < 32; j += blockDim.y) {
      const int64_t c = c0 + j, r = r0 + threadIdx.x;
      if (r < rows && c < cols) dst[c * rows + r] = tile[threadIdx.x][j];
    }
    __syncthreads();
  }
}

// 2-byte elements, both dimensions multiples of 64: 64x64 tiles moved with
// 16-byte global loads and stores.  Shared memory holds the tile as 64 rows
// of eight 16-byte chunks, chunk c of row r stored at position c ^ ((r/8)%8),
// so both the row-vector writes and the column gathers are free of bank
// conflicts.  256 threads: each writes two row vectors, then gathers two
// 8-element column vectors.
__global__ void __launch_bounds__(256) transpose_b16_kernel(const uint16_t* __restrict__ src,
                                                            uint16_t* __restrict__ dst, int rows, int cols) {
  __shared__ __align__(16) uint16_t tile[64 * 64];
  src += (int64_t)blockIdx.y * rows * cols;
  dst += (int64_t)blockIdx.y * rows * cols;
  const int tiles_c = cols / 64;
  const int ntiles = (rows / 64) * tiles_c;
  for (int t = blockIdx.x; t < ntiles; t += gridDim.x) {
    const int r0 = (t / tiles_c) * 64, c0 = (t % tiles_c) * 64;
#pragma unroll
    for (int it = 0; it < 2; ++it) {
      const int idx = threadIdx.x + it * 256;  // 64 rows x 8 chunks
      const int r = idx / 8, cv = idx % 8;
      const uint4 v = __ldg(reinterpret_cast<const uint4*>(src + (int64_t)(r0 + r) * cols + c0 + cv * 8));
      *reinterpret_cast<uint4*>(&tile[r * 64 + ((cv ^ ((r / 8) & 7)) * 8)]) = v;
    }
    __syncthreads();
#pragma unroll
    for (int it = 0; it < 2; ++it) {
      const int idx = threadIdx.x + it * 256;  // output: 64 rows (source columns) x 8 chunks
      const int c = idx / 8, rv = idx % 8;     // source column c, source rows rv*8 .. rv*8+7
      const int pos = (((c / 8) ^ rv) * 8) + (c % 8);
      uint16_t e[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) e[k] = tile[(rv * 8 + k) * 64 + pos];
      uint4 v;
      v.x = e[0] | (uint32_t(e[1]) << 16);
      v.y = e[2] | (uint32_t(e[3]) << 16);
      v.z = e[4] | (uint32_t(e[5]) << 16);
      v.w = e[6] | (uint32_t(e[7]) << 16);
      *reinterpret_cast<uint4*>(dst + (int64_t)(c0 + c) * rows + r0 + rv * 8) = v;
    }
    __syncthreads();
  }
}

// gu [T][2F] packed gate/up (128-blocks) -> m [T][F] = SiLU(g) * u, fp32.
__global__ void swiglu_f32_kernel(const float* __restrict__ gu, float* __restrict__ m, int64_t T, int F) {
  const int64_t total = T * F;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t t = i / F;
    const int f = (int)(i - t * F);
    const int64_t gcol = (int64_t)(f / 128) * 256 + (f % 128);
    const float g = gu[t * 2 * F + gcol];
    const float u = gu[t * 2 * F + gcol + 128];
    m[i] = g / (1.0f + expf(-g)) * u;
  }
}

// Packs canonical weights into (or unpacks from) the layouts of tsp.h.
// Each packed element (row n, column k) maps to one canonical element.
template <typename T>
__global__ void pack_kernel(const T* __restrict__ Wq, const T* __restrict__ Wk, const T* __restrict__ Wv,
                            const T* __restrict__ Wo, const T* __restrict__ Wg, const T* __restrict__ Wu,
                            const T* __restrict__ Wd, T* __restrict__ Pqkv, T* __restrict__ Po,
                            T* __restrict__ Pgu, T* __restrict__ Pd, int h, int hk, int F, int D, bool unpack) {
  const int64_t n_qkv = (int64_t)(h + 2 * hk) * h, n_o = (int64_t)h * h, n_gu = 2LL * F * h, n_d = (int64_t)h * F;
  const int64_t total = n_qkv + n_o + n_gu + n_d;
  const int hs = h / D, ks = hk / D;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += (int64_t)gridDim.x * blockDim.x) {
    T* packed;
    const T* canon;
    int64_t pidx, cidx;
    if (i < n_qkv) {
      // packed row n (shard s: Q h/D rows | K hk/D | V hk/D), column k
      const int64_t n = i / h, k = i % h;
      const int64_t s = n / (hs + 2 * ks), within = n % (hs + 2 * ks);
      if (within < hs) {
        canon = Wq;
        cidx = k * h + s * hs + within;
      } else {
        const int64_t kv = within - hs;
        canon = kv < ks ? Wk : Wv;
        cidx = k * hk + s * ks + (kv < ks ? kv : kv - ks);
      }
      packed = Pqkv;
      pidx = i;
    } else if (i < n_qkv + n_o) {
      const int64_t j = i - n_qkv, n = j / h, k = j % h;
      canon = Wo;
      cidx = k * h + n;
      packed = Po;
      pidx = j;
    } else if (i < n_qkv + n_o + n_gu) {
      const int64_t j = i - n_qkv - n_o, n = j / h, k = j % h;
      const int64_t blk = n / 256, off = n % 256;
      const int64_t f = blk * 128 + (off % 128);
      canon = off < 128 ? Wg : Wu;
      cidx = k * F + f;
      packed = Pgu;
      pidx = j;
    } else {
      const int64_t j = i - n_qkv - n_o - n_gu, n = j / F, k = j % F;
      canon = Wd;
      cidx = k * h + n;
      packed = Pd;
      pidx = j;
    }
    if (unpack)
      const_cast<T*>(canon)[cidx] = packed[pidx];
    else
      packed[pidx] = canon[cidx];
  }
}

int grid_for(int64_t work, int threads) {
  int64_t blocks = (work + threads - 1) / threads;
  const int64_t cap = (int64_t)num_sms() * 8;
  if (blocks > cap) blocks = cap;
  return blocks < 1 ? 1 : (int)blocks;
}

}  // namespace

cudaError_t launch_zigzag_rows(const void* src, void* dst, int64_t row_bytes, int D, int B, int64_t S,
                               bool to_zigzag, cudaStream_t stream) {
  const int64_t vpr = row_bytes / 16;
  const int64_t seg_vecs = S / (2 * D) * vpr;
  if ((int64_t)B * S * vpr == 0) return cudaSuccess;
  // about 8 resident CTAs per SM, spread evenly over the 2*D*B chunk copies
  const int64_t nseg = 2LL * D * B;
  const int64_t want = (int64_t)num_sms() * 8;
  const int64_t max_parts = (seg_vecs + kCopyThreads * kCopyUnroll - 1) / (kCopyThreads * kCopyUnroll);
  int64_t parts = (want + nseg - 1) / nseg;
  if (parts > max_parts) parts = max_parts;
  if (parts < 1) parts = 1;
  const int64_t items = nseg * parts;
  const int grid = (int)(items < want ? items : want);
  zigzag_rows_kernel<<<grid, kCopyThreads, 0, stream>>>(static_cast<const uint4*>(src), static_cast<uint4*>(dst),
                                                        vpr, D, B, S, (int)parts, to_zigzag);
  return cudaGetLastError();
}

cudaError_t launch_kv_gather(const void* kz, const void* vz, void* k, void* v, int elem_bytes, int D, int B,
                             int64_t S, int H, int dh, cudaStream_t stream) {
  return launch_kv_gather_ld(kz, vz, k, v, elem_bytes, D, B, S, H, dh, (int64_t)H * dh, stream);
}

cudaError_t launch_kv_gather_vt(const void* src, int64_t ld, int64_t v_col0, void* vt, int D, int B, int64_t S,
                                int H, int dh, cudaStream_t stream) {
  const int64_t C = S / (2 * D);
  if (C % 64 || dh % 64 || ld % 8 || v_col0 % 8) return cudaErrorInvalidValue;
  const int64_t ntiles = (int64_t)B * H * (S / 64) * (dh / 64);
  if (ntiles == 0) return cudaSuccess;
  const int64_t cap = (int64_t)num_sms() * 8;
  kv_gather_vt_kernel<<<(int)(ntiles < cap ? ntiles : cap), 256, 0, stream>>>(
      static_cast<const uint16_t*>(src), ld, v_col0, static_cast<uint16_t*>(vt), D, B, S, H, dh);
  return cudaGetLastError();
}

cudaError_t launch_kv_gather_ld(const void* kz, const void* vz, void* k, void* v, int elem_bytes, int D, int B,
                                int64_t S, int H, int dh, int64_t src_ld, cudaStream_t stream, int ntens) {
  const int vph = dh * elem_bytes / 16;
  int lg = 0;
  while ((1 << lg) < vph) ++lg;
  if ((1 << lg) != vph) return cudaErrorInvalidValue;  // dh * elem_bytes is 64, 128, 256 or 512
  const int64_t items = (int64_t)ntens * B * H * 2 * D;
  if ((int64_t)B * H * S == 0) return cudaSuccess;
  const int64_t cap = (int64_t)num_sms() * 8;
  kv_gather_kernel<<<(int)(items < cap ? items : cap), kCopyThreads, 0, stream>>>(
      static_cast<const uint4*>(kz), static_cast<const uint4*>(vz), static_cast<uint4*>(k), static_cast<uint4*>(v),
      lg, D, B, S, H, src_ld * elem_bytes / 16, ntens);
  return cudaGetLastError();
}

cudaError_t launch_copy_rows(const void* src, int64_t src_pitch_bytes, void* dst, int64_t dst_pitch_bytes,
                             int64_t rows, int64_t row_bytes, cudaStream_t stream) {
  if (rows == 0 || row_bytes == 0) return cudaSuccess;
  if ((src_pitch_bytes | dst_pitch_bytes | row_bytes) % 16) return cudaErrorInvalidValue;
  const int64_t total = rows * (row_bytes / 16);
  copy_rows_kernel<<<grid_for(total, kCopyThreads), kCopyThreads, 0, stream>>>(
      static_cast<const uint4*>(src), src_pitch_bytes / 16, static_cast<uint4*>(dst), dst_pitch_bytes / 16, rows,
      row_bytes / 16);
  return cudaGetLastError();
}

cudaError_t launch_assemble_dqkv(const void* dq, const void* dk, const void* dv, void* dqkv, int D, int B,
                                 int64_t S, int H, int Hk, int dh, cudaStream_t stream) {
  const int vph = dh * 2 / 16;
  const int64_t T = (int64_t)B * S;
  if (T == 0) return cudaSuccess;
  assemble_dqkv_kernel<<<(unsigned)T, 256, 0, stream>>>(static_cast<const uint4*>(dq), static_cast<const uint4*>(dk),
                                                         static_cast<const uint4*>(dv), static_cast<uint4*>(dqkv),
                                                         vph, D, B, S, H, Hk);
  return cudaGetLastError();
}

cudaError_t launch_assemble_dqkv_f32q(const float* dq_acc, float scale, const void* dk, const void* dv, void* dqkv,
                                      int D, int B, int64_t S, int H, int Hk, int dh, cudaStream_t stream) {
  const int vph = dh * 2 / 16;
  const int64_t T = (int64_t)B * S;
  if (T == 0) return cudaSuccess;
  assemble_dqkv_f32q_kernel<<<(unsigned)T, 256, 0, stream>>>(reinterpret_cast<const float4*>(dq_acc), scale,
                                                              static_cast<const uint4*>(dk),
                                                              static_cast<const uint4*>(dv),
                                                              static_cast<uint4*>(dqkv), vph, D, B, S, H, Hk);
  return cudaGetLastError();
}

cudaError_t launch_transpose(const void* src, void* dst, int64_t rows, int64_t cols, int elem_bytes,
                             cudaStream_t stream, int batch) {
  if (rows == 0 || cols == 0 || batch == 0) return cudaSuccess;
  const int64_t tiles = ((rows + 31) / 32) * ((cols + 31) / 32);
  const int64_t cap = ((int64_t)num_sms() * 16 + batch - 1) / batch;
  dim3 grid((unsigned)(tiles < cap ? tiles : cap), (unsigned)batch);
  dim3 block(32, 8);
  if (elem_bytes == 2 && rows % 64 == 0 && cols % 64 == 0 && rows * cols < (int64_t(1) << 31)) {
    const int64_t t64 = (rows / 64) * (cols / 64);
    const int64_t cap64 = ((int64_t)num_sms() * 8 + batch - 1) / batch;
    dim3 g64((unsigned)(t64 < cap64 ? t64 : cap64), (unsigned)batch);
    transpose_b16_kernel<<<g64, 256, 0, stream>>>(static_cast<const uint16_t*>(src), static_cast<uint16_t*>(dst),
                                                 (int)rows, (int)cols);
  } else if (elem_bytes == 2)
    transpose_kernel<uint16_t><<<grid, block, 0, stream>>>(static_cast<const uint16_t*>(src),
                                                           static_cast<uint16_t*>(dst), rows, cols);
  else
    transpose_kernel<uint32_t><<<grid, block, 0, stream>>>(static_cast<const uint32_t*>(src),
                                                           static_cast<uint32_t*>(dst), rows, cols);
  return cudaGetLastError();
}

cudaError_t launch_swiglu_f32(const float* gu, float* m, int64_t T, int F, cudaStream_t stream) {
  const int64_t total = T * F;
  if (total == 0) return cudaSuccess;
  swiglu_f32_kernel<<<grid_for(total, 256), 256, 0, stream>>>(gu, m, T, F);
  return cudaGetLastError();
}

cudaError_t launch_pack_weights(const tsp_plan* p, const void* const c[7], const tsp_weight_grads* w, bool unpack,
                                cudaStream_t stream) {
  const int h = p->hidden, F = p->ffn, D = p->D, hk = p->kv_heads * p->head_dim;
  const int64_t total = (int64_t)(h + 2 * hk) * h + (int64_t)h * h + 3LL * h * F;
  if (p->dtype == TSP_BF16)
    pack_kernel<uint16_t><<<grid_for(total, 256), 256, 0, stream>>>(
        (const uint16_t*)c[0], (const uint16_t*)c[1], (const uint16_t*)c[2], (const uint16_t*)c[3],
        (const uint16_t*)c[4], (const uint16_t*)c[5], (const uint16_t*)c[6], (uint16_t*)w->qkv, (uint16_t*)w->o,
        (uint16_t*)w->gate_up, (uint16_t*)w->down, h, hk, F, D, unpack);
  else
    pack_kernel<uint32_t><<<grid_for(total, 256), 256, 0, stream>>>(
        (const uint32_t*)c[0], (const uint32_t*)c[1], (const uint32_t*)c[2], (const uint32_t*)c[3],
        (const uint32_t*)c[4], (const uint32_t*)c[5], (const uint32_t*)c[6], (uint32_t*)w->qkv, (uint32_t*)w->o,
        (uint32_t*)w->gate_up, (uint32_t*)w->down, h, hk, F, D, unpack);
  return cudaGetLastError();
}

}  // namespace tsp
