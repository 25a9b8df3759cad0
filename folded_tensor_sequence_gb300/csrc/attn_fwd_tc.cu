// Causal flash attention forward on the 5th-generation tensor cores
// (tcgen05 + TMEM), zigzag token layout, head_dim 128, bf16 in, fp32 softmax.
//
// Queries come from the zigzag rows of the rank that owns them; keys and
// values from the gathered natural-order tensors (K as [B][Hk][S][128], V
// transposed as [B][Hk][128][S]; with grouped-query attention Hk < H and a
// query head reads K/V head head / (H / Hk)) -- the K/V all-gather of the TSP attention
// schedule (ai-trends.today TSP article, "How to Fold a Book").  Online
// softmax as in FlashAttention / ring attention (r007 chapter, "Параллелизм по
// контексту: Ring Attention против Ulysses").
//
// Block: two 128-row query tiles A and B of one (batch, head); only each
// tile's last key tile crosses the diagonal and is masked.  Chunks of whole
// 256-query blocks: a block is 256 consecutive queries (tile A stops one key
// tile before B), and a work unit is the mirror pair of blocks (G,
// 2D*nb-1-G), which lie in chunks c and 2D-1-c of the same rank.  Chunks of an
// odd number of 128-query tiles: a unit's one block is the mirror pair of
// tiles itself (tile A the light one in chunk c, tile B the heavy one in chunk
// 2D-1-c); A runs out of key tiles first and B finishes alone.  Either way
// every unit does the same number of key tiles.
//
// Per CTA: warp 16 issues TMA loads (a block's Q tiles, then K_j / V_j^T
// tiles through a 5-stage ring), warp 17 issues tcgen05.mma from one thread,
// and warps 0-15 run the softmax: for each tile and TMEM lane quadrant two
// warps, each on half of the row's 128 key columns.  TMEM (512 columns): S_A,
// S_B, O_A, O_B, 128 fp32 columns each.  Issue order per key tile j:
//   PV_A(j), S_A(j+1), PV_B(j), S_B(j+1)
// so the tensor core works on one tile while the other tile's softmax runs.
// The softmax warps hand P_x(j) over through named barriers (the MMA warp
// never waits on an mbarrier inside a block; one softmax thread has checked
// the K/V tiles that the following MMAs read).
// P = exp2(S*log2e/sqrt(dh) - m) is written as packed bf16 back into S's TMEM
// (each half over the first 32 of its 64 columns) and consumed from there by
// the PV MMA (A operand in tensor memory), which leaves shared memory for a
// deep K/V ring.  The running max is only raised (and O rescaled in TMEM)
// when it grows by more than 2^8, which keeps P <= 256 and makes the rescale
// rare; the test for it is the half-row's sum of P, not a max.
//
// Without the key split the CTAs are persistent (one per SM, units taken
// round-robin): the next block's Q tiles load as soon as a block's last S MMA
// is done, and TMEM allocation and barrier set-up happen once per CTA (8K
// tokens: 0.409 -> 0.403 ms; no change at 2 x 16K tokens).
//
// Why two warps per row and no per-tile max: the MMA warp shares its SM
// sub-partition with softmax warps, and every softmax instruction issued
// there delays its MMA issue (measured: a key-tile step takes 2230 cycles
// with no softmax arithmetic, 3140 with the one-warp softmax and its max
// tree, 2790 now).  Fewer softmax instructions per score, not shorter
// softmax latency, is what keeps the tensor pipe fed.
#include "common.cuh"
#include "internal.h"

namespace tsp {

namespace {

constexpr int QT = 128;    // rows per query tile (MMA M)
constexpr int KT = 128;    // keys per key tile
constexpr int HD = 128;    // head dim
constexpr int STAGES = 5;  // K / V^T tile ring
constexpr uint32_t SUB_BYTES = 128 * 64 * 2;     // one [128][64] bf16 swizzled sub-tile
constexpr uint32_t TILE_BYTES = 2 * SUB_BYTES;   // [128][128]
// Softmax warps 0-15 (two per query tile and TMEM lane quadrant, each taking
// half of a row's 128 key columns), then the TMA warp and the MMA warp.
constexpr int THREADS = 576;
constexpr int kTmaWarp = 16, kMmaWarp = 17;
constexpr int kHandoff = 256 + 32;  // a tile's softmax threads + the MMA warp
// Q tiles, K/V ring, mbarriers, one fp32 per row of both tiles (the row sums
// the two halves exchange).
constexpr size_t SMEM_BYTES = 1024 + (2 + STAGES) * (size_t)TILE_BYTES + 256 + 2 * 128 * sizeof(float);
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleThreshold = 8.0f;  // log2 units
constexpr float kRescaleSum = 256.0f;      // 2^kRescaleThreshold
// Named barriers handing P_x(j) from the softmax warps of tile x to the MMA
// warp, two per tile (alternating with j): A uses 1-2, B uses 3-4.  Barriers
// 5-12 pair the two warps that share the rows of one TMEM lane quadrant of one
// tile (5 + 4x + quadrant).
constexpr int kBarPA = 1, kBarPB = 3, kBarPair = 5;

struct FaParams {
  int B, H, D, nb;  // nb = blocks per chunk: 256-query blocks (nblk 2) or 128-query tiles (nblk 1)
  int nblk;         // blocks per CTA: 2 (a mirror pair of 256-query blocks) or 1 (a mirror pair of tiles)
  int Hk;           // K/V heads; query head `head` reads K/V head head / (H / Hk)
  int64_t S, C;
  int h;
  int g_off;        // first light block of the grid (rank * nb when one rank's queries run)
  // Without the key split the CTAs are persistent: CTA c takes units c, c +
  // gridDim.x, ... of the npairs * H * B units (mirror pair u % npairs, head
  // (u / npairs) % H, batch u / (npairs * H)).
  int npairs;
  int nunits;
  int64_t row_off;  // zigzag row held by row 0 of Q and O (rank * B * 2C likewise)
  // Key split: nsplit CTAs share a mirror pair, part sp taking key tiles
  // [n*sp/nsplit, n*(sp+1)/nsplit) of each block (n = the block's tile-B key
  // tiles), and write unnormalised O and (max, sum) per row to part_o /
  // part_ml ([nsplit][rows of Q][H][...]) for attn_combine_kernel; nsplit 1
  // writes O and lse directly.
  int nsplit;
  int64_t part_rows;
  float* part_o;
  float2* part_ml;
  __nv_bfloat16* o;
  float* lse;
  unsigned int* err;
};

__device__ __forceinline__ float ex2f(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// Max of 32 raw scores (3-input max tree).
__device__ __forceinline__ float max_quarter(const uint32_t (&h)[32]) {
  float m[11];
#pragma unroll
  for (int i = 0; i < 10; ++i)
    m[i] = fmax3(__uint_as_float(h[3 * i]), __uint_as_float(h[3 * i + 1]), __uint_as_float(h[3 * i + 2]));
  m[10] = fmaxf(__uint_as_float(h[30]), __uint_as_float(h[31]));
  const float a = fmax3(m[0], m[1], m[2]), b = fmax3(m[3], m[4], m[5]), c = fmax3(m[6], m[7], m[8]);
  return fmax3(fmax3(a, b, c), m[9], m[10]);
}

// Causal mask of the diagonal key tile for 32 columns starting at c0.
__device__ __forceinline__ void mask_quarter(uint32_t (&h)[32], int c0, int row) {
#pragma unroll
  for (int c = 0; c < 32; ++c)
    if (c0 + c > row) h[c] = __float_as_uint(-INFINITY);
}

// p = 2^(s * sl2 - m) for 32 scores, packed as 16 bf16 pairs (low half = even
// key) into pk; accumulates the fp32 sum of p in acc (packed pairs).
__device__ __forceinline__ void exp_pack_quarter(const uint32_t (&h)[32], uint32_t* pk, uint64_t sl2x2,
                                                 uint64_t negm2, uint64_t (&acc)[2]) {
#pragma unroll
  for (int q = 0; q < 16; ++q) {
    const uint64_t x2 = f2fma(f2pack(__uint_as_float(h[2 * q]), __uint_as_float(h[2 * q + 1])), sl2x2, negm2);
    float x0, x1;
    f2unpack(x2, x0, x1);
    const float e0 = ex2f(x0), e1 = ex2f(x1);
    acc[q & 1] = f2add(acc[q & 1], f2pack(e0, e1));
    pk[q] = pack_bf16x2(e0, e1);
  }
}

// 16-column forms of the mask and max helpers above.
__device__ __forceinline__ void mask16(uint32_t (&h)[16], int c0, int row) {
#pragma unroll
  for (int c = 0; c < 16; ++c)
    if (c0 + c > row) h[c] = __float_as_uint(-INFINITY);
}
__device__ __forceinline__ float max16(const uint32_t (&h)[16], float m) {
  const float a0 = fmax3(__uint_as_float(h[0]), __uint_as_float(h[1]), __uint_as_float(h[2]));
  const float a1 = fmax3(__uint_as_float(h[3]), __uint_as_float(h[4]), __uint_as_float(h[5]));
  const float a2 = fmax3(__uint_as_float(h[6]), __uint_as_float(h[7]), __uint_as_float(h[8]));
  const float a3 = fmax3(__uint_as_float(h[9]), __uint_as_float(h[10]), __uint_as_float(h[11]));
  const float a4 = fmax3(__uint_as_float(h[12]), __uint_as_float(h[13]), __uint_as_float(h[14]));
  return fmax3(fmax3(a0, a1, a2), fmax3(a3, a4, __uint_as_float(h[15])), m);
}
// Low-word offset of the K step k (16 elements) in a [128][128] tile of two
// 64-column sub-tiles: 2 (32 bytes) within a sub-tile, SUB_BYTES >> 4 between them.
__host__ __device__ constexpr uint32_t kstep_lo(int k) { return (k / 4) * (SUB_BYTES >> 4) + 2 * (k % 4); }

struct BlockGeo {
  int64_t zrow[2];  // row of Q / O holding tile x's first query
  int64_t p0[2];    // global position of tile x's first query
  int n[2];         // key tiles of tile x (the last one is its diagonal tile)
};

// Zigzag row and position of the 128-query tile starting `off` queries into chunk c.
__device__ __forceinline__ void tile_at(int c, int64_t off, const FaParams& p, int b, int64_t& zrow, int64_t& p0) {
  const int64_t r = c < p.D ? c : 2 * p.D - 1 - c;
  zrow = (r * p.B + b) * 2 * p.C + (c < p.D ? 0 : p.C) + off - p.row_off;
  p0 = (int64_t)c * p.C + off;
}

// blk: the CTA's block index (0: heavy, 1: light when nblk == 2).
__device__ __forceinline__ BlockGeo block_geo(int blk, int light, const FaParams& p, int b) {
  BlockGeo g;
  const int total = 2 * p.D * p.nb;
  if (p.nblk == 2) {
    const int G = blk == 0 ? total - 1 - light : light;
    const int c = G / p.nb, i = G % p.nb;
    tile_at(c, (int64_t)i * 2 * QT, p, b, g.zrow[0], g.p0[0]);
    g.zrow[1] = g.zrow[0] + QT;
    g.p0[1] = g.p0[0] + QT;
  } else {
    const int GH = total - 1 - light;  // tile B: the heavy mirror of the light tile A
    tile_at(light / p.nb, (int64_t)(light % p.nb) * QT, p, b, g.zrow[0], g.p0[0]);
    tile_at(GH / p.nb, (int64_t)(GH % p.nb) * QT, p, b, g.zrow[1], g.p0[1]);
  }
  g.n[0] = (int)(g.p0[0] / KT) + 1;
  g.n[1] = (int)(g.p0[1] / KT) + 1;
  return g;
}

// SPLIT: the key-split instantiation (parts written for attn_combine_kernel);
// without it the kernel takes every key tile and writes O and lse itself.
template <bool SPLIT>
__global__ void __launch_bounds__(THREADS, 1)
    attn_fwd_tc_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                       const __grid_constant__ CUtensorMap tmVt, const FaParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* Qs = smem;                                   // [2 tiles], block 0 then block 1
  uint8_t* KVs = smem + 2 * TILE_BYTES;                 // [STAGES] tiles
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + (2 + STAGES) * TILE_BYTES);
  uint64_t* q_full = bars + 0;              // a block's Q tiles landed (one phase per block)
  uint64_t* q_empty = bars + 2;             // a block's last S MMA done: the Q buffer may be refilled
  uint64_t* kv_full = bars + 3;             // [STAGES]
  uint64_t* kv_empty = kv_full + STAGES;    // [STAGES]
  uint64_t* s_full = kv_empty + STAGES;     // [2]
  uint64_t* o_done = s_full + 2;            // [2]
  uint64_t* drain = o_done + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  float* lx = reinterpret_cast<float*>(smem + (2 + STAGES) * TILE_BYTES + 256);  // [2 tiles][128 rows]

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int nsplit = SPLIT ? p.nsplit : 1;
  const int sp = SPLIT ? (int)blockIdx.x % nsplit : 0;  // part of the key range (key split)
  // The CTA's units: with the key split, the one of its grid position;
  // otherwise (persistent) u = blockIdx.x, blockIdx.x + gridDim.x, ...  A unit
  // is (light block or tile of a mirror pair, head, batch); with two blocks the
  // heavy one goes first.
  const int u_first = SPLIT ? 0 : (int)blockIdx.x;
  const int u_end = SPLIT ? 1 : p.nunits;
  const int u_step = SPLIT ? 1 : (int)gridDim.x;
  auto unit_of = [&](int u, int& light, int& head, int& b) {
    if constexpr (SPLIT) {
      head = (int)blockIdx.y;
      b = (int)blockIdx.z;
      light = p.g_off + (int)blockIdx.x / nsplit;
    } else {
      head = (u / p.npairs) % p.H;
      b = u / (p.npairs * p.H);
      light = p.g_off + u % p.npairs;
    }
  };
  // key tiles [lo, hiB) of this part of a block; tile A takes [lo, hiA), empty if hiA <= lo
  auto key_part = [&](const BlockGeo& g, int& lo, int& hiA, int& hiB) {
    if constexpr (SPLIT) {
      lo = (int)((int64_t)g.n[1] * sp / nsplit);
      hiB = (int)((int64_t)g.n[1] * (sp + 1) / nsplit);
      hiA = g.n[0] < hiB ? g.n[0] : hiB;
    } else {
      lo = 0;
      hiB = g.n[1];
      hiA = g.n[0];
    }
  };

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    mbar_init(q_empty, 1);
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&kv_full[s], 1);
      mbar_init(&kv_empty[s], 1);
    }
    for (int x = 0; x < 2; ++x) {
      mbar_init(&s_full[x], 1);
      mbar_init(&o_done[x], 1);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbarrier_init();
  }
  if (warp == kTmaWarp && lane == 0) {
    tma_prefetch_desc(&tmQ);
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmVt);
  }
  if (warp == kMmaWarp) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const unsigned code = KID_ATTN_FWD << 8;

  if (warp == kTmaWarp) {
    // ------------------------------ TMA producer ------------------------------
    if (lane == 0) {
      uint32_t item = 0, kb = 0;  // K/V tiles and blocks loaded so far
      bool ok = true;
      for (int u = u_first; u < u_end && ok; u += u_step) {
      int light, head, b;
      unit_of(u, light, head, b);
      const int kvh = head / (p.H / p.Hk);                        // the K/V head this query head reads
      const int64_t kv_row0 = ((int64_t)b * p.Hk + kvh) * p.S;   // K rows of that head
      const int64_t vt_row0 = ((int64_t)b * p.Hk + kvh) * HD;    // V^T rows of that head
      for (int blk = 0; blk < p.nblk && ok; ++blk, ++kb) {
        const BlockGeo g = block_geo(blk, light, p, b);
        // a block's query tiles go into the buffer once the previous block's last S MMA is done
        if (kb > 0 && !mbar_wait(q_empty, (kb - 1) & 1, abort_flag, p.err, code | 1)) {
          ok = false;
          break;
        }
        mbar_arrive_expect_tx(q_full, 2 * TILE_BYTES);
        for (int x = 0; x < 2; ++x)
          for (int c = 0; c < 2; ++c)
            tma_load_2d(Qs + x * TILE_BYTES + c * SUB_BYTES, &tmQ, head * HD + c * 64, (int)g.zrow[x], q_full);
        int lo, hiA, hiB;
        key_part(g, lo, hiA, hiB);
        for (int j = lo; j < hiB && ok; ++j) {
          for (int kv = 0; kv < 2; ++kv, ++item) {
            const int s = item % STAGES;
            if (!mbar_wait(&kv_empty[s], ((item / STAGES) & 1) ^ 1, abort_flag, p.err, code | 2)) {
              ok = false;
              break;
            }
            mbar_arrive_expect_tx(&kv_full[s], TILE_BYTES);
            uint8_t* dst = KVs + s * TILE_BYTES;
            if (kv == 0) {
              for (int c = 0; c < 2; ++c)
                tma_load_2d(dst + c * SUB_BYTES, &tmK, c * 64, (int)(kv_row0 + (int64_t)j * KT), &kv_full[s]);
            } else {
              for (int c = 0; c < 2; ++c)
                tma_load_2d(dst + c * SUB_BYTES, &tmVt, j * KT + c * 64, (int)vt_row0, &kv_full[s]);
            }
          }
        }
      }
      }
      // wait for the copies still in flight (bounded) before the CTA may exit;
      // a block's Q copies completed before any MMA of its could run, except
      // possibly the last block's if the CTA gave up
      const uint32_t first = item > (uint32_t)STAGES ? item - STAGES : 0;
      volatile int dummy = 0;
      for (uint32_t n = first; n < item; ++n) mbar_wait(&kv_full[n % STAGES], (n / STAGES) & 1, &dummy, p.err, code | 3);
      if (kb > 0) mbar_wait(q_full, (kb - 1) & 1, &dummy, p.err, code | 3);
    }
  } else if (warp == kMmaWarp) {
    // ------------------------------ MMA issuer ------------------------------
    // The whole warp walks the schedule (named barriers are warp-aligned) and
    // issues through the warp-collective MMA helpers (one elected lane
    // issues).  Inside a block the warp never waits on an mbarrier: the
    // softmax warps that hand over P_x(j) have also checked that the K/V
    // tiles the following MMAs read have landed.
    constexpr uint32_t idesc = idesc_bf16_f32(QT, KT);
    uint32_t item = 0;
    bool ok = true;  // warp-uniform: false once this warp gave up waiting
    // The MMA warp shares its SM sub-partition with softmax warps that keep
    // it from issuing; its own stream is kept short: descriptor low words per
    // tile and stage computed once, K/V stages advanced incrementally.
    const uint32_t q_lo = sdesc_lo(smem_u32(Qs));     // tile x: + x * (TILE_BYTES >> 4)
    const uint32_t kv_lo = sdesc_lo(smem_u32(KVs));   // stage s: + s * (TILE_BYTES >> 4)
    const uint32_t kv_empty_at = smem_u32(kv_empty);  // stage s: + 8 s
    const uint32_t s_full_at = smem_u32(s_full), o_done_at = smem_u32(o_done);
    auto next_stage = [](uint32_t s) { return s == STAGES - 1 ? 0u : s + 1; };
    auto mma_s = [&](int x, uint32_t s) {  // S_x = Q_x K^T, K = head dim
      const uint32_t alo = q_lo + x * (TILE_BYTES >> 4), blo = kv_lo + s * (TILE_BYTES >> 4);
#pragma unroll
      for (int k = 0; k < HD / 16; ++k)
        mma_ss_lo(tmem_base + x * 128, alo + kstep_lo(k), blo + kstep_lo(k), idesc, k > 0);
    };
    // O_x += P_x V, K = keys; P_x in TMEM over S_x's columns: keys 16k..16k+15
    // are the 8 packed columns at 64*(k/4) + 8*(k%4) (each half's P over the
    // first 32 of its own 64 columns)
    auto mma_pv = [&](int x, uint32_t s, bool acc) {
      const uint32_t blo = kv_lo + s * (TILE_BYTES >> 4);
#pragma unroll
      for (int k = 0; k < KT / 16; ++k) {
        const uint32_t pcol = 64 * (k / 4) + 8 * (k % 4);
        mma_ts_lo(tmem_base + 256 + x * 128, tmem_base + x * 128 + pcol, blo + kstep_lo(k), idesc,
                  (acc || k > 0) ? 1u : 0u);
      }
    };
    const uint32_t q_empty_at = smem_u32(q_empty);
    uint32_t kb = 0;  // blocks so far (phase of q_full)
    for (int u = u_first; u < u_end; u += u_step) {
    int light, head, b;
    unit_of(u, light, head, b);
    for (int blk = 0; blk < p.nblk; ++blk, ++kb) {
      const BlockGeo g = block_geo(blk, light, p, b);
      int lo, nA, nB;  // this part's key tiles: [lo, nB) for tile B, [lo, nA) for tile A (possibly none)
      key_part(g, lo, nA, nB);
      const bool actA = lo < nA;
      // another block follows in this CTA: its Q tiles may load once this
      // block's last S MMA (tile B's, issued after tile A's) is done
      const bool more = blk + 1 < p.nblk || u + u_step < u_end;
      const uint32_t base = item - 2 * lo;  // K_j = base + 2j, V_j = base + 2j + 1
      if (ok) {
        bool w = true;
        if (lane == 0)
          w = mbar_wait(q_full, kb & 1, abort_flag, p.err, code | 6) &&
              mbar_wait(&kv_full[item % STAGES], (item / STAGES) & 1, abort_flag, p.err, code | 4);
        ok = __shfl_sync(0xffffffffu, w ? 1 : 0, 0) != 0;
      }
      tc_fence_after();
      const uint32_t s0 = item % STAGES;  // stage of K_lo
      if (ok) {
        if (actA) {
          mma_s(0, s0);
          commit_to(s_full_at);
        }
        mma_s(1, s0);
        commit_to(s_full_at + 8);
        commit_to(kv_empty_at + 8 * s0);
        if (more && nB == lo + 1) commit_to(q_empty_at);
      }
      uint32_t sv = next_stage(s0);  // stage of V_j
      for (int j = lo; j < nB; ++j) {
        const uint32_t sk = next_stage(sv);  // stage of K_{j+1}
        if (j < nA) {
          __syncwarp();
          named_bar_sync(kBarPA + (j & 1), kHandoff);
          tc_fence_after();
          if (ok) {
            mma_pv(0, sv, j > lo);
            if (j + 1 < nA) {
              mma_s(0, sk);
              commit_to(s_full_at);
            } else {
              commit_to(o_done_at);
            }
          }
        }
        __syncwarp();
        named_bar_sync(kBarPB + (j & 1), kHandoff);
        tc_fence_after();
        if (ok) {
          mma_pv(1, sv, j > lo);
          commit_to(kv_empty_at + 8 * sv);
          if (j + 1 < nB) {
            mma_s(1, sk);
            commit_to(s_full_at + 8);
            commit_to(kv_empty_at + 8 * sk);
            if (more && j + 2 == nB) commit_to(q_empty_at);
          } else {
            commit_to(o_done_at + 8);
          }
        }
        sv = next_stage(sk);
      }
      item = base + 2 * nB;
    }
    }
    umma_commit_warp(drain);
    if (lane == 0) {
      volatile int dummy = 0;
      mbar_wait(drain, 0, &dummy, p.err, code | 7);
    }
    __syncwarp();
  } else {
    // -------------- softmax, two warps per tile and lane quadrant (warps 0-15) --------------
    // Warp w: tile x = (w / 4) % 2, rows of TMEM lane quadrant w % 4, key
    // columns [64 hf, 64 hf + 64) with hf = w / 8.  Both halves of a row keep
    // the same running max m_used (a block's first key tile and every raise
    // take the max over the whole row, which both compute alike).  Per key
    // tile no max is taken: an exponential above 2^8 (the max grew by more
    // than the threshold) makes the half's sum of P exceed 2^8, and the two
    // halves vote on that on their pair barrier; only then is the row's max
    // read to decide the raise.  Half hf writes its P over the first 32 of its
    // own 64 columns, rescales and stores O's columns [64 hf, 64 hf + 64), and
    // the halves add their row sums through shared memory at the end of a block.
    const int x = (warp / 4) & 1;
    const int hf = warp / 8;
    const int quad = warp % 4;  // the TMEM lane quadrant a warp may access
    const int row = quad * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(quad * 32) << 16;
    const uint32_t tSx = tmem_base + lane_off + x * 128;  // the whole row of S_x
    const uint32_t tS = tSx + 64 * hf;                    // this half's columns
    const uint32_t tO = tmem_base + lane_off + 256 + x * 128 + 64 * hf;
    const int pbar = kBarPair + 4 * x + quad;
    const float sl2 = kLog2e * rsqrtf((float)HD);
    uint32_t scnt = 0, ocnt = 0, item = 0;
    bool alive = true;
    const bool checker = hf == 0 && quad == 0 && lane == 0;
    // Raw max of the row's 128 scores (masked on the diagonal tile).  With
    // 18 warps the kernel has 96 registers a thread, so the TMEM loads here
    // and below are not double-buffered; what costs the tensor pipe is the
    // number of softmax instructions, not their latency.
    auto row_max = [&](bool diag) {
      float mx = -INFINITY;
#pragma unroll 1
      for (int k = 0; k < 8; ++k) {
        uint32_t bf[16];
        tmem_ld16_issue(tSx + 16 * k, bf);
        tmem_wait_ld16(bf);
        if (diag) mask16(bf, 16 * k, row);
        mx = max16(bf, mx);
      }
      return mx;
    };
    // P = 2^(s sl2 - m) over this half's 64 columns, packed into pk; returns
    // the row sum of P in sum
    auto half_exp = [&](bool diag, float m, uint32_t (&pk)[32], float& sum) {
      const uint64_t sl2x2 = f2pack(sl2, sl2), negm2 = f2pack(-m, -m);
      uint64_t acc[2] = {0, 0};
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        uint32_t bf[32];
        tmem_ld32_issue(tS + 32 * k, bf);
        tmem_wait_ld32(bf);
        if (diag) mask_quarter(bf, 64 * hf + 32 * k, row);
        exp_pack_quarter(bf, pk + 16 * k, sl2x2, negm2, acc);
      }
      float a0, a1, a2, a3;
      f2unpack(acc[0], a0, a1);
      f2unpack(acc[1], a2, a3);
      sum = (a0 + a1) + (a2 + a3);
    };
    for (int u = u_first; u < u_end; u += u_step) {
    int light, head, b;
    unit_of(u, light, head, b);
    for (int blk = 0; blk < p.nblk; ++blk) {
      const BlockGeo g = block_geo(blk, light, p, b);
      const int n = x ? g.n[1] : g.n[0];
      int lo, hiA, hiB;
      key_part(g, lo, hiA, hiB);
      const int hi = x ? hiB : hiA;
      const uint32_t base = item - 2 * lo;
      item = item + 2 * (hiB - lo);
      float m_used = -INFINITY, l = 0.f;
      // Every warp arrives once per key tile whatever happened, so the MMA
      // warp's barrier count always completes; the checker first makes sure
      // V_j and K_{j+1} have landed (the MMAs that follow read them).  A warp
      // that has given up waiting uses the blocking form, which keeps it from
      // running ahead and completing a barrier phase in the MMA warp's place.
      auto hand_off = [&](int jj) {
        if (checker && alive) {
          const uint32_t iv = base + 2 * jj + 1;
          if (mbar_wait(&kv_full[iv % STAGES], (iv / STAGES) & 1, abort_flag, p.err, code | 10) && jj + 1 < hi)
            mbar_wait(&kv_full[(iv + 1) % STAGES], ((iv + 1) / STAGES) & 1, abort_flag, p.err, code | 10);
        }
        __syncwarp();
        if (alive)
          named_bar_arrive((x == 0 ? kBarPA : kBarPB) + (jj & 1), kHandoff);
        else
          named_bar_sync((x == 0 ? kBarPA : kBarPB) + (jj & 1), kHandoff);
      };
      for (int j = lo; j < hi; ++j) {
        const bool got = alive && mbar_wait(&s_full[x], scnt & 1, abort_flag, p.err, code | 8);
        ++scnt;
        alive = __all_sync(0xffffffffu, got);
        if (!alive) {
          named_bar_red_or(pbar, 64, false);  // one vote per key tile whatever happened
          hand_off(j);
          continue;
        }
        tc_fence_after();
        const bool diag = (j == n - 1);
        if (j == lo) m_used = row_max(diag) * sl2;  // a block's (or part's) first key tile: the exact max
        uint32_t pk[32];
        float sum;
        half_exp(diag, m_used, pk, sum);
        // exponentials against the running max (exact on the first tile, so
        // the sum there is at most 64); the row's max is read only when some
        // half of the pair's rows summed above 2^8 (NaN sums count too)
        if (named_bar_red_or(pbar, 64, !(sum <= kRescaleSum))) {
          const float m_new = row_max(diag) * sl2;
          const bool up = m_new > m_used + kRescaleThreshold;
          if (__any_sync(0xffffffffu, up)) {
            const float factor = up ? ex2f(m_used - m_new) : 1.0f;
#pragma unroll 1
            for (int c2 = 0; c2 < 2; ++c2) {
              float ov[32];
              uint32_t part[32];
              tmem_ld32(tO + c2 * 32, ov);
#pragma unroll
              for (int c = 0; c < 32; ++c) part[c] = __float_as_uint(ov[c] * factor);
              tmem_st32(tO + c2 * 32, part);
            }
            if (up) {
              l *= factor;
              m_used = m_new;
            }
            half_exp(diag, m_used, pk, sum);
          }
        }
        l += sum;
        // P over this half's first 32 columns (already read); the next S MMA
        // into S_x is issued after the PV MMA that reads P.
        tmem_st32_nowait(tS, pk);
        tmem_wait_st();
        tc_fence_before();
        hand_off(j);
      }
      // the row sum over both halves (both warps of the pair take part whatever happened)
      if (lo < hi) {
        float* slot = lx + x * 128 + row;
        if (hf == 1) *slot = l;
        named_bar_sync(pbar, 64);
        if (hf == 0) {
          l += *slot;
          *slot = l;
        }
        named_bar_sync(pbar, 64);
        if (hf == 1) l = *slot;
      }
      if (!alive) continue;
      const int64_t zrow = (x ? g.zrow[1] : g.zrow[0]) + row;
      if constexpr (SPLIT) {
        float4* po =
            reinterpret_cast<float4*>(p.part_o + (((int64_t)sp * p.part_rows + zrow) * p.H + head) * HD + 64 * hf);
        const int64_t mli = ((int64_t)sp * p.part_rows + zrow) * p.H + head;
        if (lo >= hi) {
#pragma unroll 4
          for (int q = 0; q < 16; ++q) po[q] = make_float4(0.f, 0.f, 0.f, 0.f);
          if (hf == 0) p.part_ml[mli] = make_float2(-INFINITY, 0.f);
          continue;
        }
        const bool got = mbar_wait(&o_done[x], ocnt & 1, abort_flag, p.err, code | 9);
        ++ocnt;
        alive = __all_sync(0xffffffffu, got);
        if (!alive) continue;
        tc_fence_after();
#pragma unroll 1
        for (int c2 = 0; c2 < 2; ++c2) {
          float ov[32];
          tmem_ld32(tO + c2 * 32, ov);
#pragma unroll
          for (int q = 0; q < 8; ++q) po[c2 * 8 + q] = make_float4(ov[4 * q], ov[4 * q + 1], ov[4 * q + 2], ov[4 * q + 3]);
        }
        if (hf == 0) p.part_ml[mli] = make_float2(m_used, l);
        tc_fence_before();
        continue;
      }
      const bool got = mbar_wait(&o_done[x], ocnt & 1, abort_flag, p.err, code | 9);
      ++ocnt;
      alive = __all_sync(0xffffffffu, got);
      if (!alive) continue;
      tc_fence_after();
      uint32_t orr[64];
      tmem_ld64_issue(tO, orr);
      tmem_wait_ld64(orr);
      const float inv = 1.0f / l;
      uint4* dst = reinterpret_cast<uint4*>(p.o + zrow * p.h + head * HD + 64 * hf);
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        dst[q] = make_uint4(pack_bf16x2(__uint_as_float(orr[q * 8 + 0]) * inv, __uint_as_float(orr[q * 8 + 1]) * inv),
                            pack_bf16x2(__uint_as_float(orr[q * 8 + 2]) * inv, __uint_as_float(orr[q * 8 + 3]) * inv),
                            pack_bf16x2(__uint_as_float(orr[q * 8 + 4]) * inv, __uint_as_float(orr[q * 8 + 5]) * inv),
                            pack_bf16x2(__uint_as_float(orr[q * 8 + 6]) * inv, __uint_as_float(orr[q * 8 + 7]) * inv));
      }
      if (p.lse && hf == 0)
        p.lse[((int64_t)b * p.H + head) * p.S + (x ? g.p0[1] : g.p0[0]) + row] = (m_used + __log2f(l)) * kLn2;
      tc_fence_before();
    }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem_base, 512);
  }
}

// Merges the key-split parts: O = sum_s 2^(m_s - M) O_s / sum_s 2^(m_s - M) l_s with
// M = max_s m_s (m in log2 units), one warp per (row, head), four head dims per lane.
__global__ void attn_combine_kernel(const float4* __restrict__ part_o, const float2* __restrict__ part_ml, int nsplit,
                                    int64_t rows, int H, __nv_bfloat16* __restrict__ o, int h) {
  const int64_t w = (int64_t)blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  if (w >= rows * H) return;
  const int64_t row = w / H;
  const int head = (int)(w - row * H);
  float M = -INFINITY;
  for (int s = 0; s < nsplit; ++s) M = fmaxf(M, part_ml[s * rows * H + w].x);
  float L = 0.f;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int s = 0; s < nsplit; ++s) {
    const float2 ml = part_ml[s * rows * H + w];
    const float f = ex2f(ml.x - M);  // 0 for a part with no key tile (m = -inf)
    L += f * ml.y;
    const float4 v = part_o[(s * rows * H + w) * (HD / 4) + lane];
    acc.x += f * v.x;
    acc.y += f * v.y;
    acc.z += f * v.z;
    acc.w += f * v.w;
  }
  const float inv = 1.0f / L;
  uint2 out;
  out.x = pack_bf16x2(acc.x * inv, acc.y * inv);
  out.y = pack_bf16x2(acc.z * inv, acc.w * inv);
  *reinterpret_cast<uint2*>(o + row * h + head * HD + 4 * lane) = out;
}

}  // namespace

bool attn_tc_supported(int head_dim, int64_t chunk) { return head_dim == HD && chunk % QT == 0; }

size_t attn_tc_split_bytes(int64_t rows, int H) {
  return 2 * (size_t)rows * H * HD * sizeof(float) + 2 * (size_t)rows * H * sizeof(float2) + 256;
}

tsp_status attn_fwd_bf16_tc(const AttnParams& a, cudaStream_t stream) {
  if (!attn_tc_supported(a.dh, a.C)) return TSP_ERR_UNSUPPORTED;
  if (a.B * a.S == 0) return TSP_OK;
  // Q / O rows: every rank's, or one rank's B * 2C
  const int64_t T = a.rank < 0 ? (int64_t)a.B * a.S : (int64_t)a.B * 2 * a.C;
  const int h = a.H * HD;
  CUtensorMap mq, mk, mv;
  if (!make_tma_2d_bf16(&mq, a.q, T, h, h, 128) ||
      !make_tma_2d_bf16(&mk, a.k, (int64_t)a.B * a.Hk * a.S, HD, HD, 128) ||
      !make_tma_2d_bf16(&mv, a.v, (int64_t)a.B * a.Hk * HD, a.S, a.S, 128))
    return TSP_ERR_CUDA;
  static std::atomic<unsigned long long> configured{0};  // devices set up
  if (needs_setup(configured)) {
    if (cudaFuncSetAttribute(attn_fwd_tc_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)SMEM_BYTES) != cudaSuccess ||
        cudaFuncSetAttribute(attn_fwd_tc_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)SMEM_BYTES) != cudaSuccess)
      return TSP_ERR_CUDA;
    mark_setup_done(configured);
  }
  FaParams p;
  p.B = a.B;
  p.H = a.H;
  p.Hk = a.Hk;
  p.D = a.D;
  p.nblk = a.C % (2 * QT) == 0 ? 2 : 1;
  p.nb = (int)(a.C / (p.nblk * QT));
  p.S = a.S;
  p.C = a.C;
  p.h = h;
  p.o = static_cast<__nv_bfloat16*>(a.o);
  p.lse = a.lse;
  p.err = dev_error_word();
  p.g_off = a.rank < 0 ? 0 : a.rank * p.nb;
  p.row_off = a.rank < 0 ? 0 : (int64_t)a.rank * a.B * 2 * a.C;
  const int pairs = a.rank < 0 ? a.D * p.nb : p.nb;
  // A grid under one wave (one rank's queries of one weight shard) splits every
  // CTA's key range in two when the caller gave room for the parts (no lse then).
  p.nsplit = 1;
  p.part_rows = T;
  p.part_o = nullptr;
  p.part_ml = nullptr;
  if (a.split_ws && !a.lse && a.split_ws_bytes >= attn_tc_split_bytes(T, a.H) &&
      (int64_t)pairs * a.H * a.B < num_sms()) {
    p.nsplit = 2;
    p.part_o = static_cast<float*>(a.split_ws);
    p.part_ml = reinterpret_cast<float2*>(static_cast<char*>(a.split_ws) + 2 * (size_t)T * a.H * HD * sizeof(float));
  }
  p.npairs = pairs;
  p.nunits = pairs * a.H * a.B;
  if (p.nsplit > 1) {
    attn_fwd_tc_kernel<true><<<dim3(pairs * p.nsplit, a.H, a.B), THREADS, SMEM_BYTES, stream>>>(mq, mk, mv, p);
  } else {
    // persistent: one CTA per SM walks the units (the next block's Q tiles
    // load while a block finishes, and set-up is paid once per CTA)
    const int sms = num_sms();
    attn_fwd_tc_kernel<false><<<(unsigned)(p.nunits < sms ? p.nunits : sms), THREADS, SMEM_BYTES, stream>>>(mq, mk, mv, p);
  }
  if (cudaGetLastError() != cudaSuccess) return TSP_ERR_CUDA;
  if (p.nsplit > 1) {
    const int64_t warps = T * a.H;
    attn_combine_kernel<<<(unsigned)((warps + 7) / 8), 256, 0, stream>>>(
        reinterpret_cast<const float4*>(p.part_o), p.part_ml, p.nsplit, T, a.H, p.o, h);
    if (cudaGetLastError() != cudaSuccess) return TSP_ERR_CUDA;
  }
  return TSP_OK;
}

}  // namespace tsp
