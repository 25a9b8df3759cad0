// libtsp C ABI: plan validation, workspace layout and the orchestration of
// one TSP transformer layer on one GPU.
//
// Schedule of the layer (ai-trends.today, "Zyphra Introduces Tensor and
// Sequence Parallelism (TSP)", section "How to Fold a Book"; edge.aivizor.me
// TSP news post), with the D ranks emulated as partitions of device memory:
//   1. zigzag permute: rank r's tokens are chunks r and 2D-1-r;
//   2. attention: for every weight shard s, every rank projects its local
//      tokens with {W_Q, W_K, W_V}^s, K/V are all-gathered into natural
//      order, causal attention runs, and O_s W_O^s is accumulated locally.
//      Here: one projection GEMM over all shards (N = h + 2hk, hk the K/V
//      width: h for multi-head attention, less with grouped-query attention,
//      where a shard owns H/D query heads and Hk/D K/V heads) whose epilogue does
//      the gather, the zigzag-balanced attention kernel, and one output GEMM
//      whose K loop is the sum over shards (+ residual);
//   3. gated MLP ring: each rank accumulates SiLU(H W_g^j)(H W_u^j) W_d^j over
//      the shards j passing around the ring, with no all-reduce.  Here: one
//      gate/up GEMM with the SiLU*up epilogue and one down GEMM whose K loop is
//      the ring's sum over shards (+ residual);
//   4. unpermute back to natural order.
// For bf16 plans whose chunks are whole 128-row tiles the permute of x and
// the unpermute of y (and, in training, of dx) are not separate passes: the
// GEMMs read and write those rows through remapped row coordinates.
#include <stdarg.h>
#include <stdio.h>
#include <string.h>

#include <atomic>
#include <cmath>
#include <initializer_list>
#include <mutex>
#include <new>
#include <vector>

#include "common.cuh"
#include "internal.h"

namespace tsp {

__device__ unsigned int g_dev_error_word = 0;

// One warp waits (bounded) on a barrier that nothing will signal: the wait
// gives up after timeout_ns, records the error word and the kernel returns.
__global__ void wait_probe_kernel(unsigned int* err, unsigned long long timeout_ns) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    abort_flag = 0;
    fence_mbarrier_init();
  }
  __syncwarp();
  if (threadIdx.x == 0) mbar_wait_for(&bar, 0, &abort_flag, err, (KID_WAIT_PROBE << 8) | 1, timeout_ns);
}

namespace {

thread_local char t_last_error[512] = "";
thread_local tsp_status t_fail_status = TSP_OK;
thread_local int t_fail_count = 0;

tsp_status fail(tsp_status s, const char* fmt, ...) __attribute__((format(printf, 2, 3)));
tsp_status fail(tsp_status s, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(t_last_error, sizeof(t_last_error), fmt, ap);
  va_end(ap);
  return s;
}

tsp_status cuda_status(cudaError_t e, const char* what) {
  if (e == cudaSuccess) return TSP_OK;
  return fail(TSP_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

// Consumes one armed injected failure, if any.
bool injected(tsp_status* out) {
  if (t_fail_count > 0) {
    --t_fail_count;
    *out = fail(t_fail_status, "injected failure (tsp_debug_fail_next)");
    return true;
  }
  return false;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

size_t esize(const tsp_plan* p) { return p->dtype == TSP_BF16 ? 2 : 4; }

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

int kv_hidden(const tsp_plan* p) { return p->kv_heads * p->head_dim; }

// Offsets of the layer's activations inside one buffer (the `saved` buffer
// for the backward and the forward's workspace share this layout).
struct Layout {
  size_t xz, qz, k, v, oz, lse, hz, gu, mz, yz;  // yz: forward workspace only
  size_t saved_end, fwd_end;
};

Layout layer_layout(const tsp_plan* p, int batch) {
  const size_t T = (size_t)batch * p->seq, h = p->hidden, F = p->ffn, e = esize(p);
  Layout L;
  size_t o = 0;
  auto take = [&](size_t bytes) {
    size_t at = o;
    o = align256(o + bytes);
    return at;
  };
  const size_t hk = kv_hidden(p);
  L.xz = take(T * h * e);
  L.qz = take(T * h * e);
  L.k = take(T * hk * e);
  L.v = take(T * hk * e);
  L.oz = take(T * h * e);
  L.lse = take((size_t)batch * p->heads * p->seq * 4);
  L.hz = take(T * h * e);
  L.gu = take(T * 2 * F * e);
  L.mz = take(T * F * e);
  L.saved_end = o;
  L.yz = take(T * h * e);
  L.fwd_end = o;
  return L;
}

struct BwdLayout {
  size_t dyz, dgu, dhz, doz, dq, dk, dv, dsum, dqkv, dxz, vnat, end;
};

BwdLayout bwd_layout(const tsp_plan* p, int batch) {
  const size_t T = (size_t)batch * p->seq, h = p->hidden, F = p->ffn, e = esize(p);
  BwdLayout L;
  size_t o = 0;
  auto take = [&](size_t bytes) {
    size_t at = o;
    o = align256(o + bytes);
    return at;
  };
  L.dyz = take(T * h * e);
  L.dgu = take(T * 2 * F * e);
  L.dhz = take(T * h * e);
  L.doz = take(T * h * e);
  const size_t hk = kv_hidden(p);
  L.dq = take(T * h * 4);  // fp32 dQ accumulator [B][H][S][dh] (bf16 zigzag [T][h] on the warp-MMA path)
  L.dk = take(T * hk * e);
  L.dv = take(T * hk * e);
  L.dsum = take((size_t)batch * p->heads * p->seq * 4);
  L.dqkv = take(T * (h + 2 * hk) * e);
  L.dxz = take(T * h * e);
  L.vnat = take(T * hk * e);  // V in [B][Hk][S][dh] when the forward saved it transposed
  L.end = o;
  return L;
}

size_t attn_ws_bytes(const tsp_plan* p, int batch) {
  const size_t T = (size_t)batch * p->seq, h = p->hidden, e = esize(p);
  return 4 * align256(T * h * e);
}

size_t mlp_ws_bytes(const tsp_plan* p, int batch) {
  const size_t T = (size_t)batch * p->seq, F = p->ffn, e = esize(p);
  return align256(T * F * e) + align256(T * 2 * F * e);
}

// bf16 plans whose chunks are whole 128-row tiles move natural-order
// activations through remapped GEMM rows instead of zigzag copies: x and y in
// inference, y and dx in training.
bool folded_io(const tsp_plan* p) { return p->dtype == TSP_BF16 && p->chunk % 128 == 0; }

tsp_status check_plan_batch(const tsp_plan* p, int batch) {
  if (!p) return fail(TSP_ERR_INVALID_ARG, "plan is NULL");
  if (batch < 0) return fail(TSP_ERR_INVALID_ARG, "batch %d < 0", batch);
  if ((int64_t)batch * p->seq > (int64_t)INT32_MAX / 4)
    return fail(TSP_ERR_UNSUPPORTED, "batch*seq = %lld too large", (long long)batch * p->seq);
  return TSP_OK;
}

tsp_status check_ptrs(std::initializer_list<const void*> ptrs, const char* what) {
  for (const void* q : ptrs) {
    if (!q) return fail(TSP_ERR_INVALID_ARG, "%s: NULL pointer", what);
    if (!aligned16(q)) return fail(TSP_ERR_INVALID_ARG, "%s: pointer %p not 16-byte aligned", what, q);
  }
  return TSP_OK;
}

tsp_status check_bf16_shapes(const tsp_plan* p) {
  if (p->dtype != TSP_BF16) return TSP_OK;
  if (p->hidden % 256 || p->ffn % 256)
    return fail(TSP_ERR_UNSUPPORTED, "bf16 kernels need hidden %% 256 == 0 and ffn %% 256 == 0 (got %d, %d)",
                p->hidden, p->ffn);
  if (p->head_dim != 128) return fail(TSP_ERR_UNSUPPORTED, "bf16 attention needs head_dim 128 (got %d)", p->head_dim);
  return TSP_OK;
}

cudaStream_t as_stream(void* s) { return static_cast<cudaStream_t>(s); }


// ---- optional per-step timing (tsp_profile_*) --------------------------------
// When enabled, each launched step is bracketed by two CUDA events on its
// stream; tsp_profile_report() sums the elapsed times per step name.
struct ProfState {
  std::mutex mu;
  bool enabled = false;
  struct Rec {
    const char* name;
    cudaEvent_t a, b;
  };
  std::vector<Rec> recs;
  std::vector<cudaEvent_t> pool;
  cudaEvent_t get() {
    cudaEvent_t e = nullptr;
    if (!pool.empty()) {
      e = pool.back();
      pool.pop_back();
    } else if (cudaEventCreate(&e) != cudaSuccess) {
      e = nullptr;
    }
    return e;
  }
};
ProfState& prof() {
  static ProfState* s = new ProfState;  // never destroyed: events may outlive static teardown order
  return *s;
}

struct Prof {
  const char* name;
  cudaStream_t st;
  cudaEvent_t a = nullptr;
  Prof(const char* n, cudaStream_t s) : name(n), st(s) {
    ProfState& P = prof();
    std::lock_guard<std::mutex> g(P.mu);
    if (!P.enabled) return;
    a = P.get();
    if (a) cudaEventRecord(a, st);
  }
  ~Prof() {
    if (!a) return;
    ProfState& P = prof();
    std::lock_guard<std::mutex> g(P.mu);
    cudaEvent_t b = P.get();
    if (!b) {
      P.pool.push_back(a);  // no closing event: the step goes unrecorded, the event is reused
      return;
    }
    cudaEventRecord(b, st);
    P.recs.push_back({name, a, b});
  }
};

thread_local std::vector<Prof*> t_prof_stack;

// ---- the layer pieces ------------------------------------------------------

EpiParams base_epi(const tsp_plan* p, int batch) {
  EpiParams ep;
  ep.D = p->D;
  ep.B = batch;
  ep.S = (int)p->seq;
  ep.C = (int)p->chunk;
  ep.H = p->heads;
  ep.Hk = p->kv_heads;
  ep.dh = p->head_dim;
  ep.h = p->hidden;
  ep.err = dev_error_word();
  return ep;
}

// The tcgen05 attention kernel reads V transposed ([B][H][dh][S]); the QKV
// epilogue writes V in that layout whenever that kernel will run.
bool use_tc_attention(const tsp_plan* p) {
  return p->dtype == TSP_BF16 && attn_tc_supported(p->head_dim, p->chunk);
}

// a_mn / b_mn: operand stored [K][M] / [K][N] (tensor-core path only).
tsp_status run_gemm(const tsp_plan* p, const void* A, int64_t lda, const void* B, int64_t ldb, int M, int N, int K,
                    EpiKind epi, const EpiParams& ep, cudaStream_t st, const char* what, bool a_mn = false,
                    bool b_mn = false) {
  Prof pr(what, st);
  if (p->dtype != TSP_BF16 && (a_mn || b_mn)) return fail(TSP_ERR_UNSUPPORTED, "%s: MN-major fp32 GEMM", what);
  tsp_status s = p->dtype == TSP_BF16
                     ? gemm_bf16_tc(A, lda, B, ldb, M, N, K, epi, ep, st, a_mn, b_mn)
                     : gemm_f32_simt(static_cast<const float*>(A), lda, static_cast<const float*>(B), ldb, M, N, K,
                                     epi, ep, st);
  if (s != TSP_OK) return fail(s, "%s GEMM (M=%d N=%d K=%d) failed: %s", what, M, N, K, tsp_status_string(s));
  return TSP_OK;
}

// a_out = (Attn(xz Wq, xz Wk, xz Wv)) Wo [+ resid]
// x_natural: xz (and resid) are natural-order rows, read through the GEMMs'
// zigzag row remapping instead of a separate permute.
tsp_status attention_impl(const tsp_plan* p, int batch, const void* xz, const tsp_weights* w, void* a_out,
                          const void* resid, float* lse, char* qz, char* k, char* v, char* oz, cudaStream_t st,
                          bool x_natural = false) {
  const int T = batch * (int)p->seq, h = p->hidden;
  EpiParams ep = base_epi(p, batch);
  ep.q = qz;
  ep.k = k;
  ep.v = v;
  ep.v_transposed = use_tc_attention(p);
  ep.a_natural = x_natural;
  tsp_status s = run_gemm(p, xz, h, w->qkv, h, T, h + 2 * kv_hidden(p), h, EPI_QKV, ep, st, "QKV projection");
  if (s != TSP_OK) return s;
  AttnParams ap;
  ap.q = qz;
  ap.k = k;
  ap.v = v;
  ap.o = oz;
  ap.lse = lse;
  ap.D = p->D;
  ap.B = batch;
  ap.H = p->heads;
  ap.Hk = p->kv_heads;
  ap.dh = p->head_dim;
  ap.S = p->seq;
  ap.C = p->chunk;
  {
    Prof pr("attention", st);
    s = p->dtype != TSP_BF16 ? attn_fwd_f32(ap, st)
                             : (use_tc_attention(p) ? attn_fwd_bf16_tc(ap, st) : attn_fwd_bf16(ap, st));
  }
  if (s != TSP_OK) return fail(s, "attention kernel failed: %s", tsp_status_string(s));
  EpiParams eo = base_epi(p, batch);
  eo.out = a_out;
  eo.ldo = h;
  eo.resid = resid;
  eo.ldr = h;
  eo.resid_natural = x_natural;
  return run_gemm(p, oz, h, w->o, h, T, h, h, resid ? EPI_RESID : EPI_STORE, eo, st, "output projection");
}

// out = (SiLU(hz Wg) * (hz Wu)) Wd [+ resid]; optionally keeps the raw gate/up in gu_save
// out_natural: the down projection writes natural-order rows.
tsp_status mlp_impl(const tsp_plan* p, int batch, const void* hz, const tsp_weights* w, void* out, const void* resid,
                    char* mz, char* gu, bool save_gu, cudaStream_t st, bool out_natural = false) {
  const int T = batch * (int)p->seq, h = p->hidden, F = p->ffn;
  tsp_status s;
  if (p->dtype == TSP_BF16) {
    EpiParams eg = base_epi(p, batch);
    eg.out = mz;
    eg.ldo = F;
    eg.aux = save_gu ? gu : nullptr;
    eg.ldx = 2 * F;
    s = run_gemm(p, hz, h, w->gate_up, h, T, 2 * F, h, EPI_SWIGLU, eg, st, "gate/up projection");
  } else {
    EpiParams eg = base_epi(p, batch);
    eg.out = gu;
    eg.ldo = 2 * F;
    s = run_gemm(p, hz, h, w->gate_up, h, T, 2 * F, h, EPI_STORE, eg, st, "gate/up projection");
    Prof pr("swiglu", st);
    if (s == TSP_OK)
      s = cuda_status(launch_swiglu_f32(reinterpret_cast<const float*>(gu), reinterpret_cast<float*>(mz), T, F, st),
                      "swiglu");
  }
  if (s != TSP_OK) return s;
  EpiParams ed = base_epi(p, batch);
  ed.out = out;
  ed.ldo = h;
  ed.resid = resid;
  ed.ldr = h;
  ed.out_natural = out_natural;
  return run_gemm(p, mz, F, w->down, F, T, h, F, resid ? EPI_RESID : EPI_STORE, ed, st, "down projection");
}

// ---- one rank of a multi-GPU layer (tsp_rank_*) --------------------------------

struct RankDims {
  int64_t L;       // local rows: batch * 2C
  int hs, ks, fs;  // h/D, hk/D, F/D
};

RankDims rank_dims(const tsp_plan* p, int batch) {
  return RankDims{(int64_t)batch * 2 * p->chunk, p->hidden / p->D, kv_hidden(p) / p->D, p->ffn / p->D};
}

// Element offsets of the second matrix in each shard buffer (o_s, down_j).
size_t attn_shard_o_offset(const tsp_plan* p) {
  const RankDims d = rank_dims(p, 0);
  return (size_t)(d.hs + 2 * d.ks) * p->hidden;
}
size_t mlp_shard_down_offset(const tsp_plan* p) { return (size_t)2 * (p->ffn / p->D) * p->hidden; }

tsp_status check_rank_shapes(const tsp_plan* p, const char* what) {
  const RankDims d = rank_dims(p, 0);
  const size_t e = esize(p);
  if (d.fs % 128)
    return fail(TSP_ERR_UNSUPPORTED, "%s: ffn/D = %d is not a multiple of 128 (a shard holds whole gate/up blocks)",
                what, d.fs);
  if ((d.hs * e) % 16 || (2 * d.ks * e) % 16)
    return fail(TSP_ERR_UNSUPPORTED, "%s: hidden/D and 2*kv_hidden/D rows must be multiples of 16 bytes", what);
  if (p->dtype == TSP_BF16) {
    tsp_status s = check_bf16_shapes(p);
    if (s != TSP_OK) return s;
    if (d.hs % 256 || (2 * d.ks) % 256)
      return fail(TSP_ERR_UNSUPPORTED, "%s: bf16 needs hidden/D %% 256 == 0 and 2*kv_hidden/D %% 256 == 0 (got %d, %d)",
                  what, d.hs, 2 * d.ks);
  }
  return TSP_OK;
}

struct RankAttnLayout {
  size_t k, v, vt, o, split, end;  // split: parts of the attention kernel's key split (tcgen05 path)
};

RankAttnLayout rank_attn_layout(const tsp_plan* p, int batch) {
  const RankDims d = rank_dims(p, batch);
  const size_t e = esize(p), kvb = (size_t)batch * p->seq * d.ks * e;
  RankAttnLayout L;
  size_t o = 0;
  auto take = [&](size_t bytes) {
    size_t at = o;
    o = align256(o + bytes);
    return at;
  };
  L.k = take(kvb);
  // natural V for the warp-MMA kernel, V^T (gathered straight into it) for the tcgen05 kernel
  L.v = take(kvb);
  L.vt = L.v;
  L.o = take((size_t)d.L * d.hs * e);
  L.split = use_tc_attention(p) ? take(attn_tc_split_bytes(d.L, p->heads / p->D)) : L.o;
  L.end = o;
  return L;
}

size_t rank_mlp_ws_bytes(const tsp_plan* p, int batch) {
  const RankDims d = rank_dims(p, batch);
  const size_t e = esize(p);
  return align256((size_t)d.L * d.fs * e) + (p->dtype == TSP_BF16 ? 0 : align256((size_t)d.L * 2 * d.fs * e));
}

}  // namespace

tsp_status report_error(tsp_status s, const char* msg) { return fail(s, "%s", msg); }

// Every device address the library looks up (error word, static scratch, SM
// count, kernel attributes) is the current device's, so the work must be
// enqueued on a stream of that device.
tsp_status check_stream_device(void* stream, const char* what) {
  int cur = 0, sdev = 0;
  cudaError_t e = cudaGetDevice(&cur);
  if (e == cudaSuccess) e = cudaStreamGetDevice(as_stream(stream), &sdev);
  if (e != cudaSuccess) return fail(TSP_ERR_CUDA, "%s: device of the stream: %s", what, cudaGetErrorString(e));
  if (sdev != cur)
    return fail(TSP_ERR_INVALID_ARG, "%s: the stream belongs to device %d but device %d is current", what, sdev,
                cur);
  return TSP_OK;
}

void prof_begin(const char* name, cudaStream_t st) { t_prof_stack.push_back(new Prof(name, st)); }

void prof_end(cudaStream_t) {
  if (t_prof_stack.empty()) return;
  delete t_prof_stack.back();  // records the closing event
  t_prof_stack.pop_back();
}

// Per-device caches below are filled on first use by whichever host thread
// gets there; every thread computes the same value, so a relaxed atomic store
// is enough.
unsigned int* dev_error_word() {
  static std::atomic<unsigned int*> ptrs[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  unsigned int* p = ptrs[dev].load(std::memory_order_relaxed);
  if (!p) {
    void* a = nullptr;
    if (cudaGetSymbolAddress(&a, g_dev_error_word) != cudaSuccess) return nullptr;
    p = static_cast<unsigned int*>(a);
    ptrs[dev].store(p, std::memory_order_relaxed);
  }
  return p;
}

namespace {
unsigned long long device_bit() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  return 1ull << dev;
}
}  // namespace

bool needs_setup(const std::atomic<unsigned long long>& done) {
  const unsigned long long bit = device_bit();
  return bit == 0 || (done.load() & bit) == 0;
}

void mark_setup_done(std::atomic<unsigned long long>& done) { done.fetch_or(device_bit()); }

int num_sms() {
  static std::atomic<int> cache[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 1;
  int n = cache[dev].load(std::memory_order_relaxed);
  if (!n) {
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 1;
    cache[dev].store(n, std::memory_order_relaxed);
  }
  return n;
}

}  // namespace tsp

using namespace tsp;

extern "C" {

const char* tsp_status_string(tsp_status s) {
  switch (s) {
    case TSP_OK: return "TSP_OK";
    case TSP_ERR_INVALID_ARG: return "TSP_ERR_INVALID_ARG";
    case TSP_ERR_UNSUPPORTED: return "TSP_ERR_UNSUPPORTED";
    case TSP_ERR_CUDA: return "TSP_ERR_CUDA";
    case TSP_ERR_TIMEOUT: return "TSP_ERR_TIMEOUT";
    case TSP_ERR_WORKSPACE: return "TSP_ERR_WORKSPACE";
  }
  return "TSP_ERR_UNKNOWN";
}

const char* tsp_last_error_message(void) { return t_last_error; }

void tsp_debug_fail_next(tsp_status status, int count) {
  t_fail_status = status;
  t_fail_count = count > 0 ? count : 0;
}

tsp_status tsp_plan_create(int D, int64_t seq, int hidden, int heads, int head_dim, int ffn, tsp_dtype dtype,
                           tsp_plan** out) {
  return tsp_plan_create_gqa(D, seq, hidden, heads, heads, head_dim, ffn, dtype, out);
}

tsp_status tsp_plan_create_gqa(int D, int64_t seq, int hidden, int heads, int kv_heads, int head_dim, int ffn,
                               tsp_dtype dtype, tsp_plan** out) {
  if (!out) return fail(TSP_ERR_INVALID_ARG, "out is NULL");
  *out = nullptr;
  if (D < 1) return fail(TSP_ERR_INVALID_ARG, "D = %d < 1", D);
  if (seq < 2 * (int64_t)D || seq % (2 * (int64_t)D))
    return fail(TSP_ERR_INVALID_ARG, "seq %lld not a positive multiple of 2D = %d", (long long)seq, 2 * D);
  if (heads < 1 || head_dim < 1 || hidden != heads * head_dim)
    return fail(TSP_ERR_INVALID_ARG, "hidden %d != heads %d * head_dim %d", hidden, heads, head_dim);
  if (head_dim != 32 && head_dim != 64 && head_dim != 128)
    return fail(TSP_ERR_INVALID_ARG, "head_dim %d not in {32, 64, 128}", head_dim);
  if (heads % D) return fail(TSP_ERR_INVALID_ARG, "heads %d not divisible by D %d", heads, D);
  if (kv_heads < 1 || heads % kv_heads)
    return fail(TSP_ERR_INVALID_ARG, "kv_heads %d does not divide heads %d", kv_heads, heads);
  if (kv_heads % D)
    return fail(TSP_ERR_INVALID_ARG, "kv_heads %d not divisible by D %d (a shard owns whole K/V heads)", kv_heads, D);
  if (ffn < 1 || ffn % D) return fail(TSP_ERR_INVALID_ARG, "ffn %d not a positive multiple of D %d", ffn, D);
  if (hidden % 8) return fail(TSP_ERR_INVALID_ARG, "hidden %d not a multiple of 8", hidden);
  if (ffn % 128) return fail(TSP_ERR_INVALID_ARG, "ffn %d not a multiple of 128", ffn);
  if (dtype != TSP_F32 && dtype != TSP_BF16) return fail(TSP_ERR_INVALID_ARG, "unknown dtype %d", (int)dtype);
  if (seq > (int64_t)INT32_MAX / 4) return fail(TSP_ERR_UNSUPPORTED, "seq %lld too large", (long long)seq);
  tsp_plan* p = new (std::nothrow) tsp_plan;
  if (!p) return fail(TSP_ERR_INVALID_ARG, "out of host memory");
  p->D = D;
  p->seq = seq;
  p->hidden = hidden;
  p->heads = heads;
  p->kv_heads = kv_heads;
  p->head_dim = head_dim;
  p->ffn = ffn;
  p->dtype = dtype;
  p->chunk = seq / (2 * D);
  *out = p;
  return TSP_OK;
}

void tsp_plan_destroy(tsp_plan* plan) { delete plan; }

tsp_status tsp_plan_set_deterministic(tsp_plan* plan, int deterministic) {
  if (!plan) return fail(TSP_ERR_INVALID_ARG, "plan is NULL");
  if (deterministic != 0 && deterministic != 1)
    return fail(TSP_ERR_INVALID_ARG, "deterministic = %d (0 or 1)", deterministic);
  plan->deterministic = deterministic;
  return TSP_OK;
}

int tsp_plan_get_deterministic(const tsp_plan* plan) { return plan ? plan->deterministic : -1; }

size_t tsp_workspace_bytes(const tsp_plan* p, int batch, tsp_op op) {
  if (!p || batch < 0) return 0;
  switch (op) {
    case TSP_OP_ATTENTION_FWD: return attn_ws_bytes(p, batch);
    case TSP_OP_GATED_MLP_FWD: return mlp_ws_bytes(p, batch);
    case TSP_OP_LAYER_FWD: return layer_layout(p, batch).fwd_end;
    case TSP_OP_LAYER_BWD: return bwd_layout(p, batch).end;
    case TSP_OP_DECODE: return decode_ws_bytes(p, batch);
    case TSP_OP_RANK_ATTENTION: return rank_attn_layout(p, batch).end;
    case TSP_OP_RANK_MLP: return rank_mlp_ws_bytes(p, batch);
  }
  return 0;
}

size_t tsp_saved_bytes(const tsp_plan* p, int batch) {
  if (!p || batch < 0) return 0;
  return layer_layout(p, batch).saved_end;
}

tsp_status tsp_pack_weights(const tsp_plan* p, const void* const canonical[7], const tsp_weight_grads* packed,
                            void* stream) {
  tsp_status s;
  if (injected(&s)) return s;
  if (!p || !canonical || !packed) return fail(TSP_ERR_INVALID_ARG, "NULL argument");
  if ((s = check_ptrs({canonical[0], canonical[1], canonical[2], canonical[3], canonical[4], canonical[5],
                       canonical[6], packed->qkv, packed->o, packed->gate_up, packed->down},
                      "tsp_pack_weights")) != TSP_OK)
    return s;
  if ((s = check_stream_device(stream, "tsp_pack_weights")) != TSP_OK) return s;
  return cuda_status(launch_pack_weights(p, canonical, packed, false, as_stream(stream)), "pack weights");
}

tsp_status tsp_unpack_weights(const tsp_plan* p, const tsp_weights* packed, void* const canonical[7], void* stream) {
  tsp_status s;
  if (injected(&s)) return s;
  if (!p || !canonical || !packed) return fail(TSP_ERR_INVALID_ARG, "NULL argument");
  if ((s = check_ptrs({canonical[0], canonical[1], canonical[2], canonical[3], canonical[4], canonical[5],
                       canonical[6], packed->qkv, packed->o, packed->gate_up, packed->down},
                      "tsp_unpack_weights")) != TSP_OK)
    return s;
  if ((s = check_stream_device(stream, "tsp_unpack_weights")) != TSP_OK) return s;
  tsp_weight_grads w{const_cast<void*>(packed->qkv), const_cast<void*>(packed->o), const_cast<void*>(packed->gate_up),
                     const_cast<void*>(packed->down)};
  return cuda_status(launch_pack_weights(p, const_cast<const void* const*>(canonical), &w, true, as_stream(stream)),
                     "unpack weights");
}

tsp_status tsp_zigzag_permute(const tsp_plan* p, int batch, const void* x, void* xz, void* stream) {
  tsp_status s;
  if (injected(&s)) return s;
  if ((s = check_plan_batch(p, batch)) != TSP_OK) return s;
  if (batch == 0) return TSP_OK;
  if ((s = check_ptrs({x, xz}, "tsp_zigzag_permute")) != TSP_OK) return s;
  if ((s = check_stream_device(stream, "tsp_zigzag_permute")) != TSP_OK) return s;
  Prof pr("zigzag permute", as_stream(stream));
  return cuda_status(
      launch_zigzag_rows(x, xz, (int64_t)p->hidden * esize(p), p->D, batch, p->seq, true, as_stream(stream)),
      "zigzag permute");
}

tsp_status tsp_zigzag_unpermute(const tsp_plan* p, int batch, const void* xz, void* x, void* stream) {
  tsp_status s;
  if (injected(&s)) return s;
  if ((s = check_plan_batch(p, batch)) != TSP_OK) return s;
  if (batch == 0) return TSP_OK;
  if ((s = check_ptrs({x, xz}, "tsp_zigzag_unpermute")) != TSP_OK) return s;
  if ((s = check_stream_device(stream, "tsp_zigzag_unpermute")) != TSP_OK) return s;
  Prof pr("zigzag unpermute", as_stream(stream));
  return cuda_status(
      launch_zigzag_rows(xz, x, (int64_t)p->hidden * esize(p), p->D, batch, p->seq, false, as_stream(stream)),
      "zigzag unpermute");
}

tsp_status tsp_kv_gather(const tsp_plan* p, int batch, const void* kz, const void* vz, void* k, void* v,
                         void* stream) {
  tsp_status s;
  if (injected(&s)) return s;
  if ((s = check_plan_batch(p, batch)) != TSP_OK) return s;
  if (batch == 0) return TSP_OK;
  if ((s = check_ptrs({kz, vz, k, v}, "tsp_kv_gather")) != TSP_OK) return s;
  if ((s = check_stream_device(stream, "tsp_kv_gather")) != TSP_OK) return s;
  Prof pr("kv gather", as_stream(stream));
  return cuda_status(launch_kv_gather(kz, vz, k, v, (int)esize(p), p->D, batch, p->seq, p->kv_heads, p->head_dim,
                                      as_stream(stream)),
                     "kv gather");
}

tsp_status tsp_attention_fwd(const tsp_plan* p, int batch, const void* xz, const tsp_weights* w, void* a_out,
                             void* lse, void* ws, size_t ws_bytes, void* stream) {
  tsp_status s;
  if (injected(&s)) return s;
  if ((s = check_plan_batch(p, batch)) != TSP_OK) return s;
  if (batch == 0) return TSP_OK;
  if (!w) return fail(TSP_ERR_INVALID_ARG, "weights is NULL");
  if ((s = check_ptrs({xz, a_out, w->qkv, w->o, ws}, "tsp_attention_fwd")) != TSP_OK) return s;
  if (lse && !aligned16(lse)) return fail(TSP_ERR_INVALID_ARG, "lse not 16-byte aligned");
  if ((s = check_bf16_shapes(p)) != TSP_OK) return s;
  if (ws_bytes < attn_ws_bytes(p, batch))
    return fail(TSP_ERR_WORKSPACE, "workspace %zu < %zu bytes", ws_bytes, attn_ws_bytes(p, batch));
  if ((s = check_stream_device(stream, "tsp_attention_fwd")) != TSP_OK) return s;
  const size_t blk = attn_ws_bytes(p, batch) / 4;
  char* base = static_cast<char*>(ws);
  return attention_impl(p, batch, xz, w, a_out, nullptr, static_cast<float*>(lse), base, base + blk, base + 2 * blk,
                        base + 3 * blk, as_stream(stream));
}

tsp_status tsp_gated_mlp_fwd(const tsp_plan* p, int batch, const void* hz, const tsp_weights* w, void* m_out,
                             void* ws, size_t ws_bytes, void* stream) {
  tsp_status s;
  if (injected(&s)) return s;
  if ((s = check_plan_batch(p, batch)) != TSP_OK) return s;
  if (batch == 0) return TSP_OK;
  if (!w) return fail(TSP_ERR_INVALID_ARG, "weights is NULL");
  if ((s = check_ptrs({hz, m_out, w->gate_up, w->down, ws}, "tsp_gated_mlp_fwd")) != TSP_OK) return s;
  if ((s = check_bf16_shapes(p)) != TSP_OK) return s;
  if (ws_bytes < mlp_ws_bytes(p, batch))
    return fail(TSP_ERR_WORKSPACE, "workspace %zu < %zu bytes", ws_bytes, mlp_ws_bytes(p, batch));
  if ((s = check_stream_device(stream, "tsp_gated_mlp_fwd")) != TSP_OK) return s;
  const size_t T = (size_t)batch * p->seq;
  char* mz = static_cast<char*>(ws);
  char* gu = mz + align256(T * p->ffn * esize(p));
  return mlp_impl(p, batch, hz, w, m_out, nullptr, mz, gu, false, as_stream(stream));
}

tsp_status tsp_layer_fwd(const tsp_plan* p, int batch, const void* x, const tsp_weights* w, void* y, void* saved,
                         void* ws, size_t ws_bytes, void* stream) {
  tsp_status s;
  if (injected(&s)) return s;
  if ((s = check_plan_batch(p, batch)) != TSP_OK) return s;
  if (batch == 0) return TSP_OK;
  if (!w) return fail(TSP_ERR_INVALID_ARG, "weights is NULL");
  if ((s = check_ptrs({x, y, w->qkv, w->o, w->gate_up, w->down, ws}, "tsp_layer_fwd")) != TSP_OK) return s;
  if (saved && !aligned16(saved)) return fail(TSP_ERR_INVALID_ARG, "saved not 16-byte aligned");
  if ((s = check_bf16_shapes(p)) != TSP_OK) return s;
  const Layout L = layer_layout(p, batch);
  if (ws_bytes < L.fwd_end) return fail(TSP_ERR_WORKSPACE, "workspace %zu < %zu bytes", ws_bytes, L.fwd_end);
  if ((s = check_stream_device(stream, "tsp_layer_fwd")) != TSP_OK) return s;
  cudaStream_t st = as_stream(stream);
  char* wsb = static_cast<char*>(ws);
  char* act = saved ? static_cast<char*>(saved) : wsb;  // where the saved activations go
  char* xz = act + L.xz;
  char* yz = wsb + L.yz;
  if (!saved && folded_io(p)) {
    // The zigzag permute and unpermute ride on the GEMMs: every 128-row tile
    // of zigzag rows is one contiguous run of natural rows, so the QKV GEMM
    // reads x through remapped TMA coordinates, the output projection adds x
    // by remapped row, and the down projection writes y in natural order.
    s = attention_impl(p, batch, x, w, act + L.hz, x, nullptr, act + L.qz, act + L.k, act + L.v, act + L.oz, st,
                       true);
    if (s != TSP_OK) return s;
    return mlp_impl(p, batch, act + L.hz, w, y, act + L.hz, act + L.mz, act + L.gu, false, st, true);
  }
  {
    Prof pr("zigzag permute", st);
    s = cuda_status(launch_zigzag_rows(x, xz, (int64_t)p->hidden * esize(p), p->D, batch, p->seq, true, st),
                    "zigzag permute");
  }
  if (s != TSP_OK) return s;
  s = attention_impl(p, batch, xz, w, act + L.hz, xz, saved ? reinterpret_cast<float*>(act + L.lse) : nullptr,
                     act + L.qz, act + L.k, act + L.v, act + L.oz, st);
  if (s != TSP_OK) return s;
  // Training (the backward's weight gradients read x as a zigzag copy, which
  // they stream faster than remapped natural rows): x is permuted and saved,
  // y still leaves in natural order through the down projection.
  if (folded_io(p)) return mlp_impl(p, batch, act + L.hz, w, y, act + L.hz, act + L.mz, act + L.gu, true, st, true);
  s = mlp_impl(p, batch, act + L.hz, w, yz, act + L.hz, act + L.mz, act + L.gu, saved != nullptr, st);
  if (s != TSP_OK) return s;
  Prof pr("zigzag unpermute", st);
  return cuda_status(launch_zigzag_rows(yz, y, (int64_t)p->hidden * esize(p), p->D, batch, p->seq, false, st),
                     "zigzag unpermute");
}

tsp_status tsp_layer_bwd(const tsp_plan* p, int batch, const void* x, const tsp_weights* w, const void* saved,
                         const void* dy, void* dx, const tsp_weight_grads* dw, void* ws, size_t ws_bytes,
                         void* stream) {
  tsp_status s;
  if (injected(&s)) return s;
  if ((s = check_plan_batch(p, batch)) != TSP_OK) return s;
  if (batch == 0) return TSP_OK;
  if (!w || !dw) return fail(TSP_ERR_INVALID_ARG, "weights or grads is NULL");
  if ((s = check_ptrs({x, saved, dy, dx, w->qkv, w->o, w->gate_up, w->down, dw->qkv, dw->o, dw->gate_up, dw->down,
                       ws},
                      "tsp_layer_bwd")) != TSP_OK)
    return s;
  if (p->dtype != TSP_BF16) return fail(TSP_ERR_UNSUPPORTED, "layer backward is implemented for bf16 plans");
  if ((s = check_bf16_shapes(p)) != TSP_OK) return s;
  if (p->kv_heads != p->heads && !attn_bwd_tc_supported(p->head_dim, p->chunk))
    return fail(TSP_ERR_UNSUPPORTED, "grouped-query backward needs chunk %% 128 == 0 (got %lld)",
                (long long)p->chunk);
  const int64_t T64 = (int64_t)batch * p->seq;
  if (T64 % 64) return fail(TSP_ERR_UNSUPPORTED, "backward needs batch*seq %% 64 == 0 (got %lld)", (long long)T64);
  const BwdLayout L = bwd_layout(p, batch);
  if (ws_bytes < L.end) return fail(TSP_ERR_WORKSPACE, "workspace %zu < %zu bytes", ws_bytes, L.end);
  if ((s = check_stream_device(stream, "tsp_layer_bwd")) != TSP_OK) return s;
  const Layout A = layer_layout(p, batch);
  cudaStream_t st = as_stream(stream);
  const char* sv = static_cast<const char*>(saved);
  char* wb = static_cast<char*>(ws);
  const int T = (int)T64, h = p->hidden, F = p->ffn, W3 = h + 2 * kv_hidden(p);
  const int64_t eb = (int64_t)esize(p);
  // transposes `nmat` consecutive [rows][cols] matrices into workspace
  auto tr = [&](const void* src, size_t dst_off, int64_t rows, int64_t cols, const char* what, int nmat = 1) {
    Prof pr(what, st);
    return cuda_status(launch_transpose(src, wb + dst_off, rows, cols, (int)eb, st, nmat), what);
  };
#define TSP_TRY(expr)              \
  do {                             \
    if ((s = (expr)) != TSP_OK) return s; \
  } while (0)
  // dy enters through a zigzag copy (the weight gradients stream it faster
  // than remapped natural rows); dx leaves in natural order through the dx GEMM.
  const bool fold = folded_io(p);
  {
    Prof pr("permute dy", st);
    TSP_TRY(cuda_status(launch_zigzag_rows(dy, wb + L.dyz, h * eb, p->D, batch, p->seq, true, st), "permute dy"));
  }
  // MLP backward
  // Every weight and activation is read in the layout it is stored in: the
  // GEMM takes operands stored [K][M] / [K][N] (MN-major) where the product
  // needs their transpose.
  {
    EpiParams e = base_epi(p, batch);
    e.out = wb + L.dgu;
    e.ldo = 2 * F;
    e.resid = sv + A.gu;
    e.ldr = 2 * F;
    // dM = dY Wd^T: B = W_down^T, i.e. the packed down weight [h][F] read MN-major
    TSP_TRY(run_gemm(p, wb + L.dyz, h, w->down, F, T, F, h, EPI_DSWIGLU, e, st, "dM = dY Wd^T", false, true));
  }
  {
    EpiParams e = base_epi(p, batch);
    e.out = dw->down;
    e.ldo = F;
    // dWd^T = dY^T M: A = dY [T][h], B = M [T][F], both MN-major
    TSP_TRY(run_gemm(p, wb + L.dyz, h, sv + A.mz, F, h, F, T, EPI_STORE, e, st, "dW_down", true, true));
  }
  {
    EpiParams e = base_epi(p, batch);
    e.out = wb + L.dhz;
    e.ldo = h;
    e.resid = wb + L.dyz;
    e.ldr = h;
    // dH = dY + dGU Wgu: B = packed gate_up [2F][h] read MN-major
    TSP_TRY(run_gemm(p, wb + L.dgu, 2 * F, w->gate_up, h, T, h, 2 * F, EPI_RESID, e, st, "dH", false, true));
  }
  {
    EpiParams e = base_epi(p, batch);
    e.out = dw->gate_up;
    e.ldo = h;
    // dWgu = dGU^T H: A = dGU [T][2F], B = H [T][h], both MN-major
    TSP_TRY(run_gemm(p, wb + L.dgu, 2 * F, sv + A.hz, h, 2 * F, h, T, EPI_STORE, e, st, "dW_gate_up", true,
                     true));
  }
  // attention output projection backward
  {
    EpiParams e = base_epi(p, batch);
    e.out = wb + L.doz;
    e.ldo = h;
    // dO = dH Wo^T: B = packed o [h][h] read MN-major
    TSP_TRY(run_gemm(p, wb + L.dhz, h, w->o, h, T, h, h, EPI_STORE, e, st, "dO", false, true));
  }
  {
    EpiParams e = base_epi(p, batch);
    e.out = dw->o;
    e.ldo = h;
    // dWo^T = dH^T O: A = dH [T][h], B = O [T][h], both MN-major
    TSP_TRY(run_gemm(p, wb + L.dhz, h, sv + A.oz, h, h, h, T, EPI_STORE, e, st, "dW_O", true, true));
  }
  // attention core backward
  const void* v_nat = sv + A.v;
  if (use_tc_attention(p)) {
    TSP_TRY(tr(sv + A.v, L.vnat, p->head_dim, p->seq, "transpose V^T", batch * p->kv_heads));
    v_nat = wb + L.vnat;
  }
  const bool tc_bwd = attn_bwd_tc_supported(p->head_dim, p->chunk);
  if (tc_bwd) {
    const bool fused = !p->deterministic;
    {
      Prof pr("attention bwd dsum", st);
      // the fused kernel adds dQ partial sums into the accumulator: zero it in the same pass
      TSP_TRY(cuda_status(launch_attn_dsum(sv + A.oz, wb + L.doz, reinterpret_cast<float*>(wb + L.dsum), p->D, batch,
                                         p->heads, p->seq, p->chunk, st,
                                         fused ? reinterpret_cast<float*>(wb + L.dq) : nullptr),
                          "attention dsum"));
    }
    AttnBwdTcArgs ab;
    ab.q = sv + A.qz;
    ab.k = sv + A.k;
    ab.v = v_nat;
    ab.dO = wb + L.doz;
    ab.lse = reinterpret_cast<const float*>(sv + A.lse);
    ab.dsum = reinterpret_cast<const float*>(wb + L.dsum);
    ab.dq_acc = reinterpret_cast<float*>(wb + L.dq);
    ab.dk = wb + L.dk;
    ab.dv = wb + L.dv;
    ab.D = p->D;
    ab.B = batch;
    ab.H = p->heads;
    ab.Hk = p->kv_heads;
    ab.dh = p->head_dim;
    ab.S = p->seq;
    ab.C = p->chunk;
    if (fused) {
      Prof pr("attention bwd fused", st);
      s = attn_bwd_bf16_tc(ab, st, 4);
    } else {
      {
        Prof pr("attention bwd dK/dV", st);
        s = attn_bwd_bf16_tc(ab, st, 1);
      }
      if (s == TSP_OK) {
        Prof pr("attention bwd dQ", st);
        s = attn_bwd_bf16_tc(ab, st, 2);
      }
    }
    if (s != TSP_OK) return fail(s, "attention backward (tensor cores) failed: %s", tsp_status_string(s));
  } else {
    AttnBwdParams ab;
    ab.q = sv + A.qz;
    ab.k = sv + A.k;
    ab.v = v_nat;
    ab.o = sv + A.oz;
    ab.dO = wb + L.doz;
    ab.lse = reinterpret_cast<const float*>(sv + A.lse);
    ab.dsum = reinterpret_cast<float*>(wb + L.dsum);
    ab.dq = wb + L.dq;
    ab.dk = wb + L.dk;
    ab.dv = wb + L.dv;
    ab.D = p->D;
    ab.B = batch;
    ab.H = p->heads;
    ab.dh = p->head_dim;
    ab.S = p->seq;
    ab.C = p->chunk;
    {
      Prof pr("attention bwd", st);
      s = attn_bwd_bf16(ab, st);
    }
    if (s != TSP_OK) return fail(s, "attention backward failed: %s", tsp_status_string(s));
  }
  {
    Prof pr_asm("assemble dQKV", st);
    if (tc_bwd)
      TSP_TRY(cuda_status(launch_assemble_dqkv_f32q(reinterpret_cast<const float*>(wb + L.dq),
                                                    1.0f / std::sqrt((float)p->head_dim), wb + L.dk, wb + L.dv,
                                                    wb + L.dqkv, p->D, batch, p->seq, p->heads, p->kv_heads,
                                                    p->head_dim, st),
                          "assemble dQKV"));
    else
      TSP_TRY(cuda_status(launch_assemble_dqkv(wb + L.dq, wb + L.dk, wb + L.dv, wb + L.dqkv, p->D, batch, p->seq,
                                               p->heads, p->kv_heads, p->head_dim, st),
                          "assemble dQKV"));
  }
  {
    EpiParams e = base_epi(p, batch);
    e.out = fold ? dx : wb + L.dxz;
    e.ldo = h;
    e.out_natural = fold;
    e.resid = wb + L.dhz;
    e.ldr = h;
    // dx = dH + dQKV Wqkv: B = packed qkv [h + 2hk][h] read MN-major
    TSP_TRY(run_gemm(p, wb + L.dqkv, W3, w->qkv, h, T, h, W3, EPI_RESID, e, st, "dx", false, true));
  }
  {
    EpiParams e = base_epi(p, batch);
    e.out = dw->qkv;
    e.ldo = h;
    // dWqkv = dQKV^T xz: A = dQKV [T][h + 2hk], B = xz [T][h], both MN-major
    TSP_TRY(run_gemm(p, wb + L.dqkv, W3, sv + A.xz, h, W3, h, T, EPI_STORE, e, st, "dW_QKV", true, true));
  }
  if (fold) return TSP_OK;
  Prof pr_dx("unpermute dx", st);
  return cuda_status(launch_zigzag_rows(wb + L.dxz, dx, h * eb, p->D, batch, p->seq, false, st), "unpermute dx");
#undef TSP_TRY
}

tsp_status tsp_decode_step(const tsp_plan* p, int batch, int64_t pos, const void* x_new, const tsp_weights* w,
                           void* k_cache, void* v_cache, void* y_new, void* ws, size_t ws_bytes, void* stream) {
  tsp_status s;
  if (injected(&s)) return s;
  if (!p) return fail(TSP_ERR_INVALID_ARG, "plan is NULL");
  if (batch < 1 || batch > 8) return fail(TSP_ERR_INVALID_ARG, "decode batch %d not in [1, 8]", batch);
  if (pos < 0 || pos >= p->seq)
    return fail(TSP_ERR_INVALID_ARG, "pos %lld not in [0, seq = %lld)", (long long)pos, (long long)p->seq);
  if (!w) return fail(TSP_ERR_INVALID_ARG, "weights is NULL");
  if ((s = check_ptrs({x_new, k_cache, v_cache, y_new, w->qkv, w->o, w->gate_up, w->down, ws}, "tsp_decode_step")) !=
      TSP_OK)
    return s;
  if (p->dtype != TSP_BF16) return fail(TSP_ERR_UNSUPPORTED, "decode is implemented for bf16 plans");
  if ((s = check_bf16_shapes(p)) != TSP_OK) return s;
  const int g = p->heads / p->kv_heads;
  if (g != 1 && g != 2 && g != 4 && g != 8)
    return fail(TSP_ERR_UNSUPPORTED, "decode needs heads / kv_heads in {1, 2, 4, 8} (got %d)", g);
  if (ws_bytes < decode_ws_bytes(p, batch))
    return fail(TSP_ERR_WORKSPACE, "workspace %zu < %zu bytes", ws_bytes, decode_ws_bytes(p, batch));
  if ((s = check_stream_device(stream, "tsp_decode_step")) != TSP_OK) return s;
  s = decode_step_bf16(p, batch, pos, x_new, w, k_cache, v_cache, y_new, ws, as_stream(stream));
  if (s != TSP_OK) return fail(s, "decode step failed: %s", tsp_status_string(s));
  return TSP_OK;
}

size_t tsp_rank_shard_bytes(const tsp_plan* p, tsp_shard_kind kind) {
  if (!p) return 0;
  const RankDims d = rank_dims(p, 0);
  const size_t e = esize(p), h = p->hidden;
  if (kind == TSP_SHARD_ATTENTION) return ((size_t)(d.hs + 2 * d.ks) * h + h * d.hs) * e;
  if (kind == TSP_SHARD_MLP) return ((size_t)2 * d.fs * h + h * d.fs) * e;
  return 0;
}

tsp_status tsp_rank_extract_shard(const tsp_plan* p, const tsp_weights* w, int shard, tsp_shard_kind kind, void* out,
                                  void* stream) {
  tsp_status s;
  if (injected(&s)) return s;
  if (!p || !w) return fail(TSP_ERR_INVALID_ARG, "tsp_rank_extract_shard: NULL plan or weights");
  if (shard < 0 || shard >= p->D) return fail(TSP_ERR_INVALID_ARG, "shard %d not in [0, D = %d)", shard, p->D);
  if (kind != TSP_SHARD_ATTENTION && kind != TSP_SHARD_MLP)
    return fail(TSP_ERR_INVALID_ARG, "unknown shard kind %d", (int)kind);
  if ((s = check_rank_shapes(p, "tsp_rank_extract_shard")) != TSP_OK) return s;
  const void* a = kind == TSP_SHARD_ATTENTION ? w->qkv : w->gate_up;
  const void* b = kind == TSP_SHARD_ATTENTION ? w->o : w->down;
  if ((s = check_ptrs({a, b, out}, "tsp_rank_extract_shard")) != TSP_OK) return s;
  if ((s = check_stream_device(stream, "tsp_rank_extract_shard")) != TSP_OK) return s;
  const RankDims d = rank_dims(p, 0);
  const int64_t e = (int64_t)esize(p), h = p->hidden;
  cudaStream_t st = as_stream(stream);
  char* dst = static_cast<char*>(out);
  cudaError_t ce;
  if (kind == TSP_SHARD_ATTENTION) {
    const int64_t rows = d.hs + 2 * d.ks;  // the shard's rows of packed qkv, then its input rows of W_O
    ce = launch_copy_rows(static_cast<const char*>(a) + shard * rows * h * e, h * e, dst, h * e, rows, h * e, st);
    if (ce == cudaSuccess)
      ce = launch_copy_rows(static_cast<const char*>(b) + (int64_t)shard * d.hs * e, h * e,
                            dst + attn_shard_o_offset(p) * e, d.hs * e, h, d.hs * e, st);
  } else {
    const int64_t F = p->ffn;
    ce = launch_copy_rows(static_cast<const char*>(a) + (int64_t)shard * 2 * d.fs * h * e, h * e, dst, h * e,
                          2 * d.fs, h * e, st);
    if (ce == cudaSuccess)
      ce = launch_copy_rows(static_cast<const char*>(b) + (int64_t)shard * d.fs * e, F * e,
                            dst + mlp_shard_down_offset(p) * e, d.fs * e, h, d.fs * e, st);
  }
  return cuda_status(ce, "extract shard");
}

tsp_status tsp_rank_qkv(const tsp_plan* p, int batch, const void* x_local, const void* attn_shard, void* q_local,
                        void* kv_local, void* stream) {
  tsp_status s;
  if (injected(&s)) return s;
  if ((s = check_plan_batch(p, batch)) != TSP_OK) return s;
  if (batch == 0) return TSP_OK;
  if ((s = check_ptrs({x_local, attn_shard, q_local, kv_local}, "tsp_rank_qkv")) != TSP_OK) return s;
  if ((s = check_rank_shapes(p, "tsp_rank_qkv")) != TSP_OK) return s;
  if ((s = check_stream_device(stream, "tsp_rank_qkv")) != TSP_OK) return s;
  const RankDims d = rank_dims(p, batch);
  const int h = p->hidden;
  cudaStream_t st = as_stream(stream);
  // one GEMM over the shard's Q|K|V rows (they share the A operand); its
  // epilogue sends the Q columns to q_local and the K|V columns to kv_local
  EpiParams e = base_epi(p, batch);
  e.out = q_local;
  e.ldo = d.hs;
  e.aux = kv_local;
  e.ldx = 2 * d.ks;
  e.split_col = d.hs;
  return run_gemm(p, x_local, h, attn_shard, h, (int)d.L, d.hs + 2 * d.ks, h, EPI_STORE, e, st,
                  "rank QKV projection");
}

tsp_status tsp_rank_attention(const tsp_plan* p, int rank, int batch, const void* q_local, const void* kv_all,
                              const void* attn_shard, const void* resid, void* h_out, void* ws, size_t ws_bytes,
                              void* stream) {
  tsp_status s;
  if (injected(&s)) return s;
  if ((s = check_plan_batch(p, batch)) != TSP_OK) return s;
  if (rank < 0 || rank >= p->D) return fail(TSP_ERR_INVALID_ARG, "rank %d not in [0, D = %d)", rank, p->D);
  if (batch == 0) return TSP_OK;
  if ((s = check_ptrs({q_local, kv_all, attn_shard, h_out, ws}, "tsp_rank_attention")) != TSP_OK) return s;
  if (resid && !aligned16(resid)) return fail(TSP_ERR_INVALID_ARG, "tsp_rank_attention: resid not 16-byte aligned");
  if ((s = check_rank_shapes(p, "tsp_rank_attention")) != TSP_OK) return s;
  const RankAttnLayout W = rank_attn_layout(p, batch);
  if (ws_bytes < W.end) return fail(TSP_ERR_WORKSPACE, "workspace %zu < %zu bytes", ws_bytes, W.end);
  if ((s = check_stream_device(stream, "tsp_rank_attention")) != TSP_OK) return s;
  const RankDims d = rank_dims(p, batch);
  const int h = p->hidden, hk_heads = p->kv_heads / p->D;
  const size_t e = esize(p);
  cudaStream_t st = as_stream(stream);
  char* wb = static_cast<char*>(ws);
  // the all-gathered rows [D][L][2 ks] (K columns, then V) into natural positions:
  // K [B][Hk/D][S][dh]; V likewise, or for the tcgen05 kernel straight into V^T [B][Hk/D][dh][S]
  const bool tc = use_tc_attention(p);
  {
    Prof pr("rank K/V reorder", st);
    s = cuda_status(launch_kv_gather_ld(kv_all, static_cast<const char*>(kv_all) + (size_t)d.ks * e, wb + W.k,
                                        tc ? nullptr : wb + W.v, (int)e, p->D, batch, p->seq, hk_heads,
                                        p->head_dim, 2 * d.ks, st, tc ? 1 : 2),
                    "rank K/V reorder");
    if (s == TSP_OK && tc)
      s = cuda_status(launch_kv_gather_vt(kv_all, 2 * d.ks, d.ks, wb + W.vt, p->D, batch, p->seq, hk_heads,
                                          p->head_dim, st),
                      "rank V^T gather");
  }
  if (s != TSP_OK) return s;
  AttnParams ap;
  ap.q = q_local;
  ap.k = wb + W.k;
  ap.v = wb + W.vt;
  ap.o = wb + W.o;
  ap.lse = nullptr;
  ap.D = p->D;
  ap.B = batch;
  ap.H = p->heads / p->D;
  ap.Hk = hk_heads;
  ap.dh = p->head_dim;
  ap.S = p->seq;
  ap.C = p->chunk;
  ap.rank = rank;
  if (tc) {  // one rank's queries of one shard rarely fill the GPU: room for the key split
    ap.split_ws = wb + W.split;
    ap.split_ws_bytes = W.end - W.split;
  }
  {
    Prof pr("rank attention", st);
    s = p->dtype != TSP_BF16 ? attn_fwd_f32(ap, st) : (tc ? attn_fwd_bf16_tc(ap, st) : attn_fwd_bf16(ap, st));
  }
  if (s != TSP_OK) return fail(s, "rank attention kernel failed: %s", tsp_status_string(s));
  EpiParams eo = base_epi(p, batch);
  eo.out = h_out;
  eo.ldo = h;
  eo.resid = resid;
  eo.ldr = h;
  const char* wo = static_cast<const char*>(attn_shard) + attn_shard_o_offset(p) * e;
  return run_gemm(p, wb + W.o, d.hs, wo, d.hs, (int)d.L, h, d.hs, resid ? EPI_RESID : EPI_STORE, eo, st,
                  "rank output projection");
}

tsp_status tsp_rank_mlp(const tsp_plan* p, int batch, const void* h_local, const void* mlp_shard, const void* resid,
                        void* y_out, void* ws, size_t ws_bytes, void* stream) {
  tsp_status s;
  if (injected(&s)) return s;
  if ((s = check_plan_batch(p, batch)) != TSP_OK) return s;
  if (batch == 0) return TSP_OK;
  if ((s = check_ptrs({h_local, mlp_shard, y_out, ws}, "tsp_rank_mlp")) != TSP_OK) return s;
  if (resid && !aligned16(resid)) return fail(TSP_ERR_INVALID_ARG, "tsp_rank_mlp: resid not 16-byte aligned");
  if ((s = check_rank_shapes(p, "tsp_rank_mlp")) != TSP_OK) return s;
  if (ws_bytes < rank_mlp_ws_bytes(p, batch))
    return fail(TSP_ERR_WORKSPACE, "workspace %zu < %zu bytes", ws_bytes, rank_mlp_ws_bytes(p, batch));
  if ((s = check_stream_device(stream, "tsp_rank_mlp")) != TSP_OK) return s;
  const RankDims d = rank_dims(p, batch);
  const int h = p->hidden;
  const size_t e = esize(p);
  cudaStream_t st = as_stream(stream);
  char* mz = static_cast<char*>(ws);
  if (p->dtype == TSP_BF16) {
    EpiParams eg = base_epi(p, batch);
    eg.out = mz;
    eg.ldo = d.fs;
    s = run_gemm(p, h_local, h, mlp_shard, h, (int)d.L, 2 * d.fs, h, EPI_SWIGLU, eg, st, "rank gate/up projection");
  } else {
    char* gu = mz + align256((size_t)d.L * d.fs * e);
    EpiParams eg = base_epi(p, batch);
    eg.out = gu;
    eg.ldo = 2 * d.fs;
    s = run_gemm(p, h_local, h, mlp_shard, h, (int)d.L, 2 * d.fs, h, EPI_STORE, eg, st, "rank gate/up projection");
    if (s == TSP_OK) {
      Prof pr("rank swiglu", st);
      s = cuda_status(launch_swiglu_f32(reinterpret_cast<const float*>(gu), reinterpret_cast<float*>(mz), d.L, d.fs,
                                        st),
                      "rank swiglu");
    }
  }
  if (s != TSP_OK) return s;
  EpiParams ed = base_epi(p, batch);
  ed.out = y_out;
  ed.ldo = h;
  ed.resid = resid;
  ed.ldr = h;
  const char* wd = static_cast<const char*>(mlp_shard) + mlp_shard_down_offset(p) * e;
  return run_gemm(p, mz, d.fs, wd, d.fs, (int)d.L, h, d.fs, resid ? EPI_RESID : EPI_STORE, ed, st,
                  "rank down projection");
}

tsp_status tsp_debug_wait_timeout(unsigned int timeout_us, void* stream) {
  tsp_status s;
  if (injected(&s)) return s;
  if (timeout_us == 0 || timeout_us > 10000000u)
    return fail(TSP_ERR_INVALID_ARG, "timeout_us %u not in (0, 10 s]", timeout_us);
  if ((s = check_stream_device(stream, "tsp_debug_wait_timeout")) != TSP_OK) return s;
  unsigned int* err = dev_error_word();
  if (!err) return fail(TSP_ERR_CUDA, "device error word unavailable");
  wait_probe_kernel<<<1, 32, 0, as_stream(stream)>>>(err, (unsigned long long)timeout_us * 1000ull);
  return cuda_status(cudaGetLastError(), "wait probe launch");
}

void tsp_profile_enable(int on) {
  ProfState& P = prof();
  std::lock_guard<std::mutex> g(P.mu);
  P.enabled = on != 0;
}

int tsp_profile_report(const char** names, double* total_ms, int* counts, int max_entries) {
  ProfState& P = prof();
  std::lock_guard<std::mutex> g(P.mu);
  std::vector<const char*> nm;
  std::vector<double> ms;
  std::vector<int> cnt;
  for (auto& r : P.recs) {
    float t = 0.f;
    if (cudaEventSynchronize(r.b) == cudaSuccess) cudaEventElapsedTime(&t, r.a, r.b);
    size_t i = 0;
    while (i < nm.size() && strcmp(nm[i], r.name) != 0) ++i;
    if (i == nm.size()) {
      nm.push_back(r.name);
      ms.push_back(0.0);
      cnt.push_back(0);
    }
    ms[i] += t;
    cnt[i] += 1;
    P.pool.push_back(r.a);
    P.pool.push_back(r.b);
  }
  P.recs.clear();
  for (size_t i = 0; i < nm.size() && (int)i < max_entries; ++i) {
    if (names) names[i] = nm[i];
    if (total_ms) total_ms[i] = ms[i];
    if (counts) counts[i] = cnt[i];
  }
  return (int)nm.size();
}

tsp_status tsp_sync_check(void* stream) {
  cudaError_t e = cudaStreamSynchronize(as_stream(stream));
  if (e != cudaSuccess) return fail(TSP_ERR_CUDA, "stream synchronize: %s", cudaGetErrorString(e));
  e = cudaGetLastError();
  if (e != cudaSuccess) return fail(TSP_ERR_CUDA, "pending CUDA error: %s", cudaGetErrorString(e));
  unsigned int word = 0;
  e = cudaMemcpyFromSymbol(&word, g_dev_error_word, sizeof(word));
  if (e != cudaSuccess) return fail(TSP_ERR_CUDA, "reading device error word: %s", cudaGetErrorString(e));
  if (word) {
    const unsigned int zero = 0;
    cudaMemcpyToSymbol(g_dev_error_word, &zero, sizeof(zero));
    return fail(TSP_ERR_TIMEOUT, "device wait gave up (kernel %u, site %u)", word >> 8, word & 0xFF);
  }
  return TSP_OK;
}

}  // extern "C"
