/*
 * tsp.h -- C ABI of libtsp: one transformer layer computed the TSP way
 * (Tensor and Sequence Parallelism folded onto one axis of size D) on one
 * GPU (sm_103a), with the D ranks emulated as token and weight partitions in
 * device memory.
 *
 * The method (ai-trends.today, "Zyphra Introduces Tensor and Sequence
 * Parallelism (TSP)", section "How to Fold a Book"; edge.aivizor.me TSP
 * news post, paragraph on layer execution):
 *   - every rank holds 1/D of the tokens (zigzag: the sequence is cut into
 *     2D chunks, rank r holds chunk r then chunk 2D-1-r) and 1/D of the
 *     weights;
 *   - attention iterates over packed {W_Q, W_K, W_V, W_O} shards: each rank
 *     projects its local tokens, local K/V are all-gathered and put in zigzag
 *     order, causal FlashAttention runs, and the W_O partial products are
 *     accumulated locally;
 *   - the gated MLP is a ring over gate/up/down shards; each rank accumulates
 *     its partial outputs, so there is no output all-reduce.
 * On one GPU the broadcast becomes a loop over shards and the ring becomes
 * the K-loop of one GEMM whose accumulator never leaves tensor memory.
 *
 * Layer computed (row-vector convention y = x W; no norm, bias or position
 * term; softmax scale 1/sqrt(head_dim); key j visible to query i iff j <= i
 * in global positions):
 *     A = Attn(x Wq, x Wk, x Wv) Wo,   H = x + A,
 *     M = SiLU(H Wg) * (H Wu),         Y = H + M Wd.
 *
 * Conventions for every call
 *   - All tensor pointers are DEVICE pointers owned by the caller; the
 *     library never allocates device memory.  Scratch comes from the caller
 *     as a workspace of tsp_workspace_bytes() bytes.
 *   - Element type is the plan's dtype (fp32 or bf16) unless stated; lse is
 *     always fp32.  Every pointer must be 16-byte aligned.
 *   - `stream` is a cudaStream_t (NULL = legacy default stream) of the
 *     CURRENT device (cudaSetDevice): the library's per-device state (error
 *     word, static scratch, kernel set-up) is looked up for the current
 *     device, so a stream of another device is refused with
 *     TSP_ERR_INVALID_ARG before anything is enqueued.  Calls only enqueue
 *     work; they return before it runs.
 *   - Arguments are validated on the host before any launch; an invalid call
 *     enqueues nothing and returns a status.  A launch failure returns
 *     TSP_ERR_CUDA.  Kernels never trap: a device-side wait that exceeds its
 *     bound records an error word and returns; tsp_sync_check() reports it
 *     as TSP_ERR_TIMEOUT.
 *   - tsp_last_error_message() gives a thread-local description of the last
 *     non-OK status.
 *   - batch = 0 (no tokens) is valid for every call that takes a batch of
 *     sequences except tsp_decode_step: it returns TSP_OK, reads no pointer
 *     and enqueues nothing; the workspace and saved sizes for it are 0.
 *
 * Grouped-query attention (plans from tsp_plan_create_gqa): K and V have
 * Hk <= H heads, Wk and Wv are [h][hk] with hk = Hk * head_dim, and query
 * head e reads K/V head e / (H / Hk).  The r007 chapter (section
 * "Параллелизм по контексту: Ring Attention против Ulysses") names GQA, with
 * the K/V head count often cut to 8, as what bounds a head split; here a
 * weight shard owns H/D query heads and Hk/D K/V heads, so Hk % D == 0.
 * Multi-head attention is the case Hk == H.
 *
 * Layouts (T = batch * seq tokens, C = seq / (2D), h = heads * head_dim,
 * hk = kv_heads * head_dim, equal to h for multi-head attention)
 *   natural   x[b][p][h]               (row b*seq + p)
 *   zigzag    xz[r][b][k][h]            (row (r*batch + b)*2C + k) holding
 *             natural position pos(r,k) = r*C + k for k < C, and
 *             (2D-1-r)*C + (k-C) for k >= C
 *   gathered  K[b][kv_head][p][head_dim], V likewise (natural positions)
 *   lse       lse[b][head][p] fp32: natural log of sum_j exp(score_pj)
 *   packed weights (each row holds one output column, contiguous over the
 *   input dimension, i.e. the transposed weight, ready as a K-major operand):
 *     qkv     [h+2hk][h]: for shard s = 0..D-1: the Q columns of query
 *             heads s*H/D .. (s+1)*H/D-1 (h/D rows), then the K, then the
 *             V columns of K/V heads s*Hk/D .. (s+1)*Hk/D-1 (hk/D rows each);
 *     o       [h][h]:  row n = column n of W_O (input rows of shard s are
 *             input indices s*h/D .. (s+1)*h/D-1);
 *     gate_up [2F][h]: blocks of 256 rows; block j holds gate columns
 *             j*128 .. j*128+127 then up columns j*128 .. j*128+127;
 *     down    [h][F]:  row n = column n of W_down.
 */
#ifndef TSP_H
#define TSP_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  TSP_OK = 0,
  TSP_ERR_INVALID_ARG = 1, /* null/misaligned pointer, bad size, shape rule broken */
  TSP_ERR_UNSUPPORTED = 2, /* valid layer, but no kernel for this shape/dtype */
  TSP_ERR_CUDA = 3,        /* a CUDA runtime/launch error */
  TSP_ERR_TIMEOUT = 4,     /* a bounded device-side wait gave up */
  TSP_ERR_WORKSPACE = 5    /* workspace or saved buffer too small */
} tsp_status;

typedef enum { TSP_F32 = 0, TSP_BF16 = 1 } tsp_dtype;

typedef enum {
  TSP_OP_ATTENTION_FWD = 0,
  TSP_OP_GATED_MLP_FWD = 1,
  TSP_OP_LAYER_FWD = 2,
  TSP_OP_LAYER_BWD = 3,
  TSP_OP_DECODE = 4,
  TSP_OP_RANK_ATTENTION = 5, /* tsp_rank_attention */
  TSP_OP_RANK_MLP = 6        /* tsp_rank_mlp */
} tsp_op;

/* The two kinds of weight shard that travel between ranks in a multi-GPU TSP
 * layer (tsp_rank_*). */
typedef enum { TSP_SHARD_ATTENTION = 0, TSP_SHARD_MLP = 1 } tsp_shard_kind;

/* Opaque and host-only.  Configure it (tsp_plan_set_deterministic) before
 * sharing it; from then on it is read-only and safe to share between threads. */
typedef struct tsp_plan tsp_plan;

/* Packed weights (device pointers, layouts above). */
typedef struct {
  const void* qkv;
  const void* o;
  const void* gate_up;
  const void* down;
} tsp_weights;

/* Packed weight gradients, same layouts as tsp_weights (written, not accumulated). */
typedef struct {
  void* qkv;
  void* o;
  void* gate_up;
  void* down;
} tsp_weight_grads;

/* ---- plan and sizes (host only; no CUDA call is made) -------------------- */

/* Validates and records the layer shape.  Rules: D >= 1; seq % (2D) == 0;
 * heads % D == 0; ffn % D == 0; hidden == heads * head_dim; head_dim in
 * {32, 64, 128}; hidden % 8 == 0; ffn % 128 == 0.  The bf16 kernels further
 * need hidden % 256 == 0, ffn % 256 == 0 and head_dim == 128, else calls return
 * TSP_ERR_UNSUPPORTED.  *out receives a new plan (free with tsp_plan_destroy). */
tsp_status tsp_plan_create(int D, int64_t seq, int hidden, int heads, int head_dim, int ffn,
                           tsp_dtype dtype, tsp_plan** out);
/* The same with grouped-query attention: kv_heads K/V heads shared by the
 * `heads` query heads (consecutive groups of heads/kv_heads).  Extra rules:
 * kv_heads >= 1, heads % kv_heads == 0, kv_heads % D == 0 (TSP_ERR_INVALID_ARG
 * otherwise).  tsp_layer_bwd of such a plan also needs seq/(2D) % 128 == 0
 * (TSP_ERR_UNSUPPORTED otherwise).  kv_heads == heads gives tsp_plan_create. */
tsp_status tsp_plan_create_gqa(int D, int64_t seq, int hidden, int heads, int kv_heads, int head_dim, int ffn,
                               tsp_dtype dtype, tsp_plan** out);
void tsp_plan_destroy(tsp_plan* plan);
/* Attention backward algorithm of tsp_layer_bwd (tensor-core path: bf16,
 * head_dim 128, seq/(2D) % 128 == 0).  0 (the default): one fused kernel per
 * 128-key tile computes dK, dV and the tile's share of dQ, and the shares are
 * summed with fp32 reductions in L2, whose order varies, so dQ -- and dx and
 * the Q rows of dW_QKV through it -- can differ in the last bits from run to
 * run.  1: separate dK/dV and dQ kernels (the dQ kernel recomputes the scores
 * and dP), slower but bitwise reproducible.  Anything else:
 * TSP_ERR_INVALID_ARG.  Not thread-safe: call before the plan is shared. */
tsp_status tsp_plan_set_deterministic(tsp_plan* plan, int deterministic);
/* The setting above (0 or 1), or -1 for a NULL plan. */
int tsp_plan_get_deterministic(const tsp_plan* plan);

/* Workspace bytes needed by `op` for `batch` sequences (0 on invalid input). */
size_t tsp_workspace_bytes(const tsp_plan* plan, int batch, tsp_op op);
/* Bytes of the activation buffer tsp_layer_fwd saves for tsp_layer_bwd. */
size_t tsp_saved_bytes(const tsp_plan* plan, int batch);

const char* tsp_status_string(tsp_status s);
const char* tsp_last_error_message(void);

/* ---- weight packing (bit-exact reindex) ---------------------------------- */

/* canonical[7] = {Wq, Wk, Wv, Wo [h][h], Wg, Wu [h][F], Wd [F][h]}, row-major
 * with y = x W.  Writes the four packed tensors of `packed`. */
tsp_status tsp_pack_weights(const tsp_plan* plan, const void* const canonical[7],
                            const tsp_weight_grads* packed, void* stream);
/* Inverse of tsp_pack_weights (also maps packed gradients back). */
tsp_status tsp_unpack_weights(const tsp_plan* plan, const tsp_weights* packed,
                              void* const canonical[7], void* stream);

/* ---- zigzag token partition (bit-exact) ---------------------------------- */

/* x natural [batch][seq][h] -> xz zigzag [D][batch][2C][h]. */
tsp_status tsp_zigzag_permute(const tsp_plan* plan, int batch, const void* x, void* xz, void* stream);
/* xz zigzag -> x natural. */
tsp_status tsp_zigzag_unpermute(const tsp_plan* plan, int batch, const void* xz, void* x, void* stream);
/* The K/V all-gather with zigzag reorder: kz, vz zigzag [D][batch][2C][hk]
 * (head-major columns) -> k, v gathered [batch][kv_heads][seq][head_dim]. */
tsp_status tsp_kv_gather(const tsp_plan* plan, int batch, const void* kz, const void* vz,
                         void* k, void* v, void* stream);

/* ---- layer pieces ---------------------------------------------------------- */

/* Attention half on zigzag tokens: a_out = Attn(xz Wq, xz Wk, xz Wv) Wo (no
 * residual), zigzag [D][batch][2C][h].  Uses weights->qkv and weights->o.
 * lse (fp32 [batch][heads][seq]) may be NULL. */
tsp_status tsp_attention_fwd(const tsp_plan* plan, int batch, const void* xz,
                             const tsp_weights* weights, void* a_out, void* lse,
                             void* workspace, size_t workspace_bytes, void* stream);

/* Gated-MLP ring on zigzag tokens: m_out = (SiLU(hz Wg) * (hz Wu)) Wd (no
 * residual).  Uses weights->gate_up and weights->down. */
tsp_status tsp_gated_mlp_fwd(const tsp_plan* plan, int batch, const void* hz,
                             const tsp_weights* weights, void* m_out,
                             void* workspace, size_t workspace_bytes, void* stream);

/* Whole layer, natural order in and out: y = H + MLP(H), H = x + A.
 * If `saved` is non-NULL (tsp_saved_bytes bytes) the activations tsp_layer_bwd
 * needs are kept there. */
tsp_status tsp_layer_fwd(const tsp_plan* plan, int batch, const void* x, const tsp_weights* weights,
                         void* y, void* saved, void* workspace, size_t workspace_bytes,
                         void* stream);

/* Gradient of the layer: given x, weights, the `saved` buffer of the matching
 * tsp_layer_fwd and dy (natural), writes dx (natural) and every packed weight
 * gradient.  bf16 plans only (fp32 returns TSP_ERR_UNSUPPORTED). */
tsp_status tsp_layer_bwd(const tsp_plan* plan, int batch, const void* x, const tsp_weights* weights,
                         const void* saved, const void* dy, void* dx, const tsp_weight_grads* dw,
                         void* workspace, size_t workspace_bytes, void* stream);

/* ---- decoding ---------------------------------------------------------------- */

/* One decode step: each of `batch` sequences (1..8) holds `pos` cached tokens
 * (positions 0..pos-1) and appends x_new[b] at position `pos` (0 <= pos <
 * seq; the plan's seq is the cache capacity).  The step writes the new
 * token's key and value into row `pos` of the caches and y_new[b] = the
 * layer's output for that token, which attends to positions 0..pos.
 *   x_new, y_new      [batch][h] bf16
 *   k_cache, v_cache  [batch][kv_heads][seq][head_dim] bf16, natural positions;
 *                     rows >= pos are not read (row pos is overwritten)
 * TSP reading (ai-trends.today TSP article: the scheme serves inference as
 * well as training): the cache is sharded over the D virtual ranks by the
 * zigzag rule, each rank computes a partial softmax of the new query over
 * its own cached positions, and the partials are merged by log-sum-exp; the
 * projections stream every packed weight shard once.  bf16 plans only,
 * head_dim 128, heads / kv_heads in {1, 2, 4, 8} (else TSP_ERR_UNSUPPORTED);
 * workspace: tsp_workspace_bytes(plan, batch, TSP_OP_DECODE). */
tsp_status tsp_decode_step(const tsp_plan* plan, int batch, int64_t pos, const void* x_new,
                           const tsp_weights* weights, void* k_cache, void* v_cache, void* y_new,
                           void* workspace, size_t workspace_bytes, void* stream);

/* ---- one rank of a multi-GPU TSP layer ------------------------------------ */
/*
 * The calls above run all D ranks of a layer on one GPU.  The calls below are
 * ONE rank's compute steps of the same layer when each of D GPUs is a rank
 * and holds 1/D of the tokens and 1/D of the weights (ai-trends.today TSP
 * article, "How to Fold a Book"); the exchanges between them (broadcast of an
 * attention shard by its owner, all-gather of K/V, the MLP ring) are the
 * caller's, e.g. NCCL.  Every pointer is local device memory of the calling
 * rank's GPU: a shard that came from another rank has already been received
 * into a local buffer.  Rank r's layer, with x_r its local zigzag rows:
 *
 *   H_r = x_r;  for s = 0..D-1 (owner s broadcasts attention shard s):
 *       tsp_rank_qkv(x_r, shard s)          -> q_r, kv_r
 *       all-gather kv_r over the ranks      -> kv_all (rank order)
 *       tsp_rank_attention(rank r, q_r, kv_all, shard s, resid = H_r) -> H_r
 *   Y_r = H_r;  for t = 0..D-1, j = (r - t) mod D (the ring; at t = 0 the
 *       rank's own MLP shard, then the one received from rank r-1):
 *       tsp_rank_mlp(H_r, shard j, resid = Y_r) -> Y_r
 *
 * after which Y_r equals rows of rank r of tsp_layer_fwd's output (zigzag
 * rows (r*batch + b)*2C + k) up to rounding.  There is no output all-reduce.
 *
 * Local layouts (L = batch * 2C local rows, row b*2C + k holding natural
 * position pos(r, k) of sequence b; hs = h/D, ks = hk/D, fs = ffn/D):
 *   x_r, H_r, Y_r [L][h];  q_r [L][hs];  kv_r [L][2*ks] (the shard's K
 *   columns then its V columns);  kv_all [D][L][2*ks] (rank r' at r'*L rows).
 * Shard layouts (one contiguous buffer each, tsp_rank_shard_bytes bytes):
 *   attention shard s:  qkv_s [hs + 2*ks][h]  = rows of packed qkv for shard
 *                       s (Q columns of its H/D heads, then K, then V), then
 *                       o_s [h][hs] with o_s[n][i] = W_O[s*hs + i][n];
 *   MLP shard j:        gu_j [2*fs][h] = rows j*2*fs .. of packed gate_up
 *                       (its 128-column gate/up blocks), then
 *                       down_j [h][fs] with down_j[n][i] = W_down[j*fs + i][n].
 * Shape rules on top of the plan's: ffn/D % 128 == 0 (a shard holds whole
 * gate/up blocks); for bf16 also hidden/D % 256 == 0 and 2*kv_hidden/D % 256
 * == 0 (TSP_ERR_UNSUPPORTED otherwise).
 */

/* Bytes of one shard of `kind` in the layout above (0 for a NULL plan). */
size_t tsp_rank_shard_bytes(const tsp_plan* plan, tsp_shard_kind kind);

/* Writes shard `shard` (0..D-1) of `kind` from the whole packed weights into
 * `out` (tsp_rank_shard_bytes bytes): what the rank owning that shard holds. */
tsp_status tsp_rank_extract_shard(const tsp_plan* plan, const tsp_weights* packed, int shard, tsp_shard_kind kind,
                                  void* out, void* stream);

/* Projection of the rank's tokens by one attention shard: q_r = x_r Wq_s,
 * kv_r = x_r [Wk_s | Wv_s] (kv_r is what the rank contributes to the K/V
 * all-gather). */
tsp_status tsp_rank_qkv(const tsp_plan* plan, int batch, const void* x_local, const void* attn_shard,
                        void* q_local, void* kv_local, void* stream);

/* Causal attention of rank `rank`'s queries (its H/D heads of the shard) over
 * the gathered K/V of every rank, then h_out = resid + O_s Wo_s.  kv_all is
 * reordered into natural positions inside the call.  resid may equal h_out
 * (accumulation in place); resid NULL means 0.  Workspace:
 * tsp_workspace_bytes(plan, batch, TSP_OP_RANK_ATTENTION). */
tsp_status tsp_rank_attention(const tsp_plan* plan, int rank, int batch, const void* q_local, const void* kv_all,
                              const void* attn_shard, const void* resid, void* h_out, void* workspace,
                              size_t workspace_bytes, void* stream);

/* One step of the MLP ring: y_out = resid + (SiLU(H_r Wg_j) * (H_r Wu_j)) Wd_j.
 * resid may equal y_out (in place); NULL means 0.  Workspace:
 * tsp_workspace_bytes(plan, batch, TSP_OP_RANK_MLP). */
tsp_status tsp_rank_mlp(const tsp_plan* plan, int batch, const void* h_local, const void* mlp_shard,
                        const void* resid, void* y_out, void* workspace, size_t workspace_bytes, void* stream);

/* ---- status ---------------------------------------------------------------- */

/* Synchronizes `stream`, then reports a pending CUDA error (TSP_ERR_CUDA) or a
 * device-side wait that gave up (TSP_ERR_TIMEOUT, error word cleared). */
tsp_status tsp_sync_check(void* stream);

/* Host-side fault injection for tests: the next `count` tsp_* compute calls on
 * this thread return `status` before enqueuing anything (count 0 disarms). */
void tsp_debug_fail_next(tsp_status status, int count);

/* Failure-detection check: enqueues a one-warp kernel whose bounded wait on a
 * barrier that nothing signals gives up after `timeout_us` microseconds
 * (1 us .. 10 s), records the device error word and returns; the next
 * tsp_sync_check on that stream reports TSP_ERR_TIMEOUT and clears the word.
 * Nothing traps; the context stays usable. */
tsp_status tsp_debug_wait_timeout(unsigned int timeout_us, void* stream);

/* ---- attention without a caller workspace -------------------------------- */

/* Size of the static scratch array behind tsp_attention_fwd_static. */
#define TSP_STATIC_SCRATCH_BYTES (32u << 20)

/* Same computation and arguments as tsp_attention_fwd, minus the workspace:
 * for callers that cannot allocate device memory (a plug-in inside a host
 * application that owns all device allocations, or a latency-critical loop
 * that must not call cudaMalloc, which can synchronize the device).  The
 * scratch (Q, K, V, O) lives in one static device array of
 * TSP_STATIC_SCRATCH_BYTES that every GPU loading the library holds until
 * the library is unloaded; the call allocates and frees nothing.
 * - A batch whose tsp_workspace_bytes(plan, batch, TSP_OP_ATTENTION_FWD)
 *   exceeds TSP_STATIC_SCRATCH_BYTES is rejected with TSP_ERR_WORKSPACE
 *   before anything is enqueued.
 * - All calls share the array: calls whose GPU work overlaps (other streams,
 *   unordered host threads) race and corrupt each other; order them.  Each
 *   call writes all the scratch it reads, so nothing needs clearing.
 * - The first call on a device looks up the array's address on that device
 *   (cudaGetSymbolAddress, with the device current); make it before any
 *   stream capture starts.
 * The TSP posts have no counterpart of this entry point. */
tsp_status tsp_attention_fwd_static(const tsp_plan* plan, int batch, const void* xz,
                                    const tsp_weights* weights, void* a_out, void* lse, void* stream);

/* ---- measurement ----------------------------------------------------------- */

/* Per-step timing for measurement (off by default).  While enabled, every
 * kernel step a tsp_* call enqueues is bracketed by two CUDA events on the
 * call's stream (a small gap between kernels).  Thread-safe. */
void tsp_profile_enable(int on);
/* Waits for the recorded events, then writes up to max_entries rows of
 * (step name, total milliseconds, launch count) aggregated by name in
 * first-seen order; names point to static strings of the library.  Returns
 * the number of distinct names and clears the records. */
int tsp_profile_report(const char** names, double* total_ms, int* counts, int max_entries);

#ifdef __cplusplus
}
#endif

#endif /* TSP_H */
