// Internal declarations shared by the libtsp translation units.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>

#include "../../include/tsp.h"

struct tsp_plan {
  int D;
  int64_t seq;
  int hidden;
  int heads;
  int kv_heads;  // K/V heads (== heads for multi-head attention, fewer for grouped-query attention)
  int head_dim;
  int ffn;
  tsp_dtype dtype;
  int64_t chunk;  // seq / (2D)
  int deterministic = 0;  // backward: split dK/dV and dQ kernels (bitwise reproducible) instead of the fused one
};

namespace tsp {

// Epilogues of the projection GEMMs (C = A * B^T, A [M][K], B [N][K]).
enum EpiKind : int {
  EPI_STORE = 0,    // out[m][n] = acc
  EPI_RESID = 1,    // out[m][n] = resid[m][n] + acc
  EPI_QKV = 2,      // scatter packed Q|K|V columns: Q to zigzag rows, K/V gathered per K/V head
  EPI_SWIGLU = 3,   // gate/up 128-column blocks -> out[m][f] = SiLU(g) * u; optional raw copy to aux
  EPI_DSWIGLU = 4,  // acc = dM[m][f]; reads saved G/U (resid, packed gate_up order) -> dGU to out
};

struct EpiParams {
  void* out = nullptr;
  int64_t ldo = 0;
  const void* resid = nullptr;
  int64_t ldr = 0;
  void* aux = nullptr;
  int64_t ldx = 0;
  void* q = nullptr;
  void* k = nullptr;
  void* v = nullptr;
  int D = 1, B = 1, S = 0, C = 0, H = 1, dh = 1, h = 0;
  int Hk = 1;                   // EPI_QKV: K/V heads; a shard's packed columns are Q (h/D) | K (Hk*dh/D) | V
  unsigned int* err = nullptr;  // device error word
  bool v_transposed = false;    // EPI_QKV: write V as [B][Hk][dh][S] instead of [B][Hk][S][dh]
  // Zigzag row m <-> natural row remapping (uses D, B, S, C; needs C % 128 == 0):
  //   a_natural:     the A operand is natural-order rows; tile rows of zigzag
  //                  rows m0.. are read from natural row nat(m0)..
  //   resid_natural: EPI_RESID reads resid row nat(m)
  //   out_natural:   EPI_RESID writes out row nat(m)
  bool a_natural = false, resid_natural = false, out_natural = false;
  // EPI_STORE: columns n >= split_col (> 0, a multiple of 32) go to aux[m][n - split_col]
  // (row stride ldx) instead of out -- two outputs of one GEMM that shares its A operand.
  int64_t split_col = 0;
};

int num_sms();
// One-time setup per device (kernel attributes such as the dynamic shared-memory
// limit are per device): needs_setup() is true until mark_setup_done() has been
// called on the current device.  Devices 0..63.
bool needs_setup(const std::atomic<unsigned long long>& done);
void mark_setup_done(std::atomic<unsigned long long>& done);
// Records `msg` as this thread's tsp_last_error_message() and returns `s`.
tsp_status report_error(tsp_status s, const char* msg);
// TSP_OK if `stream` belongs to the current device; TSP_ERR_INVALID_ARG (with a
// message naming both devices) if not, TSP_ERR_CUDA if either cannot be read.
tsp_status check_stream_device(void* stream, const char* what);
unsigned int* dev_error_word();  // device address of this device's error word (nullptr on failure)

// bf16 tcgen05 GEMM: C[M][N] = sum_k A[m][k] B[n][k] with fp32 accumulation in
// tensor memory.  A is stored [M][K] (row stride lda), or with a_mn [K][M]
// (row stride lda, M contiguous); likewise B [N][K] or, with b_mn, [K][N].
// Needs N % 256 == 0, K % 64 == 0 (and M % 64 == 0 with a_mn), 16-byte
// aligned rows.
tsp_status gemm_bf16_tc(const void* A, int64_t lda, const void* B, int64_t ldb, int M, int N, int K,
                        EpiKind epi, const EpiParams& ep, cudaStream_t stream, bool a_mn = false,
                        bool b_mn = false);

// 2-D bf16 TMA descriptor: row-major [rows][cols], row stride ld elements,
// box = 64 columns x box_rows rows, 128-byte swizzle.
bool make_tma_2d_bf16(CUtensorMap* m, const void* base, int64_t rows, int64_t cols, int64_t ld, int box_rows);

// fp32 SIMT GEMM, same contract (any M, N, K; SWIGLU/DSWIGLU not supported).
tsp_status gemm_f32_simt(const float* A, int64_t lda, const float* B, int64_t ldb, int M, int N, int K,
                         EpiKind epi, const EpiParams& ep, cudaStream_t stream);

// Elementwise / layout kernels.
cudaError_t launch_zigzag_rows(const void* src, void* dst, int64_t row_bytes, int D, int B, int64_t S,
                               bool to_zigzag, cudaStream_t stream);
cudaError_t launch_kv_gather(const void* kz, const void* vz, void* k, void* v, int elem_bytes, int D, int B,
                             int64_t S, int H, int dh, cudaStream_t stream);
// The same with source rows src_ld elements apart (a multiple of 16 bytes);
// ntens 1 gathers K only (vz and v unused).
cudaError_t launch_kv_gather_ld(const void* kz, const void* vz, void* k, void* v, int elem_bytes, int D, int B,
                                int64_t S, int H, int dh, int64_t src_ld, cudaStream_t stream, int ntens = 2);
// 16-bit V of zigzag rows [T][ld] (head e at columns v_col0 + e*dh) -> vt
// [B][H][dh][S] in natural positions; needs seq/(2D) % 64 == 0 and dh % 64 == 0.
cudaError_t launch_kv_gather_vt(const void* src, int64_t ld, int64_t v_col0, void* vt, int D, int B, int64_t S,
                                int H, int dh, cudaStream_t stream);
// 2-D copy of `rows` rows of row_bytes (pitches and row_bytes multiples of 16).
cudaError_t launch_copy_rows(const void* src, int64_t src_pitch_bytes, void* dst, int64_t dst_pitch_bytes,
                             int64_t rows, int64_t row_bytes, cudaStream_t stream);
cudaError_t launch_swiglu_f32(const float* gu, float* m, int64_t T, int F, cudaStream_t stream);
cudaError_t launch_transpose(const void* src, void* dst, int64_t rows, int64_t cols, int elem_bytes,
                             cudaStream_t stream, int batch = 1);
cudaError_t launch_pack_weights(const tsp_plan* p, const void* const c[7], const tsp_weight_grads* w, bool unpack,
                                cudaStream_t stream);

// Attention.
// Query head `head` reads K/V head head / (H / Hk) (grouped-query attention;
// Hk == H is multi-head attention).
struct AttnParams {
  const void* q;  // zigzag rows [T][h]
  const void* k;  // [B][Hk][S][dh]
  const void* v;
  void* o;        // zigzag rows [T][h]
  float* lse;     // [B][H][S] natural log, may be null
  int D, B, H, dh;
  int64_t S, C;
  int Hk;
  // -1: the queries of every rank.  r >= 0: only rank r's queries; q and o
  // then hold just that rank's zigzag rows ([B][2C][H*dh], row b*2C + k).
  int rank = -1;
  // Optional scratch for the tcgen05 kernel's key split (attn_tc_split_bytes):
  // used, with lse NULL, when the grid would not fill the GPU once.
  void* split_ws = nullptr;
  size_t split_ws_bytes = 0;
};
tsp_status attn_fwd_bf16(const AttnParams& p, cudaStream_t stream);
tsp_status attn_fwd_f32(const AttnParams& p, cudaStream_t stream);
// tcgen05 attention (V given transposed, [B][Hk][dh][S]); needs head_dim 128 and chunk % 128 == 0.
bool attn_tc_supported(int head_dim, int64_t chunk);
tsp_status attn_fwd_bf16_tc(const AttnParams& p, cudaStream_t stream);
// Scratch bytes of the tcgen05 kernel's two-way key split for `rows` query rows of H heads.
size_t attn_tc_split_bytes(int64_t rows, int H);

struct AttnBwdParams {
  const void* q;   // zigzag [T][h]
  const void* k;   // [B][H][S][dh] (multi-head attention only)
  const void* v;
  const void* o;   // zigzag [T][h]
  const void* dO;  // zigzag [T][h]
  const float* lse;
  float* dsum;     // [B][H][S] scratch
  void* dq;        // zigzag [T][h]
  void* dk;        // [B][H][S][dh]
  void* dv;
  int D, B, H, dh;
  int64_t S, C;
};
tsp_status attn_bwd_bf16(const AttnBwdParams& p, cudaStream_t stream);
// dsum[b][head][p] = rowsum(dO * O) (fp32), the softmax-Jacobian row term of the backward.
// dq_zero (optional): an fp32 [B][H][S][dh] buffer zeroed in the same pass.
cudaError_t launch_attn_dsum(const void* o, const void* dO, float* dsum, int D, int B, int H, int64_t S, int64_t C,
                             cudaStream_t stream, float* dq_zero = nullptr);

// tcgen05 attention backward (head_dim 128, chunk % 128 == 0).
struct AttnBwdTcArgs {
  const void* q;    // zigzag [T][h]
  const void* k;    // [B][Hk][S][dh]
  const void* v;    // [B][Hk][S][dh]
  const void* dO;   // zigzag [T][h]
  const float* lse;
  const float* dsum;
  float* dq_acc;    // [B][H][S][dh] fp32, unscaled sum of dS K (1/sqrt(dh) is applied when assembled);
                    // the fused kernel adds into it (zero it first), the dQ kernel overwrites it
  void* dk;         // [B][Hk][S][dh]: summed over the query heads that read the K/V head
  void* dv;
  int D, B, H, dh;
  int64_t S, C;
  int Hk;
};
bool attn_bwd_tc_supported(int head_dim, int64_t chunk);
// which: 1 = the dK/dV kernel, 2 = the dQ kernel (3 = both: bitwise reproducible),
// 4 = the fused dK/dV/dQ kernel (dQ summed with fp32 L2 reductions).
tsp_status attn_bwd_bf16_tc(const AttnBwdTcArgs& a, cudaStream_t stream, int which = 3);

// Backward helpers.
// dqkv [T][h + 2*Hk*dh] in the packed column order <- dq zigzag [T][h], dk/dv [B][Hk][S][dh].
cudaError_t launch_assemble_dqkv(const void* dq, const void* dk, const void* dv, void* dqkv, int D, int B,
                                 int64_t S, int H, int Hk, int dh, cudaStream_t stream);
// The same with dQ taken from the tensor-core backward's fp32 accumulator
// [B][H][S][dh] (times `scale`) instead of a bf16 zigzag [T][h] buffer.
cudaError_t launch_assemble_dqkv_f32q(const float* dq_acc, float scale, const void* dk, const void* dv, void* dqkv,
                                      int D, int B, int64_t S, int H, int Hk, int dh, cudaStream_t stream);

// Decode step (bf16; batch 1..8; head_dim 128; H / Hk in {1, 2, 4, 8}).
size_t decode_ws_bytes(const tsp_plan* p, int batch);
int decode_split(int D, int H, int Hk, int B, int64_t C);
tsp_status decode_step_bf16(const tsp_plan* p, int batch, int64_t pos, const void* x_new, const tsp_weights* w,
                            void* k_cache, void* v_cache, void* y_new, void* ws, cudaStream_t st);

// Optional per-step timing (tsp_profile_*): CUDA events around enqueued work,
// summed per name.  No-ops unless profiling is enabled; calls nest like braces.
void prof_begin(const char* name, cudaStream_t st);
void prof_end(cudaStream_t st);

}  // namespace tsp
