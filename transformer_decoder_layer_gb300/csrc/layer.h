// The layer handle, the packed-weight and workspace layouts, and the internal
// entry points of the prefill / decode / MoE orchestration.
#pragma once

#include <cstddef>
#include <cstdint>

#include "internal.h"

namespace qwen {

struct PackedLayout {
  size_t status, rope, rope_t, gamma_attn, gamma_mlp, gamma_q, gamma_k, w_qkv, b_qkv, w_o, w_gu, w_down,
      w_router, b_router, w_sgu, w_sdown, total;
};

struct WorkspaceLayout {
  size_t xh, q, k16, v16, attn, r32, z, h;
  // MoE
  size_t logits, topk_idx, topk_w, blk_counts, offsets, act, perm, inv, zp, hp, yp;
  // MoE shared expert: H_s [M][sf] FP16, its output [M][d] FP32, gate g [M]
  size_t hs, ys32, gscale;
  // decode (T == 1)
  size_t part, attn_o, attn_ml;
  size_t total;
  // the regions above in layout order, named (qwen_layer_workspace_regions)
  struct Region {
    const char* name;
    size_t off, bytes;
  };
  static constexpr int kMaxRegions = 32;
  Region reg[kMaxRegions];
  int n_reg;
};

}  // namespace qwen

struct qwen_layer_s {
  qwen_layer_config cfg;
  uint8_t* packed;
  qwen::PackedLayout L;
  int* status;
  float2* rope;    // [max_position][dh/2] (cos, sin)
  float2* rope_t;  // the same table frequency-major, [dh/2][max_position]
  __nv_bfloat16 *gamma_attn, *gamma_mlp, *gamma_q, *gamma_k;
  // projection weights are held as FP16 (converted exactly from BF16 at create)
  __half* w_qkv;
  float* b_qkv;
  __half* w_o;
  __half *w_gu, *w_down;  // gate/up rows interleaved in 64-row blocks
  // router weights as FP16 [router_rows][2d], each row twice ([W_r | W_r]):
  // the logits are one GEMM over [Z_hi | Z_lo] (Z split into two FP16 parts).
  // With a shared expert, row E holds its gate column W_sg (rows E+1.. are
  // zero), so logit E is the shared gate's pre-activation.
  __half* w_router;
  float* b_router;
  // shared expert: gate/up interleaved like w_gu, FP16 [2sf][d]; down [d][sf]
  __half *w_sgu, *w_sdown;
  // optional per-stage events (qwen_layer_set_trace)
  bool tracing = false;
  void* trace[2 * QWEN_STAGE_COUNT] = {};
};

namespace qwen {

bool config_valid(const qwen_layer_config& c);
// Rows of the router GEMM: E, plus 8 (the shared gate and zero padding) when
// the layer has a shared expert.
inline int router_rows(const qwen_layer_config& c) {
  return c.n_experts + (c.shared_ffn > 0 ? 8 : 0);
}
PackedLayout packed_layout(const qwen_layer_config& c);
WorkspaceLayout workspace_layout(const qwen_layer_config& c, int B, int T);

QkvParams make_qkv_params(const qwen_layer_s* L, const int32_t* positions, const int32_t* slot0,
                          void* q, bool q_f16, __nv_bfloat16* kc, __nv_bfloat16* vc,
                          __half* k16, __half* v16, int T);

// x (BF16) or x32 (FP32) is the input; y (BF16) and/or y32 (FP32) the output.
qwen_status layer_prefill(qwen_layer_s* L, const __nv_bfloat16* x, const float* x32,
                          __nv_bfloat16* y, float* y32, int B, int T, const int32_t* positions,
                          const int32_t* slot0, __nv_bfloat16* kc, __nv_bfloat16* vc,
                          uint8_t* ws, const WorkspaceLayout& W, cudaStream_t st);

qwen_status layer_decode(qwen_layer_s* L, const __nv_bfloat16* x, const float* x32,
                         __nv_bfloat16* y, float* y32, int B, const int32_t* positions,
                         const int32_t* cache_len, __nv_bfloat16* kc, __nv_bfloat16* vc,
                         uint8_t* ws, const WorkspaceLayout& W, cudaStream_t st);

// MoE block: residual input r (BF16) or r32 (FP32); output y (BF16) and/or y32.
// z_ready: the workspace already holds [Z_hi | Z_lo] = RMSNorm_2(R) (the decode
// step fuses the norm into the O projection's split reduction).
qwen_status moe_forward(qwen_layer_s* L, const __nv_bfloat16* r, const float* r32,
                        __nv_bfloat16* y, float* y32, int T, int32_t* topk_idx_out,
                        float* topk_w_out, float* logits_out, uint8_t* ws,
                        const WorkspaceLayout& W, cudaStream_t st, bool z_ready = false);

// ---- decode building blocks (decode_gemm.cu, attention_decode.cu)

// Number of K splits the swap-AB decode GEMM uses for an [N, K] weight (or for
// `groups` such weights in grouped mode) and B tokens.
int decode_splits(int N, int K, int B, int groups = 1);
// MoE blocks on at most this many tokens run the experts through the grouped
// swap-AB decode GEMM (the tokens sit on the MMA's N side, padded to 16..64).
constexpr int kMoeDecodeMaxRows = 64;
// Bytes of FP32 partials the decode GEMM of the layer needs for batch B.
size_t decode_part_bytes(const qwen_layer_config& c, int B);

// Expert GEMMs with the weights on the MMA's M side (moe_gemm.cu): W a packed
// blocked stack [E][Nw][K], X the routed rows [rows][K] grouped by expert
// (rows [offsets[e], offsets[e+1]) for expert e, offsets on the device).
// swiglu: W interleaves gate and up rows in 64-row blocks and out = H [rows]
// [Nw / 2] = SiLU(gate) * up; else out = X W_e^T [rows][Nw].  FP16 out, row
// stride ldo.  Supported when Nw % 256 == 0, K % 64 == 0 and E <= 256.
bool gemm_expert_supported(int E, int Nw, int K);
qwen_status gemm_expert(const __half* W, int E, int Nw, int K, const __half* X, int rows, int ldx,
                        const int32_t* offsets, __half* out, int ldo, bool swiglu, int* err,
                        cudaStream_t st);

// CTAs of the MoE permutation for `entries` (token, slot) pairs (1024 each).
int moe_perm_blocks(size_t entries);
// Attention split-KV plan: number of splits per (sequence, KV head) for batch B.
void decode_attn_plan(const qwen_layer_config& c, int B, int* splits);

// part[s][b][n] = sum over split s's k-range of W[n, k] X[b, k].
// W [N, K], X [B, K] (row stride ldx).
// w_packed: W is a packed layer weight: stored in the blocked layout (128 x 64
// tiles, rows padded to 128) and never written by the kernel launched just
// before, so its first tiles may be fetched before waiting on it.  Otherwise
// W is row-major [N, K] (the caller's lm_head).
// swiglu_out: W is an interleaved gate/up weight (64-row blocks); run with one
// split and write H[b][f] = SiLU(gate) * up (FP16) instead of partials.
// late_release: the kernel lets the kernels after it launch only once its
// threads have passed their dependency wait (not at its start): everything
// enqueued before the kernel before it has then completed.
qwen_status gemm_decode_splitk(const void* W, const void* X, int ldx, int B, int N, int K,
                               int splits, bool op_f16, float* part, int* err, cudaStream_t st,
                               bool w_packed = false, __half* swiglu_out = nullptr,
                               bool late_release = false);

// Grouped (mixture-of-experts) decode GEMM.  W: E stacked FP16 [N, K] weights;
// X: `rows` FP16 rows of K, grouped by expert: rows [offsets[e], offsets[e+1])
// belong to expert e (offsets [E + 1], device).  act (device): [0] = number of
// non-empty experts (at most max_groups), then their ids.  No expert has more
// than max_m rows.  Output: part[s][row][N] FP32 partials, or with swiglu_out
// (one split, W interleaved gate/up) H[row][N/2] = SiLU(gate) * up as FP16.
qwen_status gemm_decode_grouped(const void* W, int E, const void* X, int rows, int max_m, int N,
                                int K, int splits, const int32_t* act, const int32_t* offsets,
                                int max_groups, float* part, __half* swiglu_out, int* err,
                                cudaStream_t st);

// Token mode of the grouped decode GEMM for an interleaved gate/up stack W
// [E][N][K]: X = the T token rows (ldx apart); for each non-empty expert e in
// act, H[inv[t*k + j]] = SiLU(gate) * up of token t wherever idx[t*k + j] == e
// (H rows N/2 wide, FP16).
qwen_status gemm_decode_grouped_tokens(const void* W, int E, const void* X, int ldx, int T,
                                       int N, int K, const int32_t* act, const int32_t* idx,
                                       const int32_t* inv, int k, int max_groups, __half* h_out,
                                       int* err, cudaStream_t st);

// Reductions over the splits followed by the step's epilogue.
qwen_status reduce_resid(const float* part, int splits, int B, int N, const __nv_bfloat16* resid,
                         const float* resid32, __nv_bfloat16* out, float* out32, cudaStream_t st);
// R = sum of splits + residual (FP32, out32), then Z = RMSNorm(R) (FP16, rows
// z_stride apart, 0 = N).  With z_lo the FP16 rounding residual of Z is written
// there as well (same row stride): the [Z_hi | Z_lo] operand of the router.
// Z values beyond the FP16 range are stored saturated and recorded in *err as
// QWEN_ERR_OVERFLOW (as are H values in reduce_swiglu).
qwen_status reduce_resid_norm(const float* part, int splits, int B, int N,
                              const __nv_bfloat16* resid, const float* resid32, float* out32,
                              const __nv_bfloat16* gamma, float eps, __half* z, int* err,
                              cudaStream_t st, size_t z_stride = 0, __half* z_lo = nullptr);
qwen_status reduce_swiglu(const float* part, int splits, int B, int f, __half* h, int* err,
                          cudaStream_t st);
qwen_status reduce_qkv(const float* part, int splits, int B, int Nqkv, const QkvParams& p,
                       int* err, cudaStream_t st);
qwen_status reduce_f32(const float* part, int splits, int B, int N, float* out, int ldo,
                       cudaStream_t st);

// Split-KV decode attention and its merge: q [B][Hq][dh]; query b sits in cache
// slot cache_len[b] and attends slots 0..cache_len[b].  out [B][Hq*dh].
// early: an earlier kernel of the step released its dependents only after its
// own dependency wait, so all work enqueued before the step has completed and
// the attention may load cache rows below slot cache_len[b] without waiting.
qwen_status attention_decode(const __nv_bfloat16* q, const __nv_bfloat16* kc,
                             const __nv_bfloat16* vc, const int32_t* cache_len, int B, int Hq,
                             int Hkv, int dh, int max_seq, int splits, float* part_o,
                             float* part_ml, __half* out, int* err, cudaStream_t st,
                             bool early = false);

}  // namespace qwen
