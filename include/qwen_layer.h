/*
 * qwen_layer.h -- C ABI of a GB300 (sm_103a) forward pass of one Qwen-style
 * pre-norm decoder layer, dense or mixture-of-experts, prefill or decode.
 *
 * What is computed (sources cited by page title and section):
 *   R = X + Attention(RMSNorm_1(X)),  Y = R + MLP(RMSNorm_2(R))
 *   -- "推理系统 03：逐项算清一个真实 Qwen3 Transformer 层" (Qwen3 layer page), §2.
 *   RMSNorm: gamma * x / sqrt(mean(x^2) + eps), mean square in FP32 (§3).
 *   Q/K/V = X^ W^T (+ b) with weights stored [out, in] (§4; "Qwen2.5-7B 结构拆解"
 *   §03.1, §04 for the qkv bias).  Qwen3 QK-norm: RMSNorm over dh of every Q
 *   and K head with one shared gamma each (§5).  RoPE with the rotate_half
 *   pairing (i, i + dh/2), omega_r = theta^(-2r/dh) (§6).  GQA: query head h
 *   reads KV head floor(h / (Hq/Hkv)) (§7).  Scores / sqrt(dh) + causal mask,
 *   stable softmax, P V, head concat, O projection, residual (§8, §9).
 *   SwiGLU MLP: (SiLU(Z Wg^T) * (Z Wu^T)) Wd^T (§10).  KV cache: K (after
 *   QK-norm and RoPE) and V of every position, appended ("Qwen2.5-7B 结构拆解"
 *   §09.1; Qwen3 layer page §12).  MoE: router logits z Wr^T (+ per-expert
 *   bias), top-k, softmax over the k selected logits (or, Qwen2-MoE, the
 *   selected entries of the softmax over all E), weighted sum of SwiGLU
 *   experts, plus an optional shared SwiGLU expert scaled per token by
 *   sigmoid(z W_sg) ("Qwen2.5-7B 结构拆解" §10.1, §10.2; "MoE 初步" lecture,
 *   Router / Expert sections).
 *
 * Conventions shared by every entry point:
 *   - Every tensor argument is a DEVICE pointer unless marked "host".  BF16
 *     tensors are IEEE bfloat16, row-major, densely packed, 16-byte aligned.
 *   - The caller allocates every device buffer (packed weights, workspace, KV
 *     cache, inputs, outputs).  The library never allocates device memory and
 *     never synchronises inside prefill/decode/moe/head; work is enqueued on
 *     `stream` (a cudaStream_t passed as void*, NULL = legacy default stream).
 *   - Host-checkable problems (bad shapes, NULL pointers, capacity) return an
 *     error before anything is launched.  Device-side range problems (a cache
 *     slot >= max_seq, a position >= max_position, a bounded wait that ran
 *     out) set a sticky status word that qwen_layer_poll_error returns.
 *   - The tensor-core operands inside a layer are FP16 (weights converted from
 *     BF16 at create; normalised activations, attention output and the SwiGLU
 *     product H rounded to FP16).  FP16 stops at 65504: a weight of larger
 *     magnitude makes qwen_layer_create fail with QWEN_ERR_OVERFLOW, and an
 *     activation that would round past it (or is NaN) is stored as +-65504
 *     and sets QWEN_ERR_OVERFLOW in the status word.  Results are never
 *     silently infinite.
 *   - Only head_dim 64 or 128, d % 64 == 0, ffn % 64 == 0 and Hq % Hkv == 0
 *     are supported on the GPU; anything else returns QWEN_ERR_UNSUPPORTED.
 *     There is no CPU fallback.
 */
#ifndef QWEN_LAYER_H_
#define QWEN_LAYER_H_

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define QWEN_API __attribute__((visibility("default")))
#else
#define QWEN_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  QWEN_OK = 0,
  QWEN_ERR_INVALID_ARG = 1, /* NULL pointer, bad size, bad config value      */
  QWEN_ERR_UNSUPPORTED = 2, /* shape the GPU kernels do not implement        */
  QWEN_ERR_CAPACITY = 3,    /* B, T or buffer larger than the handle allows   */
  QWEN_ERR_CUDA = 4,        /* a CUDA runtime/driver call failed             */
  QWEN_ERR_TIMEOUT = 5,     /* device: a bounded wait ran out                */
  QWEN_ERR_RANGE = 6,       /* device: cache slot or position out of range   */
  QWEN_ERR_OVERFLOW = 7     /* a value beyond the FP16 operand range: a weight
                               at create, or (device) an activation written as
                               an FP16 GEMM operand                           */
} qwen_status;

/* Layer shape and capacities.  Plain data, validated by qwen_layer_create. */
typedef struct {
  int32_t d;            /* hidden size                                         */
  int32_t n_q_heads;    /* Hq                                                  */
  int32_t n_kv_heads;   /* Hkv (Hq % Hkv == 0)                                 */
  int32_t head_dim;     /* dh: 64 or 128                                       */
  int32_t ffn;          /* f (dense) or per-expert width mf (MoE); % 64 == 0   */
  int32_t qkv_bias;     /* 1: Q/K/V projections carry a bias                   */
  int32_t qk_norm;      /* 1: Qwen3 per-head RMSNorm on Q and K                */
  double rope_theta;    /* RoPE base, 1e6 for the Qwen configurations          */
  float rms_eps;        /* epsilon of every RMSNorm (also QK-norm)             */
  int32_t n_experts;    /* E; 0 = dense MLP; else a multiple of 8, <= 248     */
  int32_t top_k;        /* k experts per token (MoE)                           */
  int32_t norm_topk_prob; /* 1: gate weights = softmax over the k selected
                           * logits; 0: the selected entries of the softmax over
                           * all E logits, as they are (Qwen2-MoE)             */
  int32_t router_bias;  /* 1: per-expert FP32 bias added to the router logits  */
  int32_t max_tokens;   /* capacity: largest B*T of one prefill call           */
  int32_t max_batch;    /* capacity: largest B of one call                     */
  int32_t max_seq;      /* KV cache slots per sequence                         */
  int32_t max_position; /* RoPE table length: positions must be < this         */
  int32_t shared_ffn;   /* sf: width of the shared expert (MoE only); 0 = none;
                         * else % 64 == 0                                       */
} qwen_layer_config;

/* Source weights (device, BF16, [out, in] row-major) handed to create.  NULL
 * where the config says absent.  Dense: w_gate/w_up [f, d], w_down [d, f].
 * MoE: w_gate/w_up [E, mf, d], w_down [E, d, mf], w_router [E, d] BF16,
 * b_router [E] FP32.  Shared expert (shared_ffn = sf > 0): w_shared_gate and
 * w_shared_up [sf, d], w_shared_down [d, sf], w_shared_expert_gate [d] (the
 * one-column gate W_sg, no bias), all BF16.  The library copies them into its
 * packed buffer; the caller may free these after the stream passed to create
 * has synchronised. */
typedef struct {
  const void* gamma_attn; /* [d]   RMSNorm_1 gamma                       */
  const void* gamma_mlp;  /* [d]   RMSNorm_2 gamma                       */
  const void* gamma_q;    /* [dh]  QK-norm gamma for Q (qk_norm)         */
  const void* gamma_k;    /* [dh]  QK-norm gamma for K (qk_norm)         */
  const void* w_q;        /* [Hq*dh, d]                                  */
  const void* w_k;        /* [Hkv*dh, d]                                 */
  const void* w_v;        /* [Hkv*dh, d]                                 */
  const void* b_q;        /* [Hq*dh]  (qkv_bias)                         */
  const void* b_k;        /* [Hkv*dh] (qkv_bias)                         */
  const void* b_v;        /* [Hkv*dh] (qkv_bias)                         */
  const void* w_o;        /* [d, Hq*dh]                                  */
  const void* w_gate;
  const void* w_up;
  const void* w_down;
  const void* w_router;   /* MoE only                                    */
  const float* b_router;  /* MoE with router_bias                        */
  const void* w_shared_gate;        /* [sf, d]  (shared_ffn)             */
  const void* w_shared_up;          /* [sf, d]  (shared_ffn)             */
  const void* w_shared_down;        /* [d, sf]  (shared_ffn)             */
  const void* w_shared_expert_gate; /* [d]      (shared_ffn)             */
} qwen_layer_weights;

typedef struct qwen_layer_s* qwen_layer_t;

/* Human-readable name of a status code (static string). */
QWEN_API const char* qwen_status_string(qwen_status s);

/* Bytes of the caller-allocated packed-weight buffer for `cfg` (includes the
 * FP32 RoPE cos/sin table and the device status word).  0 if cfg is invalid. */
QWEN_API size_t qwen_layer_packed_bytes(const qwen_layer_config* cfg);

/* Bytes of scratch a prefill of B sequences x T tokens (decode: T = 1) needs,
 * for qwen_layer_prefill / qwen_layer_decode / qwen_moe_ffn with the same
 * B*T.  The workspace is caller-owned device memory, 256-byte aligned, and
 * holds only transient values: it may be reused across calls on one stream. */
QWEN_API size_t qwen_layer_workspace_bytes(const qwen_layer_config* cfg, int32_t B, int32_t T);

/* One region of a layer workspace: a name, its byte offset and its size. */
typedef struct qwen_workspace_region {
  const char* name; /* static string owned by the library */
  size_t offset;
  size_t bytes;
} qwen_workspace_region;

/* The regions the library places in a workspace for (B, T) under `cfg`, in
 * layout order.  Host only: no device is touched.  Writes up to
 * `max_regions` entries to `out` (which may be NULL when max_regions is 0)
 * and returns the number of regions, or -1 when cfg is invalid, B or T is not
 * positive, or out is NULL with max_regions > 0.  Offsets are 256-byte
 * aligned, regions do not overlap, and each ends at or before
 * qwen_layer_workspace_bytes(cfg, B, T).  For inspection and tests; the
 * kernels use exactly these offsets. */
QWEN_API int32_t qwen_layer_workspace_regions(const qwen_layer_config* cfg, int32_t B, int32_t T,
                                              qwen_workspace_region* out, int32_t max_regions);

/* Validate cfg, pack the weights into `packed` (device, packed_bytes as
 * returned above, 256-byte aligned), build the RoPE table and return a handle.
 * Enqueues the packing on `stream` and synchronises it before returning.
 * The handle (host memory, owned by the library) remembers `packed`, which
 * must outlive the handle.  Returns QWEN_ERR_OVERFLOW, and no handle, when a
 * projection, expert or router weight is too large for FP16 (it would round
 * to infinity; |w| >= 65520). */
QWEN_API qwen_status qwen_layer_create(const qwen_layer_config* cfg, const qwen_layer_weights* w,
                              void* packed, size_t packed_bytes, void* stream,
                              qwen_layer_t* out);

/* Release the handle (host memory only; `packed` stays the caller's). */
QWEN_API void qwen_layer_destroy(qwen_layer_t layer);

/* Prefill: the full layer over B sequences of T new tokens each.
 *   x, y        [B, T, d] BF16 (y may not alias x)
 *   positions   [B*T] int32, RoPE positions (< max_position)
 *   cache_start [B] int32: sequence b's tokens go to cache slots
 *               cache_start[b] + t; query slot s sees cache slots <= s.
 *   k_cache, v_cache [B, Hkv, max_seq, dh] BF16, updated in place.
 * Dense layers run the SwiGLU MLP; MoE layers run qwen_moe_ffn's path.   */
QWEN_API qwen_status qwen_layer_prefill(qwen_layer_t layer, const void* x, void* y, int32_t B,
                               int32_t T, const int32_t* positions, const int32_t* cache_start,
                               void* k_cache, void* v_cache, void* workspace,
                               size_t workspace_bytes, void* stream);

/* Decode: one new token per sequence.
 *   x, y      [B, d] BF16;  positions [B] int32;
 *   cache_len [B] int32: number of filled slots; the new K/V row is written
 *             to slot cache_len[b] and the query attends slots 0..cache_len[b].
 *   k_cache, v_cache as for prefill.                                       */
QWEN_API qwen_status qwen_layer_decode(qwen_layer_t layer, const void* x, void* y, int32_t B,
                              const int32_t* positions, const int32_t* cache_len,
                              void* k_cache, void* v_cache, void* workspace,
                              size_t workspace_bytes, void* stream);

/* The same two calls with the residual stream in FP32 across calls (the
 * hidden state a stack of layers passes from layer to layer): exactly one of
 * x (BF16) / x_fp32 (FP32, [B, T, d] resp. [B, d]) is the input, and y (BF16)
 * and/or y_fp32 (FP32) receive the output (at least one non-NULL; y_fp32 may
 * not alias x_fp32).  Rounding the hidden state to BF16 between layers is the
 * dominant error of a deep stack; keeping it in FP32 removes it. */
QWEN_API qwen_status qwen_layer_prefill_ex(qwen_layer_t layer, const void* x, const float* x_fp32,
                                           void* y, float* y_fp32, int32_t B, int32_t T,
                                           const int32_t* positions, const int32_t* cache_start,
                                           void* k_cache, void* v_cache, void* workspace,
                                           size_t workspace_bytes, void* stream);
QWEN_API qwen_status qwen_layer_decode_ex(qwen_layer_t layer, const void* x, const float* x_fp32,
                                          void* y, float* y_fp32, int32_t B,
                                          const int32_t* positions, const int32_t* cache_len,
                                          void* k_cache, void* v_cache, void* workspace,
                                          size_t workspace_bytes, void* stream);

/* One decode step with the inputs and the output in HOST memory (the call a
 * serving loop makes): x_host (BF16 [B, d]), positions_host and
 * cache_len_host (int32 [B]) in, y_host (BF16 [B, d]) out.  When all four are
 * pinned host memory mapped for the device, the step's kernels read the inputs
 * and write the output through the host link directly (no copies between
 * kernels); otherwise the inputs are copied to staging space inside the
 * workspace, the step runs, and y is copied back, all enqueued on `stream`.
 * Nothing synchronises: the caller synchronises the stream before reading
 * y_host or changing the host inputs.  The workspace must hold
 * qwen_layer_host_workspace_bytes(cfg, B).  Errors as qwen_layer_decode, plus
 * QWEN_ERR_CUDA if a copy cannot be enqueued. */
QWEN_API size_t qwen_layer_host_workspace_bytes(const qwen_layer_config* cfg, int32_t B);
QWEN_API qwen_status qwen_layer_decode_host(qwen_layer_t layer, const void* x_host, void* y_host,
                                            int32_t B, const int32_t* positions_host,
                                            const int32_t* cache_len_host, void* k_cache,
                                            void* v_cache, void* workspace,
                                            size_t workspace_bytes, void* stream);

/* MoE block alone on T tokens: Y = R + sum_j w_j Expert_{idx_j}(Z)
 * [+ sigmoid(Z W_sg) SharedExpert(Z)],  Z = RMSNorm_2(R).
 *   r        [T, d] BF16 residual-stream input; y [T, d] BF16 output.
 *   r_fp32   optional [T, d] FP32 copy of r used for the norm and router
 *            (NULL: r is widened from BF16).
 *   topk_idx optional [T, k] int32, topk_w optional [T, k] FP32,
 *   logits   optional [T, E] FP32 router logits (outputs for inspection).  */
QWEN_API qwen_status qwen_moe_ffn(qwen_layer_t layer, const void* r, const float* r_fp32, void* y,
                         int32_t T, int32_t* topk_idx, float* topk_w, float* logits,
                         void* workspace, size_t workspace_bytes, void* stream);

/* Bytes of scratch qwen_head_last_token needs for B sequences of width d. */
QWEN_API size_t qwen_head_workspace_bytes(int32_t B, int32_t d, int32_t V);

/* Final RMSNorm + lm_head on the last position of each sequence
 * ("Qwen2.5-7B 结构拆解" §03.8): logits[b] = RMSNorm(y[b, T-1]) W_lm^T.
 *   y [B, T, d] BF16; gamma_final [d] BF16; w_lm [V, d] BF16;
 *   logits [B, V] FP32.                                                   */
QWEN_API qwen_status qwen_head_last_token(const void* y, int32_t B, int32_t T, int32_t d,
                                 const void* gamma_final, const void* w_lm, int32_t V,
                                 float eps, float* logits, void* workspace,
                                 size_t workspace_bytes, void* stream);

/* qwen_head_last_token without a workspace, for callers that cannot allocate
 * device memory at call time (for example a server that has committed all of
 * its HBM to a fixed arena, or a loop where an allocation would synchronise
 * the device).  The pages have no counterpart: this is a library convenience.
 * Same arguments and result as qwen_head_last_token minus the workspace.  The
 * normalised last rows (B * d BF16 values) live in a 2 MiB device array inside
 * the library, held on every GPU that loads it until the process exits:
 * B * d * 2 must be <= 2 MiB (e.g. B = 256 at d = 4096, B = 128 at d = 8192)
 * and B <= 256, else QWEN_ERR_CAPACITY.  The array's device address is looked
 * up on the first call made on each device (make that first call before any
 * stream capture) and kept until the process exits, so the device must not be
 * reset (cudaDeviceReset) between calls.  All calls share the array: calls
 * that overlap on the GPU race on it.  Nothing is allocated or freed. */
QWEN_API qwen_status qwen_head_last_token_noalloc(const void* y, int32_t B, int32_t T, int32_t d,
                                                  const void* gamma_final, const void* w_lm,
                                                  int32_t V, float eps, float* logits,
                                                  void* stream);

/* One RMSNorm pass (the layer's norm step on its own, Qwen3 layer page §3):
 *   y[r] = gamma * x[r] / sqrt(mean(x[r]^2) + eps), rows x d, BF16 in/out,
 *   optional FP32 copy of y (y_fp32 may be NULL).  d % 8 == 0.            */
QWEN_API qwen_status qwen_rmsnorm(const void* x, const void* gamma, void* y, float* y_fp32,
                         int32_t rows, int32_t d, float eps, void* stream);

/* Plain projection y = x W^T on the tensor cores ("Qwen2.5-7B 结构拆解"
 * §03.1-03.2): x [M, K] BF16, w [N, K] BF16, y [M, N] BF16, FP32 accumulate.
 * K % 8 == 0, N % 8 == 0.                                                 */
QWEN_API qwen_status qwen_linear(const void* x, const void* w, void* y, int32_t M, int32_t N,
                        int32_t K, void* stream);

/* Stages of one prefill / decode call, in launch order (a call runs the
 * stages its path needs; the *_FINISH stages are the decode path's split-K
 * reductions, ATTN_MERGE its split-KV merge). */
typedef enum {
  QWEN_STAGE_NORM1 = 0,
  QWEN_STAGE_QKV = 1,
  QWEN_STAGE_QKV_FINISH = 2,
  QWEN_STAGE_ATTN = 3,
  QWEN_STAGE_ATTN_MERGE = 4,
  QWEN_STAGE_O = 5,
  QWEN_STAGE_O_FINISH = 6,
  QWEN_STAGE_NORM2 = 7,
  QWEN_STAGE_GATE_UP = 8,
  QWEN_STAGE_GATE_UP_FINISH = 9,
  QWEN_STAGE_DOWN = 10,
  QWEN_STAGE_DOWN_FINISH = 11,
  QWEN_STAGE_MOE = 12, /* the whole MoE block of a MoE layer */
  QWEN_STAGE_COUNT = 13
} qwen_stage;

/* Optional per-stage timing.  `events` (host array of 2 * QWEN_STAGE_COUNT
 * cudaEvent_t handles, entries may be NULL) is remembered by the handle; every
 * later prefill/decode call records events[2*s] on its stream right before
 * stage s and events[2*s+1] right after it, for each stage it runs and each
 * non-NULL entry.  Pass events = NULL to stop.  The array must stay valid
 * until tracing is switched off. */
QWEN_API qwen_status qwen_layer_set_trace(qwen_layer_t layer, void* const* events);

/* Number of kernel launches this library has issued in this process (all
 * handles, all entry points); a host-side counter. */
QWEN_API uint64_t qwen_launch_count(void);

/* Synchronise `stream`, then read and clear the handle's device status word.
 * Returns QWEN_OK, QWEN_ERR_TIMEOUT, QWEN_ERR_RANGE or QWEN_ERR_OVERFLOW (or
 * QWEN_ERR_CUDA); the first error recorded since the last poll wins. */
QWEN_API qwen_status qwen_layer_poll_error(qwen_layer_t layer, void* stream);

/* Synchronise `stream`, then read and clear the library-wide device status
 * word that the handle-less entry points (qwen_rmsnorm, qwen_linear,
 * qwen_head_last_token) record into. */
QWEN_API qwen_status qwen_poll_error(void* stream);

/* Number of SMs of the current CUDA device (1 if it cannot be queried). */
QWEN_API int32_t qwen_device_sm_count(void);

#ifdef __cplusplus
}
#endif

#endif /* QWEN_LAYER_H_ */
