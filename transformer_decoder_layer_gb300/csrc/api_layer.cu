// C ABI of the layer handle: validation, weight packing, workspace layout and
// the orchestration of prefill / decode / MoE on the caller's stream.
//
// Layer structure, Qwen3 layer page ("推理系统 03"), §2:
//   R = X + Attention(RMSNorm_1(X)),  Y = R + MLP(RMSNorm_2(R)).
#include <cmath>
#include <cstring>
#include <new>
#include <vector>

#include "common.cuh"
#include "internal.h"
#include "layer.h"

namespace qwen {

static size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }
static size_t round128(size_t x) { return (x + 127) & ~static_cast<size_t>(127); }

bool config_valid(const qwen_layer_config& c) {
  if (c.d <= 0 || c.d % 64 || c.d > 8192) return false;
  if (c.n_q_heads <= 0 || c.n_kv_heads <= 0 || c.n_q_heads % c.n_kv_heads) return false;
  if (c.n_q_heads / c.n_kv_heads > 16) return false;
  if (c.head_dim != 64 && c.head_dim != 128) return false;
  if (c.ffn <= 0 || c.ffn % 64) return false;
  if (!(c.rope_theta > 0.0) || !(c.rms_eps >= 0.f)) return false;
  if (c.qkv_bias != 0 && c.qkv_bias != 1) return false;
  if (c.qk_norm != 0 && c.qk_norm != 1) return false;
  // the router is one tensor-core GEMM with N = E (a multiple of 8), and the
  // grouped expert GEMM schedules at most 248 groups
  if (c.n_experts < 0 || c.n_experts > 248 || (c.n_experts & 7)) return false;
  if (c.n_experts > 0) {
    if (c.top_k < 1 || c.top_k > 8 || c.top_k > c.n_experts) return false;
    if (c.norm_topk_prob != 0 && c.norm_topk_prob != 1) return false;
  }
  // shared expert: MoE layers only, width a multiple of 64 (SwiGLU tiles)
  if (c.shared_ffn < 0 || c.shared_ffn % 64) return false;
  if (c.shared_ffn > 0 && c.n_experts == 0) return false;
  if (c.max_tokens <= 0 || c.max_batch <= 0 || c.max_seq <= 0 || c.max_position <= 0) return false;
  return true;
}

PackedLayout packed_layout(const qwen_layer_config& c) {
  PackedLayout L{};
  const size_t d = c.d, dh = c.head_dim, nq = (size_t)c.n_q_heads * dh,
               nkv = (size_t)c.n_kv_heads * dh, nqkv = nq + 2 * nkv, f = c.ffn;
  size_t o = 0;
  auto take = [&](size_t bytes) {
    const size_t at = o;
    o = align256(o + bytes);
    return at;
  };
  L.status = take(256);
  L.rope = take((size_t)c.max_position * (dh / 2) * sizeof(float2));
  L.rope_t = take((size_t)c.max_position * (dh / 2) * sizeof(float2));
  L.gamma_attn = take(d * 2);
  L.gamma_mlp = take(d * 2);
  L.gamma_q = take(dh * 2);
  L.gamma_k = take(dh * 2);
  // FP16 weights in the blocked layout: every matrix (every expert's) rows
  // padded to a multiple of 128
  L.b_qkv = take(nqkv * 4);
  L.w_qkv = take(round128(nqkv) * d * 2);
  L.w_o = take(round128(d) * nq * 2);
  if (c.n_experts == 0) {
    L.w_gu = take(2 * f * d * 2);
    L.w_down = take(round128(d) * f * 2);
  } else {
    const size_t e = c.n_experts;
    L.b_router = take(e * 4);
    L.w_router = take(round128(router_rows(c)) * 2 * d * 2);  // rows [W_r | W_r]
    L.w_gu = take(e * 2 * f * d * 2);
    L.w_down = take(e * round128(d) * f * 2);
    if (c.shared_ffn) {
      const size_t sf = c.shared_ffn;
      L.w_sgu = take(2 * sf * d * 2);
      L.w_sdown = take(round128(d) * sf * 2);
    }
  }
  L.total = o;
  return L;
}

WorkspaceLayout workspace_layout(const qwen_layer_config& c, int B, int T) {
  WorkspaceLayout W{};
  const size_t M = (size_t)B * T, d = c.d, dh = c.head_dim, nq = (size_t)c.n_q_heads * dh,
               f = c.ffn;
  size_t o = 0;
  auto take = [&](const char* name, size_t bytes) {
    const size_t at = o;
    o = align256(o + bytes);
    if (W.n_reg < WorkspaceLayout::kMaxRegions) W.reg[W.n_reg++] = {name, at, bytes};
    return at;
  };
  W.xh = take("xh", M * d * 2);
  W.q = take("q", M * nq * 2);
  // FP16 copies of the call's K/V rows for the prefill attention.  Laid out for
  // every T: a prefill of one token per sequence uses this (B, 1) layout too,
  // and its copies must not share memory with each other or with X-hat.
  W.k16 = take("k16", M * (size_t)c.n_kv_heads * dh * 2);
  W.v16 = take("v16", M * (size_t)c.n_kv_heads * dh * 2);
  W.attn = take("attn", M * nq * 2);
  W.r32 = take("r32", M * d * 4);  // residual stream R kept in FP32
  // MoE: Z rows are [Z_hi | Z_lo] (2d FP16), the router's split-precision operand
  W.z = take("z", M * d * 2 * (c.n_experts ? 2 : 1));
  if (c.n_experts == 0) {
    W.h = take("h", M * f * 2);
  } else {
    const size_t e = c.n_experts, k = c.top_k, mk = M * k;
    W.logits = take("logits", M * (size_t)router_rows(c) * 4);
    W.topk_idx = take("topk_idx", mk * 4);
    W.topk_w = take("topk_w", mk * 4);
    W.blk_counts = take("blk_counts", moe_perm_blocks(mk) * e * 4);
    W.offsets = take("offsets", (e + 1) * 4);
    W.act = take("act", (e + 1) * 4);
    W.perm = take("perm", mk * 4);
    W.inv = take("inv", mk * 4);
    W.zp = take("zp", mk * d * 2);
    W.hp = take("hp", mk * f * 2);
    W.yp = take("yp", mk * d * 2);
    if (c.shared_ffn) {
      W.hs = take("hs", M * (size_t)c.shared_ffn * 2);
      W.ys32 = take("ys32", M * d * 4);
      W.gscale = take("gscale", M * 4);
    }
  }
  if (T == 1) {
    int splits = 0;
    decode_attn_plan(c, B, &splits);
    W.part = take("part", decode_part_bytes(c, B));
    W.attn_o = take("attn_o", (size_t)B * c.n_q_heads * splits * dh * 4);
    W.attn_ml = take("attn_ml", (size_t)B * c.n_q_heads * splits * 2 * 4);
  }
  W.total = o;
  return W;
}

// ------------------------------------------------------------- packing

__global__ void bf16_to_f32_kernel(const bf16* __restrict__ src, float* __restrict__ dst, int n) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < n) dst[i] = __bfloat162float(src[i]);
}

static bool copy_d2d(void* dst, const void* src, size_t bytes, cudaStream_t st) {
  return cudaMemcpyAsync(dst, src, bytes, cudaMemcpyDeviceToDevice, st) == cudaSuccess;
}

// Copy BF16 weight rows into the packed FP16 buffer.  BF16 -> FP16 is exact
// for magnitudes in [2^-14, 65504] (FP16 keeps more mantissa bits); smaller
// magnitudes land on the FP16 subnormal grid (absolute error <= 2^-25).  A
// weight that FP16 cannot hold (it would round to infinity) records
// QWEN_ERR_OVERFLOW in *err and qwen_layer_create fails.
//
// Destination: the blocked layout, a [rows][dst_cols] matrix stored as 128 x 64
// tiles of 16 KB, tile (row / 128, col / 64) at ((row/128) * dst_cols/64 +
// col/64) * 16 KB, row-major inside the tile.  Weight tiles then stream as
// whole contiguous 16 KB blocks (measured ~6% faster HBM streaming than 128
// rows of 128 bytes each from a row-major matrix).
// Row placement: source row r belongs to group r / gsz (an expert); inside a
// group, mode 0 keeps the row order and modes 1 and 2 interleave gate (1) and
// up (2) rows in 64-row blocks, block 2i = gate block i and block 2i+1 = up
// block i, so one GEMM tile holds both halves of every SwiGLU output feature;
// group g starts at destination row roff + g * gpad.  Columns go to coff + c.
__global__ void pack_blocked_f16_kernel(f16* __restrict__ dst, const bf16* __restrict__ src,
                                        size_t rows, int cols, int mode, size_t gsz, size_t gpad,
                                        size_t roff, int dst_cols, int coff, int* err) {
  const int cpr = cols / 8;  // 16-byte chunks per source row
  const size_t nch = rows * (size_t)cpr;
  const size_t kt = (size_t)dst_cols / 64;
  bool bad = false;
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < nch;
       i += (size_t)gridDim.x * blockDim.x) {
    const size_t r = i / cpr;
    const int c = (int)(i - r * cpr);
    const size_t g = r / gsz, rin = r - g * gsz;
    const size_t din = mode == 0 ? rin : (rin / 64) * 128 + (rin % 64) + (mode == 2 ? 64 : 0);
    const size_t dr = roff + g * gpad + din;
    const size_t dc = (size_t)coff + 8 * (size_t)c;
    const size_t off = (((dr / 128) * kt + dc / 64) * 128 + dr % 128) * 64 + dc % 64;
    const uint4 u = reinterpret_cast<const uint4*>(src)[i];
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
    uint32_t o[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float2 f = unpack_bf16x2(w[j]);
      o[j] = pack_f16x2_chk(f.x, f.y, bad);
    }
    *reinterpret_cast<uint4*>(dst + off) = make_uint4(o[0], o[1], o[2], o[3]);
  }
  record_overflow(err, bad);
}

// BF16 [rows][cols] -> blocked FP16 (see pack_blocked_f16_kernel); gsz = 0:
// one group; dst_cols = 0: cols.
static bool pack_blocked(f16* dst, const void* src, size_t rows, size_t cols, int mode, int* err,
                         cudaStream_t st, size_t gsz = 0, size_t gpad = 0, size_t roff = 0,
                         size_t dst_cols = 0, size_t coff = 0) {
  if (rows == 0) return true;
  const size_t nch = rows * (cols / 8);
  const int blocks = (int)((nch + 255) / 256 < 65535 ? (nch + 255) / 256 : 65535);
  pack_blocked_f16_kernel<<<blocks, 256, 0, st>>>(dst, static_cast<const bf16*>(src), rows,
                                                  (int)cols, mode, gsz ? gsz : rows, gpad, roff,
                                                  (int)(dst_cols ? dst_cols : cols), (int)coff,
                                                  err);
  count_launches();
  return cudaGetLastError() == cudaSuccess;
}

}  // namespace qwen

using namespace qwen;

extern "C" {

size_t qwen_layer_packed_bytes(const qwen_layer_config* cfg) {
  if (!cfg || !config_valid(*cfg)) return 0;
  return packed_layout(*cfg).total;
}

size_t qwen_layer_workspace_bytes(const qwen_layer_config* cfg, int32_t B, int32_t T) {
  if (!cfg || !config_valid(*cfg) || B <= 0 || T <= 0) return 0;
  return workspace_layout(*cfg, B, T).total;
}

int32_t qwen_layer_workspace_regions(const qwen_layer_config* cfg, int32_t B, int32_t T,
                                     qwen_workspace_region* out, int32_t max_regions) {
  if (!cfg || !config_valid(*cfg) || B <= 0 || T <= 0 || max_regions < 0) return -1;
  if (max_regions > 0 && !out) return -1;
  const WorkspaceLayout W = workspace_layout(*cfg, B, T);
  for (int i = 0; i < W.n_reg && i < max_regions; ++i)
    out[i] = {W.reg[i].name, W.reg[i].off, W.reg[i].bytes};
  return W.n_reg;
}

qwen_status qwen_layer_create(const qwen_layer_config* cfg, const qwen_layer_weights* w,
                              void* packed, size_t packed_bytes, void* stream,
                              qwen_layer_t* out) {
  if (!cfg || !w || !packed || !out) return QWEN_ERR_INVALID_ARG;
  *out = nullptr;
  if (!config_valid(*cfg)) {
    if (cfg->head_dim != 64 && cfg->head_dim != 128 && cfg->head_dim > 0)
      return QWEN_ERR_UNSUPPORTED;
    return QWEN_ERR_INVALID_ARG;
  }
  const qwen_layer_config& c = *cfg;
  const PackedLayout L = packed_layout(c);
  if (packed_bytes < L.total) return QWEN_ERR_CAPACITY;
  if (reinterpret_cast<uintptr_t>(packed) & 255) return QWEN_ERR_INVALID_ARG;
  const bool moe = c.n_experts > 0;
  if (!w->gamma_attn || !w->gamma_mlp || !w->w_q || !w->w_k || !w->w_v || !w->w_o ||
      !w->w_gate || !w->w_up || !w->w_down)
    return QWEN_ERR_INVALID_ARG;
  if (c.qk_norm && (!w->gamma_q || !w->gamma_k)) return QWEN_ERR_INVALID_ARG;
  if (c.qkv_bias && (!w->b_q || !w->b_k || !w->b_v)) return QWEN_ERR_INVALID_ARG;
  if (moe && (!w->w_router || (c.router_bias && !w->b_router))) return QWEN_ERR_INVALID_ARG;
  if (c.shared_ffn && (!w->w_shared_gate || !w->w_shared_up || !w->w_shared_down ||
                       !w->w_shared_expert_gate))
    return QWEN_ERR_INVALID_ARG;

  cudaStream_t st = static_cast<cudaStream_t>(stream);
  uint8_t* P = static_cast<uint8_t*>(packed);
  const size_t d = c.d, dh = c.head_dim, nq = (size_t)c.n_q_heads * dh,
               nkv = (size_t)c.n_kv_heads * dh, f = c.ffn;

  qwen_layer_s* h = new (std::nothrow) qwen_layer_s();
  if (!h) return QWEN_ERR_CAPACITY;
  h->cfg = c;
  h->packed = P;
  h->L = L;
  h->status = reinterpret_cast<int*>(P + L.status);
  h->rope = reinterpret_cast<float2*>(P + L.rope);
  h->rope_t = reinterpret_cast<float2*>(P + L.rope_t);
  h->gamma_attn = reinterpret_cast<bf16*>(P + L.gamma_attn);
  h->gamma_mlp = reinterpret_cast<bf16*>(P + L.gamma_mlp);
  h->gamma_q = c.qk_norm ? reinterpret_cast<bf16*>(P + L.gamma_q) : nullptr;
  h->gamma_k = c.qk_norm ? reinterpret_cast<bf16*>(P + L.gamma_k) : nullptr;
  h->w_qkv = reinterpret_cast<f16*>(P + L.w_qkv);
  h->b_qkv = c.qkv_bias ? reinterpret_cast<float*>(P + L.b_qkv) : nullptr;
  h->w_o = reinterpret_cast<f16*>(P + L.w_o);
  h->w_gu = reinterpret_cast<f16*>(P + L.w_gu);
  h->w_down = reinterpret_cast<f16*>(P + L.w_down);
  h->w_router = moe ? reinterpret_cast<f16*>(P + L.w_router) : nullptr;
  h->b_router = (moe && c.router_bias) ? reinterpret_cast<float*>(P + L.b_router) : nullptr;
  h->w_sgu = c.shared_ffn ? reinterpret_cast<f16*>(P + L.w_sgu) : nullptr;
  h->w_sdown = c.shared_ffn ? reinterpret_cast<f16*>(P + L.w_sdown) : nullptr;

  bool ok = cudaMemsetAsync(h->status, 0, 256, st) == cudaSuccess;
  ok = ok && copy_d2d(h->gamma_attn, w->gamma_attn, d * 2, st);
  ok = ok && copy_d2d(h->gamma_mlp, w->gamma_mlp, d * 2, st);
  if (c.qk_norm) {
    ok = ok && copy_d2d(h->gamma_q, w->gamma_q, dh * 2, st);
    ok = ok && copy_d2d(h->gamma_k, w->gamma_k, dh * 2, st);
  }
  // zero the weight area first: the rows that pad matrices to 128 stay zero
  ok = ok && cudaMemsetAsync(P + L.w_qkv, 0, L.total - L.w_qkv, st) == cudaSuccess;
  ok = ok && pack_blocked(h->w_qkv, w->w_q, nq, d, 0, h->status, st);
  ok = ok && pack_blocked(h->w_qkv, w->w_k, nkv, d, 0, h->status, st, 0, 0, nq);
  ok = ok && pack_blocked(h->w_qkv, w->w_v, nkv, d, 0, h->status, st, 0, 0, nq + nkv);
  if (c.qkv_bias && ok) {
    bf16_to_f32_kernel<<<(int)((nq + 255) / 256), 256, 0, st>>>(
        static_cast<const bf16*>(w->b_q), h->b_qkv, (int)nq);
    bf16_to_f32_kernel<<<(int)((nkv + 255) / 256), 256, 0, st>>>(
        static_cast<const bf16*>(w->b_k), h->b_qkv + nq, (int)nkv);
    bf16_to_f32_kernel<<<(int)((nkv + 255) / 256), 256, 0, st>>>(
        static_cast<const bf16*>(w->b_v), h->b_qkv + nq + nkv, (int)nkv);
    count_launches(3);
    ok = cudaGetLastError() == cudaSuccess;
  }
  ok = ok && pack_blocked(h->w_o, w->w_o, d, nq, 0, h->status, st);
  const size_t n_exp = moe ? (size_t)c.n_experts : 1;
  ok = ok && pack_blocked(h->w_gu, w->w_gate, n_exp * f, d, 1, h->status, st, f, 2 * f);
  ok = ok && pack_blocked(h->w_gu, w->w_up, n_exp * f, d, 2, h->status, st, f, 2 * f);
  ok = ok && pack_blocked(h->w_down, w->w_down, n_exp * d, f, 0, h->status, st, d, round128(d));
  if (moe) {
    // rows [W_r | W_r]; with a shared expert W_sg is row E (rows after it zero)
    ok = ok && pack_blocked(h->w_router, w->w_router, n_exp, d, 0, h->status, st, 0, 0, 0, 2 * d, 0);
    ok = ok && pack_blocked(h->w_router, w->w_router, n_exp, d, 0, h->status, st, 0, 0, 0, 2 * d, d);
    if (c.router_bias) ok = ok && copy_d2d(h->b_router, w->b_router, n_exp * 4, st);
  }
  if (c.shared_ffn) {
    const size_t sf = c.shared_ffn;
    ok = ok && pack_blocked(h->w_router, w->w_shared_expert_gate, 1, d, 0, h->status, st, 0, 0, n_exp, 2 * d, 0);
    ok = ok && pack_blocked(h->w_router, w->w_shared_expert_gate, 1, d, 0, h->status, st, 0, 0, n_exp, 2 * d, d);
    ok = ok && pack_blocked(h->w_sgu, w->w_shared_gate, sf, d, 1, h->status, st, sf, 2 * sf);
    ok = ok && pack_blocked(h->w_sgu, w->w_shared_up, sf, d, 2, h->status, st, sf, 2 * sf);
    ok = ok && pack_blocked(h->w_sdown, w->w_shared_down, d, sf, 0, h->status, st, d, round128(d));
  }
  // RoPE table: (cos, sin) of p * theta^(-2i/dh), angles and trig in FP64.
  // Qwen3 layer page, §6 (frequency equation).  Position-major for the decode
  // reduction (a warp reads one position's row), frequency-major for the
  // prefill epilogue (its lanes hold consecutive positions, so each load of
  // one frequency is contiguous across the warp).
  if (ok) {
    const int half = c.head_dim / 2;
    const size_t P_ = (size_t)c.max_position;
    std::vector<float2> tab(P_ * half), tab_t(P_ * half);
    for (int i = 0; i < half; ++i) {
      const double omega = std::pow(c.rope_theta, -2.0 * i / (double)c.head_dim);
      for (int p = 0; p < c.max_position; ++p) {
        const double ang = (double)p * omega;
        const float2 cs = make_float2((float)std::cos(ang), (float)std::sin(ang));
        tab[(size_t)p * half + i] = cs;
        tab_t[(size_t)i * P_ + p] = cs;
      }
    }
    ok = cudaMemcpyAsync(h->rope, tab.data(), tab.size() * sizeof(float2), cudaMemcpyHostToDevice,
                         st) == cudaSuccess;
    ok = ok && cudaMemcpyAsync(h->rope_t, tab_t.data(), tab_t.size() * sizeof(float2),
                               cudaMemcpyHostToDevice, st) == cudaSuccess;
    ok = ok && cudaStreamSynchronize(st) == cudaSuccess;
  }
  // a weight beyond the FP16 range was recorded by the packing kernels
  int packed_status = 0;
  ok = ok && cudaMemcpy(&packed_status, h->status, sizeof(int), cudaMemcpyDeviceToHost) ==
                 cudaSuccess;
  if (!ok || packed_status) {
    delete h;
    return ok ? static_cast<qwen_status>(packed_status) : QWEN_ERR_CUDA;
  }
  *out = h;
  return QWEN_OK;
}

void qwen_layer_destroy(qwen_layer_t layer) { delete layer; }

qwen_status qwen_layer_set_trace(qwen_layer_t layer, void* const* events) {
  if (!layer) return QWEN_ERR_INVALID_ARG;
  if (!events) {
    layer->tracing = false;
    return QWEN_OK;
  }
  for (int i = 0; i < 2 * QWEN_STAGE_COUNT; ++i) layer->trace[i] = events[i];
  layer->tracing = true;
  return QWEN_OK;
}

qwen_status qwen_layer_poll_error(qwen_layer_t layer, void* stream) {
  if (!layer) return QWEN_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(st) != cudaSuccess) return QWEN_ERR_CUDA;
  int v = 0;
  if (cudaMemcpy(&v, layer->status, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess)
    return QWEN_ERR_CUDA;
  if (v) {
    if (cudaMemset(layer->status, 0, sizeof(int)) != cudaSuccess) return QWEN_ERR_CUDA;
  }
  return static_cast<qwen_status>(v);
}

// Shared argument checks of the prefill/decode entry points.
static qwen_status check_io(const void* x, const float* x32, const void* y, const float* y32,
                            const void* workspace, const void* kc, const void* vc) {
  if ((x == nullptr) == (x32 == nullptr)) return QWEN_ERR_INVALID_ARG;
  if (!y && !y32) return QWEN_ERR_INVALID_ARG;
  if (!workspace || !kc || !vc) return QWEN_ERR_INVALID_ARG;
  const void* in = x ? x : static_cast<const void*>(x32);
  if (in == y || in == static_cast<const void*>(y32)) return QWEN_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(workspace) | reinterpret_cast<uintptr_t>(in) |
       reinterpret_cast<uintptr_t>(y) | reinterpret_cast<uintptr_t>(y32) |
       reinterpret_cast<uintptr_t>(kc) | reinterpret_cast<uintptr_t>(vc)) & 15)
    return QWEN_ERR_INVALID_ARG;
  return QWEN_OK;
}

qwen_status qwen_layer_prefill_ex(qwen_layer_t layer, const void* x, const float* x_fp32, void* y,
                                  float* y_fp32, int32_t B, int32_t T, const int32_t* positions,
                                  const int32_t* cache_start, void* k_cache, void* v_cache,
                                  void* workspace, size_t workspace_bytes, void* stream) {
  if (!layer) return QWEN_ERR_INVALID_ARG;
  const qwen_layer_config& c = layer->cfg;
  if (B < 0 || T < 0) return QWEN_ERR_INVALID_ARG;
  if (B == 0 || T == 0) return QWEN_OK;
  if (!positions || !cache_start) return QWEN_ERR_INVALID_ARG;
  if (qwen_status s = check_io(x, x_fp32, y, y_fp32, workspace, k_cache, v_cache)) return s;
  if (B > c.max_batch || (int64_t)B * T > c.max_tokens || T > c.max_seq) return QWEN_ERR_CAPACITY;
  const WorkspaceLayout W = workspace_layout(c, B, T);
  if (workspace_bytes < W.total) return QWEN_ERR_CAPACITY;
  return layer_prefill(layer, static_cast<const bf16*>(x), x_fp32, static_cast<bf16*>(y), y_fp32,
                       B, T, positions, cache_start, static_cast<bf16*>(k_cache),
                       static_cast<bf16*>(v_cache), static_cast<uint8_t*>(workspace), W,
                       static_cast<cudaStream_t>(stream));
}

qwen_status qwen_layer_prefill(qwen_layer_t layer, const void* x, void* y, int32_t B, int32_t T,
                               const int32_t* positions, const int32_t* cache_start,
                               void* k_cache, void* v_cache, void* workspace,
                               size_t workspace_bytes, void* stream) {
  if (!x || !y) return QWEN_ERR_INVALID_ARG;
  return qwen_layer_prefill_ex(layer, x, nullptr, y, nullptr, B, T, positions, cache_start,
                               k_cache, v_cache, workspace, workspace_bytes, stream);
}

qwen_status qwen_layer_decode_ex(qwen_layer_t layer, const void* x, const float* x_fp32, void* y,
                                 float* y_fp32, int32_t B, const int32_t* positions,
                                 const int32_t* cache_len, void* k_cache, void* v_cache,
                                 void* workspace, size_t workspace_bytes, void* stream) {
  if (!layer) return QWEN_ERR_INVALID_ARG;
  const qwen_layer_config& c = layer->cfg;
  if (B < 0) return QWEN_ERR_INVALID_ARG;
  if (B == 0) return QWEN_OK;
  if (!positions || !cache_len) return QWEN_ERR_INVALID_ARG;
  if (qwen_status s = check_io(x, x_fp32, y, y_fp32, workspace, k_cache, v_cache)) return s;
  if (B > c.max_batch || B > c.max_tokens) return QWEN_ERR_CAPACITY;
  const WorkspaceLayout W = workspace_layout(c, B, 1);
  if (workspace_bytes < W.total) return QWEN_ERR_CAPACITY;
  return layer_decode(layer, static_cast<const bf16*>(x), x_fp32, static_cast<bf16*>(y), y_fp32, B,
                      positions, cache_len, static_cast<bf16*>(k_cache),
                      static_cast<bf16*>(v_cache), static_cast<uint8_t*>(workspace), W,
                      static_cast<cudaStream_t>(stream));
}

qwen_status qwen_layer_decode(qwen_layer_t layer, const void* x, void* y, int32_t B,
                              const int32_t* positions, const int32_t* cache_len, void* k_cache,
                              void* v_cache, void* workspace, size_t workspace_bytes,
                              void* stream) {
  if (!x || !y) return QWEN_ERR_INVALID_ARG;
  return qwen_layer_decode_ex(layer, x, nullptr, y, nullptr, B, positions, cache_len, k_cache,
                              v_cache, workspace, workspace_bytes, stream);
}

// Device address of host memory the GPU can access (pinned and mapped), else
// nullptr.
static const void* host_device_view(const void* p) {
  cudaPointerAttributes a{};
  if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
    cudaGetLastError();  // clear the query's error
    return nullptr;
  }
  return a.type == cudaMemoryTypeHost ? a.devicePointer : nullptr;
}

// Host staging for qwen_layer_decode_host, after the decode workspace: x, y
// (BF16 [B][d]) and positions, cache lengths (int32 [B]).
size_t qwen_layer_host_workspace_bytes(const qwen_layer_config* cfg, int32_t B) {
  if (!cfg || !config_valid(*cfg) || B <= 0) return 0;
  const size_t act = align256((size_t)B * cfg->d * 2), idx = align256((size_t)B * 4);
  return align256(workspace_layout(*cfg, B, 1).total) + 2 * act + 2 * idx;
}

qwen_status qwen_layer_decode_host(qwen_layer_t layer, const void* x_host, void* y_host,
                                   int32_t B, const int32_t* positions_host,
                                   const int32_t* cache_len_host, void* k_cache, void* v_cache,
                                   void* workspace, size_t workspace_bytes, void* stream) {
  if (!layer) return QWEN_ERR_INVALID_ARG;
  const qwen_layer_config& c = layer->cfg;
  if (B < 0) return QWEN_ERR_INVALID_ARG;
  if (B == 0) return QWEN_OK;
  if (!x_host || !y_host || !positions_host || !cache_len_host || !workspace)
    return QWEN_ERR_INVALID_ARG;
  if (B > c.max_batch || B > c.max_tokens) return QWEN_ERR_CAPACITY;
  if (workspace_bytes < qwen_layer_host_workspace_bytes(&c, B)) return QWEN_ERR_CAPACITY;
  // Host memory the GPU can address (pinned and mapped): the kernels read the
  // inputs and write the output over the host link themselves, so no copy
  // sits between the step's kernels.  Otherwise: staged copies.
  const void* xv = host_device_view(x_host);
  const void* pv = host_device_view(positions_host);
  const void* lv = host_device_view(cache_len_host);
  void* yv = const_cast<void*>(host_device_view(y_host));
  if (xv && pv && lv && yv)
    return qwen_layer_decode_ex(layer, xv, nullptr, yv, nullptr, B,
                                static_cast<const int32_t*>(pv), static_cast<const int32_t*>(lv),
                                k_cache, v_cache, workspace, workspace_bytes, stream);
  const size_t act = (size_t)B * c.d * 2, idx = (size_t)B * 4;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  size_t o = align256(workspace_layout(c, B, 1).total);
  void* xd = ws + o;
  o += align256(act);
  void* yd = ws + o;
  o += align256(act);
  int32_t* pd = reinterpret_cast<int32_t*>(ws + o);
  o += align256(idx);
  int32_t* ld = reinterpret_cast<int32_t*>(ws + o);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (cudaMemcpyAsync(xd, x_host, act, cudaMemcpyHostToDevice, st) != cudaSuccess ||
      cudaMemcpyAsync(pd, positions_host, idx, cudaMemcpyHostToDevice, st) != cudaSuccess ||
      cudaMemcpyAsync(ld, cache_len_host, idx, cudaMemcpyHostToDevice, st) != cudaSuccess)
    return QWEN_ERR_CUDA;
  const qwen_status s = qwen_layer_decode_ex(layer, xd, nullptr, yd, nullptr, B, pd, ld, k_cache,
                                             v_cache, workspace, workspace_bytes, stream);
  if (s != QWEN_OK) return s;
  return cudaMemcpyAsync(y_host, yd, act, cudaMemcpyDeviceToHost, st) == cudaSuccess
             ? QWEN_OK
             : QWEN_ERR_CUDA;
}

qwen_status qwen_moe_ffn(qwen_layer_t layer, const void* r, const float* r_fp32, void* y,
                         int32_t T, int32_t* topk_idx, float* topk_w, float* logits,
                         void* workspace, size_t workspace_bytes, void* stream) {
  if (!layer) return QWEN_ERR_INVALID_ARG;
  const qwen_layer_config& c = layer->cfg;
  if (c.n_experts == 0) return QWEN_ERR_UNSUPPORTED;
  if (T < 0) return QWEN_ERR_INVALID_ARG;
  if (T == 0) return QWEN_OK;
  if (!r || !y || !workspace || r == y) return QWEN_ERR_INVALID_ARG;
  if (T > c.max_tokens) return QWEN_ERR_CAPACITY;
  const WorkspaceLayout W = workspace_layout(c, 1, T);
  if (workspace_bytes < W.total) return QWEN_ERR_CAPACITY;
  if ((reinterpret_cast<uintptr_t>(workspace) | reinterpret_cast<uintptr_t>(r) |
       reinterpret_cast<uintptr_t>(y) | reinterpret_cast<uintptr_t>(r_fp32)) & 15)
    return QWEN_ERR_INVALID_ARG;
  return moe_forward(layer, static_cast<const bf16*>(r), r_fp32, static_cast<bf16*>(y), nullptr, T,
                     topk_idx, topk_w, logits, static_cast<uint8_t*>(workspace), W,
                     static_cast<cudaStream_t>(stream));
}

size_t qwen_head_workspace_bytes(int32_t B, int32_t d, int32_t V) {
  if (B <= 0 || d <= 0 || V <= 0) return 0;
  const size_t xn = align256((size_t)B * d * 2);
  if (B > 256) return xn;
  return xn + align256((size_t)decode_splits(V, d, B) * V * (size_t)B * 4);
}

qwen_status qwen_head_last_token(const void* y, int32_t B, int32_t T, int32_t d,
                                 const void* gamma_final, const void* w_lm, int32_t V, float eps,
                                 float* logits, void* workspace, size_t workspace_bytes,
                                 void* stream) {
  if (B < 0 || T <= 0 || d <= 0 || V <= 0) return QWEN_ERR_INVALID_ARG;
  if (B == 0) return QWEN_OK;
  if (!y || !gamma_final || !w_lm || !logits || !workspace) return QWEN_ERR_INVALID_ARG;
  if ((d & 63) || d > 8192 || (V & 7)) return QWEN_ERR_UNSUPPORTED;
  if (workspace_bytes < qwen_head_workspace_bytes(B, d, V)) return QWEN_ERR_CAPACITY;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  bf16* xn = static_cast<bf16*>(workspace);
  const bf16* last = static_cast<const bf16*>(y) + (size_t)(T - 1) * d;
  qwen_status s = rmsnorm_launch(last, static_cast<const bf16*>(gamma_final), xn, false, nullptr,
                                 nullptr, B, d, eps, st, (size_t)T * d);
  if (s) return s;
  int* err = lib_status_ptr();
  if (B > 256) {
    GemmEpilogue e{};
    e.mode = EPI_F32;
    e.out32 = logits;
    e.ldo32 = V;
    return gemm_tc(xn, d, w_lm, d, B, V, d, /*op_f16=*/false, e, err, st);
  }
  float* part = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) +
                                         align256((size_t)B * d * 2));
  const int S = decode_splits(V, d, B);
  if ((s = gemm_decode_splitk(w_lm, xn, d, B, V, d, S, /*op_f16=*/false, part, err, st)))
    return s;
  return reduce_f32(part, S, B, V, logits, V, st);
}

}  // extern "C"

namespace qwen {

// Record the trace event of `stage` (begin = 0, end = 1) when tracing is on.
// Inside a CUDA-graph capture the event becomes an external event-record node,
// so it is recorded (and timed) on every replay.
static inline void mark(const qwen_layer_s* L, int stage, int end, cudaStream_t st) {
  if (!L->tracing) return;
  void* e = L->trace[2 * stage + end];
  if (!e) return;
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  cudaStreamIsCapturing(st, &cs);
  if (cs == cudaStreamCaptureStatusActive)
    cudaEventRecordWithFlags(static_cast<cudaEvent_t>(e), st, cudaEventRecordExternal);
  else
    cudaEventRecord(static_cast<cudaEvent_t>(e), st);
}

#define QWEN_STAGE_RUN(stage, expr)            \
  do {                                         \
    mark(L, (stage), 0, st);                   \
    const qwen_status s_ = (expr);             \
    if (s_ != QWEN_OK) return s_;              \
    mark(L, (stage), 1, st);                   \
  } while (0)

// One projection of a decode step: swap-AB split-K on the tensor cores; the
// reduction that follows applies the step's epilogue.
static qwen_status decode_proj(const f16* Wt, const f16* X, int B, int N, int K, float* part,
                               int* err, cudaStream_t st, int& splits, bool late_release = false) {
  splits = decode_splits(N, K, B);
  return gemm_decode_splitk(Wt, X, K, B, N, K, splits, /*op_f16=*/true, part, err, st,
                            /*w_packed=*/true, nullptr, late_release);
}

qwen_status layer_decode(qwen_layer_s* L, const bf16* x, const float* x32, bf16* y, float* y32,
                         int B, const int32_t* positions, const int32_t* cache_len, bf16* kc,
                         bf16* vc, uint8_t* ws, const WorkspaceLayout& W, cudaStream_t st) {
  const qwen_layer_config& c = L->cfg;
  const int d = c.d, dh = c.head_dim, Hq = c.n_q_heads, Hkv = c.n_kv_heads;
  const int nq = Hq * dh, nqkv = nq + 2 * Hkv * dh, f = c.ffn;
  f16* xh = reinterpret_cast<f16*>(ws + W.xh);
  bf16* q = reinterpret_cast<bf16*>(ws + W.q);
  f16* attn = reinterpret_cast<f16*>(ws + W.attn);
  float* r32 = reinterpret_cast<float*>(ws + W.r32);
  float* part = reinterpret_cast<float*>(ws + W.part);
  f16* z = reinterpret_cast<f16*>(ws + W.z);
  f16* hbuf = reinterpret_cast<f16*>(ws + W.h);
  int* err = L->status;
  int S = 1;
  // swap-AB needs the batch on the MMA's N (<= 256); larger batches take the
  // prefill-shaped GEMMs with the same fused epilogues
  const bool swap = B <= 256;

  // RMSNorm_1 -> X-hat (FP16 operand)
  QWEN_STAGE_RUN(QWEN_STAGE_NORM1, rmsnorm_launch(x, L->gamma_attn, xh, true, nullptr, x32, B,
                                                  d, c.rms_eps, st, 0, 0, nullptr, err));
  // Q/K/V, then bias, QK-norm, RoPE, Q store and K/V append at slot cache_len[b]
  const QkvParams qp = make_qkv_params(L, positions, cache_len, q, false, kc, vc, nullptr,
                                       nullptr, 1);
  if (swap) {
    // the QKV GEMM releases the kernels after it only once its threads have
    // waited for RMSNorm_1, i.e. once everything enqueued before the step has
    // completed: the attention then streams cache rows of earlier steps before
    // its own wait
    QWEN_STAGE_RUN(QWEN_STAGE_QKV, decode_proj(L->w_qkv, xh, B, nqkv, d, part, err, st, S,
                                               /*late_release=*/true));
    QWEN_STAGE_RUN(QWEN_STAGE_QKV_FINISH, reduce_qkv(part, S, B, nqkv, qp, err, st));
  } else {
    GemmEpilogue e{};
    e.mode = EPI_QKV;
    e.b_static = 1;
    e.b_blocked = 1;
    e.qkv = qp;
    QWEN_STAGE_RUN(QWEN_STAGE_QKV, gemm_tc(xh, d, L->w_qkv, d, B, nqkv, d, true, e, err, st));
  }
  // split-KV attention over slots 0..cache_len[b], then the merge
  int splits = 0;
  decode_attn_plan(c, B, &splits);
  QWEN_STAGE_RUN(QWEN_STAGE_ATTN,
                 attention_decode(q, kc, vc, cache_len, B, Hq, Hkv, dh, c.max_seq, splits,
                                  reinterpret_cast<float*>(ws + W.attn_o),
                                  reinterpret_cast<float*>(ws + W.attn_ml), attn, err, st,
                                  /*early=*/swap));
  // O projection + residual -> R (FP32)
  if (swap && !c.n_experts) {
    // O projection; its split reduction + residual is fused with RMSNorm_2
    QWEN_STAGE_RUN(QWEN_STAGE_O, decode_proj(L->w_o, attn, B, d, nq, part, err, st, S));
    QWEN_STAGE_RUN(QWEN_STAGE_O_FINISH,
                   reduce_resid_norm(part, S, B, d, x, x32, r32, L->gamma_mlp, c.rms_eps, z, err,
                                     st));
    // gate/up in one K split with SiLU*up in the epilogue -> H, then down
    QWEN_STAGE_RUN(QWEN_STAGE_GATE_UP,
                   gemm_decode_splitk(L->w_gu, z, d, B, 2 * f, d, 1, /*op_f16=*/true, nullptr,
                                      err, st, /*w_packed=*/true, hbuf));
    QWEN_STAGE_RUN(QWEN_STAGE_DOWN, decode_proj(L->w_down, hbuf, B, d, f, part, err, st, S));
    QWEN_STAGE_RUN(QWEN_STAGE_DOWN_FINISH,
                   reduce_resid(part, S, B, d, nullptr, r32, y, y32, st));
    return QWEN_OK;
  }
  if (swap) {
    // MoE: the split reduction + residual also writes [Z_hi | Z_lo] = RMSNorm_2(R)
    QWEN_STAGE_RUN(QWEN_STAGE_O, decode_proj(L->w_o, attn, B, d, nq, part, err, st, S));
    QWEN_STAGE_RUN(QWEN_STAGE_O_FINISH,
                   reduce_resid_norm(part, S, B, d, x, x32, r32, L->gamma_mlp, c.rms_eps, z, err,
                                     st, 2 * (size_t)d, z + d));
  } else {
    GemmEpilogue e{};
    e.mode = EPI_RESID;
    e.b_static = 1;
    e.b_blocked = 1;
    e.resid = x;
    e.resid32 = x32;
    e.ldr = d;
    e.out32 = r32;
    e.ldo32 = d;
    QWEN_STAGE_RUN(QWEN_STAGE_O, gemm_tc(attn, nq, L->w_o, nq, B, d, nq, true, e, err, st));
  }
  if (c.n_experts) {
    QWEN_STAGE_RUN(QWEN_STAGE_MOE, moe_forward(L, nullptr, r32, y, y32, B, nullptr, nullptr,
                                               nullptr, ws, W, st, /*z_ready=*/swap));
    return QWEN_OK;
  }
  // RMSNorm_2 -> Z, gate/up + SiLU*up -> H, down + residual -> Y
  QWEN_STAGE_RUN(QWEN_STAGE_NORM2, rmsnorm_launch(nullptr, L->gamma_mlp, z, true, nullptr, r32, B,
                                                  d, c.rms_eps, st, 0, 0, nullptr, err));
  if (swap) {
    QWEN_STAGE_RUN(QWEN_STAGE_GATE_UP, decode_proj(L->w_gu, z, B, 2 * f, d, part, err, st, S));
    QWEN_STAGE_RUN(QWEN_STAGE_GATE_UP_FINISH, reduce_swiglu(part, S, B, f, hbuf, err, st));
    QWEN_STAGE_RUN(QWEN_STAGE_DOWN, decode_proj(L->w_down, hbuf, B, d, f, part, err, st, S));
    QWEN_STAGE_RUN(QWEN_STAGE_DOWN_FINISH,
                   reduce_resid(part, S, B, d, nullptr, r32, y, y32, st));
    return QWEN_OK;
  }
  GemmEpilogue eg{};
  eg.mode = EPI_SWIGLU;
  eg.b_static = 1;
  eg.b_blocked = 1;
  eg.out = hbuf;
  eg.out_f16 = 1;
  eg.ldo = f;
  QWEN_STAGE_RUN(QWEN_STAGE_GATE_UP, gemm_tc(z, d, L->w_gu, d, B, 2 * f, d, true, eg, err, st));
  GemmEpilogue ed{};
  ed.mode = EPI_RESID;
  ed.b_static = 1;
  ed.b_blocked = 1;
  ed.out = y;
  ed.ldo = d;
  ed.resid32 = r32;
  ed.ldr = d;
  ed.out32 = y32;
  ed.ldo32 = d;
  QWEN_STAGE_RUN(QWEN_STAGE_DOWN, gemm_tc(hbuf, f, L->w_down, f, B, d, f, true, ed, err, st));
  return QWEN_OK;
}

qwen_status layer_prefill(qwen_layer_s* L, const bf16* x, const float* x32, bf16* y, float* y32,
                          int B, int T, const int32_t* positions, const int32_t* slot0, bf16* kc,
                          bf16* vc, uint8_t* ws, const WorkspaceLayout& W, cudaStream_t st) {
  const qwen_layer_config& c = L->cfg;
  const int M = B * T, d = c.d, dh = c.head_dim, Hq = c.n_q_heads, Hkv = c.n_kv_heads;
  const int nq = Hq * dh, nqkv = nq + 2 * Hkv * dh, f = c.ffn;
  f16* xh = reinterpret_cast<f16*>(ws + W.xh);
  f16* q = reinterpret_cast<f16*>(ws + W.q);
  f16* k16 = reinterpret_cast<f16*>(ws + W.k16);
  f16* v16 = reinterpret_cast<f16*>(ws + W.v16);
  f16* attn = reinterpret_cast<f16*>(ws + W.attn);
  float* r32 = reinterpret_cast<float*>(ws + W.r32);
  f16* z = reinterpret_cast<f16*>(ws + W.z);
  f16* hbuf = reinterpret_cast<f16*>(ws + W.h);
  int* err = L->status;

  // RMSNorm_1 -> X-hat (FP16 operand)
  QWEN_STAGE_RUN(QWEN_STAGE_NORM1, rmsnorm_launch(x, L->gamma_attn, xh, true, nullptr, x32, M,
                                                  d, c.rms_eps, st, 0, 0, nullptr, err));
  // fused QKV: bias, QK-norm, RoPE, Q store, K/V cache append
  GemmEpilogue e{};
  e.mode = EPI_QKV;
  e.b_static = 1;
  e.b_blocked = 1;
  e.qkv = make_qkv_params(L, positions, slot0, q, true, kc, vc, k16, v16, T);
  QWEN_STAGE_RUN(QWEN_STAGE_QKV, gemm_tc(xh, d, L->w_qkv, d, M, nqkv, d, true, e, err, st));
  // causal GQA attention over the cache
  QWEN_STAGE_RUN(QWEN_STAGE_ATTN, attention_prefill(q, kc, vc, k16, v16, slot0, attn, B, T, Hq,
                                                    Hkv, dh, c.max_seq, err, st));
  // O projection + residual; R stays in FP32 (it reaches Y unchanged through
  // the second residual, so rounding it to BF16 would put that rounding on Y)
  GemmEpilogue eo{};
  eo.mode = EPI_RESID;
  eo.b_static = 1;
  eo.b_blocked = 1;
  eo.resid = x;
  eo.resid32 = x32;
  eo.ldr = d;
  eo.out32 = r32;
  eo.ldo32 = d;
  QWEN_STAGE_RUN(QWEN_STAGE_O, gemm_tc(attn, nq, L->w_o, nq, M, d, nq, true, eo, err, st));
  if (c.n_experts) {
    QWEN_STAGE_RUN(QWEN_STAGE_MOE,
                   moe_forward(L, nullptr, r32, y, y32, M, nullptr, nullptr, nullptr, ws, W, st));
    return QWEN_OK;
  }
  // RMSNorm_2, gate/up + SiLU*mul, down + residual
  QWEN_STAGE_RUN(QWEN_STAGE_NORM2, rmsnorm_launch(nullptr, L->gamma_mlp, z, true, nullptr, r32, M,
                                                  d, c.rms_eps, st, 0, 0, nullptr, err));
  GemmEpilogue eg{};
  eg.mode = EPI_SWIGLU;
  eg.b_static = 1;
  eg.b_blocked = 1;
  eg.out = hbuf;
  eg.out_f16 = 1;
  eg.ldo = f;
  QWEN_STAGE_RUN(QWEN_STAGE_GATE_UP, gemm_tc(z, d, L->w_gu, d, M, 2 * f, d, true, eg, err, st));
  GemmEpilogue ed{};
  ed.mode = EPI_RESID;
  ed.b_static = 1;
  ed.b_blocked = 1;
  ed.out = y;
  ed.ldo = d;
  ed.resid32 = r32;
  ed.ldr = d;
  ed.out32 = y32;
  ed.ldo32 = d;
  QWEN_STAGE_RUN(QWEN_STAGE_DOWN, gemm_tc(hbuf, f, L->w_down, f, M, d, f, true, ed, err, st));
  return QWEN_OK;
}

QkvParams make_qkv_params(const qwen_layer_s* L, const int32_t* positions, const int32_t* slot0,
                          void* q, bool q_f16, bf16* kc, bf16* vc, f16* k16, f16* v16, int T) {
  const qwen_layer_config& c = L->cfg;
  QkvParams p{};
  p.bias = L->b_qkv;
  p.gamma_q = L->gamma_q;
  p.gamma_k = L->gamma_k;
  p.rope = L->rope;
  p.rope_t = L->rope_t;
  p.positions = positions;
  p.slot0 = slot0;
  p.q_out = q;
  p.q_f16 = q_f16 ? 1 : 0;
  p.k_cache = kc;
  p.v_cache = vc;
  p.k16 = k16;
  p.v16 = v16;
  p.T = T;
  p.Hq = c.n_q_heads;
  p.Hkv = c.n_kv_heads;
  p.dh = c.head_dim;
  p.max_seq = c.max_seq;
  p.max_position = c.max_position;
  p.eps = c.rms_eps;
  return p;
}

}  // namespace qwen
