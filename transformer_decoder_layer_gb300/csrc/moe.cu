// Mixture-of-experts block: router, top-k gating, token permutation, grouped
// expert GEMMs on the tensor cores, weighted combine with the residual.
//
// "Qwen2.5-7B 结构拆解" §10.2: router logits = x W_router, top-k, and with
// norm_topk_prob the k weights are renormalised (equal to a softmax over the k
// selected logits, "MoE 初步" lecture, Router section); without it (Qwen2) they
// are the selected probabilities of the softmax over all experts.  Each expert
// is a SwiGLU; the output is the plain weighted element-wise sum of the k
// expert outputs, plus (§10.1, Qwen2-MoE) a shared SwiGLU expert of width sf
// scaled per token by g = sigmoid(z W_sg), then the residual add.  Selection
// ties go to the lower expert index.
//
// Steps (all on the caller's stream, no host synchronisation):
//   1. RMSNorm_2 of R -> Z as two FP16 parts per row, [Z_hi | Z_lo]: Z_hi is
//      the experts' GEMM operand, Z_hi + Z_lo carries the FP32 value to ~2^-22
//   2. router: logits = [Z_hi | Z_lo] [W_r | W_r]^T on the tensor cores (one
//      GEMM over K = 2d, FP32 accumulate), i.e. Z W_r^T with FP32-grade inputs:
//      the logits differ from an FP32 evaluation by ~1e-6, far below the 1e-3
//      selection gaps the top-k must reproduce
//   3. top-k: one warp per token, k rounds of a warp arg-max; adds b_r and
//      writes the biased logits back.  The shared gate W_sg rides along as
//      router row E, so its logit comes out of the same GEMM
//   4. shared expert: dense gate/up (+SiLU*up) and down GEMMs on Z_hi, FP32 out
//   5. permutation (stable counting sort by expert, in entry order t*k + j):
//      per-block expert counts, then per block the starting position of each
//      expert (all counts of earlier experts, plus this expert's counts in
//      earlier blocks) and warp-level ranks; the list of non-empty experts;
//      gather of Z_hi rows
//   6. grouped GEMM gate/up (+SiLU*up) and grouped GEMM down over per-expert
//      row ranges, one persistent tensor-core kernel each: 128-row tiles of
//      routed rows, or for up to 64 tokens the swap-AB decode GEMM per
//      touched expert (weights streamed once, tokens on the MMA's N side)
//   7. combine: Y[t] = R[t] + sum_j w[t][j] Y_e[pos(t, j)] in slot order
//      (+ g[t] Y_s[t])
#include "common.cuh"
#include "internal.h"
#include "layer.h"

namespace qwen {

namespace {

constexpr int kPermBlock = 1024;  // permutation entries per CTA
constexpr int kRouteMaxSplits = 8;  // router K splits when the routing is one CTA
constexpr int kRankMaxT = 2;        // tokens up to which the routing ranks experts CTA-wide

// One warp: top-k of the logits row `lrow` (columns [0, E) are Z W_r^T on entry
// and Z W_r^T + b_r on exit) and its gate weights: norm != 0, a softmax over
// the k selected logits; norm == 0, the selected entries of the softmax over
// all E logits.  Lane 0 writes idx_row/w_row [k] and, with g_out, the sigmoid
// of the shared gate's logit lrow[E].
__device__ __forceinline__ void topk_warp(float* lrow, const float* __restrict__ bias, int E,
                                          int k, int norm, int32_t* idx_row, float* w_row,
                                          float* g_out, int32_t* sel_out = nullptr) {
  const int lane = threadIdx.x & 31;
  const int per = (E + 31) / 32;  // <= 8
  float v[8];
  unsigned taken = 0;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int e = lane + 32 * i;
    if (i < per && e < E) {
      float x = lrow[e] + (bias ? bias[e] : 0.f);
      lrow[e] = x;
      v[i] = x == x ? x : -INFINITY;  // a NaN logit is never preferred
    } else {
      v[i] = -INFINITY;
    }
  }
  // fixed-bound loops with j < k guards keep these in registers
  float sel[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
  int sel_i[8] = {0, 0, 0, 0, 0, 0, 0, 0};
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    if (j >= k) break;
    float bv = -INFINITY;
    int bi = 0x7fffffff;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int e = lane + 32 * i;
      if (i < per && e < E && !(taken >> i & 1u)) {
        if (v[i] > bv || (v[i] == bv && e < bi)) {
          bv = v[i];
          bi = e;
        }
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
      const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
      if (ov > bv || (ov == bv && oi < bi)) {
        bv = ov;
        bi = oi;
      }
    }
    if ((bi & 31) == lane) taken |= 1u << (bi >> 5);
    sel[j] = bv;
    sel_i[j] = bi;
  }
  // sel[0] is the largest logit of the row
  float all = 0.f;  // sum over all E of exp(logit - max), for norm == 0
  if (!norm) {
#pragma unroll
    for (int i = 0; i < 8; ++i) all += v[i] == -INFINITY ? 0.f : expf(v[i] - sel[0]);
    all = warp_sum(all);
  }
  if (lane == 0) {
    float s = 0.f, p[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      p[j] = j < k ? expf(sel[j] - sel[0]) : 0.f;
      s += p[j];
    }
    const float den = norm ? s : all;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      if (j < k) {
        idx_row[j] = sel_i[j];
        w_row[j] = p[j] / den;
        if (sel_out) sel_out[j] = sel_i[j];
      }
    }
    if (g_out) *g_out = 1.f / (1.f + expf(-lrow[E]));
  }
}

// One warp per token; logits rows are `ldl` apart (column E: the shared gate).
__global__ void topk_kernel(float* __restrict__ logits, int ldl, const float* __restrict__ bias,
                            int T, int E, int k, int norm, int32_t* __restrict__ idx,
                            float* __restrict__ w, float* __restrict__ gscale) {
  pdl_trigger();
  pdl_wait();
  const int t = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  if (t >= T) return;
  topk_warp(logits + (size_t)t * ldl, bias, E, k, norm, idx + (size_t)t * k, w + (size_t)t * k,
            gscale ? gscale + t : nullptr);
}

// Run by one warp: exclusive scan of tot[0..E) (E <= 256, 8 experts per
// lane).  base[e] becomes the scan value (plus its old value when `add`);
// when `publish`, offsets[0..E] get the scan and act the compacted list of
// non-empty experts in increasing order, act = [count, ids...].
__device__ __forceinline__ void expert_scan_warp(const int32_t* tot, int E, int32_t* base,
                                                 bool add, bool publish, int32_t* offsets,
                                                 int32_t* act) {
  const int lane = threadIdx.x & 31;
  int c[8], sum = 0, nz = 0;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const int x = lane * 8 + j;
    c[j] = x < E ? tot[x] : 0;
    sum += c[j];
    nz += c[j] > 0;
  }
  int incl = sum, nzi = nz;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, incl, o);
    const int u = __shfl_up_sync(0xffffffffu, nzi, o);
    if (lane >= o) {
      incl += v;
      nzi += u;
    }
  }
  int off = incl - sum, na = nzi - nz;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const int x = lane * 8 + j;
    if (x < E) {
      base[x] = (add ? base[x] : 0) + off;
      if (publish) {
        offsets[x] = off;
        if (c[j]) act[1 + na++] = x;
      }
    }
    off += c[j];
  }
  if (publish && lane == 31) {
    offsets[E] = incl;
    act[0] = nzi;
  }
}

// Per-block expert counts: block g counts entries [g*1024, (g+1)*1024).
__global__ void __launch_bounds__(kPermBlock) perm_count_kernel(const int32_t* __restrict__ idx,
                                                                int n, int E,
                                                                int32_t* __restrict__ blk_counts) {
  pdl_trigger();
  pdl_wait();
  extern __shared__ int32_t h[];
  for (int e = threadIdx.x; e < E; e += blockDim.x) h[e] = 0;
  __syncthreads();
  const int i = blockIdx.x * kPermBlock + threadIdx.x;
  if (i < n) atomicAdd(&h[min(max(idx[i], 0), E - 1)], 1);
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) blk_counts[(size_t)blockIdx.x * E + e] = h[e];
}

// Stable positions: entry i of block g with expert e goes to
//   offsets[e] + (entries of e in blocks < g) + (entries of e before i in block g),
// the last term from warp match masks plus the counts of earlier warps.
// perm[pos] = entry, inv[entry] = pos; block 0 writes offsets[0..E] and the
// list of non-empty experts act = [count, ids in increasing order].
__global__ void __launch_bounds__(kPermBlock) perm_scatter_kernel(
    const int32_t* __restrict__ idx, int n, int E, int G, const int32_t* __restrict__ blk_counts,
    int32_t* __restrict__ offsets, int32_t* __restrict__ act, int32_t* __restrict__ perm,
    int32_t* __restrict__ inv) {
  pdl_trigger();
  pdl_wait();
  extern __shared__ int32_t sm[];
  int32_t* tot = sm;               // [E] all entries of e
  int32_t* base = sm + E;          // [E] first position of e for this block
  int32_t* wcnt = sm + 2 * E;      // [32][E] entries of e per warp of this block
  const int g = blockIdx.x, lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    int all = 0, before = 0;
    for (int b0 = 0; b0 < G; b0 += 8) {
      int c[8];  // eight independent loads in flight
#pragma unroll
      for (int j = 0; j < 8; ++j) c[j] = b0 + j < G ? blk_counts[(size_t)(b0 + j) * E + e] : 0;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        all += c[j];
        before += b0 + j < g ? c[j] : 0;
      }
    }
    tot[e] = all;
    base[e] = before;
  }
  for (int i = threadIdx.x; i < 32 * E; i += blockDim.x) wcnt[i] = 0;
  __syncthreads();
  if (wid == 0) expert_scan_warp(tot, E, base, true, g == 0, offsets, act);
  const int i = g * kPermBlock + threadIdx.x;
  const bool valid = i < n;
  const int e = valid ? min(max(idx[i], 0), E - 1) : -1;
  const unsigned same = __match_any_sync(0xffffffffu, e);
  const int rank_w = __popc(same & ((1u << lane) - 1u));
  if (valid && rank_w == 0) wcnt[wid * E + e] = __popc(same);
  __syncthreads();
  if (valid) {
    int pos = base[e] + rank_w;
    for (int w = 0; w < wid; ++w) pos += wcnt[w * E + e];
    perm[pos] = i;
    inv[i] = pos;
  }
}

// Decode-sized routing in one CTA of 1024 threads (T * k <= 1024, T <= 64,
// S <= kRouteMaxSplits):
//   1. logits[t] = sum over the S router split partials part[s][t][0..R) (in
//      split order; one thread per logit);
//   2-3. the top-k and gate weights of every token.  Up to kRankMaxT tokens,
//      spread over the whole CTA: b_r is added (the biased logits written
//      back, as topk_warp does) with a copy in shared memory (NaN as -inf);
//      (t, e) is selected in slot j when j experts of token t precede it, a
//      larger logit or an equal one of lower index ahead (the order of
//      topk_warp's k rounds of warp arg-max); then one warp per token forms
//      the weights with topk_warp's arithmetic.  More tokens: topk_warp, one
//      warp per token (its k rounds beat T * E rank counts there);
//   4. the stable counting sort by expert: counts, then thread e takes the
//      sum of the counts below e (its first sorted position) and its place in
//      the list of non-empty experts, then perm / inv as perm_scatter_kernel.
// No Z rows are gathered: the expert gate/up GEMM reads the token rows
// directly.  Shared memory: route_small_smem(T, E) bytes.
__global__ void __launch_bounds__(1024) route_small_kernel(
    const float* __restrict__ part, int S, int T, int R, const float* __restrict__ bias, int E,
    int k, int norm, float* __restrict__ logits, int32_t* __restrict__ idx,
    float* __restrict__ w, float* __restrict__ gscale, int32_t* __restrict__ offsets,
    int32_t* __restrict__ act, int32_t* __restrict__ perm, int32_t* __restrict__ inv) {
  pdl_trigger();
  pdl_wait();
  extern __shared__ int32_t sm[];
  int32_t* tot = sm;                                    // [E] entries per expert
  int32_t* base = tot + E;                              // [E] first sorted position
  int32_t* wcnt = base + E;                             // [32][E] entries of e per warp
  int32_t* si = wcnt + 32 * E;                          // [T][8] selected experts
  float* sv = reinterpret_cast<float*>(si + 8 * T);     // [T][8] their logits
  float* xs = sv + 8 * T;                               // [T][E] biased logits, NaN -> -inf
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  const int n = T * k;
  const size_t plane = (size_t)T * R;
  const bool by_rank = T <= kRankMaxT;
  // 1. split sums (all S loads of a logit issued before the in-order adds)
  for (int i = threadIdx.x; i < T * R; i += blockDim.x) {
    float p[kRouteMaxSplits];
#pragma unroll
    for (int sp = 0; sp < kRouteMaxSplits; ++sp) p[sp] = sp < S ? part[sp * plane + i] : 0.f;
    float a = 0.f;
#pragma unroll
    for (int sp = 0; sp < kRouteMaxSplits; ++sp) a += p[sp];
    const int t = i / R, e = i - t * R;
    if (by_rank && e < E) {
      a += bias ? bias[e] : 0.f;
      xs[t * E + e] = a == a ? a : -INFINITY;  // a NaN logit is never preferred
    }
    logits[i] = a;
  }
  for (int e = threadIdx.x; e < E; e += blockDim.x) tot[e] = 0;
  for (int i = threadIdx.x; i < 32 * E; i += blockDim.x) wcnt[i] = 0;
  __syncthreads();
  if (!by_rank) {
    for (int t = wid; t < T; t += 32)
      topk_warp(logits + (size_t)t * R, bias, E, k, norm, idx + (size_t)t * k,
                w + (size_t)t * k, gscale ? gscale + t : nullptr, si + t * 8);
  }
  // 2. ranks (a warp's lanes read the same logit of one token: broadcast)
  for (int i = threadIdx.x; by_rank && i < T * E; i += blockDim.x) {
    const int t = i / E, e = i - t * E;
    const float* row = xs + t * E;
    const float x = row[e];
    int r = 0;
#pragma unroll 8
    for (int f = 0; f < E; ++f) {
      const float y = row[f];
      r += (y > x) | ((y == x) & (f < e));
    }
    if (r < k) {
      si[t * 8 + r] = e;
      sv[t * 8 + r] = x;
    }
  }
  __syncthreads();
  // 3. gate weights: norm != 0, a softmax over the k selected logits; norm == 0,
  // the selected entries of the softmax over all E logits; the shared gate's
  // sigmoid from logit column E
  for (int t = wid; by_rank && t < T; t += 32) {
    const float top = sv[t * 8];
    float all = 0.f;
    if (!norm) {
#pragma unroll
      for (int i2 = 0; i2 < 8; ++i2) {
        const int e = lane + 32 * i2;
        const float x = e < E ? xs[t * E + e] : -INFINITY;
        all += x == -INFINITY ? 0.f : expf(x - top);
      }
      all = warp_sum(all);
    }
    if (lane == 0) {
      float s = 0.f, p[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        p[j] = j < k ? expf(sv[t * 8 + j] - top) : 0.f;
        s += p[j];
      }
      const float den = norm ? s : all;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        if (j < k) {
          idx[(size_t)t * k + j] = si[t * 8 + j];
          w[(size_t)t * k + j] = p[j] / den;
        }
      }
      if (gscale) gscale[t] = 1.f / (1.f + expf(-logits[(size_t)t * R + E]));
    }
  }
  // 4. counting sort of the entries t * k + j by expert, stable in entry order
  const bool valid = threadIdx.x < n;
  const int e = valid ? si[(threadIdx.x / k) * 8 + threadIdx.x % k] : -1;
  if (valid) atomicAdd(&tot[e], 1);
  const unsigned same = __match_any_sync(0xffffffffu, e);
  const int rank_w = __popc(same & ((1u << lane) - 1u));
  if (valid && rank_w == 0) wcnt[wid * E + e] = __popc(same);
  __syncthreads();
  if (threadIdx.x < E) {
    const int x = threadIdx.x;
    int off = 0, na = 0;
    for (int f = 0; f < x; ++f) {
      const int c = tot[f];
      off += c;
      na += c > 0;
    }
    base[x] = off;
    offsets[x] = off;
    const int c = tot[x];
    if (c > 0) act[1 + na] = x;
    if (x == E - 1) {
      offsets[E] = off + c;
      act[0] = na + (c > 0);
    }
  }
  __syncthreads();
  if (valid) {
    int pos = base[e] + rank_w;
    for (int q = 0; q < wid; ++q) pos += wcnt[q * E + e];
    perm[pos] = threadIdx.x;
    inv[threadIdx.x] = pos;
  }
}

// Shared memory of route_small_kernel.
inline size_t route_small_smem(int T, int E) {
  return ((size_t)34 * E + 16 * (size_t)T + (size_t)T * E) * 4;
}

// zp[pos] = z[perm[pos] / k]  (16-bit rows of d elements; z rows `zs` apart),
// one warp per row
__global__ void gather_rows_kernel(const uint16_t* __restrict__ z, size_t zs,
                                   const int32_t* __restrict__ perm, int n, int k, int d,
                                   uint16_t* __restrict__ zp) {
  pdl_trigger();
  pdl_wait();
  const int row = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (row >= n) return;
  const int t = perm[row] / k;
  const uint4* src = reinterpret_cast<const uint4*>(z + (size_t)t * zs);
  uint4* dst = reinterpret_cast<uint4*>(zp + (size_t)row * d);
  for (int c = lane; c < d / 8; c += 32) dst[c] = src[c];
}

// y[t] = R[t] + (sum_j w[t][j] * Y_e[inv[t*k + j]] summed in slot order j
//        [+ gs[t] * ys[t], the gated shared expert, when ys is given]).
// Expert outputs Y_e: FP16 rows yp, or (PART) the sum over `ys_n` FP32 split
// partials ypart[s][row][d], splits added in order.
template <bool PART>
__global__ void combine_kernel(const f16* __restrict__ yp, const float* __restrict__ ypart,
                               int y_splits, size_t y_plane, const int32_t* __restrict__ inv,
                               const float* __restrict__ w, const float* __restrict__ ys,
                               const float* __restrict__ gs, const float* __restrict__ r32,
                               const bf16* __restrict__ r, int T, int k, int d,
                               bf16* __restrict__ y, float* __restrict__ y32) {
  pdl_trigger();
  pdl_wait();
  // one thread per 8-column chunk of one token; the k expert rows are loaded
  // together (k <= 8) and summed in slot order
  const int nch = d / 8;
  const long long gi = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (gi >= (long long)T * nch) return;
  const int t = (int)(gi / nch), c = (int)(gi - (long long)t * nch);
  float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
  if constexpr (PART) {
    float v[8][8];
    float wj[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      if (j < k) {
        wj[j] = w[(size_t)t * k + j];
        const float4* src =
            reinterpret_cast<const float4*>(ypart + (size_t)inv[(size_t)t * k + j] * d) + 2 * c;
        const float4 a = src[0], b = src[1];
        v[j][0] = a.x; v[j][1] = a.y; v[j][2] = a.z; v[j][3] = a.w;
        v[j][4] = b.x; v[j][5] = b.y; v[j][6] = b.z; v[j][7] = b.w;
      }
    }
    for (int sp = 1; sp < y_splits; ++sp) {
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        if (j < k) {
          const float4* src = reinterpret_cast<const float4*>(
                                  ypart + sp * y_plane + (size_t)inv[(size_t)t * k + j] * d) +
                              2 * c;
          const float4 a = src[0], b = src[1];
          v[j][0] += a.x; v[j][1] += a.y; v[j][2] += a.z; v[j][3] += a.w;
          v[j][4] += b.x; v[j][5] += b.y; v[j][6] += b.z; v[j][7] += b.w;
        }
      }
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      if (j < k) {
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[e] = fmaf(wj[j], v[j][e], acc[e]);
      }
    }
  } else {
    uint4 u[8];
    float wj[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      if (j < k) {
        wj[j] = w[(size_t)t * k + j];
        u[j] = reinterpret_cast<const uint4*>(yp + (size_t)inv[(size_t)t * k + j] * d)[c];
      }
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      if (j < k) {
        const uint32_t q[4] = {u[j].x, u[j].y, u[j].z, u[j].w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float2 f = unpack_f16x2(q[e]);
          acc[2 * e] = fmaf(wj[j], f.x, acc[2 * e]);
          acc[2 * e + 1] = fmaf(wj[j], f.y, acc[2 * e + 1]);
        }
      }
    }
  }
  if (ys) {
    const float g = gs[t];
    const float4 a = reinterpret_cast<const float4*>(ys + (size_t)t * d)[2 * c];
    const float4 b = reinterpret_cast<const float4*>(ys + (size_t)t * d)[2 * c + 1];
    acc[0] = fmaf(g, a.x, acc[0]); acc[1] = fmaf(g, a.y, acc[1]);
    acc[2] = fmaf(g, a.z, acc[2]); acc[3] = fmaf(g, a.w, acc[3]);
    acc[4] = fmaf(g, b.x, acc[4]); acc[5] = fmaf(g, b.y, acc[5]);
    acc[6] = fmaf(g, b.z, acc[6]); acc[7] = fmaf(g, b.w, acc[7]);
  }
  float o[8];
  if (r32) {
    const float4 a = reinterpret_cast<const float4*>(r32 + (size_t)t * d)[2 * c];
    const float4 b = reinterpret_cast<const float4*>(r32 + (size_t)t * d)[2 * c + 1];
    o[0] = a.x + acc[0]; o[1] = a.y + acc[1]; o[2] = a.z + acc[2]; o[3] = a.w + acc[3];
    o[4] = b.x + acc[4]; o[5] = b.y + acc[5]; o[6] = b.z + acc[6]; o[7] = b.w + acc[7];
  } else {
    const uint4 ur = reinterpret_cast<const uint4*>(r + (size_t)t * d)[c];
    const uint32_t q[4] = {ur.x, ur.y, ur.z, ur.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float2 f = unpack_bf16x2(q[e]);
      o[2 * e] = f.x + acc[2 * e];
      o[2 * e + 1] = f.y + acc[2 * e + 1];
    }
  }
  if (y) {
    uint4 out;
    out.x = pack_bf16x2(o[0], o[1]);
    out.y = pack_bf16x2(o[2], o[3]);
    out.z = pack_bf16x2(o[4], o[5]);
    out.w = pack_bf16x2(o[6], o[7]);
    reinterpret_cast<uint4*>(y + (size_t)t * d)[c] = out;
  }
  if (y32) {
    float4* o4 = reinterpret_cast<float4*>(y32 + (size_t)t * d);
    o4[2 * c] = make_float4(o[0], o[1], o[2], o[3]);
    o4[2 * c + 1] = make_float4(o[4], o[5], o[6], o[7]);
  }
}

inline int nblk(long long n, int t) { return (int)((n + t - 1) / t); }

// Optional copies of the routing for inspection (logits rows are R apart).
qwen_status copy_routing(const int32_t* idx, const float* wts, const float* logits,
                         int32_t* idx_out, float* w_out, float* logits_out, int T, int E, int R,
                         int k, cudaStream_t st) {
  const size_t n = (size_t)T * k;
  if (idx_out &&
      cudaMemcpyAsync(idx_out, idx, n * 4, cudaMemcpyDeviceToDevice, st) != cudaSuccess)
    return QWEN_ERR_CUDA;
  if (w_out && cudaMemcpyAsync(w_out, wts, n * 4, cudaMemcpyDeviceToDevice, st) != cudaSuccess)
    return QWEN_ERR_CUDA;
  if (logits_out && cudaMemcpy2DAsync(logits_out, (size_t)E * 4, logits, (size_t)R * 4,
                                      (size_t)E * 4, T, cudaMemcpyDeviceToDevice,
                                      st) != cudaSuccess)
    return QWEN_ERR_CUDA;
  return QWEN_OK;
}

}  // namespace

int moe_perm_blocks(size_t entries) { return (int)((entries + kPermBlock - 1) / kPermBlock); }

qwen_status moe_forward(qwen_layer_s* L, const bf16* r, const float* r32, bf16* y, float* y32, int T,
                        int32_t* topk_idx_out, float* topk_w_out, float* logits_out, uint8_t* ws,
                        const WorkspaceLayout& W, cudaStream_t st, bool z_ready) {
  const qwen_layer_config& c = L->cfg;
  const int d = c.d, E = c.n_experts, k = c.top_k, mf = c.ffn, sf = c.shared_ffn;
  const int R = router_rows(c);  // E, or E + 8 with the shared gate at column E
  const int n = T * k;
  int* err = L->status;
  f16* z = reinterpret_cast<f16*>(ws + W.z);  // rows [Z_hi | Z_lo], 2d apart
  float* logits = reinterpret_cast<float*>(ws + W.logits);
  int32_t* idx = reinterpret_cast<int32_t*>(ws + W.topk_idx);
  float* wts = reinterpret_cast<float*>(ws + W.topk_w);
  int32_t* blk_counts = reinterpret_cast<int32_t*>(ws + W.blk_counts);
  int32_t* offsets = reinterpret_cast<int32_t*>(ws + W.offsets);
  int32_t* act = reinterpret_cast<int32_t*>(ws + W.act);
  int32_t* perm = reinterpret_cast<int32_t*>(ws + W.perm);
  int32_t* inv = reinterpret_cast<int32_t*>(ws + W.inv);
  f16* zp = reinterpret_cast<f16*>(ws + W.zp);
  f16* hp = reinterpret_cast<f16*>(ws + W.hp);
  f16* yp = reinterpret_cast<f16*>(ws + W.yp);
  f16* hs = sf ? reinterpret_cast<f16*>(ws + W.hs) : nullptr;
  float* ys32 = sf ? reinterpret_cast<float*>(ws + W.ys32) : nullptr;
  float* gsc = sf ? reinterpret_cast<float*>(ws + W.gscale) : nullptr;
  float* part = reinterpret_cast<float*>(ws + W.part);
  // decode-sized batches use the swap-AB split-K GEMMs (one 128-row weight
  // tile would otherwise run its whole K on a single SM), and up to 64 tokens
  // the grouped swap-AB GEMM for the experts (1-8 routed rows per expert
  // would waste most of a 128-row tile)
  const bool small = T <= 256 && W.part != 0;
  const bool grouped_dec = small && T <= kMoeDecodeMaxRows;
  qwen_status s;

  // 1. RMSNorm_2 -> [Z_hi | Z_lo] (FP16 parts of the FP32 result)
  if (!z_ready && (s = rmsnorm_launch(r, L->gamma_mlp, z, true, nullptr, r32, T, d, c.rms_eps,
                                      st, 0, 2 * (size_t)d, z + d, err)))
    return s;
  // 2. router logits (and the shared gate's, column E): one tensor-core GEMM
  // over K = 2d against [W_r | W_r]
  if (small) {
    // the one-CTA routing sums the split partials: keep their number small
    const int S = grouped_dec ? min(decode_splits(R, 2 * d, T), kRouteMaxSplits)
                              : decode_splits(R, 2 * d, T);
    if ((s = gemm_decode_splitk(L->w_router, z, 2 * d, T, R, 2 * d, S, true, part, err, st,
                                /*w_packed=*/true)))
      return s;
    if (grouped_dec) {
      // 3 + 5 in one CTA: split sum, top-k, counting sort (it reads the
      // router partials, so it runs before the shared expert reuses them)
      static std::atomic<uint64_t> attr{0};  // one bit per device
      const size_t smem = route_small_smem(T, E);
      // the limit is raised once per device, for the largest use
      if (!smem_attr_once(route_small_kernel, (int)route_small_smem(kMoeDecodeMaxRows, 256), attr))
        return QWEN_ERR_CUDA;
      launch_k(route_small_kernel, dim3(1), dim3(1024), smem, st,
               (const float*)part, S, T, R, (const float*)L->b_router, E, k, c.norm_topk_prob,
               logits, idx, wts, gsc, offsets, act, perm, inv);
      count_launches();
      if (cudaGetLastError() != cudaSuccess) return QWEN_ERR_CUDA;
    } else if ((s = reduce_f32(part, S, T, R, logits, R, st))) {
      return s;
    }
  } else {
    GemmEpilogue er{};
    er.mode = EPI_F32;
    er.out32 = logits;
    er.ldo32 = R;
    er.b_static = 1;
    er.b_blocked = 1;
    if ((s = gemm_tc(z, 2 * d, L->w_router, 2 * d, T, R, 2 * d, true, er, err, st))) return s;
  }
  // 3. top-k (+ router bias), gate weights, shared gate sigmoid
  if (!grouped_dec) {
    launch_k(topk_kernel, dim3(nblk(32LL * T, 256)), dim3(256), 0, st, logits, R,
             (const float*)L->b_router, T, E, k, c.norm_topk_prob, idx, wts, gsc);
    count_launches();
  }
  // 4. shared expert on Z_hi: H_s = SiLU(Z W_sg^T) * (Z W_su^T), Y_s = H_s W_sd^T
  // (FP32); before the routed experts, whose decode partials reuse `part`
  if (sf) {
    if (small) {
      if ((s = gemm_decode_splitk(L->w_sgu, z, 2 * d, T, 2 * sf, d, 1, true, nullptr, err, st,
                                  /*w_packed=*/true, hs)))
        return s;
      const int S = decode_splits(d, sf, T);
      if ((s = gemm_decode_splitk(L->w_sdown, hs, sf, T, d, sf, S, true, part, err, st,
                                  /*w_packed=*/true)))
        return s;
      if ((s = reduce_f32(part, S, T, d, ys32, d, st))) return s;
    } else {
      GemmEpilogue sg{};
      sg.mode = EPI_SWIGLU;
      sg.out = hs;
      sg.out_f16 = 1;
      sg.ldo = sf;
      sg.b_static = 1;
      sg.b_blocked = 1;
      if ((s = gemm_tc(z, 2 * d, L->w_sgu, d, T, 2 * sf, d, true, sg, err, st))) return s;
      GemmEpilogue sd{};
      sd.mode = EPI_F32;
      sd.out32 = ys32;
      sd.ldo32 = d;
      sd.b_static = 1;
      sd.b_blocked = 1;
      if ((s = gemm_tc(hs, sf, L->w_sdown, sf, T, d, sf, true, sd, err, st))) return s;
    }
  }
  // 5. permutation by expert (stable in entry order) and gather of Z_hi rows
  if (!grouped_dec) {
    const int G = moe_perm_blocks(n);
    launch_k(perm_count_kernel, dim3(G), dim3(kPermBlock), E * sizeof(int32_t), st,
             (const int32_t*)idx, n, E, blk_counts);
    launch_k(perm_scatter_kernel, dim3(G), dim3(kPermBlock), (2 + 32) * E * sizeof(int32_t), st,
             (const int32_t*)idx, n, E, G, (const int32_t*)blk_counts, offsets, act, perm, inv);
    launch_k(gather_rows_kernel, dim3(nblk(32LL * n, 256)), dim3(256), 0, st,
             reinterpret_cast<const uint16_t*>(z), 2 * (size_t)d, (const int32_t*)perm, n, k, d,
             reinterpret_cast<uint16_t*>(zp));
    count_launches(3);
    if (cudaGetLastError() != cudaSuccess) return QWEN_ERR_CUDA;
  }
  // 6. grouped expert GEMMs: gate/up with SiLU*up, then down
  if (grouped_dec) {
    // swap-AB per touched expert: gate/up on the token rows of Z_hi (each
    // expert keeps its routed tokens), down on the sorted H rows; the down
    // partials are summed by the combine
    const int groups = n < E ? n : E;
    if ((s = gemm_decode_grouped_tokens(L->w_gu, E, z, 2 * d, T, 2 * mf, d, act, idx, inv, k,
                                        groups, hp, err, st)))
      return s;
    const int S = decode_splits(d, mf, T, groups);
    if ((s = gemm_decode_grouped(L->w_down, E, hp, n, T, d, mf, S, act, offsets, groups, part,
                                 nullptr, err, st)))
      return s;
    launch_k(combine_kernel<true>, dim3(nblk((long long)T * (d / 8), 256)), dim3(256), 0, st,
             (const f16*)nullptr, (const float*)part, S, (size_t)n * d, (const int32_t*)inv,
             (const float*)wts, (const float*)ys32, (const float*)gsc, r32, r, T, k, d, y, y32);
    count_launches();
    if (cudaGetLastError() != cudaSuccess) return QWEN_ERR_CUDA;
    return copy_routing(idx, wts, logits, topk_idx_out, topk_w_out, logits_out, T, E, R, k, st);
  }
  if (gemm_expert_supported(E, 2 * mf, d) && gemm_expert_supported(E, d, mf)) {
    // weights on the M side, routed rows in chunks of up to 256 (moe_gemm.cu)
    if ((s = gemm_expert(L->w_gu, E, 2 * mf, d, zp, n, d, offsets, hp, mf, true, err, st)))
      return s;
    if ((s = gemm_expert(L->w_down, E, d, mf, hp, n, mf, offsets, yp, d, false, err, st)))
      return s;
  } else {
    GemmEpilogue eg{};
    eg.mode = EPI_SWIGLU;
    eg.out = hp;
    eg.out_f16 = 1;
    eg.ldo = mf;
    eg.group_offsets = offsets;
    eg.n_groups = E;
    eg.b_blocked = 1;
    if ((s = gemm_tc(zp, d, L->w_gu, d, n, 2 * mf, d, true, eg, err, st))) return s;
    GemmEpilogue ed{};
    ed.mode = EPI_STORE;
    ed.out = yp;
    ed.out_f16 = 1;
    ed.ldo = d;
    ed.group_offsets = offsets;
    ed.n_groups = E;
    ed.b_blocked = 1;
    if ((s = gemm_tc(hp, mf, L->w_down, mf, n, d, mf, true, ed, err, st))) return s;
  }
  // 7. weighted combine (+ gated shared expert) + residual
  launch_k(combine_kernel<false>, dim3(nblk((long long)T * (d / 8), 256)), dim3(256), 0, st,
           (const f16*)yp, (const float*)nullptr, 1, (size_t)0, (const int32_t*)inv,
           (const float*)wts, (const float*)ys32, (const float*)gsc, r32, r, T, k, d, y, y32);
  count_launches();
  if (cudaGetLastError() != cudaSuccess) return QWEN_ERR_CUDA;
  return copy_routing(idx, wts, logits, topk_idx_out, topk_w_out, logits_out, T, E, R, k, st);
}

}  // namespace qwen
