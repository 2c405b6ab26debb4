// Mixture-of-experts block: router, top-k gating, token permutation, grouped
// expert GEMMs on the tensor cores, weighted combine with the residual.
//
// "Qwen2.5-7B 结构拆解" §10.2: router logits = x W_router, top-k, and with
// norm_topk_prob the k weights are renormalised (equal to a softmax over the k
// selected logits, "MoE 初步" lecture, Router section); each expert is a SwiGLU;
// the output is the plain weighted element-wise sum of the k expert outputs,
// then the residual add.  Selection ties go to the lower expert index.
//
// Steps (all on the caller's stream, no host synchronisation):
//   1. RMSNorm_2 of R -> Z (FP16 GEMM operand) and Z32 (FP32, for the router)
//   2. router: logits = Z32 W_r^T + b_r in FP32 (SIMT FMA, smem-tiled)
//   3. top-k: one warp per token, k rounds of a warp arg-max
//   4. permutation: expert histogram (integer atomics, order-free), then one
//      CTA per expert writes its (token, slot) entries in token order (stable
//      counting sort) and the group offsets; gather of Z rows
//   5. grouped GEMM gate/up (+SiLU*up) and grouped GEMM down over per-expert
//      row ranges, one persistent tensor-core kernel each
//   6. combine: Y[t] = R[t] + sum_j w[t][j] Y_e[pos(t, j)] in slot order
#include "common.cuh"
#include "internal.h"
#include "layer.h"

namespace qwen {

namespace {

constexpr int kRT = 32;   // router: tokens per CTA
constexpr int kRE = 128;  // router: experts per CTA
constexpr int kRK = 32;   // router: k chunk

__global__ void __launch_bounds__(256) router_kernel(const float* __restrict__ z32,
                                                     const bf16* __restrict__ wr,
                                                     const float* __restrict__ br,
                                                     float* __restrict__ logits, int T, int E,
                                                     int d) {
  pdl_trigger();
  pdl_wait();
  __shared__ float zs[kRK][kRT];       // [k][token]
  __shared__ float ws[kRK][kRE + 4];   // [k][expert]
  const int t0 = blockIdx.x * kRT, e0 = blockIdx.y * kRE;
  const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;  // experts 4tx.., tokens 4ty..
  float acc[4][4] = {};
  for (int k0 = 0; k0 < d; k0 += kRK) {
    for (int i = threadIdx.x; i < kRT * kRK; i += 256) {
      const int t = i / kRK, kk = i % kRK;
      zs[kk][t] = (t0 + t < T) ? z32[(size_t)(t0 + t) * d + k0 + kk] : 0.f;
    }
    for (int i = threadIdx.x; i < kRE * kRK; i += 256) {
      const int e = i / kRK, kk = i % kRK;
      ws[kk][e] = (e0 + e < E) ? __bfloat162float(wr[(size_t)(e0 + e) * d + k0 + kk]) : 0.f;
    }
    __syncthreads();
#pragma unroll 8
    for (int kk = 0; kk < kRK; ++kk) {
      const float4 a = *reinterpret_cast<const float4*>(&zs[kk][4 * ty]);
      const float4 b = *reinterpret_cast<const float4*>(&ws[kk][4 * tx]);
      const float av[4] = {a.x, a.y, a.z, a.w}, bv[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(av[i], bv[j], acc[i][j]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int t = t0 + 4 * ty + i;
    if (t >= T) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int e = e0 + 4 * tx + j;
      if (e < E) logits[(size_t)t * E + e] = acc[i][j] + (br ? br[e] : 0.f);
    }
  }
}

// One warp per token: k rounds of arg-max (larger logit first, lower index on
// ties), then the weights softmax(selected logits).
__global__ void topk_kernel(const float* __restrict__ logits, int T, int E, int k,
                            int32_t* __restrict__ idx, float* __restrict__ w) {
  pdl_trigger();
  pdl_wait();
  const int t = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (t >= T) return;
  const int per = (E + 31) / 32;  // <= 8
  float v[8];
  unsigned taken = 0;
#pragma unroll
  for (int i = 0; i < 8; ++i)
    v[i] = (i < per && lane + 32 * i < E) ? logits[(size_t)t * E + lane + 32 * i] : -INFINITY;
  float sel[8];
  int sel_i[8];
  for (int j = 0; j < k; ++j) {
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
  if (lane == 0) {
    float m = sel[0];
    for (int j = 1; j < k; ++j) m = fmaxf(m, sel[j]);
    float s = 0.f, p[8];
    for (int j = 0; j < k; ++j) {
      p[j] = __expf(sel[j] - m);
      s += p[j];
    }
    for (int j = 0; j < k; ++j) {
      idx[(size_t)t * k + j] = sel_i[j];
      w[(size_t)t * k + j] = p[j] / s;
    }
  }
}

__global__ void expert_hist_kernel(const int32_t* __restrict__ idx, int n, int E,
                                   int32_t* __restrict__ counts) {
  pdl_trigger();
  pdl_wait();
  extern __shared__ int32_t h[];
  for (int e = threadIdx.x; e < E; e += blockDim.x) h[e] = 0;
  __syncthreads();
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x) {
    const int e = idx[i];
    if (e >= 0 && e < E) atomicAdd(&h[e], 1);
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x)
    if (h[e]) atomicAdd(&counts[e], h[e]);
}

// One CTA per expert: stable positions of its entries (entry = t*k + j, in
// entry order), perm[pos] = entry, inv[entry] = pos.  CTA 0 also writes the
// group offsets [E+1].
__global__ void __launch_bounds__(256) expert_scatter_kernel(const int32_t* __restrict__ idx,
                                                             int n, int E,
                                                             const int32_t* __restrict__ counts,
                                                             int32_t* __restrict__ offsets,
                                                             int32_t* __restrict__ perm,
                                                             int32_t* __restrict__ inv) {
  pdl_trigger();
  pdl_wait();
  __shared__ int32_t warp_tot[8];
  __shared__ int32_t base_s;
  const int e = blockIdx.x;
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  if (threadIdx.x == 0) {
    int acc = 0;
    for (int i = 0; i < e; ++i) acc += counts[i];
    base_s = acc;
    if (e == 0) {
      int o = 0;
      for (int i = 0; i < E; ++i) {
        offsets[i] = o;
        o += counts[i];
      }
      offsets[E] = o;
    }
  }
  __syncthreads();
  int base = base_s;
  for (int c0 = 0; c0 < n; c0 += 256) {
    const int i = c0 + threadIdx.x;
    const bool hit = i < n && idx[i] == e;
    const unsigned bal = __ballot_sync(0xffffffffu, hit);
    const int rank_in_warp = __popc(bal & ((1u << lane) - 1u));
    if (lane == 0) warp_tot[wid] = __popc(bal);
    __syncthreads();
    int before = 0, total = 0;
#pragma unroll
    for (int w = 0; w < 8; ++w) {
      before += (w < wid) ? warp_tot[w] : 0;
      total += warp_tot[w];
    }
    if (hit) {
      const int pos = base + before + rank_in_warp;
      perm[pos] = i;
      inv[i] = pos;
    }
    base += total;
    __syncthreads();
  }
}

// zp[pos] = z[perm[pos] / k]  (16-bit rows of d elements), one warp per row
__global__ void gather_rows_kernel(const uint16_t* __restrict__ z, const int32_t* __restrict__ perm,
                                   int n, int k, int d, uint16_t* __restrict__ zp) {
  pdl_trigger();
  pdl_wait();
  const int row = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (row >= n) return;
  const int t = perm[row] / k;
  const uint4* src = reinterpret_cast<const uint4*>(z + (size_t)t * d);
  uint4* dst = reinterpret_cast<uint4*>(zp + (size_t)row * d);
  for (int c = lane; c < d / 8; c += 32) dst[c] = src[c];
}

// y[t] = R[t] + sum_j w[t][j] * yp[inv[t*k + j]], summed in slot order j.
__global__ void combine_kernel(const f16* __restrict__ yp, const int32_t* __restrict__ inv,
                               const float* __restrict__ w, const float* __restrict__ r32,
                               const bf16* __restrict__ r, int T, int k, int d,
                               bf16* __restrict__ y, float* __restrict__ y32) {
  pdl_trigger();
  pdl_wait();
  const int t = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (t >= T) return;
  for (int c = lane; c < d / 8; c += 32) {
    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    for (int j = 0; j < k; ++j) {
      const float wj = w[(size_t)t * k + j];
      const int pos = inv[(size_t)t * k + j];
      const uint4 u = reinterpret_cast<const uint4*>(yp + (size_t)pos * d)[c];
      const uint32_t q[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float2 f = unpack_f16x2(q[e]);
        acc[2 * e] = fmaf(wj, f.x, acc[2 * e]);
        acc[2 * e + 1] = fmaf(wj, f.y, acc[2 * e + 1]);
      }
    }
    float o[8];
    if (r32) {
      const float4 a = reinterpret_cast<const float4*>(r32 + (size_t)t * d)[2 * c];
      const float4 b = reinterpret_cast<const float4*>(r32 + (size_t)t * d)[2 * c + 1];
      o[0] = a.x + acc[0]; o[1] = a.y + acc[1]; o[2] = a.z + acc[2]; o[3] = a.w + acc[3];
      o[4] = b.x + acc[4]; o[5] = b.y + acc[5]; o[6] = b.z + acc[6]; o[7] = b.w + acc[7];
    } else {
      const uint4 u = reinterpret_cast<const uint4*>(r + (size_t)t * d)[c];
      const uint32_t q[4] = {u.x, u.y, u.z, u.w};
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
}

inline int nblk(long long n, int t) { return (int)((n + t - 1) / t); }

}  // namespace

qwen_status moe_forward(qwen_layer_s* L, const bf16* r, const float* r32, bf16* y, float* y32, int T,
                        int32_t* topk_idx_out, float* topk_w_out, float* logits_out, uint8_t* ws,
                        const WorkspaceLayout& W, cudaStream_t st) {
  const qwen_layer_config& c = L->cfg;
  const int d = c.d, E = c.n_experts, k = c.top_k, mf = c.ffn;
  const int n = T * k;
  int* err = L->status;
  f16* z = reinterpret_cast<f16*>(ws + W.z);
  float* z32 = reinterpret_cast<float*>(ws + W.z32);
  float* logits = reinterpret_cast<float*>(ws + W.logits);
  int32_t* idx = reinterpret_cast<int32_t*>(ws + W.topk_idx);
  float* wts = reinterpret_cast<float*>(ws + W.topk_w);
  int32_t* counts = reinterpret_cast<int32_t*>(ws + W.counts);
  int32_t* offsets = reinterpret_cast<int32_t*>(ws + W.offsets);
  int32_t* perm = reinterpret_cast<int32_t*>(ws + W.perm);
  int32_t* inv = reinterpret_cast<int32_t*>(ws + W.inv);
  f16* zp = reinterpret_cast<f16*>(ws + W.zp);
  f16* hp = reinterpret_cast<f16*>(ws + W.hp);
  f16* yp = reinterpret_cast<f16*>(ws + W.yp);
  qwen_status s;

  // 1. RMSNorm_2 -> Z (FP16) and Z32 (FP32 router input)
  if ((s = rmsnorm_launch(r, L->gamma_mlp, z, true, z32, r32, T, d, c.rms_eps, st))) return s;
  // 2. router logits in FP32
  launch_k(router_kernel, dim3(nblk(T, kRT), nblk(E, kRE)), dim3(256), 0, st, (const float*)z32,
           (const bf16*)L->w_router, (const float*)L->b_router, logits, T, E, d);
  count_launches();
  // 3. top-k + softmax over the selected logits
  launch_k(topk_kernel, dim3(nblk(32LL * T, 256)), dim3(256), 0, st, (const float*)logits, T, E, k,
           idx, wts);
  count_launches();
  // 4. permutation by expert (stable in token order) and gather of Z rows
  if (cudaMemsetAsync(counts, 0, (size_t)E * sizeof(int32_t), st) != cudaSuccess)
    return QWEN_ERR_CUDA;
  launch_k(expert_hist_kernel, dim3(nblk(n, 1024) < 148 ? nblk(n, 1024) : 148), dim3(1024),
           E * sizeof(int32_t), st, (const int32_t*)idx, n, E, counts);
  launch_k(expert_scatter_kernel, dim3(E), dim3(256), 0, st, (const int32_t*)idx, n, E,
           (const int32_t*)counts, offsets, perm, inv);
  launch_k(gather_rows_kernel, dim3(nblk(32LL * n, 256)), dim3(256), 0, st,
           reinterpret_cast<const uint16_t*>(z), (const int32_t*)perm, n, k, d,
           reinterpret_cast<uint16_t*>(zp));
  count_launches(3);
  if (cudaGetLastError() != cudaSuccess) return QWEN_ERR_CUDA;
  // 5. grouped expert GEMMs: gate/up with SiLU*up, then down
  GemmEpilogue eg{};
  eg.mode = EPI_SWIGLU;
  eg.out = hp;
  eg.out_f16 = 1;
  eg.ldo = mf;
  eg.group_offsets = offsets;
  eg.n_groups = E;
  if ((s = gemm_tc(zp, d, L->w_gu, d, n, 2 * mf, d, true, eg, err, st))) return s;
  GemmEpilogue ed{};
  ed.mode = EPI_STORE;
  ed.out = yp;
  ed.out_f16 = 1;
  ed.ldo = d;
  ed.group_offsets = offsets;
  ed.n_groups = E;
  if ((s = gemm_tc(hp, mf, L->w_down, mf, n, d, mf, true, ed, err, st))) return s;
  // 6. weighted combine + residual
  launch_k(combine_kernel, dim3(nblk(32LL * T, 256)), dim3(256), 0, st, (const f16*)yp,
           (const int32_t*)inv, (const float*)wts, r32, r, T, k, d, y, y32);
  count_launches();
  if (cudaGetLastError() != cudaSuccess) return QWEN_ERR_CUDA;
  // optional copies of the routing for inspection
  if (topk_idx_out &&
      cudaMemcpyAsync(topk_idx_out, idx, (size_t)n * 4, cudaMemcpyDeviceToDevice, st) != cudaSuccess)
    return QWEN_ERR_CUDA;
  if (topk_w_out &&
      cudaMemcpyAsync(topk_w_out, wts, (size_t)n * 4, cudaMemcpyDeviceToDevice, st) != cudaSuccess)
    return QWEN_ERR_CUDA;
  if (logits_out && cudaMemcpyAsync(logits_out, logits, (size_t)T * E * 4,
                                    cudaMemcpyDeviceToDevice, st) != cudaSuccess)
    return QWEN_ERR_CUDA;
  return QWEN_OK;
}

}  // namespace qwen
