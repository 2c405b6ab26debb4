// RMSNorm over the feature axis, 128-bit loads/stores.
//
// Qwen3 layer page ("推理系统 03"), §3: y_j = gamma_j x_j / sqrt(mean_k x_k^2 + eps),
// with the mean square accumulated in FP32.
#include "common.cuh"
#include "internal.h"

namespace qwen {

// 8 elements of chunk c of a row (BF16 or FP32 input) as FP32.
__device__ __forceinline__ void rms_load8(const bf16* __restrict__ xr, const float* __restrict__ xr32,
                                          int c, float (&v)[8]) {
  if (xr32) {
    const float4 a = reinterpret_cast<const float4*>(xr32)[2 * c];
    const float4 b = reinterpret_cast<const float4*>(xr32)[2 * c + 1];
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
    v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
  } else {
    const uint4 u = reinterpret_cast<const uint4*>(xr)[c];
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float2 f = unpack_bf16x2(w[j]);
      v[2 * j] = f.x;
      v[2 * j + 1] = f.y;
    }
  }
}

// One warp per row, two passes: the sum of squares over the row (loads of
// several 512-byte row segments in flight per warp), then the row again (now
// in L1 or L2), scaled and stored.  Keeping the whole row in registers
// instead (128 values per lane at d = 4096) left room for 8 warps per SM and
// reached a quarter to half of the HBM bandwidth.
__global__ void __launch_bounds__(256) rmsnorm_kernel(const bf16* __restrict__ x,
                                                      const float* __restrict__ x32,
                                                      const bf16* __restrict__ gamma,
                                                      void* __restrict__ y, bool y_f16,
                                                      float* __restrict__ y32, int rows, int d,
                                                      float eps, size_t xs, size_t ys,
                                                      __half* __restrict__ y_lo, int* err) {
  pdl_trigger();
  pdl_wait();
  const int row = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (row >= rows) return;
  const int nch = d >> 3;  // 8-element chunks
  const bf16* xr = x32 ? nullptr : x + (size_t)row * xs;
  const float* xr32 = x32 ? x32 + (size_t)row * xs : nullptr;
  float ss = 0.f;
#pragma unroll 8
  for (int c = lane; c < nch; c += 32) {
    float v[8];
    rms_load8(xr, xr32, c, v);
#pragma unroll
    for (int j = 0; j < 8; ++j) ss = fmaf(v[j], v[j], ss);
  }
  ss = warp_sum(ss);
  const float rstd = rsqrtf(ss / (float)d + eps);
  const uint4* gr = reinterpret_cast<const uint4*>(gamma);
  uint4* yr = reinterpret_cast<uint4*>(static_cast<uint16_t*>(y) + (size_t)row * ys);
  uint4* lr = y_lo ? reinterpret_cast<uint4*>(y_lo + (size_t)row * ys) : nullptr;
  bool bad = false;
#pragma unroll 4
  for (int c = lane; c < nch; c += 32) {
    float v[8];
    rms_load8(xr, xr32, c, v);
    const uint4 gu = gr[c];
    const uint32_t gw[4] = {gu.x, gu.y, gu.z, gu.w};
    float o[8];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float2 g = unpack_bf16x2(gw[j]);
      o[2 * j] = g.x * (v[2 * j] * rstd);
      o[2 * j + 1] = g.y * (v[2 * j + 1] * rstd);
    }
    uint4 out;
    out.x = pack2_chk(o[0], o[1], y_f16, bad);
    out.y = pack2_chk(o[2], o[3], y_f16, bad);
    out.z = pack2_chk(o[4], o[5], y_f16, bad);
    out.w = pack2_chk(o[6], o[7], y_f16, bad);
    yr[c] = out;
    if (lr) {
      // residual of the FP16 rounding, itself rounded to FP16
      const uint32_t hw[4] = {out.x, out.y, out.z, out.w};
      uint32_t lo[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float2 h = unpack_f16x2(hw[j]);
        lo[j] = pack_f16x2_chk(o[2 * j] - h.x, o[2 * j + 1] - h.y, bad);
      }
      lr[c] = make_uint4(lo[0], lo[1], lo[2], lo[3]);
    }
    if (y32) {
      float4* y4 = reinterpret_cast<float4*>(y32 + (size_t)row * d);
      y4[2 * c] = make_float4(o[0], o[1], o[2], o[3]);
      y4[2 * c + 1] = make_float4(o[4], o[5], o[6], o[7]);
    }
  }
  record_overflow(err, bad);
}

// Up to a few rows per SM (decode batches, short prefills): one CTA per row,
// one 8-element chunk per thread, so the row is read, reduced and written in
// one round trip each.
__global__ void __launch_bounds__(1024) rmsnorm_row_kernel(
    const bf16* __restrict__ x, const float* __restrict__ x32, const bf16* __restrict__ gamma,
    void* __restrict__ y, bool y_f16, float* __restrict__ y32, int d, float eps, size_t xs,
    size_t ys, __half* __restrict__ y_lo, int* err) {
  pdl_trigger();
  __shared__ float red[32];
  const int row = blockIdx.x;
  const int c = threadIdx.x;  // chunk
  const int nch = d >> 3;
  const int lane = c & 31, wid = c >> 5;
  // gamma is a weight (no kernel writes it): read before the wait
  const uint4 gu = c < nch ? reinterpret_cast<const uint4*>(gamma)[c] : make_uint4(0, 0, 0, 0);
  pdl_wait();
  float v[8];
  float ss = 0.f;
  if (c < nch) {
    if (x32) {
      const float4* xr = reinterpret_cast<const float4*>(x32 + (size_t)row * xs);
      const float4 a = xr[2 * c], b = xr[2 * c + 1];
      v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
      v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
    } else {
      const uint4 u = reinterpret_cast<const uint4*>(x + (size_t)row * xs)[c];
      const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float2 f = unpack_bf16x2(w[j]);
        v[2 * j] = f.x;
        v[2 * j + 1] = f.y;
      }
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) ss = fmaf(v[j], v[j], ss);
  }
  ss = warp_sum(ss);
  if (lane == 0) red[wid] = ss;
  __syncthreads();
  float tot = 0.f;
  const int nw = (blockDim.x + 31) >> 5;
  for (int w = 0; w < nw; ++w) tot += red[w];
  if (c >= nch) return;
  const float rstd = rsqrtf(tot / (float)d + eps);
  const uint32_t gw[4] = {gu.x, gu.y, gu.z, gu.w};
  float o[8];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const float2 g = unpack_bf16x2(gw[j]);
    o[2 * j] = g.x * (v[2 * j] * rstd);
    o[2 * j + 1] = g.y * (v[2 * j + 1] * rstd);
  }
  bool bad = false;
  uint4 out;
  out.x = pack2_chk(o[0], o[1], y_f16, bad);
  out.y = pack2_chk(o[2], o[3], y_f16, bad);
  out.z = pack2_chk(o[4], o[5], y_f16, bad);
  out.w = pack2_chk(o[6], o[7], y_f16, bad);
  reinterpret_cast<uint4*>(static_cast<uint16_t*>(y) + (size_t)row * ys)[c] = out;
  if (y_lo) {
    const uint32_t hw[4] = {out.x, out.y, out.z, out.w};
    uint32_t lo[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float2 h = unpack_f16x2(hw[j]);
      lo[j] = pack_f16x2_chk(o[2 * j] - h.x, o[2 * j + 1] - h.y, bad);
    }
    reinterpret_cast<uint4*>(y_lo + (size_t)row * ys)[c] = make_uint4(lo[0], lo[1], lo[2], lo[3]);
  }
  if (y32) {
    float4* y4 = reinterpret_cast<float4*>(y32 + (size_t)row * d);
    y4[2 * c] = make_float4(o[0], o[1], o[2], o[3]);
    y4[2 * c + 1] = make_float4(o[4], o[5], o[6], o[7]);
  }
  record_overflow(err, bad);
}

qwen_status rmsnorm_launch(const bf16* x, const bf16* gamma, void* y, bool y_f16, float* y32,
                           const float* x32, int rows, int d, float eps, cudaStream_t st,
                           size_t x_stride, size_t y_stride, __half* y_lo, int* err) {
  if (rows == 0) return QWEN_OK;
  if (d <= 0 || (d & 7) || d > 8192) return QWEN_ERR_UNSUPPORTED;
  const size_t xs = x_stride ? x_stride : (size_t)d;
  const size_t ys = y_stride ? y_stride : (size_t)d;
  if (y_lo && !y_f16) return QWEN_ERR_INVALID_ARG;
  // one CTA per row up to 8 rows per SM: at 1024 rows (T = 1024 prefill) the
  // warp-per-row kernel, with two passes over each row and 8 warps per SM, is
  // bound by the latency of its dependent loads (12.5 -> ~6 us in the layer's
  // timeline); at 4096 rows and above both kernels measure the same
  if (rows <= 8 * device_sm_count()) {
    const int threads = ((d >> 3) + 31) & ~31;  // <= 1024 for d <= 8192
    launch_k(rmsnorm_row_kernel, dim3(rows), dim3(threads), 0, st, x, x32, gamma, y, y_f16, y32, d,
             eps, xs, ys, y_lo, err);
    count_launches();
    return cudaGetLastError() == cudaSuccess ? QWEN_OK : QWEN_ERR_CUDA;
  }
  const int threads = 256;
  const int blocks = (rows * 32 + threads - 1) / threads;
  launch_k(rmsnorm_kernel, dim3(blocks), dim3(threads), 0, st, x, x32, gamma, y, y_f16, y32, rows,
           d, eps, xs, ys, y_lo, err);
  count_launches();
  return cudaGetLastError() == cudaSuccess ? QWEN_OK : QWEN_ERR_CUDA;
}

}  // namespace qwen
