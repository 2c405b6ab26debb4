// Per-(token, head) finish of the fused QKV projection: bias, Qwen3 QK-norm,
// rotate_half RoPE, then Q store or K/V cache append.  Used by the prefill GEMM
// epilogue and by the decode split-K reduction, so both paths share one
// definition of the step.
//
// Qwen3 layer page ("推理系统 03"): §4 projections, §5 per-head RMSNorm over dh
// with one shared gamma for Q and one for K (V untouched), §6 RoPE pairing
// (i, i + dh/2) by angle p * theta^(-2i/dh) (cos/sin read from a table built in
// FP64 on the host), §12 the cache keeps K after QK-norm and RoPE.
#pragma once

#include "common.cuh"
#include "internal.h"

namespace qwen {

template <int DH>
__device__ __forceinline__ void qkv_head_finish(float (&v)[DH], int m, int head,
                                                const QkvParams& p, int* err) {
  const int kind = head < p.Hq ? 0 : (head < p.Hq + p.Hkv ? 1 : 2);  // q, k, v
  // the token's position and its sequence's first slot, loaded first: their
  // latency then overlaps the bias and QK-norm arithmetic
  const int b = m / p.T, t = m - (m / p.T) * p.T;
  const int pos = kind < 2 ? p.positions[m] : 0;
  const int s0 = p.slot0[b];
  if (p.bias) {
    const float4* bb = reinterpret_cast<const float4*>(p.bias + (size_t)head * DH);
#pragma unroll
    for (int i = 0; i < DH / 4; ++i) {
      const float4 b4 = __ldg(bb + i);
      v[4 * i] += b4.x;
      v[4 * i + 1] += b4.y;
      v[4 * i + 2] += b4.z;
      v[4 * i + 3] += b4.w;
    }
  }
  if (kind < 2) {
    if (p.gamma_q) {
      float ss = 0.f;
#pragma unroll
      for (int i = 0; i < DH; ++i) ss = fmaf(v[i], v[i], ss);
      const float rstd = rsqrtf(ss / (float)DH + p.eps);
      const uint4* g4 = reinterpret_cast<const uint4*>(kind == 0 ? p.gamma_q : p.gamma_k);
#pragma unroll
      for (int i = 0; i < DH / 8; ++i) {
        const uint4 gu = __ldg(g4 + i);
        const uint32_t gw[4] = {gu.x, gu.y, gu.z, gu.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const float2 g = unpack_bf16x2(gw[j]);
          v[8 * i + 2 * j] = g.x * (v[8 * i + 2 * j] * rstd);
          v[8 * i + 2 * j + 1] = g.y * (v[8 * i + 2 * j + 1] * rstd);
        }
      }
    }
    if (pos < 0 || pos >= p.max_position) {
      record_error(err, QWEN_ERR_RANGE);
      return;
    }
    // frequency-major table: the lanes of a warp hold consecutive tokens, so
    // each frequency's (cos, sin) loads are contiguous across the warp
    const float2* tab = p.rope_t + pos;
#pragma unroll
    for (int i = 0; i < DH / 2; ++i) {
      const float2 cs = __ldg(tab + (size_t)i * p.max_position);  // pair (i, i + dh/2)
      const float a = v[i], b = v[i + DH / 2];
      v[i] = a * cs.x - b * cs.y;
      v[i + DH / 2] = b * cs.x + a * cs.y;
    }
  }
  bool bad = false;  // an FP16 value (prefill Q, K/V copies) beyond the format's range
  auto store = [&](void* dst, bool f16_out, bool streaming = false) {
    uint4* d4 = reinterpret_cast<uint4*>(dst);
#pragma unroll
    for (int i = 0; i < DH / 8; ++i) {
      uint4 o;
      o.x = pack2_chk(v[8 * i], v[8 * i + 1], f16_out, bad);
      o.y = pack2_chk(v[8 * i + 2], v[8 * i + 3], f16_out, bad);
      o.z = pack2_chk(v[8 * i + 4], v[8 * i + 5], f16_out, bad);
      o.w = pack2_chk(v[8 * i + 6], v[8 * i + 7], f16_out, bad);
      if (streaming)
        __stcs(d4 + i, o);
      else
        d4[i] = o;
    }
  };
  if (kind == 0) {
    // prefill: FP16 when the sequence starts at slot 0 (every key is this
    // call's, read from FP16 copies), BF16 when earlier keys come from the
    // BF16 cache, so the attention's two operands always share a type
    store(static_cast<uint16_t*>(p.q_out) + (((size_t)b * p.Hq + head) * p.T + t) * DH,
          p.q_f16 != 0 && s0 == 0);
    record_overflow(err, bad);
    return;
  }
  const int slot = s0 + t;
  if (slot < 0 || slot >= p.max_seq) {
    record_error(err, QWEN_ERR_RANGE);
    return;
  }
  const int g = kind == 1 ? head - p.Hq : head - p.Hq - p.Hkv;
  __half* fresh = kind == 1 ? p.k16 : p.v16;
  // a sequence from slot 0 has its attention read the FP16 copies, so its
  // cache rows are not read again in this call: streaming stores keep them
  // from displacing Q and the copies in L2
  const bool fresh_read = fresh != nullptr && s0 == 0;
  store((kind == 1 ? p.k_cache : p.v_cache) + (((size_t)b * p.Hkv + g) * p.max_seq + slot) * DH,
        false, fresh_read);
  if (fresh) store(fresh + (((size_t)b * p.Hkv + g) * p.T + t) * DH, true);
  record_overflow(err, bad);
}

}  // namespace qwen
