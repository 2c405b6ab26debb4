// Decode-step projections: one token per sequence, so every projection is a
// skinny product [B x K] x [N x K]^T that is bound by streaming the weight
// from HBM ("Qwen2.5-7B 结构拆解" §11: single-stream decode speed is bandwidth
// divided by weight bytes).
//
// Swap-AB: the weight is the MMA's A operand (128 weight rows fill the M=128
// tensor-core tile), the B tokens are its N operand (padded to 16..256).  The
// K dimension is split so that (n-tile, k-split) units cover every SM; a
// persistent CTA walks its units with a deep TMA ring so enough weight bytes
// are in flight.  Each unit writes FP32 partials part[s][n][b]; a reduction
// kernel sums the splits in a fixed order (deterministic) and applies the
// step's epilogue (residual add, SiLU*up, or the fused QKV finish).
//
// Grouped mode (mixture-of-experts decode): W is a stack of E weights [E][N][K]
// and X holds the routed rows grouped by expert, rows [offsets[e],
// offsets[e+1]) for expert e.  A unit is (non-empty expert, n-tile, k-split);
// its X tile starts at the expert's first row and results are kept for that
// expert's rows only, so each touched expert's weights stream from HBM once.
// Token mode (grouped, SwiGLU only): X holds the T token rows themselves;
// every expert's tile multiplies all of them and the epilogue keeps the
// tokens routed to the expert, writing each to its sorted row inv[t*k + j]
// (idx[t*k + j] == e), so no gathered copy of X is needed.
#include "common.cuh"
#include "internal.h"
#include "layer.h"
#include "qkv_epilogue.cuh"

#include <cudaTypedefs.h>

namespace qwen {

namespace {

constexpr int kDBM = 128;
constexpr int kDBK = 64;
constexpr int kDThreads = 192;

// Epilogues of the decode GEMM: FP32 split partials, or (one split only) the
// SwiGLU of an interleaved gate/up tile written straight to H.
enum DecEpi : int { DEC_PARTIAL = 0, DEC_SWIGLU = 1 };

template <int BP, int EPI>
struct DecCfg {
  static constexpr int A_BYTES = kDBM * kDBK * 2;  // 16 KB of weight per stage
  static constexpr int B_BYTES = BP * kDBK * 2;
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  // gate half of a tile handed to the up warps: [64 rows][BP] FP32
  static constexpr int XCH_BYTES = EPI == DEC_SWIGLU ? 64 * BP * 4 : 0;
  static constexpr int RING = (200 * 1024 - XCH_BYTES) / STAGE_BYTES;
  static constexpr int STAGES = RING > 12 ? 12 : RING;
  // the epilogue reads 32 columns at a time, so with BP = 16 the second
  // accumulator's read reaches column 47: allocate at least 64 columns
  static constexpr int TMEM_COLS = 2 * BP < 64 ? 64 : 2 * BP;
  static constexpr int SMEM_BYTES = 1024 + STAGES * STAGE_BYTES + XCH_BYTES + 256;
};

}  // namespace

// B: rows of X (all routed rows in grouped mode, the tokens in token mode).
// gact (grouped mode, else null): [0] = number of non-empty experts, then
// their ids; goff: [E + 1] row offsets; tidx/tinv (token mode, else null):
// [B][tk] expert ids and sorted rows of each (token, slot).  All are written
// by the kernel before this one.
template <int BP, int EPI>
__global__ void __launch_bounds__(kDThreads, 1)
    gemm_decode_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX,
                       int B, int N, int K, int splits, uint32_t idesc, int w_packed,
                       float* __restrict__ part, f16* __restrict__ hout,
                       const int32_t* gact, const int32_t* goff, const int32_t* tidx,
                       const int32_t* tinv, int tk, int late, int* err) {
  using C = DecCfg<BP, EPI>;
  bool f16_bad = false;  // an H value beyond the FP16 range (SwiGLU epilogue)
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* sA = smem;
  uint8_t* sB = smem + C::STAGES * C::A_BYTES;
  float* xch = reinterpret_cast<float*>(sB + C::STAGES * C::B_BYTES);
  uint64_t* full = reinterpret_cast<uint64_t*>(sB + C::STAGES * C::B_BYTES + C::XCH_BYTES);
  uint64_t* empty = full + C::STAGES;
  uint64_t* tfull = empty + C::STAGES;
  uint64_t* tempty = tfull + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(tempty + 2);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  // late: each thread releases the next kernel only after its own dependency
  // wait (warp 1 waits for that alone), so the kernels after this one start
  // once the kernel before it, and everything before that, has completed
  if (!late) pdl_trigger();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_tiles = (N + kDBM - 1) / kDBM;
  const int n_kblk = (K + kDBK - 1) / kDBK;
  const int per_group = n_tiles * splits;
  const bool grouped = gact != nullptr;
  const bool tokens = tidx != nullptr;  // token mode (grouped SwiGLU only)
  // grouped: the unit count is device data, read after pdl_wait by each role
  int units = grouped ? 0 : per_group;

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tfull[a], 1);
      mbar_init(&tempty[a], 128);
    }
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  // unit u -> row tile of its weight tile (wrow: the blocked layout's tile
  // index for packed weights, else the first weight row), n0 within the
  // expert's N, the k-block range of split s, and the X rows [row0, row0 + m)
  auto unit_range = [&](int u, int& wrow, int& n0, int& kb0, int& kb1, int& s, int& row0,
                        int& m, int& e) {
    const int a = u / per_group;
    const int r = u - a * per_group;
    const int tile = r / splits;
    s = r - tile * splits;
    n0 = tile * kDBM;
    if (grouped) {
      e = gact[1 + a];
      row0 = tokens ? 0 : goff[e];
      m = tokens ? B : goff[e + 1] - row0;
      wrow = w_packed ? e * n_tiles + tile : e * N + n0;
    } else {
      e = 0;
      row0 = 0;
      m = B;
      wrow = w_packed ? tile : n0;
    }
    kb0 = (int)(((long long)s * n_kblk) / splits);
    kb1 = (int)(((long long)(s + 1) * n_kblk) / splits);
  };

  // weight tile of k-block kb: packed weights are in the blocked layout (4-D
  // map, one 128 x 64 tile), others row-major (2-D map from row wrow)
  auto load_w = [&](uint8_t* dst, uint64_t* bar, int kb, int wrow, uint64_t pol) {
    if (w_packed)
      tma_load_4d_hint_w(dst, &tmW, bar, 0, 0, kb, wrow, pol);
    else
      tma_load_2d_hint_w(dst, &tmW, bar, kb * kDBK, wrow, pol);
  };

  // warps 0 and 1 run converged and issue from one elected lane
  if (warp == 0) {
    {
      tma_prefetch_desc(&tmW);
      tma_prefetch_desc(&tmX);
      // weights are read once per step: evicted first, so the activations
      // the small kernels between the GEMMs read stay in L2
      const uint64_t wpol = l2_evict_first();
      // weights are never written by the kernels before this one: stream the
      // first stages of weight tiles while the previous kernel finishes
      int pre = 0;
      if (w_packed && !grouped && blockIdx.x < units) {
        int wrow, n0, kb0, kb1, s, row0, m, e;
        unit_range(blockIdx.x, wrow, n0, kb0, kb1, s, row0, m, e);
        pre = min(C::STAGES, kb1 - kb0);
        for (int i = 0; i < pre; ++i) {
          mbar_arrive_expect_tx_w(&full[i], C::STAGE_BYTES);
          load_w(sA + i * C::A_BYTES, &full[i], kb0 + i, wrow, wpol);
        }
      }
      pdl_wait();
      if (late) pdl_trigger();
      if (grouped) units = gact[0] * per_group;
      int stage = 0;
      uint32_t phase = 0;
      int g = 0;
      for (int u = blockIdx.x; u < units; u += gridDim.x) {
        int wrow, n0, kb0, kb1, s, row0, m, e;
        unit_range(u, wrow, n0, kb0, kb1, s, row0, m, e);
        for (int kb = kb0; kb < kb1; ++kb, ++g) {
          if (g < pre) {
            tma_load_2d_w(sB + stage * C::B_BYTES, &tmX, &full[stage], kb * kDBK, row0);
          } else {
            if (!mbar_wait_w(&empty[stage], phase ^ 1u, abort_flag, err)) goto prod_done;
            mbar_arrive_expect_tx_w(&full[stage], C::STAGE_BYTES);
            load_w(sA + stage * C::A_BYTES, &full[stage], kb, wrow, wpol);
            tma_load_2d_w(sB + stage * C::B_BYTES, &tmX, &full[stage], kb * kDBK, row0);
          }
          if (++stage == C::STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      for (int i = 0; i < C::STAGES; ++i) {
        if (!mbar_wait_w(&empty[stage], phase ^ 1u, abort_flag, err)) break;
        if (++stage == C::STAGES) {
          stage = 0;
          phase ^= 1u;
        }
      }
    prod_done:;
    }
  } else if (warp == 1) {
    {
      if (grouped || late) pdl_wait();
      if (late) pdl_trigger();
      if (grouped) units = gact[0] * per_group;
      int stage = 0;
      uint32_t phase = 0;
      int local = 0;
      for (int u = blockIdx.x; u < units; u += gridDim.x, ++local) {
        int wrow, n0, kb0, kb1, s, row0, m, e;
        unit_range(u, wrow, n0, kb0, kb1, s, row0, m, e);
        const int acc = local & 1;
        if (!mbar_wait_w(&tempty[acc], ((local >> 1) & 1) ^ 1u, abort_flag, err)) break;
        tc_fence_after();
        const uint32_t d = tmem + acc * BP;
        bool ok = true;
        for (int kb = kb0; kb < kb1; ++kb) {
          if (!mbar_wait_w(&full[stage], phase, abort_flag, err)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a0 = smem_u32(sA + stage * C::A_BYTES);
          const uint32_t b0 = smem_u32(sB + stage * C::B_BYTES);
#pragma unroll
          for (int k = 0; k < kDBK / 16; ++k)
            umma_f16_w(d, smem_desc_sw128(a0 + 32 * k, 16, 1024), smem_desc_sw128(b0 + 32 * k, 16, 1024),
                     idesc, (kb != kb0) || k);
          umma_commit_w(&empty[stage]);
          if (++stage == C::STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        umma_commit_w(&tfull[acc]);
      }
    }
  } else {
    pdl_wait();  // the partials may still be read by the previous kernel
    if (late) pdl_trigger();
    if (grouped) units = gact[0] * per_group;
    const int q = warp & 3;
    int local = 0;
    for (int u = blockIdx.x; u < units; u += gridDim.x, ++local) {
      int wrow, n0, kb0, kb1, s, row0, m, e;
      unit_range(u, wrow, n0, kb0, kb1, s, row0, m, e);
      if (m > BP) {  // the host sizes BP for the largest group: never taken
        record_error(err, QWEN_ERR_CAPACITY);
        m = BP;
      }
      const int acc = local & 1;
      if (!mbar_wait(&tfull[acc], (local >> 1) & 1, abort_flag, err)) break;
      tc_fence_after();
      const int n = n0 + q * 32 + lane;
      if constexpr (EPI == DEC_PARTIAL) {
        // part[s][row][n]: for each X row the 32 lanes (consecutive weight
        // rows n) write 128 contiguous bytes
        float* dst = part + (size_t)s * B * N + (size_t)row0 * N + n;
#pragma unroll 1
        for (int c = 0; c < BP; c += 32) {
          uint32_t r[32];
          tmem_ld32(tmem + (static_cast<uint32_t>(q * 32) << 16) + acc * BP + c, r);
          tmem_ld_wait();
          if (n < N) {
#pragma unroll
            for (int i = 0; i < 32; ++i)
              if (c + i < m) dst[(size_t)(c + i) * N] = __uint_as_float(r[i]);
          }
        }
        tc_fence_before();
        mbar_arrive(&tempty[acc]);
      } else {
        // tile rows 0-63 are gate rows (warps q = 0, 1), rows 64-127 the up rows
        // of the same 64 features (q = 2, 3): gate values go through shared
        // memory, the up warps form h = SiLU(gate) * up and store H[b][f]
        const int f_tile = (n0 >> 7) * 64;  // first feature of this tile
        if (q < 2) {
#pragma unroll 1
          for (int c = 0; c < BP; c += 32) {
            uint32_t r[32];
            tmem_ld32(tmem + (static_cast<uint32_t>(q * 32) << 16) + acc * BP + c, r);
            tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 32; ++i)  // xch holds BP columns (16 when BP = 16)
              if (c + i < BP) xch[(c + i) * 64 + q * 32 + lane] = __uint_as_float(r[i]);
          }
        }
        asm volatile("bar.sync 2, 128;" ::: "memory");
        if (q >= 2) {
          const int fr = (q - 2) * 32 + lane;  // feature within the tile
          const int fdim = N / 2;
#pragma unroll 1
          for (int c = 0; c < BP; c += 32) {
            uint32_t r[32];
            tmem_ld32(tmem + (static_cast<uint32_t>(q * 32) << 16) + acc * BP + c, r);
            tmem_ld_wait();
            // output row of column c + lane: the X row itself, or in token
            // mode the sorted row of the token's slot that chose this expert
            int orow = c + lane < m ? row0 + c + lane : -1;
            if (tokens && orow >= 0) {
              int found = -1;
              for (int j = 0; j < tk; ++j)
                if (tidx[(size_t)orow * tk + j] == e) found = tinv[(size_t)orow * tk + j];
              orow = found;
            }
#pragma unroll
            for (int i = 0; i < 32; ++i) {
              const int row = __shfl_sync(0xffffffffu, orow, i);
              if (row >= 0 && f_tile + fr < fdim) {
                const float gv = xch[(c + i) * 64 + fr];
                hout[(size_t)row * fdim + f_tile + fr] =
                    f16_chk(silu_f(gv) * __uint_as_float(r[i]), f16_bad);
              }
            }
          }
        }
        tc_fence_before();
        mbar_arrive(&tempty[acc]);
        asm volatile("bar.sync 2, 128;" ::: "memory");  // xch free for the next tile
      }
    }
  }
  record_overflow(err, f16_bad);
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

// ------------------------------------------------------------------ reductions
// Partials are part[s][b][n]; the splits are summed in order s = 0, 1, ...

// v[e] += src[s * plane + e * estride] for s = 0 .. splits-1 in order, for the
// first nvalid of the PER values.  The loads of CH splits are issued together
// before their adds: these reductions are bound by load latency, not bytes.
template <int PER, int CH>
__device__ __forceinline__ void add_splits(const float* __restrict__ src, size_t plane,
                                           int estride, int splits, int nvalid,
                                           float (&v)[PER]) {
  for (int s0 = 0; s0 < splits; s0 += CH) {
    float t[CH][PER];
#pragma unroll
    for (int c = 0; c < CH; ++c)
#pragma unroll
      for (int e = 0; e < PER; ++e)
        t[c][e] = (s0 + c < splits && e < nvalid)
                      ? src[(size_t)(s0 + c) * plane + (size_t)e * estride]
                      : 0.f;
#pragma unroll
    for (int c = 0; c < CH; ++c)
#pragma unroll
      for (int e = 0; e < PER; ++e)
        if (s0 + c < splits) v[e] += t[c][e];
  }
}

__global__ void reduce_resid_kernel(const float* __restrict__ part, int splits, int B, int N,
                                    const bf16* __restrict__ resid,
                                    const float* __restrict__ resid32, bf16* __restrict__ out,
                                    float* __restrict__ out32) {
  pdl_trigger();
  pdl_wait();
  const int i = blockIdx.x * blockDim.x + threadIdx.x;  // over B * N, n fastest
  if (i >= N * B) return;
  const size_t plane = (size_t)B * N;
  float acc[1] = {0.f};
  add_splits<1, 8>(part + i, plane, 0, splits, 1, acc);
  const float r = acc[0] + (resid32 ? resid32[i] : __bfloat162float(resid[i]));
  if (out) out[i] = __float2bfloat16_rn(r);
  if (out32) out32[i] = r;
}

// h[b][j] = SiLU(gate_j) * up_j with gate row (j/64)*128 + j%64 and up row +64.
__global__ void reduce_swiglu_kernel(const float* __restrict__ part, int splits, int B, int f,
                                     f16* __restrict__ h, int* err) {
  pdl_trigger();
  pdl_wait();
  const int i = blockIdx.x * blockDim.x + threadIdx.x;  // over B * f, j fastest
  if (i >= f * B) return;
  const int b = i / f, j = i - b * f;
  const int N = 2 * f;
  const int n_gate = (j >> 6) * 128 + (j & 63);
  const size_t plane = (size_t)B * N;
  const float* src = part + (size_t)b * N + n_gate;
  float gu[2] = {0.f, 0.f};  // gate, up
  add_splits<2, 8>(src, plane, 64, splits, 2, gu);
  bool bad = false;
  h[i] = f16_chk(silu_f(gu[0]) * gu[1], bad);
  record_overflow(err, bad);
}

// One warp per (b, head): lane e holds channels e, e+32, e+64, e+96 (dh = 128)
// or e, e+32 (dh = 64), so the rotate_half pairs (i, i + dh/2) stay in a lane.
// The same step as qkv_head_finish: bias, QK-norm (warp reduction over dh),
// RoPE from the FP64-built table, then Q store or K/V cache append.
template <int DH>
__global__ void reduce_qkv_kernel(const float* __restrict__ part, int splits, int B, int Nqkv,
                                  QkvParams p, int* err) {
  pdl_trigger();
  pdl_wait();
  constexpr int PER = DH / 32;
  const int wid = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  const int heads = p.Hq + 2 * p.Hkv;
  if (wid >= B * heads) return;
  const int b = wid / heads, head = wid - b * heads;
  const size_t plane = (size_t)B * Nqkv;
  const float* src = part + (size_t)b * Nqkv + (size_t)head * DH + lane;
  float v[PER];
#pragma unroll
  for (int e = 0; e < PER; ++e) v[e] = 0.f;
  add_splits<PER, 32 / PER>(src, plane, 32, splits, PER, v);
  const int kind = head < p.Hq ? 0 : (head < p.Hq + p.Hkv ? 1 : 2);
  if (p.bias) {
#pragma unroll
    for (int e = 0; e < PER; ++e) v[e] += p.bias[(size_t)head * DH + lane + 32 * e];
  }
  if (kind < 2) {
    if (p.gamma_q) {
      float ss = 0.f;
#pragma unroll
      for (int e = 0; e < PER; ++e) ss = fmaf(v[e], v[e], ss);
      ss = warp_sum(ss);
      const float rstd = rsqrtf(ss / (float)DH + p.eps);
      const bf16* gm = kind == 0 ? p.gamma_q : p.gamma_k;
#pragma unroll
      for (int e = 0; e < PER; ++e) v[e] = __bfloat162float(gm[lane + 32 * e]) * (v[e] * rstd);
    }
    const int pos = p.positions[b];
    if (pos < 0 || pos >= p.max_position) {
      if (lane == 0) record_error(err, QWEN_ERR_RANGE);
      return;
    }
    const float2* tab = p.rope + (size_t)pos * (DH / 2);
#pragma unroll
    for (int e = 0; e < PER / 2; ++e) {
      const float2 cs = tab[lane + 32 * e];
      const float lo = v[e], hi = v[e + PER / 2];
      v[e] = lo * cs.x - hi * cs.y;
      v[e + PER / 2] = hi * cs.x + lo * cs.y;
    }
  }
  bf16* dst;
  if (kind == 0) {
    dst = static_cast<bf16*>(p.q_out) + ((size_t)b * p.Hq + head) * DH;  // T == 1, BF16
  } else {
    const int slot = p.slot0[b];
    if (slot < 0 || slot >= p.max_seq) {
      if (lane == 0) record_error(err, QWEN_ERR_RANGE);
      return;
    }
    const int g = kind == 1 ? head - p.Hq : head - p.Hq - p.Hkv;
    dst = (kind == 1 ? p.k_cache : p.v_cache) + (((size_t)b * p.Hkv + g) * p.max_seq + slot) * DH;
  }
#pragma unroll
  for (int e = 0; e < PER; ++e) dst[lane + 32 * e] = __float2bfloat16_rn(v[e]);
}

// One CTA per sequence row b: R[b] = sum_s part[s][b] + residual (FP32 out),
// then Z[b] = gamma * R[b] / sqrt(mean(R[b]^2) + eps) as the FP16 operand of
// the next projection: the O-projection reduction fused with RMSNorm_2.
template <int PER>
__global__ void __launch_bounds__(1024) reduce_resid_norm_kernel(
    const float* __restrict__ part, int splits, int B, int N, const bf16* __restrict__ resid,
    const float* __restrict__ resid32, float* __restrict__ out32, const bf16* __restrict__ gamma,
    float eps, f16* __restrict__ z, size_t zs, f16* __restrict__ z_lo, int* err) {
  pdl_trigger();
  __shared__ float red[32];
  const int b = blockIdx.x;
  const size_t plane = (size_t)B * N;
  const size_t row = (size_t)b * N;
  // gamma is a weight (no kernel writes it): read before the wait, so the
  // scaling after the row reduction needs no further load
  float gm[PER];
#pragma unroll
  for (int j = 0; j < PER; ++j) {
    const int n = threadIdx.x + 1024 * j;
    gm[j] = n < N ? __bfloat162float(gamma[n]) : 0.f;
  }
  pdl_wait();
  float v[PER];
#pragma unroll
  for (int j = 0; j < PER; ++j) {
    const int n = threadIdx.x + 1024 * j;
    v[j] = 0.f;
    if (n < N) v[j] = resid32 ? resid32[row + n] : __bfloat162float(resid[row + n]);
  }
  // columns threadIdx.x + 1024 j, j < nvalid, are inside the row
  const int nvalid = (int)threadIdx.x < N ? min(PER, (N - 1 - (int)threadIdx.x) / 1024 + 1) : 0;
  add_splits<PER, 32 / PER>(part + row + threadIdx.x, plane, 1024, splits, nvalid, v);
  float ss = 0.f;
#pragma unroll
  for (int j = 0; j < PER; ++j) {
    const int n = threadIdx.x + 1024 * j;
    if (n < N) {
      out32[row + n] = v[j];
      ss = fmaf(v[j], v[j], ss);
    }
  }
  ss = warp_sum(ss);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = ss;
  __syncthreads();
  float tot = 0.f;
#pragma unroll
  for (int w = 0; w < 32; ++w) tot += red[w];
  const float rstd = rsqrtf(tot / (float)N + eps);
  const size_t zrow = (size_t)b * zs;
  bool bad = false;
#pragma unroll
  for (int j = 0; j < PER; ++j) {
    const int n = threadIdx.x + 1024 * j;
    if (n < N) {
      const float o = gm[j] * (v[j] * rstd);
      const f16 hi = f16_chk(o, bad);
      z[zrow + n] = hi;
      if (z_lo) z_lo[zrow + n] = f16_chk(o - __half2float(hi), bad);
    }
  }
  record_overflow(err, bad);
}

__global__ void reduce_f32_kernel(const float* __restrict__ part, int splits, int B, int N,
                                  float* __restrict__ out, int ldo) {
  pdl_trigger();
  pdl_wait();
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= N * B) return;
  const int b = i / N, n = i - b * N;
  const size_t plane = (size_t)B * N;
  float acc[1] = {0.f};
  add_splits<1, 8>(part + i, plane, 0, splits, 1, acc);
  out[(size_t)b * ldo + n] = acc[0];
}

// ------------------------------------------------------------------ host side

static PFN_cuTensorMapEncodeTiled_v12000 enc_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}

// Packed weights: 128 x 64 tiles of 16 KB (see the prefill GEMM), one tile a box.
static bool tmap_blocked(CUtensorMap* m, const void* base, uint64_t row_tiles, uint64_t K,
                         bool f16) {
  auto enc = enc_fn();
  if (!enc || (reinterpret_cast<uintptr_t>(base) & 15) || (K % kDBK)) return false;
  const uint64_t kt = K / kDBK;
  cuuint64_t dims[4] = {(cuuint64_t)kDBK, (cuuint64_t)kDBM, kt, row_tiles};
  cuuint64_t strides[3] = {kDBK * 2, kDBM * kDBK * 2, kt * kDBM * kDBK * 2};
  cuuint32_t box[4] = {(cuuint32_t)kDBK, (cuuint32_t)kDBM, 1, 1};
  cuuint32_t es[4] = {1, 1, 1, 1};
  return enc(m, f16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4,
             const_cast<void*>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
             CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

static bool tmap2d(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols, uint64_t ld,
                   uint32_t box_rows, bool f16) {
  auto enc = enc_fn();
  if (!enc || (reinterpret_cast<uintptr_t>(base) & 15) || ((ld * 2) & 15)) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {ld * 2};
  cuuint32_t box[2] = {(cuuint32_t)kDBK, box_rows};
  cuuint32_t es[2] = {1, 1};
  return enc(m, f16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
             const_cast<void*>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

static int pad_batch(int B) {
  if (B <= 16) return 16;
  if (B <= 32) return 32;
  if (B <= 64) return 64;
  if (B <= 128) return 128;
  return 256;
}

// K splits for an [N, K] weight (times `groups` in grouped mode) and B tokens:
// the split count with the smallest modelled time, where a launch takes the
// longer of streaming all weight bytes from HBM and the busiest SM pulling its
// units through TMA, plus the split partials (written, then read by the
// reduction) and a fixed cost per unit on the busiest SM.  Few splits leave
// SMs idle; many make small units whose partials and hand-offs cost more than
// the extra SMs gain.  Rates: measured GB300 copy bandwidth and per-SM TMA
// ingress (about 6.6 TB/s and 100-120 GB/s; 70 GB/s is used to keep a margin).
int decode_splits(int N, int K, int B, int groups) {
  const int sms = device_sm_count();
  const int tiles = (N + kDBM - 1) / kDBM * groups;
  const int kblk = (K + kDBK - 1) / kDBK;
  const int bp = pad_batch(B < 1 ? 1 : (B > 256 ? 256 : B));
  constexpr double kHbm = 6.6e12, kSmIngress = 7.0e10, kUnitCost = 2.0e-7;
  const double w_time = (double)tiles * kblk * kDBM * kDBK * 2 / kHbm;
  const double kblk_bytes = (double)(kDBM + bp) * kDBK * 2;  // weight + X tile
  const double part_bytes = (double)kDBM * B * 4;            // one unit's partials
  int best = 1;
  double best_t = 1e30;
  for (int s = 1; s <= 32 && (s == 1 || s <= kblk / 2); ++s) {
    const int units = tiles * s;
    const int per_sm = (units + sms - 1) / sms;
    const int kb = (kblk + s - 1) / s;
    const double sm_time = (double)per_sm * kb * kblk_bytes / kSmIngress;
    const double t = (w_time > sm_time ? w_time : sm_time) +
                     (s > 1 ? 2.0 * units * part_bytes / kHbm : 0.0) + per_sm * kUnitCost;
    if (t < best_t * (1.0 - 1e-9)) {
      best_t = t;
      best = s;
    }
  }
  return best;
}

size_t decode_part_bytes(const qwen_layer_config& c, int B) {
  const size_t d = c.d, nq = (size_t)c.n_q_heads * c.head_dim,
               nqkv = nq + 2 * (size_t)c.n_kv_heads * c.head_dim, f = c.ffn;
  size_t m = 0;
  auto upd = [&](size_t N, size_t K) {
    const size_t s = decode_splits((int)N, (int)K, B);
    const size_t need = s * N * (size_t)B * 4;
    if (need > m) m = need;
  };
  upd(nqkv, d);
  upd(d, nq);
  if (c.n_experts == 0) {
    upd(2 * f, d);
    upd(d, f);
  } else {
    upd(router_rows(c), 2 * d);  // the router over [Z_hi | Z_lo]
    if (c.shared_ffn) upd(d, c.shared_ffn);  // the shared expert's down projection
    if (B <= kMoeDecodeMaxRows) {  // grouped expert down projection, B*k rows
      const int rows = B * c.top_k;
      const int groups = rows < c.n_experts ? rows : c.n_experts;
      const size_t need = (size_t)decode_splits(d, f, B, groups) * rows * d * 4;
      if (need > m) m = need;
    }
  }
  return m;
}

template <int BP, int EPI>
static qwen_status launch_dec(const CUtensorMap& tw, const CUtensorMap& tx, int B, int N, int K,
                              int splits, bool op_f16, bool w_packed, float* part, f16* hout,
                              const int32_t* gact, const int32_t* goff, const int32_t* tidx,
                              const int32_t* tinv, int tk, int max_groups, bool late, int* err,
                              cudaStream_t st) {
  using C = DecCfg<BP, EPI>;
  auto kern = gemm_decode_kernel<BP, EPI>;
  static std::atomic<uint64_t> attr{0};  // one bit per device
  if (!smem_attr_once(kern, C::SMEM_BYTES, attr)) return QWEN_ERR_CUDA;
  const int units = ((N + kDBM - 1) / kDBM) * splits * max_groups;
  const int sms = device_sm_count();
  const int grid = units < sms ? units : sms;
  launch_k(kern, dim3(grid), dim3(kDThreads), C::SMEM_BYTES, st, tw, tx, B, N, K, splits,
           idesc_f32acc(kDBM, BP, op_f16), w_packed ? 1 : 0, part, hout, gact, goff, tidx, tinv,
           tk, late ? 1 : 0, err);
  count_launches();
  return cudaGetLastError() == cudaSuccess ? QWEN_OK : QWEN_ERR_CUDA;
}

// Shared host path of the dense and grouped decode GEMMs.  W: `groups` stacked
// [N, K] weights, packed (blocked layout, each weight's rows padded to 128) or
// row-major; X: B rows, ldx apart; BP covers max_m rows.
static qwen_status decode_gemm_launch(const void* W, int groups, const void* X, int ldx, int B,
                                      int max_m, int N, int K, int splits, bool op_f16,
                                      bool w_packed, float* part, f16* hout,
                                      const int32_t* gact, const int32_t* goff,
                                      const int32_t* tidx, const int32_t* tinv, int tk,
                                      int max_groups, int* err, cudaStream_t st,
                                      bool late = false) {
  if (B <= 0 || max_m <= 0 || max_m > 256) return QWEN_ERR_UNSUPPORTED;
  if ((K & 7) || splits < 1 || max_groups < 1) return QWEN_ERR_UNSUPPORTED;
  const int bp = pad_batch(max_m);
  CUtensorMap tw, tx;
  if (w_packed) {
    if (!tmap_blocked(&tw, W, (uint64_t)groups * ((N + kDBM - 1) / kDBM), (uint64_t)K, op_f16))
      return QWEN_ERR_CUDA;
  } else if (!tmap2d(&tw, W, (uint64_t)groups * N, (uint64_t)K, (uint64_t)K, kDBM, op_f16)) {
    return QWEN_ERR_CUDA;
  }
  if (!tmap2d(&tx, X, (uint64_t)B, (uint64_t)K, (uint64_t)ldx, bp, op_f16)) return QWEN_ERR_CUDA;
#define QWEN_DEC_CASE(BPV)                                                                        \
  case BPV:                                                                                       \
    return hout ? launch_dec<BPV, DEC_SWIGLU>(tw, tx, B, N, K, 1, op_f16, w_packed, nullptr,      \
                                              hout, gact, goff, tidx, tinv, tk, max_groups, late, \
                                              err, st)                                            \
                : launch_dec<BPV, DEC_PARTIAL>(tw, tx, B, N, K, splits, op_f16, w_packed, part,   \
                                               nullptr, gact, goff, nullptr, nullptr, 0,          \
                                               max_groups, late, err, st);
  switch (bp) {
    QWEN_DEC_CASE(16)
    QWEN_DEC_CASE(32)
    QWEN_DEC_CASE(64)
    QWEN_DEC_CASE(128)
    QWEN_DEC_CASE(256)
    default: return QWEN_ERR_UNSUPPORTED;
  }
#undef QWEN_DEC_CASE
}

qwen_status gemm_decode_splitk(const void* W, const void* X, int ldx, int B, int N, int K,
                               int splits, bool op_f16, float* part, int* err, cudaStream_t st,
                               bool w_packed, f16* swiglu_out, bool late_release) {
  return decode_gemm_launch(W, 1, X, ldx, B, B, N, K, splits, op_f16, w_packed, part, swiglu_out,
                            nullptr, nullptr, nullptr, nullptr, 0, 1, err, st, late_release);
}

qwen_status gemm_decode_grouped(const void* W, int E, const void* X, int rows, int max_m, int N,
                                int K, int splits, const int32_t* act, const int32_t* offsets,
                                int max_groups, float* part, f16* swiglu_out, int* err,
                                cudaStream_t st) {
  if (!act || !offsets || E <= 0) return QWEN_ERR_INVALID_ARG;
  return decode_gemm_launch(W, E, X, K, rows, max_m, N, K, splits, /*op_f16=*/true,
                            /*w_packed=*/true, part, swiglu_out, act, offsets, nullptr, nullptr, 0,
                            max_groups, err, st);
}

qwen_status gemm_decode_grouped_tokens(const void* W, int E, const void* X, int ldx, int T,
                                       int N, int K, const int32_t* act, const int32_t* idx,
                                       const int32_t* inv, int k, int max_groups, f16* h_out,
                                       int* err, cudaStream_t st) {
  if (!act || !idx || !inv || !h_out || E <= 0 || k < 1) return QWEN_ERR_INVALID_ARG;
  return decode_gemm_launch(W, E, X, ldx, T, T, N, K, 1, /*op_f16=*/true, /*w_packed=*/true,
                            nullptr, h_out, act, nullptr, idx, inv, k,
                            max_groups, err, st);
}

static inline int blocks_for(long long n, int t) { return (int)((n + t - 1) / t); }

qwen_status reduce_resid(const float* part, int splits, int B, int N, const bf16* resid,
                         const float* resid32, bf16* out, float* out32, cudaStream_t st) {
  launch_k(reduce_resid_kernel, dim3(blocks_for((long long)N * B, 256)), dim3(256), 0, st, part,
           splits, B, N, resid, resid32, out, out32);
  count_launches();
  return cudaGetLastError() == cudaSuccess ? QWEN_OK : QWEN_ERR_CUDA;
}

qwen_status reduce_swiglu(const float* part, int splits, int B, int f, f16* h, int* err,
                          cudaStream_t st) {
  launch_k(reduce_swiglu_kernel, dim3(blocks_for((long long)f * B, 256)), dim3(256), 0, st, part,
           splits, B, f, h, err);
  count_launches();
  return cudaGetLastError() == cudaSuccess ? QWEN_OK : QWEN_ERR_CUDA;
}

qwen_status reduce_qkv(const float* part, int splits, int B, int Nqkv, const QkvParams& p, int* err,
                       cudaStream_t st) {
  const long long threads = 32LL * B * (p.Hq + 2 * p.Hkv);
  if (p.dh == 128)
    launch_k(reduce_qkv_kernel<128>, dim3(blocks_for(threads, 128)), dim3(128), 0, st, part, splits,
             B, Nqkv, p, err);
  else
    launch_k(reduce_qkv_kernel<64>, dim3(blocks_for(threads, 128)), dim3(128), 0, st, part, splits,
             B, Nqkv, p, err);
  count_launches();
  return cudaGetLastError() == cudaSuccess ? QWEN_OK : QWEN_ERR_CUDA;
}

qwen_status reduce_resid_norm(const float* part, int splits, int B, int N, const bf16* resid,
                              const float* resid32, float* out32, const bf16* gamma, float eps,
                              f16* z, int* err, cudaStream_t st, size_t z_stride, f16* z_lo) {
  if (N > 1024 * 8) return QWEN_ERR_UNSUPPORTED;
  const size_t zs = z_stride ? z_stride : (size_t)N;
  if (N <= 1024 * 4)
    launch_k(reduce_resid_norm_kernel<4>, dim3(B), dim3(1024), 0, st, part, splits, B, N, resid,
             resid32, out32, gamma, eps, z, zs, z_lo, err);
  else
    launch_k(reduce_resid_norm_kernel<8>, dim3(B), dim3(1024), 0, st, part, splits, B, N, resid,
             resid32, out32, gamma, eps, z, zs, z_lo, err);
  count_launches();
  return cudaGetLastError() == cudaSuccess ? QWEN_OK : QWEN_ERR_CUDA;
}

qwen_status reduce_f32(const float* part, int splits, int B, int N, float* out, int ldo,
                       cudaStream_t st) {
  launch_k(reduce_f32_kernel, dim3(blocks_for((long long)N * B, 256)), dim3(256), 0, st, part,
           splits, B, N, out, ldo);
  count_launches();
  return cudaGetLastError() == cudaSuccess ? QWEN_OK : QWEN_ERR_CUDA;
}

}  // namespace qwen
