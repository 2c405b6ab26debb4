// Causal GQA flash attention for prefill on tcgen05 tensor cores (sm_103a).
//
// Qwen3 layer page ("推理系统 03"), §7-§9: query head h of token t reads KV head
// g = floor(h / (Hq/Hkv)); S = q.k / sqrt(dh) plus the causal mask (a key in
// slot s is visible to the query in slot s_q iff s <= s_q); stable softmax over
// visible keys; o = sum_s a_s v_s; heads are concatenated along features.
// "Qwen2.5-7B 结构拆解" §05.2 / §05.4: K/V are indexed per group (no physical
// repeat) and tiles above the diagonal are skipped.  §12 of the Qwen3 page: the
// [T,T] probability matrix is never written to memory.
//
// Operands: the queries and the keys/values this call computed are FP16 (the
// QKV epilogue writes FP16 copies of the new K/V rows besides the BF16 cache),
// so S = Q K^T and O += P V run on FP16 tensor-core operands with P in FP16.
// Key tiles that reach below the sequence's first new slot (chunked prefill
// onto a filled cache) come from the BF16 cache instead; for those the
// softmax warps convert Q to a BF16 copy once and P is rounded to BF16.
//
// One CTA = one (sequence b, query head h, tile of 128 query rows).
//   warp 0      TMA: Q tile once, then K/V tiles of 128 keys (2-stage ring)
//   warp 1      TMEM allocator + MMA issuer:
//                 S_j = Q K_j^T  -> TMEM (two S buffers, 128 cols each)
//                 O  += P_j V_j  -> TMEM (dh cols), P_j from shared memory,
//                 V_j read MN-major (dh contiguous) straight from the cache tile
//   warps 2..5  softmax: thread = query row; online max/sum in FP32 with the
//               rescale of O deferred until the max grows by 2^8; P -> FP16
//               (BF16 for cache tiles) in the 128-byte-swizzled K-major layout
//               the MMA reads; final O / l.
#include "common.cuh"
#include "internal.h"

#include <cudaTypedefs.h>

namespace qwen {

namespace {

constexpr int kQT = 128;  // query rows per CTA
constexpr int kKT = 128;  // keys per tile
constexpr int kAttnThreads = 192;
constexpr float kRescaleLog2 = 8.0f;  // defer O rescale until the max grew by 2^8

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

template <int DH>
struct AttnCfg {
  static constexpr int TILE_BYTES = kKT * DH * 2;  // one [128 x DH] 16-bit tile
  static constexpr int Q_OFF = 0;                            // Q (FP16)
  static constexpr int QB_OFF = TILE_BYTES;                  // BF16 copy of Q
  static constexpr int P_OFF = 2 * TILE_BYTES;               // P [128 x 128] 16-bit
  static constexpr int K_OFF = P_OFF + kQT * kKT * 2;        // 2 stages
  static constexpr int V_OFF = K_OFF + 2 * TILE_BYTES;       // 2 stages
  static constexpr int BAR_OFF = V_OFF + 2 * TILE_BYTES;
  static constexpr int SMEM_BYTES = 1024 + BAR_OFF + 256;
  static constexpr int S_COL0 = 0;    // S buffers at columns 0 and 128
  static constexpr int O_COL = 256;   // O accumulator
  static constexpr int TMEM_COLS = 512;
};

struct AttnArgs {
  int B, T, Hq, Hkv, max_seq;
  const int32_t* slot0;  // [B] cache slot of the first new token
  f16* out;              // [B*T][Hq*DH], FP16 operand of the O projection
  float scale_log2;      // log2(e) / sqrt(dh)
  int* err;
};

}  // namespace

template <int DH>
__global__ void __launch_bounds__(kAttnThreads, 1)
    attn_prefill_kernel(const __grid_constant__ CUtensorMap tmQ,
                        const __grid_constant__ CUtensorMap tmK,
                        const __grid_constant__ CUtensorMap tmV,
                        const __grid_constant__ CUtensorMap tmK16,
                        const __grid_constant__ CUtensorMap tmV16, AttnArgs a) {
  pdl_trigger();
  pdl_wait();
  using C = AttnCfg<DH>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* sQ = smem + C::Q_OFF;
  uint8_t* sQb = smem + C::QB_OFF;
  uint8_t* sP = smem + C::P_OFF;
  uint8_t* sK = smem + C::K_OFF;
  uint8_t* sV = smem + C::V_OFF;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::BAR_OFF);
  uint64_t* q_full = bars + 0;
  uint64_t* k_full = bars + 1;    // [2]
  uint64_t* v_full = bars + 3;    // [2]
  uint64_t* kv_empty = bars + 5;  // [2]
  uint64_t* s_full = bars + 7;    // [2]
  uint64_t* s_free = bars + 9;    // [2]
  uint64_t* p_full = bars + 11;
  uint64_t* o_done = bars + 12;
  uint64_t* qb_ready = bars + 13;  // BF16 copy of Q written (chunked prefill only)
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 14);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // heaviest (last) query tiles first
  const int n_qt = (a.T + kQT - 1) / kQT;
  const int bh_count = a.B * a.Hq;
  const int qt = n_qt - 1 - blockIdx.x / bh_count;
  const int bh = blockIdx.x % bh_count;
  const int b = bh / a.Hq, h = bh - b * a.Hq;
  const int g = h / (a.Hq / a.Hkv);
  const int t0 = qt * kQT;
  const int s0 = a.slot0[b];
  const int q_last = min(t0 + kQT, a.T) - 1;   // last valid query row of the tile
  const int kmax = s0 + q_last;                // largest visible key slot
  const int n_kv = kmax / kKT + 1;             // key tiles 0..n_kv-1
  const int q_row0 = (b * a.Hq + h) * a.T + t0;        // row in the Q view
  const int kv_row0 = (b * a.Hkv + g) * a.max_seq;     // row in the cache view
  const int kv16_row0 = (b * a.Hkv + g) * a.T - s0;    // + key slot = row in the fresh view

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&k_full[i], 1);
      mbar_init(&v_full[i], 1);
      mbar_init(&kv_empty[i], 1);
      mbar_init(&s_full[i], 1);
      mbar_init(&s_free[i], 128);
    }
    mbar_init(p_full, 128);
    mbar_init(o_done, 1);
    mbar_init(qb_ready, 128);
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

  if (warp == 0) {
    if (lane == 0) {
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
      tma_prefetch_desc(&tmK16);
      tma_prefetch_desc(&tmV16);
      mbar_arrive_expect_tx(q_full, C::TILE_BYTES);
#pragma unroll
      for (int c = 0; c < DH / 64; ++c)
        tma_load_2d(sQ + c * kQT * 128, &tmQ, q_full, c * 64, q_row0);
      for (int j = 0; j < n_kv; ++j) {
        const int st = j & 1;
        if (!mbar_wait(&kv_empty[st], ((j >> 1) & 1) ^ 1u, abort_flag, a.err)) break;
        // tiles entirely at or above the first new slot come from the FP16
        // copies of this call's rows, the others from the BF16 cache
        const bool fresh = j * kKT >= s0;
        const CUtensorMap* mk = fresh ? &tmK16 : &tmK;
        const CUtensorMap* mv = fresh ? &tmV16 : &tmV;
        const int row = fresh ? kv16_row0 + j * kKT : kv_row0 + j * kKT;
        mbar_arrive_expect_tx(&k_full[st], C::TILE_BYTES);
#pragma unroll
        for (int c = 0; c < DH / 64; ++c)
          tma_load_2d(sK + st * C::TILE_BYTES + c * kKT * 128, mk, &k_full[st], c * 64, row);
        mbar_arrive_expect_tx(&v_full[st], C::TILE_BYTES);
#pragma unroll
        for (int c = 0; c < DH / 64; ++c)
          tma_load_2d(sV + st * C::TILE_BYTES + c * kKT * 128, mv, &v_full[st], c * 64, row);
      }
      // drain: every issued tile is consumed before exit
      for (int j = n_kv; j < n_kv + 2; ++j) {
        if (!mbar_wait(&kv_empty[j & 1], ((j >> 1) & 1) ^ 1u, abort_flag, a.err)) break;
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t idesc_s16 = idesc_f32acc(kQT, kKT, true);
      constexpr uint32_t idesc_sb = idesc_f32acc(kQT, kKT, false);
      constexpr uint32_t idesc_o16 = idesc_f32acc(kQT, DH, true, false, /*b_mn_major=*/true);
      constexpr uint32_t idesc_ob = idesc_f32acc(kQT, DH, false, false, /*b_mn_major=*/true);
      bool qb_waited = false;
      auto issue_s = [&](int j) -> bool {
        const int st = j & 1;
        const bool fresh = j * kKT >= s0;
        if (!fresh && !qb_waited) {
          if (!mbar_wait(qb_ready, 0, abort_flag, a.err)) return false;
          tc_fence_after();
          qb_waited = true;
        }
        const uint32_t q0 = smem_u32(fresh ? sQ : sQb);
        const uint32_t k0 = smem_u32(sK + st * C::TILE_BYTES);
        const uint32_t d = tmem + C::S_COL0 + st * kKT;
#pragma unroll
        for (int k = 0; k < DH / 16; ++k) {
          const uint32_t off = (k >> 2) * (kQT * 128) + (k & 3) * 32;
          umma_f16(d, smem_desc_sw128(q0 + off, 16, 1024), smem_desc_sw128(k0 + off, 16, 1024),
                   fresh ? idesc_s16 : idesc_sb, k != 0);
        }
        umma_commit(&s_full[st]);
        return true;
      };
      bool ok = mbar_wait(q_full, 0, abort_flag, a.err) &&
                mbar_wait(&k_full[0], 0, abort_flag, a.err);
      if (ok) {
        tc_fence_after();
        ok = issue_s(0);
      }
      const uint32_t p0 = smem_u32(sP);
      for (int j = 0; ok && j < n_kv; ++j) {
        const int st = j & 1;
        if (j + 1 < n_kv) {
          const int j1 = j + 1, st1 = j1 & 1;
          if (!mbar_wait(&k_full[st1], (j1 >> 1) & 1, abort_flag, a.err)) break;
          if (j1 >= 2 && !mbar_wait(&s_free[st1], ((j1 >> 1) - 1) & 1, abort_flag, a.err)) break;
          tc_fence_after();
          if (!issue_s(j1)) break;
        }
        if (!mbar_wait(p_full, j & 1, abort_flag, a.err)) break;
        if (!mbar_wait(&v_full[st], (j >> 1) & 1, abort_flag, a.err)) break;
        tc_fence_after();
        const uint32_t v0 = smem_u32(sV + st * C::TILE_BYTES);
#pragma unroll
        for (int k = 0; k < kKT / 16; ++k) {
          // A = P rows x keys (K-major, two 64-key swizzle blocks of 16 KB)
          const uint32_t pa = p0 + (k >> 2) * (kQT * 128) + (k & 3) * 32;
          // B = V keys x dh read MN-major: 16 keys = 16 rows of 128 B; next 64-wide
          // dh block 16 KB away (LBO), next 8 keys 1 KB away (SBO)
          const uint32_t vb = v0 + k * 16 * 128;
          umma_f16(tmem + C::O_COL, smem_desc_sw128(pa, 16, 1024),
                   smem_desc_sw128(vb, kKT * 128, 1024), (j * kKT >= s0) ? idesc_o16 : idesc_ob,
                   (j | k) != 0);
        }
        umma_commit(o_done);
        umma_commit(&kv_empty[st]);
      }
    }
  } else {
    // softmax / epilogue warps
    const int qw = warp & 3;
    const int r = qw * 32 + lane;  // query row within the tile
    const int t = t0 + r;
    const int s_q = s0 + t;        // this row's cache slot
    const uint32_t lane_base = static_cast<uint32_t>(qw * 32) << 16;
    float m_used = -INFINITY, l_sum = 0.f;
    bool ok = true;
    if (s0 > 0) {
      // some key tiles come from the BF16 cache: convert this row of Q once
      // (element by element, so the swizzled placement is kept)
      if (!mbar_wait(q_full, 0, abort_flag, a.err)) ok = false;
      if (ok) {
#pragma unroll
        for (int blk = 0; blk < DH / 64; ++blk) {
          const uint4* src = reinterpret_cast<const uint4*>(sQ + blk * (kQT * 128) + r * 128);
          uint4* dst = reinterpret_cast<uint4*>(sQb + blk * (kQT * 128) + r * 128);
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            const uint4 u = src[c];
            const uint32_t w[4] = {u.x, u.y, u.z, u.w};
            uint32_t o[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const float2 f = unpack_f16x2(w[e]);
              o[e] = pack_bf16x2(f.x, f.y);
            }
            dst[c] = make_uint4(o[0], o[1], o[2], o[3]);
          }
        }
        fence_proxy_async_smem();
        mbar_arrive(qb_ready);
      }
    }
    for (int j = 0; ok && j < n_kv; ++j) {
      const bool fresh = j * kKT >= s0;
      const int st = j & 1;
      if (!mbar_wait(&s_full[st], (j >> 1) & 1, abort_flag, a.err)) { ok = false; break; }
      tc_fence_after();
      float s[kKT];
#pragma unroll
      for (int c = 0; c < kKT / 32; ++c) {
        uint32_t rr[32];
        tmem_ld32(tmem + lane_base + C::S_COL0 + st * kKT + 32 * c, rr);
        tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < 32; ++i) s[32 * c + i] = __uint_as_float(rr[i]);
      }
      tc_fence_before();
      mbar_arrive(&s_free[st]);
      // scale (log2 domain) and causal mask
      const int key0 = j * kKT;
      float mx = -INFINITY;
#pragma unroll
      for (int i = 0; i < kKT; ++i) {
        const float v = (key0 + i <= s_q) ? s[i] * a.scale_log2 : -INFINITY;
        s[i] = v;
        mx = fmaxf(mx, v);
      }
      float alpha = 1.f;
      if (mx > m_used + kRescaleLog2 || m_used == -INFINITY) {
        const float m_new = fmaxf(mx, m_used);
        alpha = (m_used == -INFINITY) ? 0.f : ex2(m_used - m_new);
        l_sum *= alpha;
        m_used = m_new;
      }
      // P = 2^(s - m) rounded to the tile's operand type; l sums the rounded values
      uint32_t pk[kKT / 2];
#pragma unroll
      for (int i = 0; i < kKT / 2; ++i) {
        const float p0 = ex2(s[2 * i] - m_used);
        const float p1 = ex2(s[2 * i + 1] - m_used);
        pk[i] = pack2(p0, p1, fresh);
        const float2 rp = fresh ? unpack_f16x2(pk[i]) : unpack_bf16x2(pk[i]);
        l_sum += rp.x + rp.y;
      }
      if (j > 0) {
        // PV of the previous tile must be done before P is overwritten and O rescaled
        if (!mbar_wait(o_done, (j - 1) & 1, abort_flag, a.err)) { ok = false; break; }
        tc_fence_after();
        const bool need = __any_sync(0xffffffffu, alpha != 1.f);
        if (need) {
#pragma unroll
          for (int c = 0; c < DH / 32; ++c) {
            uint32_t oo[32];
            const uint32_t addr = tmem + lane_base + C::O_COL + 32 * c;
            tmem_ld32(addr, oo);
            tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 32; ++i) oo[i] = __float_as_uint(__uint_as_float(oo[i]) * alpha);
            tmem_st32(addr, oo);
          }
          tmem_st_wait();
        }
      }
      // P row -> shared memory, 128-byte swizzle: 16-byte chunk c of row r sits at
      // chunk c ^ (r & 7) of the row's 128-byte line
#pragma unroll
      for (int blk = 0; blk < 2; ++blk) {
        uint8_t* rowp = sP + blk * (kQT * 128) + r * 128;
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          const int e = blk * 32 + c * 4;  // index into pk (pairs)
          uint4 v;
          v.x = pk[e];
          v.y = pk[e + 1];
          v.z = pk[e + 2];
          v.w = pk[e + 3];
          *reinterpret_cast<uint4*>(rowp + ((c ^ (r & 7)) << 4)) = v;
        }
      }
      // keys past the CTA's last visible slot may hold stale cache contents:
      // zero their V rows so 0 * (non-finite) cannot reach O
      if (key0 + kKT - 1 > kmax) {
        if (!mbar_wait(&v_full[st], (j >> 1) & 1, abort_flag, a.err)) { ok = false; break; }
        if (key0 + r > kmax) {
#pragma unroll
          for (int c = 0; c < DH / 64; ++c) {
            uint4* vr = reinterpret_cast<uint4*>(sV + st * C::TILE_BYTES + c * kKT * 128 + r * 128);
#pragma unroll
            for (int q = 0; q < 8; ++q) vr[q] = make_uint4(0, 0, 0, 0);
          }
        }
      }
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(p_full);
    }
    if (ok && mbar_wait(o_done, (n_kv - 1) & 1, abort_flag, a.err)) {
      tc_fence_after();
      const float inv_l = 1.f / l_sum;
      const bool row_ok = t < a.T;
      f16* dst = a.out + ((size_t)b * a.T + t) * (size_t)(a.Hq * DH) + (size_t)h * DH;
#pragma unroll
      for (int c = 0; c < DH / 32; ++c) {
        uint32_t oo[32];
        tmem_ld32(tmem + lane_base + C::O_COL + 32 * c, oo);
        tmem_ld_wait();
        if (row_ok) {
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            uint4 w;
            w.x = pack_f16x2(__uint_as_float(oo[8 * q]) * inv_l, __uint_as_float(oo[8 * q + 1]) * inv_l);
            w.y = pack_f16x2(__uint_as_float(oo[8 * q + 2]) * inv_l, __uint_as_float(oo[8 * q + 3]) * inv_l);
            w.z = pack_f16x2(__uint_as_float(oo[8 * q + 4]) * inv_l, __uint_as_float(oo[8 * q + 5]) * inv_l);
            w.w = pack_f16x2(__uint_as_float(oo[8 * q + 6]) * inv_l, __uint_as_float(oo[8 * q + 7]) * inv_l);
            reinterpret_cast<uint4*>(dst + 32 * c)[q] = w;
          }
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

// ------------------------------------------------------------------ host side

static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
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

static bool tmap_rows_dh(CUtensorMap* m, const void* base, uint64_t rows, int dh, bool f16) {
  auto enc = encode_fn();
  if (!enc || (reinterpret_cast<uintptr_t>(base) & 15)) return false;
  cuuint64_t dims[2] = {(cuuint64_t)dh, rows};
  cuuint64_t strides[1] = {(cuuint64_t)dh * 2};
  cuuint32_t box[2] = {64, 128};
  cuuint32_t es[2] = {1, 1};
  return enc(m, f16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
             const_cast<void*>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
             CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int DH>
static qwen_status launch_dh(const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v,
                             const CUtensorMap& k16, const CUtensorMap& v16, const AttnArgs& a,
                             cudaStream_t st) {
  auto kern = attn_prefill_kernel<DH>;
  static bool attr = false;
  if (!attr) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             AttnCfg<DH>::SMEM_BYTES) != cudaSuccess)
      return QWEN_ERR_CUDA;
    attr = true;
  }
  const int n_qt = (a.T + kQT - 1) / kQT;
  const int grid = n_qt * a.B * a.Hq;
  launch_k(kern, dim3(grid), dim3(kAttnThreads), AttnCfg<DH>::SMEM_BYTES, st, q, k, v, k16, v16,
           a);
  count_launches();
  return cudaGetLastError() == cudaSuccess ? QWEN_OK : QWEN_ERR_CUDA;
}

// q [B][Hq][T][dh], caches [B][Hkv][max_seq][dh], out [B*T][Hq*dh].
qwen_status attention_prefill(const f16* q, const bf16* k_cache, const bf16* v_cache,
                              const f16* k16, const f16* v16, const int32_t* slot0, f16* out,
                              int B, int T, int Hq, int Hkv, int dh, int max_seq, int* err,
                              cudaStream_t st) {
  if (B == 0 || T == 0) return QWEN_OK;
  CUtensorMap tq, tk, tv, tk16, tv16;
  if (!tmap_rows_dh(&tq, q, (uint64_t)B * Hq * T, dh, true)) return QWEN_ERR_CUDA;
  if (!tmap_rows_dh(&tk, k_cache, (uint64_t)B * Hkv * max_seq, dh, false)) return QWEN_ERR_CUDA;
  if (!tmap_rows_dh(&tv, v_cache, (uint64_t)B * Hkv * max_seq, dh, false)) return QWEN_ERR_CUDA;
  if (!tmap_rows_dh(&tk16, k16, (uint64_t)B * Hkv * T, dh, true)) return QWEN_ERR_CUDA;
  if (!tmap_rows_dh(&tv16, v16, (uint64_t)B * Hkv * T, dh, true)) return QWEN_ERR_CUDA;
  AttnArgs a;
  a.B = B; a.T = T; a.Hq = Hq; a.Hkv = Hkv; a.max_seq = max_seq;
  a.slot0 = slot0; a.out = out; a.err = err;
  a.scale_log2 = 1.4426950408889634f / sqrtf((float)dh);
  if (dh == 128) return launch_dh<128>(tq, tk, tv, tk16, tv16, a, st);
  if (dh == 64) return launch_dh<64>(tq, tk, tv, tk16, tv16, a, st);
  return QWEN_ERR_UNSUPPORTED;
}

}  // namespace qwen
