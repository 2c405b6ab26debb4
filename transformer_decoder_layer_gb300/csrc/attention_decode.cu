// Split-KV decode attention (one new query per sequence) and its merge.
//
// "Qwen2.5-7B 结构拆解" §09.1: at decode the single query of each head attends
// every cached row 0..t of its sequence, the new K/V row included; §05.2: the
// G = Hq/Hkv query heads of a group read the same K/V rows, so one staged K/V
// block serves all G heads.  Qwen3 layer page §7-§9 for scores / sqrt(dh), the
// stable softmax and the weighted sum of V.
//
// The step reads the whole cache once and does ~G FLOPs per byte, so it is
// bound by HBM bandwidth: K/V blocks of 64 keys are streamed by TMA (128-byte
// swizzle) through a 4-stage ring; the tiny contraction runs on mma.sync
// (m16n8k16, BF16 -> FP32) with the group's heads as the 16 rows.
//
// Work unit = (sequence b, KV head g, key chunk sp).  A persistent CTA walks
// its units; 4 compute warps each take 16 keys of every block and keep their own
// running max / sum / O; the warps merge through shared memory and the unit's
// unnormalised partial (m, l, O) goes to a workspace.  A merge kernel combines
// the chunks of each head in a fixed order (deterministic).
#include "common.cuh"
#include "internal.h"
#include "layer.h"

#include <cudaTypedefs.h>

namespace qwen {

namespace {

constexpr int kKB = 64;          // keys per stage
constexpr int kCW = 4;           // compute warps (16 keys each)
constexpr int kDecAttnThreads = 32 * (kCW + 1);
constexpr int kDStages = 4;

__device__ __forceinline__ float ex2f(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                        uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                          uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

// D(16x8, f32) += A(16x16, bf16, row) * B(16x8, bf16, col)
__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, "
      "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

template <int DH>
struct DecAttnCfg {
  static constexpr int BOX_BYTES = kKB * 128;          // 64 keys x 64 dims
  static constexpr int KV_BYTES = (DH / 64) * BOX_BYTES;
  static constexpr int STAGE_BYTES = 2 * KV_BYTES;      // K then V
  static constexpr int SCRATCH_FLOATS = kCW * 16 * (DH + 2);
  static constexpr int SMEM_BYTES = 1024 + kDStages * STAGE_BYTES + SCRATCH_FLOATS * 4 + 256;
};

struct DecAttnArgs {
  const bf16* q;  // [B][Hq][DH]
  const int32_t* cache_len;
  int B, Hq, Hkv, max_seq, chunk, splits;
  float scale_log2;
  float* part_o;   // [B*Hq][splits][DH]
  float* part_ml;  // [B*Hq][splits][2]
  int* err;
};

}  // namespace

template <int DH>
__global__ void __launch_bounds__(kDecAttnThreads, 1)
    attn_decode_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                       DecAttnArgs a) {
  pdl_trigger();
  pdl_wait();
  using C = DecAttnCfg<DH>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  float* scratch = reinterpret_cast<float*>(smem + kDStages * C::STAGE_BYTES);
  uint64_t* full = reinterpret_cast<uint64_t*>(scratch + C::SCRATCH_FLOATS);
  uint64_t* empty = full + kDStages;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(empty + kDStages);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = a.Hq / a.Hkv;
  const int units = a.B * a.Hkv * a.splits;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kDStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kCW);
    }
    *abort_flag = 0;
    fence_barrier_init();
  }
  __syncthreads();

  if (warp == kCW) {
    // ---------------- producer
    if (lane == 0) {
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
      int stage = 0;
      uint32_t phase = 0;
      for (int u = blockIdx.x; u < units; u += gridDim.x) {
        const int pair = u / a.splits, sp = u - pair * a.splits;
        const int b = pair / a.Hkv;
        const int n_keys = min(a.cache_len[b] + 1, a.max_seq);
        const int k0 = sp * a.chunk, k1 = min(k0 + a.chunk, n_keys);
        const int row0 = pair * a.max_seq;  // (b * Hkv + g) * max_seq
        for (int blk = k0; blk < k1; blk += kKB) {
          if (!mbar_wait(&empty[stage], phase ^ 1u, abort_flag, a.err)) goto prod_done;
          uint8_t* st = smem + stage * C::STAGE_BYTES;
          mbar_arrive_expect_tx(&full[stage], C::STAGE_BYTES);
#pragma unroll
          for (int c = 0; c < DH / 64; ++c) {
            tma_load_2d(st + c * C::BOX_BYTES, &tmK, &full[stage], c * 64, row0 + blk);
            tma_load_2d(st + C::KV_BYTES + c * C::BOX_BYTES, &tmV, &full[stage], c * 64, row0 + blk);
          }
          if (++stage == kDStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      for (int i = 0; i < kDStages; ++i) {
        if (!mbar_wait(&empty[stage], phase ^ 1u, abort_flag, a.err)) break;
        if (++stage == kDStages) {
          stage = 0;
          phase ^= 1u;
        }
      }
    prod_done:;
    }
    return;
  }

  // ---------------- compute warps
  const int gid = lane >> 2, tq = lane & 3;
  int stage = 0;
  uint32_t phase = 0;
  const uint32_t smem_base = smem_u32(smem);
  for (int u = blockIdx.x; u < units; u += gridDim.x) {
    const int pair = u / a.splits, sp = u - pair * a.splits;
    const int b = pair / a.Hkv, g = pair - b * a.Hkv;
    // the new token sits in slot cache_len[b]: keys 0..cache_len[b] (clamped to the cache)
    const int n_keys = min(a.cache_len[b] + 1, a.max_seq);
    const int L = n_keys - 1;  // last visible key
    const int k0 = sp * a.chunk, k1 = min(k0 + a.chunk, n_keys);
    const int h0 = g * G;
    // Q fragments (rows = heads of the group, zero beyond G)
    uint32_t qa[DH / 16][4];
    {
      const uint32_t* qrow0 = reinterpret_cast<const uint32_t*>(a.q + ((size_t)b * a.Hq + h0 + gid) * DH);
      const uint32_t* qrow1 = reinterpret_cast<const uint32_t*>(a.q + ((size_t)b * a.Hq + h0 + gid + 8) * DH);
      const bool v0 = gid < G, v1 = gid + 8 < G;
#pragma unroll
      for (int kk = 0; kk < DH / 16; ++kk) {
        qa[kk][0] = v0 ? qrow0[(16 * kk + 2 * tq) / 2] : 0u;
        qa[kk][1] = v1 ? qrow1[(16 * kk + 2 * tq) / 2] : 0u;
        qa[kk][2] = v0 ? qrow0[(16 * kk + 8 + 2 * tq) / 2] : 0u;
        qa[kk][3] = v1 ? qrow1[(16 * kk + 8 + 2 * tq) / 2] : 0u;
      }
    }
    float m_r[2] = {-INFINITY, -INFINITY}, l_r[2] = {0.f, 0.f};
    float o[DH / 8][4];
#pragma unroll
    for (int i = 0; i < DH / 8; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;

    for (int blk = k0; blk < k1; blk += kKB) {
      if (!mbar_wait(&full[stage], phase, abort_flag, a.err)) break;
      const uint32_t sK = smem_base + stage * C::STAGE_BYTES;
      const uint32_t sV = sK + C::KV_BYTES;
      const int kb = blk + 16 * warp;  // first key of this warp's slice
      // ---- S = Q K^T for 16 keys (two n-blocks of 8)
      float s[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
      const int mi = lane >> 3, rr = lane & 7;
#pragma unroll
      for (int kk = 0; kk < DH / 16; ++kk) {
        const int r = 16 * warp + 8 * (mi >> 1) + rr;        // key row in the block
        const int box = (16 * kk) / 64;
        const int ch = 2 * (kk & 3) + (mi & 1);
        const uint32_t addr = sK + box * C::BOX_BYTES + r * 128 + ((ch ^ (r & 7)) << 4);
        uint32_t b00, b01, b10, b11;
        ldsm_x4(addr, b00, b01, b10, b11);
        mma16816(s[0], qa[kk], b00, b01);
        mma16816(s[1], qa[kk], b10, b11);
      }
      // ---- mask, scale (log2 domain), online softmax per head row
      float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
      for (int nb = 0; nb < 2; ++nb)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int key = kb + 8 * nb + 2 * tq + (e & 1);
          const float v = key <= L ? s[nb][e] * a.scale_log2 : -INFINITY;
          s[nb][e] = v;
          mx[e >> 1] = fmaxf(mx[e >> 1], v);
        }
      float alpha[2];
#pragma unroll
      for (int rI = 0; rI < 2; ++rI) {
        mx[rI] = fmaxf(mx[rI], __shfl_xor_sync(0xffffffffu, mx[rI], 1));
        mx[rI] = fmaxf(mx[rI], __shfl_xor_sync(0xffffffffu, mx[rI], 2));
        const float m_new = fmaxf(m_r[rI], mx[rI]);
        alpha[rI] = (m_new == -INFINITY) ? 1.f : ex2f(m_r[rI] - m_new);
        m_r[rI] = m_new;
      }
      uint32_t pa[4];
      {
        float p[2][4];
#pragma unroll
        for (int nb = 0; nb < 2; ++nb)
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float mrow = m_r[e >> 1];
            p[nb][e] = (mrow == -INFINITY) ? 0.f : ex2f(s[nb][e] - mrow);
          }
        pa[0] = pack_bf16x2(p[0][0], p[0][1]);
        pa[1] = pack_bf16x2(p[0][2], p[0][3]);
        pa[2] = pack_bf16x2(p[1][0], p[1][1]);
        pa[3] = pack_bf16x2(p[1][2], p[1][3]);
        const float2 f0 = unpack_bf16x2(pa[0]), f1 = unpack_bf16x2(pa[1]);
        const float2 f2 = unpack_bf16x2(pa[2]), f3 = unpack_bf16x2(pa[3]);
        l_r[0] = l_r[0] * alpha[0] + (f0.x + f0.y + f2.x + f2.y);
        l_r[1] = l_r[1] * alpha[1] + (f1.x + f1.y + f3.x + f3.y);
      }
#pragma unroll
      for (int i = 0; i < DH / 8; ++i) {
        o[i][0] *= alpha[0];
        o[i][1] *= alpha[0];
        o[i][2] *= alpha[1];
        o[i][3] *= alpha[1];
      }
      // ---- keys past the new token may hold stale cache rows: zero their V
      const bool tail = kb + 15 > L;
      if (tail) {
#pragma unroll
        for (int it = 0; it < (16 * (DH / 64) * 8) / 32; ++it) {
          const int idx = it * 32 + lane;           // (row, box, chunk)
          const int row = idx / ((DH / 64) * 8);
          const int rem = idx - row * ((DH / 64) * 8);
          const int box = rem >> 3, chn = rem & 7;
          if (kb + row > L) {
            uint8_t* p = smem + stage * C::STAGE_BYTES + C::KV_BYTES + box * C::BOX_BYTES +
                         (16 * warp + row) * 128 + chn * 16;
            *reinterpret_cast<uint4*>(p) = make_uint4(0, 0, 0, 0);
          }
        }
        __syncwarp();
      }
      // ---- O += P V over this warp's 16 keys
#pragma unroll
      for (int d0 = 0; d0 < DH; d0 += 16) {
        const int r = 16 * warp + 8 * (mi & 1) + rr;  // key row
        const int box = d0 / 64;
        const int ch = ((d0 & 63) >> 3) + (mi >> 1);
        const uint32_t addr = sV + box * C::BOX_BYTES + r * 128 + ((ch ^ (r & 7)) << 4);
        uint32_t v00, v01, v10, v11;
        ldsm_x4_t(addr, v00, v01, v10, v11);
        mma16816(o[d0 / 8], pa, v00, v01);
        mma16816(o[d0 / 8 + 1], pa, v10, v11);
      }
      __syncwarp();
      if (tail) fence_proxy_async_smem();
      if (lane == 0) mbar_arrive(&empty[stage]);
      if (++stage == kDStages) {
        stage = 0;
        phase ^= 1u;
      }
    }
    if (*abort_flag) break;
    // ---- merge the 4 warps of this unit through shared memory
#pragma unroll
    for (int rI = 0; rI < 2; ++rI) {
      l_r[rI] += __shfl_xor_sync(0xffffffffu, l_r[rI], 1);
      l_r[rI] += __shfl_xor_sync(0xffffffffu, l_r[rI], 2);
    }
    float* my = scratch + (size_t)warp * 16 * (DH + 2);
#pragma unroll
    for (int rI = 0; rI < 2; ++rI) {
      const int hrow = gid + 8 * rI;
      float* row = my + hrow * (DH + 2);
#pragma unroll
      for (int i = 0; i < DH / 8; ++i) {
        row[8 * i + 2 * tq] = o[i][2 * rI];
        row[8 * i + 2 * tq + 1] = o[i][2 * rI + 1];
      }
      if (tq == 0) {
        row[DH] = m_r[rI];
        row[DH + 1] = l_r[rI];
      }
    }
    asm volatile("bar.sync 1, %0;" ::"r"(kCW * 32) : "memory");
    for (int idx = threadIdx.x; idx < G * DH; idx += kCW * 32) {
      const int hrow = idx / DH, dd = idx - hrow * DH;
      float M = -INFINITY;
#pragma unroll
      for (int w = 0; w < kCW; ++w) M = fmaxf(M, scratch[(w * 16 + hrow) * (DH + 2) + DH]);
      float acc = 0.f, lsum = 0.f;
#pragma unroll
      for (int w = 0; w < kCW; ++w) {
        const float* row = scratch + (w * 16 + hrow) * (DH + 2);
        const float f = (row[DH] == -INFINITY) ? 0.f : ex2f(row[DH] - M);
        acc += f * row[dd];
        lsum += f * row[DH + 1];
      }
      const size_t ph = (size_t)(b * a.Hq + h0 + hrow) * a.splits + sp;
      a.part_o[ph * DH + dd] = acc;
      if (dd == 0) {
        a.part_ml[ph * 2] = M;
        a.part_ml[ph * 2 + 1] = lsum;
      }
    }
    asm volatile("bar.sync 1, %0;" ::"r"(kCW * 32) : "memory");
  }
}

// out[b][h*DH + d] = sum_s 2^(m_s - M) o_s[d] / sum_s 2^(m_s - M) l_s
template <int DH>
__global__ void attn_decode_merge_kernel(const float* __restrict__ part_o,
                                         const float* __restrict__ part_ml, int BH, int splits,
                                         f16* __restrict__ out) {
  pdl_trigger();
  pdl_wait();
  const int wid = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (wid >= BH) return;
  const float* ml = part_ml + (size_t)wid * splits * 2;
  float M = -INFINITY;
  for (int s = 0; s < splits; ++s) M = fmaxf(M, ml[2 * s]);
  float acc[DH / 32];
#pragma unroll
  for (int i = 0; i < DH / 32; ++i) acc[i] = 0.f;
  float lsum = 0.f;
  for (int s = 0; s < splits; ++s) {
    const float m = ml[2 * s];
    if (m == -INFINITY) continue;
    const float f = ex2f(m - M);
    lsum += f * ml[2 * s + 1];
    const float* po = part_o + ((size_t)wid * splits + s) * DH;
#pragma unroll
    for (int i = 0; i < DH / 32; ++i) acc[i] += f * po[lane + 32 * i];
  }
  const float inv = 1.f / lsum;
#pragma unroll
  for (int i = 0; i < DH / 32; ++i)
    out[(size_t)wid * DH + lane + 32 * i] = __float2half_rn(acc[i] * inv);
}

// ------------------------------------------------------------------ host side

static PFN_cuTensorMapEncodeTiled_v12000 enc() {
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

static bool tmap_cache(CUtensorMap* m, const void* base, uint64_t rows, int dh) {
  auto e = enc();
  if (!e || (reinterpret_cast<uintptr_t>(base) & 15)) return false;
  cuuint64_t dims[2] = {(cuuint64_t)dh, rows};
  cuuint64_t strides[1] = {(cuuint64_t)dh * 2};
  cuuint32_t box[2] = {64, (cuuint32_t)kKB};
  cuuint32_t es[2] = {1, 1};
  return e(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, es,
           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
           CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

void decode_attn_plan(const qwen_layer_config& c, int B, int* chunk, int* splits) {
  const int sms = device_sm_count();
  const long long pairs = (long long)B * c.n_kv_heads;
  long long target = (16LL * sms + pairs - 1) / pairs;  // splits per (b, g)
  if (target < 1) target = 1;
  long long ch = (c.max_seq + target - 1) / target;
  ch = ((ch + kKB - 1) / kKB) * kKB;
  if (ch < kKB) ch = kKB;
  *chunk = (int)ch;
  *splits = (int)((c.max_seq + ch - 1) / ch);
}

template <int DH>
static qwen_status launch_attn_dec(const CUtensorMap& tk, const CUtensorMap& tv,
                                   const DecAttnArgs& a, f16* out, cudaStream_t st) {
  auto kern = attn_decode_kernel<DH>;
  static bool attr = false;
  if (!attr) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             DecAttnCfg<DH>::SMEM_BYTES) != cudaSuccess)
      return QWEN_ERR_CUDA;
    attr = true;
  }
  const int units = a.B * a.Hkv * a.splits;
  const int sms = device_sm_count();
  const int grid = units < sms ? units : sms;
  launch_k(kern, dim3(grid), dim3(kDecAttnThreads), DecAttnCfg<DH>::SMEM_BYTES, st, tk, tv, a);
  count_launches();
  if (cudaGetLastError() != cudaSuccess) return QWEN_ERR_CUDA;
  const int BH = a.B * a.Hq;
  launch_k(attn_decode_merge_kernel<DH>, dim3((BH * 32 + 255) / 256), dim3(256), 0, st,
           (const float*)a.part_o, (const float*)a.part_ml, BH, a.splits, out);
  count_launches();
  return cudaGetLastError() == cudaSuccess ? QWEN_OK : QWEN_ERR_CUDA;
}

qwen_status attention_decode(const bf16* q, const bf16* kc, const bf16* vc,
                             const int32_t* cache_len, int B, int Hq, int Hkv, int dh, int max_seq,
                             int chunk, int splits, float* part_o, float* part_ml, f16* out,
                             int* err, cudaStream_t st) {
  if (B == 0) return QWEN_OK;
  if (Hq / Hkv > 16 || chunk % kKB) return QWEN_ERR_UNSUPPORTED;
  CUtensorMap tk, tv;
  if (!tmap_cache(&tk, kc, (uint64_t)B * Hkv * max_seq, dh)) return QWEN_ERR_CUDA;
  if (!tmap_cache(&tv, vc, (uint64_t)B * Hkv * max_seq, dh)) return QWEN_ERR_CUDA;
  DecAttnArgs a;
  a.q = q;
  a.cache_len = cache_len;
  a.B = B;
  a.Hq = Hq;
  a.Hkv = Hkv;
  a.max_seq = max_seq;
  a.chunk = chunk;
  a.splits = splits;
  a.scale_log2 = 1.4426950408889634f / sqrtf((float)dh);
  a.part_o = part_o;
  a.part_ml = part_ml;
  a.err = err;
  if (dh == 128) return launch_attn_dec<128>(tk, tv, a, out, st);
  if (dh == 64) return launch_attn_dec<64>(tk, tv, a, out, st);
  return QWEN_ERR_UNSUPPORTED;
}

}  // namespace qwen
