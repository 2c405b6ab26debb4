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
// Work split (stream-K style): the (sequence, KV head) pairs' 64-key blocks are
// laid end to end, each pair taking nbv = ceil(max_seq / 64) places, and CTA c
// takes the contiguous range [c * per, (c + 1) * per): every CTA gets the same
// number of blocks, its range covering the end of one pair and the start of
// the next.  A work unit = the part of one pair inside one CTA's range (blocks
// past the sequence's length are skipped); it writes its partial to slot
// c - (first CTA of the pair).  A persistent CTA walks its units;
// the producer warp streams each unit's query rows (bulk copy) and K/V blocks
// (TMA) through rings of equal depth, so it can run ahead across unit
// boundaries.  In the decode step the first unit's blocks that lie wholly below
// the new token's slot are requested before the dependency wait (see
// DecAttnArgs::early).  4 compute warps each take 16 keys of every block and keep their
// own running max / sum / O; the warps merge through shared memory and the
// unit's unnormalised partial (m, l, O) goes to a workspace.  A merge kernel
// combines the slots of each head in a fixed order (deterministic).
#include <algorithm>
#include <cmath>

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
  static constexpr int Q_BYTES = 16 * DH * 2;           // one unit's query rows (<= 16 heads)
  // merge scratch, double-buffered by unit parity: per warp its O fragments
  // lane-major ([DH/2][32] floats) and per head row (max, sum)
  static constexpr int FRAG_FLOATS = (DH / 2) * 32;
  static constexpr int SCRATCH_FLOATS = 2 * kCW * (FRAG_FLOATS + 16 * 2);
  static constexpr int LEN_SLOTS = 1024;  // cache lengths staged in shared memory
  static constexpr int SMEM_BYTES = 1024 + kDStages * STAGE_BYTES + kDStages * Q_BYTES +
                                    SCRATCH_FLOATS * 4 + LEN_SLOTS * 4 + 256;
};

struct DecAttnArgs {
  const bf16* q;  // [B][Hq][DH]
  const int32_t* cache_len;
  int B, Hq, Hkv, max_seq;
  int nbv, per, slots;  // key blocks per pair, blocks per CTA, partial slots per pair
  float scale_log2;
  float* part_o;   // [B*Hq][slots][DH]
  float* part_ml;  // [B*Hq][slots][2]
  int* err;
  // A kernel of this step before the previous one released the kernels after
  // it only once its threads had passed their dependency wait, so everything
  // enqueued before the step has completed when this kernel starts: the
  // producer may load cache blocks that lie wholly below the new token's slot
  // (written by earlier steps) before waiting for the kernel before this one.
  int early;
};

}  // namespace

template <int DH>
__global__ void __launch_bounds__(kDecAttnThreads, 1)
    attn_decode_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                       DecAttnArgs a) {
  pdl_trigger();
  // early: the set-up reads only cache_len (written before the step) and the
  // producer waits after its first loads; otherwise everyone waits here
  if (!a.early) pdl_wait();
  using C = DecAttnCfg<DH>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  bf16* sQ = reinterpret_cast<bf16*>(smem + kDStages * C::STAGE_BYTES);  // [kDStages][16][DH]
  float* scratch =
      reinterpret_cast<float*>(smem + kDStages * C::STAGE_BYTES + kDStages * C::Q_BYTES);
  uint64_t* full = reinterpret_cast<uint64_t*>(scratch + C::SCRATCH_FLOATS);
  uint64_t* empty = full + kDStages;
  uint64_t* q_full = empty + kDStages;   // [kDStages]
  uint64_t* q_empty = q_full + kDStages; // [kDStages]
  volatile int* abort_flag = reinterpret_cast<volatile int*>(q_empty + kDStages);
  int* s_len = const_cast<int*>(abort_flag) + 4;  // [LEN_SLOTS] cache lengths

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = a.Hq / a.Hkv;
  // this CTA's lu-th unit: pair, key range [k0, k1) (empty when the range lies
  // past the sequence's length) and partial slot; false when there is none
  const long long v_end = (long long)a.B * a.Hkv * a.nbv;
  const long long v0 = (long long)blockIdx.x * a.per;
  const long long v1 = v0 + a.per < v_end ? v0 + a.per : v_end;
  auto unit_of = [&](int lu, int& pair, int& k0, int& k1, int& slot, int& n_keys) -> bool {
    const long long p = v0 / a.nbv + lu;
    if (p * a.nbv >= v1) return false;
    pair = (int)p;
    const long long lo = (v0 > p * a.nbv ? v0 : p * a.nbv) - p * a.nbv;
    const long long hi = (v1 < (p + 1) * a.nbv ? v1 : (p + 1) * a.nbv) - p * a.nbv;
    const int b = pair / a.Hkv;
    // the new token sits in slot cache_len[b]: keys 0..cache_len[b] (clamped to the cache)
    n_keys = min((b < DecAttnCfg<DH>::LEN_SLOTS ? s_len[b] : a.cache_len[b]) + 1, a.max_seq);
    k0 = (int)lo * kKB;
    k1 = min((int)hi * kKB, n_keys);
    slot = (int)blockIdx.x - (int)((p * a.nbv) / a.per);
    return true;
  };

  if (threadIdx.x == 0) {
    for (int s = 0; s < kDStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kCW);
    }
    for (int s = 0; s < kDStages; ++s) {
      mbar_init(&q_full[s], 1);
      mbar_init(&q_empty[s], kCW);
    }
    *abort_flag = 0;
    fence_barrier_init();
  }
  // query rows beyond the group stay zero (the bulk copies fill rows < G only)
  for (int i = threadIdx.x; i < kDStages * C::Q_BYTES / 16; i += blockDim.x)
    reinterpret_cast<uint4*>(sQ)[i] = make_uint4(0, 0, 0, 0);
  // every unit needs its sequence's cache length: stage them once
  for (int i = threadIdx.x; i < a.B && i < C::LEN_SLOTS; i += blockDim.x) s_len[i] = a.cache_len[i];
  fence_proxy_async_smem();
  __syncthreads();

  if (warp == kCW) {
    // ---------------- producer (converged; one elected lane issues)
    {
      if (lane == 0) {
        tma_prefetch_desc(&tmK);
        tma_prefetch_desc(&tmV);
      }
      __syncwarp();
      const uint64_t pol = l2_evict_first();
      auto load_block = [&](int stage, int row) {
        uint8_t* st = smem + stage * C::STAGE_BYTES;
        mbar_arrive_expect_tx_w(&full[stage], C::STAGE_BYTES);
#pragma unroll
        for (int c = 0; c < DH / 64; ++c) {
          // the cache is read once per step: evicted first
          tma_load_2d_hint_w(st + c * C::BOX_BYTES, &tmK, &full[stage], c * 64, row, pol);
          tma_load_2d_hint_w(st + C::KV_BYTES + c * C::BOX_BYTES, &tmV, &full[stage], c * 64, row,
                             pol);
        }
      };
      int stage = 0;
      uint32_t phase = 0;
      int pair, k0, k1, slot, n_keys;
      // first unit: the blocks wholly below the new token's slot (written by
      // earlier steps) into the empty ring, before the wait
      int pre = 0;
      if (a.early) {
        if (unit_of(0, pair, k0, k1, slot, n_keys)) {
          const int b = pair / a.Hkv;
          const int cl = b < C::LEN_SLOTS ? s_len[b] : a.cache_len[b];
          for (int blk = k0; blk < k1 && pre < kDStages && blk + kKB <= cl; blk += kKB, ++pre)
            load_block(pre, pair * a.max_seq + blk);
        }
        pdl_wait();
      }
      for (int lu = 0; unit_of(lu, pair, k0, k1, slot, n_keys); ++lu) {
        const int b = pair / a.Hkv, g = pair - b * a.Hkv;
        const int row0 = pair * a.max_seq;  // (b * Hkv + g) * max_seq
        // the unit's G query rows (contiguous in q) into its slot of the Q ring
        const int qs = lu % kDStages;
        if (!mbar_wait_w(&q_empty[qs], ((lu / kDStages) & 1) ^ 1u, abort_flag, a.err)) goto prod_done;
        mbar_arrive_expect_tx_w(&q_full[qs], (uint32_t)(G * DH * 2));
        bulk_load_w(sQ + qs * 16 * DH, a.q + ((size_t)b * a.Hq + (size_t)g * G) * DH,
                  (uint32_t)(G * DH * 2), &q_full[qs]);
        for (int blk = k0, i = 0; blk < k1; blk += kKB, ++i) {
          if (lu > 0 || i >= pre) {  // else loaded before the wait
            if (!mbar_wait_w(&empty[stage], phase ^ 1u, abort_flag, a.err)) goto prod_done;
            load_block(stage, row0 + blk);
          }
          if (++stage == kDStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      for (int i = 0; i < kDStages; ++i) {
        if (!mbar_wait_w(&empty[stage], phase ^ 1u, abort_flag, a.err)) break;
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
  if (a.early) pdl_wait();  // the query rows come from the kernel before
  const int gid = lane >> 2, tq = lane & 3;
  int stage = 0;
  uint32_t phase = 0;
  const uint32_t smem_base = smem_u32(smem);
  int pair, k0, k1, slot, n_keys;
  for (int lu = 0; unit_of(lu, pair, k0, k1, slot, n_keys); ++lu) {
    const int b = pair / a.Hkv, g = pair - b * a.Hkv;
    const int L = n_keys - 1;  // last visible key
    const int h0 = g * G;
    // Q fragments (rows = heads of the group, zero beyond G) from the slot the
    // producer filled.  The slot is released at the end of the unit: only then
    // are the shared-memory loads certain to have completed (their consumers,
    // the S MMAs, have issued), so the next bulk copy cannot overtake them.
    uint32_t qa[DH / 16][4];
    const int qs = lu % kDStages;
    {
      if (!mbar_wait(&q_full[qs], (lu / kDStages) & 1, abort_flag, a.err)) break;
      const uint32_t* qrow0 = reinterpret_cast<const uint32_t*>(sQ + (qs * 16 + gid) * DH);
      const uint32_t* qrow1 = reinterpret_cast<const uint32_t*>(sQ + (qs * 16 + gid + 8) * DH);
#pragma unroll
      for (int kk = 0; kk < DH / 16; ++kk) {
        qa[kk][0] = qrow0[(16 * kk + 2 * tq) / 2];
        qa[kk][1] = qrow1[(16 * kk + 2 * tq) / 2];
        qa[kk][2] = qrow0[(16 * kk + 8 + 2 * tq) / 2];
        qa[kk][3] = qrow1[(16 * kk + 8 + 2 * tq) / 2];
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
    __syncwarp();
    if (lane == 0) mbar_arrive(&q_empty[qs]);
    // ---- merge the warps of this unit: fragments lane-major into the scratch
    // buffer of this unit's parity, one barrier, then each warp combines a
    // share of the fragment entries across all warps (the other buffer may
    // still be read by slower threads of the previous unit; the barrier of
    // the next unit orders reuse of this one)
#pragma unroll
    for (int rI = 0; rI < 2; ++rI) {
      l_r[rI] += __shfl_xor_sync(0xffffffffu, l_r[rI], 1);
      l_r[rI] += __shfl_xor_sync(0xffffffffu, l_r[rI], 2);
    }
    float* buf = scratch + (lu & 1) * kCW * (C::FRAG_FLOATS + 32);
    float* frag = buf + warp * C::FRAG_FLOATS;
    float* ml = buf + kCW * C::FRAG_FLOATS;  // [kCW][16 rows][2]
#pragma unroll
    for (int i = 0; i < DH / 8; ++i)
#pragma unroll
      for (int e = 0; e < 4; ++e) frag[(4 * i + e) * 32 + lane] = o[i][e];
    if (tq == 0) {
      ml[(warp * 16 + gid) * 2] = m_r[0];
      ml[(warp * 16 + gid) * 2 + 1] = l_r[0];
      ml[(warp * 16 + gid + 8) * 2] = m_r[1];
      ml[(warp * 16 + gid + 8) * 2 + 1] = l_r[1];
    }
    asm volatile("bar.sync 1, %0;" ::"r"(kCW * 32) : "memory");
    constexpr int PER_W = (DH / 2) / kCW;  // fragment entries each warp combines
    float Mr[2], wr[2][kCW], Lr[2];
#pragma unroll
    for (int rI = 0; rI < 2; ++rI) {
      const int row = gid + 8 * rI;
      float M = -INFINITY;
#pragma unroll
      for (int w = 0; w < kCW; ++w) M = fmaxf(M, ml[(w * 16 + row) * 2]);
      float L = 0.f;
#pragma unroll
      for (int w = 0; w < kCW; ++w) {
        const float mw = ml[(w * 16 + row) * 2];
        wr[rI][w] = (mw == -INFINITY) ? 0.f : ex2f(mw - M);
        L += wr[rI][w] * ml[(w * 16 + row) * 2 + 1];
      }
      Mr[rI] = M;
      Lr[rI] = L;
    }
#pragma unroll
    for (int j = 0; j < PER_W; ++j) {
      const int i = warp * PER_W + j;       // fragment entry
      const int e = i & 3, nb = i >> 2;
      const int rI = e >> 1;
      const int row = gid + 8 * rI;
      const int col = 8 * nb + 2 * tq + (e & 1);
      float acc = 0.f;
#pragma unroll
      for (int w = 0; w < kCW; ++w) acc += wr[rI][w] * buf[w * C::FRAG_FLOATS + i * 32 + lane];
      if (row < G) {
        const size_t ph = (size_t)(b * a.Hq + h0 + row) * a.slots + slot;
        a.part_o[ph * DH + col] = acc;
      }
    }
    if (warp == 0 && tq == 0) {
#pragma unroll
      for (int rI = 0; rI < 2; ++rI) {
        const int row = gid + 8 * rI;
        if (row < G) {
          const size_t ph = (size_t)(b * a.Hq + h0 + row) * a.slots + slot;
          a.part_ml[ph * 2] = Mr[rI];
          a.part_ml[ph * 2 + 1] = Lr[rI];
        }
      }
    }
  }
}

// out[b][h*DH + d] = sum_s 2^(m_s - M) o_s[d] / sum_s 2^(m_s - M) l_s over the
// slots s that CTAs wrote for head h's (sequence, KV head) pair: the CTAs whose
// block ranges meet the pair's [p * nbv, (p + 1) * nbv).  One CTA per (b, h)
// of SG groups of DH threads: thread (j, t) takes slots j, j + SG, ... of
// element t, up to 8 slots' loads in flight at once, and merges them in slot
// order with a running maximum (sums rescaled by 2^(old max - new max) when it
// grows); the groups' results are then merged in order j = 0, 1, .. through
// shared memory.  A slot whose key range was empty has m = -inf and adds
// nothing.
__device__ __forceinline__ void merge_in(float m, float l, float o, float& M, float& L, float& A) {
  if (m == -INFINITY) return;
  if (m > M) {
    const float f = ex2f(M - m);  // 0 while M is -inf
    L = fmaf(L, f, l);
    A = fmaf(A, f, o);
    M = m;
  } else {
    const float f = ex2f(m - M);
    L = fmaf(f, l, L);
    A = fmaf(f, o, A);
  }
}

template <int DH>
__global__ void __launch_bounds__(1024) attn_decode_merge_kernel(
    const float* __restrict__ part_o, const float* __restrict__ part_ml, int BH, int slots,
    int G, int nbv, int per, f16* __restrict__ out, int* err) {
  pdl_trigger();
  pdl_wait();
  __shared__ float sm_m[1024 / DH], sm_l[1024 / DH];
  __shared__ float sm_a[1024];
  const int wid = blockIdx.x;  // b * Hq + h
  const int t = threadIdx.x % DH, j = threadIdx.x / DH;
  const int SG = blockDim.x / DH;
  if (wid >= BH) return;
  const long long pair = wid / G;  // (b * Hq + h) / G = b * Hkv + h / G
  const int splits = (int)(((pair + 1) * nbv - 1) / per - (pair * nbv) / per) + 1;
  const float* ml = part_ml + (size_t)wid * slots * 2;
  const float* po = part_o + (size_t)wid * slots * DH + t;
  float M = -INFINITY, L = 0.f, A = 0.f;
  for (int s0 = j; s0 < splits; s0 += 8 * SG) {
    float m[8], l[8], o[8];
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      const int sl = s0 + c * SG;
      const bool in = sl < splits;
      m[c] = in ? ml[2 * sl] : -INFINITY;
      l[c] = in ? ml[2 * sl + 1] : 0.f;
      o[c] = in ? po[(size_t)sl * DH] : 0.f;
    }
#pragma unroll
    for (int c = 0; c < 8; ++c) merge_in(m[c], l[c], o[c], M, L, A);
  }
  if (SG > 1) {
    if (t == 0) {
      sm_m[j] = M;
      sm_l[j] = L;
    }
    sm_a[threadIdx.x] = A;
    __syncthreads();
    if (j != 0) return;
    M = -INFINITY;
    L = A = 0.f;
    for (int q = 0; q < SG; ++q) merge_in(sm_m[q], sm_l[q], sm_a[q * DH + t], M, L, A);
  }
  bool bad = false;  // C is the next GEMM's FP16 operand: V rows past 65504 reach it
  out[(size_t)wid * DH + t] = f16_chk(A / L, bad);
  record_overflow(err, bad);
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

// The stream-K split: pairs x nbv blocks over the SMs, `per` blocks per CTA;
// a pair meets at most (nbv - 1) / per + 2 CTA ranges, its partial slots.
struct AttnSplit {
  int nbv, per, slots, grid;
};

static AttnSplit attn_split(int B, int Hkv, int max_seq) {
  AttnSplit sp;
  const long long sms = device_sm_count();
  sp.nbv = (max_seq + kKB - 1) / kKB;
  const long long total = (long long)B * Hkv * sp.nbv;
  sp.per = (int)((total + sms - 1) / sms);
  sp.grid = (int)((total + sp.per - 1) / sp.per);
  sp.slots = (sp.nbv - 1) / sp.per + 2;
  return sp;
}

void decode_attn_plan(const qwen_layer_config& c, int B, int* splits) {
  *splits = attn_split(B, c.n_kv_heads, c.max_seq).slots;
}

template <int DH>
static qwen_status launch_attn_dec(const CUtensorMap& tk, const CUtensorMap& tv,
                                   const DecAttnArgs& a, int grid, f16* out, cudaStream_t st) {
  auto kern = attn_decode_kernel<DH>;
  static std::atomic<uint64_t> attr{0};  // one bit per device
  if (!smem_attr_once(kern, DecAttnCfg<DH>::SMEM_BYTES, attr)) return QWEN_ERR_CUDA;
  launch_k(kern, dim3(grid), dim3(kDecAttnThreads), DecAttnCfg<DH>::SMEM_BYTES, st, tk, tv, a);
  count_launches();
  if (cudaGetLastError() != cudaSuccess) return QWEN_ERR_CUDA;
  const int BH = a.B * a.Hq;
  // slot groups: about 4 slots per thread, at most 1024 threads
  const int sg = std::max(1, std::min(1024 / DH, (a.slots + 3) / 4));
  launch_k(attn_decode_merge_kernel<DH>, dim3(BH), dim3(DH * sg), 0, st, (const float*)a.part_o,
           (const float*)a.part_ml, BH, a.slots, a.Hq / a.Hkv, a.nbv, a.per, out, a.err);
  count_launches();
  return cudaGetLastError() == cudaSuccess ? QWEN_OK : QWEN_ERR_CUDA;
}

qwen_status attention_decode(const bf16* q, const bf16* kc, const bf16* vc,
                             const int32_t* cache_len, int B, int Hq, int Hkv, int dh, int max_seq,
                             int splits, float* part_o, float* part_ml, f16* out,
                             int* err, cudaStream_t st, bool early) {
  if (B == 0) return QWEN_OK;
  if (Hq / Hkv > 16) return QWEN_ERR_UNSUPPORTED;
  const AttnSplit sp = attn_split(B, Hkv, max_seq);
  if (splits < sp.slots) return QWEN_ERR_CAPACITY;  // partial space sized for fewer slots
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
  a.nbv = sp.nbv;
  a.per = sp.per;
  a.slots = sp.slots;
  a.scale_log2 = 1.4426950408889634f / sqrtf((float)dh);
  a.part_o = part_o;
  a.part_ml = part_ml;
  a.err = err;
  a.early = early ? 1 : 0;
  if (dh == 128) return launch_attn_dec<128>(tk, tv, a, sp.grid, out, st);
  if (dh == 64) return launch_attn_dec<64>(tk, tv, a, sp.grid, out, st);
  return QWEN_ERR_UNSUPPORTED;
}

}  // namespace qwen
