// Persistent tcgen05 GEMM for sm_103a: D[M,N] = A[M,K] * B[N,K]^T with FP16
// operands (the layer's packed weights and activations) or BF16 operands
// (qwen_linear), FP32 accumulation in tensor memory, fed by TMA through an
// mbarrier ring, with fused epilogues for the decoder layer's projections.
//
// Every projection of the layer is a "token rows x weight rows" product of this
// shape ("Qwen2.5-7B 结构拆解" §03.2: [B,S,d] is flattened to [B*S,d] and each
// projection is one GEMM against the [out,in] weight, §03.1).
//
// CTA layout (192 threads, one CTA per SM, persistent over output tiles):
//   warp 0      TMA producer: A tile [128 x 64] and B tile [BN x 64] per stage
//               (pair tiles: this CTA's [BN/2 x 64] half of B)
//   warp 1      TMEM allocator + MMA issuer (one elected lane; pair tiles:
//               only the even CTA of the cluster issues)
//   warps 2..5  epilogue: tcgen05.ld of the 128 x BN FP32 accumulator, fused
//               math, global stores.  Warp w reads TMEM lanes 32*(w%4)..+31.
// Two accumulators in TMEM (2 x BN columns) let the epilogue of tile i overlap
// the main loop of tile i+1.  Tile shapes: 1-SM tiles of 128 x BN, or pair
// tiles of 256 x BN on a cluster of two CTAs (see GemmCfg); the host picks
// the shape with the shorter estimated run (gemm_tc).
#include "common.cuh"
#include "internal.h"
#include "qkv_epilogue.cuh"

#include <cudaTypedefs.h>

namespace qwen {

constexpr int kBM = 128;
constexpr int kBK = 64;  // 64 bf16 = 128 bytes = one swizzle row
constexpr int kGemmThreads = 192;
constexpr int kGroupM = 16;  // raster: 16 m-blocks share a sweep over n

// PAIR: a 2-CTA cluster computes a 256 x BN tile with cta_group::2 MMAs; each
// CTA stages 128 rows of A and BN/2 rows of B per k-block, so a 256 x 256 x 64
// step moves 32 KB into each SM per 512 MMA cycles instead of 48 KB (the
// per-SM TMA ingress, about 57-76 bytes per cycle, bounds 1-SM 128 x 256 tiles).
template <int BN, bool PAIR = false>
struct GemmCfg {
  static constexpr int STAGES = PAIR ? 6 : (BN == 256 ? 4 : 6);
  static constexpr int TILE_M = PAIR ? 2 * kBM : kBM;  // output rows per tile
  static constexpr int A_BYTES = kBM * kBK * 2;
  static constexpr int B_BYTES = (PAIR ? BN / 2 : BN) * kBK * 2;
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr int TMEM_COLS = 2 * BN;  // two accumulators
  static constexpr int SMEM_BYTES = 1024 /*align slack*/ + STAGES * STAGE_BYTES + 256 + 1024;
};

struct TileInfo {
  int m0, n0, row_end, b_row0;
  int b_tile;  // blocked B: index of the tile's first 128-row block
  int bw;      // tile width: BN, or 128 for the split tail of a dense GEMM
};

// Map a linear tile id to output coordinates.  Dense mode: groups of kGroupM
// m-blocks are swept across all n-blocks so the active B tiles and A rows both
// stay in L2.  Grouped mode: (group, m-block within group, n-block).
//
// Dense mode with epi.split_tail: tiles from epi.split_from on (the last,
// partial wave) are cut in two 128-wide halves, so that wave spreads over
// twice as many SMs: tile split_from + 2 i + h is half h of tile split_from + i.
__device__ __forceinline__ bool get_tile(int tile, int M, int N, int BN, int n_nblk,
                                         const GemmEpilogue& epi, const int* s_tile_prefix,
                                         TileInfo& ti, int bm = kBM) {
  if (epi.group_offsets == nullptr) {
    const int n_mblk = (M + bm - 1) / bm;
    int half = -1;
    ti.bw = BN;
    if (epi.split_tail && tile >= epi.split_from) {
      const int r = tile - epi.split_from;
      half = r & 1;
      tile = epi.split_from + (r >> 1);
      ti.bw = 128;
    }
    if (tile >= n_mblk * n_nblk) return false;
    const int per_group = kGroupM * n_nblk;
    const int g = tile / per_group;
    const int first_m = g * kGroupM;
    const int gm = min(kGroupM, n_mblk - first_m);
    const int r = tile - g * per_group;
    const int mb = first_m + r % gm;
    const int nb = r / gm;
    ti.m0 = mb * bm;
    ti.n0 = nb * BN + (half > 0 ? 128 : 0);
    ti.row_end = M;
    ti.b_row0 = ti.n0;
    ti.b_tile = ti.n0 / 128;
    return true;
  }
  // grouped: s_tile_prefix[g] = m-tiles of groups < g (n_groups+1 entries)
  const int total_m = s_tile_prefix[epi.n_groups];
  if (tile >= total_m * n_nblk) return false;
  const int mt = tile / n_nblk;
  const int nb = tile - mt * n_nblk;
  int lo = 0, hi = epi.n_groups - 1;  // last g with prefix[g] <= mt
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (s_tile_prefix[mid] <= mt) lo = mid; else hi = mid - 1;
  }
  const int g = lo;
  const int row_begin = epi.group_offsets[g];
  ti.m0 = row_begin + (mt - s_tile_prefix[g]) * bm;
  ti.row_end = epi.group_offsets[g + 1];
  ti.n0 = nb * BN;
  ti.b_row0 = g * N + ti.n0;
  ti.b_tile = g * ((N + 127) / 128) + ti.n0 / 128;  // each group's rows padded to 128
  ti.bw = BN;
  return true;
}

template <int BN, int EPI>
__device__ __forceinline__ void epilogue_tile(uint32_t taddr, int row, bool row_ok, int n0,
                                              int N, const GemmEpilogue& epi, int* err, int bw) {
  if constexpr (EPI == EPI_QKV) {
    const int dh = epi.qkv.dh;
    if (dh == 128) {
#pragma unroll 1
      for (int h0 = 0; h0 < bw; h0 += 128) {
        float v[128];
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          uint32_t r[32];
          tmem_ld32(taddr + h0 + 32 * c, r);
          tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 32; ++i) v[32 * c + i] = __uint_as_float(r[i]);
        }
        if (row_ok && n0 + h0 < N) qkv_head_finish<128>(v, row, (n0 + h0) / 128, epi.qkv, err);
      }
    } else {
#pragma unroll 1
      for (int h0 = 0; h0 < bw; h0 += 64) {
        float v[64];
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          uint32_t r[32];
          tmem_ld32(taddr + h0 + 32 * c, r);
          tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 32; ++i) v[32 * c + i] = __uint_as_float(r[i]);
        }
        if (row_ok && n0 + h0 < N) qkv_head_finish<64>(v, row, (n0 + h0) / 64, epi.qkv, err);
      }
    }
  } else if constexpr (EPI == EPI_SWIGLU) {
    // columns [128j, 128j+64) are gate rows, [128j+64, 128j+128) the matching up rows
    bool bad = false;  // an H value beyond the FP16 range
#pragma unroll 1
    for (int j = 0; j < bw; j += 128) {
#pragma unroll 1
      for (int h = 0; h < 64; h += 32) {
        uint32_t g[32], u[32];
        tmem_ld32(taddr + j + h, g);
        tmem_ld32(taddr + j + 64 + h, u);
        tmem_ld_wait();
        const int col = (n0 + j) / 2 + h;  // output feature
        if (row_ok && n0 + j < N) {
          uint4* dst = reinterpret_cast<uint4*>(static_cast<uint16_t*>(epi.out) +
                                                (size_t)row * epi.ldo + col);
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            float o[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) {
              const float gv = __uint_as_float(g[8 * q + e]);
              o[e] = silu_f(gv) * __uint_as_float(u[8 * q + e]);
            }
            uint4 w;
            w.x = pack2_chk(o[0], o[1], epi.out_f16, bad);
            w.y = pack2_chk(o[2], o[3], epi.out_f16, bad);
            w.z = pack2_chk(o[4], o[5], epi.out_f16, bad);
            w.w = pack2_chk(o[6], o[7], epi.out_f16, bad);
            dst[q] = w;
          }
        }
      }
    }
    record_overflow(err, bad);
  } else {
    bool bad = false;  // an FP16 output beyond the format's range
#pragma unroll 1
    for (int c = 0; c < bw; c += 32) {
      uint32_t r[32];
      tmem_ld32(taddr + c, r);
      tmem_ld_wait();
      const int col = n0 + c;
      if (!row_ok || col >= N) continue;
      const bool full = col + 32 <= N;
      if constexpr (EPI == EPI_F32) {
        float* dst = epi.out32 + (size_t)row * epi.ldo32 + col;
        if (full) {
#pragma unroll
          for (int q = 0; q < 8; ++q)
            reinterpret_cast<float4*>(dst)[q] =
                make_float4(__uint_as_float(r[4 * q]), __uint_as_float(r[4 * q + 1]),
                            __uint_as_float(r[4 * q + 2]), __uint_as_float(r[4 * q + 3]));
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i)
            if (i < N - col) dst[i] = __uint_as_float(r[i]);
        }
      } else {
        float o[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) o[i] = __uint_as_float(r[i]);
        if constexpr (EPI == EPI_RESID) {
          if (epi.resid32) {
            const float* rs = epi.resid32 + (size_t)row * epi.ldr + col;
            if (full) {
#pragma unroll
              for (int q = 0; q < 8; ++q) {
                const float4 f = reinterpret_cast<const float4*>(rs)[q];
                o[4 * q] += f.x;
                o[4 * q + 1] += f.y;
                o[4 * q + 2] += f.z;
                o[4 * q + 3] += f.w;
              }
            } else {
#pragma unroll
              for (int i = 0; i < 32; ++i)
                if (i < N - col) o[i] += rs[i];
            }
          } else {
            const bf16* rs = epi.resid + (size_t)row * epi.ldr + col;
            if (full) {
#pragma unroll
              for (int q = 0; q < 4; ++q) {
                const uint4 u = reinterpret_cast<const uint4*>(rs)[q];
                const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                  const float2 f = unpack_bf16x2(w[e]);
                  o[8 * q + 2 * e] += f.x;
                  o[8 * q + 2 * e + 1] += f.y;
                }
              }
            } else {
#pragma unroll
              for (int i = 0; i < 32; ++i)
                if (i < N - col) o[i] += bf2f(rs[i]);
            }
          }
          if (epi.out32) {
            float* d32 = epi.out32 + (size_t)row * epi.ldo32 + col;
            if (full) {
#pragma unroll
              for (int q = 0; q < 8; ++q)
                reinterpret_cast<float4*>(d32)[q] =
                    make_float4(o[4 * q], o[4 * q + 1], o[4 * q + 2], o[4 * q + 3]);
            } else {
#pragma unroll
              for (int i = 0; i < 32; ++i)
                if (i < N - col) d32[i] = o[i];
            }
          }
          if (epi.out == nullptr) continue;
        }
        uint16_t* dst = static_cast<uint16_t*>(epi.out) + (size_t)row * epi.ldo + col;
        if (full) {
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            uint4 w;
            w.x = pack2_chk(o[8 * q], o[8 * q + 1], epi.out_f16, bad);
            w.y = pack2_chk(o[8 * q + 2], o[8 * q + 3], epi.out_f16, bad);
            w.z = pack2_chk(o[8 * q + 4], o[8 * q + 5], epi.out_f16, bad);
            w.w = pack2_chk(o[8 * q + 6], o[8 * q + 7], epi.out_f16, bad);
            reinterpret_cast<uint4*>(dst)[q] = w;
          }
        } else {
#pragma unroll
          for (int i = 0; i < 32; i += 2)
            if (i < N - col) {
              const uint32_t p = pack2_chk(o[i], o[i + 1], epi.out_f16, bad);
              dst[i] = static_cast<uint16_t>(p & 0xFFFFu);
              if (i + 1 < N - col) dst[i + 1] = static_cast<uint16_t>(p >> 16);
            }
        }
      }
    }
    record_overflow(err, bad);
  }
}

template <int BN, int EPI, bool PAIR>
__global__ void __launch_bounds__(kGemmThreads, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const __grid_constant__ CUtensorMap tmBh, int M, int N, int K, uint32_t idesc,
                   uint32_t idesc_half, GemmEpilogue epi, int* err) {
  using C = GemmCfg<BN, PAIR>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* sA = smem;
  uint8_t* sB = smem + C::STAGES * C::A_BYTES;
  uint64_t* full = reinterpret_cast<uint64_t*>(sB + C::STAGES * C::B_BYTES);
  uint64_t* empty = full + C::STAGES;
  uint64_t* tfull = empty + C::STAGES;
  uint64_t* tempty = tfull + 2;
  uint64_t* mma_done = tempty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(mma_done + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  int* s_tile_prefix = reinterpret_cast<int*>(tmem_slot + 4);  // up to 256 groups

  pdl_trigger();
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int n_nblk = (N + BN - 1) / BN;
  const int n_kblk = (K + kBK - 1) / kBK;
  // pair mode: both CTAs of a cluster walk the same tiles; rank 0 issues the MMAs
  const int rank = PAIR ? static_cast<int>(cluster_ctarank()) : 0;
  const int unit = PAIR ? static_cast<int>(blockIdx.x >> 1) : static_cast<int>(blockIdx.x);
  const int n_units = PAIR ? static_cast<int>(gridDim.x >> 1) : static_cast<int>(gridDim.x);

  if (threadIdx.x == 0) {
    if (epi.group_offsets) pdl_wait();  // the group offsets come from the previous kernel
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tfull[a], 1);
      mbar_init(&tempty[a], PAIR ? 256 : 128);  // the epilogue threads of both CTAs
    }
    mbar_init(mma_done, 1);
    *abort_flag = 0;
    if (epi.group_offsets) {
      int acc = 0;
      for (int g = 0; g < epi.n_groups; ++g) {
        s_tile_prefix[g] = acc;
        const int rows = epi.group_offsets[g + 1] - epi.group_offsets[g];
        acc += (rows + C::TILE_M - 1) / C::TILE_M;
      }
      s_tile_prefix[epi.n_groups] = acc;
    }
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
    if (epi.split_tail || PAIR) tma_prefetch_desc(&tmBh);  // pair mode: tmB only for split tails
  }
  if (warp == 1) {
    if constexpr (PAIR) {
      tmem_alloc_pair(tmem_slot, C::TMEM_COLS);
      tmem_relinquish_pair();
    } else {
      tmem_alloc(tmem_slot, C::TMEM_COLS);
      tmem_relinquish();
    }
  }
  tc_fence_before();
  if constexpr (PAIR)
    cluster_sync_all();  // both CTAs' barriers exist before any cross-CTA signal
  else
    __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  // B tile of k-block kb: row-major [N, K] (2-D map, rows from b_row0) or the
  // blocked layout of packed weights (4-D map, 128 x 64 tiles from b_tile).
  // 1-SM tiles: tmB carries a whole BN-row tile, tmBh the 128 rows of a
  // split-tail tile.  Pair tiles: each CTA loads its half of B, 128 rows by
  // tmBh, or 64 rows by tmB for a 128-wide split-tail tile.
  auto load_b = [&](uint8_t* dst, uint64_t* bar, int kb, const TileInfo& t) {
    if constexpr (PAIR) {
      const uint32_t bar0 = cluster_addr(bar, 0);
      if (t.bw == BN) {
        if (epi.b_blocked)
          tma_load_4d_pair_w(dst, &tmBh, bar0, 0, 0, kb, t.b_tile + rank);
        else
          tma_load_2d_pair_w(dst, &tmBh, bar0, kb * kBK, t.b_row0 + rank * (BN / 2));
      } else {
        if (epi.b_blocked)
          tma_load_4d_pair_w(dst, &tmB, bar0, 0, rank * 64, kb, t.b_tile);
        else
          tma_load_2d_pair_w(dst, &tmB, bar0, kb * kBK, t.b_row0 + rank * 64);
      }
    } else {
      const CUtensorMap* m = t.bw == BN ? &tmB : &tmBh;
      if (epi.b_blocked)
        tma_load_4d_w(dst, m, bar, 0, 0, kb, t.b_tile);
      else
        tma_load_2d_w(dst, m, bar, kb * kBK, t.b_row0);
    }
  };
  auto load_a = [&](uint8_t* dst, uint64_t* bar, int kb, const TileInfo& t) {
    if constexpr (PAIR)
      tma_load_2d_pair_w(dst, &tmA, cluster_addr(bar, 0), kb * kBK, t.m0 + rank * kBM);
    else
      tma_load_2d_w(dst, &tmA, bar, kb * kBK, t.m0);
  };
  // bytes the stage's barrier waits for (in pair mode: rank 0's barrier, both CTAs' tiles)
  auto stage_bytes = [&](const TileInfo& t) -> uint32_t {
    return PAIR ? (uint32_t)(2 * (C::A_BYTES + (t.bw / 2) * kBK * 2))
                : (uint32_t)(C::A_BYTES + t.bw * kBK * 2);
  };

  // warps 0 and 1 run converged and issue from one elected lane (a lone lane
  // next to busy epilogue warps gets too few issue slots)
  if (warp == 0) {
    {
      // stream the first B (weight) tiles while the previous kernel finishes
      int pre = 0;
      TileInfo ti;
      if (epi.b_static && !epi.group_offsets &&
          get_tile(unit, M, N, BN, n_nblk, epi, s_tile_prefix, ti, C::TILE_M)) {
        pre = min(C::STAGES, n_kblk);
        for (int i = 0; i < pre; ++i) {
          if (rank == 0) mbar_arrive_expect_tx_w(&full[i], stage_bytes(ti));
          load_b(sB + i * C::B_BYTES, &full[i], i, ti);
        }
      }
      pdl_wait();
      int stage = 0;
      uint32_t phase = 0;
      int g = 0;
      for (int tile = unit; get_tile(tile, M, N, BN, n_nblk, epi, s_tile_prefix, ti, C::TILE_M);
           tile += n_units) {
        for (int kb = 0; kb < n_kblk; ++kb, ++g) {
          if (g >= pre) {
            if (!mbar_wait_w(&empty[stage], phase ^ 1u, abort_flag, err)) goto producer_done;
            if (rank == 0) mbar_arrive_expect_tx_w(&full[stage], stage_bytes(ti));
            load_b(sB + stage * C::B_BYTES, &full[stage], kb, ti);
          }
          load_a(sA + stage * C::A_BYTES, &full[stage], kb, ti);
          if (++stage == C::STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      // drain: wait until the MMAs have consumed every stage we filled, so no
      // TMA write is still in flight when the CTA exits
      for (int s = 0; s < C::STAGES; ++s) {
        if (!mbar_wait_w(&empty[stage], phase ^ 1u, abort_flag, err)) break;
        if (++stage == C::STAGES) {
          stage = 0;
          phase ^= 1u;
        }
      }
    producer_done:;
    }
  } else if (warp == 1) {
    if (rank == 0) {
      int stage = 0;
      uint32_t phase = 0;
      int local = 0;
      TileInfo ti;
      for (int tile = unit; get_tile(tile, M, N, BN, n_nblk, epi, s_tile_prefix, ti, C::TILE_M);
           tile += n_units, ++local) {
        const int acc = local & 1;
        const uint32_t acc_phase = (local >> 1) & 1;
        if (!mbar_wait_w(&tempty[acc], acc_phase ^ 1u, abort_flag, err)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + acc * BN;
        bool ok = true;
        for (int kb = 0; kb < n_kblk; ++kb) {
          if (!mbar_wait_w(&full[stage], phase, abort_flag, err)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a0 = smem_u32(sA + stage * C::A_BYTES);
          const uint32_t b0 = smem_u32(sB + stage * C::B_BYTES);
#pragma unroll
          for (int k = 0; k < kBK / 16; ++k) {
            const uint64_t ad = smem_desc_sw128(a0 + 32 * k, 16, 1024);
            const uint64_t bd = smem_desc_sw128(b0 + 32 * k, 16, 1024);
            if constexpr (PAIR)
              umma_f16_pair_w(d_tmem, ad, bd, ti.bw == BN ? idesc : idesc_half, (kb | k) != 0);
            else
              umma_f16_w(d_tmem, ad, bd, ti.bw == BN ? idesc : idesc_half, (kb | k) != 0);
          }
          if constexpr (PAIR)
            umma_commit_pair_w(&empty[stage], 0x3);
          else
            umma_commit_w(&empty[stage]);
          if (++stage == C::STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        if constexpr (PAIR)
          umma_commit_pair_w(&tfull[acc], 0x3);
        else
          umma_commit_w(&tfull[acc]);
      }
      if constexpr (PAIR) {
        // the MMAs read the other CTA's shared memory: all of them have to be
        // complete before that CTA may leave (also on an early exit)
        umma_commit_pair_w(mma_done, 0x1);
        __syncwarp();
        if (!mbar_wait_drain(mma_done, 0, err)) *abort_flag = 1;
      }
    }
  } else {
    pdl_wait();  // residuals and outputs are shared with earlier kernels
    const int q = warp & 3;  // TMEM lane quarter this warp may access
    int local = 0;
    TileInfo ti;
    const uint32_t tempty0 = PAIR ? cluster_addr(&tempty[0], 0) : 0u;
    const uint32_t tempty1 = PAIR ? cluster_addr(&tempty[1], 0) : 0u;
    for (int tile = unit; get_tile(tile, M, N, BN, n_nblk, epi, s_tile_prefix, ti, C::TILE_M);
         tile += n_units, ++local) {
      const int acc = local & 1;
      const uint32_t acc_phase = (local >> 1) & 1;
      if (!mbar_wait(&tfull[acc], acc_phase, abort_flag, err)) break;
      tc_fence_after();
      const int row = ti.m0 + rank * kBM + q * 32 + lane;
      const uint32_t taddr = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + acc * BN;
      epilogue_tile<BN, EPI>(taddr, row, row < ti.row_end, ti.n0, N, epi, err, ti.bw);
      tc_fence_before();
      if constexpr (PAIR)
        mbar_arrive_cluster(acc ? tempty1 : tempty0);
      else
        mbar_arrive(&tempty[acc]);
    }
  }

  tc_fence_before();
  if constexpr (PAIR)
    cluster_sync_all();  // neither CTA leaves while the pair's MMAs may read it
  else
    __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    if constexpr (PAIR)
      tmem_dealloc_pair(tmem_base, C::TMEM_COLS);
    else
      tmem_dealloc(tmem_base, C::TMEM_COLS);
  }
}

// ------------------------------------------------------------------ host side

static PFN_cuTensorMapEncodeTiled_v12000 get_encode_fn() {
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

// 2-D BF16 tensor [rows][cols] with row stride `ld` elements; box [box_rows][64]
// with the 128-byte swizzle.
static bool make_tmap_16(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols,
                         uint64_t ld, uint32_t box_rows, bool f16) {
  auto enc = get_encode_fn();
  if (!enc) return false;
  if ((reinterpret_cast<uintptr_t>(base) & 15) || ((ld * 2) & 15)) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {ld * 2};
  cuuint32_t box[2] = {static_cast<cuuint32_t>(kBK), box_rows};
  cuuint32_t estr[2] = {1, 1};
  return enc(map, f16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
             const_cast<void*>(base), dims, strides,
             box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The blocked layout of packed weights: 128 x 64 tiles of 16 KB, tile (t, kt)
// at ((t * K/64) + kt) * 16 KB, rows of 64 elements inside a tile.  4-D map
// {64 elements, 128 rows, K/64 tiles, row tiles}; a box of `box_tiles`
// consecutive row tiles lands in shared memory as box_tiles * 128 rows.
static bool make_tmap_blocked(CUtensorMap* map, const void* base, uint64_t row_tiles, uint64_t K,
                              uint32_t box_tiles, bool f16, uint32_t box_rows = 128) {
  auto enc = get_encode_fn();
  if (!enc || (reinterpret_cast<uintptr_t>(base) & 15)) return false;
  const uint64_t kt = K / kBK;
  cuuint64_t dims[4] = {(cuuint64_t)kBK, 128, kt, row_tiles};
  cuuint64_t strides[3] = {kBK * 2, 128 * kBK * 2, kt * 128 * kBK * 2};
  cuuint32_t box[4] = {(cuuint32_t)kBK, box_rows, 1, box_tiles};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  return enc(map, f16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4,
             const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
             CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 2-CTA clusters of the pair kernel that fit on the device at once (every
// epilogue variant has the same shared memory and thread count); 0 if the
// query fails, which keeps every GEMM on 1-SM tiles.
static int pair_clusters() {
  // per device: 0 = not queried yet, else the count plus one
  static std::atomic<int> known[kMaxDevices] = {};
  const int dev = current_device();
  if (dev < 0) return 0;
  const int k = known[dev].load(std::memory_order_relaxed);
  if (k) return k - 1;
  int n = 0;
  auto kern = gemm_tc_kernel<256, EPI_STORE, true>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           GemmCfg<256, true>::SMEM_BYTES) == cudaSuccess) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * (device_sm_count() / 2));
    cfg.blockDim = dim3(kGemmThreads);
    cfg.dynamicSmemBytes = GemmCfg<256, true>::SMEM_BYTES;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int c = 0;
    if (cudaOccupancyMaxActiveClusters(&c, kern, &cfg) == cudaSuccess && c > 0) n = c;
  }
  cudaGetLastError();  // a failed query leaves no sticky error behind
  known[dev].store(n + 1, std::memory_order_relaxed);
  return n;
}

template <int BN, int EPI, bool PAIR>
static qwen_status launch_bn(const CUtensorMap& ta, const CUtensorMap& tb, const CUtensorMap& tbh,
                             int M, int N, int K, uint32_t idesc, uint32_t idesc_half,
                             const GemmEpilogue& epi, int* err, int units, cudaStream_t st) {
  auto kern = gemm_tc_kernel<BN, EPI, PAIR>;
  using C = GemmCfg<BN, PAIR>;
  static std::atomic<uint64_t> attr_done{0};  // per template instance, one bit per device
  cudaLaunchConfig_t cfg = {};
  cfg.blockDim = dim3(kGemmThreads);
  cfg.dynamicSmemBytes = C::SMEM_BYTES;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  int na = 0;
  if (PAIR) {
    attr[na].id = cudaLaunchAttributeClusterDimension;
    attr[na].val.clusterDim.x = 2;
    attr[na].val.clusterDim.y = 1;
    attr[na].val.clusterDim.z = 1;
    ++na;
  }
  if (!smem_attr_once(kern, C::SMEM_BYTES, attr_done)) return QWEN_ERR_CUDA;
  // persistent grid: co-resident CTAs (pair mode: clusters)
  const int max_units = PAIR ? pair_clusters() : device_sm_count();
  if (pdl_enabled()) {
    attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[na].val.programmaticStreamSerializationAllowed = 1;
    ++na;
  }
  const int grid_units = units < max_units ? units : max_units;
  cfg.gridDim = dim3((PAIR ? 2 : 1) * grid_units);
  cfg.attrs = attr;
  cfg.numAttrs = na;
  if (cudaLaunchKernelEx(&cfg, kern, ta, tb, tbh, M, N, K, idesc, idesc_half, epi, err) !=
      cudaSuccess)
    return QWEN_ERR_CUDA;
  count_launches();
  return cudaGetLastError() == cudaSuccess ? QWEN_OK : QWEN_ERR_CUDA;
}

template <int EPI>
static qwen_status launch_epi(bool pair, const CUtensorMap& ta, const CUtensorMap& tb,
                              const CUtensorMap& tbh, int M, int N, int K, uint32_t idesc,
                              uint32_t idesc_half, const GemmEpilogue& epi, int* err, int units,
                              cudaStream_t st) {
  return pair ? launch_bn<256, EPI, true>(ta, tb, tbh, M, N, K, idesc, idesc_half, epi, err, units,
                                          st)
              : launch_bn<256, EPI, false>(ta, tb, tbh, M, N, K, idesc, idesc_half, epi, err,
                                           units, st);
}

qwen_status gemm_tc(const void* A, int lda, const void* B, int ldb, int M, int N, int K,
                    bool op_f16, const GemmEpilogue& epi_in, int* err, cudaStream_t st) {
  if (M == 0 || N == 0) return QWEN_OK;
  if (K <= 0 || (K & 7) || (N & 7)) return QWEN_ERR_UNSUPPORTED;
  if (epi_in.group_offsets && (epi_in.n_groups <= 0 || epi_in.n_groups > 250))
    return QWEN_ERR_UNSUPPORTED;
  constexpr int BN = 256;
  GemmEpilogue epi = epi_in;
  const int sms = device_sm_count();
  epi.split_tail = 0;
  epi.split_from = 0;
  // 1-SM tiles (128 x 256) or pair tiles (256 x 256 on a 2-CTA cluster).  A
  // 1-SM tile is bound by its SM's TMA ingress and took about 1.1x the time of
  // a pair tile in measurements (T=4096 gate/up and down projections); the
  // choice compares the two wave counts on that basis.
  //
  // Wave quantisation: with T tiles on S units (SMs or clusters) the last wave
  // holds T mod S tiles.  Cutting those in two 128-wide halves spreads them
  // over twice as many units.  A 1-SM half tile takes about 2/3 of a full one
  // (its B box is half, its A box the same); a pair half tile (each CTA: 128
  // rows of A and 64 of B per k-block, 24 KB per 256 MMA cycles) about 0.78 at
  // the ingress rate.  Split when that shortens the estimate by 4 % or more
  // (below that, measured gains and losses were within noise).
  auto tail_split = [](int tiles, int units, double half_cost, double& t) -> bool {
    const int full_waves = tiles / units, rem = tiles - full_waves * units;
    t = full_waves + (rem > 0 ? 1.0 : 0.0);
    if (rem == 0) return false;
    const double t_split = full_waves + ((2 * rem + units - 1) / units) * half_cost;
    if (t_split >= 0.96 * t) return false;
    t = t_split;
    return true;
  };
  bool pair = false;
  int grid;
  if (epi.group_offsets) {
    // expert groups: the row count per group is only known on the device; a
    // 256-row tile wastes more of a group's ragged last tile, which measured as
    // a loss at 256 routed rows per expert on average and a gain at 512
    pair = M >= 384 * epi.n_groups && pair_clusters() > 0;
    grid = sms;  // the number of tiles is only known on the device
  } else {
    const int tiles = ((M + kBM - 1) / kBM) * ((N + BN - 1) / BN);
    double t_one;
    const bool split_one = tail_split(tiles, sms, 2.0 / 3.0, t_one);
    const int clusters = M >= 2 * kBM ? pair_clusters() : 0;
    const int ptiles = ((M + 2 * kBM - 1) / (2 * kBM)) * ((N + BN - 1) / BN);
    double t_pair = 0.0;
    const bool split_pair = clusters > 0 && tail_split(ptiles, clusters, 0.78, t_pair);
    pair = clusters > 0 && t_pair < 1.1 * t_one;
    const bool split = pair ? split_pair : split_one;
    const int n = pair ? ptiles : tiles, units = pair ? clusters : sms;
    grid = n;
    if (split) {
      const int full_waves = n / units;
      epi.split_tail = 1;
      epi.split_from = full_waves * units;
      grid = epi.split_from + 2 * (n - epi.split_from);
    }
    if (!pair && grid > sms) grid = sms;
  }
  const uint64_t b_rows = epi.group_offsets ? (uint64_t)N * epi.n_groups : (uint64_t)N;
  CUtensorMap ta, tb, tbh;
  if (!make_tmap_16(&ta, A, (uint64_t)M, (uint64_t)K, (uint64_t)lda, kBM, op_f16))
    return QWEN_ERR_CUDA;
  // B boxes.  1-SM tiles: tb a whole tile (BN rows), tbh a split-tail half
  // (128 rows).  Pair tiles: tbh one CTA's half of a tile (128 rows), tb one
  // CTA's half of a split-tail tile (64 rows).
  const uint32_t tb_rows = pair ? 64 : BN;
  if (epi.b_blocked) {
    if (K % kBK) return QWEN_ERR_UNSUPPORTED;
    const uint64_t tiles = (uint64_t)(epi.group_offsets ? epi.n_groups : 1) * ((N + 127) / 128);
    const bool ok_tb = pair ? make_tmap_blocked(&tb, B, tiles, (uint64_t)K, 1, op_f16, 64)
                            : make_tmap_blocked(&tb, B, tiles, (uint64_t)K, BN / 128, op_f16);
    if (!ok_tb || !make_tmap_blocked(&tbh, B, tiles, (uint64_t)K, 1, op_f16))
      return QWEN_ERR_CUDA;
  } else if (!make_tmap_16(&tb, B, b_rows, (uint64_t)K, (uint64_t)ldb, tb_rows, op_f16) ||
             !make_tmap_16(&tbh, B, b_rows, (uint64_t)K, (uint64_t)ldb, 128, op_f16)) {
    return QWEN_ERR_CUDA;
  }
  const uint32_t idesc = idesc_f32acc(pair ? 2 * kBM : kBM, BN, op_f16);
  const uint32_t idesc_half = idesc_f32acc(pair ? 2 * kBM : kBM, 128, op_f16);
  switch (epi.mode) {
    case EPI_STORE:
      return launch_epi<EPI_STORE>(pair, ta, tb, tbh, M, N, K, idesc, idesc_half, epi, err, grid, st);
    case EPI_RESID:
      return launch_epi<EPI_RESID>(pair, ta, tb, tbh, M, N, K, idesc, idesc_half, epi, err, grid, st);
    case EPI_SWIGLU:
      return launch_epi<EPI_SWIGLU>(pair, ta, tb, tbh, M, N, K, idesc, idesc_half, epi, err, grid, st);
    case EPI_QKV:
      return launch_epi<EPI_QKV>(pair, ta, tb, tbh, M, N, K, idesc, idesc_half, epi, err, grid, st);
    case EPI_F32:
      return launch_epi<EPI_F32>(pair, ta, tb, tbh, M, N, K, idesc, idesc_half, epi, err, grid, st);
    default: return QWEN_ERR_INVALID_ARG;
  }
}

}  // namespace qwen
