// Expert GEMMs of the mixture-of-experts block in prefill, with the expert
// weights on the tensor core's M side.
//
// "Qwen2.5-7B 结构拆解" §10.2 / the "MoE 初步" lecture (Expert section): each
// routed (token, slot) row goes through its expert's SwiGLU, gate/up then
// down.  After the permutation the routed rows of expert e are the rows
// [offsets[e], offsets[e+1]) of one matrix.  Tiling those rows by 128 (the
// M side of an MMA) pads every expert's last tile: with skewed loads of ~256
// rows per expert that is about 28 % extra MMA work, and 62 % with 256-row
// tiles.  Here the weight rows take the M side instead (a 2-CTA pair holds
// 256 weight rows, cta_group::2) and an expert's routed rows are the N side,
// taken in chunks of up to 256 rounded up to a multiple of 16: about 3 %
// padding, and each CTA stages 16 KB of weights plus at most 16 KB of rows per
// k-block, within what one SM's TMA delivers per 512 MMA cycles.
//
// Work unit = (expert e, 256-row weight tile w, chunk c of <= 256 routed rows),
// numbered expert by expert, weight tile by weight tile, chunks fastest, so
// the chunks that share a weight tile run on neighbouring clusters and find it
// in L2.  The accumulator D[256 weight rows][N rows] sits in tensor memory,
// each CTA holding its 128 weight rows; so in the epilogue a lane holds one
// output feature of every row.  Each warp stages its 32 features of 32 rows
// in shared memory and stores them as 64-byte row segments, 8 rows per
// instruction (one row per instruction measured 2-3x slower than the MMAs).
//
//   warp 0      TMA producer (one elected lane): this CTA's 128 weight rows
//               (one blocked 128 x 64 tile) and its half of the chunk's rows
//               (one 128-row box; a short last chunk loads rows it does not
//               use: 32- and 64-row boxes measured slower) per k-block; both
//               CTAs signal the even CTA's barrier
//   warp 1      TMEM allocation; in the even CTA, the pair MMA issuer
//   warps 2..5  epilogue.  SwiGLU: a 128-row weight tile holds 64 gate rows
//               (TMEM lanes 0-63) and the 64 matching up rows (lanes 64-127),
//               so the gate warps compute SiLU(gate) and hand it to the up
//               warps through shared memory, 32 routed rows at a time.
#include "common.cuh"
#include "internal.h"
#include "layer.h"

#include <cudaTypedefs.h>

namespace qwen {

namespace {

constexpr int kXT = 256;      // routed rows per chunk: the MMA's N at most
constexpr int kXBox = 128;    // rows per TMA box of the routed-row operand (one CTA's half)
constexpr int kEBK = 64;      // k-block (128 bytes of FP16)
constexpr int kEThreads = 192;
constexpr int kEStages = 6;
constexpr int kEMaxExperts = 256;
constexpr int kEA = 128 * kEBK * 2;  // this CTA's 128 weight rows of a k-block
constexpr int kEB = 128 * kEBK * 2;  // this CTA's half (<= 128) of the chunk's rows
constexpr int kEXch = 32 * 64 * 4;   // gate hand-off: 32 rows x 64 features, FP32
constexpr int kEOffA = 0;
constexpr int kEOffB = kEOffA + kEStages * kEA;
constexpr int kEOffXch = kEOffB + kEStages * kEB;
constexpr int kEStg = 32 * 32 * 2;    // one epilogue warp's 32 x 32 FP16 output block
constexpr int kEOffStg = kEOffXch + kEXch;
constexpr int kEOffPre = kEOffStg + 4 * kEStg;                    // chunk prefix [E + 1]
constexpr int kEOffRows = kEOffPre + (kEMaxExperts + 1) * 4;      // row offsets [E + 1]
constexpr int kEOffBar = (kEOffRows + (kEMaxExperts + 1) * 4 + 7) & ~7;
constexpr int kESmem = 1024 + kEOffBar + 256;
static_assert(kESmem <= 232448, "shared memory budget");

enum ExpEpi : int { EXP_SWIGLU = 0, EXP_STORE = 1 };

}  // namespace

// One epilogue warp's output block: rows c .. c + 31 of the chunk (a thread
// holds one feature of each) are staged in shared memory, stg[row * 32 +
// lane], then stored as 64-byte row segments, four lanes per row: 8 rows per
// instruction instead of one 64-byte row.  Rows >= nrows are not stored.
__device__ __forceinline__ void expert_store_block(const uint16_t* stg, int lane, f16* dst,
                                                   size_t ldo, int nrows) {
  __syncwarp();
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int rr = j * 8 + (lane >> 2), ch = lane & 3;
    if (rr < nrows)
      *reinterpret_cast<uint4*>(dst + (size_t)rr * ldo + ch * 8) =
          *reinterpret_cast<const uint4*>(stg + rr * 32 + ch * 8);
  }
  __syncwarp();
}

// 32 values of this lane's feature, rows 0..31 of the block, into the staging
// area as FP16.  One max of |v| decides whether any value would pass FP16's
// range; only then the saturating conversion runs (and records it in bad).
__device__ __forceinline__ void stage_f16(const float (&v)[32], uint16_t* stg, int lane,
                                          bool& bad) {
  float mx = 0.f;
#pragma unroll
  for (int i = 0; i < 32; ++i) mx = fmaxf(mx, fabsf(v[i]));
  if (mx < 65520.f) {
#pragma unroll
    for (int i = 0; i < 32; ++i) stg[i * 32 + lane] = __half_as_ushort(__float2half_rn(v[i]));
  } else {
#pragma unroll
    for (int i = 0; i < 32; ++i) stg[i * 32 + lane] = __half_as_ushort(f16_chk(v[i], bad));
  }
}

// W: blocked FP16 [E][Nw][K] (each expert's rows padded to 128; for SwiGLU the
// gate and up rows interleaved in 64-row blocks), X: FP16 routed rows
// [rows][K], row stride ldx.  out: SwiGLU -> H [rows][Nw / 2], store -> Y
// [rows][Nw], FP16, row stride ldo.
template <int EPI>
__global__ void __launch_bounds__(kEThreads, 1)
    gemm_expert_kernel(const __grid_constant__ CUtensorMap tmW,
                       const __grid_constant__ CUtensorMap tmX, int E, int Nw, int K,
                       const int32_t* __restrict__ offsets, f16* __restrict__ out, int ldo,
                       int* err) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* sA = smem + kEOffA;
  uint8_t* sB = smem + kEOffB;
  float* xch = reinterpret_cast<float*>(smem + kEOffXch);
  uint16_t* stg = reinterpret_cast<uint16_t*>(smem + kEOffStg + (threadIdx.x >> 5 & 3) * kEStg);
  int* s_pre = reinterpret_cast<int*>(smem + kEOffPre);
  int* s_off = reinterpret_cast<int*>(smem + kEOffRows);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kEOffBar);
  uint64_t* empty = full + kEStages;
  uint64_t* tfull = empty + kEStages;
  uint64_t* tempty = tfull + 2;
  uint64_t* x_full = tempty + 2;   // gate values of 32 rows in xch
  uint64_t* x_empty = x_full + 1;  // xch read by the up warps
  uint64_t* mma_done = x_empty + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(mma_done + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  pdl_trigger();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int rank = static_cast<int>(cluster_ctarank());
  const int cl = static_cast<int>(blockIdx.x >> 1), n_cl = static_cast<int>(gridDim.x >> 1);
  const int n_wt = Nw / 256;         // 256-row weight tiles per expert
  const int n_t128 = (Nw + 127) / 128;  // blocked 128-row tiles per expert
  const int n_kblk = K / kEBK;

  if (threadIdx.x == 0) {
    pdl_wait();  // the row offsets come from the permutation kernel
    int acc = 0;
    for (int e = 0; e < E; ++e) {
      const int o0 = offsets[e], o1 = offsets[e + 1];
      s_off[e] = o0;
      s_pre[e] = acc;
      acc += (o1 - o0 + kXT - 1) / kXT;
    }
    s_off[E] = offsets[E];
    s_pre[E] = acc;
    for (int s = 0; s < kEStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tfull[a], 1);
      mbar_init(&tempty[a], 256);  // the epilogue threads of both CTAs
    }
    mbar_init(x_full, 64);
    mbar_init(x_empty, 64);
    mbar_init(mma_done, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmW);
    tma_prefetch_desc(&tmX);
  }
  if (warp == 1) {
    tmem_alloc_pair(tmem_slot, 512);  // two accumulators of up to 256 columns
    tmem_relinquish_pair();
  }
  tc_fence_before();
  cluster_sync_all();  // both CTAs' barriers exist before any cross-CTA signal
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const int n_units = s_pre[E] * n_wt;

  // unit -> expert e, weight tile w, first routed row row0 and row count m
  auto unit_of = [&](int u, int& e, int& w, int& row0, int& m) {
    const int key = u / n_wt;  // base of expert e is n_wt * s_pre[e]
    int lo = 0, hi = E - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (s_pre[mid] <= key) lo = mid; else hi = mid - 1;
    }
    e = lo;
    const int nc = s_pre[e + 1] - s_pre[e];
    const int r = u - n_wt * s_pre[e];
    w = r / nc;
    row0 = s_off[e] + (r - w * nc) * kXT;
    m = min(kXT, s_off[e + 1] - row0);
  };
  // the MMA's N: the chunk's rows rounded up to 16; each CTA holds half
  auto n_of = [](int m) { return (m + 15) & ~15; };

  if (warp == 0) {
    pdl_wait();  // the routed rows come from the kernels before
    const uint32_t bar0 = cluster_addr(&full[0], 0);
    int stage = 0;
    uint32_t phase = 0;
    for (int u = cl; u < n_units; u += n_cl) {
      int e, w, row0, m;
      unit_of(u, e, w, row0, m);
      const int half = n_of(m) >> 1;
      const int nbox = (half + kXBox - 1) / kXBox;
      const uint32_t bytes = 2u * (uint32_t)(kEA + nbox * kXBox * kEBK * 2);
      const int wtile = e * n_t128 + 2 * w + rank;
      for (int kb = 0; kb < n_kblk; ++kb) {
        if (!mbar_wait_w(&empty[stage], phase ^ 1u, abort_flag, err)) goto prod_done;
        if (rank == 0) mbar_arrive_expect_tx_w(&full[stage], bytes);
        const uint32_t bar = bar0 + (uint32_t)(stage * sizeof(uint64_t));
        tma_load_4d_pair_w(sA + stage * kEA, &tmW, bar, 0, 0, kb, wtile);
        for (int i = 0; i < nbox; ++i)
          tma_load_2d_pair_w(sB + stage * kEB + i * kXBox * 128, &tmX, bar, kb * kEBK,
                             row0 + rank * half + i * kXBox);
        if (++stage == kEStages) {
          stage = 0;
          phase ^= 1u;
        }
      }
    }
    // drain: every stage filled has been consumed before the CTA may exit
    for (int s = 0; s < kEStages; ++s) {
      if (!mbar_wait_w(&empty[stage], phase ^ 1u, abort_flag, err)) break;
      if (++stage == kEStages) {
        stage = 0;
        phase ^= 1u;
      }
    }
  prod_done:;
  } else if (warp == 1) {
    if (rank == 0) {
      int stage = 0;
      uint32_t phase = 0;
      int local = 0;
      for (int u = cl; u < n_units; u += n_cl, ++local) {
        int e, w, row0, m;
        unit_of(u, e, w, row0, m);
        const uint32_t idesc = idesc_f32acc(256, n_of(m), true);
        const int acc = local & 1;
        if (!mbar_wait_w(&tempty[acc], ((local >> 1) & 1) ^ 1u, abort_flag, err)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + acc * kXT;
        bool ok = true;
        for (int kb = 0; kb < n_kblk; ++kb) {
          if (!mbar_wait_w(&full[stage], phase, abort_flag, err)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a0 = smem_u32(sA + stage * kEA);
          const uint32_t b0 = smem_u32(sB + stage * kEB);
#pragma unroll
          for (int k = 0; k < kEBK / 16; ++k)
            umma_f16_pair_w(d_tmem, smem_desc_sw128(a0 + 32 * k, 16, 1024),
                            smem_desc_sw128(b0 + 32 * k, 16, 1024), idesc, (kb | k) != 0);
          umma_commit_pair_w(&empty[stage], 0x3);
          if (++stage == kEStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        umma_commit_pair_w(&tfull[acc], 0x3);
      }
      // the MMAs read the other CTA's shared memory: all of them complete
      // before that CTA may leave (also on an early exit)
      umma_commit_pair_w(mma_done, 0x1);
      __syncwarp();
      if (!mbar_wait_drain(mma_done, 0, err)) *abort_flag = 1;
    }
  } else {
    pdl_wait();  // the outputs may still be read by an earlier kernel
    const int q = warp & 3;  // TMEM lane quarter of this warp
    const uint32_t tempty0 = cluster_addr(&tempty[0], 0);
    const uint32_t tempty1 = cluster_addr(&tempty[1], 0);
    int local = 0, ch = 0;  // units done; 32-row hand-offs done (SwiGLU)
    bool bad = false;       // an FP16 output beyond the format's range
    for (int u = cl; u < n_units; u += n_cl, ++local) {
      int e, w, row0, m;
      unit_of(u, e, w, row0, m);
      const int acc = local & 1;
      if (!mbar_wait(&tfull[acc], (local >> 1) & 1, abort_flag, err)) break;
      tc_fence_after();
      const uint32_t taddr = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + acc * kXT;
      bool ok = true;
      if constexpr (EPI == EXP_STORE) {
        // this warp's 32 features of the CTA's 128 weight rows
        f16* dst = out + (size_t)row0 * ldo + (w * 256 + rank * 128 + q * 32);
        for (int c = 0; c < m; c += 32) {
          uint32_t r[32];
          tmem_ld32(taddr + c, r);
          tmem_ld_wait();
          float v[32];
#pragma unroll
          for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
          stage_f16(v, stg, lane, bad);
          expert_store_block(stg, lane, dst + (size_t)c * ldo, ldo, m - c);
        }
      } else {
        // this CTA's 128-row weight tile: features 64 (2w + rank) + 0..63; the
        // gate warps pass SiLU(gate) on, the up warps multiply and store
        f16* dst = out + (size_t)row0 * ldo + ((2 * w + rank) * 64 + (q & 1) * 32);
        for (int c = 0; c < m; c += 32, ++ch) {
          uint32_t r[32];
          tmem_ld32(taddr + c, r);
          tmem_ld_wait();
          if (q < 2) {
            float sg[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) sg[i] = silu_f(__uint_as_float(r[i]));
            if (!mbar_wait(x_empty, (ch & 1) ^ 1u, abort_flag, err)) { ok = false; break; }
#pragma unroll
            for (int i = 0; i < 32; ++i) xch[i * 64 + q * 32 + lane] = sg[i];
            mbar_arrive(x_full);
          } else {
            if (!mbar_wait(x_full, ch & 1, abort_flag, err)) { ok = false; break; }
            float v[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) v[i] = xch[i * 64 + (q - 2) * 32 + lane] * __uint_as_float(r[i]);
            mbar_arrive(x_empty);
            stage_f16(v, stg, lane, bad);
            expert_store_block(stg, lane, dst + (size_t)c * ldo, ldo, m - c);
          }
        }
      }
      if (!ok) break;
      tc_fence_before();
      mbar_arrive_cluster(acc ? tempty1 : tempty0);
    }
    record_overflow(err, bad);
  }

  tc_fence_before();
  cluster_sync_all();  // neither CTA leaves while the pair's MMAs may read it
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, 512);
  }
}

// ------------------------------------------------------------------ host side

namespace {

PFN_cuTensorMapEncodeTiled_v12000 expert_encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult qr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &qr) == cudaSuccess &&
        qr == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}

// Clusters of two gemm_expert_kernel CTAs that fit on the device at once.
int expert_clusters() {
  static std::atomic<int> known[kMaxDevices] = {};  // count + 1; 0 = not queried
  const int dev = current_device();
  if (dev < 0) return 0;
  const int k = known[dev].load(std::memory_order_relaxed);
  if (k) return k - 1;
  int n = 0;
  auto kern = gemm_expert_kernel<EXP_SWIGLU>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kESmem) ==
      cudaSuccess) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * (device_sm_count() / 2));
    cfg.blockDim = dim3(kEThreads);
    cfg.dynamicSmemBytes = kESmem;
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

}  // namespace

bool gemm_expert_supported(int E, int Nw, int K) {
  return E > 0 && E <= kEMaxExperts && Nw % 256 == 0 && K % kEBK == 0 && expert_clusters() > 0;
}

qwen_status gemm_expert(const f16* W, int E, int Nw, int K, const f16* X, int rows, int ldx,
                        const int32_t* offsets, f16* out, int ldo, bool swiglu, int* err,
                        cudaStream_t st) {
  if (rows == 0) return QWEN_OK;
  if (!gemm_expert_supported(E, Nw, K)) return QWEN_ERR_UNSUPPORTED;
  auto enc = expert_encode_fn();
  if (!enc || (reinterpret_cast<uintptr_t>(W) & 15) || (reinterpret_cast<uintptr_t>(X) & 15) ||
      ((ldx * 2) & 15))
    return QWEN_ERR_CUDA;
  // weights: the blocked layout, 4-D {64 elements, 128 rows, K/64 tiles, row tiles}
  CUtensorMap tw, tx;
  {
    const uint64_t kt = (uint64_t)K / kEBK, tiles = (uint64_t)E * ((Nw + 127) / 128);
    cuuint64_t dims[4] = {(cuuint64_t)kEBK, 128, kt, tiles};
    cuuint64_t strides[3] = {kEBK * 2, 128 * kEBK * 2, kt * 128 * kEBK * 2};
    cuuint32_t box[4] = {(cuuint32_t)kEBK, 128, 1, 1};
    cuuint32_t es[4] = {1, 1, 1, 1};
    if (enc(&tw, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 4, const_cast<f16*>(W), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return QWEN_ERR_CUDA;
  }
  {
    // routed rows: 2-D [rows][K], boxes of 64 columns x 32 rows (rows past the
    // end read as zero)
    cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)ldx * 2};
    cuuint32_t box[2] = {(cuuint32_t)kEBK, (cuuint32_t)kXBox};
    cuuint32_t es[2] = {1, 1};
    if (enc(&tx, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<f16*>(X), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return QWEN_ERR_CUDA;
  }
  auto kern = swiglu ? gemm_expert_kernel<EXP_SWIGLU> : gemm_expert_kernel<EXP_STORE>;
  static std::atomic<uint64_t> attr_sw{0}, attr_st{0};  // one bit per device
  if (!smem_attr_once(kern, kESmem, swiglu ? attr_sw : attr_st)) return QWEN_ERR_CUDA;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * expert_clusters());  // persistent; units are known on the device
  cfg.blockDim = dim3(kEThreads);
  cfg.dynamicSmemBytes = kESmem;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  int na = 1;
  if (pdl_enabled()) {
    attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[na].val.programmaticStreamSerializationAllowed = 1;
    ++na;
  }
  cfg.attrs = attr;
  cfg.numAttrs = na;
  if (cudaLaunchKernelEx(&cfg, kern, tw, tx, E, Nw, K, offsets, out, ldo, err) != cudaSuccess)
    return QWEN_ERR_CUDA;
  count_launches();
  return cudaGetLastError() == cudaSuccess ? QWEN_OK : QWEN_ERR_CUDA;
}

}  // namespace qwen
