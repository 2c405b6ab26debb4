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
// Persistent: one CTA per SM walks a list of work items.  A work item = one
// sequence b, one KV group g, two query heads of that group (A and B; B absent
// for the last head of an odd-sized group, or in every item when one head per
// item is chosen for short sequences) and one tile of 128 query rows.  Both
// heads read every staged K/V tile: a single SM's TMA delivers about 64 bytes
// per cycle, and one head alone would need a 64 KB K/V tile per 1024 cycles of
// MMA work; two heads halve that.  Items are numbered heaviest first and dealt
// to the CTAs in a snake order; the K/V ring and the S/P/O hand-offs carry
// over from one item to the next.
//   warp 0      TMA: Q_A, Q_B once, then K (2 stages) and V (1 stage) tiles of
//               128 keys, in the order K(j+1), V(j)
//   warps 1, 2  MMA issuers of head A and head B (TMEM allocation by warp 1):
//               S_x(j+1) = Q_x K_{j+1}^T as soon as the softmax has read S_x(j)
//               into registers, and O_x += P_x(j) V_j once it has written P_x(j)
//               to shared memory.  Each issuer runs its loop as a converged warp
//               and issues from one elected lane: a lone lane next to busy
//               softmax warps gets too few issue slots.
//   warps 3-6   softmax of head A, warps 7-10 softmax of head B: one thread per
//               query row; online max / sum in FP32 with the rescale of O
//               deferred until the running max grows by 2^8; P in the
//               128-byte-swizzled K-major layout the MMA reads; final O / l.
// Tensor memory: S_A, S_B (128 columns each), O_A, O_B (dh columns each).
//
// Operands: when the sequence starts at slot 0 every key comes from this call,
// so Q, K, V and P are FP16 (the QKV epilogue writes FP16 copies of the new K/V
// rows besides the BF16 cache).  A chunk appended to a filled cache reads the
// BF16 cache instead; then the QKV epilogue has written Q in BF16 and P is
// rounded to BF16.
#include "common.cuh"
#include "internal.h"

#include <cudaTypedefs.h>

namespace qwen {

namespace {

constexpr int kQT = 128;      // query rows per CTA
constexpr int kKT = 128;      // keys per tile
constexpr int kKStages = 2;   // K ring; V has a single stage
constexpr int kAttnThreads = 352;
constexpr float kRescaleLog2 = 8.0f;  // defer O rescale until the max grew by 2^8

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Two FP32 values as one 64-bit operand of the packed f32x2 instructions (lo
// in the low word).
__device__ __forceinline__ uint64_t f32x2(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}

// Two exponent arguments s0 c + n, s1 c + n by one packed FP32 FMA.
__device__ __forceinline__ void fma_pair(float s0, float s1, uint64_t c2, uint64_t n2, float& x0,
                                         float& x1) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(f32x2(s0, s1)), "l"(c2), "l"(n2));
  asm("mov.b64 {%0, %1}, %2;" : "=f"(x0), "=f"(x1) : "l"(d));
}

// Two products x0 c, x1 c by one packed FP32 multiply.
__device__ __forceinline__ void mul_pair(float x0, float x1, uint64_t c2, float& y0, float& y1) {
  uint64_t d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(f32x2(x0, x1)), "l"(c2));
  asm("mov.b64 {%0, %1}, %2;" : "=f"(y0), "=f"(y1) : "l"(d));
}

__device__ __forceinline__ float max3(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

// 128 consecutive TMEM columns of this warp's 32 lanes -> registers; the wait
// for the load sits in the same statement, so no use can move above it.
__device__ __forceinline__ void tmem_ld128_wait(uint32_t taddr, uint32_t (&r)[128]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x128.b32 {"
      "%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, "
      "%32, %33, %34, %35, %36, %37, %38, %39, %40, %41, %42, %43, %44, %45, %46, %47, "
      "%48, %49, %50, %51, %52, %53, %54, %55, %56, %57, %58, %59, %60, %61, %62, %63, "
      "%64, %65, %66, %67, %68, %69, %70, %71, %72, %73, %74, %75, %76, %77, %78, %79, "
      "%80, %81, %82, %83, %84, %85, %86, %87, %88, %89, %90, %91, %92, %93, %94, %95, "
      "%96, %97, %98, %99, %100, %101, %102, %103, %104, %105, %106, %107, %108, %109, %110, %111, "
      "%112, %113, %114, %115, %116, %117, %118, %119, %120, %121, %122, %123, %124, %125, %126, %127"
      "}, [%128];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]),
        "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]), "=r"(r[37]), "=r"(r[38]), "=r"(r[39]),
        "=r"(r[40]), "=r"(r[41]), "=r"(r[42]), "=r"(r[43]), "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]),
        "=r"(r[48]), "=r"(r[49]), "=r"(r[50]), "=r"(r[51]), "=r"(r[52]), "=r"(r[53]), "=r"(r[54]), "=r"(r[55]),
        "=r"(r[56]), "=r"(r[57]), "=r"(r[58]), "=r"(r[59]), "=r"(r[60]), "=r"(r[61]), "=r"(r[62]), "=r"(r[63]),
        "=r"(r[64]), "=r"(r[65]), "=r"(r[66]), "=r"(r[67]), "=r"(r[68]), "=r"(r[69]), "=r"(r[70]), "=r"(r[71]),
        "=r"(r[72]), "=r"(r[73]), "=r"(r[74]), "=r"(r[75]), "=r"(r[76]), "=r"(r[77]), "=r"(r[78]), "=r"(r[79]),
        "=r"(r[80]), "=r"(r[81]), "=r"(r[82]), "=r"(r[83]), "=r"(r[84]), "=r"(r[85]), "=r"(r[86]), "=r"(r[87]),
        "=r"(r[88]), "=r"(r[89]), "=r"(r[90]), "=r"(r[91]), "=r"(r[92]), "=r"(r[93]), "=r"(r[94]), "=r"(r[95]),
        "=r"(r[96]), "=r"(r[97]), "=r"(r[98]), "=r"(r[99]), "=r"(r[100]), "=r"(r[101]), "=r"(r[102]), "=r"(r[103]),
        "=r"(r[104]), "=r"(r[105]), "=r"(r[106]), "=r"(r[107]), "=r"(r[108]), "=r"(r[109]), "=r"(r[110]), "=r"(r[111]),
        "=r"(r[112]), "=r"(r[113]), "=r"(r[114]), "=r"(r[115]), "=r"(r[116]), "=r"(r[117]), "=r"(r[118]), "=r"(r[119]),
        "=r"(r[120]), "=r"(r[121]), "=r"(r[122]), "=r"(r[123]), "=r"(r[124]), "=r"(r[125]), "=r"(r[126]), "=r"(r[127])
      : "r"(taddr)
      : "memory");
}

__device__ __forceinline__ void tmem_ld32_wait(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {"
      "%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31"
      "}, [%32];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
        "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
        "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
        "=r"(r[31])
      : "r"(taddr)
      : "memory");
}

template <int DH>
struct AttnCfg {
  static constexpr int TILE_BYTES = kKT * DH * 2;  // one [128 x DH] 16-bit tile
  static constexpr int P_BYTES = kQT * kKT * 2;    // one [128 x 128] 16-bit P tile
  static constexpr int Q_OFF = 0;                  // Q_A, Q_B
  static constexpr int K_OFF = 2 * TILE_BYTES;     // kKStages tiles
  static constexpr int V_OFF = K_OFF + kKStages * TILE_BYTES;
  static constexpr int P_OFF = V_OFF + TILE_BYTES;  // P_A, P_B
  static constexpr int BAR_OFF = P_OFF + 2 * P_BYTES;
  static constexpr int SMEM_BYTES = 1024 + BAR_OFF + 256;
  static constexpr int S_COL = 0;     // S_x at x * 128
  static constexpr int O_COL = 256;   // O_x at 256 + x * DH
  static constexpr int TMEM_COLS = 512;
  static_assert(SMEM_BYTES <= 232448, "shared memory budget");
};

struct AttnArgs {
  int B, T, Hq, Hkv, max_seq;
  const int32_t* slot0;  // [B] cache slot of the first new token
  f16* out;              // [B*T][Hq*DH], FP16 operand of the O projection
  float scale_log2;      // log2(e) / sqrt(dh)
  int hpi;               // query heads per work item: 2, or 1 when 2 leave SMs idle
  int* err;
};

}  // namespace

// One work item: sequence b, KV group g, query heads hA (and hA + 1 when
// nq = 2), query rows [t0, t0 + 128).  Items are numbered heaviest first (the
// last query tiles see the most keys).  With one head per item (a.hpi = 1)
// there are twice as many items, each half the work per key tile: for short
// sequences the longest item, not the total, sets the time.
struct AttnItem {
  int b, g, hA, nq, t0, s0, kmax, n_kv, kv_row0;
  bool fresh;  // every key is this call's (slot0 == 0): FP16 operands
};

__device__ __forceinline__ AttnItem attn_item(int it, const AttnArgs& a) {
  const int gs = a.Hq / a.Hkv;
  const int npair = (gs + a.hpi - 1) / a.hpi;
  const int n_qt = (a.T + kQT - 1) / kQT;
  const int per_qt = a.B * a.Hkv * npair;
  AttnItem I;
  const int qt = n_qt - 1 - it / per_qt;
  int u = it % per_qt;
  const int pr = u % npair;
  u /= npair;
  I.g = u % a.Hkv;
  I.b = u / a.Hkv;
  I.hA = I.g * gs + a.hpi * pr;
  I.nq = (a.hpi == 2 && 2 * pr + 1 < gs) ? 2 : 1;
  I.t0 = qt * kQT;
  I.s0 = a.slot0[I.b];
  I.fresh = I.s0 == 0;
  const int q_last = min(I.t0 + kQT, a.T) - 1;  // last valid query row of the tile
  I.kmax = I.s0 + q_last;                       // largest visible key slot
  I.n_kv = I.kmax / kKT + 1;                    // key tiles 0..n_kv-1
  // row of key slot 0 in the K/V view (FP16 copies of this call, or the cache)
  I.kv_row0 = I.fresh ? (I.b * a.Hkv + I.g) * a.T : (I.b * a.Hkv + I.g) * a.max_seq;
  return I;
}

// Persistent: each CTA walks its items (a snake order, see item_of).  The K/V
// ring, the S/P/O hand-offs and the Q buffers carry over from item to item
// (running counters give every barrier phase), so the next item's Q and first
// K tiles load, and its first S is computed, while the softmax warps still
// write the previous item's output.
// Barrier phases are tracked by parity, so no thread may wait on a phase more
// than one ahead of, or two behind, a barrier's current one.  The barriers both
// heads share (Q, K and V full / empty) therefore see every phase from both
// issuers: in an item without head B (the last of an odd-sized group) issuer B
// still waits for each Q, K and V load and makes head B's release arrival.
// The softmax warps only wait on their own head's barriers and on V tiles of
// their own items.
template <int DH>
__global__ void __launch_bounds__(kAttnThreads, 1)
    attn_prefill_kernel(const __grid_constant__ CUtensorMap tmQ,
                        const __grid_constant__ CUtensorMap tmK,
                        const __grid_constant__ CUtensorMap tmV,
                        const __grid_constant__ CUtensorMap tmK16,
                        const __grid_constant__ CUtensorMap tmV16,
                        const __grid_constant__ CUtensorMap tmO, AttnArgs a) {
  pdl_trigger();
  using C = AttnCfg<DH>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* sQ = smem + C::Q_OFF;
  uint8_t* sK = smem + C::K_OFF;
  uint8_t* sV = smem + C::V_OFF;
  uint8_t* sP = smem + C::P_OFF;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::BAR_OFF);
  uint64_t* q_full = bars + 0;
  uint64_t* q_empty = bars + 2;   // the item's S MMAs no longer read Q
  uint64_t* k_full = bars + 3;    // [2]
  uint64_t* k_empty = bars + 5;   // [2]
  uint64_t* v_full = bars + 7;
  uint64_t* v_empty = bars + 8;
  uint64_t* s_full = bars + 9;    // [2] per head: S_x in TMEM
  uint64_t* s_free = bars + 11;   // [2] per head: S_x read into registers
  uint64_t* p_full = bars + 13;   // [2] per head: P_x in shared memory
  uint64_t* o_done = bars + 15;   // [2] per head: O_x += P_x V complete
  uint64_t* o_free = bars + 17;   // [2] per head: the item's O_x has been read out
  uint64_t* mma_idle = bars + 19; // [2] per head
  uint64_t* staged = bars + 21;   // [2] per head: the item's output rows are in P_x
  uint64_t* st_read = bars + 23;  // [2] per head: the output store has read P_x
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 25);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int gs = a.Hq / a.Hkv;
  const int n_items = ((a.T + kQT - 1) / kQT) * a.B * a.Hkv * ((gs + a.hpi - 1) / a.hpi);
  // this CTA's ni-th item (-1: none left).  Snake order over the heaviest-first
  // item list: round r takes items [r G, (r+1) G), CTA k the k-th of them in
  // even rounds and the (G-1-k)-th in odd rounds, which balances the summed
  // work about as well as handing out items dynamically.
  auto item_of = [&](int ni) -> int {
    const int G = (int)gridDim.x, k = (int)blockIdx.x;
    for (int r = 0, seen = 0;; ++r) {
      const int base = r * G;
      if (base >= n_items) return -1;
      const int it = base + ((r & 1) ? G - 1 - k : k);
      if (it < n_items && seen++ == ni) return it;
    }
  };

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    mbar_init(q_empty, 2);   // each head's issuer, present in the item or not
    for (int i = 0; i < kKStages; ++i) {
      mbar_init(&k_full[i], 1);
      mbar_init(&k_empty[i], 2);
    }
    mbar_init(v_full, 1);
    mbar_init(v_empty, 2);
    for (int x = 0; x < 2; ++x) {
      mbar_init(&s_full[x], 1);
      mbar_init(&s_free[x], 128);
      mbar_init(&p_full[x], 128);
      mbar_init(&o_done[x], 1);
      mbar_init(&o_free[x], 128);
      mbar_init(&mma_idle[x], 1);
      mbar_init(&staged[x], 128);
      mbar_init(&st_read[x], 1);
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
  // barrier and TMEM set-up overlap the previous kernel's tail; everything
  // below reads what it wrote (Q, the K/V rows, the slot offsets)
  pdl_wait();

  if (warp == 0) {
    // TMA producer, converged; one elected lane issues.  Per item: Q once the
    // previous item's S MMAs are done with it, then K(0), and per tile j
    // K(j+1) ahead of V(j): S(j+1) is issued early in the softmax of tile j,
    // P(j).V only at its end.
    if (lane == 0) {
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
      tma_prefetch_desc(&tmK16);
      tma_prefetch_desc(&tmV16);
    }
    __syncwarp();
    int nk = 0, nv = 0, nql = 0;  // K, V and Q loads issued
    for (int ni = 0, it = item_of(0); it >= 0; it = item_of(++ni)) {
      const AttnItem I = attn_item(it, a);
      const CUtensorMap* mk = I.fresh ? &tmK16 : &tmK;
      const CUtensorMap* mv = I.fresh ? &tmV16 : &tmV;
      if (ni > 0 && !mbar_wait_w(q_empty, (ni - 1) & 1, abort_flag, a.err)) break;
      mbar_arrive_expect_tx_w(q_full, I.nq * C::TILE_BYTES);
      for (int x = 0; x < I.nq; ++x) {
#pragma unroll
        for (int c = 0; c < DH / 64; ++c)
          tma_load_2d_w(sQ + x * C::TILE_BYTES + c * kQT * 128, &tmQ, q_full, c * 64,
                        (I.b * a.Hq + I.hA + x) * a.T + I.t0);
      }
      ++nql;
      auto load_k = [&](int j) -> bool {
        const int st = nk % kKStages;
        if (!mbar_wait_w(&k_empty[st], ((nk / kKStages) & 1) ^ 1u, abort_flag, a.err))
          return false;
        mbar_arrive_expect_tx_w(&k_full[st], C::TILE_BYTES);
#pragma unroll
        for (int c = 0; c < DH / 64; ++c)
          tma_load_2d_w(sK + st * C::TILE_BYTES + c * kKT * 128, mk, &k_full[st], c * 64,
                        I.kv_row0 + j * kKT);
        ++nk;
        return true;
      };
      auto load_v = [&](int j) -> bool {
        if (!mbar_wait_w(v_empty, (nv & 1) ^ 1u, abort_flag, a.err)) return false;
        mbar_arrive_expect_tx_w(v_full, C::TILE_BYTES);
#pragma unroll
        for (int c = 0; c < DH / 64; ++c)
          tma_load_2d_w(sV + c * kKT * 128, mv, v_full, c * 64, I.kv_row0 + j * kKT);
        ++nv;
        return true;
      };
      bool ok = load_k(0);
      for (int j = 0; ok && j < I.n_kv; ++j) {
        if (j + 1 < I.n_kv && !load_k(j + 1)) ok = false;
        if (ok && !load_v(j)) ok = false;
      }
      if (!ok) break;
    }
    // the CTA does not retire while a copy is still landing (also on abort)
    for (int j = max(0, nk - kKStages); j < nk; ++j)
      mbar_wait_drain(&k_full[j % kKStages], (j / kKStages) & 1, a.err);
    if (nv > 0) mbar_wait_drain(v_full, (nv - 1) & 1, a.err);
    if (nql > 0) mbar_wait_drain(q_full, (nql - 1) & 1, a.err);
  } else if (warp <= 2) {
    const int x = warp - 1;  // head whose MMAs this warp issues
    // descriptors computed once; each MMA adds a constant (start address >> 4
    // stays below 2^14, so the add never carries out of its field)
    const uint64_t dq = smem_desc_sw128(smem_u32(sQ + x * C::TILE_BYTES), 16, 1024);
    const uint64_t dk0 = smem_desc_sw128(smem_u32(sK), 16, 1024);
    const uint64_t dv = smem_desc_sw128(smem_u32(sV), kKT * 128, 1024);
    const uint64_t dp = smem_desc_sw128(smem_u32(sP + x * C::P_BYTES), 16, 1024);
    const uint32_t d_s = tmem + C::S_COL + x * kKT;
    const uint32_t d_o = tmem + C::O_COL + x * DH;
    // kc, vc: this CTA's K and V tiles before the item; c: head x's tiles before
    // the item; hi: items head x took part in
    int kc = 0, vc = 0, c = 0, hi = 0;
    bool ok = true;
    for (int ni = 0, it = item_of(0); ok && it >= 0; it = item_of(++ni)) {
      const AttnItem I = attn_item(it, a);
      if (x >= I.nq) {
        // head absent: observe each shared load and arrive for this head
        ok = mbar_wait_w(q_full, ni & 1, abort_flag, a.err);
        if (ok && lane == 0) mbar_arrive(q_empty);
        for (int j = 0; ok && j < I.n_kv; ++j) {
          const int k1 = kc + j, v1 = vc + j;
          ok = mbar_wait_w(&k_full[k1 % kKStages], (k1 / kKStages) & 1, abort_flag, a.err);
          if (ok && lane == 0) mbar_arrive(&k_empty[k1 % kKStages]);
          if (ok) ok = mbar_wait_w(v_full, v1 & 1, abort_flag, a.err);
          if (ok && lane == 0) mbar_arrive(v_empty);
        }
        __syncwarp();
        kc += I.n_kv;
        vc += I.n_kv;
        continue;
      }
      const uint32_t idesc_s = idesc_f32acc(kQT, kKT, I.fresh);
      const uint32_t idesc_o = idesc_f32acc(kQT, DH, I.fresh, false, /*b_mn_major=*/true);
      auto issue_s = [&](int j) {
        const int kidx = kc + j;
        const uint64_t b0 = dk0 + (uint64_t)((kidx % kKStages) * (C::TILE_BYTES >> 4));
#pragma unroll
        for (int k = 0; k < DH / 16; ++k) {
          // 16 dh columns = 32 B within a 128-B swizzle row; next 64-wide block 16 KB on
          const uint32_t off = ((k >> 2) * (kQT * 128) + (k & 3) * 32) >> 4;
          umma_f16_w(d_s, dq + off, b0 + off, idesc_s, k != 0);
        }
        umma_commit_w(&s_full[x]);
        umma_commit_w(&k_empty[kidx % kKStages]);
        if (j == I.n_kv - 1) umma_commit_w(q_empty);  // the item's last read of Q
      };
      auto issue_pv = [&](int j) {
#pragma unroll
        for (int k = 0; k < kKT / 16; ++k) {
          // A = P rows x keys (K-major, two 64-key swizzle blocks of 16 KB);
          // B = V keys x dh read MN-major: 16 keys = 16 rows of 128 B, next
          // 64-wide dh block 16 KB away (LBO), next 8 keys 1 KB away (SBO)
          const uint32_t pa = ((k >> 2) * (kQT * 128) + (k & 3) * 32) >> 4;
          umma_f16_w(d_o, dp + pa, dv + ((k * 16 * 128) >> 4), idesc_o, (j | k) != 0);
        }
        umma_commit_w(&o_done[x]);
        umma_commit_w(v_empty);
      };
      // S(0): Q and K(0) landed, and the previous item's last S read out of TMEM
      ok = mbar_wait_w(q_full, ni & 1, abort_flag, a.err);
      if (ok) ok = mbar_wait_w(&k_full[kc % kKStages], (kc / kKStages) & 1, abort_flag, a.err);
      if (ok && c > 0) ok = mbar_wait_w(&s_free[x], (c - 1) & 1, abort_flag, a.err);
      if (ok) {
        tc_fence_after();
        issue_s(0);
      }
      for (int j = 0; ok && j < I.n_kv; ++j) {
        if (j + 1 < I.n_kv) {
          const int k1 = kc + j + 1;
          if (!mbar_wait_w(&k_full[k1 % kKStages], (k1 / kKStages) & 1, abort_flag, a.err)) {
            ok = false;
            break;
          }
          // S_x(j+1) overwrites S_x(j): the softmax has it in registers
          if (!mbar_wait_w(&s_free[x], (c + j) & 1, abort_flag, a.err)) {
            ok = false;
            break;
          }
          tc_fence_after();
          issue_s(j + 1);
        }
        if (!mbar_wait_w(v_full, (vc + j) & 1, abort_flag, a.err)) { ok = false; break; }
        if (!mbar_wait_w(&p_full[x], (c + j) & 1, abort_flag, a.err)) { ok = false; break; }
        // the first P.V of an item overwrites O_x: the previous item's output
        // must have been read out
        if (j == 0 && hi > 0 && !mbar_wait_w(&o_free[x], (hi - 1) & 1, abort_flag, a.err)) {
          ok = false;
          break;
        }
        tc_fence_after();
        issue_pv(j);
      }
      kc += I.n_kv;
      vc += I.n_kv;
      c += I.n_kv;
      ++hi;
    }
    // retire only after every issued MMA has completed (also on abort)
    umma_commit_w(&mma_idle[x]);
    mbar_wait_drain(&mma_idle[x], 0, a.err);
  } else {
    // softmax / epilogue warps: head x, row r of each item's query tile
    const int x = (warp - 3) >> 2;
    const int qw = warp & 3;        // TMEM lane quadrant of this warp
    const int r = qw * 32 + lane;   // query row within the tile
    const uint32_t lane_base = static_cast<uint32_t>(qw * 32) << 16;
    const uint32_t s_addr = tmem + lane_base + C::S_COL + x * kKT;
    const uint32_t o_addr = tmem + lane_base + C::O_COL + x * DH;
    uint8_t* prow = sP + x * C::P_BYTES + r * 128;  // this row in P's two swizzle blocks
    int c = 0, vcount = 0;  // head x's S tiles and this CTA's V tiles before the item
    bool ok = true;
    int n_out = 0;  // output tiles of head x staged so far
    const bool issuer = qw == 3 && lane == 0;  // issues head x's output stores
    for (int ni = 0, it = item_of(0); ok && it >= 0; it = item_of(++ni)) {
      const AttnItem I = attn_item(it, a);
      if (x >= I.nq) {
        vcount += I.n_kv;
        continue;
      }
      const int t = I.t0 + r;
      const int s_q = I.s0 + t;         // this row's cache slot
      const int s_row0 = I.s0 + I.t0;   // slot of the tile's first row
      float m_used = -INFINITY, l_sum = 0.f;
      for (int j = 0; ok && j < I.n_kv; ++j) {
        const int cj = c + j;
        if (!mbar_wait(&s_full[x], cj & 1, abort_flag, a.err)) { ok = false; break; }
        tc_fence_after();
        float s[kKT];
        {
          uint32_t raw[kKT];
          tmem_ld128_wait(s_addr, raw);
#pragma unroll
          for (int i = 0; i < kKT; ++i) s[i] = __uint_as_float(raw[i]);
        }
        tc_fence_before();
        mbar_arrive(&s_free[x]);  // S_x(j+1) may now be computed into the same columns
        const int key0 = j * kKT;
        if (key0 + kKT - 1 > s_row0) {
          // a tile that reaches past the first row's slot: causal mask
#pragma unroll
          for (int i = 0; i < kKT; ++i) s[i] = (key0 + i <= s_q) ? s[i] : -INFINITY;
        }
        float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
        for (int i = 0; i < kKT; i += 8) {
#pragma unroll
          for (int q = 0; q < 4; ++q) m4[q] = max3(m4[q], s[i + 2 * q], s[i + 2 * q + 1]);
        }
        const float mx = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3])) * a.scale_log2;
        float alpha = 1.f;
        if (mx > m_used + kRescaleLog2) {
          alpha = ex2(m_used - mx);  // 0 on the first tile (m_used = -inf)
          l_sum *= alpha;
          m_used = mx;
        }
        // P = 2^(s * scale - m), FP32 row sum, rounded to the operand type,
        // stored in the 128-byte swizzle: 16-byte chunk q of row r sits at
        // chunk q ^ (r & 7) of the row's 128-byte line.  Keys 0-63 are packed
        // before the wait for the previous P.V (which still reads the buffer),
        // keys 64-127 are stored as they are computed.  Arguments and sums of
        // two keys at a time go through the packed FP32 FMA and add.
        const float neg_m = -m_used;
        const uint64_t c2 = f32x2(a.scale_log2, a.scale_log2), n2 = f32x2(neg_m, neg_m);
        uint64_t l2 = f32x2(0.f, 0.f);
        auto p8 = [&](int k0, uint32_t (&w)[4]) {
#pragma unroll
          for (int e4 = 0; e4 < 4; ++e4) {
            float x0, x1;
            fma_pair(s[k0 + 2 * e4], s[k0 + 2 * e4 + 1], c2, n2, x0, x1);
            const float p0 = ex2(x0), p1 = ex2(x1);
            asm("add.rn.f32x2 %0, %0, %1;" : "+l"(l2) : "l"(f32x2(p0, p1)));
            w[e4] = pack2(p0, p1, I.fresh);
          }
        };
        uint32_t pk[32];
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          uint32_t w[4];
          p8(8 * q, w);
#pragma unroll
          for (int e4 = 0; e4 < 4; ++e4) pk[4 * q + e4] = w[e4];
        }
        if (j > 0) {
          // O_x += P_x(j-1) V must be done: it reads the P buffer, and O is
          // rescaled below (O_x += P_x(j) V waits for this thread).  At j = 0
          // the previous item's epilogue already waited for its last P.V.
          if (!mbar_wait(&o_done[x], (cj - 1) & 1, abort_flag, a.err)) { ok = false; break; }
          tc_fence_after();
        } else if (n_out > 0) {
          // the previous item's output store reads P_x: wait until it has
          if (issuer) {
            bulk_wait_group_read0();
            mbar_arrive(&st_read[x]);
          }
          if (!mbar_wait(&st_read[x], (n_out - 1) & 1, abort_flag, a.err)) { ok = false; break; }
        }
#pragma unroll
        for (int q = 0; q < 8; ++q)
          *reinterpret_cast<uint4*>(prow + ((q ^ (r & 7)) << 4)) =
              make_uint4(pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          uint32_t w[4];
          p8(64 + 8 * q, w);
          *reinterpret_cast<uint4*>(prow + kQT * 128 + ((q ^ (r & 7)) << 4)) =
              make_uint4(w[0], w[1], w[2], w[3]);
        }
        {
          float lo, hi;
          asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(l2));
          l_sum += lo + hi;
        }
        if (j > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll 1
          for (int q = 0; q < DH / 32; ++q) {
            uint32_t oo[32];
            tmem_ld32_wait(o_addr + 32 * q, oo);
#pragma unroll
            for (int i = 0; i < 32; ++i) oo[i] = __float_as_uint(__uint_as_float(oo[i]) * alpha);
            tmem_st32(o_addr + 32 * q, oo);
          }
          tmem_st_wait();
        }
        if (key0 + kKT - 1 > I.kmax) {
          // keys past the item's last visible slot may hold stale cache
          // contents: zero their V rows so 0 * (non-finite) cannot reach O
          // (both heads' threads write the same zeros; each head's P.V waits
          // for its own)
          if (!mbar_wait(v_full, (vcount + j) & 1, abort_flag, a.err)) { ok = false; break; }
          if (key0 + r > I.kmax) {
#pragma unroll
            for (int q = 0; q < DH / 64; ++q) {
              uint4* vr = reinterpret_cast<uint4*>(sV + q * kKT * 128 + r * 128);
#pragma unroll
              for (int e = 0; e < 8; ++e) vr[e] = make_uint4(0, 0, 0, 0);
            }
          }
        }
        fence_proxy_async_smem();
        tc_fence_before();
        mbar_arrive(&p_full[x]);
      }
      if (!ok) break;
      // epilogue: O / l of this item, then O_x is free for the next item.
      // The last P.V has completed, so P_x's buffer is free: the rows are
      // written there in P's 128-byte-swizzled layout, which is the layout a
      // TMA store of two 64-column boxes reads, and one thread of the head
      // stores the tile asynchronously (rows past the sequence's end are
      // clipped by the tensor map's T extent).
      if (!mbar_wait(&o_done[x], (c + I.n_kv - 1) & 1, abort_flag, a.err)) break;
      tc_fence_after();
      const float inv_l = 1.f / l_sum;
      const uint64_t inv2 = f32x2(inv_l, inv_l);
      bool bad = false;  // C is the next GEMM's FP16 operand: V rows past 65504 reach it
#pragma unroll 1
      for (int h = 0; h < DH / 64; ++h) {  // 64 columns = one swizzle block of the row
        uint32_t oo[64];
        tmem_ld32(o_addr + 64 * h, *reinterpret_cast<uint32_t(*)[32]>(oo));
        tmem_ld32(o_addr + 64 * h + 32, *reinterpret_cast<uint32_t(*)[32]>(oo + 32));
        tmem_ld_wait();
        float f[64];
        float mx = 0.f;
#pragma unroll
        for (int i = 0; i < 64; i += 2) {
          mul_pair(__uint_as_float(oo[i]), __uint_as_float(oo[i + 1]), inv2, f[i], f[i + 1]);
          mx = max3(mx, fabsf(f[i]), fabsf(f[i + 1]));
        }
        // the common case converts plainly; a row that FP16 cannot hold
        // (|o| >= 65520, or NaN) takes the saturating conversion
        const bool sat = !(mx < 65520.f);
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          uint32_t w[4];
          if (sat) {
#pragma unroll
            for (int e = 0; e < 4; ++e) w[e] = pack_f16x2_chk(f[8 * q + 2 * e], f[8 * q + 2 * e + 1], bad);
          } else {
#pragma unroll
            for (int e = 0; e < 4; ++e) w[e] = pack_f16x2(f[8 * q + 2 * e], f[8 * q + 2 * e + 1]);
          }
          *reinterpret_cast<uint4*>(prow + h * (kQT * 128) + ((q ^ (r & 7)) << 4)) =
              make_uint4(w[0], w[1], w[2], w[3]);
        }
      }
      tc_fence_before();
      mbar_arrive(&o_free[x]);  // O_x has been read: the next item's P.V may overwrite it
      record_overflow(a.err, bad);
      fence_proxy_async_smem();  // the staged rows are visible to the TMA store
      mbar_arrive(&staged[x]);
      if (issuer) {
        if (!mbar_wait(&staged[x], n_out & 1, abort_flag, a.err)) break;
#pragma unroll
        for (int h = 0; h < DH / 64; ++h)
          tma_store_3d(&tmO, sP + x * C::P_BYTES + h * (kQT * 128), (I.hA + x) * DH + 64 * h, I.t0,
                       I.b);
        bulk_commit_group();
      }
      ++n_out;
      c += I.n_kv;
      vcount += I.n_kv;
    }
  }

  // the output stores this CTA issued are complete before its shared memory goes
  if (warp >= 3 && (warp & 3) == 3 && lane == 0) bulk_wait_group0();
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

// The attention output [B][T][Hq * dh] FP16 as a 3-D map with boxes of 64
// columns x 128 rows of one sequence, so a tile's rows past T are clipped
// instead of landing in the next sequence.
static bool tmap_out(CUtensorMap* m, const void* base, int B, int T, int width) {
  auto enc = encode_fn();
  if (!enc || (reinterpret_cast<uintptr_t>(base) & 15) || ((width * 2) & 15)) return false;
  cuuint64_t dims[3] = {(cuuint64_t)width, (cuuint64_t)T, (cuuint64_t)B};
  cuuint64_t strides[2] = {(cuuint64_t)width * 2, (cuuint64_t)T * width * 2};
  cuuint32_t box[3] = {64, 128, 1};
  cuuint32_t es[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, const_cast<void*>(base), dims, strides, box,
             es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int DH>
static qwen_status launch_dh(const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v,
                             const CUtensorMap& k16, const CUtensorMap& v16, const CUtensorMap& o,
                             const AttnArgs& a, cudaStream_t st) {
  auto kern = attn_prefill_kernel<DH>;
  static std::atomic<uint64_t> attr{0};  // one bit per device
  if (!smem_attr_once(kern, AttnCfg<DH>::SMEM_BYTES, attr)) return QWEN_ERR_CUDA;
  const int n_qt = (a.T + kQT - 1) / kQT;
  const int npair = (a.Hq / a.Hkv + a.hpi - 1) / a.hpi;
  const long long items = (long long)n_qt * a.B * a.Hkv * npair;
  const int sms = device_sm_count();
  const int grid = items < sms ? (int)items : sms;  // persistent: one CTA per SM
  launch_k(kern, dim3(grid), dim3(kAttnThreads), AttnCfg<DH>::SMEM_BYTES, st, q, k, v, k16, v16,
           o, a);
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
  CUtensorMap to;
  if (!tmap_out(&to, out, B, T, Hq * dh)) return QWEN_ERR_CUDA;
  AttnArgs a;
  a.B = B; a.T = T; a.Hq = Hq; a.Hkv = Hkv; a.max_seq = max_seq;
  a.slot0 = slot0; a.out = out; a.err = err;
  a.scale_log2 = 1.4426950408889634f / sqrtf((float)dh);
  // two heads per item share each K/V tile (half the TMA traffic per MMA
  // cycle); below 1.5 items per SM, one head per item shortens the longest
  // item instead
  {
    const long long pairs = (long long)((T + kQT - 1) / kQT) * B * Hkv * ((Hq / Hkv + 1) / 2);
    a.hpi = pairs * 2 < 3LL * device_sm_count() ? 1 : 2;
  }
  if (dh == 128) return launch_dh<128>(tq, tk, tv, tk16, tv16, to, a, st);
  if (dh == 64) return launch_dh<64>(tq, tk, tv, tk16, tv16, to, a, st);
  return QWEN_ERR_UNSUPPORTED;
}

}  // namespace qwen
