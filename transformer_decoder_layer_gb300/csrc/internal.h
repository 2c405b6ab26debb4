// Host-side launchers shared between the C ABI (api.cu) and the kernel files.
#pragma once

#include <atomic>

#include <cstddef>
#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "../../include/qwen_layer.h"

namespace qwen {

// Epilogues of the tensor-core GEMM D = A B^T (A [M,K], B [N,K], K-major).
enum EpiMode : int {
  EPI_STORE = 0,   // out[M,N] bf16 = D
  EPI_RESID = 1,   // D + residual (bf16 or fp32): bf16 out and/or fp32 out32
  EPI_SWIGLU = 2,  // B rows interleaved gate/up in 64-row blocks: out[M,N/2] = SiLU(g)*u
  EPI_QKV = 3,     // bias, QK-norm, RoPE, Q store + K/V cache append
  EPI_F32 = 4,     // out32[M,N] fp32 = D
};

// Everything the QKV epilogue needs (shared by the prefill GEMM epilogue and
// the decode reduce kernel).
struct QkvParams {
  const float* bias;       // [Nq+2Nkv] fp32 or nullptr
  const __nv_bfloat16* gamma_q;   // [dh] or nullptr (no QK-norm)
  const __nv_bfloat16* gamma_k;   // [dh]
  const float2* rope;      // [max_position][dh/2] (cos, sin)
  const float2* rope_t;    // the same, frequency-major [dh/2][max_position]
  const int32_t* positions;  // [M]
  const int32_t* slot0;      // [B]: cache slot of the sequence's first new token
  void* q_out;             // [B][Hq][T][dh], BF16, or with q_f16 FP16 for the
  int q_f16;               // sequences with slot0[b] == 0 (BF16 for the others)
  __nv_bfloat16* k_cache;  // [B][Hkv][max_seq][dh]
  __nv_bfloat16* v_cache;
  __half* k16;             // optional FP16 copies of this call's K/V rows,
  __half* v16;             // [B][Hkv][T][dh] (prefill attention reads them)
  int T, Hq, Hkv, dh, max_seq, max_position;
  float eps;
};

struct GemmEpilogue {
  int mode;
  void* out;    // 16-bit output (BF16, or FP16 when out_f16)
  int out_f16;
  int ldo;
  const __nv_bfloat16* resid;  // residual input (EPI_RESID), BF16 ...
  const float* resid32;        // ... or FP32 (takes precedence when set)
  int ldr;
  float* out32;  // fp32 output (EPI_F32, or optional copy in EPI_RESID)
  int ldo32;
  QkvParams qkv;
  // Grouped (expert) mode when group_offsets != nullptr: A rows of group g are
  // [group_offsets[g], group_offsets[g+1]); B holds n_groups stacked [N,K]
  // matrices; output rows are A rows.
  const int32_t* group_offsets;  // [n_groups+1] (device)
  int n_groups;
  // B is never written by the kernel launched just before this one (packed
  // layer weights): its first tiles may be fetched before waiting on it.
  int b_static;
  // B is a packed layer weight in the blocked layout (128 x 64 tiles, each
  // group's rows padded to a multiple of 128); else row-major with row stride ldb.
  int b_blocked;
  // Set by gemm_tc (dense mode): tiles from split_from on are 128 wide.
  int split_tail, split_from;
};

// Devices the library tells apart (per-device set-up below).
constexpr int kMaxDevices = 64;
// The current device, or -1 if it cannot be read or is kMaxDevices or above.
int current_device();
// SM count of the current device (cached per device; 1 if it cannot be read).
int device_sm_count();

// Raise a kernel's dynamic shared memory limit on the current device, once
// per device: `done` holds one bit per device.  False on failure.
template <typename Kern>
bool smem_attr_once(Kern kern, int bytes, std::atomic<uint64_t>& done) {
  const int dev = current_device();
  if (dev < 0) return false;
  const uint64_t bit = 1ull << dev;
  if (done.load(std::memory_order_acquire) & bit) return true;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) !=
      cudaSuccess)
    return false;
  done.fetch_or(bit, std::memory_order_release);
  return true;
}

// Whether kernels are launched with programmatic dependent launch (default on;
// QWEN_PDL=0 in the environment turns it off).
bool pdl_enabled();

// Launch `kern` on `st`, with programmatic stream serialisation when enabled.
// Every kernel launched this way calls pdl_wait() before using memory that
// earlier kernels touch.
template <typename... KArgs, typename... Args>
cudaError_t launch_k(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                     Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl_enabled() ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, static_cast<KArgs>(args)...);
}
// Host-side count of kernel launches issued by the library (qwen_launch_count).
void count_launches(int n = 1);
// Device status word used by handle-less entry points, on the current device
// (its address is looked up once per device); nullptr if the lookup fails.
int* lib_status_ptr();

// The tensor-core GEMM.  A [M,K] (row stride lda elements), B [N,K] (ldb),
// both BF16 or both FP16 (op_f16).  For grouped mode, B holds n_groups stacked
// [N,K] matrices and A rows of group g live in [group_offsets[g],
// group_offsets[g+1]).
qwen_status gemm_tc(const void* A, int lda, const void* B, int ldb, int M, int N, int K,
                    bool op_f16, const GemmEpilogue& epi, int* err, cudaStream_t st);

// Causal GQA flash attention for prefill: q [B][Hq][T][dh], caches
// [B][Hkv][max_seq][dh], out [B*T][Hq*dh]; query t of sequence b sits in cache
// slot slot0[b] + t and sees slots <= its own.
// q and the fresh K/V copies (k16/v16: this call's T rows per (b, KV head)) are
// FP16; key tiles that reach below slot0[b] are read from the BF16 cache.
qwen_status attention_prefill(const __half* q, const __nv_bfloat16* k_cache,
                              const __nv_bfloat16* v_cache, const __half* k16,
                              const __half* v16, const int32_t* slot0,
                              __half* out, int B, int T, int Hq, int Hkv, int dh,
                              int max_seq, int* err, cudaStream_t st);

// y[r] = gamma * x[r] / sqrt(mean(x[r]^2) + eps); input rows `x_stride`
// elements apart (0 = d), read from x32 (FP32) when given, else x (BF16);
// y is BF16, or FP16 when y_f16, rows `y_stride` apart (0 = d).  With y_lo
// (FP16 y only) the rounding residual y - fp16(y) is written there as FP16, rows
// `y_stride` apart: y + y_lo carries the FP32 value to about 2^-22.  An FP16
// value beyond the format's range is stored saturated and QWEN_ERR_OVERFLOW is
// recorded in *err (when err is not NULL).
qwen_status rmsnorm_launch(const __nv_bfloat16* x, const __nv_bfloat16* gamma, void* y,
                           bool y_f16, float* y32, const float* x32, int rows, int d, float eps,
                           cudaStream_t st, size_t x_stride = 0, size_t y_stride = 0,
                           __half* y_lo = nullptr, int* err = nullptr);

}  // namespace qwen
