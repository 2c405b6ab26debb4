// Host-side launchers shared between the C ABI (api.cu) and the kernel files.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "../../include/qwen_layer.h"

namespace qwen {

// Epilogues of the tensor-core GEMM D = A B^T (A [M,K], B [N,K], K-major).
enum EpiMode : int {
  EPI_STORE = 0,   // out[M,N] bf16 = D
  EPI_RESID = 1,   // out = D + resid (bf16), optional fp32 copy
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
  const int32_t* positions;  // [M]
  const int32_t* slot0;      // [B]: cache slot of the sequence's first new token
  __nv_bfloat16* q_out;    // [B][Hq][T][dh]
  __nv_bfloat16* k_cache;  // [B][Hkv][max_seq][dh]
  __nv_bfloat16* v_cache;
  int T, Hq, Hkv, dh, max_seq, max_position;
  float eps;
};

struct GemmEpilogue {
  int mode;
  __nv_bfloat16* out;  // bf16 output
  int ldo;
  const __nv_bfloat16* resid;  // residual input (EPI_RESID)
  int ldr;
  float* out32;  // fp32 output (EPI_F32, or optional copy in EPI_RESID)
  int ldo32;
  QkvParams qkv;
  // Grouped (expert) mode when group_offsets != nullptr: A rows of group g are
  // [group_offsets[g], group_offsets[g+1]); B holds n_groups stacked [N,K]
  // matrices; output rows are A rows.
  const int32_t* group_offsets;  // [n_groups+1] (device)
  int n_groups;
};

int device_sm_count();
int* lib_status_ptr();  // device status word used by handle-less entry points

// The tensor-core GEMM.  A [M,K] (row stride lda elements), B [N,K] (ldb).
// For grouped mode, B holds n_groups stacked [N,K] matrices and A rows of
// group g live in [group_offsets[g], group_offsets[g+1]).
qwen_status gemm_tc(const __nv_bfloat16* A, int lda, const __nv_bfloat16* B, int ldb, int M,
                    int N, int K, const GemmEpilogue& epi, int* err, cudaStream_t st);

qwen_status rmsnorm_launch(const __nv_bfloat16* x, const __nv_bfloat16* gamma,
                           __nv_bfloat16* y, float* y32, const float* x32, int rows, int d,
                           float eps, cudaStream_t st);

}  // namespace qwen
