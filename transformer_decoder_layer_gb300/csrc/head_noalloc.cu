// qwen_head_last_token_noalloc: the last-token head (final RMSNorm + lm_head)
// for callers that cannot allocate device memory at call time.
//
// Who needs it: a serving process that hands all of its HBM to a fixed arena
// up front (weights, KV cache, activations) has no room left to carve a
// per-call workspace, and a host loop that must not trigger an allocation
// (which can synchronise the device and stall every other stream) cannot ask
// for one either.  qwen_head_last_token needs a caller workspace for the
// normalised last-position rows; this variant keeps those rows in a fixed
// device array that lives inside the library instead.
//
// The array is a file-scope __device__ variable: every GPU that loads the
// library holds its kQwenHeadScratchBytes until the process exits.  Host code
// must not use the symbol's name as an address, so the device address is
// looked up once per device with cudaGetSymbolAddress, on the first call made
// with that device current (that first call should therefore come before any
// stream capture).  The looked-up address is kept for the life of the process:
// a cudaDeviceReset between calls would reload the module and leave it stale,
// so the caller must not reset the device while using this entry point.  The
// GEMM's device status word (read by qwen_poll_error) is looked up per device
// the same way.  All calls share the one array and it keeps the last call's
// contents; every call overwrites the part it uses before reading it, so no
// clearing is needed.  Calls that overlap on the GPU (different streams, or
// different threads without ordering) race on the array.
#include <mutex>

#include "common.cuh"
#include "internal.h"
#include "layer.h"

namespace qwen {

constexpr size_t kQwenHeadScratchBytes = (size_t)2 << 20;  // 2 MiB: B * d * 2 bytes at most

static __device__ __align__(256) uint8_t g_head_scratch[kQwenHeadScratchBytes];

// Device address of g_head_scratch for the current device (set up once per
// device), or nullptr if the lookup fails.
static void* head_scratch_address() {
  static std::mutex mu;
  static void* addr[kMaxDevices] = {};
  const int dev = current_device();
  if (dev < 0) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  if (!addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_head_scratch) != cudaSuccess) return nullptr;
    addr[dev] = p;
  }
  return addr[dev];
}

}  // namespace qwen

using namespace qwen;

extern "C" {

qwen_status qwen_head_last_token_noalloc(const void* y, int32_t B, int32_t T, int32_t d,
                                         const void* gamma_final, const void* w_lm, int32_t V,
                                         float eps, float* logits, void* stream) {
  if (B < 0 || T <= 0 || d <= 0 || V <= 0) return QWEN_ERR_INVALID_ARG;
  if (B == 0) return QWEN_OK;
  if (!y || !gamma_final || !w_lm || !logits) return QWEN_ERR_INVALID_ARG;
  if ((d & 63) || d > 8192 || (V & 7)) return QWEN_ERR_UNSUPPORTED;
  if (B > 256) return QWEN_ERR_CAPACITY;
  if ((size_t)B * (size_t)d * 2 > kQwenHeadScratchBytes) return QWEN_ERR_CAPACITY;
  void* scratch = head_scratch_address();
  int* status = lib_status_ptr();
  if (!scratch || !status) return QWEN_ERR_CUDA;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  bf16* xn = static_cast<bf16*>(scratch);
  const bf16* last = static_cast<const bf16*>(y) + (size_t)(T - 1) * d;
  qwen_status s = rmsnorm_launch(last, static_cast<const bf16*>(gamma_final), xn, false, nullptr,
                                 nullptr, B, d, eps, st, (size_t)T * d);
  if (s) return s;
  // one K split: the decode GEMM writes its [B][V] FP32 result straight into
  // the logits, so no partial buffer is needed
  return gemm_decode_splitk(w_lm, xn, d, B, V, d, 1, /*op_f16=*/false, logits, status, st);
}

}  // extern "C"
