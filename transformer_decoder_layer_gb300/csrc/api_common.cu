// C ABI: status strings, device queries and the handle-less entry points
// (qwen_rmsnorm, qwen_linear).
#include <atomic>
#include <cstdio>
#include <cstdlib>
#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace qwen {

static std::atomic<unsigned long long> g_launches{0};

void count_launches(int n) { g_launches.fetch_add((unsigned long long)n, std::memory_order_relaxed); }

// Status word for entry points that have no layer handle (qwen_linear, ...).
// A module-scope device variable: no allocation is needed to use it.  Each
// device has its own copy; host code looks its address up per device.
static __device__ int g_lib_status;

int current_device() {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return -1;
  return dev;
}

int* lib_status_ptr() {
  static std::mutex mu;
  static int* addr[kMaxDevices] = {};
  const int dev = current_device();
  if (dev < 0) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  if (!addr[dev]) {
    void* a = nullptr;
    if (cudaGetSymbolAddress(&a, g_lib_status) == cudaSuccess) addr[dev] = static_cast<int*>(a);
  }
  return addr[dev];
}

bool pdl_enabled() {
  static int v = -1;
  if (v < 0) {
    const char* e = getenv("QWEN_PDL");
    v = (e && e[0] == '0') ? 0 : 1;
  }
  return v == 1;
}

int device_sm_count() {
  static std::atomic<int> cached[kMaxDevices] = {};
  const int dev = current_device();
  if (dev < 0) return 1;
  int n = cached[dev].load(std::memory_order_relaxed);
  if (!n) {
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
      return 1;
    cached[dev].store(n, std::memory_order_relaxed);
  }
  return n;
}

}  // namespace qwen

using namespace qwen;

extern "C" {

const char* qwen_status_string(qwen_status s) {
  switch (s) {
    case QWEN_OK: return "ok";
    case QWEN_ERR_INVALID_ARG: return "invalid argument";
    case QWEN_ERR_UNSUPPORTED: return "unsupported shape or option";
    case QWEN_ERR_CAPACITY: return "capacity exceeded";
    case QWEN_ERR_CUDA: return "CUDA error";
    case QWEN_ERR_TIMEOUT: return "device wait timed out";
    case QWEN_ERR_RANGE: return "cache slot or position out of range";
    case QWEN_ERR_OVERFLOW: return "value beyond the FP16 operand range (|x| > 65504)";
  }
  return "unknown status";
}

int32_t qwen_device_sm_count(void) { return device_sm_count(); }

uint64_t qwen_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

qwen_status qwen_rmsnorm(const void* x, const void* gamma, void* y, float* y_fp32, int32_t rows,
                         int32_t d, float eps, void* stream) {
  if (rows < 0 || d <= 0) return QWEN_ERR_INVALID_ARG;
  if (rows == 0) return QWEN_OK;
  if (!x || !gamma || !y) return QWEN_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(y) |
       reinterpret_cast<uintptr_t>(gamma)) & 15)
    return QWEN_ERR_INVALID_ARG;
  return rmsnorm_launch(static_cast<const bf16*>(x), static_cast<const bf16*>(gamma), y,
                        /*y_f16=*/false, y_fp32, nullptr, rows, d, eps,
                        static_cast<cudaStream_t>(stream));
}

qwen_status qwen_linear(const void* x, const void* w, void* y, int32_t M, int32_t N, int32_t K,
                        void* stream) {
  if (M < 0 || N <= 0 || K <= 0) return QWEN_ERR_INVALID_ARG;
  if (M == 0) return QWEN_OK;
  if (!x || !w || !y) return QWEN_ERR_INVALID_ARG;
  if ((K & 7) || (N & 7)) return QWEN_ERR_UNSUPPORTED;
  GemmEpilogue epi{};
  epi.mode = EPI_STORE;
  epi.out = y;
  epi.ldo = N;
  return gemm_tc(x, K, w, K, M, N, K, /*op_f16=*/false, epi, lib_status_ptr(),
                 static_cast<cudaStream_t>(stream));
}

qwen_status qwen_poll_error(void* stream) {
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return QWEN_ERR_CUDA;
  int* p = lib_status_ptr();
  if (!p) return QWEN_ERR_CUDA;
  int v = 0;
  if (cudaMemcpy(&v, p, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return QWEN_ERR_CUDA;
  if (v) {
    const int zero = 0;
    cudaMemcpy(p, &zero, sizeof(int), cudaMemcpyHostToDevice);
  }
  return static_cast<qwen_status>(v);
}

}  // extern "C"
