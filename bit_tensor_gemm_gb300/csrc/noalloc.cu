// noalloc.cu -- lbgemm_run_static: the GEMM with its re-encoding scratch in a
// fixed array compiled into the library, for callers that cannot allocate
// GPU memory and cannot provide a workspace either.  Nothing here allocates:
// the array exists once per device for the life of the process.
#include <cuda_runtime.h>

#include <cstdio>
#include <mutex>

#include "lbgemm.h"

namespace lbg {
lbgemm_status report_error(lbgemm_status st, const char* message);
lbgemm_status scratch_for_call(int bits, int64_t M, int64_t N, int64_t K, const void* A,
                               const void* B, const void* C, int variant, size_t* bytes);
}

namespace {

constexpr size_t kStaticScratchBytes = LBGEMM_STATIC_SCRATCH_BYTES;
constexpr int kMaxDevices = 64;

// The scratch.  In host code this name is only a stand-in for the symbol;
// its device address comes from cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

std::mutex g_mu;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of the array on the current device, looked up once per device.
lbgemm_status scratch_address(void** out) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess || dev < 0 || dev >= kMaxDevices)
    return lbg::report_error(LBGEMM_ERR_CUDA, "lbgemm_run_static: no usable current device");
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_static_scratch);
    if (e != cudaSuccess || !p) {
      char msg[256];
      snprintf(msg, sizeof msg, "lbgemm_run_static: cudaGetSymbolAddress failed: %s",
               cudaGetErrorString(e));
      return lbg::report_error(LBGEMM_ERR_CUDA, msg);
    }
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return LBGEMM_OK;
}

}  // namespace

extern "C" lbgemm_status lbgemm_run_static(int bits, int64_t M, int64_t N, int64_t K,
                                           const void* A, const void* B, int32_t* C, int variant,
                                           void* stream) {
  // the scratch of the route this call takes: both re-encoded operands on the
  // tensor-core route, one on the in-kernel conversion route, none on the
  // routes that read int8 directly
  size_t need = 0;
  lbgemm_status st = lbg::scratch_for_call(bits, M, N, K, A, B, C, variant, &need);
  if (st != LBGEMM_OK) return st;
  if (need > kStaticScratchBytes) {
    char msg[256];
    snprintf(msg, sizeof msg,
             "lbgemm_run_static: this problem needs %zu bytes of scratch, more than the %zu-byte "
             "static array; use lbgemm_run or lbgemm_run_ws",
             need, kStaticScratchBytes);
    return lbg::report_error(LBGEMM_ERR_WORKSPACE, msg);
  }
  if (M == 0 || N == 0) return LBGEMM_OK;
  void* scratch = nullptr;
  st = scratch_address(&scratch);
  if (st != LBGEMM_OK) return st;
  return lbgemm_run_ws(bits, M, N, K, A, B, C, variant, scratch, kStaticScratchBytes, stream);
}
