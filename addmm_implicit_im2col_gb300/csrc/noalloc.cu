// gemm_addmm_f32_noalloc: the tensor-core addmm for callers that cannot
// allocate device memory while they run.
//
// Who needs it: a program whose device memory is fixed when it starts -- a
// real-time or embedded runtime with a set memory budget, or an operator
// inside a host framework that forbids allocation in its compute callback.
// For those callers an allocation on the call path is not an option: it can
// block behind other work on the device, and it can fail under memory
// pressure in the middle of a run.  The other addmm entry points either take
// scratch from the device's memory pool or from the caller; this one uses a
// buffer that is part of the library image instead.
//
// The scratch (mat2 transposed and split into TF32 hi / lo parts, the same
// data the pool-backed path builds) lives in the file-scope device array
// below.  Every GPU that loads the library holds those kNoallocScratchBytes
// until the process exits.  Host code cannot use the array's name as a device
// address, so the first call on each device looks the address up with
// cudaGetSymbolAddress (with that device current) and caches it.
#include <cmath>
#include <mutex>

#include "imc.h"
#include "imc_internal.cuh"

namespace imc {
namespace {

constexpr size_t kNoallocScratchBytes = size_t(32) << 20;  // 32 MiB
static_assert(kNoallocScratchBytes == IMC_NOALLOC_SCRATCH_BYTES, "header and library disagree");

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoallocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_ptr[kMaxDevices];

// Device address of g_noalloc_scratch on the current device (set-up on the
// first call per device).  IMC_OK, IMC_ERR_DEVICE or IMC_ERR_CUDA.
int scratch_address(void** ptr) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return IMC_ERR_DEVICE;
  }
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) {
      cudaGetLastError();
      return IMC_ERR_CUDA;
    }
    g_scratch_ptr[dev] = p;
  }
  *ptr = g_scratch_ptr[dev];
  return IMC_OK;
}

}  // namespace
}  // namespace imc

extern "C" int gemm_addmm_f32_noalloc(const float* self, int self_2d, const float* mat1,
                                      const float* mat2, float* out, int64_t M, int64_t N,
                                      int64_t K, double beta, double alpha, int mode,
                                      void* stream) {
  using namespace imc;
  // Size check first, so that an oversized problem is rejected before any
  // CUDA call.  Nothing in the buffer needs clearing: the mat2 pre-pass
  // writes every element the main kernel reads.
  const size_t need = gemm_scratch_needed(mat1, M, N, K, alpha, mode);
  if (need > kNoallocScratchBytes) return IMC_ERR_SCRATCH;
  // The argument errors gemm_addmm_f32_ex reports before touching the device
  // come first here too (the scratch set-up below needs the device).
  if (need > 0) {
    if (self_2d != 0 && self_2d != 1) return IMC_ERR_ARG;
    if (!std::isfinite(beta) || !std::isfinite(alpha)) return IMC_ERR_ARG;
    if (!out || !mat1 || !mat2 || (beta != 0.0 && !self)) return IMC_ERR_NULL;
  }
  if (need == 0)  // SIMT, epilogue-only or invalid arguments: no scratch involved
    return gemm_with_scratch(self, self_2d, mat1, mat2, out, M, N, K, beta, alpha, mode, nullptr,
                             0, stream);
  const int dev = require_device();
  if (dev != IMC_OK) return dev;
  void* scratch = nullptr;
  const int rc = scratch_address(&scratch);
  if (rc != IMC_OK) return rc;
  return gemm_with_scratch(self, self_2d, mat1, mat2, out, M, N, K, beta, alpha, mode, scratch,
                           kNoallocScratchBytes, stream);
}
