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
// below.  Every GPU that loads this file's device code holds those
// kNoallocScratchBytes until the process exits.  With CUDA's lazy module
// loading (the default) that load -- and so the reservation of the buffer --
// happens the first time the array is used on a device: the first call of
// this entry point there, which is its set-up.  Host code cannot use the
// array's name as a device address, so every call looks the address up with
// cudaGetSymbolAddress on the current device (after the first call this only
// reads the loaded module's symbol table; it allocates nothing), which also
// keeps the address right if the program resets the device in between.
#include <cmath>

#include "imc.h"
#include "imc_internal.cuh"

namespace imc {
namespace {

constexpr size_t kNoallocScratchBytes = size_t(32) << 20;  // 32 MiB
static_assert(kNoallocScratchBytes == IMC_NOALLOC_SCRATCH_BYTES, "header and library disagree");

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoallocScratchBytes];

// Device address of g_noalloc_scratch on the current device.  IMC_OK or
// IMC_ERR_CUDA.
int scratch_address(void** ptr) {
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) {
    cudaGetLastError();
    return IMC_ERR_CUDA;
  }
  *ptr = p;
  return IMC_OK;
}

}  // namespace
}  // namespace imc

extern "C" int gemm_addmm_f32_noalloc(const float* self, int self_2d, const float* mat1,
                                      const float* mat2, float* out, int64_t M, int64_t N,
                                      int64_t K, double beta, double alpha, int mode,
                                      void* stream) {
  using namespace imc;
  // 1. The argument checks of gemm_addmm_f32_ex, on the host, in its order
  //    (flags, scalars, sizes, pointers, overlaps); no CUDA call.
  const int v = gemm_check_args(self, self_2d, mat1, mat2, out, M, N, K, beta, alpha, mode);
  if (v != IMC_OK) return v;
  // 2. The size check against the fixed buffer, still before any CUDA call.
  //    Nothing in the buffer needs clearing: the mat2 pre-pass writes every
  //    element the main kernel reads, and split-K partial sums are written
  //    in full before they are summed.
  const size_t need = gemm_scratch_needed(mat1, M, N, K, alpha, mode);
  if (need > kNoallocScratchBytes) return IMC_ERR_SCRATCH;
  if (need == 0)  // SIMT, epilogue-only or empty: no scratch involved
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
