// Internal declarations shared by the host dispatch and the kernel files of
// libimc.  Not part of the public ABI (include/imc.h).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace imc {

// One addmm problem after validation: out = beta*self + alpha*(mat1 @ mat2).
struct GemmArgs {
  const float* self;  // [N] or [M,N]; only read when read_self
  const float* mat1;  // [M,K]
  const float* mat2;  // [K,N]
  float* out;         // [M,N]
  int64_t M, N, K;
  float alpha, beta;
  int self_2d;        // 1: self is [M,N]
  int read_self;      // beta != 0
  int vec_out;        // out (and self) allow 16-byte vector access: N % 4 == 0, aligned
  int relu;           // apply max(v, 0) to every output
  int b_kmajor;       // mat2 is given transposed, [N,K] (aten.linear weight)
};

// One conv2d problem after validation, already viewed as the GEMM
// M = OC, N = B*OH*OW, K = IC*KH*KW.
struct ConvArgs {
  const float* x;     // [B,IC,H,W]
  const float* w;     // [OC,IC,KH,KW] == [OC, K]
  const float* bias;  // [OC] or nullptr
  float* out;         // [B,OC,OH,OW]
  int B, IC, H, W, OC, KH, KW;
  int sH, sW, pH, pW, dH, dW;
  int OH, OW;
  int64_t M, N, K;
  int vec_out;        // OH*OW % 4 == 0 and out 16-byte aligned
  int relu;           // apply max(v, 0) to every output
};

// SIMT fp32 FFMA kernels (any shape, any alignment).
cudaError_t launch_simt_gemm(const GemmArgs& a, cudaStream_t s);
cudaError_t launch_simt_conv(const ConvArgs& a, cudaStream_t s);

// Epilogue-only kernels: out = beta*self (addmm with K == 0 or alpha == 0)
// and out = bias (conv with K == 0).
cudaError_t launch_fill_gemm(const GemmArgs& a, cudaStream_t s);
cudaError_t launch_fill_conv(const ConvArgs& a, cudaStream_t s);

// Direct conv2d: one thread per output element, receptive field read from
// global memory for every output (the design the implicit GEMM replaces).
cudaError_t launch_direct_conv(const ConvArgs& a, cudaStream_t s);

// tcgen05 tensor-core kernels.  three_pass selects 3xTF32 (fp32 accuracy)
// over a single TF32 product.  Return cudaErrorNotSupported when the shape
// does not meet the kernel's requirements (the caller falls back to SIMT).
// The addmm kernel needs a 16-byte aligned workspace for the transposed mat2,
// a copy of mat1 with 16-byte aligned rows when its rows are not (pad_a:
// K % 4 != 0 or an unaligned mat1; pad_b likewise for a K-major linear
// weight) and, for problems with few output tiles, split-K partial sums; it
// is dead once the launch completes.  tc_gemm_workspace_bytes(.., limit) is
// the size of the best plan whose scratch fits in `limit` bytes: SIZE_MAX
// gives the preferred size, 0 the minimum (no split-K); launch_tc_gemm plans
// within the workspace it is given.
bool tc_gemm_supported(const GemmArgs& a);
bool tc_gemm_pad_a(const GemmArgs& a);
bool tc_gemm_pad_b(const GemmArgs& a);
size_t tc_gemm_workspace_bytes(int64_t M, int64_t N, int64_t K, bool three_pass, bool b_kmajor,
                               bool pad_a, bool pad_b, size_t limit);
cudaError_t launch_tc_gemm(const GemmArgs& a, bool three_pass, void* workspace,
                           size_t workspace_bytes, cudaStream_t s);
// The conv kernel needs a 16-byte aligned workspace for the padded hi / lo
// weight planes and, when the last wave of tiles is cut into K-slices, their
// partial sums; tc_conv_workspace_bytes(.., limit) follows the same rule as
// the addmm one (SIZE_MAX: preferred size, 0: minimum, no slices).
// tc_conv_shape_ok: the sizes the kernel's 32-bit indexing and tap table
// take (pointers may be null); tc_conv_supported adds the driver check.
bool tc_conv_shape_ok(const ConvArgs& a);
bool tc_conv_supported(const ConvArgs& a);
size_t tc_conv_workspace_bytes(const ConvArgs& a, bool three_pass, size_t limit);
cudaError_t launch_tc_conv(const ConvArgs& a, bool three_pass, void* workspace,
                           size_t workspace_bytes, cudaStream_t s);

// Read and clear the watchdog word of the addmm / conv tensor-core kernels on
// the current device (the caller synchronises first).
cudaError_t gemm_take_watchdog(int* value);
// A one-thread kernel whose barrier wait gives up after limit_us (addmm
// watchdog word).
cudaError_t launch_wait_selftest(int limit_us, cudaStream_t s);
cudaError_t conv_take_watchdog(int* value);

// Used by the fixed-scratch addmm entry point: the argument checks of
// gemm_addmm_f32_ex alone (host only, no CUDA call; IMC_OK or its status),
// the scratch bytes the call with these arguments would use (0 when no
// tensor-core kernel runs), the addmm itself on a caller-held scratch
// buffer, and the device check.
int gemm_check_args(const float* self, int self_2d, const float* mat1, const float* mat2,
                    float* out, int64_t M, int64_t N, int64_t K, double beta, double alpha,
                    int mode);
size_t gemm_scratch_needed(const float* mat1, int64_t M, int64_t N, int64_t K, double alpha,
                           int mode);
int gemm_with_scratch(const float* self, int self_2d, const float* mat1, const float* mat2,
                      float* out, int64_t M, int64_t N, int64_t K, double beta, double alpha,
                      int mode, void* scratch, size_t scratch_bytes, void* stream);
int require_device();

// Number of SMs of the current device (cached per device).
int device_sm_count();

// Counts one kernel launch (for imc_launch_count()).
void note_launch();
// Names the main kernel of the call in progress (imc_last_kernel_name()
// reports it once the call succeeds); a static string.
void note_kernel_name(const char* name);

// Launches `kernel` as the programmatic dependent of the previous kernel of
// the stream: it may start once that kernel's blocks have all executed
// griddepcontrol.launch_dependents, while that kernel is still running, and
// calls ptx::griddep_wait() before any global access that kernel could
// conflict with.  Every compute kernel of the library is launched this way.  A
// pre-pass waits at its first instruction and only then lets its own dependent
// (the call's main kernel) launch, so that a main kernel that follows its
// pre-pass may read the call's inputs from its start; a main kernel that
// begins a call (no pre-pass) has every global access after its wait.
template <typename... KArgs, typename... Args>
cudaError_t launch_after_previous(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                                  cudaStream_t s, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr.val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}

}  // namespace imc
