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
};

// SIMT fp32 FFMA kernels (any shape, any alignment).
cudaError_t launch_simt_gemm(const GemmArgs& a, cudaStream_t s);
cudaError_t launch_simt_conv(const ConvArgs& a, cudaStream_t s);

// Epilogue-only kernels: out = beta*self (addmm with K == 0 or alpha == 0)
// and out = bias (conv with K == 0).
cudaError_t launch_fill_gemm(const GemmArgs& a, cudaStream_t s);
cudaError_t launch_fill_conv(const ConvArgs& a, cudaStream_t s);

// tcgen05 tensor-core kernels.  three_pass selects 3xTF32 (fp32 accuracy)
// over a single TF32 product.  Return cudaErrorNotSupported when the shape
// does not meet the kernel's requirements (the caller falls back to SIMT).
bool tc_gemm_supported(const GemmArgs& a);
cudaError_t launch_tc_gemm(const GemmArgs& a, bool three_pass, cudaStream_t s);
bool tc_conv_supported(const ConvArgs& a);
cudaError_t launch_tc_conv(const ConvArgs& a, bool three_pass, cudaStream_t s);

// Reads and clears the watchdog word of the tensor-core kernels on the
// current device (synchronises `s` first).
cudaError_t tc_take_watchdog(int* value, cudaStream_t s);

// Number of SMs of the current device (cached per device).
int device_sm_count();

// Counts one kernel launch (for imc_launch_count()).
void note_launch();

}  // namespace imc
