/*
 * CPU oracle for fp32 addmm and groups==1 NCHW conv2d -- TEST INFRASTRUCTURE.
 *
 * Only the test suite, the package smoke check and the benchmark's CPU
 * baseline may load this library.  It shares no code, header or constant with
 * the CUDA path; it is a plain restatement of what the operations compute:
 *
 *   addmm  (ExecuTorch WebGPU "Add optimized addmm op", Solution and
 *           Implementation paragraphs):
 *       out[i,j] = beta * self(i,j) + alpha * sum_k mat1[i,k] * mat2[k,j]
 *       with self(i,j) = self[j] for a [N] self, self[i*N + j] for [M,N].
 *
 *   conv2d (ExecuTorch WebGPU "et_vk conv2d: route standard (groups==1) conv
 *           through an im2col tiled GEMM", Problem / Solution / Implementation):
 *       out[b,oc,oh,ow] = bias[oc] + sum_{ic,kh,kw} w[oc,ic,kh,kw] * x[b,ic,ih,iw]
 *       ih = oh*sH - pH + kh*dH, iw = ow*sW - pW + kw*dW, taps outside the
 *       input contribute nothing (zero padding).
 *
 * All arithmetic is fp64 on fp32 inputs.  Alongside each result the oracle
 * returns S = sum of |product| over the same terms, which scales the
 * per-element error bound |gpu - ref| <= c * S + 1e-6.
 */
#ifndef IMC_ORACLE_H
#define IMC_ORACLE_H
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Return codes. */
#define ORACLE_OK 0
#define ORACLE_EARG (-1)

/* addmm on a subset of output rows.
 *   rows == NULL selects every row 0..M-1 (nrows must then equal M).
 *   ref  : [nrows, N] fp64, row r holds output row rows[r].
 *   sabs : [nrows, N] fp64 (may be NULL) = sum_k |mat1[i,k] * mat2[k,j]|.
 * beta == 0: self is not read (may be NULL).  alpha == 0: mat1 and mat2 are
 * not read and S is 0.  nthreads <= 0 uses every online core. */
int oracle_addmm(const float* self, int self_2d, const float* mat1, const float* mat2,
                 int64_t M, int64_t N, int64_t K, double beta, double alpha,
                 const int64_t* rows, int64_t nrows, int nthreads,
                 double* ref, double* sabs);

/* The same sum taken the way a plain fp32 program would: one fp32 accumulator
 * per output, terms added in k order, then beta*self + alpha*acc in fp32.
 * Used only to show that the error bound is reachable by plain fp32. */
int oracle_addmm_fp32_naive(const float* self, int self_2d, const float* mat1,
                            const float* mat2, int64_t M, int64_t N, int64_t K,
                            float beta, float alpha, float* out);

/* Output spatial size of one axis:
 *   floor((in + 2*pad - dil*(k - 1) - 1) / stride) + 1, or -1 when that is < 1
 *   or an argument is out of range. */
int64_t oracle_conv_out_size(int64_t in, int64_t k, int64_t stride, int64_t pad, int64_t dil);

/* Direct (seven-loop) conv2d on a subset of output channels.
 *   ocs == NULL selects every channel (nocs must then equal OC).
 *   ref  : [B, nocs, OH, OW] fp64; channel c of ref is output channel ocs[c].
 *   sabs : same shape (may be NULL), sum over in-range taps of |w * x|.
 *   bias may be NULL (no bias). */
int oracle_conv2d(const float* x, const float* w, const float* bias,
                  int64_t B, int64_t IC, int64_t H, int64_t W, int64_t OC,
                  int64_t KH, int64_t KW, int64_t sH, int64_t sW, int64_t pH, int64_t pW,
                  int64_t dH, int64_t dW, const int64_t* ocs, int64_t nocs, int nthreads,
                  double* ref, double* sabs);

/* Number of worker threads the oracle would use for nthreads <= 0. */
int oracle_default_threads(void);

#ifdef __cplusplus
}
#endif
#endif
