/*
 * imc.h -- C ABI of libimc: fp32 addmm and groups==1 NCHW conv2d, both run as
 * one tiled GEMM with a fused epilogue on NVIDIA sm_103a (GB300).
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - All tensor pointers are DEVICE pointers to contiguous row-major fp32
 *    data owned by the caller.  The library never frees or keeps a pointer to
 *    them beyond the call; it may cache CUDA function attributes per device.
 *  - Device memory: the tensor-core kernels need scratch -- addmm a copy of
 *    mat2 transposed and split into TF32 hi / lo parts, conv2d the weight
 *    split the same way in zero-padded rows.  The *_ws entry points take it
 *    from the caller and allocate nothing; the others take it from the
 *    library's own stream-ordered memory pool on the current device
 *    (cudaMallocFromPoolAsync / cudaFreeAsync on `stream`).  The scratch is
 *    dead once the call's work completes.  The pool keeps the memory it has
 *    handed out for later calls until imc_release_memory(), and gives a block
 *    freed on one stream to another stream only once that free has completed
 *    (calls on different streams never wait for each other through it).
 *  - `stream` is a cudaStream_t (NULL = the legacy default stream).  Work is
 *    enqueued asynchronously on it; no entry point synchronises the host.
 *  - Every kernel is launched as the programmatic dependent of the kernel
 *    before it on `stream` (cudaLaunchAttributeProgrammaticStreamSerialization)
 *    and executes griddepcontrol.wait before any global access that kernel
 *    could conflict with, so stream order holds exactly as for plain launches,
 *    also after a caller's kernel that releases its dependents early; a call
 *    that follows another library call on the same stream starts sooner.  The
 *    conv kernels release the stream's next kernel once their last loads are
 *    out: a caller's kernel launched as a programmatic dependent after a conv
 *    call must execute griddepcontrol.wait before it reads the conv's output
 *    (as every programmatic dependent must); plain launches are unaffected.
 *  - The *_ws entry points enqueue only kernels on `stream` (no allocation,
 *    no host synchronisation), so they can be captured into a CUDA graph and
 *    replayed on new data written into the same buffers; make one call on the
 *    device before the capture (it sets per-device kernel attributes).
 *  - Host threads may call the entry points at the same time (the library's
 *    per-device state is set up once, under locks or atomics); calls whose
 *    buffers overlap must still be ordered by the caller's streams.
 *  - Every argument is checked before anything is launched.  A call that
 *    returns an error has enqueued nothing and written nothing.
 *  - Return value: IMC_OK (0) or one of the negative IMC_ERR_* codes below;
 *    imc_status_string() names them.  IMC_ERR_CUDA means a CUDA runtime call
 *    failed (for example a launch error); the CUDA error is left for the
 *    caller to read with cudaGetLastError().
 *  - Arithmetic is fp32 in and out.  The default mode (IMC_MODE_DEFAULT)
 *    keeps fp32 accuracy: each product is split into TF32 pieces
 *    (3xTF32) on the tensor cores, or computed with fp32 FMA on the SIMT
 *    fallback.  IMC_MODE_TF32 is an explicitly requested faster mode with
 *    single TF32 products (about 3 fewer decimal digits): the tensor core
 *    truncates both operands to TF32, so a product may be off by up to
 *    ~1.95e-3 of its magnitude (the error of out[i,j] is then bounded by
 *    about 1.95e-3 * |alpha| * sum_k |mat1[i,k] * mat2[k,j]|).
 *  - Non-finite inputs: the SIMT kernels follow IEEE arithmetic.  On the
 *    tensor cores an output whose exact value is NaN comes out non-finite
 *    (the tensor core reads a NaN whose payload lies only in the 13 low
 *    mantissa bits as an infinity), an output whose exact value is +inf or
 *    -inf comes out as that infinity -- or as NaN in the 3xTF32 mode, whose
 *    cross products can multiply an infinity by a zero low part -- and
 *    outputs no non-finite input reaches are unaffected.
 */
#ifndef IMC_H
#define IMC_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ------------------------------------------------------------ status codes */
#define IMC_OK 0
#define IMC_ERR_NULL (-1)    /* a required pointer is NULL                       */
#define IMC_ERR_SHAPE (-2)   /* a size is negative / out of range, empty output  */
#define IMC_ERR_ARG (-3)     /* bad flag or mode value, non-finite alpha / beta  */
#define IMC_ERR_ALIAS (-4)   /* the output overlaps an input it may not overlap   */
#define IMC_ERR_CUDA (-5)    /* a CUDA runtime call or kernel launch failed       */
#define IMC_ERR_TIMEOUT (-6) /* a kernel gave up waiting on one of its barriers   */
#define IMC_ERR_DEVICE (-7)  /* no usable device of compute capability 10.3       */
#define IMC_ERR_SCRATCH (-8) /* needs more than gemm_addmm_f32_noalloc's buffer  */

/* ------------------------------------------------------------------- modes */
#define IMC_MODE_DEFAULT 0 /* fp32-accurate: 3xTF32 tensor cores, SIMT when needed */
#define IMC_MODE_TF32 1    /* explicit 1xTF32 fast mode (SIMT when the shape needs) */
#define IMC_MODE_SIMT 2    /* force the fp32 FFMA SIMT kernel                       */
#define IMC_MODE_FORCE_TC3 3 /* force the tcgen05 3xTF32 kernel (IMC_ERR_SHAPE if the
                                shape cannot take it); for tests and measurement    */
#define IMC_MODE_FORCE_TC1 4 /* force the tcgen05 1xTF32 kernel, likewise          */
#define IMC_MODE_DIRECT 5    /* conv2d only: the direct kernel (one thread per output
                                element, no operand reuse) -- the pre-GEMM design the
                                conv page replaces, kept as a measured baseline       */
/* Flag OR-ed into any mode: apply max(v, 0) to every output element in the
 * fused epilogue (the ReLU of a Linear / Conv + ReLU block, ExecuTorch WebGPU
 * "Add relu op" pull request referenced from the addmm page). */
#define IMC_ACT_RELU 0x100

/* ---------------------------------------- kernel ids (imc_last_kernel()) */
#define IMC_KERNEL_NONE 0 /* nothing launched (empty problem)              */
#define IMC_KERNEL_TC3 1  /* tcgen05 3xTF32 kernel                         */
#define IMC_KERNEL_TC1 2  /* tcgen05 1xTF32 kernel                         */
#define IMC_KERNEL_SIMT 3 /* fp32 FFMA SIMT kernel                         */
#define IMC_KERNEL_FILL 4 /* epilogue only: K == 0 or alpha == 0           */
#define IMC_KERNEL_DIRECT 5 /* direct conv2d kernel (IMC_MODE_DIRECT)      */

/*
 * gemm_addmm_f32 -- aten.addmm semantics.
 *
 * Source: ExecuTorch WebGPU pull request "Add optimized addmm op",
 * Solution and Implementation paragraphs (out = beta*self + alpha*(mat1 @
 * mat2); self broadcast from [N] or given as a full [M,N]; mat2 read as
 * mat2[k*N + n]; AddmmParams carries M, N, K, self_2d, beta, alpha) and its
 * Constraints paragraph (fp32 only; 2-D operands; mat2 exactly [K,N]).
 *
 *   out[i,j] = beta * self(i,j) + alpha * sum_{k<K} mat1[i*K + k] * mat2[k*N + j]
 *   self(i,j) = self[j]          when self_2d == 0  (self is [N])
 *             = self[i*N + j]    when self_2d == 1  (self is [M,N])
 *
 * Arguments
 *   self    [N] or [M,N] fp32; may be NULL only when beta == 0.  Not read
 *           when beta == 0 (NaN / Inf in it do not propagate).
 *   self_2d 0 or 1 as above; any other value is IMC_ERR_ARG.
 *   mat1    [M,K] fp32 row-major.   mat2 [K,N] fp32 row-major.
 *           Neither is read when alpha == 0 or K == 0.
 *   out     [M,N] fp32 row-major, written in full.  out may equal self when
 *           self_2d == 1 (in-place addmm); any other overlap of out with an
 *           input is IMC_ERR_ALIAS.
 *   M, N, K sizes, each in [0, 2^31).  M == 0 or N == 0: nothing to do, OK.
 *           K == 0: out = beta*self (the empty sum is 0).
 *   beta, alpha  finite scalars (the pages default both to 1.0, which the
 *           Python binding supplies); used in fp32.
 *   stream  cudaStream_t or NULL.
 * Kernel choice: the tcgen05 path takes any K and any alignment: it reads
 * mat2 through a transposed copy in its scratch whose rows are padded to a
 * multiple of 4 floats, and copies mat1 there too when its rows are not
 * 16-byte aligned (K % 4 != 0 or an unaligned base).  Tiny problems take the
 * SIMT kernel.  imc_last_kernel() / imc_last_kernel_name() report which ran.
 */
int gemm_addmm_f32(const float* self, int self_2d, const float* mat1, const float* mat2,
                   float* out, int64_t M, int64_t N, int64_t K, double beta, double alpha,
                   void* stream);

/* gemm_addmm_f32 with an explicit mode (IMC_MODE_* other than
 * IMC_MODE_DIRECT, optionally | IMC_ACT_RELU); mode IMC_MODE_DEFAULT is
 * exactly gemm_addmm_f32.  Any other mode value is IMC_ERR_ARG. */
int gemm_addmm_f32_ex(const float* self, int self_2d, const float* mat1, const float* mat2,
                      float* out, int64_t M, int64_t N, int64_t K, double beta, double alpha,
                      int mode, void* stream);

/* Bytes of device scratch the addmm prefers for these sizes and mode: the
 * copy of mat2 transposed and split (2*N*Kp*4 bytes when the 3xTF32
 * tensor-core kernel would run, N*Kp*4 for 1xTF32; Kp = K rounded up to a
 * multiple of 4), a copy of mat1 (M*Kp*4) when K % 4 != 0, plus split-K
 * partial sums (slices*M*N*4) for problems with too few output tiles to fill
 * the GPU; 0 when the SIMT or epilogue-only kernel would run.  The size
 * assumes 16-byte aligned pointers (alpha != 0); with an unaligned mat1 the
 * call also needs the mat1 copy, and a workspace without room for it makes
 * gemm_addmm_f32_ws run the SIMT kernel (or return IMC_ERR_ARG in a forced
 * tensor-core mode).  Returns 0 for invalid sizes or mode. */
size_t gemm_addmm_f32_workspace_bytes(int64_t M, int64_t N, int64_t K, int mode);

/* gemm_addmm_f32_ex with caller-provided scratch: `workspace` is a device
 * buffer of `workspace_bytes`, 16-byte aligned, not overlapping any argument
 * (may be NULL when no scratch is needed).  It must hold at least the mat2
 * copy (2*N*K*4 or N*K*4 bytes); the kernel plans within the buffer given, so
 * gemm_addmm_f32_workspace_bytes() bytes give the fastest plan and fewer
 * bytes a plan with fewer (or no) split-K slices.  Nothing is allocated.
 * The buffer is dead once the work enqueued on `stream` completes; work using
 * it concurrently on another stream races.  Too small, NULL or unaligned:
 * IMC_ERR_ARG; overlapping: IMC_ERR_ALIAS. */
int gemm_addmm_f32_ws(const float* self, int self_2d, const float* mat1, const float* mat2,
                      float* out, int64_t M, int64_t N, int64_t K, double beta, double alpha,
                      int mode, void* workspace, size_t workspace_bytes, void* stream);

/*
 * conv2d_gemm_f32 -- groups==1, non-transposed NCHW convolution lowered to
 * an implicit-im2col GEMM.
 *
 * Source: ExecuTorch WebGPU pull request "et_vk conv2d: route standard
 * (groups==1) conv through an im2col tiled GEMM", Solution paragraph
 * (M = OC, N = B*OH*OW, K = IC*KH*KW; out-of-range taps read 0.0, which
 * implements padding) and Implementation paragraph (A = weight viewed as
 * [OC, K]; B sampled on the fly with n -> (b, oh, ow), kk -> (ic, kh, kw),
 * ih = oh*sH - pH + kh*dH and likewise iw; bias per row (OC); NCHW output).
 *
 *   out[b,oc,oh,ow] = bias[oc] + sum_{ic,kh,kw} w[oc,ic,kh,kw] * x[b,ic,ih,iw]
 *   OH = floor((H + 2*pad - dilation*(KH-1) - 1) / stride) + 1, likewise OW.
 *
 * Arguments
 *   x     [B,IC,H,W] fp32 contiguous.      w [OC,IC,KH,KW] fp32 contiguous.
 *   bias  [OC] fp32, or NULL for no bias.  out [B,OC,OH,OW] fp32, written in
 *         full; it may not overlap x, w or bias (IMC_ERR_ALIAS).
 *   B, IC, OC >= 0 (B == 0 or OC == 0: nothing to do; IC == 0: out = bias);
 *   H, W, KH, KW >= 1; stride >= 1, pad >= 0, dilation >= 1, applied to
 *   both axes; OH, OW must come out >= 1 (else IMC_ERR_SHAPE).  Every
 *   tensor must hold fewer than 2^31 elements.
 * Kernel choice: the tcgen05 path gathers the im2col operand itself and has
 * no alignment rule on x or w; tiny problems take the SIMT kernel.  With
 * fewer than 8 input channels, W and OW multiples of 4 and x, out 16-byte
 * aligned, it reads each tile's input window from shared memory, brought in
 * by one TMA box per tile ("k_tc_conv<3xtf32,slab>"); when moreover OC <= 128
 * and the output's tiles of 8 rows x 32 columns fill between 3/4 of the SMs
 * and all of them (one tile each), the product is
 * taken with the channels as the MMA's M and 256 positions as its N
 * ("k_tc_conv<3xtf32,slab_t>").
 */
int conv2d_gemm_f32(const float* x, const float* w, const float* bias, float* out, int64_t B,
                    int64_t IC, int64_t H, int64_t W, int64_t OC, int64_t KH, int64_t KW,
                    int64_t stride, int64_t pad, int64_t dilation, void* stream);

/* conv2d_gemm_f32 with an explicit mode (IMC_MODE_*, optionally
 * | IMC_ACT_RELU). */
int conv2d_gemm_f32_ex(const float* x, const float* w, const float* bias, float* out, int64_t B,
                       int64_t IC, int64_t H, int64_t W, int64_t OC, int64_t KH, int64_t KW,
                       int64_t stride, int64_t pad, int64_t dilation, int mode, void* stream);

/* conv2d_gemm_f32_ex with separate height / width stride, padding and
 * dilation, as in the per-axis index map ih = oh*sH - pH + kh*dH,
 * iw = ow*sW - pW + kw*dW of the same Implementation paragraph. */
int conv2d_gemm_f32_nd(const float* x, const float* w, const float* bias, float* out, int64_t B,
                       int64_t IC, int64_t H, int64_t W, int64_t OC, int64_t KH, int64_t KW,
                       int64_t sH, int64_t sW, int64_t pH, int64_t pW, int64_t dH, int64_t dW,
                       int mode, void* stream);

/*
 * gemm_addmm_f32_noalloc -- gemm_addmm_f32_ex for callers that cannot
 * allocate device memory while they run.  (The pages have no counterpart:
 * this is a deployment option of this library.)
 *
 * Meant for programs whose device memory is fixed when they start, such as a
 * real-time or embedded runtime with a set memory budget, or an operator in a
 * host framework that forbids allocation inside its compute callback: for
 * them an allocation on the call path can block behind other device work or
 * fail under memory pressure mid-run.  Inputs and output are still the
 * caller's.  The tensor-core path's scratch (mat2 transposed, split into hi /
 * lo parts) lives in a fixed device buffer of IMC_NOALLOC_SCRATCH_BYTES
 * inside the library, which every GPU that loads it holds until the process
 * exits; no call takes memory from a pool or frees any.
 *
 * Limit: a problem whose mat2 copy alone would exceed
 * IMC_NOALLOC_SCRATCH_BYTES -- N*K above 4 Mi elements in the default mode,
 * 8 Mi in IMC_MODE_TF32 -- returns IMC_ERR_SCRATCH before any CUDA call; the
 * kernel plans its split-K partial sums within what is left of the buffer.
 * Problems that take the SIMT kernel need no scratch.
 * Order of checks: the argument checks of gemm_addmm_f32_ex come first (the
 * same statuses in the same order, IMC_ERR_ARG, IMC_ERR_SHAPE, IMC_ERR_NULL,
 * IMC_ERR_ALIAS), then the size check (IMC_ERR_SCRATCH); none of them makes
 * a CUDA call.
 * Set-up, and when the buffer is reserved: CUDA loads a library's device
 * code into each device's memory when it is first used there (lazy module
 * loading, the default), and the buffer is part of that code's image.  So
 * the FIRST call on a device is the set-up: it loads the buffer (reserving
 * IMC_NOALLOC_SCRATCH_BYTES of device memory at that moment, which can fail
 * with IMC_ERR_CUDA if the device is full) and looks its address up with
 * cudaGetSymbolAddress, with that device current.  The same holds for the
 * code of each kernel the first time it runs.  Make the first calls -- one
 * per shape class and mode the program will use -- at start-up, before any
 * memory budget is fixed and before any stream is captured, or set the
 * environment variable CUDA_MODULE_LOADING=EAGER before the process
 * initialises CUDA, so that everything is loaded when the context is made.
 * After the set-up, calls allocate nothing (each looks the address up again,
 * which only reads the loaded code's symbol table).
 * Sharing: every call uses the same buffer, which keeps what the last call
 * left in it.  Nothing in it needs to start at zero (each call writes all it
 * reads before reading it), but calls whose work overlaps on the GPU -- on
 * different streams, or from different host threads -- race on it.
 * Other arguments, status codes and results are those of gemm_addmm_f32_ex;
 * the results equal, bit for bit, those of gemm_addmm_f32_ws given a
 * workspace of IMC_NOALLOC_SCRATCH_BYTES (the same plan runs).
 */
#define IMC_NOALLOC_SCRATCH_BYTES ((size_t)32 << 20)
int gemm_addmm_f32_noalloc(const float* self, int self_2d, const float* mat1, const float* mat2,
                           float* out, int64_t M, int64_t N, int64_t K, double beta,
                           double alpha, int mode, void* stream);

/* Bytes of device scratch conv2d_gemm_f32_ws needs for these arguments:
 * 2*OC*Kp*4 for the 3xTF32 tensor-core kernel, OC*Kp*4 for the 1xTF32 one
 * (Kp = IC*KH*KW rounded up to a multiple of 4), 0 otherwise or when the
 * arguments are invalid. */
size_t conv2d_gemm_f32_workspace_bytes(int64_t B, int64_t IC, int64_t H, int64_t W, int64_t OC,
                                       int64_t KH, int64_t KW, int64_t sH, int64_t sW,
                                       int64_t pH, int64_t pW, int64_t dH, int64_t dW, int mode);

/* conv2d_gemm_f32_nd with caller-provided scratch (same rules as
 * gemm_addmm_f32_ws); nothing is allocated. */
int conv2d_gemm_f32_ws(const float* x, const float* w, const float* bias, float* out, int64_t B,
                       int64_t IC, int64_t H, int64_t W, int64_t OC, int64_t KH, int64_t KW,
                       int64_t sH, int64_t sW, int64_t pH, int64_t pW, int64_t dH, int64_t dW,
                       int mode, void* workspace, size_t workspace_bytes, void* stream);

/*
 * linear_f32 -- aten.linear: out[M,N] = x[M,K] @ w[N,K]^T (+ bias[N]).
 *
 * Source: the same tiled GEMM as addmm with the B operand read from the
 * transposed [N, K] weight -- ExecuTorch WebGPU "Add optimized addmm op",
 * Implementation paragraph (addmm re-derives its B read for mat2's [K,N]
 * layout, "unlike linear's transposed [N,K] weight"), and the conv page's
 * Implementation paragraph (conv2d_gemm forks linear_fp32_tiled).
 *
 *   out[m,n] = bias[n] + sum_k x[m*K + k] * w[n*K + k]     (bias may be NULL)
 *
 * x [M,K], w [N,K], bias [N] or NULL, out [M,N]: contiguous row-major fp32
 * device pointers; out may not overlap x, w or bias.  M, N, K in [0, 2^31).
 * mode: IMC_MODE_* (not IMC_MODE_DIRECT), optionally | IMC_ACT_RELU.  The
 * weight is already K-major, so the tensor-core path needs scratch only for
 * its TF32 lo part (N*K*4 bytes, 3xTF32) and any split-K partial sums;
 * when K % 4 != 0 (or w / x is not 16-byte aligned) the weight (hi and lo)
 * and x are copied there with rows of K rounded up to 4 floats.  linear_f32
 * takes the scratch from the stream-ordered pool, linear_f32_ws from the
 * caller (rules as gemm_addmm_f32_ws).  Tiny problems take the SIMT kernel.
 */
int linear_f32(const float* x, const float* w, const float* bias, float* out, int64_t M,
               int64_t N, int64_t K, int mode, void* stream);
size_t linear_f32_workspace_bytes(int64_t M, int64_t N, int64_t K, int mode);
int linear_f32_ws(const float* x, const float* w, const float* bias, float* out, int64_t M,
                  int64_t N, int64_t K, int mode, void* workspace, size_t workspace_bytes,
                  void* stream);

/*
 * gemm_addmm_f32_host, conv2d_gemm_f32_host -- gemm_addmm_f32_ex and
 * conv2d_gemm_f32_nd on HOST buffers.  (The pages have no counterpart: this
 * is the library's call for callers that hold their tensors in host memory.)
 *
 * Every tensor pointer (self, mat1, mat2, out; x, w, bias, out) is a host
 * pointer to contiguous row-major fp32 data, with the layouts, the other
 * arguments, the checks and the status codes of the device entry points.
 * All argument checks run first (aliasing is checked on the host ranges;
 * out may equal a 2-D self, as there).  The call then enqueues on `stream`:
 * one device buffer from the library's pool, the host->device copies of the
 * inputs the call reads, the computation (the device entry point on those
 * copies), the device->host copy of out, and the buffer's release.  It
 * returns once that is enqueued; out holds the result when the stream's work
 * up to that point has completed (cudaStreamSynchronize).  Calls on separate
 * streams overlap one call's copies with another's computation.
 * Host memory: page-locked (cudaHostAlloc, cudaMallocHost, cudaHostRegister)
 * for copies that run asynchronously and overlap other streams' work;
 * pageable memory is accepted, but the copies then hold the calling thread.
 * The caller keeps the input buffers unchanged, and out unread, until the
 * stream's work completes.  A failure after the checks (a CUDA error while
 * copying or launching) returns IMC_ERR_CUDA.
 */
int gemm_addmm_f32_host(const float* self, int self_2d, const float* mat1, const float* mat2,
                        float* out, int64_t M, int64_t N, int64_t K, double beta, double alpha,
                        int mode, void* stream);
int conv2d_gemm_f32_host(const float* x, const float* w, const float* bias, float* out,
                         int64_t B, int64_t IC, int64_t H, int64_t W, int64_t OC, int64_t KH,
                         int64_t KW, int64_t sH, int64_t sW, int64_t pH, int64_t pW, int64_t dH,
                         int64_t dW, int mode, void* stream);

/* Human-readable name of a status code (static string, never NULL). */
const char* imc_status_string(int status);

/* IMC_KERNEL_* id of the kernel the calling host thread's last successful
 * call launched. */
int imc_last_kernel(void);

/* Name of the main kernel the calling host thread's last successful call
 * launched, with its form, e.g. "k_tc_gemm<3xtf32,a_tmem>",
 * "k_tc_conv<3xtf32>", "k_tc_conv<1xtf32,slab>", "k_tc_conv<3xtf32,slab_t>",
 * "k_simt_small"; "none"
 * when nothing ran.  A static string, never NULL. */
const char* imc_last_kernel_name(void);

/* Number of kernels this library has launched in this process. */
uint64_t imc_launch_count(void);

/* Synchronises `stream`, then reads and clears the current device's
 * watchdog word.  Returns IMC_OK, IMC_ERR_TIMEOUT if a kernel gave up on a
 * barrier wait since the last check, or IMC_ERR_CUDA. */
int imc_check_device_error(void* stream);

/* Library ABI version (major * 100 + minor). */
int imc_version(void);

/* Diagnostic of the failure path: enqueues on `stream` a one-thread kernel
 * that waits on a barrier nothing completes, with the bounded wait of the
 * library's kernels shortened to limit_us microseconds (1000 .. 1000000).
 * The wait gives up, the kernel records it in the watchdog word and returns,
 * so that imc_check_device_error(stream) then reports IMC_ERR_TIMEOUT (and
 * clears it) while the CUDA context stays usable.  IMC_OK once enqueued,
 * IMC_ERR_ARG for a limit out of range, IMC_ERR_DEVICE without a usable GPU. */
int imc_selftest_wait_timeout(int limit_us, void* stream);

/* Returns the device memory the library's pools hold but no call in flight
 * uses (cudaMemPoolTrimTo) on every device the library has used.  Call it
 * once the library's work has completed.  IMC_OK or IMC_ERR_CUDA. */
int imc_release_memory(void);

#ifdef __cplusplus
}
#endif
#endif /* IMC_H */
