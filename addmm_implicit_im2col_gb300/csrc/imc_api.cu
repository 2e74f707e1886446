// C ABI of libimc (include/imc.h): argument checks, kernel choice, launch.
//
// Every check runs before anything is enqueued, so a call that fails has
// launched nothing -- the "throw before leak" rule of the ExecuTorch WebGPU
// conv2d page (Implementation paragraph: both dispatch grids are computed
// before any buffer is allocated).  The addmm checks follow the "Add
// optimized addmm op" page's Implementation and Constraints paragraphs
// (non-null buffers, mat2 exactly [K,N], self [N] or [M,N], fp32 only -- the
// last is fixed by the float* types here).  The 65535-workgroup cap those
// pages state is a WebGPU dispatch limit and is not reproduced.
#include <atomic>
#include <cmath>
#include <cstddef>
#include <cstdint>
#include <mutex>

#include "imc.h"
#include "imc_internal.cuh"

namespace imc {

static std::atomic<uint64_t> g_launches{0};
static thread_local int t_last_kernel = IMC_KERNEL_NONE;
static thread_local const char* t_last_name = "none";
static thread_local const char* t_pending_name = "none";

void note_launch() { g_launches.fetch_add(1, std::memory_order_relaxed); }
void note_kernel_name(const char* name) { t_pending_name = name; }

namespace {
constexpr int kMaxDevices = 64;
std::mutex g_dev_mu;
int g_sm_count[kMaxDevices];
int g_dev_ok[kMaxDevices];  // 0 unknown, 1 sm_103, -1 other

// IMC_OK when the current device is compute capability 10.3.
int check_device() {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) {
    cudaGetLastError();
    return IMC_ERR_DEVICE;
  }
  if (dev >= kMaxDevices) return IMC_ERR_DEVICE;
  std::lock_guard<std::mutex> lk(g_dev_mu);
  if (g_dev_ok[dev] == 0) {
    int major = 0, minor = 0, sms = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
      cudaGetLastError();
      return IMC_ERR_DEVICE;
    }
    g_sm_count[dev] = sms;
    g_dev_ok[dev] = (major == 10 && minor == 3) ? 1 : -1;
  }
  return g_dev_ok[dev] == 1 ? IMC_OK : IMC_ERR_DEVICE;
}

bool overlaps(const void* a, uint64_t abytes, const void* b, uint64_t bbytes) {
  if (!a || !b || abytes == 0 || bbytes == 0) return false;
  const uintptr_t a0 = (uintptr_t)a, b0 = (uintptr_t)b;
  return a0 < b0 + bbytes && b0 < a0 + abytes;
}

bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

constexpr int64_t kMaxDim = 0x7fffffffLL;
// Problems smaller than this many multiply-adds run on the SIMT kernel: the
// tensor-core kernel's fixed set-up (TMEM allocation, pipeline fill) is
// larger than the whole job there.  Above it the tensor path measured faster
// (addmm 256x256x64: 10.2 against 12.3 us; 256x256x256: 13.3 against 41 us
// for the small SIMT kernel).
constexpr int64_t kTinyMacs = int64_t(1) << 22;

int finish(cudaError_t e, int kernel) {
  if (e != cudaSuccess) return IMC_ERR_CUDA;
  t_last_kernel = kernel;
  t_last_name = t_pending_name;
  return IMC_OK;
}

void set_none() {
  t_last_kernel = IMC_KERNEL_NONE;
  t_last_name = "none";
}

// The library's stream-ordered memory pool of each device, created on first
// use.  It keeps the memory it has handed out for later calls (release
// threshold: all of it; imc_release_memory gives it back), and hands a block
// freed on one stream to a call on another stream only once that free has
// completed: no dependency is added between the streams of separate calls.
std::mutex g_pool_mu;
cudaMemPool_t g_pool[kMaxDevices];

cudaError_t pool_alloc(void** p, size_t bytes, cudaStream_t s) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  cudaMemPool_t pool;
  {
    std::lock_guard<std::mutex> lk(g_pool_mu);
    if (!g_pool[dev]) {
      cudaMemPoolProps props = {};
      props.allocType = cudaMemAllocationTypePinned;
      props.location.type = cudaMemLocationTypeDevice;
      props.location.id = dev;
      cudaMemPool_t created;
      e = cudaMemPoolCreate(&created, &props);
      if (e != cudaSuccess) return e;
      uint64_t keep = UINT64_MAX;
      int no = 0;
      if ((e = cudaMemPoolSetAttribute(created, cudaMemPoolAttrReleaseThreshold, &keep)) !=
              cudaSuccess ||
          (e = cudaMemPoolSetAttribute(created, cudaMemPoolReuseAllowInternalDependencies,
                                       &no)) != cudaSuccess) {
        cudaMemPoolDestroy(created);
        return e;
      }
      g_pool[dev] = created;
    }
    pool = g_pool[dev];
  }
  return cudaMallocFromPoolAsync(p, bytes, pool, s);
}
}  // namespace

int device_sm_count() {
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < kMaxDevices) {
    std::lock_guard<std::mutex> lk(g_dev_mu);
    if (g_sm_count[dev] > 0) return g_sm_count[dev];
  }
  int n = 0;
  cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
  return n > 0 ? n : 1;
}

}  // namespace imc

using namespace imc;


namespace {

// Splits a mode argument into the kernel mode and the ReLU flag.  False for
// unknown bits or a kernel mode the operation does not have (IMC_MODE_DIRECT
// is conv-only).
bool parse_mode(int mode, bool conv, int* base, int* relu) {
  if (mode & ~(0xFF | IMC_ACT_RELU)) return false;
  *base = mode & 0xFF;
  *relu = (mode & IMC_ACT_RELU) ? 1 : 0;
  return *base >= IMC_MODE_DEFAULT && *base <= (conv ? IMC_MODE_DIRECT : IMC_MODE_FORCE_TC1);
}

// Which kernel a well-formed addmm takes.  `tc_ok` is whether the tcgen05
// path can take the operands (it reads operands whose rows are not 16-byte
// aligned through padded copies in its scratch, so: whether they are read).
int plan_gemm(int64_t M, int64_t N, int64_t K, double alpha, int mode, bool tc_ok) {
  if (M == 0 || N == 0) return IMC_KERNEL_NONE;
  if (alpha == 0.0 || K == 0) return IMC_KERNEL_FILL;
  const bool force_tc = mode == IMC_MODE_FORCE_TC3 || mode == IMC_MODE_FORCE_TC1;
  if (force_tc) return tc_ok ? (mode == IMC_MODE_FORCE_TC3 ? IMC_KERNEL_TC3 : IMC_KERNEL_TC1) : -1;
  if (mode == IMC_MODE_SIMT || !tc_ok || (double)M * N * K < (double)kTinyMacs)
    return IMC_KERNEL_SIMT;
  return mode == IMC_MODE_DEFAULT ? IMC_KERNEL_TC3 : IMC_KERNEL_TC1;
}

// workspace == nullptr and !caller_ws: the transposed-mat2 workspace comes
// from the library's stream-ordered pool (pool_alloc / cudaFreeAsync on
// `stream`).  caller_ws: the caller's buffer of ws_bytes is used, nothing is
// allocated.
// b_kmajor: mat2 is given transposed as [N,K] (linear).
// validate_only: run every argument check (pointers taken as 16-byte aligned,
// as the device copies of host buffers are) and return before any CUDA call.
int gemm_impl(const float* self, int self_2d, const float* mat1, const float* mat2, float* out,
              int64_t M, int64_t N, int64_t K, double beta, double alpha, int mode_arg,
              bool b_kmajor, void* workspace, size_t ws_bytes, bool caller_ws, void* stream,
              bool validate_only = false) {
  if (self_2d != 0 && self_2d != 1) return IMC_ERR_ARG;
  int mode = 0, relu = 0;
  if (!parse_mode(mode_arg, false, &mode, &relu)) return IMC_ERR_ARG;
  if (!std::isfinite(beta) || !std::isfinite(alpha)) return IMC_ERR_ARG;
  if (M < 0 || N < 0 || K < 0 || M > kMaxDim || N > kMaxDim || K > kMaxDim) return IMC_ERR_SHAPE;
  if (M == 0 || N == 0) {
    set_none();
    return IMC_OK;
  }
  const bool read_self = beta != 0.0;
  const bool read_ops = alpha != 0.0 && K > 0;
  if (!out) return IMC_ERR_NULL;
  if (read_self && !self) return IMC_ERR_NULL;
  if (read_ops && (!mat1 || !mat2)) return IMC_ERR_NULL;

  const uint64_t out_bytes = (uint64_t)M * (uint64_t)N * 4u;
  const uint64_t mat1_bytes = (uint64_t)M * K * 4u, mat2_bytes = (uint64_t)K * N * 4u;
  if (read_ops && (overlaps(out, out_bytes, mat1, mat1_bytes) ||
                   overlaps(out, out_bytes, mat2, mat2_bytes)))
    return IMC_ERR_ALIAS;
  const uint64_t self_bytes = (uint64_t)(self_2d ? M * N : N) * 4u;
  if (read_self) {
    const bool exact_inplace = self_2d && (const void*)self == (const void*)out;
    if (!exact_inplace && overlaps(out, out_bytes, self, self_bytes)) return IMC_ERR_ALIAS;
  }

  GemmArgs a;
  a.self = self;
  a.mat1 = mat1;
  a.mat2 = mat2;
  a.out = out;
  a.M = M;
  a.N = N;
  a.K = K;
  a.alpha = (float)alpha;
  a.beta = (float)beta;
  a.self_2d = self_2d;
  a.read_self = read_self ? 1 : 0;
  a.vec_out = (N % 4 == 0) && aligned16(out) && (!read_self || aligned16(self)) ? 1 : 0;
  a.relu = relu;
  a.b_kmajor = b_kmajor ? 1 : 0;
  const bool tc_ok = read_ops;
  int kernel = plan_gemm(M, N, K, alpha, mode, tc_ok);
  if (kernel < 0) return IMC_ERR_SHAPE;
  if (validate_only) return IMC_OK;
  bool tc = kernel == IMC_KERNEL_TC3 || kernel == IMC_KERNEL_TC1;
  const bool three = kernel == IMC_KERNEL_TC3;
  // operand copies with aligned rows: from K alone, or also from the pointers
  const bool pad_a = tc_gemm_pad_a(a), pad_b = tc_gemm_pad_b(a);
  const bool pad_a_k = K % 4 != 0, pad_b_k = b_kmajor && K % 4 != 0;
  // A caller workspace sized by the size query (which assumes 16-byte aligned
  // pointers) may lack room for the copies an unaligned operand needs: such a
  // call takes the SIMT kernel, unless a tensor-core mode was forced.
  if (tc && caller_ws && (pad_a != pad_a_k || pad_b != pad_b_k) &&
      ws_bytes < tc_gemm_workspace_bytes(M, N, K, three, b_kmajor, pad_a, pad_b, 0) &&
      mode != IMC_MODE_FORCE_TC3 && mode != IMC_MODE_FORCE_TC1) {
    kernel = IMC_KERNEL_SIMT;
    tc = false;
  }
  // minimum (no split-K) and the scratch the call will use
  const size_t need_min =
      tc ? tc_gemm_workspace_bytes(M, N, K, three, b_kmajor, pad_a, pad_b, 0) : 0;
  const size_t need = tc ? tc_gemm_workspace_bytes(M, N, K, three, b_kmajor, pad_a, pad_b,
                                                   caller_ws ? ws_bytes : SIZE_MAX)
                         : 0;
  if (caller_ws && need_min > 0) {
    if (!workspace || ws_bytes < need_min || !aligned16(workspace)) return IMC_ERR_ARG;
    if (overlaps(workspace, need, out, out_bytes) || overlaps(workspace, need, mat1, mat1_bytes) ||
        overlaps(workspace, need, mat2, mat2_bytes) ||
        (read_self && overlaps(workspace, need, self, self_bytes)))
      return IMC_ERR_ALIAS;
  }
  const int dev = check_device();
  if (dev != IMC_OK) return dev;
  cudaStream_t s = (cudaStream_t)stream;

  if (kernel == IMC_KERNEL_FILL) return finish(launch_fill_gemm(a, s), kernel);
  if (kernel == IMC_KERNEL_SIMT) return finish(launch_simt_gemm(a, s), kernel);
  if (!tc_gemm_supported(a)) return IMC_ERR_DEVICE;  // driver without tensor-map support
  void* ws = workspace;
  const bool pool = !caller_ws && need > 0;
  if (pool && pool_alloc(&ws, need, s) != cudaSuccess) return IMC_ERR_CUDA;
  const cudaError_t e = launch_tc_gemm(a, three, ws, need, s);
  if (pool) {
    const cudaError_t f = cudaFreeAsync(ws, s);
    if (e == cudaSuccess && f != cudaSuccess) return IMC_ERR_CUDA;
  }
  return finish(e, kernel);
}

}  // namespace

extern "C" {

int gemm_addmm_f32_ex(const float* self, int self_2d, const float* mat1, const float* mat2,
                      float* out, int64_t M, int64_t N, int64_t K, double beta, double alpha,
                      int mode, void* stream) {
  return gemm_impl(self, self_2d, mat1, mat2, out, M, N, K, beta, alpha, mode, false, nullptr, 0,
                   false, stream);
}

int gemm_addmm_f32(const float* self, int self_2d, const float* mat1, const float* mat2,
                   float* out, int64_t M, int64_t N, int64_t K, double beta, double alpha,
                   void* stream) {
  return gemm_impl(self, self_2d, mat1, mat2, out, M, N, K, beta, alpha, IMC_MODE_DEFAULT, false,
                   nullptr, 0, false, stream);
}

int gemm_addmm_f32_ws(const float* self, int self_2d, const float* mat1, const float* mat2,
                      float* out, int64_t M, int64_t N, int64_t K, double beta, double alpha,
                      int mode, void* workspace, size_t workspace_bytes, void* stream) {
  return gemm_impl(self, self_2d, mat1, mat2, out, M, N, K, beta, alpha, mode, false, workspace,
                   workspace_bytes, true, stream);
}

}  // extern "C"

namespace {
size_t gemm_query(int64_t M, int64_t N, int64_t K, int mode_arg, bool b_kmajor) {
  if (M <= 0 || N <= 0 || K <= 0 || M > kMaxDim || N > kMaxDim || K > kMaxDim) return 0;
  int mode = 0, relu = 0;
  if (!parse_mode(mode_arg, false, &mode, &relu)) return 0;
  const int kernel = plan_gemm(M, N, K, 1.0, mode, true);
  // pointers taken as 16-byte aligned: copies only when K % 4 != 0
  const bool pad_a = K % 4 != 0, pad_b = b_kmajor && K % 4 != 0;
  if (kernel == IMC_KERNEL_TC3)
    return tc_gemm_workspace_bytes(M, N, K, true, b_kmajor, pad_a, pad_b, SIZE_MAX);
  if (kernel == IMC_KERNEL_TC1)
    return tc_gemm_workspace_bytes(M, N, K, false, b_kmajor, pad_a, pad_b, SIZE_MAX);
  return 0;
}
}  // namespace

extern "C" {

size_t gemm_addmm_f32_workspace_bytes(int64_t M, int64_t N, int64_t K, int mode) {
  return gemm_query(M, N, K, mode, false);
}

// aten.linear on the addmm path with mat2 = w given as [N,K], self = bias [N].
int linear_f32(const float* x, const float* w, const float* bias, float* out, int64_t M,
               int64_t N, int64_t K, int mode, void* stream) {
  return gemm_impl(bias, 0, x, w, out, M, N, K, bias ? 1.0 : 0.0, 1.0, mode, true, nullptr, 0,
                   false, stream);
}

size_t linear_f32_workspace_bytes(int64_t M, int64_t N, int64_t K, int mode) {
  return gemm_query(M, N, K, mode, true);
}

int linear_f32_ws(const float* x, const float* w, const float* bias, float* out, int64_t M,
                  int64_t N, int64_t K, int mode, void* workspace, size_t workspace_bytes,
                  void* stream) {
  return gemm_impl(bias, 0, x, w, out, M, N, K, bias ? 1.0 : 0.0, 1.0, mode, true, workspace,
                   workspace_bytes, true, stream);
}

}  // extern "C"

namespace {

struct ConvShape {
  int64_t OH, OW, K;
};

// Checks sizes; fills OH, OW, K.  IMC_OK or IMC_ERR_SHAPE.
int conv_shape(int64_t B, int64_t IC, int64_t H, int64_t W, int64_t OC, int64_t KH, int64_t KW,
               int64_t sH, int64_t sW, int64_t pH, int64_t pW, int64_t dH, int64_t dW,
               ConvShape* cs) {
  if (B < 0 || IC < 0 || OC < 0 || H < 1 || W < 1 || KH < 1 || KW < 1) return IMC_ERR_SHAPE;
  if (sH < 1 || sW < 1 || pH < 0 || pW < 0 || dH < 1 || dW < 1) return IMC_ERR_SHAPE;
  if (B > kMaxDim || IC > kMaxDim || OC > kMaxDim || H > kMaxDim || W > kMaxDim ||
      KH > kMaxDim || KW > kMaxDim || sH > kMaxDim || sW > kMaxDim || pH > kMaxDim ||
      pW > kMaxDim || dH > kMaxDim || dW > kMaxDim)
    return IMC_ERR_SHAPE;
  // OH = floor((H + 2*pH - dH*(KH-1) - 1) / sH) + 1, likewise OW.
  const int64_t spanH = H + 2 * pH - dH * (KH - 1) - 1;
  const int64_t spanW = W + 2 * pW - dW * (KW - 1) - 1;
  if (spanH < 0 || spanW < 0) return IMC_ERR_SHAPE;
  cs->OH = spanH / sH + 1;
  cs->OW = spanW / sW + 1;
  // Every tensor stays below 2^31 elements (32-bit element offsets inside).
  const double lim = 2147483647.0;
  if ((double)B * IC * H * W > lim || (double)OC * IC * KH * KW > lim ||
      (double)B * OC * cs->OH * cs->OW > lim || (double)IC * KH * KW > lim ||
      (double)B * cs->OH * cs->OW > lim)
    return IMC_ERR_SHAPE;
  cs->K = IC * KH * KW;
  return IMC_OK;
}

// Which kernel a well-formed conv takes.  `tc_ok`: the tcgen05 kernel takes
// the sizes (tc_conv_shape_ok); forced tensor-core modes fail otherwise.
int plan_conv(int64_t M, int64_t N, int64_t K, int mode, bool tc_ok) {
  if (M == 0 || N == 0) return IMC_KERNEL_NONE;
  if (K == 0) return IMC_KERNEL_FILL;
  if (mode == IMC_MODE_DIRECT) return IMC_KERNEL_DIRECT;
  if (mode == IMC_MODE_FORCE_TC3 || mode == IMC_MODE_FORCE_TC1)
    return tc_ok ? (mode == IMC_MODE_FORCE_TC3 ? IMC_KERNEL_TC3 : IMC_KERNEL_TC1) : -1;
  if (mode == IMC_MODE_SIMT || !tc_ok || (double)M * N * K < (double)kTinyMacs)
    return IMC_KERNEL_SIMT;
  return mode == IMC_MODE_DEFAULT ? IMC_KERNEL_TC3 : IMC_KERNEL_TC1;
}

// The validated problem as kernel arguments (pointers may be null for a
// size query).
ConvArgs conv_args(const float* x, const float* w, const float* bias, float* out, int64_t B,
                   int64_t IC, int64_t H, int64_t W, int64_t OC, int64_t KH, int64_t KW,
                   int64_t sH, int64_t sW, int64_t pH, int64_t pW, int64_t dH, int64_t dW,
                   const ConvShape& cs, int relu) {
  ConvArgs c;
  c.x = x;
  c.w = w;
  c.bias = bias;
  c.out = out;
  c.B = (int)B;
  c.IC = (int)IC;
  c.H = (int)H;
  c.W = (int)W;
  c.OC = (int)OC;
  c.KH = (int)KH;
  c.KW = (int)KW;
  c.sH = (int)sH;
  c.sW = (int)sW;
  c.pH = (int)pH;
  c.pW = (int)pW;
  c.dH = (int)dH;
  c.dW = (int)dW;
  c.OH = (int)cs.OH;
  c.OW = (int)cs.OW;
  c.M = OC;
  c.N = B * cs.OH * cs.OW;
  c.K = cs.K;
  c.vec_out = ((cs.OH * cs.OW) % 4 == 0) && aligned16(out) ? 1 : 0;
  c.relu = relu;
  return c;
}

// validate_only: as for gemm_impl.
int conv_impl(const float* x, const float* w, const float* bias, float* out, int64_t B,
              int64_t IC, int64_t H, int64_t W, int64_t OC, int64_t KH, int64_t KW, int64_t sH,
              int64_t sW, int64_t pH, int64_t pW, int64_t dH, int64_t dW, int mode_arg,
              void* workspace, size_t ws_bytes, bool caller_ws, void* stream,
              bool validate_only = false) {
  int mode = 0, relu = 0;
  if (!parse_mode(mode_arg, true, &mode, &relu)) return IMC_ERR_ARG;
  ConvShape cs;
  const int sh = conv_shape(B, IC, H, W, OC, KH, KW, sH, sW, pH, pW, dH, dW, &cs);
  if (sh != IMC_OK) return sh;
  if (B == 0 || OC == 0) {
    set_none();
    return IMC_OK;
  }
  const int64_t K = cs.K, OH = cs.OH, OW = cs.OW;
  if (!out) return IMC_ERR_NULL;
  if (K > 0 && (!x || !w)) return IMC_ERR_NULL;
  const uint64_t out_bytes = (uint64_t)(B * OC * OH * OW) * 4u;
  const uint64_t x_bytes = (uint64_t)(B * IC * H * W) * 4u, w_bytes = (uint64_t)(OC * K) * 4u;
  if ((K > 0 && (overlaps(out, out_bytes, x, x_bytes) || overlaps(out, out_bytes, w, w_bytes))) ||
      overlaps(out, out_bytes, bias, (uint64_t)OC * 4u))
    return IMC_ERR_ALIAS;
  const ConvArgs c = conv_args(x, w, bias, out, B, IC, H, W, OC, KH, KW, sH, sW, pH, pW, dH, dW,
                               cs, relu);
  const int kernel = plan_conv(OC, B * OH * OW, K, mode, tc_conv_shape_ok(c));
  if (kernel < 0) return IMC_ERR_SHAPE;
  if (validate_only) return IMC_OK;
  const bool tc = kernel == IMC_KERNEL_TC3 || kernel == IMC_KERNEL_TC1;
  const bool three = kernel == IMC_KERNEL_TC3;
  // minimum (no K-slices) and the scratch the call will use
  const size_t need_min = tc ? tc_conv_workspace_bytes(c, three, 0) : 0;
  const size_t need =
      tc ? tc_conv_workspace_bytes(c, three, caller_ws ? ws_bytes : SIZE_MAX) : 0;
  if (caller_ws && need_min > 0) {
    if (!workspace || ws_bytes < need_min || !aligned16(workspace)) return IMC_ERR_ARG;
    if (overlaps(workspace, need, out, out_bytes) || overlaps(workspace, need, x, x_bytes) ||
        overlaps(workspace, need, w, w_bytes) ||
        overlaps(workspace, need, bias, (uint64_t)OC * 4u))
      return IMC_ERR_ALIAS;
  }
  const int dev = check_device();
  if (dev != IMC_OK) return dev;
  cudaStream_t s = (cudaStream_t)stream;

  if (kernel == IMC_KERNEL_FILL) return finish(launch_fill_conv(c, s), kernel);
  if (kernel == IMC_KERNEL_DIRECT) return finish(launch_direct_conv(c, s), kernel);
  if (kernel == IMC_KERNEL_SIMT) return finish(launch_simt_conv(c, s), kernel);
  if (!tc_conv_supported(c)) return IMC_ERR_DEVICE;  // driver without tensor-map support
  void* ws = workspace;
  if (!caller_ws) {
    if (pool_alloc(&ws, need, s) != cudaSuccess) return IMC_ERR_CUDA;
  }
  const cudaError_t e = launch_tc_conv(c, three, ws, need, s);
  if (!caller_ws) {
    const cudaError_t f = cudaFreeAsync(ws, s);
    if (e == cudaSuccess && f != cudaSuccess) return IMC_ERR_CUDA;
  }
  return finish(e, kernel);
}

}  // namespace

extern "C" {

int conv2d_gemm_f32_nd(const float* x, const float* w, const float* bias, float* out, int64_t B,
                       int64_t IC, int64_t H, int64_t W, int64_t OC, int64_t KH, int64_t KW,
                       int64_t sH, int64_t sW, int64_t pH, int64_t pW, int64_t dH, int64_t dW,
                       int mode, void* stream) {
  return conv_impl(x, w, bias, out, B, IC, H, W, OC, KH, KW, sH, sW, pH, pW, dH, dW, mode,
                   nullptr, 0, false, stream);
}

int conv2d_gemm_f32_ws(const float* x, const float* w, const float* bias, float* out, int64_t B,
                       int64_t IC, int64_t H, int64_t W, int64_t OC, int64_t KH, int64_t KW,
                       int64_t sH, int64_t sW, int64_t pH, int64_t pW, int64_t dH, int64_t dW,
                       int mode, void* workspace, size_t workspace_bytes, void* stream) {
  return conv_impl(x, w, bias, out, B, IC, H, W, OC, KH, KW, sH, sW, pH, pW, dH, dW, mode,
                   workspace, workspace_bytes, true, stream);
}

size_t conv2d_gemm_f32_workspace_bytes(int64_t B, int64_t IC, int64_t H, int64_t W, int64_t OC,
                                       int64_t KH, int64_t KW, int64_t sH, int64_t sW,
                                       int64_t pH, int64_t pW, int64_t dH, int64_t dW,
                                       int mode_arg) {
  int mode = 0, relu = 0;
  if (!parse_mode(mode_arg, true, &mode, &relu)) return 0;
  ConvShape cs;
  if (conv_shape(B, IC, H, W, OC, KH, KW, sH, sW, pH, pW, dH, dW, &cs) != IMC_OK) return 0;
  const ConvArgs c = conv_args(nullptr, nullptr, nullptr, nullptr, B, IC, H, W, OC, KH, KW, sH,
                               sW, pH, pW, dH, dW, cs, relu);
  const int kernel = plan_conv(OC, B * cs.OH * cs.OW, cs.K, mode, tc_conv_shape_ok(c));
  if (kernel == IMC_KERNEL_TC3) return tc_conv_workspace_bytes(c, true, SIZE_MAX);
  if (kernel == IMC_KERNEL_TC1) return tc_conv_workspace_bytes(c, false, SIZE_MAX);
  return 0;
}

int conv2d_gemm_f32_ex(const float* x, const float* w, const float* bias, float* out, int64_t B,
                       int64_t IC, int64_t H, int64_t W, int64_t OC, int64_t KH, int64_t KW,
                       int64_t stride, int64_t pad, int64_t dilation, int mode, void* stream) {
  return conv2d_gemm_f32_nd(x, w, bias, out, B, IC, H, W, OC, KH, KW, stride, stride, pad, pad,
                            dilation, dilation, mode, stream);
}

int conv2d_gemm_f32(const float* x, const float* w, const float* bias, float* out, int64_t B,
                    int64_t IC, int64_t H, int64_t W, int64_t OC, int64_t KH, int64_t KW,
                    int64_t stride, int64_t pad, int64_t dilation, void* stream) {
  return conv2d_gemm_f32_nd(x, w, bias, out, B, IC, H, W, OC, KH, KW, stride, stride, pad, pad,
                            dilation, dilation, IMC_MODE_DEFAULT, stream);
}

}  // extern "C"

namespace {

size_t round256(uint64_t b) { return (size_t)((b + 255) & ~uint64_t(255)); }

// The library's two copy queues of each device (created on first use):
// every host-buffer call puts its host->device copies on the first and its
// device->host copy on the second, tied to the caller's stream by events.
// The copies of calls issued on different streams then run one after another
// in call order, one per direction at a time: the link's bandwidth drops
// when several copies in one direction share it.
std::mutex g_queue_mu;
cudaStream_t g_copy_in[kMaxDevices], g_copy_out[kMaxDevices];

cudaError_t copy_queues(cudaStream_t* in, cudaStream_t* out) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lk(g_queue_mu);
  if (!g_copy_in[dev]) {
    cudaStream_t a, b;
    if ((e = cudaStreamCreateWithFlags(&a, cudaStreamNonBlocking)) != cudaSuccess) return e;
    if ((e = cudaStreamCreateWithFlags(&b, cudaStreamNonBlocking)) != cudaSuccess) {
      cudaStreamDestroy(a);
      return e;
    }
    g_copy_in[dev] = a;
    g_copy_out[dev] = b;
  }
  *in = g_copy_in[dev];
  *out = g_copy_out[dev];
  return cudaSuccess;
}

// Work enqueued on `to` after this call waits for the work on `from` so far.
cudaError_t link(cudaStream_t from, cudaStream_t to) {
  cudaEvent_t ev;
  cudaError_t e = cudaEventCreateWithFlags(&ev, cudaEventDisableTiming);
  if (e != cudaSuccess) return e;
  e = cudaEventRecord(ev, from);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(to, ev, 0);
  const cudaError_t d = cudaEventDestroy(ev);  // released once it has completed
  return e != cudaSuccess ? e : d;
}

// Device copies of a call's host buffers in one stream-ordered allocation on
// the caller's stream `s`: `n` host ranges (nullptr / 0 bytes: absent) at
// 256-byte boundaries; dev[i] is the device address of range i.  take()
// copies the inputs in on the copy-in queue, after the work already on `s`,
// and makes `s` wait for them; finish() copies the result out on the copy-out
// queue once the work on `s` (the computation) is done, makes `s` wait for
// that copy and releases the allocation on `s`.
struct DeviceCopies {
  char* base = nullptr;
  cudaStream_t s, q_in = nullptr, q_out = nullptr;
  explicit DeviceCopies(cudaStream_t st) : s(st) {}
  int take(const void* const* host, const uint64_t* bytes, const bool* copy_in, int n,
           float** dev) {
    if (copy_queues(&q_in, &q_out) != cudaSuccess) return IMC_ERR_CUDA;
    size_t total = 0;
    for (int i = 0; i < n; ++i) total += round256(bytes[i]);
    if (pool_alloc((void**)&base, total, s) != cudaSuccess) {
      base = nullptr;
      return IMC_ERR_CUDA;
    }
    if (link(s, q_in) != cudaSuccess) return IMC_ERR_CUDA;
    int rc = IMC_OK;
    size_t off = 0;
    for (int i = 0; i < n; ++i) {
      dev[i] = bytes[i] ? reinterpret_cast<float*>(base + off) : nullptr;
      off += round256(bytes[i]);
      if (rc == IMC_OK && copy_in[i] && bytes[i] &&
          cudaMemcpyAsync(dev[i], host[i], bytes[i], cudaMemcpyHostToDevice, q_in) != cudaSuccess)
        rc = IMC_ERR_CUDA;
    }
    // `s` waits for the copies even after a failed one: the allocation is
    // released on `s`.
    if (link(q_in, s) != cudaSuccess) rc = IMC_ERR_CUDA;
    return rc;
  }
  int finish(int rc, void* host_out, const float* dev_out, uint64_t bytes) {
    if (rc == IMC_OK) {
      if (link(s, q_out) != cudaSuccess ||
          cudaMemcpyAsync(host_out, dev_out, bytes, cudaMemcpyDeviceToHost, q_out) !=
              cudaSuccess)
        rc = IMC_ERR_CUDA;
      if (link(q_out, s) != cudaSuccess) rc = IMC_ERR_CUDA;
    }
    if (base && cudaFreeAsync(base, s) != cudaSuccess && rc == IMC_OK) rc = IMC_ERR_CUDA;
    return rc;
  }
};

}  // namespace

extern "C" {

int gemm_addmm_f32_host(const float* self, int self_2d, const float* mat1, const float* mat2,
                        float* out, int64_t M, int64_t N, int64_t K, double beta, double alpha,
                        int mode, void* stream) {
  const int v = gemm_impl(self, self_2d, mat1, mat2, out, M, N, K, beta, alpha, mode, false,
                          nullptr, 0, false, stream, true);
  if (v != IMC_OK || M == 0 || N == 0) return v;
  const int dev = check_device();
  if (dev != IMC_OK) return dev;
  const bool read_self = beta != 0.0, read_ops = alpha != 0.0 && K > 0;
  const void* host[4] = {self, mat1, mat2, out};
  const uint64_t bytes[4] = {read_self ? (uint64_t)(self_2d ? M * N : N) * 4u : 0,
                             read_ops ? (uint64_t)(M * K) * 4u : 0,
                             read_ops ? (uint64_t)(K * N) * 4u : 0, (uint64_t)(M * N) * 4u};
  const bool copy_in[4] = {true, true, true, false};
  float* d[4];
  DeviceCopies dc((cudaStream_t)stream);
  int rc = dc.take(host, bytes, copy_in, 4, d);
  if (rc == IMC_OK)
    rc = gemm_impl(d[0], self_2d, d[1], d[2], d[3], M, N, K, beta, alpha, mode, false, nullptr, 0,
                   false, stream);
  return dc.finish(rc, out, d[3], bytes[3]);
}

int conv2d_gemm_f32_host(const float* x, const float* w, const float* bias, float* out,
                         int64_t B, int64_t IC, int64_t H, int64_t W, int64_t OC, int64_t KH,
                         int64_t KW, int64_t sH, int64_t sW, int64_t pH, int64_t pW, int64_t dH,
                         int64_t dW, int mode, void* stream) {
  const int v = conv_impl(x, w, bias, out, B, IC, H, W, OC, KH, KW, sH, sW, pH, pW, dH, dW, mode,
                          nullptr, 0, false, stream, true);
  if (v != IMC_OK || B == 0 || OC == 0) return v;
  const int dev = check_device();
  if (dev != IMC_OK) return dev;
  ConvShape cs;
  conv_shape(B, IC, H, W, OC, KH, KW, sH, sW, pH, pW, dH, dW, &cs);  // checked above
  const void* host[4] = {x, w, bias, out};
  const uint64_t bytes[4] = {cs.K > 0 ? (uint64_t)(B * IC * H * W) * 4u : 0,
                             cs.K > 0 ? (uint64_t)(OC * cs.K) * 4u : 0,
                             bias ? (uint64_t)OC * 4u : 0,
                             (uint64_t)(B * OC * cs.OH * cs.OW) * 4u};
  const bool copy_in[4] = {true, true, true, false};
  float* d[4];
  DeviceCopies dc((cudaStream_t)stream);
  int rc = dc.take(host, bytes, copy_in, 4, d);
  if (rc == IMC_OK)
    rc = conv_impl(d[0], d[1], d[2], d[3], B, IC, H, W, OC, KH, KW, sH, sW, pH, pW, dH, dW, mode,
                   nullptr, 0, false, stream);
  return dc.finish(rc, out, d[3], bytes[3]);
}

const char* imc_status_string(int status) {
  switch (status) {
    case IMC_OK: return "IMC_OK";
    case IMC_ERR_NULL: return "IMC_ERR_NULL: a required pointer is NULL";
    case IMC_ERR_SHAPE: return "IMC_ERR_SHAPE: a size is out of range or the output is empty";
    case IMC_ERR_ARG: return "IMC_ERR_ARG: bad flag, mode or scalar";
    case IMC_ERR_ALIAS: return "IMC_ERR_ALIAS: the output overlaps an input";
    case IMC_ERR_CUDA: return "IMC_ERR_CUDA: a CUDA call or kernel launch failed";
    case IMC_ERR_TIMEOUT: return "IMC_ERR_TIMEOUT: a kernel gave up waiting on a barrier";
    case IMC_ERR_DEVICE: return "IMC_ERR_DEVICE: no usable compute capability 10.3 device";
    case IMC_ERR_SCRATCH:
      return "IMC_ERR_SCRATCH: the problem needs more scratch than the no-allocation "
             "entry point's fixed buffer holds";
    default: return "IMC_ERR_UNKNOWN";
  }
}

int imc_last_kernel(void) { return t_last_kernel; }

const char* imc_last_kernel_name(void) { return t_last_name; }

uint64_t imc_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

int imc_check_device_error(void* stream) {
  const int dev = check_device();
  if (dev != IMC_OK) return dev;
  int vg = 0, vc = 0;
  if (cudaStreamSynchronize((cudaStream_t)stream) != cudaSuccess ||
      gemm_take_watchdog(&vg) != cudaSuccess || conv_take_watchdog(&vc) != cudaSuccess)
    return IMC_ERR_CUDA;
  return (vg != 0 || vc != 0) ? IMC_ERR_TIMEOUT : IMC_OK;
}

int imc_version(void) { return 103; }

int imc_selftest_wait_timeout(int limit_us, void* stream) {
  if (limit_us < 1000 || limit_us > 1000000) return IMC_ERR_ARG;
  const int dev = check_device();
  if (dev != IMC_OK) return dev;
  return launch_wait_selftest(limit_us, (cudaStream_t)stream) == cudaSuccess ? IMC_OK
                                                                            : IMC_ERR_CUDA;
}

int imc_release_memory(void) {
  std::lock_guard<std::mutex> lk(g_pool_mu);
  for (int d = 0; d < kMaxDevices; ++d)
    if (g_pool[d] && cudaMemPoolTrimTo(g_pool[d], 0) != cudaSuccess) return IMC_ERR_CUDA;
  return IMC_OK;
}

}  // extern "C"

// Hooks for the fixed-scratch addmm entry point (noalloc.cu).
namespace imc {

int gemm_check_args(const float* self, int self_2d, const float* mat1, const float* mat2,
                    float* out, int64_t M, int64_t N, int64_t K, double beta, double alpha,
                    int mode) {
  return gemm_impl(self, self_2d, mat1, mat2, out, M, N, K, beta, alpha, mode, false, nullptr, 0,
                   false, nullptr, true);
}

size_t gemm_scratch_needed(const float* mat1, int64_t M, int64_t N, int64_t K, double alpha,
                           int mode_arg) {
  if (M <= 0 || N <= 0 || K <= 0 || M > kMaxDim || N > kMaxDim || K > kMaxDim) return 0;
  int mode = 0, relu = 0;
  if (!parse_mode(mode_arg, false, &mode, &relu)) return 0;
  const int kernel = plan_gemm(M, N, K, alpha, mode, alpha != 0.0);
  if (kernel != IMC_KERNEL_TC3 && kernel != IMC_KERNEL_TC1) return 0;
  const bool pad_a = K % 4 != 0 || !aligned16(mat1);
  return tc_gemm_workspace_bytes(M, N, K, kernel == IMC_KERNEL_TC3, false, pad_a, false, 0);
}

int gemm_with_scratch(const float* self, int self_2d, const float* mat1, const float* mat2,
                      float* out, int64_t M, int64_t N, int64_t K, double beta, double alpha,
                      int mode, void* scratch, size_t scratch_bytes, void* stream) {
  return gemm_impl(self, self_2d, mat1, mat2, out, M, N, K, beta, alpha, mode, false, scratch,
                   scratch_bytes, true, stream);
}

int require_device() { return check_device(); }

}  // namespace imc
