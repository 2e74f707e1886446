// SIMT fp32 FFMA fallback: a shared-memory tiled GEMM with register blocking
// for shapes the tensor-core path does not take (tiny problems, K or N not a
// multiple of 4, unaligned operands) and for IMC_MODE_SIMT.
//
// This is the design family of the ExecuTorch WebGPU "Add optimized addmm op"
// page (Implementation paragraph: a workgroup stages tiles of both operands in
// shared memory, synchronises, and every thread accumulates a 4x4 register
// sub-tile over the k-tiles), here with a 64x64 output tile, 16-deep k-tiles
// and 256 threads.  The conv variant samples the im2col operand on the fly as
// the "et_vk conv2d ... im2col tiled GEMM" page's Implementation paragraph
// describes (n -> (b, oh, ow), kk -> (ic, kh, kw), out-of-range taps read 0).
#include "imc_internal.cuh"
#include "ptx.cuh"

namespace imc {
namespace {

constexpr int BM = 64, BN = 64, BK = 16, THREADS = 256;

struct GemmOperands {
  GemmArgs a;
  __device__ __forceinline__ float load_a(int64_t m, int64_t k) const {
    return a.mat1[m * a.K + k];
  }
  __device__ __forceinline__ float load_b(int64_t k, int64_t n) const {
    return a.b_kmajor ? a.mat2[n * a.K + k] : a.mat2[k * a.N + n];  // linear: w[n, k]
  }
  __device__ __forceinline__ void store_row4(int64_t m, int64_t n0, const float* acc) const {
    float* o = a.out + m * a.N;
    const float* sp = a.self_2d ? a.self + m * a.N : a.self;
    if (a.vec_out && n0 + 3 < a.N) {
      float4 r;
      float4 sv = a.read_self ? *reinterpret_cast<const float4*>(sp + n0) : make_float4(0, 0, 0, 0);
      r.x = a.read_self ? fmaf(a.alpha, acc[0], a.beta * sv.x) : a.alpha * acc[0];
      r.y = a.read_self ? fmaf(a.alpha, acc[1], a.beta * sv.y) : a.alpha * acc[1];
      r.z = a.read_self ? fmaf(a.alpha, acc[2], a.beta * sv.z) : a.alpha * acc[2];
      r.w = a.read_self ? fmaf(a.alpha, acc[3], a.beta * sv.w) : a.alpha * acc[3];
      if (a.relu) r = make_float4(fmaxf(r.x, 0.f), fmaxf(r.y, 0.f), fmaxf(r.z, 0.f), fmaxf(r.w, 0.f));
      *reinterpret_cast<float4*>(o + n0) = r;
      return;
    }
    for (int j = 0; j < 4; ++j) {
      int64_t n = n0 + j;
      if (n >= a.N) break;
      const float v = a.read_self ? fmaf(a.alpha, acc[j], a.beta * sp[n]) : a.alpha * acc[j];
      o[n] = a.relu ? fmaxf(v, 0.f) : v;
    }
  }
  __device__ __forceinline__ int64_t M() const { return a.M; }
  __device__ __forceinline__ int64_t N() const { return a.N; }
  __device__ __forceinline__ int64_t K() const { return a.K; }
};

struct ConvOperands {
  ConvArgs c;
  __device__ __forceinline__ float load_a(int64_t m, int64_t k) const {
    return c.w[m * c.K + k];  // weight viewed as [OC, IC*KH*KW]
  }
  // im2col sample: column n = (b*OH + oh)*OW + ow, row kk = (ic*KH + kh)*KW + kw.
  __device__ __forceinline__ float load_b(int64_t kk, int64_t n) const {
    const int ow = (int)(n % c.OW);
    const int64_t t = n / c.OW;
    const int oh = (int)(t % c.OH);
    const int b = (int)(t / c.OH);
    const int kw = (int)(kk % c.KW);
    const int64_t u = kk / c.KW;
    const int kh = (int)(u % c.KH);
    const int ic = (int)(u / c.KH);
    const int ih = oh * c.sH - c.pH + kh * c.dH;
    const int iw = ow * c.sW - c.pW + kw * c.dW;
    if (ih < 0 || ih >= c.H || iw < 0 || iw >= c.W) return 0.0f;
    return c.x[(((int64_t)b * c.IC + ic) * c.H + ih) * c.W + iw];
  }
  __device__ __forceinline__ void store_row4(int64_t m, int64_t n0, const float* acc) const {
    const float bv = c.bias ? c.bias[m] : 0.0f;
    const int64_t P = (int64_t)c.OH * c.OW;
    for (int j = 0; j < 4; ++j) {
      int64_t n = n0 + j;
      if (n >= c.N) break;
      const int64_t b = n / P, p = n - b * P;
      const float v = acc[j] + bv;
      c.out[(b * c.OC + m) * P + p] = c.relu ? fmaxf(v, 0.f) : v;
    }
  }
  __device__ __forceinline__ int64_t M() const { return c.M; }
  __device__ __forceinline__ int64_t N() const { return c.N; }
  __device__ __forceinline__ int64_t K() const { return c.K; }
};

template <class Ops>
__global__ __launch_bounds__(THREADS) void k_simt(const Ops ops) {
  ptx::griddep_wait();  // dependent launch: the kernel before this one has completed
  __shared__ __align__(16) float As[BK][BM];
  __shared__ __align__(16) float Bs[BK][BN];
  const int t = threadIdx.x;
  const int tx = t % 16, ty = t / 16;
  const int64_t M = ops.M(), N = ops.N(), K = ops.K();
  const int64_t tiles_n = (N + BN - 1) / BN;
  const int64_t m0 = ((int64_t)blockIdx.x / tiles_n) * BM, n0 = ((int64_t)blockIdx.x % tiles_n) * BN;
  float acc[4][4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[i][j] = 0.0f;

  for (int64_t k0 = 0; k0 < K; k0 += BK) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int e = t + i * THREADS;
      const int ml = e / BK, kl = e % BK;  // consecutive threads walk k (row-major A)
      const int64_t m = m0 + ml, k = k0 + kl;
      As[kl][ml] = (m < M && k < K) ? ops.load_a(m, k) : 0.0f;
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int e = t + i * THREADS;
      const int kl = e / BN, nl = e % BN;  // consecutive threads walk n
      const int64_t k = k0 + kl, n = n0 + nl;
      Bs[kl][nl] = (k < K && n < N) ? ops.load_b(k, n) : 0.0f;
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < BK; ++kk) {
      const float4 av = *reinterpret_cast<const float4*>(&As[kk][ty * 4]);
      const float4 bv = *reinterpret_cast<const float4*>(&Bs[kk][tx * 4]);
      const float ar[4] = {av.x, av.y, av.z, av.w};
      const float br[4] = {bv.x, bv.y, bv.z, bv.w};
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(ar[i], br[j], acc[i][j]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int64_t m = m0 + ty * 4 + i;
    if (m < M) ops.store_row4(m, n0 + tx * 4, acc[i]);
  }
}

// Small problems (few outputs, short K): T = 1, 2, 4 or 8 consecutive threads
// per output (T = ceil(K / 32) rounded up to a power of two), each summing one
// contiguous run of at most 32 k in k order with all of its loads in flight
// together; the T partial sums are then added pairwise by shuffles (xor 1,
// then 2, then 4: a fixed order).  No shared-memory staging (whose load /
// barrier rounds per k-tile are the whole cost at this size).
template <int T>
__global__ void __launch_bounds__(256) k_simt_small(const GemmArgs a) {
  ptx::griddep_wait();  // dependent launch: the kernel before this one has completed
  const int64_t tid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const int64_t e = tid / T;
  const int t = (int)(tid % T);
  const bool live = e < a.M * a.N;
  float acc = 0.0f;
  if (live) {
    const int64_t m = e / a.N, n = e - m * a.N;
    const int K = (int)a.K;  // <= kSmallK = 32 * 8
    const int kc = (K + T - 1) / T, k0 = t * kc, k1 = k0 + kc < K ? k0 + kc : K;
    const float* ar = a.mat1 + m * a.K;
    float av[32], bv[32];
#pragma unroll
    for (int j = 0; j < 32; ++j) {
      const int k = k0 + j;
      av[j] = k < k1 ? __ldg(ar + k) : 0.0f;
      bv[j] = k < k1 ? (a.b_kmajor ? __ldg(a.mat2 + n * a.K + k) : __ldg(a.mat2 + (int64_t)k * a.N + n))
                     : 0.0f;
    }
#pragma unroll
    for (int j = 0; j < 32; ++j)
      if (k0 + j < k1) acc = fmaf(av[j], bv[j], acc);
  }
#pragma unroll
  for (int x = 1; x < T; x <<= 1) acc += __shfl_xor_sync(0xffffffffu, acc, x);
  if (!live || t != 0) return;
  const int64_t n = e % a.N;
  const float v = a.read_self ? fmaf(a.alpha, acc, a.beta * a.self[a.self_2d ? e : n])
                              : a.alpha * acc;
  a.out[e] = a.relu ? fmaxf(v, 0.f) : v;
}

__global__ void k_fill_gemm(const GemmArgs a) {
  ptx::griddep_wait();  // dependent launch: the kernel before this one has completed
  const int64_t total = a.M * a.N;
  for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < total;
       e += (int64_t)gridDim.x * blockDim.x) {
    const int64_t n = e % a.N;
    float v = 0.0f;
    if (a.read_self) v = a.beta * (a.self_2d ? a.self[e] : a.self[n]);
    a.out[e] = a.relu ? fmaxf(v, 0.f) : v;
  }
}

__global__ void k_fill_conv(const ConvArgs c) {
  ptx::griddep_wait();  // dependent launch: the kernel before this one has completed
  const int64_t P = (int64_t)c.OH * c.OW;
  const int64_t total = (int64_t)c.B * c.OC * P;
  for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < total;
       e += (int64_t)gridDim.x * blockDim.x) {
    const int64_t oc = (e / P) % c.OC;
    const float v = c.bias ? c.bias[oc] : 0.0f;
    c.out[e] = c.relu ? fmaxf(v, 0.f) : v;
  }
}

// Direct convolution (the conv page's Problem paragraph: one thread per output
// element re-reading its receptive field from global memory, no reuse across
// threads; its "Before" line: scalar, or vec4 over the input channels when
// their count is a multiple of 4).  Consecutive threads take consecutive ow,
// so output stores and input loads along a row are coalesced.  fp32 FMA in
// (ic, kh, kw) order; the VEC4 form adds, per tap, the 4-term dot product of
// channels ic .. ic+3 (in NCHW / OIHW those are a plane apart, so the loads
// stay scalar).
template <bool VEC4>
__global__ void __launch_bounds__(256) k_direct_conv(const ConvArgs c) {
  ptx::griddep_wait();  // dependent launch: the kernel before this one has completed
  const int64_t P = (int64_t)c.OH * c.OW;
  const int64_t total = (int64_t)c.B * c.OC * P;
  const int64_t HW = (int64_t)c.H * c.W, taps = (int64_t)c.KH * c.KW;
  for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < total;
       e += (int64_t)gridDim.x * blockDim.x) {
    const int ow = (int)(e % c.OW);
    const int64_t t = e / c.OW;
    const int oh = (int)(t % c.OH);
    const int64_t u = t / c.OH;
    const int oc = (int)(u % c.OC);
    const int b = (int)(u / c.OC);
    const float* xb = c.x + (int64_t)b * c.IC * HW;
    const float* wr = c.w + (int64_t)oc * c.K;
    float acc = 0.0f;
    for (int ic = 0; ic < c.IC; ic += VEC4 ? 4 : 1)
      for (int kh = 0; kh < c.KH; ++kh) {
        const int ih = oh * c.sH - c.pH + kh * c.dH;
        if (ih < 0 || ih >= c.H) continue;
        for (int kw = 0; kw < c.KW; ++kw) {
          const int iw = ow * c.sW - c.pW + kw * c.dW;
          if (iw < 0 || iw >= c.W) continue;
          const float* wp = wr + (ic * c.KH + kh) * c.KW + kw;
          const float* xp = xb + ic * HW + (int64_t)ih * c.W + iw;
          if (VEC4) {  // the 4 channels ic .. ic+3 as one 4-term dot product
            float d = __ldg(wp) * __ldg(xp);
            d = fmaf(__ldg(wp + taps), __ldg(xp + HW), d);
            d = fmaf(__ldg(wp + 2 * taps), __ldg(xp + 2 * HW), d);
            d = fmaf(__ldg(wp + 3 * taps), __ldg(xp + 3 * HW), d);
            acc += d;
          } else {
            acc = fmaf(__ldg(wp), __ldg(xp), acc);
          }
        }
      }
    const float v = acc + (c.bias ? __ldg(c.bias + oc) : 0.0f);
    c.out[e] = c.relu ? fmaxf(v, 0.f) : v;
  }
}

unsigned fill_blocks(int64_t total) {
  int64_t b = (total + 255) / 256;
  int64_t cap = (int64_t)device_sm_count() * 8;
  return (unsigned)(b < cap ? (b > 0 ? b : 1) : cap);
}

}  // namespace

// Up to this many outputs and k, the addmm takes k_simt_small.
constexpr int64_t kSmallOutputs = 1 << 16, kSmallK = 256;

// One CTA per 64x64 output tile, linear tile index (no per-dimension grid cap).
static bool simt_grid(int64_t M, int64_t N, unsigned* blocks) {
  const int64_t tiles = ((M + BM - 1) / BM) * ((N + BN - 1) / BN);
  if (tiles > 0x7fffffffLL) return false;
  *blocks = (unsigned)tiles;
  return true;
}

cudaError_t launch_simt_gemm(const GemmArgs& a, cudaStream_t s) {
  if (a.M * a.N <= kSmallOutputs && a.K <= kSmallK) {
    const int T = a.K <= 32 ? 1 : (a.K <= 64 ? 2 : (a.K <= 128 ? 4 : 8));
    const unsigned blocks = (unsigned)((a.M * a.N * T + 255) / 256);
    cudaError_t e;
    switch (T) {
      case 1: e = launch_after_previous(k_simt_small<1>, dim3(blocks), dim3(256), 0, s, a); break;
      case 2: e = launch_after_previous(k_simt_small<2>, dim3(blocks), dim3(256), 0, s, a); break;
      case 4: e = launch_after_previous(k_simt_small<4>, dim3(blocks), dim3(256), 0, s, a); break;
      default: e = launch_after_previous(k_simt_small<8>, dim3(blocks), dim3(256), 0, s, a); break;
    }
    note_launch();
    note_kernel_name("k_simt_small");
    return e;
  }
  unsigned grid;
  if (!simt_grid(a.M, a.N, &grid)) return cudaErrorInvalidConfiguration;
  const cudaError_t e =
      launch_after_previous(k_simt<GemmOperands>, dim3(grid), dim3(THREADS), 0, s, GemmOperands{a});
  note_launch();
  note_kernel_name("k_simt<gemm>");
  return e;
}

cudaError_t launch_simt_conv(const ConvArgs& c, cudaStream_t s) {
  unsigned grid;
  if (!simt_grid(c.M, c.N, &grid)) return cudaErrorInvalidConfiguration;
  const cudaError_t e =
      launch_after_previous(k_simt<ConvOperands>, dim3(grid), dim3(THREADS), 0, s, ConvOperands{c});
  note_launch();
  note_kernel_name("k_simt<conv>");
  return e;
}

cudaError_t launch_fill_gemm(const GemmArgs& a, cudaStream_t s) {
  const cudaError_t e =
      launch_after_previous(k_fill_gemm, dim3(fill_blocks(a.M * a.N)), dim3(256), 0, s, a);
  note_launch();
  note_kernel_name("k_fill_gemm");
  return e;
}

cudaError_t launch_direct_conv(const ConvArgs& c, cudaStream_t s) {
  const int64_t total = (int64_t)c.B * c.OC * c.OH * c.OW;
  const int64_t cap = (int64_t)device_sm_count() * 16, blocks = (total + 255) / 256;
  // as in the pages' direct kernel: the 4-channel form when IC % 4 == 0
  const dim3 grid((unsigned)(blocks < cap ? blocks : cap));
  const cudaError_t e =
      c.IC % 4 == 0 ? launch_after_previous(k_direct_conv<true>, grid, dim3(256), 0, s, c)
                    : launch_after_previous(k_direct_conv<false>, grid, dim3(256), 0, s, c);
  note_launch();
  note_kernel_name("k_direct_conv");
  return e;
}

cudaError_t launch_fill_conv(const ConvArgs& c, cudaStream_t s) {
  const cudaError_t e = launch_after_previous(
      k_fill_conv, dim3(fill_blocks((int64_t)c.B * c.OC * c.OH * c.OW)), dim3(256), 0, s, c);
  note_launch();
  note_kernel_name("k_fill_conv");
  return e;
}

}  // namespace imc
