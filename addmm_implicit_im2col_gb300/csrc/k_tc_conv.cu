// tcgen05 tensor-core conv2d (groups == 1, NCHW) as an implicit-im2col GEMM.
//
// Semantics: ExecuTorch WebGPU "et_vk conv2d: route standard (groups==1) conv
// through an im2col tiled GEMM", Solution and Implementation paragraphs:
// M = OC, N = B*OH*OW, K = IC*KH*KW; the weight is the [OC, K] operand; the
// input is im2col-sampled on the fly (n -> (b, oh, ow), kk -> (ic, kh, kw),
// ih = oh*sH - pH + kh*dH, likewise iw, out-of-range taps read 0); bias per
// output channel; NCHW output.
//
// Layout for sm_103a:
//   pre-pass    the weight is written once per call as zero-padded rows of Kp
//               (K rounded up to 4) fp32 -- hi part and, for 3xTF32, lo part --
//               so that its tiles can be TMA-loaded whatever K is
//   warp 8      TMA producer of the weight tiles (MH x 128 rows x 16, 64B swizzle)
//   warps 0-7   im2col producers: thread t owns column n = n0 + t of the tile;
//               per k-block of 16 it gathers its 16 taps (loads for the next
//               k-block are issued before the current one is stored), splits
//               them into TF32 hi / lo and writes them as one K-major row of
//               the B tiles
//   warp 9      TMEM owner + MMA issuer: MH 128-row halves share every B tile;
//               3 MMAs per k-step (A_lo*B_hi + A_hi*B_lo + A_hi*B_hi) or 1
//   warps 10-13 epilogue: tcgen05.ld, 32x32 transpose through shared memory,
//               acc + bias[oc] to NCHW rows
// One persistent CTA per SM; the tile width BN (multiple of 16, up to
// BN_MAX) is chosen per problem so the tiles fill the SMs in few waves.
// Every barrier wait is bounded (see tc_common.cuh).
#include <mutex>

#include "imc.h"
#include "imc_internal.cuh"
#include "tc_common.cuh"

namespace imc {
namespace {

using namespace tc;

constexpr int BK = 16;           // fp32 per k-block: one 64-byte swizzle row
constexpr int KSTEPS = BK / UK;  // 2
constexpr int HALF_BYTES = BM * BK * 4;  // one 128-row A tile: 8 KB
constexpr int PRODUCERS = 256;           // im2col producer threads (warps 0-7)
constexpr int TMA_WARP = 8, MMA_WARP = 9, EPI_WARP0 = 10, THREADS = 14 * 32;

__device__ int g_watchdog_conv;

template <int MH, bool THREE>
struct Cfg {
  static constexpr int BN_MAX = MH == 2 ? 192 : 256;
  static constexpr int B_BYTES = BN_MAX * BK * 4;
  static constexpr int A_HI = 0;
  static constexpr int A_LO = MH * HALF_BYTES;
  static constexpr int B_HI = (THREE ? 2 : 1) * MH * HALF_BYTES;
  static constexpr int B_LO = B_HI + B_BYTES;
  static constexpr int STAGE = B_HI + (THREE ? 2 : 1) * B_BYTES;
  static constexpr int STAGES = (196608 / STAGE) < MAX_STAGES ? (196608 / STAGE) : MAX_STAGES;
  static constexpr int SMEM = 1024 + STAGES * STAGE + EPI_BYTES + (int)sizeof(Ctl);
  static constexpr int NBUF = MH == 2 ? 1 : 2;  // accumulator buffers in TMEM
  static_assert(STAGES >= 3, "pipeline depth");
  static_assert(SMEM <= 232448, "shared memory");
};

// ------------------------------------------------------- weight pre-pass
// w_hi[oc*Kp + k] = tf32 part of w[oc*K + k] (0 for k >= K), w_lo the rest.
__global__ void k_prep_w(const float* __restrict__ w, int64_t OC, int64_t K, int64_t Kp,
                         float* __restrict__ w_hi, float* __restrict__ w_lo) {
  const int64_t total = OC * Kp;
  for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < total;
       e += (int64_t)gridDim.x * blockDim.x) {
    const int64_t oc = e / Kp, k = e - oc * Kp;
    const float v = k < K ? __ldg(w + oc * K + k) : 0.0f;
    if (w_lo) {
      w_hi[e] = tf32_hi(v);
      w_lo[e] = tf32_lo(v);
    } else {
      w_hi[e] = v;
    }
  }
}

struct Store {
  const ConvArgs& c;
  int64_t m0, n0;
  int bn;
  __device__ __forceinline__ float4 load(int r, int) const {
    const int64_t m = m0 + r;
    const float bv = (c.bias && m < c.M) ? __ldg(c.bias + m) : 0.0f;
    return make_float4(bv, bv, bv, bv);
  }
  __device__ __forceinline__ void operator()(int r, int col, float4 v, float4 b4) const {
    const int64_t m = m0 + r, n = n0 + col;
    if (col >= bn || m >= c.M || n >= c.N) return;
    const float bv = b4.x;
    const int64_t P = (int64_t)c.OH * c.OW;
    float4 o4 = make_float4(v.x + bv, v.y + bv, v.z + bv, v.w + bv);
    if (c.relu) o4 = make_float4(fmaxf(o4.x, 0.f), fmaxf(o4.y, 0.f), fmaxf(o4.z, 0.f), fmaxf(o4.w, 0.f));
    if (c.vec_out && col + 3 < bn) {  // P % 4 == 0: n .. n+3 lie in one image
      const int64_t b = n / P, p = n - b * P;
      *reinterpret_cast<float4*>(c.out + (b * c.OC + m) * P + p) = o4;
    } else {
      const float vv[4] = {o4.x, o4.y, o4.z, o4.w};
      for (int j = 0; j < 4 && n + j < c.N && col + j < bn; ++j) {
        const int64_t nn = n + j, b = nn / P, p = nn - b * P;
        c.out[(b * c.OC + m) * P + p] = vv[j];
      }
    }
  }
};

// One im2col column (output position n) and the running tap (ic, kh, kw)
// of kk = k0, kept across k-blocks so no division is needed per k-block.
struct Column {
  const float* xb;  // image b of x
  int ih0, iw0;     // oh*sH - pH, ow*sW - pW
  bool ok;
};
struct Tap {
  int ic, kh, kw;
};

// The 16 taps kk = k0 .. k0+15 of one column (zero outside the image and for
// kk >= K); advances `tap` by 16.
__device__ __forceinline__ void gather(const ConvArgs& c, const Column& col, int k0, int K,
                                       Tap& tap, float (&v)[BK]) {
#pragma unroll
  for (int j = 0; j < BK; ++j) {
    const int ih = col.ih0 + tap.kh * c.dH, iw = col.iw0 + tap.kw * c.dW;
    const bool in = col.ok && (k0 + j < K) && (unsigned)ih < (unsigned)c.H &&
                    (unsigned)iw < (unsigned)c.W;
    v[j] = in ? __ldg(col.xb + ((tap.ic * c.H + ih) * c.W + iw)) : 0.0f;
    if (++tap.kw == c.KW) {
      tap.kw = 0;
      if (++tap.kh == c.KH) {
        tap.kh = 0;
        ++tap.ic;
      }
    }
  }
}

template <int MH, bool THREE>
__global__ void __launch_bounds__(THREADS, 1)
    k_tc_conv(const __grid_constant__ CUtensorMap tmWh, const __grid_constant__ CUtensorMap tmWl,
              const ConvArgs c, const int num_m, const int num_n, const int bn) {
  using C = Cfg<MH, THREE>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  float* epi = reinterpret_cast<float*>(smem + C::STAGES * C::STAGE);
  Ctl* ctl = reinterpret_cast<Ctl*>(smem + C::STAGES * C::STAGE + EPI_BYTES);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int num_tiles = num_m * num_n;
  const int K = (int)c.K;
  const int num_kb = (K + BK - 1) / BK;
  int* wd = &g_watchdog_conv;

  if (threadIdx.x == 0) init_barriers(ctl, C::STAGES, PRODUCERS + 1, 1);
  if (warp == TMA_WARP && lane == 0) {
    ptx::tma_prefetch_desc(&tmWh);
    if (THREE) ptx::tma_prefetch_desc(&tmWl);
  }
  if (warp == MMA_WARP) {
    ptx::tmem_alloc(&ctl->tmem_base, TMEM_COLS);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = ctl->tmem_base;
  volatile int* abort = &ctl->abort;

  if (warp < 8) {
    // ----------------------------------------------------- im2col producers
    const int pt = threadIdx.x;
    const int P = c.OH * c.OW;
    int s = 0;
    uint32_t ph = 0;
    bool ok = true;
    for (int t = blockIdx.x; t < num_tiles && ok; t += gridDim.x) {
      const int nt = t / num_m;  // tiles of one column block are adjacent
      const int64_t n = (int64_t)nt * bn + pt;
      Column col{c.x, 0, 0, pt < bn && n < c.N};
      if (col.ok) {
        const int b = (int)(n / P), p = (int)(n - (int64_t)b * P);
        const int oh = p / c.OW, ow = p - oh * c.OW;
        col.ih0 = oh * c.sH - c.pH;
        col.iw0 = ow * c.sW - c.pW;
        col.xb = c.x + (int64_t)b * c.IC * c.H * c.W;
      }
      // Three register buffers, rotated by unrolling (copying a buffer whose
      // loads are in flight would wait for them): the taps of k-blocks kb+1
      // and kb+2 are in flight while k-block kb is stored.
      Tap tap{0, 0, 0};
      auto next = [&](int kb, float (&v)[BK]) { gather(c, col, kb * BK, K, tap, v); };
      float va[BK], vb[BK], vc[BK];
      auto store = [&](const float (&v)[BK]) -> bool {
        if (!warp_wait_bar(&ctl->empty[s], ph ^ 1u, abort, kSiteProducerEmpty, wd)) return false;
        if (pt < bn) {
          uint8_t* row = smem + s * C::STAGE + C::B_HI + sw64_row_base(pt);
#pragma unroll
          for (int j = 0; j < BK / 4; ++j) {
            const float4 q = make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
            const int off = sw64_unit(pt, j);
            if (THREE) {
              *reinterpret_cast<float4*>(row + off) = tf32_hi4(q);
              *reinterpret_cast<float4*>(row + (C::B_LO - C::B_HI) + off) = tf32_lo4(q);
            } else {
              *reinterpret_cast<float4*>(row + off) = q;
            }
          }
        }
        ptx::fence_proxy_async_smem();
        ptx::mbar_arrive(&ctl->full[s]);
        if (++s == C::STAGES) {
          s = 0;
          ph ^= 1u;
        }
        return true;
      };
      next(0, va);
      if (num_kb > 1) next(1, vb);
      for (int kb = 0; kb < num_kb && ok; kb += 3) {
        if (kb + 2 < num_kb) next(kb + 2, vc);
        if (!(ok = store(va)) || kb + 1 >= num_kb) break;
        if (kb + 3 < num_kb) next(kb + 3, va);
        if (!(ok = store(vb)) || kb + 2 >= num_kb) break;
        if (kb + 4 < num_kb) next(kb + 4, vb);
        ok = store(vc);
      }
    }
  } else if (warp == TMA_WARP) {
    // ------------------------------------------------ weight TMA producer
    if (lane == 0) {
      const uint32_t tx = (uint32_t)((THREE ? 2 : 1) * MH * HALF_BYTES);
      int s = 0, issued = 0;
      uint32_t ph = 0;
      for (int t = blockIdx.x; t < num_tiles && !*abort; t += gridDim.x) {
        const int mt = t % num_m;
        for (int kb = 0; kb < num_kb; ++kb) {
          if (!wait_bar(&ctl->empty[s], ph ^ 1u, abort, kSiteProducerEmpty, wd)) break;
          uint8_t* st = smem + s * C::STAGE;
          ptx::mbar_arrive_expect_tx(&ctl->full[s], tx);
#pragma unroll
          for (int h = 0; h < MH; ++h) {
            ptx::tma_load_2d(st + C::A_HI + h * HALF_BYTES, &tmWh, &ctl->full[s], kb * BK,
                             mt * MH * BM + h * BM);
            if (THREE)
              ptx::tma_load_2d(st + C::A_LO + h * HALF_BYTES, &tmWl, &ctl->full[s], kb * BK,
                               mt * MH * BM + h * BM);
          }
          ++issued;
          if (++s == C::STAGES) {
            s = 0;
            ph ^= 1u;
          }
        }
      }
      for (int j = (issued > C::STAGES ? issued - C::STAGES : 0); j < issued; ++j)
        drain_wait(&ctl->full[j % C::STAGES], (uint32_t)((j / C::STAGES) & 1));
    }
  } else if (warp == MMA_WARP) {
    // --------------------------------------------------------- MMA issuer
    if (lane == 0) {
      const uint32_t idesc = ptx::idesc_tf32(BM, (uint32_t)bn, false, false);
      int s = 0, tl = 0;
      uint32_t ph = 0;
      for (int t = blockIdx.x; t < num_tiles; t += gridDim.x, ++tl) {
        const int buf = tl % C::NBUF;
        const uint32_t use = (uint32_t)(tl / C::NBUF);
        if (!wait_bar(&ctl->acce[buf], (use & 1u) ^ 1u, abort, kSiteMmaAccEmpty, wd)) break;
        ptx::tc_fence_after();
        bool ok = true;
        for (int kb = 0; kb < num_kb; ++kb) {
          if (!wait_bar(&ctl->full[s], ph, abort, kSiteMmaOperands, wd)) {
            ok = false;
            break;
          }
          ptx::tc_fence_after();
          const uint32_t st = ptx::smem_addr(smem + s * C::STAGE);
#pragma unroll
          for (int h = 0; h < MH; ++h) {
            const uint32_t d = tmem + (uint32_t)(buf + h) * 256u;
#pragma unroll
            for (int ks = 0; ks < KSTEPS; ++ks) {
              const uint64_t ah = sw64_desc(st + C::A_HI + h * HALF_BYTES, ks);
              const uint64_t bh = sw64_desc(st + C::B_HI, ks);
              const uint32_t acc = (kb > 0 || ks > 0) ? 1u : 0u;
              if (THREE) {
                const uint64_t al = sw64_desc(st + C::A_LO + h * HALF_BYTES, ks);
                const uint64_t bl = sw64_desc(st + C::B_LO, ks);
                ptx::mma_tf32(d, al, bh, idesc, acc);
                ptx::mma_tf32(d, ah, bl, idesc, 1u);
                ptx::mma_tf32(d, ah, bh, idesc, 1u);
              } else {
                ptx::mma_tf32(d, ah, bh, idesc, acc);
              }
            }
          }
          ptx::mma_commit(&ctl->empty[s]);
          if (++s == C::STAGES) {
            s = 0;
            ph ^= 1u;
          }
        }
        if (!ok) break;
        ptx::mma_commit(&ctl->accf[buf]);
      }
      ptx::mma_commit(&ctl->drain);
      drain_wait(&ctl->drain, 0);
    }
    __syncwarp();
  } else {
    // ----------------------------------------------------------- epilogue
    const int q = warp & 3;
    float* stage = epi + (warp - EPI_WARP0) * 32 * EPI_PITCH;
    int tl = 0;
    for (int t = blockIdx.x; t < num_tiles; t += gridDim.x, ++tl) {
      const int buf = tl % C::NBUF;
      const uint32_t use = (uint32_t)(tl / C::NBUF);
      if (!warp_wait_bar(&ctl->accf[buf], use & 1u, abort, kSiteEpilogueAccFull, wd)) break;
      ptx::tc_fence_after();
      const int mt = t % num_m, nt = t / num_m;
#pragma unroll 1
      for (int h = 0; h < MH; ++h)
        drain_accumulator(tmem, q, (uint32_t)(buf + h) * 256u, (bn + 31) & ~31, stage,
                          Store{c, (int64_t)mt * MH * BM + h * BM, (int64_t)nt * bn, bn});
      ptx::tc_fence_before();
      ptx::mbar_arrive(&ctl->acce[buf]);
    }
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (warp == MMA_WARP) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, TMEM_COLS);
  }
}

// ------------------------------------------------------------------- host
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
    else
      cudaGetLastError();
  });
  return fn;
}

// Padded weight plane [OC, Kp] -> tensor map, box {16, 128}, 64-byte swizzle.
bool encode_w(CUtensorMap* m, const float* base, uint64_t Kp, uint64_t OC) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {Kp, OC};
  const cuuint64_t strides[1] = {Kp * 4};
  const cuuint32_t box[2] = {(cuuint32_t)BK, (cuuint32_t)BM};
  const cuuint32_t es[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float*>(base), dims, strides, box,
            es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Tile width: multiple of 16 up to bn_max minimising waves * (bn + 16).
int pick_bn(int64_t num_m, int64_t N, int bn_max, int sms) {
  int best = bn_max;
  int64_t best_cost = INT64_MAX;
  for (int bn = bn_max; bn >= 32; bn -= 16) {
    const int64_t tiles = num_m * ((N + bn - 1) / bn);
    const int64_t cost = ((tiles + sms - 1) / sms) * (bn + 16);
    if (cost < best_cost) {
      best_cost = cost;
      best = bn;
    }
  }
  return best;
}

constexpr int kMaxDev = 64;

template <int MH, bool THREE>
cudaError_t run(const ConvArgs& c, const float* w_hi, const float* w_lo, int64_t Kp,
                cudaStream_t s) {
  using Cf = Cfg<MH, THREE>;
  static bool ready[kMaxDev];
  auto k = k_tc_conv<MH, THREE>;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev >= kMaxDev || !ready[dev]) {
    e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, Cf::SMEM);
    if (e != cudaSuccess) return e;
    if (dev < kMaxDev) ready[dev] = true;
  }
  CUtensorMap th, tl;
  if (!encode_w(&th, w_hi, (uint64_t)Kp, (uint64_t)c.OC) ||
      !encode_w(&tl, THREE ? w_lo : w_hi, (uint64_t)Kp, (uint64_t)c.OC))
    return cudaErrorInvalidValue;
  const int sms = device_sm_count();
  const int num_m = (int)((c.M + MH * BM - 1) / (MH * BM));
  const int bn = pick_bn(num_m, c.N, Cf::BN_MAX, sms);
  const int num_n = (int)((c.N + bn - 1) / bn);
  const int tiles = num_m * num_n;
  const int grid = tiles < sms ? tiles : sms;
  k<<<grid, THREADS, Cf::SMEM, s>>>(th, tl, c, num_m, num_n, bn);
  note_launch();
  return cudaGetLastError();
}

int64_t padded_k(int64_t K) { return (K + 3) / 4 * 4; }

}  // namespace

bool tc_conv_supported(const ConvArgs& c) {
  const double tiles = (double)((c.M + BM - 1) / BM) * (double)((c.N + 31) / 32);
  return tiles < 2147483647.0 && encode_fn() != nullptr;
}

size_t tc_conv_workspace_bytes(int64_t OC, int64_t K, bool three_pass) {
  return (three_pass ? 2u : 1u) * (size_t)OC * (size_t)padded_k(K) * sizeof(float);
}

cudaError_t launch_tc_conv(const ConvArgs& c, bool three_pass, void* workspace, cudaStream_t s) {
  if (!tc_conv_supported(c) || !workspace) return cudaErrorNotSupported;
  const int64_t Kp = padded_k(c.K);
  float* w_hi = static_cast<float*>(workspace);
  float* w_lo = three_pass ? w_hi + c.OC * Kp : nullptr;
  const int64_t total = c.OC * Kp;
  const int64_t cap = (int64_t)device_sm_count() * 8;
  const int64_t blocks = (total + 255) / 256;
  k_prep_w<<<(unsigned)(blocks < cap ? blocks : cap), 256, 0, s>>>(c.w, c.OC, c.K, Kp, w_hi,
                                                                   w_lo);
  note_launch();
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  if (c.M > BM)
    return three_pass ? run<2, true>(c, w_hi, w_lo, Kp, s) : run<2, false>(c, w_hi, w_lo, Kp, s);
  return three_pass ? run<1, true>(c, w_hi, w_lo, Kp, s) : run<1, false>(c, w_hi, w_lo, Kp, s);
}

cudaError_t conv_take_watchdog(int* value) {
  cudaError_t e = cudaMemcpyFromSymbol(value, g_watchdog_conv, sizeof(int));
  if (e != cudaSuccess) return e;
  const int zero = 0;
  return cudaMemcpyToSymbol(g_watchdog_conv, &zero, sizeof(int));
}

}  // namespace imc
