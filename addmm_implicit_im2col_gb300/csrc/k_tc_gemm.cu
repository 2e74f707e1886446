// tcgen05 tensor-core addmm: out = beta*self + alpha*(mat1 @ mat2), fp32.
//
// Semantics: ExecuTorch WebGPU "Add optimized addmm op", Solution and
// Implementation paragraphs (mat2 read as mat2[k*N + n]; self broadcast from
// [N] or given as [M,N]; epilogue beta*self + alpha*acc).  The page's WGSL
// kernel stages 32x32 slabs of both operands in workgroup memory and loops
// over ceil(K/32) k-tiles; the same tiled GEMM is laid out here for sm_103a.
//
// A kind::tf32 MMA on this GPU reads its shared-memory operands K-major only.
// mat1 [M,K] already is; mat2 [K,N] is N-contiguous, so a pre-pass
// (k_prep_b) writes it once per call, transposed, into a caller- or
// pool-provided workspace: Bt_hi[n][k] and Bt_lo[n][k] (3xTF32) or Bt[n][k]
// (1xTF32), rows of Kp = K rounded up to 4 floats.  TMA needs 16-byte aligned
// rows: when K % 4 != 0 (or mat1 is not 16-byte aligned) mat1 is copied
// into the workspace with rows of Kp floats too (k_pad_rows).  The tensor maps
// keep the extent K, so the TMA reads zeros for k >= K and the columns
// between K and Kp are never read.  The main kernel is then a plain pipeline:
//
//   warp 0      TMA producer: mat1 tile (128 x 16), Bt_hi / Bt_lo tiles (BN x 16),
//               64-byte swizzle, into a 4-stage ring (5 for the TS form, 8 for
//               1xTF32)
//   warps 6-9   (3xTF32) A_lo = mat1 - tf32(mat1); in the TS form each thread
//               takes one row of the mat1 tile, splits it and writes A_hi and
//               A_lo to the stage's TMEM columns, otherwise A_lo goes to a
//               shared-memory tile elementwise
//   warp 1      TMEM owner + MMA issuer: per 8-deep k-step
//               A_lo*B_hi + A_hi*B_lo + A_hi*B_hi into an fp32 TMEM accumulator;
//               the TS form reads A from TMEM (measured: 94 % of the TF32 MMA
//               rate at N = 256, against 80 % with both operands in shared
//               memory) and has one accumulator, the other form reads the raw
//               mat1 tile as A_hi (the tensor core drops the 13 low mantissa
//               bits itself) and double-buffers the accumulator.  The TS form
//               is used when a unit runs enough k-blocks that the faster MMAs
//               outweigh the drain of the single accumulator (see kTsMinKb)
//   warps 2-5   epilogue: tcgen05.ld, then beta*self + alpha*acc: a whole
//               tile with N % 4 == 0 and no [M,N] self leaves by 2-D TMA
//               stores of 32 x 32 blocks from a 128-byte-swizzled staging
//               block (beta*self of a vector self staged once per tile in
//               shared memory); otherwise a 32x32 transpose through shared
//               memory and 16-byte row-segment stores
//
// One persistent CTA per SM walks 128 x BN tiles in a grouped raster; BN (32
// to 256: a multiple of 32, or of 16 from 112 up when K is not split) is
// picked per problem to fill the SMs with few waves.  The MMA issuer keeps
// its operand descriptors as running values (a few instructions per k-block
// in the issuing thread are on the pipeline's critical path).  Every barrier
// wait is bounded (see tc_common.cuh).
#include <atomic>
#include <mutex>

#include "imc.h"
#include "imc_internal.cuh"
#include "tc_common.cuh"

namespace imc {
namespace {

using namespace tc;

constexpr int BK = 16;           // fp32 per k-block: one 64-byte swizzle row
static_assert(BK == 2 * UK, "a k-block is two MMA k-steps");
constexpr int BN_MAX = 256;
constexpr int A_BYTES = BM * BK * 4;      // 8 KB
constexpr int B_BYTES = BN_MAX * BK * 4;  // 16 KB
constexpr uint32_t ACC_STRIDE = 256;      // TMEM columns between the two accumulators

constexpr int SROW_BYTES = BN_MAX * 4;  // beta * self[n0 ..) of the tile, for a vector self

struct Layout {
  int a, a_lo, b_hi, b_lo, bytes, stages;
};
constexpr Layout kL3 = {0, A_BYTES, 2 * A_BYTES, 2 * A_BYTES + B_BYTES, 2 * (A_BYTES + B_BYTES), 4};
constexpr Layout kL1 = {0, 0, A_BYTES, 0, A_BYTES + B_BYTES, 8};
// 3xTF32 with A from TMEM: no A_lo tile in shared memory
constexpr Layout kLts = {0, 0, A_BYTES, A_BYTES + B_BYTES, A_BYTES + 2 * B_BYTES, 5};
constexpr int smem_bytes(const Layout& L) {
  return 1024 + L.stages * L.bytes + EPI_BYTES + SROW_BYTES + (int)sizeof(Ctl);
}
static_assert(smem_bytes(kL3) <= 232448 && smem_bytes(kL1) <= 232448 &&
                  smem_bytes(kLts) <= 232448, "shared memory");
static_assert(kL1.stages <= MAX_STAGES, "stages");
// A-from-TMEM form: one accumulator (columns 0-255), A stages of 32 columns
// (hi 0-15, lo 16-31) from column 256.
constexpr uint32_t TS_A_COL0 = 256, TS_A_STAGE_COLS = 32;
static_assert(TS_A_COL0 + kLts.stages * TS_A_STAGE_COLS <= TMEM_COLS, "TMEM");
// K-blocks per unit from which the A-from-TMEM form is used: it runs the MMAs
// faster but holds the MMA while the single accumulator drains, which is slow
// when the epilogue reads an [M,N] self (measured on 32768x1024x1024: 305 us
// with the double-buffered form, 443 us with this one), cheap otherwise.
constexpr int kTsMinKb = 96, kTsMinKbLightEpilogue = 32;

__device__ int g_watchdog_gemm;

// ----------------------------------------------------------- mat2 pre-pass
// Bt_hi[n*ldk + k] = tf32 part of mat2[k*N + n] and Bt_lo[n*ldk + k] = the
// rest (3xTF32), or Bt_hi = mat2 transposed (bt_lo == nullptr); ldk >= K.
// 32x32 tiles through shared memory: reads and writes are 128-byte rows.
__global__ void __launch_bounds__(256) k_prep_b(const float* __restrict__ mat2, int64_t K,
                                                int64_t N, int64_t ldk, float* __restrict__ bt_hi,
                                                float* __restrict__ bt_lo) {
  __shared__ float tile[32][33];
  ptx::griddep_wait();    // the kernel before this one has completed
  ptx::griddep_launch();  // the main kernel may start its prologue
  const int tx = threadIdx.x, ty = threadIdx.y;
  const int64_t tiles_n = (N + 31) / 32, tiles = tiles_n * ((K + 31) / 32);
  for (int64_t t = blockIdx.x; t < tiles; t += gridDim.x) {
    const int64_t k0 = (t / tiles_n) * 32, n0 = (t % tiles_n) * 32;
#pragma unroll
    for (int i = ty; i < 32; i += 8) {
      const int64_t k = k0 + i, n = n0 + tx;
      tile[i][tx] = (k < K && n < N) ? __ldg(mat2 + k * N + n) : 0.0f;
    }
    __syncthreads();
#pragma unroll
    for (int i = ty; i < 32; i += 8) {
      const int64_t n = n0 + i, k = k0 + tx;
      if (n < N && k < K) {
        const float v = tile[tx][i];
        if (bt_lo) {
          bt_hi[n * ldk + k] = tf32_hi(v);
          bt_lo[n * ldk + k] = tf32_lo(v);
        } else {
          bt_hi[n * ldk + k] = v;
        }
      }
    }
    __syncthreads();
  }
}

// The same for N % 4 == 0 and a 16-byte aligned mat2 (ldk % 4 == 0): 64 x 64
// tiles, 16-byte loads along N and 16-byte stores along K (a group of four k
// is written whole when its first k < K; ldk >= K rounded up to 4).
__global__ void __launch_bounds__(256) k_prep_b4(const float* __restrict__ mat2, int64_t K,
                                                 int64_t N, int64_t ldk,
                                                 float* __restrict__ bt_hi,
                                                 float* __restrict__ bt_lo) {
  __shared__ float tile[64][65];
  ptx::griddep_wait();    // the kernel before this one has completed
  ptx::griddep_launch();  // the main kernel may start its prologue
  const int t = threadIdx.x, r0 = t >> 4, q4 = t & 15;
  const int64_t tiles_n = (N + 63) / 64, tiles = tiles_n * ((K + 63) / 64);
  for (int64_t tt = blockIdx.x; tt < tiles; tt += gridDim.x) {
    const int64_t k0 = (tt / tiles_n) * 64, n0 = (tt % tiles_n) * 64;
#pragma unroll
    for (int i = 0; i < 4; ++i) {  // rows k0 + r, columns n0 + 4*q4 .. +3
      const int r = r0 + 16 * i;
      const int64_t k = k0 + r, n = n0 + 4 * q4;
      const float4 v = (k < K && n < N) ? __ldg(reinterpret_cast<const float4*>(mat2 + k * N + n))
                                        : make_float4(0.f, 0.f, 0.f, 0.f);
      tile[r][4 * q4] = v.x;
      tile[r][4 * q4 + 1] = v.y;
      tile[r][4 * q4 + 2] = v.z;
      tile[r][4 * q4 + 3] = v.w;
    }
    __syncthreads();
#pragma unroll
    for (int i = 0; i < 4; ++i) {  // output rows n0 + r, columns k0 + 4*q4 .. +3
      const int r = r0 + 16 * i;
      const int64_t n = n0 + r, k = k0 + 4 * q4;
      if (n < N && k < K) {
        const float4 v = make_float4(tile[4 * q4][r], tile[4 * q4 + 1][r], tile[4 * q4 + 2][r],
                                     tile[4 * q4 + 3][r]);
        if (bt_lo) {
          *reinterpret_cast<float4*>(bt_hi + n * ldk + k) = tf32_hi4(v);
          *reinterpret_cast<float4*>(bt_lo + n * ldk + k) = tf32_lo4(v);
        } else {
          *reinterpret_cast<float4*>(bt_hi + n * ldk + k) = v;
        }
      }
    }
    __syncthreads();
  }
}

// linear: the weight w[N,K] is already K-major and serves as B_hi as it is
// (the tensor core truncates to TF32); 3xTF32 needs only w_lo = w - tf32(w).
// 16-byte elements, four in flight per thread; the grid (at most two blocks
// per SM) stays resident beside the main kernel's CTAs, so the main kernel,
// launched as its dependent, starts without waiting for pre-pass blocks.
__global__ void __launch_bounds__(256) k_prep_blo(const float4* __restrict__ w, int64_t total4,
                                                  float4* __restrict__ w_lo) {
  ptx::griddep_wait();  // the kernel before this one has completed
  ptx::griddep_launch();
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total4; i += 4 * stride) {
    float4 v[4];
#pragma unroll
    for (int j = 0; j < 4; ++j)
      v[j] = i + j * stride < total4 ? __ldg(w + i + j * stride) : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int j = 0; j < 4; ++j)
      if (i + j * stride < total4) w_lo[i + j * stride] = tf32_lo4(v[j]);
  }
}

// A [rows, K] operand whose rows are not 16-byte aligned (K % 4 != 0 or an
// unaligned base) copied to rows of ld floats: dst[r*ld + k] = src[r*K + k]
// for k < K (dst_lo, when given, gets the TF32 lo part and dst the value
// itself); the columns K .. ld-1 are left as they are (the TMA never reads
// them).  Work unit = 256 consecutive elements of one row (thread = one
// element: coalesced reads and writes); a block takes PAD_UNITS consecutive
// units at a time, all their loads before any store, so that enough reads are
// in flight to keep HBM busy (one 4-byte load per thread ran at half its
// bandwidth: 87.7 us for a 134 MB copy).  Rows are not 16-byte aligned, so
// the accesses stay 4 bytes wide.
constexpr int PAD_UNITS = 8;
__global__ void __launch_bounds__(256) k_pad_rows(const float* __restrict__ src, int64_t rows,
                                                  int64_t K, int64_t ld, float* __restrict__ dst,
                                                  float* __restrict__ dst_lo) {
  ptx::griddep_wait();  // the kernel before this one has completed
  ptx::griddep_launch();
  const int64_t cols_blocks = (K + 255) / 256, units = rows * cols_blocks;
  for (int64_t u0 = (int64_t)blockIdx.x * PAD_UNITS; u0 < units;
       u0 += (int64_t)gridDim.x * PAD_UNITS) {
    float v[PAD_UNITS];
    int64_t at[PAD_UNITS];  // destination index, -1: nothing to copy
    int64_t r = u0 / cols_blocks, cb = u0 - r * cols_blocks;
#pragma unroll
    for (int j = 0; j < PAD_UNITS; ++j) {
      const int64_t k = cb * 256 + threadIdx.x;
      const bool live = u0 + j < units && k < K;
      v[j] = live ? __ldg(src + r * K + k) : 0.0f;
      at[j] = live ? r * ld + k : -1;
      if (++cb == cols_blocks) {  // the next unit starts the next row
        cb = 0;
        ++r;
      }
    }
#pragma unroll
    for (int j = 0; j < PAD_UNITS; ++j) {
      if (at[j] < 0) continue;
      dst[at[j]] = v[j];
      if (dst_lo) dst_lo[at[j]] = tf32_lo(v[j]);
    }
  }
}

// ------------------------------------------------------------ main kernel
struct Store {
  const GemmArgs& g;
  int64_t m0, n0;
  const float* srow;  // beta * self[n0 + c] in shared memory (vector self), else nullptr
  int64_t nlim;       // min(N, n0 + tile width): the columns from there on are not this tile's
  // beta * self for the segment (row r, columns c .. c+3 of the tile), read
  // before any output of the block is written (out may be self: each element
  // is read before its own write).
  __device__ __forceinline__ float4 load(int r, int c) const {
    const int64_t m = m0 + r, n = n0 + c;
    float4 sv = make_float4(0.f, 0.f, 0.f, 0.f);
    if (!g.read_self || m >= g.M || n >= nlim) return sv;
    if (srow) return *reinterpret_cast<const float4*>(srow + c);
    const float* sp = g.self + (g.self_2d ? m * g.N : 0) + n;
    if (g.vec_out) {
      sv = *reinterpret_cast<const float4*>(sp);  // plain load: self may be out
    } else {
      sv.x = sp[0];
      if (n + 1 < g.N) sv.y = sp[1];
      if (n + 2 < g.N) sv.z = sp[2];
      if (n + 3 < g.N) sv.w = sp[3];
    }
    return make_float4(g.beta * sv.x, g.beta * sv.y, g.beta * sv.z, g.beta * sv.w);
  }
  __device__ __forceinline__ void operator()(int r, int c, float4 v, float4 bs) const {
    const int64_t m = m0 + r, n = n0 + c;
    if (m >= g.M || n >= nlim) return;
    float* o = g.out + m * g.N + n;
    float4 o4 = make_float4(fmaf(g.alpha, v.x, bs.x), fmaf(g.alpha, v.y, bs.y),
                            fmaf(g.alpha, v.z, bs.z), fmaf(g.alpha, v.w, bs.w));
    if (g.relu) o4 = make_float4(fmaxf(o4.x, 0.f), fmaxf(o4.y, 0.f), fmaxf(o4.z, 0.f), fmaxf(o4.w, 0.f));
    if (g.vec_out) {  // N % 4 == 0 and 16-byte aligned rows: n .. n+3 are in range
      *reinterpret_cast<float4*>(o) = o4;
    } else {
      const float vv[4] = {o4.x, o4.y, o4.z, o4.w};
      for (int j = 0; j < 4 && n + j < g.N; ++j) o[j] = vv[j];
    }
  }
};

// Drains a tile by TMA stores (whole-tile units, no [M,N] self, aligned out
// with N % 4 == 0): per 32-column chunk each warp computes alpha*acc +
// beta*self (+ ReLU) for its 32 rows, writes them to its 4 KB block of shared
// memory in the 128-byte swizzled layout (row r, 16-byte unit u at
// r*128 + ((u ^ (r % 8)) * 16)), and lane 0 stores the 32 x 32 block with one
// 2-D tensor store.  `srow` holds beta * self of the tile's columns (nullptr:
// no self).  The accumulator is released after its last TMEM load.  A tile
// width of 16 mod 32 ends on a half chunk: a 32-column box would overwrite the
// next tile's columns, so each lane stores its row's 16 values itself.
__device__ __forceinline__ void drain_tma(uint32_t tmem, int q, int bn, uint8_t* blk,
                                          const CUtensorMap* tm_out, const GemmArgs& g,
                                          int64_t m0, int64_t n0, const float* srow,
                                          uint64_t* release) {
  const int lane = threadIdx.x & 31;
  const uint32_t tbase = tmem + ((uint32_t)(q * 32) << 16);
  // alpha*acc + beta*self (+ ReLU) of 4 columns from c + 4u
  auto value = [&](const uint32_t (&v)[32], const float4& s4, int u) {
    float4 o = make_float4(fmaf(g.alpha, __uint_as_float(v[4 * u]), s4.x),
                           fmaf(g.alpha, __uint_as_float(v[4 * u + 1]), s4.y),
                           fmaf(g.alpha, __uint_as_float(v[4 * u + 2]), s4.z),
                           fmaf(g.alpha, __uint_as_float(v[4 * u + 3]), s4.w));
    if (g.relu)
      o = make_float4(fmaxf(o.x, 0.f), fmaxf(o.y, 0.f), fmaxf(o.z, 0.f), fmaxf(o.w, 0.f));
    return o;
  };
  int c = 0;
#pragma unroll 1
  for (; c + 32 <= bn; c += 32) {
    uint32_t v[32];
    float4 s4[8];
    ptx::tmem_ld32(tbase + (uint32_t)c, v);
    // beta*self of the chunk's columns, read before any staging store: placed
    // between the stores (two shared-memory ranges the compiler cannot tell
    // apart) each read waited for the store before it -- ~480 against ~140 clk
    // per chunk (clock64 marks, 8192x4096x4096), and the MMA waited ~6.9 k
    // against ~5.3 k clk per tile for the accumulator
#pragma unroll
    for (int u = 0; u < 8; ++u)
      s4[u] = srow ? *reinterpret_cast<const float4*>(srow + c + 4 * u)
                   : make_float4(0.f, 0.f, 0.f, 0.f);
    ptx::tmem_ld_wait();
    if (release && c + 32 >= bn) {
      ptx::tc_fence_before();
      ptx::mbar_arrive(release);
    }
    if (lane == 0) ptx::bulk_wait_read0();  // the previous chunk's store has read the block
    __syncwarp();
#pragma unroll
    for (int u = 0; u < 8; ++u)
      *reinterpret_cast<float4*>(blk + lane * 128 + ((u ^ (lane & 7)) << 4)) = value(v, s4[u], u);
    ptx::fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) {
      ptx::tma_store_2d(tm_out, blk, (int)(n0 + c), (int)(m0 + q * 32));
      ptx::bulk_commit();
    }
  }
  if (c < bn) {  // half chunk: each lane stores its row's 16 values itself
    uint32_t v[32];
    float4 s4[4];
    ptx::tmem_ld32(tbase + (uint32_t)c, v);
#pragma unroll
    for (int u = 0; u < 4; ++u)
      s4[u] = srow ? *reinterpret_cast<const float4*>(srow + c + 4 * u)
                   : make_float4(0.f, 0.f, 0.f, 0.f);
    ptx::tmem_ld_wait();
    if (release) {
      ptx::tc_fence_before();
      ptx::mbar_arrive(release);
    }
    const int64_t m = m0 + q * 32 + lane;
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int64_t n = n0 + c + 4 * u;
      const float4 o = value(v, s4[u], u);
      if (m < g.M && n < g.N)  // N % 4 == 0: the whole float4 is inside
        *reinterpret_cast<float4*>(g.out + m * g.N + n) = o;
    }
  }
}

// Split-K: a unit's raw partial tile goes to part[slice][M][N].
struct PartStore {
  float* p;
  int64_t M, N, m0, n0;
  int64_t nlim;  // min(N, n0 + tile width)
  __device__ __forceinline__ float4 load(int, int) const { return make_float4(0.f, 0.f, 0.f, 0.f); }
  __device__ __forceinline__ void operator()(int r, int c, float4 v, float4) const {
    const int64_t m = m0 + r, n = n0 + c;
    if (m >= M || n >= nlim) return;
    float* o = p + m * N + n;
    if (N % 4 == 0) {
      *reinterpret_cast<float4*>(o) = v;
    } else {
      const float vv[4] = {v.x, v.y, v.z, v.w};
      for (int j = 0; j < 4 && n + j < N; ++j) o[j] = vv[j];
    }
  }
};

// Split-K epilogue: out = beta*self + alpha * sum over slices 0, 1, ... of the
// partial tiles, always in that order (deterministic).
__global__ void __launch_bounds__(256) k_splitk_epilogue(const float* __restrict__ part,
                                                         const int splits, const GemmArgs g) {
  ptx::griddep_wait();  // the partials come from the main kernel
  const int64_t MN = g.M * g.N;
  if (g.vec_out) {
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < MN / 4;
         i += (int64_t)gridDim.x * blockDim.x) {
      const int64_t e = 4 * i, n = e % g.N;
      float4 acc = *reinterpret_cast<const float4*>(part + e);
      for (int sl = 1; sl < splits; ++sl) {
        const float4 v = *reinterpret_cast<const float4*>(part + sl * MN + e);
        acc = make_float4(acc.x + v.x, acc.y + v.y, acc.z + v.z, acc.w + v.w);
      }
      float4 bs = make_float4(0.f, 0.f, 0.f, 0.f);
      if (g.read_self) {
        const float4 sv = *reinterpret_cast<const float4*>(g.self + (g.self_2d ? e : n));
        bs = make_float4(g.beta * sv.x, g.beta * sv.y, g.beta * sv.z, g.beta * sv.w);
      }
      float4 o4 = make_float4(fmaf(g.alpha, acc.x, bs.x), fmaf(g.alpha, acc.y, bs.y),
                              fmaf(g.alpha, acc.z, bs.z), fmaf(g.alpha, acc.w, bs.w));
      if (g.relu)
        o4 = make_float4(fmaxf(o4.x, 0.f), fmaxf(o4.y, 0.f), fmaxf(o4.z, 0.f), fmaxf(o4.w, 0.f));
      *reinterpret_cast<float4*>(g.out + e) = o4;
    }
  } else {
    for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < MN;
         e += (int64_t)gridDim.x * blockDim.x) {
      float acc = part[e];
      for (int sl = 1; sl < splits; ++sl) acc += part[sl * MN + e];
      const float bs = g.read_self ? g.beta * g.self[g.self_2d ? e : e % g.N] : 0.0f;
      const float v = fmaf(g.alpha, acc, bs);
      g.out[e] = g.relu ? fmaxf(v, 0.f) : v;
    }
  }
}

template <bool THREE, bool TS>
__global__ void __launch_bounds__(THREE ? 320 : 192, 1)
    k_tc_gemm(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmBh,
              const __grid_constant__ CUtensorMap tmBl, const __grid_constant__ CUtensorMap tmOut,
              const int tma_out, const GemmArgs g, const int num_m,
              const int num_n, const int group, const int bn, const int splits, const int kps,
              float* __restrict__ part) {
  static_assert(!TS || THREE, "the A-from-TMEM form is 3xTF32");
  constexpr Layout L = TS ? kLts : (THREE ? kL3 : kL1);
  constexpr int NACC = TS ? 1 : 2;  // accumulator buffers
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_align1024(smem_raw);
  float* epi = reinterpret_cast<float*>(smem + L.stages * L.bytes);
  float* srow = reinterpret_cast<float*>(smem + L.stages * L.bytes + EPI_BYTES);
  Ctl* ctl = reinterpret_cast<Ctl*>(smem + L.stages * L.bytes + EPI_BYTES + SROW_BYTES);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // Work unit u = (tile u % num_tiles, K-slice u / num_tiles); a slice covers
  // k-blocks [slice*kps, min(num_kb, (slice+1)*kps)).  splits == 1: whole K.
  const int num_tiles = num_m * num_n;
  const int num_units = num_tiles * splits;
  const int num_kb = (int)((g.K + BK - 1) / BK);
  int* wd = &g_watchdog_gemm;

  if (threadIdx.x == 0) init_barriers(ctl, L.stages, 1, TS ? 4 : 128);
  if (warp == 0 && lane == 0) {
    ptx::tma_prefetch_desc(&tmA);
    ptx::tma_prefetch_desc(&tmBh);
    if (THREE) ptx::tma_prefetch_desc(&tmBl);
  }
  if (warp == 1) {
    ptx::tmem_alloc(&ctl->tmem_base, TMEM_COLS);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = ctl->tmem_base;
  volatile int* abort = &ctl->abort;

  if (warp == 0) {
    // ------------------------------------------------------ TMA producer
    if (lane == 0) {
      ptx::griddep_wait();  // mat2^T (or w_lo) comes from the pre-pass, or the kernel before
      const uint32_t tx = (uint32_t)(A_BYTES + (THREE ? 2 : 1) * bn * BK * 4);
      int s = 0, issued = 0;
      uint32_t ph = 0;
      for (int u = blockIdx.x; u < num_units && !*abort; u += gridDim.x) {
        int mt, nt;
        tile_coords(u % num_tiles, num_m, num_n, group, mt, nt);
        const int kb0 = (u / num_tiles) * kps, kb1 = min(num_kb, kb0 + kps);
        for (int kb = kb0; kb < kb1; ++kb) {
          if (!wait_bar(&ctl->empty[s], ph ^ 1u, abort, kSiteProducerEmpty, wd)) break;
          uint8_t* st = smem + s * L.bytes;
          ptx::mbar_arrive_expect_tx(&ctl->full[s], tx);
          ptx::tma_load_2d(st + L.a, &tmA, &ctl->full[s], kb * BK, mt * BM);
          ptx::tma_load_2d(st + L.b_hi, &tmBh, &ctl->full[s], kb * BK, nt * bn);
          if (THREE) ptx::tma_load_2d(st + L.b_lo, &tmBl, &ctl->full[s], kb * BK, nt * bn);
          ++issued;
          if (++s == L.stages) {
            s = 0;
            ph ^= 1u;
          }
        }
      }
      // the split-K sum kernel may launch now (it waits for this kernel).  The
      // next call's first kernel is not released early: launched then, its
      // blocks land on the SMs this kernel frees first, and a pre-pass spread
      // over few SMs measured slower than one launched when this kernel ends
      if (splits > 1) ptx::griddep_launch();
      // Every copy issued must have landed before the CTA's shared memory is released.
      for (int j = (issued > L.stages ? issued - L.stages : 0); j < issued; ++j)
        drain_wait(&ctl->full[j % L.stages], (uint32_t)((j / L.stages) & 1));
    }
  } else if (warp == 1) {
    // --------------------------------------------------------- MMA issuer
    if (lane == 0) {
      const uint32_t idesc = ptx::idesc_tf32(BM, (uint32_t)bn, false, false);
      // Operand addresses advance by constants (the issuing thread's few
      // instructions between MMAs are on the pipeline's critical path): a
      // descriptor holds the shared address >> 4 in its low 14 bits, so the
      // stage, the tile within it and k-step 1 (+32 bytes) are plain adds.
      constexpr uint64_t kStage = (uint64_t)(L.bytes >> 4), kA = (uint64_t)(L.a >> 4),
                         kAlo = (uint64_t)(L.a_lo >> 4), kBhi = (uint64_t)(L.b_hi >> 4),
                         kBlo = (uint64_t)(L.b_lo >> 4), kK1 = 2;
      const uint64_t d0 = sw64_desc(ptx::smem_addr(smem), 0);
      const uint32_t t0 = tmem + TS_A_COL0;
      uint64_t ds = d0;   // stage s, k-step 0
      uint32_t ts = t0;   // stage s's A columns (A-from-TMEM form)
      int s = 0, tl = 0;
      uint32_t ph = 0;
      for (int u = blockIdx.x; u < num_units; u += gridDim.x, ++tl) {
        const int buf = tl % NACC;
        const uint32_t use = (uint32_t)(tl / NACC);
        if (!wait_bar(&ctl->acce[buf], (use & 1u) ^ 1u, abort, kSiteMmaAccEmpty, wd)) break;
        ptx::tc_fence_after();
        const uint32_t d = tmem + (uint32_t)buf * ACC_STRIDE;
        const int kb0 = (u / num_tiles) * kps, kb1 = min(num_kb, kb0 + kps);
        bool ok = true;
        for (int kb = kb0; kb < kb1; ++kb) {
          if (!wait_bar(THREE ? &ctl->split[s] : &ctl->full[s], ph, abort, kSiteMmaOperands, wd)) {
            ok = false;
            break;
          }
          ptx::tc_fence_after();
          const uint32_t acc = kb > kb0 ? 1u : 0u;
          if (TS) {  // k-step 0, then k-step 1 (TMEM columns + UK, descriptors + 2)
            ptx::mma_tf32_ts(d, ts + 16u, ds + kBhi, idesc, acc);  // A_lo * B_hi
            ptx::mma_tf32_ts(d, ts, ds + kBlo, idesc, 1u);         // A_hi * B_lo
            ptx::mma_tf32_ts(d, ts, ds + kBhi, idesc, 1u);         // A_hi * B_hi
            ptx::mma_tf32_ts(d, ts + 16u + UK, ds + kBhi + kK1, idesc, 1u);
            ptx::mma_tf32_ts(d, ts + UK, ds + kBlo + kK1, idesc, 1u);
            ptx::mma_tf32_ts(d, ts + UK, ds + kBhi + kK1, idesc, 1u);
          } else if (THREE) {  // small terms first
            ptx::mma_tf32(d, ds + kAlo, ds + kBhi, idesc, acc);
            ptx::mma_tf32(d, ds + kA, ds + kBlo, idesc, 1u);
            ptx::mma_tf32(d, ds + kA, ds + kBhi, idesc, 1u);
            ptx::mma_tf32(d, ds + kAlo + kK1, ds + kBhi + kK1, idesc, 1u);
            ptx::mma_tf32(d, ds + kA + kK1, ds + kBlo + kK1, idesc, 1u);
            ptx::mma_tf32(d, ds + kA + kK1, ds + kBhi + kK1, idesc, 1u);
          } else {
            ptx::mma_tf32(d, ds + kA, ds + kBhi, idesc, acc);
            ptx::mma_tf32(d, ds + kA + kK1, ds + kBhi + kK1, idesc, 1u);
          }
          ptx::mma_commit(&ctl->empty[s]);
          if (++s == L.stages) {
            s = 0;
            ph ^= 1u;
            ds = d0;
            ts = t0;
          } else {
            ds += kStage;
            ts += TS_A_STAGE_COLS;
          }
        }
        if (!ok) break;
        ptx::mma_commit(&ctl->accf[buf]);
      }
      // Every MMA issued must be done before TMEM is released.
      ptx::mma_commit(&ctl->drain);
      drain_wait(&ctl->drain, 0);
    }
    __syncwarp();
  } else if (warp < 6) {
    // ----------------------------------------------------------- epilogue
    // self is read ahead of the first accumulator: not before the kernel
    // before this one (a dependent launch) has completed
    ptx::griddep_wait();
    const int q = warp & 3;  // TMEM lane quadrant this warp may read
    float* stage = epi + (warp - 2) * 32 * EPI_PITCH;
    int tl = 0;
    for (int u = blockIdx.x; u < num_units; u += gridDim.x, ++tl) {
      const int buf = tl % NACC;
      const uint32_t use = (uint32_t)(tl / NACC);
      int mt, nt;
      tile_coords(u % num_tiles, num_m, num_n, group, mt, nt);
      if (g.read_self && g.self_2d && splits == 1) {
        // while the tile's MMAs run: pull its [M,N] self rows into L2 (one row
        // of up to BN floats per thread, 128-byte lines)
        const int64_t m = (int64_t)mt * BM + (warp - 2) * 32 + lane, n0 = (int64_t)nt * bn;
        if (m < g.M) {
          const float* row = g.self + m * g.N + n0;
          const int64_t cols = g.N - n0 < bn ? g.N - n0 : bn;
          for (int64_t c = 0; c < cols; c += 32) ptx::prefetch_l2(row + c);
        }
      }
      // A vector self is the same for every row of the tile: beta * self of the
      // tile's columns goes to shared memory while its MMAs run.
      const bool vec_self = g.read_self && !g.self_2d && splits == 1;
      if (vec_self) {
        epi_sync();  // the previous tile's drain has read the row
        const int64_t n0 = (int64_t)nt * bn;
        for (int c = (warp - 2) * 32 + lane; c < bn; c += 128)
          srow[c] = n0 + c < g.N ? g.beta * g.self[n0 + c] : 0.0f;
        epi_sync();
      }
      const bool ok = warp_wait_bar(&ctl->accf[buf], use & 1u, abort, kSiteEpilogueAccFull, wd);
      if (epi_any(!ok)) break;
      ptx::tc_fence_after();
      // the single accumulator is handed back as soon as it is read
      uint64_t* early = TS ? &ctl->acce[buf] : nullptr;
      if (tma_out && splits == 1 && !(g.read_self && g.self_2d))
        drain_tma(tmem + (uint32_t)buf * ACC_STRIDE, q, bn, reinterpret_cast<uint8_t*>(epi) + (warp - 2) * 4096,
                  &tmOut, g, (int64_t)mt * BM, (int64_t)nt * bn, vec_self ? srow : nullptr, early);
      else if (splits == 1)
        drain_accumulator(tmem, q, (uint32_t)buf * ACC_STRIDE, bn, stage,
                          Store{g, (int64_t)mt * BM, (int64_t)nt * bn, vec_self ? srow : nullptr,
                                min(g.N, (int64_t)(nt + 1) * bn)},
                          early);
      else
        drain_accumulator(tmem, q, (uint32_t)buf * ACC_STRIDE, bn, stage,
                          PartStore{part + (int64_t)(u / num_tiles) * g.M * g.N, g.M, g.N,
                                    (int64_t)mt * BM, (int64_t)nt * bn,
                                    min(g.N, (int64_t)(nt + 1) * bn)},
                          early);
      if (!TS) {
        ptx::tc_fence_before();
        ptx::mbar_arrive(&ctl->acce[buf]);
      }
    }
    if (lane == 0) ptx::bulk_wait_all();  // every TMA store has landed before the CTA ends
  } else if (TS) {
    // ------------------------------- split warps: A_hi / A_lo into TMEM
    // Thread = row r of the A tile (TMEM lane r): its 16 values of a k-block
    // are read from the swizzled tile, split, and written to the stage's
    // TMEM columns; one arrival per warp on split[s].
    const int r = (warp & 3) * 32 + lane;
    const uint32_t trow = tmem + ((uint32_t)((warp & 3) * 32) << 16) + TS_A_COL0;
    int s = 0;
    uint32_t ph = 0;
    for (int u = blockIdx.x; u < num_units; u += gridDim.x) {
      bool ok = true;
      const int kb0 = (u / num_tiles) * kps, kb1 = min(num_kb, kb0 + kps);
      for (int kb = kb0; kb < kb1; ++kb) {
        if (!warp_wait_bar(&ctl->empty[s], ph ^ 1u, abort, kSiteProducerEmpty, wd) ||
            !warp_wait_bar(&ctl->full[s], ph, abort, kSiteSplitFull, wd)) {
          ok = false;
          break;
        }
        ptx::tc_fence_after();
        const uint8_t* row = smem + s * L.bytes + L.a + sw64_row_base(r);
        float hi[16], lo[16];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const float4 v = *reinterpret_cast<const float4*>(row + sw64_unit(r, j));
          const float vv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            hi[4 * j + e] = tf32_hi(vv[e]);
            lo[4 * j + e] = tf32_lo(vv[e]);
          }
        }
        const uint32_t ta = trow + (uint32_t)s * TS_A_STAGE_COLS;
        ptx::tmem_st16(ta, hi);
        ptx::tmem_st16(ta + 16, lo);
        ptx::tmem_st_wait();
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(&ctl->split[s]);
        if (++s == L.stages) {
          s = 0;
          ph ^= 1u;
        }
      }
      if (!ok) break;
    }
  } else if (THREE) {
    // ------------------------------------------------ split warps: A_lo
    const int tid = threadIdx.x - 192;
    int s = 0;
    uint32_t ph = 0;
    for (int u = blockIdx.x; u < num_units; u += gridDim.x) {
      bool ok = true;
      const int kb0 = (u / num_tiles) * kps, kb1 = min(num_kb, kb0 + kps);
      for (int kb = kb0; kb < kb1; ++kb) {
        // every thread polls: measured faster here than one lane per warp
        if (!wait_bar(&ctl->full[s], ph, abort, kSiteSplitFull, wd)) {
          ok = false;
          break;
        }
        const float4* a = reinterpret_cast<const float4*>(smem + s * L.bytes + L.a);
        float4* alo = reinterpret_cast<float4*>(smem + s * L.bytes + L.a_lo);
#pragma unroll
        for (int i = tid; i < A_BYTES / 16; i += 128) alo[i] = tf32_lo4(a[i]);
        ptx::fence_proxy_async_smem();
        ptx::mbar_arrive(&ctl->split[s]);
        if (++s == L.stages) {
          s = 0;
          ph ^= 1u;
        }
      }
      if (!ok) break;
    }
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
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

// Row-major fp32 matrix [outer, inner] with rows ld >= inner floats apart
// (ld % 4 == 0) -> tensor map with a {16, box_outer} box (64-byte rows),
// 64-byte swizzle, zero fill outside the matrix.
bool encode_k16(CUtensorMap* m, const float* base, uint64_t inner, uint64_t outer,
                uint32_t box_outer, uint64_t ld) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {inner, outer};
  const cuuint64_t strides[1] = {ld * 4};
  const cuuint32_t box[2] = {(cuuint32_t)BK, box_outer};
  const cuuint32_t es[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float*>(base), dims, strides, box,
            es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Raster group (M-tiles sharing each N-tile): with `sms` tiles resident, a
// group of G M-tiles keeps G mat1 panels and about sms/G mat2^T panels live.
// Pick G to minimise the estimated panel re-reads from DRAM:
// mat1_bytes * ceil(num_n / (sms / G)) + mat2t_bytes * ceil(num_m / G).
int pick_group(int64_t num_m, int64_t num_n, int sms, double a_bytes, double b_bytes) {
  // A wave of `sms` tiles grouped g along M spans sms / g N-tiles: every A
  // panel is read once per ceil(num_n / (sms / g)) and the whole B once per
  // ceil(num_m / g) (and symmetrically for groups along N, returned as -g).
  // Ties go to groups along N (on 8192x4096x4096, 4 N-tiles per group measured
  // 1 % faster than 16 M-tiles, at the same modelled traffic).
  int best = 1;
  double best_cost = 1e300;
  for (int dir = 1; dir >= 0; --dir) {
    const int64_t major = dir ? num_n : num_m, minor = dir ? num_m : num_n;
    const double major_bytes = dir ? b_bytes : a_bytes, minor_bytes = dir ? a_bytes : b_bytes;
    // groups above 16 measured slower on the 32768x1024x1024 workload
    for (int g = 1; g <= major && g <= sms && g <= 16; ++g) {
      const int64_t span = sms / g > 0 ? sms / g : 1;
      const double cost = major_bytes * (double)((minor + span - 1) / span) +
                          minor_bytes * (double)((major + g - 1) / g);
      if (cost < best_cost * 0.999) {
        best_cost = cost;
        best = dir ? -g : g;
      }
    }
  }
  return best;
}

// out [M, N] -> tensor map with a {32, 32} box, 128-byte swizzle (the
// epilogue's staging layout); rows and columns past the end are not written.
bool encode_out(CUtensorMap* m, const GemmArgs& g) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {(cuuint64_t)g.N, (cuuint64_t)g.M};
  const cuuint64_t strides[1] = {(cuuint64_t)g.N * 4};
  const cuuint32_t box[2] = {32, 32};
  const cuuint32_t es[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, g.out, dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Launch plan.  It depends on the problem only (not on the device), so the
// scratch size can be queried before a device is chosen; kPlanSMs is the SM
// count of the GB300 it is tuned for.
constexpr int kPlanSMs = 152;

struct Plan {
  int bn, num_m, num_n, splits, kps;
  int64_t ld;           // row length (floats) of the B copies and of a padded A copy
  int64_t a_offset;     // byte offset of the padded mat1 copy (when there is one)
  int64_t part_offset;  // byte offset of the split-K partials in the scratch
};

// Picks the tile width BN (a multiple of 32, or of 16 from 112 up for an
// unsplit K) and the number of K-slices by an
// estimate of the last SM's time in MMA column-k-blocks: waves * kps * (BN +
// 32), plus, when split, the slice-sum pass ((splits + 1) * M*N*4 bytes at
// HBM speed, ~1.5 ns per unit).  Ties go to wider tiles and fewer slices.
// Only plans whose scratch fits in `limit` bytes are considered (a single
// slice is always allowed: its scratch is the operand copies alone).
// pad_a / pad_b: mat1 / a K-major B (linear weight) needs a copy with
// 16-byte aligned rows.
Plan make_plan(int64_t M, int64_t N, int64_t K, bool three, bool b_kmajor, bool pad_a,
               bool pad_b, size_t limit) {
  const int64_t num_kb = (K + BK - 1) / BK;
  const int64_t ld = (K + 3) / 4 * 4;
  Plan best{BN_MAX, (int)((M + BM - 1) / BM), 0, 1, (int)num_kb, ld, 0, 0};
  // B copies: mat2 transposed, hi (+ lo); a K-major B needs only its lo part,
  // or hi (+ lo) copies when its rows are not 16-byte aligned
  const int64_t copies =
      b_kmajor ? (pad_b ? (three ? 2 : 1) : (three ? 1 : 0)) : (three ? 2 : 1);
  const int64_t bt = copies * N * ld * (int64_t)sizeof(float);
  const int64_t a_offset = (bt + 255) / 256 * 256;
  const int64_t a_bytes = pad_a ? M * ld * (int64_t)sizeof(float) : 0;
  const int64_t part_offset = (a_offset + a_bytes + 255) / 256 * 256;
  double best_cost = 1e300;
  for (int bn = BN_MAX; bn >= 32; bn -= 16) {
    if (bn % 32 != 0 && bn < 112) continue;  // narrow tiles: steps of 32
    const int64_t tiles = best.num_m * ((N + bn - 1) / bn);
    for (int sp = 1; sp <= (bn % 32 != 0 ? 1 : 16); ++sp) {  // half steps: unsplit tiles only
      const int64_t kps = (num_kb + sp - 1) / sp;
      const int64_t eff = (num_kb + kps - 1) / kps;  // non-empty slices
      if (sp > 1 && (kps < 4 || eff != sp)) continue;
      if (sp > 1 && (double)part_offset + (double)sp * M * N * 4.0 > (double)limit) continue;
      const int64_t units = tiles * sp;
      const double waves = (double)((units + kPlanSMs - 1) / kPlanSMs);
      double cost = waves * (double)kps * (bn + 32);
      if (sp > 1) cost += (double)(sp + 1) * (double)M * (double)N * 4.0 / 9750.0;
      if (cost < best_cost * 0.999) {
        best_cost = cost;
        best.bn = bn;
        best.splits = sp;
        best.kps = (int)kps;
      }
    }
  }
  best.num_n = (int)((N + best.bn - 1) / best.bn);
  best.a_offset = a_offset;
  best.part_offset = part_offset;
  return best;
}

size_t plan_bytes(const Plan& p, int64_t M, int64_t N) {
  return (size_t)p.part_offset + (p.splits > 1 ? (size_t)p.splits * M * N * sizeof(float) : 0);
}

constexpr int kMaxDev = 64;

// after_prep: a pre-pass of this call ran just before (the main kernel may
// then start early and waits for it before loading B).
// a / lda: the A operand as the TMA reads it (mat1, or its padded copy);
// ldb: the row length of the B operand (bt_hi / bt_lo).
template <bool THREE, bool TS>
cudaError_t run(const GemmArgs& g, const Plan& p, const float* a, int64_t lda, const float* bt_hi,
                const float* bt_lo, int64_t ldb, float* part, cudaStream_t s) {
  constexpr int smem = smem_bytes(TS ? kLts : (THREE ? kL3 : kL1));
  static std::atomic<bool> ready[kMaxDev];  // per device: the attribute is set (calls may race)
  auto k = k_tc_gemm<THREE, TS>;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev >= kMaxDev || !ready[dev].load(std::memory_order_acquire)) {
    e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    if (dev < kMaxDev) ready[dev].store(true, std::memory_order_release);
  }
  const int sms = device_sm_count();
  CUtensorMap ta, tbh, tbl;
  if (!encode_k16(&ta, a, (uint64_t)g.K, (uint64_t)g.M, BM, (uint64_t)lda) ||
      !encode_k16(&tbh, bt_hi, (uint64_t)g.K, (uint64_t)g.N, (uint32_t)p.bn, (uint64_t)ldb) ||
      !encode_k16(&tbl, THREE ? bt_lo : bt_hi, (uint64_t)g.K, (uint64_t)g.N, (uint32_t)p.bn,
                  (uint64_t)ldb))
    return cudaErrorInvalidValue;
  const int units = p.num_m * p.num_n * p.splits;
  const int grid = units < sms ? units : sms;
  const int group = pick_group(p.num_m, p.num_n, kPlanSMs, (double)g.M * g.K * 4.0,
                               (THREE ? 8.0 : 4.0) * (double)g.N * g.K);
  const dim3 block(THREE ? 320 : 192);
  // whole-tile units leave by TMA store when out allows it (N % 4 == 0, aligned)
  CUtensorMap tout;
  const int tma_out = p.splits == 1 && g.vec_out && encode_out(&tout, g) ? 1 : 0;
  if (!tma_out) tout = ta;  // not read
  // a dependent launch whether or not a pre-pass comes first: every global
  // access of the kernel follows a griddepcontrol.wait
  e = launch_after_previous(k, dim3(grid), block, (size_t)smem, s, ta, tbh, tbl, tout, tma_out, g,
                            p.num_m, p.num_n, group, p.bn, p.splits, p.kps, part);
  note_launch();
  note_kernel_name(TS ? "k_tc_gemm<3xtf32,a_tmem>" : (THREE ? "k_tc_gemm<3xtf32>" : "k_tc_gemm<1xtf32>"));
  if (e != cudaSuccess || p.splits == 1) return e;
  const int64_t items = g.vec_out ? g.M * g.N / 4 : g.M * g.N;
  const int64_t cap = (int64_t)sms * 8, blocks = (items + 255) / 256;
  e = launch_after_previous(k_splitk_epilogue, dim3((unsigned)(blocks < cap ? blocks : cap)),
                            dim3(256), 0, s, (const float*)part, p.splits, g);
  note_launch();
  return e;
}

}  // namespace

bool tc_gemm_supported(const GemmArgs& a) {
  const double tiles = (double)((a.M + BM - 1) / BM) * (double)((a.N + 31) / 32);
  return tiles < 2147483647.0 && encode_fn() != nullptr;
}

bool tc_gemm_pad_a(const GemmArgs& a) {
  return a.K % 4 != 0 || (reinterpret_cast<uintptr_t>(a.mat1) & 15u) != 0;
}

bool tc_gemm_pad_b(const GemmArgs& a) {
  return a.b_kmajor && (a.K % 4 != 0 || (reinterpret_cast<uintptr_t>(a.mat2) & 15u) != 0);
}

size_t tc_gemm_workspace_bytes(int64_t M, int64_t N, int64_t K, bool three_pass, bool b_kmajor,
                               bool pad_a, bool pad_b, size_t limit) {
  return plan_bytes(make_plan(M, N, K, three_pass, b_kmajor, pad_a, pad_b, limit), M, N);
}

cudaError_t launch_tc_gemm(const GemmArgs& g, bool three_pass, void* workspace,
                           size_t workspace_bytes, cudaStream_t s) {
  if (!tc_gemm_supported(g)) return cudaErrorNotSupported;
  const bool pad_a = tc_gemm_pad_a(g), pad_b = tc_gemm_pad_b(g);
  const Plan p =
      make_plan(g.M, g.N, g.K, three_pass, g.b_kmajor != 0, pad_a, pad_b, workspace_bytes);
  if (plan_bytes(p, g.M, g.N) > workspace_bytes || (plan_bytes(p, g.M, g.N) > 0 && !workspace))
    return cudaErrorInvalidValue;
  float* ws = static_cast<float*>(workspace);
  float* part = reinterpret_cast<float*>(static_cast<char*>(workspace) + p.part_offset);
  const int64_t ld = p.ld;
  const float *b_hi, *b_lo, *a = g.mat1;
  int64_t lda = g.K, ldb = ld;
  const int64_t cap = (int64_t)device_sm_count() * 8;
  if (pad_a) {  // mat1 rows to 16-byte aligned rows of ld floats
    float* a_copy = reinterpret_cast<float*>(static_cast<char*>(workspace) + p.a_offset);
    const int64_t blocks = (g.M * ((g.K + 255) / 256) + PAD_UNITS - 1) / PAD_UNITS;
    const dim3 grid((unsigned)(blocks < cap ? blocks : cap));
    const cudaError_t e = launch_after_previous(k_pad_rows, grid, dim3(256), 0, s, g.mat1, g.M,
                                                g.K, ld, a_copy, (float*)nullptr);
    note_launch();
    if (e != cudaSuccess) return e;
    a = a_copy;
    lda = ld;
  }
  if (g.b_kmajor && pad_b) {  // w[N,K] to aligned rows, hi (+ lo)
    b_hi = ws;
    b_lo = three_pass ? ws + g.N * ld : nullptr;
    const int64_t blocks = (g.N * ((g.K + 255) / 256) + PAD_UNITS - 1) / PAD_UNITS;
    const dim3 grid((unsigned)(blocks < cap ? blocks : cap));
    const cudaError_t e = launch_after_previous(k_pad_rows, grid, dim3(256), 0, s, g.mat2, g.N,
                                                g.K, ld, ws,
                                                three_pass ? ws + g.N * ld : (float*)nullptr);
    note_launch();
    if (e != cudaSuccess) return e;
  } else if (g.b_kmajor) {  // w[N,K] is B_hi; 3xTF32 adds w_lo in the scratch
    b_hi = g.mat2;
    b_lo = three_pass ? ws : nullptr;
    ldb = g.K;  // == ld: K % 4 == 0 here
    if (three_pass) {
      // K % 4 == 0 and 16-byte aligned rows here: whole float4s
      const int64_t total4 = g.N * g.K / 4, blocks = (total4 + 255) / 256;
      const int64_t cap2 = 2 * (int64_t)device_sm_count();
      const cudaError_t e = launch_after_previous(
          k_prep_blo, dim3((unsigned)(blocks < cap2 ? blocks : cap2)), dim3(256), 0, s,
          reinterpret_cast<const float4*>(g.mat2), total4, reinterpret_cast<float4*>(ws));
      note_launch();
      if (e != cudaSuccess) return e;
    }
  } else {  // transpose mat2[K,N] into Bt_hi[N,ld] (+ Bt_lo)
    b_hi = ws;
    b_lo = three_pass ? ws + g.N * ld : nullptr;
    if (g.N % 4 == 0 && (reinterpret_cast<uintptr_t>(g.mat2) & 15u) == 0) {
      const int64_t tiles = ((g.N + 63) / 64) * ((g.K + 63) / 64);
      const cudaError_t e = launch_after_previous(
          k_prep_b4, dim3((unsigned)(tiles < cap ? tiles : cap)), dim3(256), 0, s, g.mat2, g.K,
          g.N, ld, ws, three_pass ? ws + g.N * ld : (float*)nullptr);
      if (e != cudaSuccess) return e;
    } else {
      const int64_t tiles = ((g.N + 31) / 32) * ((g.K + 31) / 32);
      const cudaError_t e = launch_after_previous(
          k_prep_b, dim3((unsigned)(tiles < cap ? tiles : cap)), dim3(32, 8), 0, s, g.mat2, g.K,
          g.N, ld, ws, three_pass ? ws + g.N * ld : (float*)nullptr);
      if (e != cudaSuccess) return e;
    }
    note_launch();
  }
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  if (!three_pass) return run<false, false>(g, p, a, lda, b_hi, nullptr, ldb, part, s);
  const bool light = !(g.read_self && g.self_2d) || p.splits > 1;  // no [M,N] self read per tile
  const bool ts = p.kps >= kTsMinKb || (light && p.kps >= kTsMinKbLightEpilogue);
  return ts ? run<true, true>(g, p, a, lda, b_hi, b_lo, ldb, part, s)
            : run<true, false>(g, p, a, lda, b_hi, b_lo, ldb, part, s);
}

namespace {
// One thread waits on a barrier that nothing will complete: the wait gives up
// after limit_ns and reports through the addmm watchdog word, as a real
// timeout does (imc_selftest_wait_timeout).
__global__ void k_wait_selftest(uint64_t limit_ns) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    ptx::mbar_init(&bar, 1);
    abort_flag = 0;
    ptx::fence_mbar_init();
    wait_bar(&bar, 0, &abort_flag, kSiteSelfTest, &g_watchdog_gemm, limit_ns);
  }
}
}  // namespace

cudaError_t launch_wait_selftest(int limit_us, cudaStream_t s) {
  k_wait_selftest<<<1, 32, 0, s>>>((uint64_t)limit_us * 1000ull);
  note_launch();
  return cudaGetLastError();
}

cudaError_t gemm_take_watchdog(int* value) {
  cudaError_t e = cudaMemcpyFromSymbol(value, g_watchdog_gemm, sizeof(int));
  if (e != cudaSuccess) return e;
  const int zero = 0;
  return cudaMemcpyToSymbol(g_watchdog_gemm, &zero, sizeof(int));
}

}  // namespace imc
