// tcgen05 tensor-core kernels for fp32 addmm and implicit-im2col conv2d.
//
// What they compute is fixed by two ExecuTorch WebGPU pull-request pages:
// "Add optimized addmm op" (Solution / Implementation: out = beta*self +
// alpha*(mat1 @ mat2), mat2 read as mat2[k*N + n], self from [N] or [M,N]) and
// "et_vk conv2d: route standard (groups==1) conv through an im2col tiled GEMM"
// (Solution / Implementation: M = OC, N = B*OH*OW, K = IC*KH*KW, weight as
// the [OC, K] operand, the input im2col-sampled on the fly with out-of-range
// taps reading 0, bias per output channel, NCHW output).  Their WGSL design
// (32x32 workgroup tiles, 4x4 register blocking) targets a scalar ALU; here
// the same tiled GEMM is laid out for sm_103a:
//
//  * one persistent CTA per SM walks 128 x 128 output tiles;
//  * operands are staged in a multi-stage ring of shared-memory tiles in the
//    K-major, 128-byte-swizzled layout the tensor core reads (on this GPU a
//    kind::tf32 MMA only accepts K-major operands);
//  * one thread issues tcgen05.mma kind::tf32 into an fp32 accumulator in
//    tensor memory (TMEM), double-buffered so the epilogue of one tile
//    overlaps the main loop of the next;
//  * fp32 accuracy (the default mode) comes from splitting every operand
//    element v into hi = v with the low 13 mantissa bits cleared (exactly a
//    TF32 number) and lo = v - hi (exact in fp32) and accumulating
//    A_lo*B_hi + A_hi*B_lo + A_hi*B_hi ("3xTF32"; the dropped A_lo*B_lo term is
//    below 2^-20 relative).  The 1xTF32 mode issues A*B once;
//  * the epilogue reads the accumulator with tcgen05.ld, transposes each
//    32x32 block through shared memory and writes whole 128-byte row
//    segments: beta*self + alpha*acc (addmm) or acc + bias[oc] scattered to
//    NCHW (conv).
//
// addmm: mat1 and mat2 tiles arrive by TMA (cp.async.bulk.tensor, no
// multicast).  mat1 is K-major already; mat2 is N-contiguous, so four
// transform warps transpose its tile into the K-major layout while splitting
// it (and split mat1 in place).  conv: four producer warps gather the im2col
// rows (zero for padding taps and the ragged K / N edges) and the weight rows
// and write hi and lo tiles directly.
//
// Every mbarrier wait is bounded (about 2 s): on expiry the kernel records
// the wait site in a device word, stops all roles, waits for its own copies
// and MMAs in flight, frees its TMEM and returns.  No trap, no hang.
#include <mutex>

#include "imc.h"
#include "imc_internal.cuh"
#include "ptx.cuh"

namespace imc {
namespace {

constexpr int BM = 128;                  // rows of a tile (TMEM lanes)
constexpr int BN = 128;                  // columns of a tile (MMA N)
constexpr int BK = 32;                   // fp32 per k-block: one 128-byte swizzle row
constexpr int UK = 8;                    // K of one tcgen05.mma kind::tf32
constexpr int KSTEPS = BK / UK;
constexpr int TILE_BYTES = 128 * BK * 4;  // one 128-row K-major operand tile: 16 KB
constexpr int B_CHUNK_BYTES = BK * 128;   // 32 columns x BK rows of an N-contiguous tile
constexpr int EPI_PITCH = 36;             // floats per staged epilogue row
constexpr int EPI_BYTES = 4 * 32 * EPI_PITCH * 4;
constexpr int MAX_STAGES = 8;
constexpr uint32_t TMEM_COLS = 2 * BN;    // two accumulator buffers
constexpr uint64_t kWaitLimitNs = 2000000000ull;
constexpr uint64_t kDrainLimitNs = 200000000ull;

// Watchdog word: first wait site that timed out (0 = none).
__device__ int g_watchdog;

struct Ctl {
  uint64_t full[MAX_STAGES];   // raw operands of a stage are in shared memory
  uint64_t split[MAX_STAGES];  // addmm: the MMA-ready tiles of a stage are written
  uint64_t empty[MAX_STAGES];  // the MMAs reading a stage are done
  uint64_t accf[2];            // accumulator buffer holds a finished tile
  uint64_t acce[2];            // epilogue has drained an accumulator buffer
  uint64_t drain;              // all MMAs of this CTA are done
  uint32_t tmem_base;
  int abort;
};

// Byte offsets of the tiles inside one pipeline stage.
struct Layout {
  int a_hi, b_hi, a_lo, b_lo, b_raw, bytes, stages;
};
// addmm, 3xTF32: mat1 tile (TMA, truncated in place = A_hi) | mat2 tile as
// loaded | A_lo | B_hi | B_lo.   1xTF32: mat1 | mat2 as loaded | B (K-major).
constexpr Layout kGemm3 = {0, 3 * TILE_BYTES, 2 * TILE_BYTES, 4 * TILE_BYTES, TILE_BYTES,
                           5 * TILE_BYTES, 2};
constexpr Layout kGemm1 = {0, 2 * TILE_BYTES, 0, 0, TILE_BYTES, 3 * TILE_BYTES, 4};
// conv, 3xTF32: A_hi | B_hi | A_lo | B_lo.   1xTF32: A | B.
constexpr Layout kConv3 = {0, TILE_BYTES, 2 * TILE_BYTES, 3 * TILE_BYTES, 0, 4 * TILE_BYTES, 3};
constexpr Layout kConv1 = {0, TILE_BYTES, 0, 0, 0, 2 * TILE_BYTES, 6};

constexpr int smem_bytes(const Layout& L) {
  return 1024 + L.stages * L.bytes + EPI_BYTES + (int)sizeof(Ctl);
}
static_assert(smem_bytes(kGemm3) <= 232448 && smem_bytes(kGemm1) <= 232448 &&
                  smem_bytes(kConv3) <= 232448 && smem_bytes(kConv1) <= 232448,
              "shared memory");
static_assert(kGemm1.stages <= MAX_STAGES && kConv1.stages <= MAX_STAGES, "stages");

enum WaitSite {
  kSiteProducerEmpty = 1,
  kSiteSplitFull = 2,
  kSiteMmaAccEmpty = 3,
  kSiteMmaOperands = 4,
  kSiteEpilogueAccFull = 5,
};

__device__ __forceinline__ bool wait_bar(uint64_t* bar, uint32_t parity, volatile int* abort,
                                         int site) {
  if (ptx::mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = ptx::globaltimer_ns();
  for (uint32_t it = 1;; ++it) {
    if (ptx::mbar_try_wait(bar, parity)) return true;
    if ((it & 127u) == 0) {
      if (*abort) return false;
      if (ptx::globaltimer_ns() - t0 > kWaitLimitNs) {
        *abort = 1;
        atomicCAS(&g_watchdog, 0, site);
        return false;
      }
    }
  }
}

// Teardown wait: ignores the abort flag, gives up after kDrainLimitNs.
__device__ __forceinline__ void drain_wait(uint64_t* bar, uint32_t parity) {
  const uint64_t t0 = ptx::globaltimer_ns();
  while (!ptx::mbar_try_wait(bar, parity)) {
    if (ptx::globaltimer_ns() - t0 > kDrainLimitNs) break;
  }
}

__device__ __forceinline__ float tf32_hi(float v) {
  return __uint_as_float(__float_as_uint(v) & 0xFFFFE000u);
}
__device__ __forceinline__ float tf32_lo(float v, float hi) {
  return isfinite(v) ? v - hi : 0.0f;
}

// Byte offset of element (row, k) in a 128-row, BK-deep K-major tile with the
// 128-byte swizzle: 8-row groups of 1024 B, 16-byte units XOR-ed with row % 8.
__device__ __forceinline__ int kmajor_offset(int row, int k) {
  return (row >> 3) * 1024 + (row & 7) * 128 + ((((k >> 2) ^ (row & 7))) << 4) + (k & 3) * 4;
}

// Writes 32 consecutive-k values of one tile row: hi (and lo at +lo_delta).
__device__ __forceinline__ void store_row(uint8_t* tile, int row, const float (&v)[BK], bool three,
                                          int lo_delta) {
  uint8_t* base = tile + (row >> 3) * 1024 + (row & 7) * 128;
#pragma unroll
  for (int j = 0; j < BK / 4; ++j) {
    const int off = (j ^ (row & 7)) << 4;
    const float4 q = make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
    if (three) {
      const float4 h = make_float4(tf32_hi(q.x), tf32_hi(q.y), tf32_hi(q.z), tf32_hi(q.w));
      *reinterpret_cast<float4*>(base + off) = h;
      *reinterpret_cast<float4*>(base + lo_delta + off) =
          make_float4(tf32_lo(q.x, h.x), tf32_lo(q.y, h.y), tf32_lo(q.z, h.z), tf32_lo(q.w, h.w));
    } else {
      *reinterpret_cast<float4*>(base + off) = q;
    }
  }
}

// Grouped raster: `group` M-tiles share each N-tile before moving on, so the
// CTAs resident at one time reuse the same operand panels from L2.
__device__ __forceinline__ void tile_coords(int t, int num_m, int num_n, int group, int& mt,
                                            int& nt) {
  const int per = group * num_n;
  const int gi = t / per;
  const int m_first = gi * group;
  const int rows = min(group, num_m - m_first);
  const int r = t - gi * per;
  mt = m_first + r % rows;
  nt = r / rows;
}

// ---------------------------------------------------------------- MMA role
// One thread: for every tile, wait for a free accumulator buffer, then for
// each k-block wait for its operands, issue KSTEPS (x3 for 3xTF32) MMAs and
// release the stage with a commit.
__device__ void mma_role(Ctl* ctl, uint8_t* smem, uint32_t tmem, int num_tiles, int num_kb,
                         const Layout L, bool three, bool wait_split) {
  volatile int* abort = &ctl->abort;
  const uint32_t idesc = ptx::idesc_tf32(BM, BN, /*a_mn_major=*/false, /*b_mn_major=*/false);
  int s = 0;
  uint32_t ph = 0;
  int tl = 0;
  for (int t = blockIdx.x; t < num_tiles; t += gridDim.x, ++tl) {
    const int buf = tl & 1;
    const uint32_t use = (uint32_t)(tl >> 1);
    if (!wait_bar(&ctl->acce[buf], (use & 1u) ^ 1u, abort, kSiteMmaAccEmpty)) break;
    ptx::tc_fence_after();
    const uint32_t d = tmem + (uint32_t)(buf * BN);
    bool ok = true;
    for (int kb = 0; kb < num_kb; ++kb) {
      uint64_t* ready = wait_split ? &ctl->split[s] : &ctl->full[s];
      if (!wait_bar(ready, ph, abort, kSiteMmaOperands)) {
        ok = false;
        break;
      }
      ptx::tc_fence_after();
      const uint32_t st = ptx::smem_addr(smem + s * L.bytes);
#pragma unroll
      for (int k = 0; k < KSTEPS; ++k) {
        // K-major tiles: 8-row groups 1024 B apart, one k-step = 32 B inside the row.
        const uint64_t ah = ptx::smem_desc(st + L.a_hi + k * 32, 16, 1024, ptx::kSwizzle128B);
        const uint64_t bh = ptx::smem_desc(st + L.b_hi + k * 32, 16, 1024, ptx::kSwizzle128B);
        const uint32_t acc = (kb > 0 || k > 0) ? 1u : 0u;
        if (three) {
          const uint64_t al = ptx::smem_desc(st + L.a_lo + k * 32, 16, 1024, ptx::kSwizzle128B);
          const uint64_t bl = ptx::smem_desc(st + L.b_lo + k * 32, 16, 1024, ptx::kSwizzle128B);
          ptx::mma_tf32(d, al, bh, idesc, acc);
          ptx::mma_tf32(d, ah, bl, idesc, 1u);
          ptx::mma_tf32(d, ah, bh, idesc, 1u);
        } else {
          ptx::mma_tf32(d, ah, bh, idesc, acc);
        }
      }
      ptx::mma_commit(&ctl->empty[s]);
      if (++s == L.stages) {
        s = 0;
        ph ^= 1u;
      }
    }
    if (!ok) break;
    ptx::mma_commit(&ctl->accf[buf]);
  }
  // Wait for every MMA this thread issued before TMEM can be released.
  ptx::mma_commit(&ctl->drain);
  drain_wait(&ctl->drain, 0);
}

// ----------------------------------------------------------- epilogue role
// Four warps; warp w may read TMEM lanes 32*(w%4) .. +31 (rows of the tile).
struct GemmStore {
  const GemmArgs& g;
  __device__ __forceinline__ void store4(int64_t m, int64_t n, float4 v) const {
    float* o = g.out + m * g.N + n;
    if (g.vec_out) {  // N % 4 == 0 on this path, so n .. n+3 are in range
      float4 r;
      if (g.read_self) {
        const float4 sv =
            __ldg(reinterpret_cast<const float4*>(g.self + (g.self_2d ? m * g.N : 0) + n));
        r.x = fmaf(g.alpha, v.x, g.beta * sv.x);
        r.y = fmaf(g.alpha, v.y, g.beta * sv.y);
        r.z = fmaf(g.alpha, v.z, g.beta * sv.z);
        r.w = fmaf(g.alpha, v.w, g.beta * sv.w);
      } else {
        r = make_float4(g.alpha * v.x, g.alpha * v.y, g.alpha * v.z, g.alpha * v.w);
      }
      *reinterpret_cast<float4*>(o) = r;
    } else {
      const float vv[4] = {v.x, v.y, v.z, v.w};
      const float* sp = g.self + (g.self_2d ? m * g.N : 0);
      for (int j = 0; j < 4 && n + j < g.N; ++j)
        o[j] = g.read_self ? fmaf(g.alpha, vv[j], g.beta * sp[n + j]) : g.alpha * vv[j];
    }
  }
  __device__ __forceinline__ int64_t M() const { return g.M; }
  __device__ __forceinline__ int64_t N() const { return g.N; }
};

struct ConvStore {
  const ConvArgs& c;
  __device__ __forceinline__ void store4(int64_t m, int64_t n, float4 v) const {
    const float bv = c.bias ? __ldg(c.bias + m) : 0.0f;
    const int64_t P = (int64_t)c.OH * c.OW;
    if (c.vec_out) {  // P % 4 == 0: n .. n+3 lie in one image
      const int64_t b = n / P, p = n - b * P;
      *reinterpret_cast<float4*>(c.out + (b * c.OC + m) * P + p) =
          make_float4(v.x + bv, v.y + bv, v.z + bv, v.w + bv);
    } else {
      const float vv[4] = {v.x, v.y, v.z, v.w};
      for (int j = 0; j < 4 && n + j < c.N; ++j) {
        const int64_t nn = n + j, b = nn / P, p = nn - b * P;
        c.out[(b * c.OC + m) * P + p] = vv[j] + bv;
      }
    }
  }
  __device__ __forceinline__ int64_t M() const { return c.M; }
  __device__ __forceinline__ int64_t N() const { return c.N; }
};

template <class Store>
__device__ void epilogue_role(Ctl* ctl, float* stage, uint32_t tmem, int num_tiles, int num_m,
                              int num_n, int group, int q, const Store& st) {
  volatile int* abort = &ctl->abort;
  const int lane = threadIdx.x & 31;
  int tl = 0;
  for (int t = blockIdx.x; t < num_tiles; t += gridDim.x, ++tl) {
    const int buf = tl & 1;
    const uint32_t use = (uint32_t)(tl >> 1);
    int ok = 1;
    if (lane == 0) ok = wait_bar(&ctl->accf[buf], use & 1u, abort, kSiteEpilogueAccFull) ? 1 : 0;
    ok = __shfl_sync(0xffffffffu, ok, 0);
    if (!ok) break;
    ptx::tc_fence_after();
    int mt, nt;
    tile_coords(t, num_m, num_n, group, mt, nt);
    const int64_t row0 = (int64_t)mt * BM + q * 32;
    const uint32_t tbase = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(buf * BN);
#pragma unroll 1
    for (int c = 0; c < BN / 32; ++c) {
      uint32_t r[32];
      ptx::tmem_ld32(tbase + (uint32_t)(c * 32), r);
      ptx::tmem_ld_wait();
      float4* dst = reinterpret_cast<float4*>(stage + lane * EPI_PITCH);
#pragma unroll
      for (int j = 0; j < 8; ++j)
        dst[j] = make_float4(__uint_as_float(r[4 * j]), __uint_as_float(r[4 * j + 1]),
                             __uint_as_float(r[4 * j + 2]), __uint_as_float(r[4 * j + 3]));
      __syncwarp();
      const int64_t col0 = (int64_t)nt * BN + c * 32;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int rr = i * 4 + (lane >> 3), cc = (lane & 7) * 4;
        const int64_t gm = row0 + rr, gn = col0 + cc;
        if (gm < st.M() && gn < st.N())
          st.store4(gm, gn, *reinterpret_cast<const float4*>(stage + rr * EPI_PITCH + cc));
      }
      __syncwarp();
    }
    ptx::tc_fence_before();
    ptx::mbar_arrive(&ctl->acce[buf]);
  }
}

__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
  return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

__device__ __forceinline__ void init_barriers(Ctl* ctl, int stages, uint32_t full_count) {
  for (int s = 0; s < stages; ++s) {
    ptx::mbar_init(&ctl->full[s], full_count);
    ptx::mbar_init(&ctl->split[s], 128);
    ptx::mbar_init(&ctl->empty[s], 1);
  }
  for (int b = 0; b < 2; ++b) {
    ptx::mbar_init(&ctl->accf[b], 1);
    ptx::mbar_init(&ctl->acce[b], 128);
  }
  ptx::mbar_init(&ctl->drain, 1);
  ctl->abort = 0;
  ptx::fence_mbar_init();
}

// ------------------------------------------------------------- addmm kernel
// warp 0: TMA producer; warp 1: TMEM owner + MMA issuer; warps 2-5: epilogue;
// warps 6-9: transform warps (K-major mat2 tile; hi / lo split in 3xTF32).
template <bool THREE>
__global__ void __launch_bounds__(320, 1)
    k_tc_gemm(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
              const GemmArgs g, const int num_m, const int num_n, const int group) {
  constexpr Layout L = THREE ? kGemm3 : kGemm1;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  float* epi = reinterpret_cast<float*>(smem + L.stages * L.bytes);
  Ctl* ctl = reinterpret_cast<Ctl*>(smem + L.stages * L.bytes + EPI_BYTES);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int num_tiles = num_m * num_n;
  const int num_kb = (int)((g.K + BK - 1) / BK);

  if (threadIdx.x == 0) init_barriers(ctl, L.stages, 1);
  if (warp == 0 && lane == 0) {
    ptx::tma_prefetch_desc(&tmA);
    ptx::tma_prefetch_desc(&tmB);
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
    if (lane == 0) {
      int s = 0;
      uint32_t ph = 0;
      int issued = 0;
      for (int t = blockIdx.x; t < num_tiles && !*abort; t += gridDim.x) {
        int mt, nt;
        tile_coords(t, num_m, num_n, group, mt, nt);
        for (int kb = 0; kb < num_kb; ++kb) {
          if (!wait_bar(&ctl->empty[s], ph ^ 1u, abort, kSiteProducerEmpty)) break;
          uint8_t* st = smem + s * L.bytes;
          ptx::mbar_arrive_expect_tx(&ctl->full[s], 2 * TILE_BYTES);
          ptx::tma_load_2d(st + L.a_hi, &tmA, &ctl->full[s], kb * BK, mt * BM);
#pragma unroll
          for (int c = 0; c < BN / 32; ++c)
            ptx::tma_load_2d(st + L.b_raw + c * B_CHUNK_BYTES, &tmB, &ctl->full[s],
                             nt * BN + c * 32, kb * BK);
          ++issued;
          if (++s == L.stages) {
            s = 0;
            ph ^= 1u;
          }
        }
      }
      // Every copy issued must have landed before the CTA's shared memory is released.
      for (int j = (issued > L.stages ? issued - L.stages : 0); j < issued; ++j)
        drain_wait(&ctl->full[j % L.stages], (uint32_t)((j / L.stages) & 1));
    }
  } else if (warp == 1) {
    if (lane == 0) mma_role(ctl, smem, tmem, num_tiles, num_kb, L, THREE, true);
    __syncwarp();
  } else if (warp < 6) {
    epilogue_role(ctl, epi + (warp - 2) * 32 * EPI_PITCH, tmem, num_tiles, num_m, num_n, group,
                  warp & 3, GemmStore{g});
  } else {
    // Transform warps.  mat1 tile: split in place (hi) and into A_lo.  mat2
    // tile (32 k-rows x 128 n, N-contiguous, 128B-swizzled per 32-column
    // chunk): lane = k; each lane reads 4 consecutive n of its row and writes
    // them to rows n of the K-major B_hi (and B_lo) tiles.  Both the 16-byte
    // reads and the 4-byte writes hit 32 distinct banks per warp.
    const int tid = threadIdx.x - 192, tw = tid >> 5;
    int s = 0;
    uint32_t ph = 0;
    for (int t = blockIdx.x; t < num_tiles; t += gridDim.x) {
      bool ok = true;
      for (int kb = 0; kb < num_kb; ++kb) {
        if (!wait_bar(&ctl->full[s], ph, abort, kSiteSplitFull)) {
          ok = false;
          break;
        }
        uint8_t* st = smem + s * L.bytes;
        if (THREE) {
          float4* ahi = reinterpret_cast<float4*>(st + L.a_hi);
          float4* alo = reinterpret_cast<float4*>(st + L.a_lo);
#pragma unroll 4
          for (int i = tid; i < TILE_BYTES / 16; i += 128) {
            const float4 v = ahi[i];
            const float4 h = make_float4(tf32_hi(v.x), tf32_hi(v.y), tf32_hi(v.z), tf32_hi(v.w));
            ahi[i] = h;
            alo[i] = make_float4(tf32_lo(v.x, h.x), tf32_lo(v.y, h.y), tf32_lo(v.z, h.z),
                                 tf32_lo(v.w, h.w));
          }
        }
        const uint8_t* braw = st + L.b_raw;
        uint8_t* bhi = st + L.b_hi;
        const int k = lane;
#pragma unroll 2
        for (int qd = tw; qd < BN / 4; qd += 4) {  // qd: group of 4 columns n = 4qd .. 4qd+3
          const float4 v = *reinterpret_cast<const float4*>(
              braw + (qd >> 3) * B_CHUNK_BYTES + k * 128 + ((((qd & 7) ^ (k & 7))) << 4));
          const float vv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const int off = kmajor_offset(4 * qd + j, k);
            if (THREE) {
              const float h = tf32_hi(vv[j]);
              *reinterpret_cast<float*>(bhi + off) = h;
              *reinterpret_cast<float*>(bhi + (L.b_lo - L.b_hi) + off) = tf32_lo(vv[j], h);
            } else {
              *reinterpret_cast<float*>(bhi + off) = vv[j];
            }
          }
        }
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

// -------------------------------------------------------------- conv kernel
// warps 0-3: producers (im2col gather of B, weight rows of A, hi/lo split);
// warp 4: TMEM owner + MMA issuer; warps 5-8: epilogue.
template <bool THREE>
__global__ void __launch_bounds__(288, 1)
    k_tc_conv(const ConvArgs c, const int num_m, const int num_n, const int group,
              const int a_vec) {
  constexpr Layout L = THREE ? kConv3 : kConv1;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  float* epi = reinterpret_cast<float*>(smem + L.stages * L.bytes);
  Ctl* ctl = reinterpret_cast<Ctl*>(smem + L.stages * L.bytes + EPI_BYTES);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int num_tiles = num_m * num_n;
  const int K = (int)c.K;
  const int num_kb = (K + BK - 1) / BK;

  if (threadIdx.x == 0) init_barriers(ctl, L.stages, 128);
  if (warp == 4) {
    ptx::tmem_alloc(&ctl->tmem_base, TMEM_COLS);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = ctl->tmem_base;
  volatile int* abort = &ctl->abort;

  if (warp < 4) {
    const int pt = threadIdx.x;  // owns row pt of the B tile (column n) and row pt of A
    const int P = c.OH * c.OW;
    int s = 0;
    uint32_t ph = 0;
    for (int t = blockIdx.x; t < num_tiles && !*abort; t += gridDim.x) {
      int mt, nt;
      tile_coords(t, num_m, num_n, group, mt, nt);
      // im2col column n = (b*OH + oh)*OW + ow of this thread.
      const int64_t n = (int64_t)nt * BN + pt;
      const bool col_ok = n < c.N;
      int ih0 = 0, iw0 = 0;
      const float* xb = c.x;
      if (col_ok) {
        const int b = (int)(n / P), p = (int)(n - (int64_t)b * P);
        const int oh = p / c.OW, ow = p - oh * c.OW;
        ih0 = oh * c.sH - c.pH;
        iw0 = ow * c.sW - c.pW;
        xb = c.x + (int64_t)b * c.IC * c.H * c.W;
      }
      const int64_t m = (int64_t)mt * BM + pt;
      const bool row_ok = m < c.M;
      const float* wrow = c.w + (row_ok ? m : 0) * (int64_t)K;
      bool ok = true;
      for (int kb = 0; kb < num_kb; ++kb) {
        if (!wait_bar(&ctl->empty[s], ph ^ 1u, abort, kSiteProducerEmpty)) {
          ok = false;
          break;
        }
        uint8_t* st = smem + s * L.bytes;
        const int k0 = kb * BK;
        // ---- B: im2col rows k0 .. k0+31 of column n; kk -> (ic, kh, kw).
        float v[BK];
        {
          int kw = k0 % c.KW;
          const int u = k0 / c.KW;
          int kh = u % c.KH;
          int ic = u / c.KH;
#pragma unroll
          for (int j = 0; j < BK; ++j) {
            const int ih = ih0 + kh * c.dH, iw = iw0 + kw * c.dW;
            const bool in = col_ok && (k0 + j < K) && (unsigned)ih < (unsigned)c.H &&
                            (unsigned)iw < (unsigned)c.W;
            v[j] = in ? __ldg(xb + ((ic * c.H + ih) * c.W + iw)) : 0.0f;
            if (++kw == c.KW) {
              kw = 0;
              if (++kh == c.KH) {
                kh = 0;
                ++ic;
              }
            }
          }
        }
        // ---- A: weight row m, columns k0 .. k0+31.
        float a[BK];
        if (a_vec && row_ok && k0 + BK <= K) {
#pragma unroll
          for (int j = 0; j < BK / 4; ++j) {
            const float4 q4 = __ldg(reinterpret_cast<const float4*>(wrow + k0) + j);
            a[4 * j] = q4.x;
            a[4 * j + 1] = q4.y;
            a[4 * j + 2] = q4.z;
            a[4 * j + 3] = q4.w;
          }
        } else {
#pragma unroll
          for (int j = 0; j < BK; ++j) a[j] = (row_ok && k0 + j < K) ? __ldg(wrow + k0 + j) : 0.0f;
        }
        store_row(st + L.b_hi, pt, v, THREE, L.b_lo - L.b_hi);
        store_row(st + L.a_hi, pt, a, THREE, L.a_lo - L.a_hi);
        ptx::fence_proxy_async_smem();
        ptx::mbar_arrive(&ctl->full[s]);
        if (++s == L.stages) {
          s = 0;
          ph ^= 1u;
        }
      }
      if (!ok) break;
    }
  } else if (warp == 4) {
    if (lane == 0) mma_role(ctl, smem, tmem, num_tiles, num_kb, L, THREE, false);
    __syncwarp();
  } else {
    epilogue_role(ctl, epi + (warp - 5) * 32 * EPI_PITCH, tmem, num_tiles, num_m, num_n, group,
                  warp & 3, ConvStore{c});
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 4) {
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

// Row-major fp32 matrix [outer, inner] -> tensor map with a {32, box_outer}
// box, 128-byte swizzle, zero fill outside the matrix.
bool encode_2d(CUtensorMap* m, const float* base, uint64_t inner, uint64_t outer,
               uint32_t box_outer) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {inner, outer};
  const cuuint64_t strides[1] = {inner * 4};
  const cuuint32_t box[2] = {32, box_outer};
  const cuuint32_t es[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float*>(base), dims, strides, box,
            es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

constexpr int kMaxDev = 64;

template <class KernelPtr>
cudaError_t prepare(KernelPtr k, int smem, bool* done_per_device) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < kMaxDev && done_per_device[dev]) return cudaSuccess;
  e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e == cudaSuccess && dev < kMaxDev) done_per_device[dev] = true;
  return e;
}

template <bool THREE>
cudaError_t run_gemm(const GemmArgs& g, const CUtensorMap& ta, const CUtensorMap& tb,
                     cudaStream_t s) {
  constexpr int smem = smem_bytes(THREE ? kGemm3 : kGemm1);
  static bool ready[kMaxDev];
  auto k = k_tc_gemm<THREE>;
  cudaError_t e = prepare(k, smem, ready);
  if (e != cudaSuccess) return e;
  const int num_m = (int)((g.M + BM - 1) / BM), num_n = (int)((g.N + BN - 1) / BN);
  const int tiles = num_m * num_n;
  const int sms = device_sm_count();
  const int grid = tiles < sms ? tiles : sms;
  const int group = num_m < 8 ? num_m : 8;
  k<<<grid, 320, smem, s>>>(ta, tb, g, num_m, num_n, group);
  note_launch();
  return cudaGetLastError();
}

template <bool THREE>
cudaError_t run_conv(const ConvArgs& c, cudaStream_t s) {
  constexpr int smem = smem_bytes(THREE ? kConv3 : kConv1);
  static bool ready[kMaxDev];
  auto k = k_tc_conv<THREE>;
  cudaError_t e = prepare(k, smem, ready);
  if (e != cudaSuccess) return e;
  const int num_m = (int)((c.M + BM - 1) / BM), num_n = (int)((c.N + BN - 1) / BN);
  const int tiles = num_m * num_n;
  const int sms = device_sm_count();
  const int grid = tiles < sms ? tiles : sms;
  const int a_vec = (c.K % 4 == 0) && ((reinterpret_cast<uintptr_t>(c.w) & 15u) == 0);
  k<<<grid, 288, smem, s>>>(c, num_m, num_n, num_m, a_vec);
  note_launch();
  return cudaGetLastError();
}

}  // namespace

bool tc_gemm_supported(const GemmArgs& a) {
  const bool aligned = ((reinterpret_cast<uintptr_t>(a.mat1) | reinterpret_cast<uintptr_t>(a.mat2)) &
                        15u) == 0;
  const double tiles = (double)((a.M + BM - 1) / BM) * (double)((a.N + BN - 1) / BN);
  return a.K % 4 == 0 && a.N % 4 == 0 && aligned && tiles < 2147483647.0 && encode_fn() != nullptr;
}

cudaError_t launch_tc_gemm(const GemmArgs& g, bool three_pass, cudaStream_t s) {
  if (!tc_gemm_supported(g)) return cudaErrorNotSupported;
  CUtensorMap ta, tb;
  if (!encode_2d(&ta, g.mat1, (uint64_t)g.K, (uint64_t)g.M, BM)) return cudaErrorInvalidValue;
  if (!encode_2d(&tb, g.mat2, (uint64_t)g.N, (uint64_t)g.K, BK)) return cudaErrorInvalidValue;
  return three_pass ? run_gemm<true>(g, ta, tb, s) : run_gemm<false>(g, ta, tb, s);
}

bool tc_conv_supported(const ConvArgs& c) {
  const double tiles = (double)((c.M + BM - 1) / BM) * (double)((c.N + BN - 1) / BN);
  return tiles < 2147483647.0;
}

cudaError_t launch_tc_conv(const ConvArgs& c, bool three_pass, cudaStream_t s) {
  if (!tc_conv_supported(c)) return cudaErrorNotSupported;
  return three_pass ? run_conv<true>(c, s) : run_conv<false>(c, s);
}

cudaError_t tc_take_watchdog(int* value, cudaStream_t s) {
  cudaError_t e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return e;
  e = cudaMemcpyFromSymbol(value, g_watchdog, sizeof(int));
  if (e != cudaSuccess) return e;
  const int zero = 0;
  return cudaMemcpyToSymbol(g_watchdog, &zero, sizeof(int));
}

}  // namespace imc
