// Device pieces shared by the tcgen05 kernels: bounded barrier waits, the
// TF32 hi / lo split, K-major swizzled tile addressing, tile rasterisation and
// the TMEM -> global epilogue.  Each kernel file includes this header once.
#pragma once

#include <cuda.h>

#include "imc_internal.cuh"
#include "ptx.cuh"

namespace imc {
namespace tc {

constexpr int BM = 128;     // rows of one MMA tile (TMEM lanes)
constexpr int UK = 8;       // K of one tcgen05.mma kind::tf32
constexpr int EPI_PITCH = 36;  // floats per staged epilogue row
constexpr int EPI_BYTES = 4 * 32 * EPI_PITCH * 4;
constexpr int MAX_STAGES = 8;
constexpr uint32_t TMEM_COLS = 512;
constexpr uint64_t kWaitLimitNs = 2000000000ull;
constexpr uint64_t kDrainLimitNs = 200000000ull;

enum WaitSite {
  kSiteProducerEmpty = 1,
  kSiteSplitFull = 2,
  kSiteMmaAccEmpty = 3,
  kSiteMmaOperands = 4,
  kSiteEpilogueAccFull = 5,
  kSiteSelfTest = 6,  // imc_selftest_wait_timeout: a wait nothing completes
  kSiteSlabFull = 7,   // conv gather waiting for its input slab
  kSiteSlabEmpty = 8,  // conv slab producer waiting for a free slab buffer
};

struct Ctl {
  uint64_t full[MAX_STAGES];   // operands of a stage are in shared memory
  uint64_t split[MAX_STAGES];  // the split / transform step of a stage is done
  uint64_t empty[MAX_STAGES];  // the MMAs reading a stage are done
  uint64_t accf[2];            // accumulator buffer holds a finished tile
  uint64_t acce[2];            // epilogue has drained an accumulator buffer
  uint64_t drain;              // all MMAs of this CTA are done
  uint32_t tmem_base;
  int abort;
};

// Waits for the phase with the given parity; gives up after limit_ns
// (recording `site` in *watchdog and raising the CTA's abort flag) or when
// another role has raised the abort flag.
__device__ __forceinline__ bool wait_bar(uint64_t* bar, uint32_t parity, volatile int* abort,
                                         int site, int* watchdog,
                                         uint64_t limit_ns = kWaitLimitNs) {
  if (ptx::mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = ptx::globaltimer_ns();
  for (uint32_t it = 1;; ++it) {
    if (ptx::mbar_try_wait(bar, parity)) return true;
    if ((it & 127u) == 0) {
      if (*abort) return false;
      if (ptx::globaltimer_ns() - t0 > limit_ns) {
        *abort = 1;
        atomicCAS(watchdog, 0, site);
        return false;
      }
    }
  }
}

// wait_bar for a whole warp: lane 0 polls, the result is broadcast, and the
// warp leaves converged (32 lanes spinning on one barrier only add shared-
// memory traffic and issue slots).
__device__ __forceinline__ bool warp_wait_bar(uint64_t* bar, uint32_t parity, volatile int* abort,
                                              int site, int* watchdog) {
  int ok = 1;
  if ((threadIdx.x & 31) == 0) ok = wait_bar(bar, parity, abort, site, watchdog) ? 1 : 0;
  return __shfl_sync(0xffffffffu, ok, 0) != 0;
}

// Teardown wait: ignores the abort flag, gives up after kDrainLimitNs.
__device__ __forceinline__ void drain_wait(uint64_t* bar, uint32_t parity) {
  const uint64_t t0 = ptx::globaltimer_ns();
  while (!ptx::mbar_try_wait(bar, parity)) {
    if (ptx::globaltimer_ns() - t0 > kDrainLimitNs) break;
  }
}

// Named barrier 1 over the four epilogue warps; epi_any also ORs a flag
// across them (so that they leave their loop together).
__device__ __forceinline__ void epi_sync() { asm volatile("bar.sync 1, 128;" ::: "memory"); }
__device__ __forceinline__ bool epi_any(bool v) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "bar.red.or.pred q, 1, 128, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"((uint32_t)v)
      : "memory");
  return r != 0;
}

__device__ __forceinline__ void init_barriers(Ctl* ctl, int stages, uint32_t full_count,
                                              uint32_t split_count) {
  for (int s = 0; s < stages; ++s) {
    ptx::mbar_init(&ctl->full[s], full_count);
    ptx::mbar_init(&ctl->split[s], split_count);
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

// The tensor core reads an fp32 operand as TF32 by dropping its 13 low
// mantissa bits (measured on GB300: round toward zero), so hi = v with those
// bits cleared is what it sees of v, and lo = v - hi is exact in fp32.
__device__ __forceinline__ float tf32_hi(float v) {
  return __uint_as_float(__float_as_uint(v) & 0xFFFFE000u);
}
__device__ __forceinline__ float tf32_lo(float v) {
  return isfinite(v) ? v - tf32_hi(v) : 0.0f;
}
__device__ __forceinline__ float4 tf32_lo4(float4 v) {
  return make_float4(tf32_lo(v.x), tf32_lo(v.y), tf32_lo(v.z), tf32_lo(v.w));
}
__device__ __forceinline__ float4 tf32_hi4(float4 v) {
  return make_float4(tf32_hi(v.x), tf32_hi(v.y), tf32_hi(v.z), tf32_hi(v.w));
}

// K-major tile with 64-byte rows (16 fp32 of K) and the 64-byte swizzle:
// 8-row groups of 512 B; inside a row the 16-byte unit u sits at u ^ ((row/2) % 4).
// This is the layout a TMA box {16, rows} with CU_TENSOR_MAP_SWIZZLE_64B writes.
__device__ __forceinline__ int sw64_row_base(int row) { return (row >> 3) * 512 + (row & 7) * 64; }
__device__ __forceinline__ int sw64_unit(int row, int u) { return ((u ^ ((row >> 1) & 3))) << 4; }

// UMMA shared-memory descriptor of a K-major SW64 tile; k-step `ks` (8 fp32)
// is 32 B into the 64-byte row.
__device__ __forceinline__ uint64_t sw64_desc(uint32_t tile_addr, int ks) {
  return ptx::smem_desc(tile_addr + ks * 32, 16, 512, ptx::kSwizzle64B);
}

// Grouped raster.  group > 0: `group` M-tiles share each N-tile before moving
// on to the next N-tile; group < 0: -group N-tiles share each M-tile.  Either
// way the CTAs resident at one time reuse the same operand panels from L2.
__device__ __forceinline__ void tile_coords(int t, int num_m, int num_n, int group, int& mt,
                                            int& nt) {
  const bool along_n = group < 0;
  const int g = along_n ? -group : group;
  const int major = along_n ? num_n : num_m, minor = along_n ? num_m : num_n;
  const int per = g * minor;
  const int gi = t / per;
  const int first = gi * g;
  const int width = min(g, major - first);
  const int r = t - gi * per;
  const int a = first + r % width, b = r / width;
  mt = along_n ? b : a;
  nt = along_n ? a : b;
}

// The first 1024-byte aligned byte of the dynamic shared memory, as an offset
// into the __shared__ array: pointers derived from it stay shared-memory
// pointers (one made from an integer would be generic, and generic accesses
// measured ~1 % slower on the addmm, ~6 % on a short one).
__device__ __forceinline__ uint8_t* smem_align1024(uint8_t* smem_raw) {
  return smem_raw + ((1024u - (ptx::smem_addr(smem_raw) & 1023u)) & 1023u);
}

// Reads `ncols` (a multiple of 16) accumulator columns of the 32 rows this
// warp owns (TMEM lanes 32q .. 32q+31, starting at column `col`), transposes
// each 32x32 block through the warp's staging area and hands 16-byte row
// segments to the store functor: first store.load(row, col) for all eight
// segments a lane handles in the block (so their global reads are in flight
// together), then store(row, col, acc, loaded) for each.
// With `release` given, the thread arrives on it (after a tcgen05 fence) as
// soon as its last columns are in registers, so the MMA can reuse the
// accumulator while the stores finish; otherwise the caller arrives after.
// When ncols ends halfway through a 32-column block, the block's last load
// reads 16 columns past the tile (inside the TMEM allocation) and the store
// functor, which bounds its columns by the tile's end, drops them.
template <class StoreFn>
__device__ __forceinline__ void drain_accumulator(uint32_t tmem, int q, uint32_t col, int ncols,
                                                  float* stage, const StoreFn& store,
                                                  uint64_t* release = nullptr) {
  const int lane = threadIdx.x & 31;
  const uint32_t tbase = tmem + ((uint32_t)(q * 32) << 16) + col;
#pragma unroll 1
  for (int c = 0; c < ncols; c += 32) {
    uint32_t r[32];
    ptx::tmem_ld32(tbase + (uint32_t)c, r);
    ptx::tmem_ld_wait();
    if (release && c + 32 >= ncols) {
      ptx::tc_fence_before();
      ptx::mbar_arrive(release);
    }
    float4* dst = reinterpret_cast<float4*>(stage + lane * EPI_PITCH);
#pragma unroll
    for (int j = 0; j < 8; ++j)
      dst[j] = make_float4(__uint_as_float(r[4 * j]), __uint_as_float(r[4 * j + 1]),
                           __uint_as_float(r[4 * j + 2]), __uint_as_float(r[4 * j + 3]));
    __syncwarp();
    float4 pre[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) pre[i] = store.load(q * 32 + i * 4 + (lane >> 3), c + (lane & 7) * 4);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int rr = i * 4 + (lane >> 3), cc = (lane & 7) * 4;
      store(q * 32 + rr, c + cc, *reinterpret_cast<const float4*>(stage + rr * EPI_PITCH + cc),
            pre[i]);
    }
    __syncwarp();
  }
}

}  // namespace tc
}  // namespace imc
