// tcgen05 tensor-core conv2d (groups == 1, NCHW) as an implicit-im2col GEMM.
//
// Semantics: ExecuTorch WebGPU "et_vk conv2d: route standard (groups==1) conv
// through an im2col tiled GEMM", Solution and Implementation paragraphs:
// GEMM M = OC, N = B*OH*OW, K = IC*KH*KW; the weight is the [OC, K] operand;
// the input is im2col-sampled on the fly (n -> (b, oh, ow), kk -> (ic, kh, kw),
// ih = oh*sH - pH + kh*dH, likewise iw, out-of-range taps read 0); bias per
// output channel; NCHW output.
//
// Layout for sm_103a.  The kernel forms the transposed product
// D[p, oc] = sum_k im2col[p, k] * w[oc, k], so that the operand built on the
// fly is the MMA's A operand and lives in tensor memory (the tensor core then
// reads only the weight tile from shared memory, and the gather never writes
// shared memory):
//   tile        128 output positions p (TMEM lanes) x BN output channels
//               (BN at most 256, a multiple of 16, of 32 when OC needs
//               several channel tiles)
//   K order     with IC >= 8, k runs over (kh, kw, ic) inside the kernel --
//               input channel fastest -- instead of the pages' (ic, kh, kw):
//               a sum does not depend on the order of its terms up to
//               rounding, and this way the 16 k a thread gathers per k-block
//               usually share one spatial tap (one bounds check, then reads
//               at a fixed channel-plane stride).  Few channels keep the pages'
//               order, where consecutive k reuse the same input rows.
//   pre-pass    the weight is written once per call, in the kernel's K order,
//               as zero-padded rows of Kp (K rounded up to 4) fp32 -- hi part
//               and, for 3xTF32, lo part -- so that its tiles can be
//               TMA-loaded whatever K is
//   warps 0-7   im2col gather: warp w fills TMEM lanes 32*(w%4) .. +31 (32
//               positions) with all 16 k of every other k-block (those whose
//               index has parity w/4); the values of its next k-block are in
//               flight while one is split into TF32 hi / lo and written to its
//               stage (tcgen05.st)
//   warp 8      TMA producer of the weight tiles (BN x 16 fp32, 64B swizzle)
//   warp 9      TMEM owner + MMA issuer, A from TMEM and B from shared memory:
//               A_lo*B_hi + A_hi*B_lo + A_hi*B_hi per k-step of 8, or A*B
//   warps 10-13 epilogue: tcgen05.ld (one position per lane), transposed
//               through shared memory, + bias; a whole tile inside one image
//               leaves by one 3-D TMA store per 32-channel chunk, other tiles
//               (and K-slice partial sums) as 512-byte runs of positions per
//               channel
//   warp 14     slab form only (few input channels, see slab_geometry): the
//               position tile is 4 output rows x 32 output columns, and this
//               warp brings each tile's input window [IC][rows][columns] into
//               one of two shared-memory slabs by one 4-D TMA box (zeros
//               outside the image); the gather warps then read the im2col
//               values from the slab through a k offset table, and whole
//               tiles leave by 4-D TMA stores clipped at the image edges
// TMEM columns 0-255 hold the accumulator (two of 128 when BN <= 128, so the
// epilogue of one tile overlaps the next), columns 256-511 the A stages (32
// columns each: hi 0-15, lo 16-31).
// A second kernel, k_tc_conv_t (the transposed slab form, further down), takes
// the stem-like convs (IC < 8, OC <= 128, one 256-position tile per SM) the
// other way round: channels as the MMA's M, positions as N.
// Scheduling: persistent CTAs take whole tiles first.  When the last wave
// would leave SMs idle, its tiles are cut into S K-slices; a slice writes its
// partial sums to scratch and k_conv_tail adds the S partial tiles in slice
// order (the result does not depend on which CTA ran which slice).
// Every barrier wait is bounded (see tc_common.cuh).
#include <algorithm>
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
constexpr int GATHER_WARPS = 8;
constexpr int TMA_WARP = 8, MMA_WARP = 9, EPI_WARP0 = 10, SLAB_WARP = 14;
// gather forms (kernel template argument)
constexpr int GM_PAGES = 0;  // K order (ic, kh, kw), reads from global memory
constexpr int GM_ICF = 1;    // K order (kh, kw, ic), reads from global memory
constexpr int GM_SLAB = 2;   // K order (ic, kh, kw), reads an input slab in shared memory
// threads of a CTA: 14 warps, 15 with the slab producer
constexpr int threads_of(int gm) { return (gm == GM_SLAB ? 15 : 14) * 32; }
constexpr int SLAB_ROWS = 4, SLAB_COLS = 32;  // 2-D position tile of the slab form
constexpr int kSlabMaxBytes = 48 * 1024;      // one slab buffer (two are resident)
constexpr int kSlabMaxK = 2048;               // k offset table of the slab form (8 KB)
constexpr uint32_t A_COL0 = 256, A_STAGE_COLS = 32;
constexpr int MAX_TAPS = 1024;  // KH*KW entries of the per-CTA tap table
constexpr int EPI_CHUNK_FLOATS = 32 * BM;  // one 32-channel chunk of a tile
constexpr int EPI_STAGE_BYTES = 2 * EPI_CHUNK_FLOATS * 4;  // two chunk buffers
constexpr int SMEM_LIMIT = 232448;
constexpr int kPlanSMs = 152;            // SM count the K-slice plan is made for
constexpr double kSliceLaunchKb = 8.0;   // fix-up launch, in k-block times
constexpr double kHbmBytesPerClkSm = 24.0;  // one SM's share of HBM bandwidth

__device__ int g_watchdog_conv;

// Work split and shared-memory layout, the same for every CTA of a launch.
struct Sched {
  int bn, n_oc, kb;         // channel-tile width, channel tiles, k-blocks of a whole tile
  int full, slices, units;  // whole-tile units, K-slices per tail tile, all units
  int stages, nacc;         // pipeline stages, accumulator buffers
  int w_bytes;              // weight tiles of a stage (hi [+ lo])
  int tab_bytes;            // tap table
  int tma_out;              // whole tiles inside one image leave by TMA store
  int tpi;                  // position tiles per image (0: tiles run across images)
  // slab form: a position tile is SLAB_ROWS output rows x SLAB_COLS output
  // columns (tw tiles across a row); its input window [IC][srows][sbw] (first
  // column soff floats before the first tap) comes in by one TMA box
  int slab, tw, sbw, srows, soff;
  int slab_tx, slab_stride;  // bytes of one box, bytes between the two buffers
  float* part;              // tail partial sums [units - full][bn][128]
};

struct Unit {
  int pt, ot;    // position tile, channel tile
  int kb0, kb1;  // k-block range
  int slot;      // partial-sum slot, -1 for a whole tile
};

__device__ __forceinline__ Unit decode(const Sched& q, int u) {
  Unit r;
  int t;
  if (u < q.full) {
    t = u;
    r.kb0 = 0;
    r.kb1 = q.kb;
    r.slot = -1;
  } else {
    const int v = u - q.full, tt = v / q.slices, sl = v - tt * q.slices;
    t = q.full + tt;
    r.kb0 = (int)((int64_t)sl * q.kb / q.slices);
    r.kb1 = (int)((int64_t)(sl + 1) * q.kb / q.slices);
    r.slot = v;
  }
  r.pt = t / q.n_oc;
  r.ot = t - r.pt * q.n_oc;
  return r;
}

// Positions of tile pt: p0 .. p0 + count - 1 (global position = b*OH*OW +
// oh*OW + ow).  With q.tpi > 0 each image has its own tiles (the last one of
// an image may be short), so no tile runs into the next image.
struct TilePos {
  int64_t p0;
  int count;
};
__device__ __forceinline__ TilePos tile_pos(const ConvArgs& c, const Sched& q, int pt) {
  TilePos t;
  if (q.tpi > 0) {
    const int b = pt / q.tpi, pix0 = (pt - b * q.tpi) * BM, P = c.OH * c.OW;
    t.p0 = (int64_t)b * P + pix0;
    t.count = P - pix0 < BM ? P - pix0 : BM;
  } else {
    t.p0 = (int64_t)pt * BM;
    t.count = c.N - t.p0 < BM ? (int)(c.N - t.p0) : BM;
  }
  return t;
}

// Slab form: image and top-left output position of position tile pt.
struct Tile2 {
  int b, oh0, ow0;
};
__device__ __forceinline__ Tile2 tile2d(const Sched& q, int pt) {
  Tile2 t;
  t.b = pt / q.tpi;
  const int r = pt - t.b * q.tpi, rt = r / q.tw;
  t.oh0 = rt * SLAB_ROWS;
  t.ow0 = (r - rt * q.tw) * SLAB_COLS;
  return t;
}

// ------------------------------------------------------- weight pre-pass
// Column k of row oc takes w[oc, ic, kh, kw]: k = ic*taps + tap (the pages'
// order) or, with icf, k = tap*IC + ic (tap = kh*KW + kw).  w_hi gets its TF32
// part (0 for k >= K), w_lo the rest.  Thread = column k (grid-stride in x),
// rows 4 at a time (loads first) from 4*blockIdx.y in steps of 4*gridDim.y.
// The grid is sized to be resident at once beside the main kernel's CTAs, so
// that the main kernel (launched as its dependent) starts without waiting for
// pre-pass blocks to drain.  The pre-pass is itself launched as the dependent
// of the kernel before it: its blocks wait for that kernel to complete (it may
// still read the planes, or write w or x), and only then let the main kernel
// launch, so that the main kernel may read x from its first instruction.
__global__ void __launch_bounds__(256) k_prep_w(const float* __restrict__ w, int OC, int K, int Kp,
                                                int IC, int taps, int icf, float* __restrict__ w_hi,
                                                float* __restrict__ w_lo) {
  ptx::griddep_wait();    // the kernel before this one has completed
  ptx::griddep_launch();  // the main kernel may start its prologue and gathers
  for (int k = blockIdx.x * blockDim.x + threadIdx.x; k < Kp; k += gridDim.x * blockDim.x) {
    int src = k;
    if (icf) {
      const int tap = k / IC;
      src = (k - tap * IC) * taps + tap;
    }
    for (int oc0 = 4 * (int)blockIdx.y; oc0 < OC; oc0 += 4 * (int)gridDim.y) {
      float v[4];
#pragma unroll
      for (int i = 0; i < 4; ++i)
        v[i] = (oc0 + i < OC && k < K) ? __ldg(w + (int64_t)(oc0 + i) * K + src) : 0.0f;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        if (oc0 + i >= OC) break;
        const int64_t e = (int64_t)(oc0 + i) * Kp + k;
        if (w_lo) {
          w_hi[e] = tf32_hi(v[i]);
          w_lo[e] = tf32_lo(v[i]);
        } else {
          w_hi[e] = v[i];
        }
      }
    }
  }
}

// Two register buffers of gathered values, alternated by unrolling (copying a
// buffer whose loads are in flight would wait for them): the 16 values of a
// warp's next k-block are in flight while one k-block is stored.
template <class Gather, class Store>
__device__ __forceinline__ bool rotate2(int nkb, Gather& gather, Store& store) {
  float va[BK], vb[BK];
  gather(va);
  for (int i = 0; i < nkb; i += 2) {
    if (i + 1 < nkb) gather(vb);
    if (!store(va)) return false;
    if (i + 1 >= nkb) break;
    if (i + 2 < nkb) gather(va);
    if (!store(vb)) return false;
  }
  return true;
}

// ------------------------------------------------------------ main kernel
template <bool THREE, int GM>
__global__ void __launch_bounds__(threads_of(GM), 1)
    k_tc_conv(const __grid_constant__ CUtensorMap tmWh, const __grid_constant__ CUtensorMap tmWl,
              const __grid_constant__ CUtensorMap tmO, const __grid_constant__ CUtensorMap tmX,
              const ConvArgs c, const Sched q) {
  constexpr bool ICF = GM == GM_ICF, SLAB = GM == GM_SLAB;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_align1024(smem_raw);
  const int b_tile = q.bn * BK * 4;  // one weight tile (hi or lo)
  // [weight stages][2 input slabs (slab form)][tap table][epilogue staging]
  // [barriers][slab barriers: full 0, 1, empty 0, 1]
  float* slab = reinterpret_cast<float*>(smem + q.stages * q.w_bytes);
  int2* tab = reinterpret_cast<int2*>(reinterpret_cast<uint8_t*>(slab) +
                                      (SLAB ? 2 * q.slab_stride : 0));
  float* epi_stage = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(tab) + q.tab_bytes);
  Ctl* ctl = reinterpret_cast<Ctl*>(reinterpret_cast<uint8_t*>(epi_stage) + EPI_STAGE_BYTES);
  uint64_t* sbar = reinterpret_cast<uint64_t*>(ctl + 1);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int taps = c.KH * c.KW;
  int* wd = &g_watchdog_conv;

  if constexpr (SLAB) {
    // k offset table: k = ic*taps + kh*KW + kw -> ic*srows*sbw + kh*dH*sbw +
    // kw*dW, the value's place in a slab relative to its position's first
    // tap (0 for k >= K, masked by the gather)
    int* koff = reinterpret_cast<int*>(tab);
    for (int k = threadIdx.x; k < q.kb * BK; k += blockDim.x) {
      int o = 0;
      if (k < c.K) {
        const int ic = k / taps, r = k - ic * taps, kh = r / c.KW, kw = r - kh * c.KW;
        o = (ic * q.srows + kh * c.dH) * q.sbw + kw * c.dW;
      }
      koff[k] = o;
    }
  } else {
    // tap table: r = kh*KW + kw -> (kh*dH, kw*dW)
    for (int r = threadIdx.x; r < taps; r += blockDim.x) {
      const int kh = r / c.KW, kw = r - kh * c.KW;
      tab[r] = make_int2(kh * c.dH, kw * c.dW);
    }
  }
  // full: the 4 gather warps of the stage's k-block parity + the weight TMA
  if (threadIdx.x == 0) init_barriers(ctl, q.stages, GATHER_WARPS / 2 + 1, 1);
  // Slab form: the producer sets up its own barriers and sends the first
  // box before the CTA's set-up barrier (the input does not come from the
  // pre-pass), so that its memory latency overlaps the set-up.
  auto slab_load = [&](int u, int sb) {
    const Tile2 t = tile2d(q, decode(q, u).pt);
    ptx::mbar_arrive_expect_tx(&sbar[sb], (uint32_t)q.slab_tx);
    ptx::tma_load_4d(slab + sb * (q.slab_stride / 4), &tmX, &sbar[sb],
                     t.ow0 * c.sW - c.pW - q.soff, t.oh0 * c.sH - c.pH, 0, t.b);
  };
  if (SLAB && warp == SLAB_WARP && lane == 0) {
    for (int i = 0; i < 2; ++i) {
      ptx::mbar_init(&sbar[i], 1);                 // the producer's expect-tx
      ptx::mbar_init(&sbar[2 + i], GATHER_WARPS);  // every gather warp is done with it
    }
    ptx::fence_mbar_init();
    if ((int)blockIdx.x < q.units) slab_load((int)blockIdx.x, 0);
  }
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

  if (warp < GATHER_WARPS) {
    // ------------------------------------------------------ im2col gather
    // Warp w fills TMEM lanes 32*(w%4) .. +31 with all 16 k of the k-blocks
    // whose index in this CTA's sequence has parity w/4: each warp hands over
    // one k-block in two, so the store-and-signal latency of one k-block
    // overlaps the gather of the next in the other warp.
    const int quarter = warp & 3, par = warp >> 2;
    const int HW = c.H * c.W, ICHW = c.IC * HW, P = c.OH * c.OW;
    const uint32_t trow = tmem + ((uint32_t)(quarter * 32) << 16) + A_COL0;
    int s = 0;
    uint32_t ph = 0;
    int64_t g0 = 0;  // index of the unit's first k-block in this CTA's sequence
    bool ok = true;
    // Splits the 16 values of a k-block into TF32 hi / lo and writes them to
    // the stage's TMEM columns; then arrives on the stage's full barrier and
    // moves to this warp's next stage (two k-blocks on).
    auto put_issue = [&](const float (&v)[BK]) {
      const uint32_t ta = trow + (uint32_t)s * A_STAGE_COLS;
      if (THREE) {
        float hi[BK], lo[BK];
#pragma unroll
        for (int j = 0; j < BK; ++j) {
          hi[j] = tf32_hi(v[j]);
          lo[j] = tf32_lo(v[j]);
        }
        ptx::tmem_st16(ta, hi);
        ptx::tmem_st16(ta + 16, lo);
      } else {
        ptx::tmem_st16(ta, v);  // the tensor core reads it as TF32
      }
    };
    auto put_commit = [&]() {
      ptx::tmem_st_wait();
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(&ctl->full[s]);
      s += 2;
      if (s >= q.stages) {
        s -= q.stages;
        ph ^= 1u;
      }
    };
    auto put = [&](const float (&v)[BK]) {
      put_issue(v);
      put_commit();
    };
    auto store = [&](const float (&v)[BK]) -> bool {
      if (!warp_wait_bar(&ctl->empty[s], ph ^ 1u, abort, kSiteProducerEmpty, wd)) return false;
      ptx::tc_fence_after();
      put(v);
      return true;
    };
    int ul = 0;  // units of this CTA so far
    for (int u = blockIdx.x; u < q.units && ok; u += gridDim.x, ++ul) {
      const Unit un = decode(q, u);
      const int nkb_unit = un.kb1 - un.kb0;
      const int i0 = (int)((par ^ g0) & 1);  // this warp's first k-block of the unit
      const int nkb = nkb_unit > i0 ? (nkb_unit - i0 + 1) / 2 : 0;
      {
        const int64_t g = g0 + i0;
        s = (int)(g % q.stages);
        ph = (uint32_t)((g / q.stages) & 1);
      }
      g0 += nkb_unit;
      const int k0 = (un.kb0 + i0) * BK;
      if constexpr (SLAB) {
        // Every gather warp waits for the unit's slab (so that its arrival
        // below counts toward this use of the buffer), reads it, and hands
        // the buffer back.  Lane = output column ow0 + lane, quarter = output
        // row oh0 + quarter; the slab holds input rows oh0*sH - pH .. and
        // columns ow0*sW - pW - soff .., zeros outside the image.
        const int sb = ul & 1;
        if (!warp_wait_bar(&sbar[sb], (uint32_t)(ul >> 1) & 1u, abort, kSiteSlabFull, wd)) {
          ok = false;
          break;
        }
        if (nkb > 0) {
          const float* sl = slab + sb * (q.slab_stride / 4) + quarter * c.sH * q.sbw +
                            lane * c.sW + q.soff;
          const int* koff = reinterpret_cast<const int*>(tab);
          int kk = k0;  // first k of this warp's next k-block
          // 16 offsets by four broadcast loads, then 16 independent loads
          // (an offset past K is 0, inside the slab; the value is masked)
          auto gather = [&](float (&v)[BK]) {
            int o[BK];
#pragma unroll
            for (int j = 0; j < BK; j += 4) {
              const int4 t = *reinterpret_cast<const int4*>(koff + kk + j);
              o[j] = t.x;
              o[j + 1] = t.y;
              o[j + 2] = t.z;
              o[j + 3] = t.w;
            }
#pragma unroll
            for (int j = 0; j < BK; ++j) {
              const float xv = sl[o[j]];
              v[j] = kk + j < c.K ? xv : 0.0f;
            }
            kk += 2 * BK;
          };
          // the TMEM stores of one k-block complete while the next is gathered
          float va[BK], vb[BK];
          gather(va);
          for (int i = 0; i < nkb; i += 2) {
            if (!warp_wait_bar(&ctl->empty[s], ph ^ 1u, abort, kSiteProducerEmpty, wd)) {
              ok = false;
              break;
            }
            ptx::tc_fence_after();
            put_issue(va);
            if (i + 1 < nkb) gather(vb);
            put_commit();
            if (i + 1 >= nkb) break;
            if (!warp_wait_bar(&ctl->empty[s], ph ^ 1u, abort, kSiteProducerEmpty, wd)) {
              ok = false;
              break;
            }
            ptx::tc_fence_after();
            put_issue(vb);
            if (i + 2 < nkb) gather(va);
            put_commit();
          }
        }
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(&sbar[2 + sb]);
        continue;
      }
      if (nkb == 0) continue;
      const TilePos tp = tile_pos(c, q, un.pt);
      const int64_t p = tp.p0 + quarter * 32 + lane;
      const bool pok = quarter * 32 + lane < tp.count;
      int b = 0, ih0 = 0, iw0 = 0;
      if (pok) {
        b = (int)(p / P);
        const int pix = (int)(p - (int64_t)b * P);
        const int oh = pix / c.OW, ow = pix - oh * c.OW;
        ih0 = oh * c.sH - c.pH;
        iw0 = ow * c.sW - c.pW;
      }
      const float* xb = c.x + (int64_t)b * ICHW;
      if constexpr (ICF) {
        // running position of this warp's next k = tap*IC + ic: the tap's
        // validity and in-plane offset, and the channel plane offset ic*H*W
        int tap = k0 / c.IC, ic = k0 - tap * c.IC, ic_hw = ic * HW;
        bool tap_in = false;
        int tap_off = 0;
        auto set_tap = [&]() {
          tap_in = false;
          if (pok && tap < taps) {
            const int2 d = tab[tap];
            const int ih = ih0 + d.x, iw = iw0 + d.y;
            tap_in = (unsigned)ih < (unsigned)c.H && (unsigned)iw < (unsigned)c.W;
            tap_off = ih * c.W + iw;
          }
        };
        set_tap();
        // The 16 values of one k-block (0 past K, outside the image, or past
        // the last position), then skip the other warp's k-block.
        auto gather = [&](float (&v)[BK]) {
#pragma unroll
          for (int j = 0; j < BK; ++j) {
            v[j] = tap_in ? __ldg(xb + (ic_hw + tap_off)) : 0.0f;
            ic_hw += HW;
            if (++ic == c.IC) {
              ic = 0;
              ic_hw = 0;
              ++tap;
              set_tap();
            }
          }
          ic += BK;
          if (ic >= c.IC) {
            while (ic >= c.IC) {
              ic -= c.IC;
              ++tap;
            }
            set_tap();
          }
          ic_hw = ic * HW;
        };
        if (c.IC % BK == 0) {
          // a k-block lies in one tap: one bounds check per k-block, then 16
          // loads at the channel-plane stride (ic, tap: this warp's next k)
          auto gather16 = [&](float (&v)[BK]) {
            const float* src = xb + (ic_hw + tap_off);
#pragma unroll
            for (int j = 0; j < BK; ++j) v[j] = tap_in ? __ldg(src + j * HW) : 0.0f;
            ic += 2 * BK;
            if (ic >= c.IC) {  // a later tap: ic stays a multiple of 16
              while (ic >= c.IC) {
                ic -= c.IC;
                ++tap;
              }
              set_tap();
            }
            ic_hw = ic * HW;
          };
          ok = rotate2(nkb, gather16, store);
        } else {
          ok = rotate2(nkb, gather, store);
        }
      } else {
        // running (ic, r) of this warp's next k = ic*taps + r
        int ic_hw = (k0 / taps) * HW, r = k0 - (k0 / taps) * taps;
        auto gather = [&](float (&v)[BK]) {
#pragma unroll
          for (int j = 0; j < BK; ++j) {
            const int2 d = tab[r];
            const int ih = ih0 + d.x, iw = iw0 + d.y;
            const bool in = pok && ic_hw < ICHW && (unsigned)ih < (unsigned)c.H &&
                            (unsigned)iw < (unsigned)c.W;
            v[j] = in ? __ldg(xb + (ic_hw + ih * c.W + iw)) : 0.0f;
            if (++r == taps) {
              r = 0;
              ic_hw += HW;
            }
          }
          r += BK;
          while (r >= taps) {
            r -= taps;
            ic_hw += HW;
          }
        };
        ok = rotate2(nkb, gather, store);
      }
    }
  } else if (warp == TMA_WARP) {
    // ------------------------------------------------ weight TMA producer
    if (lane == 0) {
      ptx::griddep_wait();  // the weight planes come from the pre-pass
      int s = 0, issued = 0;
      uint32_t ph = 0;
      for (int u = blockIdx.x; u < q.units && !*abort; u += gridDim.x) {
        const Unit un = decode(q, u);
        for (int kb = un.kb0; kb < un.kb1; ++kb) {
          if (!wait_bar(&ctl->empty[s], ph ^ 1u, abort, kSiteProducerEmpty, wd)) break;
          uint8_t* st = smem + s * q.w_bytes;
          ptx::mbar_arrive_expect_tx(&ctl->full[s], (uint32_t)q.w_bytes);
          ptx::tma_load_2d(st, &tmWh, &ctl->full[s], kb * BK, un.ot * q.bn);
          if (THREE) ptx::tma_load_2d(st + b_tile, &tmWl, &ctl->full[s], kb * BK, un.ot * q.bn);
          ++issued;
          if (++s == q.stages) {
            s = 0;
            ph ^= 1u;
          }
        }
      }
      // this CTA's last loads are out: the slice-sum kernel or the next call's
      // weight pre-pass may launch (each waits for this kernel).  Its blocks
      // fit beside this kernel's CTAs, so they spread over all SMs (unlike the
      // addmm's, see k_tc_gemm), and the pre-pass starts the moment this
      // kernel ends (measured 2-3 us faster per call back to back)
      ptx::griddep_launch();
      for (int j = (issued > q.stages ? issued - q.stages : 0); j < issued; ++j)
        drain_wait(&ctl->full[j % q.stages], (uint32_t)((j / q.stages) & 1));
    }
  } else if (warp == MMA_WARP) {
    // --------------------------------------------------------- MMA issuer
    if (lane == 0) {
      const uint32_t idesc = ptx::idesc_tf32(BM, (uint32_t)q.bn, false, false);
      // Operand addresses advance by constants (the issuing thread's few
      // instructions between MMAs are on the pipeline's critical path):
      // B descriptors of stage s at k-step 0 = b0 + s * (w_bytes >> 4) (a
      // descriptor holds the address >> 4 in its low 14 bits); k-step 1 adds
      // 32 bytes (2), the lo tile b_tile bytes; the A stage's TMEM columns.
      const uint64_t b0 = sw64_desc(ptx::smem_addr(smem), 0);
      const uint64_t b_step = (uint64_t)(q.w_bytes >> 4), lo = (uint64_t)(b_tile >> 4);
      const uint32_t a0 = tmem + A_COL0;
      uint64_t bs = b0;
      uint32_t as = a0;
      int s = 0, ul = 0;
      uint32_t ph = 0;
      for (int u = blockIdx.x; u < q.units; u += gridDim.x, ++ul) {
        const Unit un = decode(q, u);
        const int buf = ul % q.nacc;
        const uint32_t use = (uint32_t)(ul / q.nacc);
        if (!wait_bar(&ctl->acce[buf], (use & 1u) ^ 1u, abort, kSiteMmaAccEmpty, wd)) break;
        ptx::tc_fence_after();
        const uint32_t d = tmem + (uint32_t)buf * 128u;
        bool ok = true;
        for (int kb = un.kb0; kb < un.kb1; ++kb) {
          if (!wait_bar(&ctl->full[s], ph, abort, kSiteMmaOperands, wd)) {
            ok = false;
            break;
          }
          ptx::tc_fence_after();
          const uint32_t acc = kb > un.kb0 ? 1u : 0u;
          if (THREE) {  // k-step 0, then k-step 1 (TMEM columns + UK, descriptors + 2)
            ptx::mma_tf32_ts(d, as + 16u, bs, idesc, acc);       // A_lo * B_hi
            ptx::mma_tf32_ts(d, as, bs + lo, idesc, 1u);         // A_hi * B_lo
            ptx::mma_tf32_ts(d, as, bs, idesc, 1u);              // A_hi * B_hi
            ptx::mma_tf32_ts(d, as + 16u + UK, bs + 2, idesc, 1u);
            ptx::mma_tf32_ts(d, as + UK, bs + lo + 2, idesc, 1u);
            ptx::mma_tf32_ts(d, as + UK, bs + 2, idesc, 1u);
          } else {
            ptx::mma_tf32_ts(d, as, bs, idesc, acc);
            ptx::mma_tf32_ts(d, as + UK, bs + 2, idesc, 1u);
          }
          ptx::mma_commit(&ctl->empty[s]);
          // next stage, by selects (no branch between this k-block's MMAs and the next wait)
          const bool wrap = ++s == q.stages;
          s = wrap ? 0 : s;
          ph ^= wrap ? 1u : 0u;
          bs = wrap ? b0 : bs + b_step;
          as = wrap ? a0 : as + A_STAGE_COLS;
        }
        if (!ok) break;
        ptx::mma_commit(&ctl->accf[buf]);
      }
      ptx::mma_commit(&ctl->drain);
      drain_wait(&ctl->drain, 0);
    }
    __syncwarp();
  } else if (warp == SLAB_WARP) {
    // ------------------------------------- input slab producer (slab form)
    // One TMA box [IC][srows][sbw] per unit, into buffer (unit & 1) once the
    // gather warps have handed it back; the box may start before the image
    // (column a multiple of 4, zeros there) and run past its end.
    if (SLAB && lane == 0) {
      int ul = (int)blockIdx.x < q.units ? 1 : 0;  // the first box went out before set-up
      for (int u = blockIdx.x + ul * gridDim.x; u < q.units && !*abort; u += gridDim.x, ++ul) {
        const int sb = ul & 1;
        if (!wait_bar(&sbar[2 + sb], ((uint32_t)(ul >> 1) & 1u) ^ 1u, abort, kSiteSlabEmpty, wd))
          break;
        slab_load(u, sb);
      }
      for (int j = (ul > 2 ? ul - 2 : 0); j < ul; ++j)  // the boxes still in flight land
        drain_wait(&sbar[j & 1], (uint32_t)(j >> 1) & 1u);
    }
  } else {
    // ----------------------------------------------------------- epilogue
    // Per 32-channel chunk: TMEM -> registers -> a [32 channels][128
    // positions] block in shared memory (two blocks, alternating); the
    // accumulator is released as soon as its last chunk is in registers.  A
    // whole tile inside one image (q.tma_out) gets bias / ReLU on the way into
    // the block and leaves by one TMA store per chunk; otherwise warp q writes
    // channels 8q .. 8q+7 of the chunk, each as one 512-byte run of positions
    // (lane l stores positions 4l .. 4l+3 with one 16-byte store).
    const int quarter = warp & 3, row = quarter * 32 + lane;
    const bool issuer = warp == EPI_WARP0 && lane == 0;  // TMA stores
    const int64_t P = (int64_t)c.OH * c.OW;
    int ul = 0, nchunk = 0;
    for (int u = blockIdx.x; u < q.units; u += gridDim.x, ++ul) {
      const Unit un = decode(q, u);
      const int buf = ul % q.nacc;
      const uint32_t use = (uint32_t)(ul / q.nacc);
      const bool ok = warp_wait_bar(&ctl->accf[buf], use & 1u, abort, kSiteEpilogueAccFull, wd);
      if (epi_any(!ok)) break;
      ptx::tc_fence_after();
      const TilePos tp = tile_pos(c, q, un.pt);
      const int64_t p0 = tp.p0, plast = tp.p0 + tp.count - 1;
      const int b0 = (int)(p0 / P);
      // slab form: every whole tile leaves by TMA (4-D box, clipped at the
      // image's right and bottom edges); only K-slice partial sums do not
      const bool by_tma = SLAB ? un.slot < 0 : q.tma_out && un.slot < 0 && plast / P == b0;
      // this lane's four positions in the store phase
      const int64_t pq = p0 + 4 * lane;
      const int left = tp.count - 4 * lane;
      const int nvalid = left <= 0 ? 0 : (left < 4 ? left : 4);
      int64_t obase = 0;  // out offset of (b, oc = 0, position pq)
      if (nvalid > 0) {
        const int64_t b = pq / P;
        obase = b * c.OC * P + (pq - b * P);
      }
      // P % 4 == 0 and a 16-byte aligned out: the four positions are in one
      // image and form one aligned float4
      const bool vec = nvalid == 4 && c.vec_out;
      const int oc0 = un.ot * q.bn;
      const uint32_t tacc = tmem + ((uint32_t)(quarter * 32) << 16) + (uint32_t)buf * 128u;
#pragma unroll 1
      for (int cc = 0; cc < q.bn; cc += 32, ++nchunk) {
        uint32_t r[32];
        ptx::tmem_ld32(tacc + (uint32_t)cc, r);
        ptx::tmem_ld_wait();
        if (cc + 32 >= q.bn) {  // the whole accumulator is read: hand it back
          ptx::tc_fence_before();
          ptx::mbar_arrive(&ctl->acce[buf]);
        }
        // bias of chunk channel `lane`, handed out by shuffle
        const int my_oc = oc0 + cc + lane;
        const float my_bias =
            (un.slot < 0 && c.bias && cc + lane < q.bn && my_oc < c.OC) ? __ldg(c.bias + my_oc)
                                                                          : 0.0f;
        float* blk = epi_stage + (nchunk & 1) * EPI_CHUNK_FLOATS;
        if (issuer) ptx::bulk_wait_read1();  // the store from this block two chunks ago
        epi_sync();  // ... and the plain stores of that chunk are done with it
        if (by_tma) {
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            float o = __uint_as_float(r[j]) + __shfl_sync(0xffffffffu, my_bias, j);
            if (c.relu) o = fmaxf(o, 0.0f);
            blk[j * BM + row] = o;
          }
          ptx::fence_proxy_async_smem();
          epi_sync();
          if (issuer) {
            if constexpr (SLAB) {
              const Tile2 t = tile2d(q, un.pt);
              ptx::tma_store_4d(&tmO, blk, t.ow0, t.oh0, oc0 + cc, t.b);
            } else {
              ptx::tma_store_3d(&tmO, blk, (int)(p0 - (int64_t)b0 * P), oc0 + cc, b0);
            }
            ptx::bulk_commit();
          }
          continue;
        }
#pragma unroll
        for (int j = 0; j < 32; ++j) blk[j * BM + row] = __uint_as_float(r[j]);
        epi_sync();
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const int jj = quarter * 8 + i, col = cc + jj;  // channel in chunk / in tile
          const float bv = __shfl_sync(0xffffffffu, my_bias, jj);
          const float4 v = *reinterpret_cast<const float4*>(blk + jj * BM + 4 * lane);
          if (col >= q.bn) continue;
          if (un.slot >= 0) {  // K-slice partial sums: [slot][col][128 positions]
            *reinterpret_cast<float4*>(q.part + ((int64_t)un.slot * q.bn + col) * BM + 4 * lane) =
                v;
            continue;
          }
          const int oc = oc0 + col;
          if (oc >= c.OC) continue;
          float o[4] = {v.x + bv, v.y + bv, v.z + bv, v.w + bv};
          if (c.relu) {
#pragma unroll
            for (int k = 0; k < 4; ++k) o[k] = fmaxf(o[k], 0.0f);
          }
          if (vec) {
            *reinterpret_cast<float4*>(c.out + obase + (int64_t)oc * P) =
                make_float4(o[0], o[1], o[2], o[3]);
          } else {
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              if (k < nvalid) {
                const int64_t pk = pq + k, b = pk / P;
                c.out[(b * c.OC + oc) * P + (pk - b * P)] = o[k];
              }
            }
          }
        }
      }
    }
    if (issuer) ptx::bulk_wait_all();  // every TMA store has landed before the CTA ends
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (warp == MMA_WARP) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, TMEM_COLS);
  }
}

// ------------------------------------------ transposed slab form (k_tc_conv_t)
// For few input channels, at most 128 output channels and one 256-position
// tile per CTA over 3/4 of the SMs or more, the product is taken the other
// way round:
// D[oc, p] = sum_k w[oc, k] * im2col[p, k], 128 channels (M, TMEM lanes) x 256
// positions (N, TMEM columns) per MMA, both operands in shared memory.  A
// position tile is ST_ROWS x ST_COLS outputs of one image.
//   warps 0-7   gather: warp r, lane j -> output position (oh0 + r, ow0 + j),
//               row n = 32r + j of the B tiles; per k-block the position's 16
//               im2col values are read from the input slab through the k
//               offset table, split into TF32 hi / lo and stored as its
//               64-byte row (K-major, 64-byte swizzle), then fenced for the
//               tensor core
//   warp 8      TMA producer of the weight tiles (128 x 16 fp32, rows past OC
//               read as zero)
//   warp 9      TMEM owner + MMA issuer: W_lo*B_hi + W_hi*B_lo + W_hi*B_hi per
//               k-step of 8, or W*B
//   warps 10-13 epilogue: one tcgen05.ld gives a thread one channel's 32
//               positions of an output row (+ bias, + ReLU); warp q stages its
//               32 channels x 32 positions (128-byte swizzle) in the input
//               slab's space, free once the last k-block is gathered, and
//               stores them with one 4-D TMA box {32 columns, 1 row, 32
//               channels, 1 image} clipped at the output's edges
//   warp 14     the CTA's input slab [IC][srows][sbw]: one 4-D TMA box
// Stage: W_hi | W_lo | B_hi | B_lo (3xTF32) or W | B.
constexpr int ST_ROWS = 8, ST_COLS = 32, ST_POS = ST_ROWS * ST_COLS;
constexpr int ST_W_TILE = BM * BK * 4;      // 8 KB: 128 channels x 16 k
constexpr int ST_B_TILE = ST_POS * BK * 4;  // 16 KB: 256 positions x 16 k
constexpr int ST_THREADS = 15 * 32;
constexpr int kStSlabMaxBytes = 64 * 1024;
constexpr int kStEpiBytes = 4 * 2 * 4096;  // epilogue: two 4 KB blocks per warp

template <bool THREE>
__global__ void __launch_bounds__(ST_THREADS, 1)
    k_tc_conv_t(const __grid_constant__ CUtensorMap tmWh, const __grid_constant__ CUtensorMap tmWl,
                const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmO,
                const ConvArgs c, const Sched q) {
  constexpr int B_OFF = THREE ? 2 * ST_W_TILE : ST_W_TILE;  // B tiles within a stage
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_align1024(smem_raw);
  // [stages][input slab][k offset table][barriers][slab barrier]
  float* slab = reinterpret_cast<float*>(smem + q.stages * q.w_bytes);
  int* koff = reinterpret_cast<int*>(reinterpret_cast<uint8_t*>(slab) + q.slab_stride);
  Ctl* ctl = reinterpret_cast<Ctl*>(reinterpret_cast<uint8_t*>(koff) + q.tab_bytes);
  uint64_t* sbar = reinterpret_cast<uint64_t*>(ctl + 1);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int taps = c.KH * c.KW;
  int* wd = &g_watchdog_conv;
  // this CTA's position tile: image b, output rows oh0.., columns ow0..
  const int b = (int)blockIdx.x / q.tpi, r = (int)blockIdx.x - b * q.tpi, rt = r / q.tw;
  const int oh0 = rt * ST_ROWS, ow0 = (r - rt * q.tw) * ST_COLS;

  // k = ic*taps + kh*KW + kw -> ic*srows*sbw + kh*dH*sbw + kw*dW (0 past K)
  for (int k = threadIdx.x; k < q.kb * BK; k += blockDim.x) {
    int o = 0;
    if (k < c.K) {
      const int ic = k / taps, rr = k - ic * taps, kh = rr / c.KW, kw = rr - kh * c.KW;
      o = (ic * q.srows + kh * c.dH) * q.sbw + kw * c.dW;
    }
    koff[k] = o;
  }
  // full: the 8 gather warps + the weight TMA
  if (threadIdx.x == 0) init_barriers(ctl, q.stages, GATHER_WARPS + 1, 1);
  if (warp == SLAB_WARP && lane == 0) {  // the input box goes out before the set-up barrier
    ptx::mbar_init(sbar, 1);
    ptx::fence_mbar_init();
    ptx::mbar_arrive_expect_tx(sbar, (uint32_t)q.slab_tx);
    ptx::tma_load_4d(slab, &tmX, sbar, ow0 * c.sW - c.pW - q.soff, oh0 * c.sH - c.pH, 0, b);
  }
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

  if (warp < GATHER_WARPS) {
    // ------------------------------------------------------ im2col gather
    const int n = warp * 32 + lane;  // row of the B tiles
    const int row_off = sw64_row_base(n);
    if (warp_wait_bar(sbar, 0, abort, kSiteSlabFull, wd)) {
      const float* sl = slab + warp * c.sH * q.sbw + lane * c.sW + q.soff;
      int kk = 0;  // first k of the next k-block to gather
      auto gather = [&](float (&v)[BK]) {
        int o[BK];
#pragma unroll
        for (int j = 0; j < BK; j += 4) {
          const int4 t = *reinterpret_cast<const int4*>(koff + kk + j);
          o[j] = t.x;
          o[j + 1] = t.y;
          o[j + 2] = t.z;
          o[j + 3] = t.w;
        }
#pragma unroll
        for (int j = 0; j < BK; ++j) {
          const float xv = sl[o[j]];
          v[j] = kk + j < c.K ? xv : 0.0f;
        }
        kk += BK;
      };
      int s = 0;
      uint32_t ph = 0;
      auto store = [&](const float (&v)[BK]) -> bool {
        if (!warp_wait_bar(&ctl->empty[s], ph ^ 1u, abort, kSiteProducerEmpty, wd)) return false;
        uint8_t* row = smem + s * q.w_bytes + B_OFF + row_off;
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const float4 x4 = make_float4(v[4 * u], v[4 * u + 1], v[4 * u + 2], v[4 * u + 3]);
          if (THREE) {
            *reinterpret_cast<float4*>(row + sw64_unit(n, u)) = tf32_hi4(x4);
            *reinterpret_cast<float4*>(row + ST_B_TILE + sw64_unit(n, u)) = tf32_lo4(x4);
          } else {
            *reinterpret_cast<float4*>(row + sw64_unit(n, u)) = x4;  // read as TF32
          }
        }
        ptx::fence_proxy_async_smem();  // the tensor core reads what was just stored
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(&ctl->full[s]);
        if (++s == q.stages) {
          s = 0;
          ph ^= 1u;
        }
        return true;
      };
      rotate2(q.kb, gather, store);
    }
  } else if (warp == TMA_WARP) {
    // ------------------------------------------------ weight TMA producer
    if (lane == 0) {
      ptx::griddep_wait();  // the weight planes come from the pre-pass
      int s = 0, issued = 0;
      uint32_t ph = 0;
      for (int kb = 0; kb < q.kb && !*abort; ++kb) {
        if (!wait_bar(&ctl->empty[s], ph ^ 1u, abort, kSiteProducerEmpty, wd)) break;
        uint8_t* st = smem + s * q.w_bytes;
        ptx::mbar_arrive_expect_tx(&ctl->full[s], (uint32_t)(THREE ? 2 * ST_W_TILE : ST_W_TILE));
        ptx::tma_load_2d(st, &tmWh, &ctl->full[s], kb * BK, 0);
        if (THREE) ptx::tma_load_2d(st + ST_W_TILE, &tmWl, &ctl->full[s], kb * BK, 0);
        ++issued;
        if (++s == q.stages) {
          s = 0;
          ph ^= 1u;
        }
      }
      ptx::griddep_launch();  // as in k_tc_conv: the next call's weight pre-pass may launch
      for (int j = (issued > q.stages ? issued - q.stages : 0); j < issued; ++j)
        drain_wait(&ctl->full[j % q.stages], (uint32_t)((j / q.stages) & 1));
    }
  } else if (warp == MMA_WARP) {
    // --------------------------------------------------------- MMA issuer
    if (lane == 0) {
      const uint32_t idesc = ptx::idesc_tf32(BM, ST_POS, false, false);
      // descriptors as running values: stage s at k-step 0 = d0 + s * (w_bytes
      // >> 4); the W_lo / B tiles at fixed offsets; k-step 1 adds 32 bytes (2)
      const uint64_t d0 = sw64_desc(ptx::smem_addr(smem), 0);
      const uint64_t step = (uint64_t)(q.w_bytes >> 4);
      constexpr uint64_t kWlo = ST_W_TILE >> 4, kB = B_OFF >> 4,
                         kBlo = (B_OFF + ST_B_TILE) >> 4, kK1 = 2;
      uint64_t ds = d0;
      int s = 0;
      uint32_t ph = 0;
      bool ok = true;
      for (int kb = 0; kb < q.kb; ++kb) {
        if (!wait_bar(&ctl->full[s], ph, abort, kSiteMmaOperands, wd)) {
          ok = false;
          break;
        }
        ptx::tc_fence_after();
        const uint32_t acc = kb > 0 ? 1u : 0u;
        if (THREE) {
          ptx::mma_tf32(tmem, ds + kWlo, ds + kB, idesc, acc);        // W_lo * B_hi
          ptx::mma_tf32(tmem, ds, ds + kBlo, idesc, 1u);              // W_hi * B_lo
          ptx::mma_tf32(tmem, ds, ds + kB, idesc, 1u);                // W_hi * B_hi
          ptx::mma_tf32(tmem, ds + kWlo + kK1, ds + kB + kK1, idesc, 1u);
          ptx::mma_tf32(tmem, ds + kK1, ds + kBlo + kK1, idesc, 1u);
          ptx::mma_tf32(tmem, ds + kK1, ds + kB + kK1, idesc, 1u);
        } else {
          ptx::mma_tf32(tmem, ds, ds + kB, idesc, acc);
          ptx::mma_tf32(tmem, ds + kK1, ds + kB + kK1, idesc, 1u);
        }
        ptx::mma_commit(&ctl->empty[s]);
        const bool wrap = ++s == q.stages;
        s = wrap ? 0 : s;
        ph ^= wrap ? 1u : 0u;
        ds = wrap ? d0 : ds + step;
      }
      if (ok) ptx::mma_commit(&ctl->accf[0]);
      ptx::mma_commit(&ctl->drain);
      drain_wait(&ctl->drain, 0);
    }
    __syncwarp();
  } else if (warp == SLAB_WARP) {
    if (lane == 0) drain_wait(sbar, 0);  // the box has landed before the CTA ends
  } else {
    // ----------------------------------------------------------- epilogue
    const int quarter = warp & 3, oc = quarter * 32 + lane;
    const float bias = (c.bias && oc < c.OC) ? __ldg(c.bias + oc) : 0.0f;
    // a warp whose 32 channels all lie past OC has nothing to store
    if (quarter * 32 < c.OC && warp_wait_bar(&ctl->accf[0], 0, abort, kSiteEpilogueAccFull, wd)) {
      // every k-block has been gathered and consumed: the slab's space is free
      ptx::tc_fence_after();
      const uint32_t trow = tmem + ((uint32_t)(quarter * 32) << 16);
      uint8_t* stage = reinterpret_cast<uint8_t*>(slab) + quarter * 8192;  // two 4 KB blocks
      const int rows = c.OH - oh0 < ST_ROWS ? c.OH - oh0 : ST_ROWS;  // output rows of the tile
#pragma unroll 1
      for (int rr = 0; rr < rows; ++rr) {
        uint32_t v[32];
        __syncwarp();  // converged for the warp-wide TMEM load
        ptx::tmem_ld32(trow + (uint32_t)(rr * ST_COLS), v);
        ptx::tmem_ld_wait();
        uint8_t* blk = stage + (rr & 1) * 4096;
        if (lane == 0) ptx::bulk_wait_read1();  // the store from this block two rows ago
        __syncwarp();
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          float4 o = make_float4(__uint_as_float(v[4 * u]) + bias, __uint_as_float(v[4 * u + 1]) + bias,
                                 __uint_as_float(v[4 * u + 2]) + bias, __uint_as_float(v[4 * u + 3]) + bias);
          if (c.relu)
            o = make_float4(fmaxf(o.x, 0.f), fmaxf(o.y, 0.f), fmaxf(o.z, 0.f), fmaxf(o.w, 0.f));
          *reinterpret_cast<float4*>(blk + lane * 128 + ((u ^ (lane & 7)) << 4)) = o;
        }
        ptx::fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          ptx::tma_store_4d(&tmO, blk, ow0, oh0 + rr, quarter * 32, b);
          ptx::bulk_commit();
        }
      }
      if (lane == 0) ptx::bulk_wait_all();  // every store has landed before the CTA ends
    }
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (warp == MMA_WARP) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, TMEM_COLS);
  }
}

// Adds the K-slice partial tiles of the sliced tiles in slice order, then bias
// (and ReLU), and writes NCHW.  Thread = (tile, channel, 4 positions); the
// slice loads are unrolled (at most 16) so that they are all in flight.
constexpr int MAX_SLICES = 16;
__global__ void __launch_bounds__(256) k_conv_tail(const ConvArgs c, const Sched q, int tail) {
  ptx::griddep_wait();  // the partial tiles come from the main kernel
  const int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const int quad = (int)(idx & 31);
  const int64_t rest = idx >> 5;
  const int col = (int)(rest % q.bn), tt = (int)(rest / q.bn);
  if (tt >= tail) return;
  const int t = q.full + tt, pt = t / q.n_oc, ot = t - pt * q.n_oc;
  const int r0 = 4 * quad, oc = ot * q.bn + col;
  if (oc >= c.OC) return;
  int64_t obase = -1;  // slab form: out offset of (b, oc, oh, ow), -1 if off the image
  TilePos tp{0, BM};
  if (q.slab) {  // row r0 of the tile is output (oh0 + r0/32, ow0 + r0%32 ..+3), OW % 4 == 0
    const Tile2 t2 = tile2d(q, pt);
    const int oh = t2.oh0 + (r0 >> 5), ow = t2.ow0 + (r0 & 31);
    if (oh >= c.OH || ow >= c.OW) return;
    obase = (((int64_t)t2.b * c.OC + oc) * c.OH + oh) * c.OW + ow;
  } else {
    tp = tile_pos(c, q, pt);
    if (r0 >= tp.count) return;
  }
  const int64_t per = (int64_t)q.bn * BM;
  const float4* src =
      reinterpret_cast<const float4*>(q.part + ((int64_t)tt * q.slices * q.bn + col) * BM + r0);
  float4 acc = src[0];
#pragma unroll
  for (int sl = 1; sl < MAX_SLICES; ++sl) {
    if (sl < q.slices) {
      const float4 v = src[sl * per / 4];
      acc = make_float4(acc.x + v.x, acc.y + v.y, acc.z + v.z, acc.w + v.w);
    }
  }
  const float bv = c.bias ? __ldg(c.bias + oc) : 0.0f;
  float o[4] = {acc.x + bv, acc.y + bv, acc.z + bv, acc.w + bv};
  if (c.relu) {
#pragma unroll
    for (int k = 0; k < 4; ++k) o[k] = fmaxf(o[k], 0.0f);
  }
  if (obase >= 0) {
    *reinterpret_cast<float4*>(c.out + obase) = make_float4(o[0], o[1], o[2], o[3]);
    return;
  }
  const int64_t P = (int64_t)c.OH * c.OW, p = tp.p0 + r0, b = p / P;
  if (c.vec_out && r0 + 3 < tp.count) {  // P % 4 == 0: p .. p+3 are in one image
    *reinterpret_cast<float4*>(c.out + (b * c.OC + oc) * P + (p - b * P)) =
        make_float4(o[0], o[1], o[2], o[3]);
  } else {
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      if (r0 + k < tp.count) {
        const int64_t pk = p + k, bk = pk / P;
        c.out[(bk * c.OC + oc) * P + (pk - bk * P)] = o[k];
      }
    }
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

// Padded weight plane [OC, Kp] -> tensor map, box {16, bn}, 64-byte swizzle;
// rows past OC read as zero.
bool encode_w(CUtensorMap* m, const float* base, uint64_t Kp, uint64_t OC, int bn) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {Kp, OC};
  const cuuint64_t strides[1] = {Kp * 4};
  const cuuint32_t box[2] = {(cuuint32_t)BK, (cuuint32_t)bn};
  const cuuint32_t es[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float*>(base), dims, strides, box,
            es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int64_t padded_k(int64_t K) { return (K + 3) / 4 * 4; }

struct Plan {
  Sched q;
  int tail;         // tiles cut into K-slices
  size_t part_off;  // byte offset of the partial sums in the workspace
  size_t bytes;     // workspace bytes
  int smem;         // dynamic shared memory of the main kernel
};

// Input channel fastest in the kernel's K order (see the file comment).
bool ic_fastest(const ConvArgs& c) { return c.IC >= 8; }

// Shared memory of the main kernel besides the weight stages.
int fixed_smem(const Sched& q) {
  return 1024 + (q.slab ? 2 * q.slab_stride : 0) + q.tab_bytes + EPI_STAGE_BYTES +
         (int)sizeof(Ctl) + 4 * (int)sizeof(uint64_t);
}

// Slab form, for few input channels (the pages' K order): position tiles of
// SLAB_ROWS x SLAB_COLS outputs, each tile's input window brought into shared
// memory by one 4-D TMA box and the im2col values read from there.  Applies
// when the box fits the TMA limits (each extent <= 256, x and its rows
// 16-byte aligned: W % 4 == 0), both buffers fit beside four weight stages,
// the output takes 4-D TMA stores (OW % 4 == 0, aligned out), K is at most
// kSlabMaxK (the k offset table), and at least 3/4 of the tiles' positions are
// real outputs.
bool slab_geometry(const ConvArgs& c, Sched& q, int w_bytes) {
  if (ic_fastest(c) || c.W % 4 != 0 || c.OW % 4 != 0 || !c.vec_out ||
      reinterpret_cast<uintptr_t>(c.x) % 16 != 0 || (int64_t)q.kb * BK > kSlabMaxK)
    return false;
  const int64_t off = (4 - c.pW % 4) % 4;  // box column start a multiple of 4
  const int64_t bw =
      (off + (SLAB_COLS - 1) * (int64_t)c.sW + (int64_t)(c.KW - 1) * c.dW + 1 + 3) / 4 * 4;
  const int64_t rows = (SLAB_ROWS - 1) * (int64_t)c.sH + (int64_t)(c.KH - 1) * c.dH + 1;
  if (bw > 256 || rows > 256 || c.IC > 256) return false;
  const int64_t bytes = (int64_t)c.IC * rows * bw * 4;
  if (bytes > kSlabMaxBytes) return false;
  const int64_t tw = (c.OW + SLAB_COLS - 1) / SLAB_COLS, th = (c.OH + SLAB_ROWS - 1) / SLAB_ROWS;
  if (4 * (int64_t)c.OW * c.OH < 3 * tw * SLAB_COLS * th * SLAB_ROWS) return false;
  if ((int64_t)c.B * tw * th * q.n_oc >= (int64_t(1) << 30)) return false;  // tile indices fit an int
  Sched t = q;
  t.slab = 1;
  t.tw = (int)tw;
  t.tpi = (int)(tw * th);
  t.sbw = (int)bw;
  t.srows = (int)rows;
  t.soff = (int)off;
  t.slab_tx = (int)bytes;
  t.slab_stride = (int)((bytes + 1023) / 1024 * 1024);
  t.tab_bytes = (t.kb * BK * 4 + 1023) / 1024 * 1024;  // k offset table
  if (fixed_smem(t) + 4 * w_bytes > SMEM_LIMIT) return false;
  q = t;
  return true;
}

// Channel tiles of at most 256 (as even as possible, multiples of 16, or of
// 32 when there are several);
// 128-position tiles (SLAB_ROWS x SLAB_COLS in the slab form); K-slices for the tail tiles when they shorten the
// longest CTA's work and the partial sums fit in `limit` bytes of workspace.
// Cost in k-block times of one CTA: whole-tile waves, the sliced wave(s), the
// fix-up launch, and the partial sums' write + read at HBM speed (one k-block
// of MMAs takes (3 or 1) * 2 * 128 * BN * 8 / 2047 clocks at ~90 % of the
// measured TF32 rate, at least 400: below that the gather sets the pace).
Plan make_plan(const ConvArgs& c, bool three, size_t limit) {
  const int64_t OC = c.M, Npix = c.N, K = c.K, P = (int64_t)c.OH * c.OW;
  Plan pl{};
  Sched& q = pl.q;
  q.n_oc = (int)((OC + BN_MAX - 1) / BN_MAX);
  // The epilogue writes 32-channel blocks, and a TMA box is clipped only at
  // OC: with several channel tiles each is a multiple of 32 wide, so that no
  // block reaches into the next tile's channels (one tile: a multiple of 16).
  const int64_t per_tile = (OC + q.n_oc - 1) / q.n_oc;
  q.bn = (int)(q.n_oc > 1 ? (per_tile + 31) / 32 * 32 : (per_tile + 15) / 16 * 16);
  q.kb = (int)((K + BK - 1) / BK);
  int64_t ptiles;
  if (slab_geometry(c, q, (three ? 2 : 1) * q.bn * BK * 4)) {
    ptiles = (int64_t)c.B * q.tpi;
  } else {
    // per-image tiles when that adds at most 1/16 empty positions
    const int64_t tpi = (P + BM - 1) / BM;
    q.tpi = (P >= BM && (tpi * BM - P) * 16 <= P) ? (int)tpi : 0;
    ptiles = q.tpi > 0 ? (int64_t)c.B * q.tpi : (Npix + BM - 1) / BM;
  }
  const int64_t tiles = ptiles * q.n_oc;
  const size_t w_bytes = (three ? 2u : 1u) * (size_t)OC * (size_t)padded_k(K) * sizeof(float);
  pl.part_off = (w_bytes + 255) / 256 * 256;
  const int64_t waves = tiles / kPlanSMs, tail = tiles - waves * kPlanSMs;
  const double kb_clk =
      std::max(400.0, (three ? 6.0 : 2.0) * BM * q.bn * UK / (2047.0 * 0.9));
  const double gpu_bytes_per_kb = kHbmBytesPerClkSm * kb_clk * kPlanSMs;
  int best_s = 1;
  double best = (double)((waves + (tail > 0 ? 1 : 0)) * q.kb);
  for (int S = 2; S <= 16 && S <= q.kb / 4 && tail > 0; ++S) {
    const size_t part = (size_t)tail * S * q.bn * BM * sizeof(float);
    if (pl.part_off + part > limit) break;
    const double cost = (double)(waves * q.kb +
                                 (tail * S + kPlanSMs - 1) / kPlanSMs * ((q.kb + S - 1) / S)) +
                        kSliceLaunchKb + 2.0 * (double)part / gpu_bytes_per_kb;
    if (cost < best) {
      best = cost;
      best_s = S;
    }
  }
  q.slices = best_s;
  pl.tail = best_s > 1 ? (int)tail : 0;
  q.full = (int)(tiles - pl.tail);
  q.units = q.full + pl.tail * best_s;
  pl.bytes = best_s > 1 ? pl.part_off + (size_t)pl.tail * best_s * q.bn * BM * sizeof(float)
                        : w_bytes;
  q.nacc = q.bn <= 128 ? 2 : 1;
  return pl;
}

// Shared-memory layout: weight stages, the tap table, the epilogue's staging
// block, the barriers.  False when fewer than three stages fit.
bool layout(Plan& pl, const ConvArgs& c, bool three) {
  Sched& q = pl.q;
  q.w_bytes = (three ? 2 : 1) * q.bn * BK * 4;
  // tap table, or the k offset table of the slab form; a multiple of 1 KB
  // keeps the epilogue blocks 1 KB-aligned
  q.tab_bytes = q.slab ? (q.kb * BK * 4 + 1023) / 1024 * 1024
                       : (c.KH * c.KW * 8 + 1023) / 1024 * 1024;
  const int avail = SMEM_LIMIT - fixed_smem(q);
  q.stages = avail / q.w_bytes < MAX_STAGES ? avail / q.w_bytes : MAX_STAGES;
  pl.smem = fixed_smem(q) + q.stages * q.w_bytes;
  return q.stages >= 3;
}

// out viewed as [B][OC][OH*OW] -> tensor map, box {128 positions, 32
// channels, 1 image}; positions and channels past the end are not written.
// Needs OH*OW % 4 == 0 and a 16-byte aligned out.
bool encode_out(CUtensorMap* m, const ConvArgs& c) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t P = (cuuint64_t)c.OH * c.OW;
  const cuuint64_t dims[3] = {P, (cuuint64_t)c.OC, (cuuint64_t)c.B};
  const cuuint64_t strides[2] = {P * 4, P * c.OC * 4};
  const cuuint32_t box[3] = {(cuuint32_t)BM, 32, 1};
  const cuuint32_t es[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, c.out, dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
            CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Slab form: out viewed as [B][OC][OH][OW] -> tensor map, box {SLAB_COLS,
// SLAB_ROWS, 32 channels, 1 image}; the parts past OW, OH or OC are not
// written.  Needs OW % 4 == 0 and a 16-byte aligned out.
bool encode_out_2d(CUtensorMap* m, const ConvArgs& c) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t OW = (cuuint64_t)c.OW, OH = (cuuint64_t)c.OH, OC = (cuuint64_t)c.OC;
  const cuuint64_t dims[4] = {OW, OH, OC, (cuuint64_t)c.B};
  const cuuint64_t strides[3] = {OW * 4, OH * OW * 4, OC * OH * OW * 4};
  const cuuint32_t box[4] = {(cuuint32_t)SLAB_COLS, (cuuint32_t)SLAB_ROWS, 32, 1};
  const cuuint32_t es[4] = {1, 1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, c.out, dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
            CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Slab form: x viewed as [B][IC][H][W] -> tensor map, box {sbw, srows, IC,
// 1 image}, unswizzled ([IC][srows][sbw] in shared memory); outside the
// image reads as zero.  Needs W % 4 == 0 and a 16-byte aligned x.
bool encode_x_slab(CUtensorMap* m, const ConvArgs& c, const Sched& q) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t W = (cuuint64_t)c.W, H = (cuuint64_t)c.H, IC = (cuuint64_t)c.IC;
  const cuuint64_t dims[4] = {W, H, IC, (cuuint64_t)c.B};
  const cuuint64_t strides[3] = {W * 4, H * W * 4, IC * H * W * 4};
  const cuuint32_t box[4] = {(cuuint32_t)q.sbw, (cuuint32_t)q.srows, (cuuint32_t)c.IC, 1};
  const cuuint32_t es[4] = {1, 1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, const_cast<float*>(c.x), dims, strides, box,
            es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
            CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Transposed slab form (k_tc_conv_t): few input channels (the pages' K
// order), OC <= 128, the output in tiles of ST_ROWS x ST_COLS, between 3/4 of
// a tile and one tile per SM over the whole batch, W % 4 == 0 and a 16-byte aligned
// x (the input box), OW % 4 == 0 and an aligned out (16-byte stores), K at
// most kSlabMaxK (the k offset table), at least 3/4 of the tiles' positions
// real outputs, and at least two stages beside the slab.
bool st_geometry(const ConvArgs& c, bool three, Sched& q, int& smem) {
  if (ic_fastest(c) || c.OC > BM || c.W % 4 != 0 || c.OW % 4 != 0 || !c.vec_out ||
      reinterpret_cast<uintptr_t>(c.x) % 16 != 0)
    return false;
  const int64_t kb = (c.K + BK - 1) / BK;
  if (kb * BK > kSlabMaxK) return false;
  const int64_t off = (4 - c.pW % 4) % 4;
  const int64_t bw =
      (off + (ST_COLS - 1) * (int64_t)c.sW + (int64_t)(c.KW - 1) * c.dW + 1 + 3) / 4 * 4;
  const int64_t rows = (ST_ROWS - 1) * (int64_t)c.sH + (int64_t)(c.KH - 1) * c.dH + 1;
  if (bw > 256 || rows > 256 || c.IC > 256) return false;
  const int64_t bytes = (int64_t)c.IC * rows * bw * 4;
  if (bytes > kStSlabMaxBytes) return false;
  const int64_t tw = (c.OW + ST_COLS - 1) / ST_COLS, th = (c.OH + ST_ROWS - 1) / ST_ROWS;
  const int64_t slab_space = std::max<int64_t>((bytes + 1023) / 1024 * 1024, kStEpiBytes);
  // one tile per SM, and enough tiles to fill 3/4 of them: with fewer, the
  // 128-position form cuts K across the idle SMs and measured faster (64
  // tiles of K = 147: 12.5 against 14.5 us; 24 tiles of K = 343: 16.5 against
  // 20.6 us)
  if ((int64_t)c.B * tw * th > kPlanSMs || 4 * (int64_t)c.B * tw * th < 3 * kPlanSMs) return false;
  if (4 * (int64_t)c.OW * c.OH < 3 * tw * ST_COLS * th * ST_ROWS) return false;
  Sched t{};
  t.kb = (int)kb;
  t.slab = 1;
  t.tw = (int)tw;
  t.tpi = (int)(tw * th);
  t.units = (int)(c.B * tw * th);
  t.sbw = (int)bw;
  t.srows = (int)rows;
  t.soff = (int)off;
  t.slab_tx = (int)bytes;
  t.slab_stride = (int)slab_space;  // the slab, then the epilogue's staging blocks
  t.tab_bytes = (int)((kb * BK * 4 + 1023) / 1024 * 1024);
  t.w_bytes = (three ? 2 : 1) * (ST_W_TILE + ST_B_TILE);
  const int fixed = 1024 + t.slab_stride + t.tab_bytes + (int)sizeof(Ctl) + (int)sizeof(uint64_t);
  const int st = (SMEM_LIMIT - fixed) / t.w_bytes;
  t.stages = st < MAX_STAGES ? st : MAX_STAGES;
  if (t.stages < 2) return false;
  t.bn = BM;
  t.n_oc = 1;
  t.nacc = 1;
  q = t;
  smem = fixed + t.stages * t.w_bytes;
  return true;
}

constexpr int kMaxDev = 64;

// Transposed slab form: out viewed as [B][OC][OH][OW] -> tensor map, box {32
// columns, 1 row, 32 channels, 1 image}, 128-byte swizzle (a staged block is
// 32 channel rows of 128 bytes); the parts past OW, OH or OC are not written.
bool encode_out_t(CUtensorMap* m, const ConvArgs& c) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t OW = (cuuint64_t)c.OW, OH = (cuuint64_t)c.OH, OC = (cuuint64_t)c.OC;
  const cuuint64_t dims[4] = {OW, OH, OC, (cuuint64_t)c.B};
  const cuuint64_t strides[3] = {OW * 4, OH * OW * 4, OC * OH * OW * 4};
  const cuuint32_t box[4] = {(cuuint32_t)ST_COLS, 1, 32, 1};
  const cuuint32_t es[4] = {1, 1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, c.out, dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <bool THREE>
cudaError_t run_t(const ConvArgs& c, const Sched& q, int smem, const float* w_hi,
                  const float* w_lo, int64_t Kp, cudaStream_t s) {
  CUtensorMap th, tl, tx, to;
  if (!encode_w(&th, w_hi, (uint64_t)Kp, (uint64_t)c.OC, BM) ||
      !encode_w(&tl, THREE ? w_lo : w_hi, (uint64_t)Kp, (uint64_t)c.OC, BM) ||
      !encode_x_slab(&tx, c, q) || !encode_out_t(&to, c))
    return cudaErrorInvalidValue;
  static std::atomic<bool> ready[kMaxDev];  // per device: the attribute is set (calls may race)
  auto k = k_tc_conv_t<THREE>;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev >= kMaxDev || !ready[dev].load(std::memory_order_acquire)) {
    e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_LIMIT);
    if (e != cudaSuccess) return e;
    if (dev < kMaxDev) ready[dev].store(true, std::memory_order_release);
  }
  e = launch_after_previous(k, dim3(q.units), dim3(ST_THREADS), (size_t)smem, s, th, tl, tx, to, c, q);
  note_launch();
  note_kernel_name(THREE ? "k_tc_conv<3xtf32,slab_t>" : "k_tc_conv<1xtf32,slab_t>");
  return e;
}

template <bool THREE, int GM>
cudaError_t launch_main(const ConvArgs& c, const Plan& pl, const CUtensorMap& th,
                        const CUtensorMap& tl, const CUtensorMap& to, const CUtensorMap& tx,
                        int grid, cudaStream_t s) {
  static std::atomic<bool> ready[kMaxDev];  // per device: the attribute is set (calls may race)
  auto k = k_tc_conv<THREE, GM>;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev >= kMaxDev || !ready[dev].load(std::memory_order_acquire)) {
    e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_LIMIT);
    if (e != cudaSuccess) return e;
    if (dev < kMaxDev) ready[dev].store(true, std::memory_order_release);
  }
  return launch_after_previous(k, dim3(grid), dim3(threads_of(GM)), (size_t)pl.smem, s, th, tl, to, tx,
                               c, pl.q);
}

template <bool THREE>
cudaError_t run(const ConvArgs& c, Plan pl, const float* w_hi, const float* w_lo, int64_t Kp,
                float* part, cudaStream_t s) {
  CUtensorMap th, tl;
  if (!encode_w(&th, w_hi, (uint64_t)Kp, (uint64_t)c.OC, pl.q.bn) ||
      !encode_w(&tl, THREE ? w_lo : w_hi, (uint64_t)Kp, (uint64_t)c.OC, pl.q.bn))
    return cudaErrorInvalidValue;
  if (!layout(pl, c, THREE)) return cudaErrorInvalidValue;
  CUtensorMap to, tx = th;  // tx: read in the slab form only
  if (pl.q.slab) {
    if (!encode_out_2d(&to, c) || !encode_x_slab(&tx, c, pl.q)) return cudaErrorInvalidValue;
    pl.q.tma_out = 1;
  } else {
    pl.q.tma_out = c.vec_out && encode_out(&to, c) ? 1 : 0;  // vec_out: P % 4 == 0, aligned out
    if (!pl.q.tma_out) to = th;                                // not read
  }
  pl.q.part = part;
  const int sms = device_sm_count();
  const int grid = pl.q.units < sms ? pl.q.units : sms;
  cudaError_t e;
  if (pl.q.slab)
    e = launch_main<THREE, GM_SLAB>(c, pl, th, tl, to, tx, grid, s);
  else if (ic_fastest(c))
    e = launch_main<THREE, GM_ICF>(c, pl, th, tl, to, tx, grid, s);
  else
    e = launch_main<THREE, GM_PAGES>(c, pl, th, tl, to, tx, grid, s);
  note_launch();
  note_kernel_name(pl.q.slab ? (THREE ? "k_tc_conv<3xtf32,slab>" : "k_tc_conv<1xtf32,slab>")
                             : (THREE ? "k_tc_conv<3xtf32>" : "k_tc_conv<1xtf32>"));
  if (e != cudaSuccess || pl.tail == 0) return e;
  const int64_t threads = (int64_t)pl.tail * pl.q.bn * 32;
  e = launch_after_previous(k_conv_tail, dim3((unsigned)((threads + 255) / 256)), dim3(256), 0,
                            s, c, pl.q, pl.tail);
  note_launch();
  return e;
}

}  // namespace

bool tc_conv_shape_ok(const ConvArgs& c) {
  const int64_t lim30 = int64_t(1) << 30, lim31 = (int64_t(1) << 31) - 1;
  if ((int64_t)c.KH * c.KW > MAX_TAPS || c.K > lim31 - 8) return false;  // Kp fits an int
  if ((int64_t)(c.KH - 1) * c.dH >= lim30 || (int64_t)(c.KW - 1) * c.dW >= lim30) return false;
  if ((int64_t)c.H + 2 * (int64_t)c.pH >= lim30 || (int64_t)c.W + 2 * (int64_t)c.pW >= lim30)
    return false;
  // the running input-channel offset may pass IC by up to 33 planes (one
  // k-block and the skipped one after the last)
  if (((int64_t)c.IC + 33) * c.H * c.W > lim31) return false;
  // position tiles are at most one per 128 positions plus one per image
  const int64_t tiles = ((c.N + BM - 1) / BM + c.B) * ((c.M + BN_MAX - 1) / BN_MAX);
  return tiles < lim31;
}

bool tc_conv_supported(const ConvArgs& c) { return tc_conv_shape_ok(c) && encode_fn() != nullptr; }

size_t tc_conv_workspace_bytes(const ConvArgs& c, bool three_pass, size_t limit) {
  return make_plan(c, three_pass, limit).bytes;
}

cudaError_t launch_tc_conv(const ConvArgs& c, bool three_pass, void* workspace,
                           size_t workspace_bytes, cudaStream_t s) {
  if (!tc_conv_supported(c) || !workspace) return cudaErrorNotSupported;
  const Plan pl = make_plan(c, three_pass, workspace_bytes);
  if (pl.bytes > workspace_bytes) return cudaErrorInvalidValue;
  const int64_t Kp = padded_k(c.K);
  float* w_hi = static_cast<float*>(workspace);
  float* w_lo = three_pass ? w_hi + c.OC * Kp : nullptr;
  float* part = reinterpret_cast<float*>(static_cast<char*>(workspace) + pl.part_off);
  // at most two pre-pass blocks per SM (see k_prep_w)
  const int gx = (int)((Kp + 255) / 256 < 64 ? (Kp + 255) / 256 : 64);
  const int gy_cap = 2 * device_sm_count() / gx > 1 ? 2 * device_sm_count() / gx : 1;
  const int gy = std::max(1, (int)((c.OC + 3) / 4 < gy_cap ? (c.OC + 3) / 4 : gy_cap));
  cudaError_t e = launch_after_previous(k_prep_w, dim3(gx, gy), dim3(256), 0, s, c.w, c.OC,
                                        (int)c.K, (int)Kp, c.IC, c.KH * c.KW,
                                        ic_fastest(c) ? 1 : 0, w_hi, w_lo);
  note_launch();
  if (e != cudaSuccess) return e;
  Sched qt;
  int smem_t = 0;
  if (st_geometry(c, three_pass, qt, smem_t))
    return three_pass ? run_t<true>(c, qt, smem_t, w_hi, w_lo, Kp, s)
                      : run_t<false>(c, qt, smem_t, w_hi, nullptr, Kp, s);
  return three_pass ? run<true>(c, pl, w_hi, w_lo, Kp, part, s)
                    : run<false>(c, pl, w_hi, nullptr, Kp, part, s);
}

cudaError_t conv_take_watchdog(int* value) {
  cudaError_t e = cudaMemcpyFromSymbol(value, g_watchdog_conv, sizeof(int));
  if (e != cudaSuccess) return e;
  const int zero = 0;
  return cudaMemcpyToSymbol(g_watchdog_conv, &zero, sizeof(int));
}

}  // namespace imc
