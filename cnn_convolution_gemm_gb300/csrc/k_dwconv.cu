// Depthwise 3x3 convolution (groups == C == K), NHWC bf16, fp32 accumulate,
// fused bias / residual / ReLU / ReLU6.
//
// The Momenta talk ("優化2：Depthwise卷積") splits a 3x3 conv into a per-channel
// spatial filter and a 1x1 channel mix; the spatial part does only 9
// multiply-adds per loaded value, so it is bound by memory bandwidth.  The
// kernel is built so HBM streams at full rate with few threads:
//   * persistent CTAs walk a list of blocks (image, channel slice of up to 256
//     channels — all of C for the usual widths, so a block reads whole
//     contiguous pixel runs —, block of RB output rows, block of output
//     columns sized to fill a buffer); for each, one 4-D TMA load per input
//     row brings the columns the block needs (its halo included) into that
//     row's slot in shared memory (a fixed pitch, so shared loads take
//     constant offsets), and out-of-bounds elements arrive as zeros, which is
//     the padding;
//   * two CTAs per SM, each with a ring of two shared-memory buffers: the
//     loads of a CTA's next block are in flight while it computes the current
//     one, so bytes in flight do not depend on registers, and the two CTAs'
//     warps hide each other's latencies;
//   * a thread owns 4 channels of two adjacent output columns and walks down
//     the block's input rows: each row's values (4 or 5 columns, one 8-byte
//     shared load each) are added into the accumulators of the up to three
//     output rows they reach; a finished output row gets bias / residual /
//     activation and is stored as bf16;
//   * the multiply-adds take the bf16 input and weight straight from their
//     packed 32-bit words (fma.rn.f32.bf16: bf16 x bf16 + fp32 -> fp32, the
//     product exact, one rounding), so no instruction widens the operands and
//     the result equals the fp32 FMA of the widened values;
//   * a warp releases a buffer through an mbarrier when it is done with it,
//     and the loading thread refills it once every warp has, so warps are not
//     held to a common pace by block-wide barriers;
//   * weights are prepacked tap-major ([9][C] bf16): one 8-byte load per tap
//     gives a thread its 4 channels.
#include <cuda_bf16.h>

#include <algorithm>

#include "internal.h"
#include "ptx.cuh"

namespace {

// Two CTAs of up to 256 threads share an SM (registers: 2 x 256 x 128), each
// with a ring of two shared-memory buffers: while a CTA computes one block, the
// loads of its next block are in flight, and the other CTA's warps cover the
// latencies of this one's.
constexpr int MAX_THREADS = 256;
constexpr int CTAS_PER_SM = 2;
constexpr int NBUF = 2;              // shared-memory ring depth per CTA
constexpr int BUF_MAX = 54 * 1024;   // bytes per buffer (2 CTAs x 2 x 54 KB fit 228 KB)

template <int ST>
struct DwCfg {
  static constexpr int RB = ST == 1 ? 8 : 4;      // output rows per block
  static constexpr int IH = (RB - 1) * ST + 3;    // input rows per block
  // input row r of a block sits at r * ROWP in its buffer: a compile-time,
  // 128-byte aligned pitch, so every shared-memory load has a constant offset
  static constexpr int ROWP = BUF_MAX / IH / 128 * 128;
  static constexpr int SMEM = NBUF * BUF_MAX + 1024 + 2 * NBUF * 8;
};

struct DwParams {
  int N, C, H, W, OH, OW, pad;
  int shuf_g;              // input channel shuffle groups (SHUF kernels)
  int cb;                  // channels per block (all of C when C <= 256)
  int owt, iw, buf_bytes;  // output columns per block, input columns, bytes per block
  int cslices, rblocks, cblocks;
  long long nblocks;
  int* err;
  unsigned long long wait_ns;
};

// work items of one block: (4-channel group, pair of output columns)
__host__ __device__ inline int gb_items(const DwParams& p) { return ((p.owt + 1) / 2) * (p.cb / 4); }

// Two fp32 values in one 64-bit register pair: channels (c, c + 1) of an
// output on their way to one bf16x2 word.
typedef unsigned long long f32x2;

__device__ __forceinline__ f32x2 f2_pack(float lo, float hi) {
  f32x2 r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void f2_unpack(f32x2 v, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
// an fp32 pair -> one bf16x2 word (round to nearest even), negative results set
// to zero when RELU; the activation commutes with the monotone rounding
template <bool RELU>
__device__ __forceinline__ uint32_t f2_to_bf16x2(f32x2 v) {
  float lo, hi;
  f2_unpack(v, lo, hi);
  uint32_t r;
  if (RELU)
    asm("cvt.rn.relu.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  else
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}
__device__ __forceinline__ uint32_t min6_bf16x2(uint32_t v) {
  const __nv_bfloat162 six = __float2bfloat162_rn(6.f);
  __nv_bfloat162 h = __hmin2(*reinterpret_cast<__nv_bfloat162*>(&v), six);
  return *reinterpret_cast<uint32_t*>(&h);
}
__device__ __forceinline__ uint2 lds64(uint32_t addr) {
  uint2 v;
  asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(addr));
  return v;
}

// a * b + c for bf16 a, b (bit patterns) and fp32 c: the product of two bf16
// values is exact in fp32, so this is the fp32 FMA of the widened operands
__device__ __forceinline__ float fma_bf16(unsigned short a, unsigned short b, float c) {
  float d;
  asm("fma.rn.f32.bf16 %0, %1, %2, %3;" : "=f"(d) : "h"(a), "h"(b), "f"(c));
  return d;
}
// the two bf16 halves of a packed word (lo: the element at the lower address)
__device__ __forceinline__ void halves(uint32_t u, unsigned short& lo, unsigned short& hi) {
  asm("mov.b32 {%0, %1}, %2;" : "=h"(lo), "=h"(hi) : "r"(u));
}

// bias / residual / activation of 4 channels, rounding to bf16, one 8-byte store
template <int ACT, bool RES>
__device__ __forceinline__ void store4(f32x2 a0, f32x2 a1, __nv_bfloat16* yp,
                                       const __nv_bfloat16* rp) {
  if (RES) {
    const uint2 rv = __ldg(reinterpret_cast<const uint2*>(rp));
    float v0, v1, v2, v3;
    f2_unpack(a0, v0, v1);
    f2_unpack(a1, v2, v3);
    a0 = f2_pack(v0 + __uint_as_float(rv.x << 16), v1 + __uint_as_float(rv.x & 0xffff0000u));
    a1 = f2_pack(v2 + __uint_as_float(rv.y << 16), v3 + __uint_as_float(rv.y & 0xffff0000u));
  }
  uint2 ov;
  ov.x = f2_to_bf16x2<(ACT >= 1)>(a0);
  ov.y = f2_to_bf16x2<(ACT >= 1)>(a1);
  if (ACT == 2) {
    ov.x = min6_bf16x2(ov.x);
    ov.y = min6_bf16x2(ov.y);
  }
  *reinterpret_cast<uint2*>(yp) = ov;
}

// One work item of one block: 4 channels x 2 output columns x RB output rows.
// Input row rho feeds output row (rho - i) / ST through filter row i; each input
// value is loaded once and added into the accumulators of the (up to three)
// output rows it reaches.  Output row o lives in slot o % 3 and is stored once
// its last input row, o * ST + 2, has been added.  FULL: all RB rows and both
// columns exist (no per-row tests).  SHUF: the 4 input channels are gathered
// one by one at byte offsets choff[] within the pixel (channel shuffle).
template <int ST, int ACT, bool RES, bool FULL, bool SHUF = false>
__device__ __forceinline__ void dw_item(uint32_t src, uint32_t col_b,
                                        const unsigned short (&wh)[9][4], const float (&bz)[4],
                                        __nv_bfloat16* y0, const __nv_bfloat16* r0, size_t y_row,
                                        int C, int nrows, bool two, const uint32_t (&choff)[4]) {
  using Cf = DwCfg<ST>;
  constexpr int NC = ST + 3;  // distinct input columns the two outputs read
  uint32_t sc[NC];            // shared address of input column cc of the pair, row 0
#pragma unroll
  for (int cc = 0; cc < NC; ++cc) sc[cc] = src + cc * col_b;
  __nv_bfloat16* y1 = y0 + C;
  const __nv_bfloat16* r1 = RES ? r0 + C : nullptr;
  float acc[3][2][4];  // [slot][output column][channel]
#pragma unroll
  for (int rho = 0; rho < Cf::IH; ++rho) {
    unsigned short xh[NC][4];  // bf16 inputs of this row: [column][channel]
#pragma unroll
    for (int cc = 0; cc < NC; ++cc) {
      if constexpr (SHUF) {
#pragma unroll
        for (int q = 0; q < 4; ++q)
          asm volatile("ld.shared.u16 %0, [%1];"
                       : "=h"(xh[cc][q])
                       : "r"(sc[cc] + rho * Cf::ROWP + choff[q]));
      } else {
        const uint2 v = lds64(sc[cc] + rho * Cf::ROWP);
        halves(v.x, xh[cc][0], xh[cc][1]);
        halves(v.y, xh[cc][2], xh[cc][3]);
      }
    }
#pragma unroll
    for (int i = 0; i < 3; ++i) {
      if (rho < i || (rho - i) % ST != 0 || (rho - i) / ST >= Cf::RB) continue;
      float(&a)[2][4] = acc[((rho - i) / ST) % 3];
#pragma unroll
      for (int s = 0; s < 3; ++s)
#pragma unroll
        for (int o = 0; o < 2; ++o)
#pragma unroll
          for (int q = 0; q < 4; ++q)
            a[o][q] = fma_bf16(xh[o * ST + s][q], wh[i * 3 + s][q],
                               (i == 0 && s == 0) ? bz[q] : a[o][q]);
    }
    if (rho < 2 || (rho - 2) % ST != 0 || (rho - 2) / ST >= Cf::RB) continue;
    const int orow = (rho - 2) / ST;
    const float(&a)[2][4] = acc[orow % 3];
    if (FULL || orow < nrows) {
      store4<ACT, RES>(f2_pack(a[0][0], a[0][1]), f2_pack(a[0][2], a[0][3]), y0, r0);
      if (FULL || two)
        store4<ACT, RES>(f2_pack(a[1][0], a[1][1]), f2_pack(a[1][2], a[1][3]), y1, r1);
    }
    y0 += y_row;
    y1 += y_row;
    if (RES) {
      r0 += y_row;
      r1 += y_row;
    }
  }
}

// Persistent CTAs walk the block list; see the file comment.
template <int ST, int ACT, bool RES, bool SHUF = false>
__global__ void __launch_bounds__(MAX_THREADS, CTAS_PER_SM)
    dwconv3x3_tma_kernel(const __grid_constant__ CUtensorMap tm_x, const DwParams p,
                         const __nv_bfloat16* __restrict__ w9c, const float* __restrict__ bias,
                         const __nv_bfloat16* __restrict__ res, __nv_bfloat16* __restrict__ y) {
  using Cf = DwCfg<ST>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + NBUF * BUF_MAX);  // tile landed
  uint64_t* empty = full + NBUF;  // every warp is done reading the tile
  const int nwarps = blockDim.x / 32;

  if (threadIdx.x == 0) {
    for (int i = 0; i < NBUF; ++i) {
      gb::mbar_init(&full[i], 1);
      gb::mbar_init(&empty[i], nwarps);
    }
    gb::fence_barrier_init();
    gb::tma_prefetch_desc(&tm_x);
  }
  __syncthreads();

  // A block index is a mixed-radix number (image n, channel slice cs, row block
  // rb, column block cb; cb fastest).  The CTA's blocks are first, first + step,
  // ..., so both cursors below (the block being computed and the one thread 0
  // loads next) advance by adding the digits of step with carries: no division
  // inside the loop.
  struct Cursor {
    int n, cs, rb, cb;
  };
  auto digits = [&](long long b) {
    Cursor c;
    c.cb = (int)(b % p.cblocks);
    b /= p.cblocks;
    c.rb = (int)(b % p.rblocks);
    b /= p.rblocks;
    c.cs = (int)(b % p.cslices);
    c.n = (int)(b / p.cslices);
    return c;
  };
  const Cursor sd = digits(gridDim.x);
  auto advance = [&](Cursor& c) {
    // each digit + step digit + carry < 2 * radix: one subtraction suffices
    c.cb += sd.cb;
    int k = c.cb >= p.cblocks;
    c.cb -= k ? p.cblocks : 0;
    c.rb += sd.rb + k;
    k = c.rb >= p.rblocks;
    c.rb -= k ? p.rblocks : 0;
    c.cs += sd.cs + k;
    k = c.cs >= p.cslices;
    c.cs -= k ? p.cslices : 0;
    c.n += sd.n + k;
  };
  // one TMA load per input row (a box one row high) into its slot at r * ROWP;
  // rows and columns outside the image arrive as zeros, which is the padding
  auto issue = [&](const Cursor& c, int buf) {
    gb::fence_proxy_async_smem();
    gb::mbar_arrive_expect_tx(&full[buf], p.buf_bytes);
    const uint32_t dst = gb::smem_u32(smem + buf * BUF_MAX);
    const int c0 = c.cs * p.cb, w0 = c.cb * p.owt * ST - p.pad, h0 = c.rb * Cf::RB * ST - p.pad;
#pragma unroll 1
    for (int r = 0; r < Cf::IH; ++r)
      asm volatile(
          "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
          " [%0], [%1, {%2, %3, %4, %5}], [%6];" ::"r"(dst + r * Cf::ROWP),
          "l"(reinterpret_cast<uint64_t>(&tm_x)), "r"(c0), "r"(w0), "r"(h0 + r), "r"(c.n),
          "r"(gb::smem_u32(&full[buf]))
          : "memory");
  };

  // The CTA's k-th block (k = 0, 1, ...) is block first + k * step and lives in
  // buffer k % NBUF.  Thread 0 keeps NBUF - 1 loads ahead of its own warp; it
  // refills a buffer once all warps have released it, so the other warps never
  // wait on one another.
  const long long first = blockIdx.x, step = gridDim.x;
  const int nmine = p.nblocks > first ? (int)((p.nblocks - first + step - 1) / step) : 0;
  Cursor cur = digits(first), ld = cur;
  int issued = 0;  // blocks thread 0 has issued
  if (threadIdx.x == 0)
    for (; issued < NBUF - 1 && issued < nmine; ++issued) {
      issue(ld, issued);
      advance(ld);
    }
  // this thread's work items: (4-channel group g, pair jp of output columns
  // 2jp, 2jp + 1), item = jp * groups + g, items threadIdx.x + r * blockDim.x
  const int groups = p.cb / 4;
  const int npairs = (p.owt + 1) / 2;
  const int g_first = threadIdx.x % groups, jp_first = threadIdx.x / groups;
  const int g_step = blockDim.x % groups, jp_step = blockDim.x / groups;
  unsigned short wf[9][4];  // this thread's bf16 weights [tap][channel] (kept while its
  float bz[4];              // channels are unchanged) and fp32 bias
  int w_c = -1;
  const uint32_t col_b = (uint32_t)p.cb * 2;  // bytes between input columns in a row slot
  const size_t y_row = (size_t)p.OW * p.C;    // elements between output rows
  int it = 0;
  for (; it < nmine; ++it, advance(cur)) {
    const int buf = it % NBUF;
    bool ok = true;
    if (threadIdx.x == 0 && issued < nmine) {
      // refill: block `issued` goes where block issued - NBUF was
      if (issued >= NBUF)
        ok = gb::mbar_wait_bounded(&empty[issued % NBUF], (uint32_t)((issued / NBUF - 1) & 1),
                                   p.wait_ns, p.err);
      if (ok) {
        issue(ld, issued % NBUF);
        advance(ld);
        ++issued;
      }
    }
    if (ok) ok = gb::mbar_wait_bounded(&full[buf], (uint32_t)((it / NBUF) & 1), p.wait_ns, p.err);
    if (!__all_sync(0xffffffffu, ok)) break;  // a wait ran out: leave (the drain is below)

    const uint32_t tile = gb::smem_u32(smem + buf * BUF_MAX);
    const int nrows = min(Cf::RB, p.OH - cur.rb * Cf::RB);  // output rows of this block
    for (int g = g_first, jp = jp_first; jp < npairs;) {
      const int j0 = 2 * jp;
      const int c = cur.cs * p.cb + g * 4;
      const int ow0 = cur.cb * p.owt + j0;
      if (c < p.C && ow0 < p.OW) {
        const bool two = j0 + 1 < p.owt && ow0 + 1 < p.OW;
        if (c != w_c) {  // weights and bias of these 4 channels, in fp32
#pragma unroll
          for (int k = 0; k < 9; ++k) {
            const uint2 v = __ldg(reinterpret_cast<const uint2*>(w9c + (size_t)k * p.C + c));
            halves(v.x, wf[k][0], wf[k][1]);
            halves(v.y, wf[k][2], wf[k][3]);
          }
          if (bias) {  // scalar loads: the caller's bias need not be 16-byte aligned
            for (int q = 0; q < 4; ++q) bz[q] = __ldg(bias + c + q);
          } else {
            for (int q = 0; q < 4; ++q) bz[q] = 0.f;
          }
          w_c = c;
        }
        // tile-local input columns of the pair: j0*ST + s (first), (j0+1)*ST + s (second)
        uint32_t choff[4] = {0, 0, 0, 0};
        uint32_t src = tile + (uint32_t)(j0 * ST) * col_b;
        if constexpr (SHUF) {
          // output channel j reads channel (j mod G) * (C / G) + j div G of the
          // input (the whole channel range is in the tile: one slice)
#pragma unroll
          for (int q = 0; q < 4; ++q)
            choff[q] = (uint32_t)(((c + q) % p.shuf_g) * (p.C / p.shuf_g) + (c + q) / p.shuf_g) * 2;
        } else {
          src += (uint32_t)g * 8;
        }
        const size_t yoff = (((size_t)cur.n * p.OH + cur.rb * Cf::RB) * p.OW + ow0) * p.C + c;
        const __nv_bfloat16* r0 = RES ? res + yoff : nullptr;
        if (nrows == Cf::RB && two)
          dw_item<ST, ACT, RES, true, SHUF>(src, col_b, wf, bz, y + yoff, r0, y_row, p.C, nrows,
                                            two, choff);
        else
          dw_item<ST, ACT, RES, false, SHUF>(src, col_b, wf, bz, y + yoff, r0, y_row, p.C, nrows,
                                             two, choff);
      }
      g += g_step;  // next item: + blockDim.x
      jp += jp_step;
      if (g >= groups) {
        g -= groups;
        ++jp;
      }
    }
    __syncwarp();
    if ((threadIdx.x & 31) == 0) gb::mbar_arrive(&empty[buf]);
  }
  // Every load thread 0 issued must land before the CTA's shared memory goes
  // away.  On normal exit all of them were consumed (it == issued); after a
  // timeout the ones still in flight are waited for here (bounded).
  if (threadIdx.x == 0)
    for (int k = it; k < issued; ++k)
      gb::mbar_wait_bounded(&full[k % NBUF], (uint32_t)((k / NBUF) & 1), p.wait_ns, p.err);
}

// [C][3][3] -> [9][C]
__global__ void pack_dw_weights_kernel(const __nv_bfloat16* __restrict__ w,
                                       __nv_bfloat16* __restrict__ wp, int C) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= 9 * C) return;
  const int k = i / C, c = i % C;
  wp[i] = w[c * 9 + k];
}

template <int ST, int ACT>
auto pick_kernel(bool res, bool shuf) {
  // (a shuffled input with a residual is not a combination networks use: the
  // shuffle variants are built without the residual)
  return shuf ? dwconv3x3_tma_kernel<ST, ACT, false, true>
              : (res ? dwconv3x3_tma_kernel<ST, ACT, true> : dwconv3x3_tma_kernel<ST, ACT, false>);
}

template <int ST>
cudaError_t launch_st(const gbconv_desc_s& d, const void* x, const void* w, const float* bias,
                      const void* res, void* y, int* err, unsigned long long wait_ns,
                      cudaStream_t st) {
  using Cf = DwCfg<ST>;
  DwParams p{};
  p.N = d.N;
  p.C = d.C;
  p.H = d.H;
  p.W = d.W;
  p.OH = d.OH;
  p.OW = d.OW;
  p.pad = d.pad;
  // channel slices of <= 256 channels (the TMA box limit), as few as possible,
  // so each block reads whole contiguous pixel rows
  p.cslices = gb_ceil_div(d.C, 256);
  p.cb = gb_ceil_div(gb_ceil_div(d.C, p.cslices), 8) * 8;
  // widest column block whose input row fits one row slot
  const int px_bytes = p.cb * 2;
  int iw_max = Cf::ROWP / px_bytes;
  int owt = (iw_max - 3) / ST + 1;
  if (owt > d.OW) owt = d.OW;
  if (owt > 256 / ST - 2) owt = 256 / ST - 2;  // TMA box dimension <= 256
  if (owt < 1) return cudaErrorInvalidConfiguration;
  owt = gb_ceil_div(d.OW, gb_ceil_div(d.OW, owt));  // equal-width column blocks
  p.owt = owt;
  p.iw = (p.owt - 1) * ST + 3;
  p.buf_bytes = Cf::IH * p.iw * px_bytes;  // transaction bytes of one block's IH row loads
  p.rblocks = gb_ceil_div(d.OH, Cf::RB);
  p.cblocks = gb_ceil_div(d.OW, p.owt);
  p.nblocks = (long long)d.N * p.cslices * p.rblocks * p.cblocks;
  if (p.nblocks >= (1LL << 31)) return cudaErrorInvalidValue;  // block counters are 32-bit
  p.err = err;
  p.wait_ns = wait_ns;
  CUtensorMap tm;
  cuuint64_t dims[4] = {(cuuint64_t)d.C, (cuuint64_t)d.W, (cuuint64_t)d.H, (cuuint64_t)d.N};
  cuuint64_t strides[3] = {(cuuint64_t)d.C * 2, (cuuint64_t)d.W * d.C * 2,
                           (cuuint64_t)d.H * d.W * d.C * 2};
  cuuint32_t box[4] = {(cuuint32_t)p.cb, (cuuint32_t)p.iw, 1, 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  if (gb_encode_tiled(&tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(x), dims,
                      strides, box, estr, CU_TENSOR_MAP_SWIZZLE_NONE) != CUDA_SUCCESS)
    return cudaErrorInvalidValue;
  const long long grid = std::min<long long>(p.nblocks, (long long)CTAS_PER_SM * gb_num_sms());
  // threads: the block's work items split into equal rounds of <= MAX_THREADS
  const int items = gb_items(p);
  const int rounds = gb_ceil_div(items, MAX_THREADS);
  const int threads = gb_ceil_div(gb_ceil_div(items, rounds), 32) * 32;
  const bool has_res = res != nullptr;
  const bool shuf = d.shuffle_groups > 1;
  if (shuf && (has_res || p.cslices != 1)) return cudaErrorInvalidValue;
  p.shuf_g = shuf ? d.shuffle_groups : 1;
  auto kern = d.act == CONV_ACT_RELU6  ? pick_kernel<ST, 2>(has_res, shuf)
              : d.act == CONV_ACT_RELU ? pick_kernel<ST, 1>(has_res, shuf)
                                       : pick_kernel<ST, 0>(has_res, shuf);
  cudaError_t e = gb_set_smem_once(reinterpret_cast<const void*>(kern), Cf::SMEM);
  if (e != cudaSuccess) return e;
  kern<<<(unsigned)grid, threads, Cf::SMEM, st>>>(
      tm, p, static_cast<const __nv_bfloat16*>(w), bias, static_cast<const __nv_bfloat16*>(res),
      static_cast<__nv_bfloat16*>(y));
  gb_count_launch();
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_pack_dw_weights(const gbconv_desc_s& d, const void* w, void* wpack,
                                   cudaStream_t st) {
  const int n = 9 * d.C;
  pack_dw_weights_kernel<<<gb_ceil_div(n, 256), 256, 0, st>>>(
      static_cast<const __nv_bfloat16*>(w), static_cast<__nv_bfloat16*>(wpack), d.C);
  gb_count_launch();
  return cudaGetLastError();
}

cudaError_t launch_dwconv3x3(const gbconv_desc_s& d, const void* x, const void* w,
                             const float* bias, const void* res, void* y, int* err,
                             unsigned long long wait_ns, cudaStream_t st) {
  if (d.stride == 1) return launch_st<1>(d, x, w, bias, res, y, err, wait_ns, st);
  return launch_st<2>(d, x, w, bias, res, y, err, wait_ns, st);
}
