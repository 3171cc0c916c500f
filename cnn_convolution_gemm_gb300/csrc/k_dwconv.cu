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
//     columns sized to fill a buffer); for each, one 4-D TMA load
//     brings the input rows/columns the block needs (its halo included) into
//     shared memory, and out-of-bounds elements arrive as zeros, which is the
//     padding;
//   * two shared-memory buffers: the load of the next block is in flight while
//     the current one is computed, so bytes in flight do not depend on
//     registers or occupancy;
//   * a thread owns 4 channels of two adjacent output columns and walks down
//     the block's rows keeping the bf16 input window in registers (4 new
//     8-byte shared loads per output row), multiplying bf16 operands into fp32
//     accumulators with fma.rn.f32.bf16;
//   * weights are prepacked tap-major ([9][C] bf16): one 16-byte load per tap.
#include <cuda_bf16.h>

#include <algorithm>

#include "internal.h"
#include "ptx.cuh"

namespace {

constexpr int MAX_THREADS = 384;
constexpr int NBUF = 3;              // shared-memory ring depth: two loads in flight
constexpr int BUF_MAX = 66 * 1024;   // bytes per buffer

template <int ST>
struct DwCfg {
  static constexpr int RB = ST == 1 ? 8 : 4;      // output rows per block
  static constexpr int IH = (RB - 1) * ST + 3;    // input rows per block
  static constexpr int SMEM = NBUF * BUF_MAX + 1024 + 64;
};

struct DwParams {
  int N, C, H, W, OH, OW, pad, act;
  int cb;                  // channels per block (all of C when C <= 256)
  int owt, iw, buf_bytes;  // output columns per block, input columns, bytes per buffer
  int cslices, rblocks, cblocks;
  long long nblocks;
  int* err;
  unsigned long long wait_ns;
};

// work items of one block: (4-channel group, pair of output columns)
__host__ __device__ inline int gb_items(const DwParams& p) { return ((p.owt + 1) / 2) * (p.cb / 4); }

// two fp32 values in one 64-bit register pair (the operand of fma.rn.f32x2)
typedef unsigned long long f32x2;

__device__ __forceinline__ f32x2 pack2(float lo, float hi) {
  f32x2 r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ float2 unpack2(f32x2 v) {
  float2 r;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(r.x), "=f"(r.y) : "l"(v));
  return r;
}
// bf16x2 (one 32-bit word) -> two fp32 in a register pair
__device__ __forceinline__ f32x2 bf16x2_to_f32x2(uint32_t u) {
  return pack2(__uint_as_float(u << 16), __uint_as_float(u & 0xffff0000u));
}
__device__ __forceinline__ void ffma2(f32x2& d, f32x2 a, f32x2 b) {
  asm("fma.rn.f32x2 %0, %1, %2, %0;" : "+l"(d) : "l"(a), "l"(b));
}

// d += a * w with bf16 operands and an fp32 accumulator, one rounding (the same
// result as converting both operands to fp32 first)
__device__ __forceinline__ void fma_bf16(float& d, unsigned short a, unsigned short w) {
  asm("fma.rn.f32.bf16 %0, %1, %2, %0;" : "+f"(d) : "h"(a), "h"(w));
}
// four bf16 values of an 8-byte load, one per 16-bit register
__device__ __forceinline__ void split4(const uint2 v, unsigned short (&h)[4]) {
  asm("mov.b32 {%0, %1}, %2;" : "=h"(h[0]), "=h"(h[1]) : "r"(v.x));
  asm("mov.b32 {%0, %1}, %2;" : "=h"(h[2]), "=h"(h[3]) : "r"(v.y));
}

template <int ST>
__global__ void __launch_bounds__(MAX_THREADS, 1)
    dwconv3x3_tma_kernel(const __grid_constant__ CUtensorMap tm_x, const DwParams p,
                         const __nv_bfloat16* __restrict__ w9c, const float* __restrict__ bias,
                         const __nv_bfloat16* __restrict__ res, __nv_bfloat16* __restrict__ y) {
  using Cf = DwCfg<ST>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + NBUF * BUF_MAX);

  if (threadIdx.x == 0) {
    for (int i = 0; i < NBUF; ++i) gb::mbar_init(&full[i], 1);
    gb::fence_barrier_init();
    gb::tma_prefetch_desc(&tm_x);
  }
  __syncthreads();

  auto block_coords = [&](long long b, int& n, int& cs, int& rb, int& cb) {
    cb = (int)(b % p.cblocks);
    b /= p.cblocks;
    rb = (int)(b % p.rblocks);
    b /= p.rblocks;
    cs = (int)(b % p.cslices);
    n = (int)(b / p.cslices);
  };
  auto issue = [&](long long b, int buf) {
    int n, cs, rb, cb;
    block_coords(b, n, cs, rb, cb);
    gb::fence_proxy_async_smem();
    gb::mbar_arrive_expect_tx(&full[buf], p.buf_bytes);
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4, %5}], [%6];" ::"r"(gb::smem_u32(smem + buf * BUF_MAX)),
        "l"(reinterpret_cast<uint64_t>(&tm_x)), "r"(cs * p.cb), "r"(cb * p.owt * ST - p.pad),
        "r"(rb * Cf::RB * ST - p.pad), "r"(n), "r"(gb::smem_u32(&full[buf]))
        : "memory");
  };

  // ring of NBUF buffers: block i of this CTA lives in buffer i % NBUF; the
  // load of block i + NBUF - 1 is issued before block i is computed
  const long long first = blockIdx.x, step = gridDim.x;
  if (threadIdx.x == 0)
    for (int i = 0; i < NBUF - 1; ++i)
      if (first + i * step < p.nblocks) issue(first + i * step, i);
  int it = 0;
  bool ok = true;
  const int groups = p.cb / 4;
  const int items = gb_items(p);
  unsigned short wr[9][4];  // this thread's weights (kept while its work item is unchanged)
  float bz[4];
  int w_item = -1, w_cs = -1;
  for (long long b = first; b < p.nblocks; b += step, ++it) {
    const int buf = it % NBUF;
    const long long nb = b + (NBUF - 1) * step;
    if (threadIdx.x == 0 && nb < p.nblocks) issue(nb, (it + NBUF - 1) % NBUF);
    const uint32_t parity = (uint32_t)((it / NBUF) & 1);
    if (!gb::mbar_wait_bounded(&full[buf], parity, p.wait_ns, p.err)) ok = false;
    if (!__syncthreads_and(ok)) {
      // a wait ran out: let every load this CTA issued land before it exits
      if (threadIdx.x == 0)
        for (int i = 0; i < NBUF; ++i) {
          const int k = it + i;
          if (first + (long long)k * step < p.nblocks)
            gb::mbar_wait_bounded(&full[k % NBUF], (uint32_t)((k / NBUF) & 1), p.wait_ns, p.err);
        }
      break;
    }
    int n, cs, rb, cb;
    block_coords(b, n, cs, rb, cb);
    const uint8_t* tile = smem + buf * BUF_MAX;
    // work items: (4-channel group g, pair of output columns j0, j0 + 1), g fastest
    for (int item = threadIdx.x; item < items; item += blockDim.x) {
      const int g = item % groups;
      const int j0 = 2 * (item / groups);
      const int c = cs * p.cb + g * 4;
      const int ow0 = cb * p.owt + j0;
      if (c >= p.C || ow0 >= p.OW || j0 >= p.owt) continue;
      const bool two = j0 + 1 < p.owt && ow0 + 1 < p.OW;
      if (item != w_item || cs != w_cs) {  // weights and bias of these 4 channels
#pragma unroll
        for (int k = 0; k < 9; ++k)
          split4(__ldg(reinterpret_cast<const uint2*>(w9c + (size_t)k * p.C + c)), wr[k]);
#pragma unroll
        for (int q = 0; q < 4; ++q) bz[q] = bias ? __ldg(bias + c + q) : 0.f;
        w_item = item;
        w_cs = cs;
      }
      // tile-local input columns of the pair: j0*ST + s (first), (j0+1)*ST + s (second)
      constexpr int NC = ST + 3;  // distinct input columns the two outputs read
      const int lc = j0 * ST;
      auto ld = [&](int row, int col, unsigned short (&h)[4]) {
        split4(*reinterpret_cast<const uint2*>(
                   tile + ((size_t)(row * p.iw + lc + col) * p.cb + g * 4) * 2),
               h);
      };
      unsigned short win[3][NC][4];  // bf16 window; input row rho lives in slot rho % 3
#pragma unroll
      for (int i = 0; i < 3; ++i)
#pragma unroll
        for (int cc = 0; cc < NC; ++cc) ld(i, cc, win[i][cc]);
#pragma unroll
      for (int k = 0; k < Cf::RB; ++k) {
        const int oh = rb * Cf::RB + k;
        if (oh >= p.OH) break;
        if (k > 0) {  // the ST new input rows of this output row's window
#pragma unroll
          for (int q = 0; q < ST; ++q) {
            const int rho = (k - 1) * ST + 3 + q;
#pragma unroll
            for (int cc = 0; cc < NC; ++cc) ld(rho, cc, win[rho % 3][cc]);
          }
        }
        float acc[2][4];
#pragma unroll
        for (int o = 0; o < 2; ++o)
#pragma unroll
          for (int q = 0; q < 4; ++q) acc[o][q] = bz[q];
#pragma unroll
        for (int i = 0; i < 3; ++i) {
          const int sl = (k * ST + i) % 3;
#pragma unroll
          for (int s = 0; s < 3; ++s) {
#pragma unroll
            for (int o = 0; o < 2; ++o)
#pragma unroll
              for (int q = 0; q < 4; ++q) fma_bf16(acc[o][q], win[sl][o * ST + s][q], wr[i * 3 + s][q]);
          }
        }
#pragma unroll
        for (int o = 0; o < 2; ++o) {
          if (o == 1 && !two) break;
          float* a = acc[o];
          const size_t off = (((size_t)n * p.OH + oh) * p.OW + ow0 + o) * p.C + c;
          if (res) {
            const uint2 rv = __ldg(reinterpret_cast<const uint2*>(res + off));
            a[0] += __uint_as_float(rv.x << 16);
            a[1] += __uint_as_float(rv.x & 0xffff0000u);
            a[2] += __uint_as_float(rv.y << 16);
            a[3] += __uint_as_float(rv.y & 0xffff0000u);
          }
          __nv_bfloat162 h0 = __floats2bfloat162_rn(a[0], a[1]);
          __nv_bfloat162 h1 = __floats2bfloat162_rn(a[2], a[3]);
          // the activation commutes with the (monotone) rounding to bf16
          if (p.act >= 1) {
            const __nv_bfloat162 z = __float2bfloat162_rn(0.f);
            h0 = __hmax2(h0, z);
            h1 = __hmax2(h1, z);
          }
          if (p.act == 2) {
            const __nv_bfloat162 six = __float2bfloat162_rn(6.f);
            h0 = __hmin2(h0, six);
            h1 = __hmin2(h1, six);
          }
          uint2 ov;
          ov.x = *reinterpret_cast<uint32_t*>(&h0);
          ov.y = *reinterpret_cast<uint32_t*>(&h1);
          *reinterpret_cast<uint2*>(y + off) = ov;
        }
      }
    }
    __syncthreads();  // the buffer is free for the load issued next iteration
  }
  // On normal exit every issued load has been waited for: a load is issued
  // only for a block index inside the list, and every such block is processed.
}

// [C][3][3] -> [9][C]
__global__ void pack_dw_weights_kernel(const __nv_bfloat16* __restrict__ w,
                                       __nv_bfloat16* __restrict__ wp, int C) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= 9 * C) return;
  const int k = i / C, c = i % C;
  wp[i] = w[c * 9 + k];
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
  p.act = d.act;
  // channel slices of <= 256 channels (the TMA box limit), as few as possible,
  // so each block reads whole contiguous pixel rows
  p.cslices = gb_ceil_div(d.C, 256);
  p.cb = gb_ceil_div(gb_ceil_div(d.C, p.cslices), 8) * 8;
  // widest column block whose input tile fits one buffer
  const int px_bytes = p.cb * 2;
  int iw_max = BUF_MAX / (Cf::IH * px_bytes);
  int owt = (iw_max - 3) / ST + 1;
  if (owt > d.OW) owt = d.OW;
  if (owt > 256 / ST - 2) owt = 256 / ST - 2;  // TMA box dimension <= 256
  if (owt < 1) return cudaErrorInvalidConfiguration;
  owt = gb_ceil_div(d.OW, gb_ceil_div(d.OW, owt));  // equal-width column blocks
  p.owt = owt;
  p.iw = (p.owt - 1) * ST + 3;
  p.buf_bytes = Cf::IH * p.iw * px_bytes;
  p.rblocks = gb_ceil_div(d.OH, Cf::RB);
  p.cblocks = gb_ceil_div(d.OW, p.owt);
  p.nblocks = (long long)d.N * p.cslices * p.rblocks * p.cblocks;
  p.err = err;
  p.wait_ns = wait_ns;
  CUtensorMap tm;
  cuuint64_t dims[4] = {(cuuint64_t)d.C, (cuuint64_t)d.W, (cuuint64_t)d.H, (cuuint64_t)d.N};
  cuuint64_t strides[3] = {(cuuint64_t)d.C * 2, (cuuint64_t)d.W * d.C * 2,
                           (cuuint64_t)d.H * d.W * d.C * 2};
  cuuint32_t box[4] = {(cuuint32_t)p.cb, (cuuint32_t)p.iw, Cf::IH, 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  if (gb_encode_tiled(&tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(x), dims,
                      strides, box, estr, CU_TENSOR_MAP_SWIZZLE_NONE) != CUDA_SUCCESS)
    return cudaErrorInvalidValue;
  cudaError_t e = cudaFuncSetAttribute(dwconv3x3_tma_kernel<ST>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, Cf::SMEM);
  if (e != cudaSuccess) return e;
  const long long grid = std::min<long long>(p.nblocks, gb_num_sms());
  // threads: the block's work items split into equal rounds of <= MAX_THREADS
  const int items = gb_items(p);
  const int rounds = gb_ceil_div(items, MAX_THREADS);
  const int threads = gb_ceil_div(gb_ceil_div(items, rounds), 32) * 32;
  dwconv3x3_tma_kernel<ST><<<(unsigned)grid, threads, Cf::SMEM, st>>>(
      tm, p, static_cast<const __nv_bfloat16*>(w), bias, static_cast<const __nv_bfloat16*>(res),
      static_cast<__nv_bfloat16*>(y));
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_pack_dw_weights(const gbconv_desc_s& d, const void* w, void* wpack,
                                   cudaStream_t st) {
  const int n = 9 * d.C;
  pack_dw_weights_kernel<<<gb_ceil_div(n, 256), 256, 0, st>>>(
      static_cast<const __nv_bfloat16*>(w), static_cast<__nv_bfloat16*>(wpack), d.C);
  return cudaGetLastError();
}

cudaError_t launch_dwconv3x3(const gbconv_desc_s& d, const void* x, const void* w,
                             const float* bias, const void* res, void* y, int* err,
                             unsigned long long wait_ns, cudaStream_t st) {
  if (d.stride == 1) return launch_st<1>(d, x, w, bias, res, y, err, wait_ns, st);
  return launch_st<2>(d, x, w, bias, res, y, err, wait_ns, st);
}
