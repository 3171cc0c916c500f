// Depthwise 3x3 convolution (groups == C == K), NHWC bf16, fp32 accumulate,
// fused bias / residual / ReLU / ReLU6.
//
// The Momenta talk ("優化2：Depthwise卷積") splits a 3x3 conv into a per-channel
// spatial filter and a 1x1 channel mix; the spatial part loads each input
// value for only 9 multiply-adds, so it is bound by memory bandwidth, not
// arithmetic.  The kernel is therefore built to move each input byte from
// DRAM once:
//   * a thread owns 8 channels (one 16-byte vector) of one output column ow
//     and walks down a strip of TH output rows, keeping the 3 x 3 input window
//     in registers (fp32) and loading only the new input row(s) per step;
//   * consecutive threads of a warp own consecutive channel vectors, then
//     consecutive columns, so every load and store is a contiguous 16-byte
//     run of the NHWC row;
//   * weights are prepacked tap-major ([9][C] bf16) so one 16-byte load
//     fetches a tap for the thread's 8 channels; they stay in registers.
#include <cuda_bf16.h>

#include <algorithm>

#include "internal.h"

namespace {

constexpr int TH = 8;  // output rows per thread

struct DwParams {
  int N, C, H, W, OH, OW, pad, CV, strips, act;
};

__device__ __forceinline__ void bf16x8_to_f32(const uint4& v, float* f) {
  const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    f[2 * j] = __uint_as_float(u[j] << 16);
    f[2 * j + 1] = __uint_as_float(u[j] & 0xffff0000u);
  }
}

template <int ST>
__global__ void __launch_bounds__(128)
    dwconv3x3_kernel(const DwParams p, const __nv_bfloat16* __restrict__ x,
                     const __nv_bfloat16* __restrict__ w9c, const float* __restrict__ bias,
                     const __nv_bfloat16* __restrict__ res, __nv_bfloat16* __restrict__ y) {
  long long t = blockIdx.x * (long long)blockDim.x + threadIdx.x;
  const long long total = (long long)p.N * p.strips * p.OW * p.CV;
  if (t >= total) return;
  const int cv = (int)(t % p.CV);
  t /= p.CV;
  const int ow = (int)(t % p.OW);
  t /= p.OW;
  const int strip = (int)(t % p.strips);
  const int n = (int)(t / p.strips);
  const int c = cv * 8;

  float wr[9][8];
#pragma unroll
  for (int k = 0; k < 9; ++k)
    bf16x8_to_f32(__ldg(reinterpret_cast<const uint4*>(w9c + (size_t)k * p.C + c)), wr[k]);
  float b[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) b[j] = bias ? __ldg(bias + c + j) : 0.f;

  const int oh0 = strip * TH;
  const int iw0 = ow * ST - p.pad;
  const __nv_bfloat16* xn = x + (size_t)n * p.H * p.W * p.C + c;

  // load one input row (3 columns) of the window as raw bf16 vectors
  auto load_row = [&](int ih, uint4 (&dst)[3]) {
#pragma unroll
    for (int j = 0; j < 3; ++j) {
      const int iw = iw0 + j;
      if (ih >= 0 && ih < p.H && iw >= 0 && iw < p.W)
        dst[j] = __ldg(reinterpret_cast<const uint4*>(xn + ((size_t)ih * p.W + iw) * p.C));
      else
        dst[j] = make_uint4(0, 0, 0, 0);
    }
  };

  // window rows win[slot][col][ch]; slot rotates with the unrolled row index
  constexpr int SLOTS = 3;
  float win[SLOTS][3][8];
  {
    uint4 raw[3];
#pragma unroll
    for (int i = 0; i < 3; ++i) {
      load_row(oh0 * ST - p.pad + i, raw);
#pragma unroll
      for (int j = 0; j < 3; ++j) bf16x8_to_f32(raw[j], win[i][j]);
    }
  }

#pragma unroll
  for (int k = 0; k < TH; ++k) {
    const int oh = oh0 + k;
    if (oh >= p.OH) break;
    // prefetch the rows the next output needs (ST new rows)
    uint4 nxt[ST][3];
    if (k + 1 < TH && oh + 1 < p.OH) {
#pragma unroll
      for (int q = 0; q < ST; ++q) load_row((oh + 1) * ST - p.pad + (3 - ST) + q, nxt[q]);
    }
    // slots: row i of the current window lives in slot (k*ST + i) % 3
    float acc[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) acc[j] = b[j];
#pragma unroll
    for (int i = 0; i < 3; ++i) {
      const int sl = (k * ST + i) % SLOTS;
#pragma unroll
      for (int jj = 0; jj < 3; ++jj)
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[j] = fmaf(win[sl][jj][j], wr[i * 3 + jj][j], acc[j]);
    }
    const size_t off = (((size_t)n * p.OH + oh) * p.OW + ow) * p.C + c;
    if (res) {
      float r[8];
      bf16x8_to_f32(__ldg(reinterpret_cast<const uint4*>(res + off)), r);
#pragma unroll
      for (int j = 0; j < 8; ++j) acc[j] += r[j];
    }
    uint4 o;
    uint32_t* ou = reinterpret_cast<uint32_t*>(&o);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      float a0 = acc[2 * j], a1 = acc[2 * j + 1];
      if (p.act >= 1) {
        a0 = fmaxf(a0, 0.f);
        a1 = fmaxf(a1, 0.f);
      }
      if (p.act == 2) {
        a0 = fminf(a0, 6.f);
        a1 = fminf(a1, 6.f);
      }
      __nv_bfloat162 h = __floats2bfloat162_rn(a0, a1);
      ou[j] = *reinterpret_cast<uint32_t*>(&h);
    }
    *reinterpret_cast<uint4*>(y + off) = o;
    // retire the oldest ST rows, install the prefetched ones
    if (k + 1 < TH && oh + 1 < p.OH) {
#pragma unroll
      for (int q = 0; q < ST; ++q) {
        const int sl = (k * ST + 3 + q) % SLOTS;
#pragma unroll
        for (int j = 0; j < 3; ++j) bf16x8_to_f32(nxt[q][j], win[sl][j]);
      }
    }
  }
}

// [C][3][3] -> [9][C]
__global__ void pack_dw_weights_kernel(const __nv_bfloat16* __restrict__ w,
                                       __nv_bfloat16* __restrict__ wp, int C) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= 9 * C) return;
  const int k = i / C, c = i % C;
  wp[i] = w[c * 9 + k];
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
                             const float* bias, const void* res, void* y, cudaStream_t st) {
  DwParams p{d.N, d.C, d.H, d.W, d.OH, d.OW, d.pad, d.C / 8, gb_ceil_div(d.OH, TH), d.act};
  const long long total = (long long)p.N * p.strips * p.OW * p.CV;
  const int block = 128;
  const long long grid = gb_ceil_div_ll(total, block);
  if (grid > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  auto xb = static_cast<const __nv_bfloat16*>(x);
  auto wb = static_cast<const __nv_bfloat16*>(w);
  auto rb = static_cast<const __nv_bfloat16*>(res);
  auto yb = static_cast<__nv_bfloat16*>(y);
  if (d.stride == 1)
    dwconv3x3_kernel<1><<<(unsigned)grid, block, 0, st>>>(p, xb, wb, bias, rb, yb);
  else
    dwconv3x3_kernel<2><<<(unsigned)grid, block, 0, st>>>(p, xb, wb, bias, rb, yb);
  return cudaGetLastError();
}
