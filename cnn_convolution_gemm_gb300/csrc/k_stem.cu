// Stride-2 convolutions over 8 (or 4) channels — the network stem, 7x7 / 2 on
// an RGB image padded to 8 (or 4) channels — as stride-1 implicit GEMMs.
//
// With 8 channels an implicit-GEMM k-step of 64 reduction elements holds 8
// filter taps, and each tap is its own 128-pixel x 16-byte TMA im2col box:
// many tiny copies per k-step, and the kernel waits on them.  A space-to-depth
// rewrite removes the stride instead.  With
//   X2[n][h2][w2][(dy*2 + dx)*8 + c] = x[n][2*h2 + dy][2*w2 + dx][c]     (32 ch)
// the output pixel (oh, ow) of the stride-2 conv reads input rows
// 2*oh - pad + i, i < R; writing i - pad = 2*a + dy (dy in {0, 1}) turns that
// into block rows oh + a, a in [floor(-pad/2), floor((R-1-pad)/2)], so
//   y[n][oh][ow][k] = sum_{a,b} sum_{dy,dx,c} X2[n][oh+a][ow+b][(dy,dx,c)] *
//                     W2[k][a][b][(dy,dx,c)],   W2 = w[k][2a+dy+pad][2b+dx+pad][c]
// (zero where that tap is outside the R x R kernel): a stride-1 R2 x R2 conv
// (R2 = 4 for R = 7) over 32 channels with asymmetric padding, which runs on
// the ordinary implicit GEMM (one 128 x 64 im2col box per k-step).  The zero
// taps cost tensor work (16 taps x 64 for 49 x 8 useful), which is cheap here.
#include <cuda_bf16.h>

#include <algorithm>

#include "internal.h"
#include "ptx.cuh"

namespace {

struct StemGeom {
  int a_min, a_max, R2;  // block-tap range of the rewritten conv
};

StemGeom stem_geom(const gbconv_desc_s& d) {
  StemGeom g;
  // floor division of -pad and (R - 1 - pad) by 2
  g.a_min = -((d.pad + 1) / 2);
  g.a_max = (d.R - 1 - d.pad) >= 0 ? (d.R - 1 - d.pad) / 2 : -((d.pad - d.R + 2) / 2);
  g.R2 = g.a_max - g.a_min + 1;
  return g;
}

// the 32-channel space-to-depth desc the implicit GEMM runs on
gbconv_desc_s stem_desc(const gbconv_desc_s& d) {
  const StemGeom g = stem_geom(d);
  gbconv_desc_s e = d;
  e.C = 32;
  e.H = d.H / 2;
  e.W = d.W / 2;
  e.R = e.S = g.R2;
  e.stride = 1;
  e.dil = 1;
  e.pad = -g.a_min;                 // rows before
  e.pad_hi_delta = g.a_max - e.pad;  // rows after minus rows before
  e.OH = d.OH;
  e.OW = d.OW;
  return e;
}

// one output pixel (64 bytes) per thread: its 2x2 input pixels, 16 bytes each
__global__ void space_to_depth8_kernel(const uint4* __restrict__ x, uint4* __restrict__ x2,
                                       int N, int H, int W) {
  const int H2 = H / 2, W2 = W / 2;
  const long long total = (long long)N * H2 * W2;
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < total;
       i += (long long)gridDim.x * blockDim.x) {
    const int w2 = (int)(i % W2);
    const long long t = i / W2;
    const int h2 = (int)(t % H2);
    const long long n = t / H2;
    const long long row0 = (n * H + 2 * h2) * W + 2 * w2;  // input pixel (2h2, 2w2)
#pragma unroll
    for (int dy = 0; dy < 2; ++dy)
#pragma unroll
      for (int dx = 0; dx < 2; ++dx) x2[i * 4 + dy * 2 + dx] = __ldg(x + row0 + dy * W + dx);
  }
}

// w [K][R][R][8] -> packed implicit-GEMM weights of the rewritten conv:
// [K][R2*R2][64], channel ch < 32 = (dy, dx, c), ch >= 32 zero
__global__ void pack_stem_weights_kernel(const __nv_bfloat16* __restrict__ w,
                                         __nv_bfloat16* __restrict__ wp, int K, int R, int pad,
                                         int a_min, int R2) {
  const long long total = (long long)K * R2 * R2 * 64;
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < total;
       i += (long long)gridDim.x * blockDim.x) {
    const int ch = (int)(i % 64);
    const long long kt = i / 64;
    const int tap = (int)(kt % (R2 * R2));
    const long long k = kt / (R2 * R2);
    float v = 0.f;
    if (ch < 32) {
      const int dy = ch / 16, dx = (ch / 8) % 2, c = ch % 8;
      const int a = tap / R2 + a_min, b = tap % R2 + a_min;
      const int ii = 2 * a + dy + pad, jj = 2 * b + dx + pad;
      if (ii >= 0 && ii < R && jj >= 0 && jj < R)
        v = __bfloat162float(w[((k * R + ii) * R + jj) * 8 + c]);
    }
    wp[i] = __float2bfloat16_rn(v);
  }
}

int grid_for(long long n) { return (int)std::min<long long>((n + 255) / 256, 152LL * 16); }

// ---------------------------------------------------------------------------
// Space-to-depth by 4.  With C = 4 (an RGB image padded to 4 channels) the
// factor-2 rewrite still moves 64-byte pixels and pads every k-step to 64
// channels; a factor of 4 gives 16 C = 64 (or 128) channels per block pixel:
//   X4[n][bh][bw][(dy*4 + dx)*C + c] = x[n][4 bh + dy][4 bw + dx][c]
// Output pixel (2 bh + py, 2 bw + px) of the stride-2 conv reads input rows
// 4 bh + (2 py - pad + i), i < R; with 2 py - pad + i = 4 a + dy that is block
// row bh + a, a in [floor(-pad / 4), floor((R + 1 - pad) / 4)], so the 2 x 2
// output pixels of a block are one stride-1 R4 x R4 conv over the block grid
// with 4 K output columns (py, px, k):
//   W4[(py*2 + px)*K + k][a][b][(dy, dx, c)] = w[k][4a + dy - 2py + pad][4b + dx - 2px + pad][c]
// (zero where that tap is outside the R x R kernel).  The implicit GEMM's
// epilogue writes column (py, px, k) of block (n, bh, bw) to output pixel
// (n, 2 bh + py, 2 bw + px), channel k.

struct Stem4Geom {
  int a_min, a_max, R4;
};

int floor_div4(int v) { return v >= 0 ? v / 4 : -((-v + 3) / 4); }

Stem4Geom stem4_geom(const gbconv_desc_s& d) {
  Stem4Geom g;
  g.a_min = floor_div4(-d.pad);
  g.a_max = floor_div4(d.R + 1 - d.pad);
  g.R4 = g.a_max - g.a_min + 1;
  return g;
}

// the block-grid desc the implicit GEMM runs on
gbconv_desc_s stem4_desc(const gbconv_desc_s& d) {
  const Stem4Geom g = stem4_geom(d);
  gbconv_desc_s e = d;
  e.C = 16 * d.C;
  e.H = d.H / 4;
  e.W = d.W / 4;
  e.K = 4 * d.K;
  e.R = e.S = g.R4;
  e.stride = 1;
  e.dil = 1;
  e.pad = -g.a_min;                  // block rows before
  e.pad_hi_delta = g.a_max - e.pad;  // block rows after minus rows before
  e.OH = d.OH / 2;
  e.OW = d.OW / 2;
  return e;
}

// one (block pixel, dy) per thread: input row 4 bh + dy, columns 4 bw .. 4 bw + 3,
// 4 C contiguous values, copied to channels dy * 4C .. of the block pixel
__global__ void space_to_depth4_kernel(const uint4* __restrict__ x, uint4* __restrict__ x4,
                                       int N, int H, int W, int C) {
  gb::allow_dependents();  // the block-grid GEMM sets up meanwhile
  const int BH = H / 4, BW = W / 4, v = C / 2;  // v: 16-byte vectors per 4 pixels
  const long long total = (long long)N * BH * BW * 4;
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < total;
       i += (long long)gridDim.x * blockDim.x) {
    const int dy = (int)(i & 3);
    const long long blk = i >> 2;
    const int bw = (int)(blk % BW);
    const long long t = blk / BW;
    const int bh = (int)(t % BH);
    const long long n = t / BH;
    const long long src = ((n * H + 4 * bh + dy) * W + 4 * bw) * C / 8;  // in 16-byte units
    const long long dst = (blk * 16 * C + dy * 4 * C) / 8;
    for (int q = 0; q < v; ++q) x4[dst + q] = __ldg(x + src + q);
  }
}

// w [K][R][R][C] -> packed implicit-GEMM weights of the block conv:
// [4K][R4*R4][16C], column (py*2 + px)*K + k, channel (dy*4 + dx)*C + c
__global__ void pack_stem4_weights_kernel(const __nv_bfloat16* __restrict__ w,
                                          __nv_bfloat16* __restrict__ wp, int K, int R, int C,
                                          int pad, int a_min, int R4) {
  const int CB = 16 * C;
  const long long total = (long long)4 * K * R4 * R4 * CB;
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < total;
       i += (long long)gridDim.x * blockDim.x) {
    const int ch = (int)(i % CB);
    const long long ct = i / CB;
    const int tap = (int)(ct % (R4 * R4));
    const int col = (int)(ct / (R4 * R4));
    const int g = col / K, k = col % K, py = g >> 1, px = g & 1;
    const int dy = ch / (4 * C), dx = (ch / C) % 4, c = ch % C;
    const int a = tap / R4 + a_min, b = tap % R4 + a_min;
    const int ii = 4 * a + dy - 2 * py + pad, jj = 4 * b + dx - 2 * px + pad;
    float v = 0.f;
    if (ii >= 0 && ii < R && jj >= 0 && jj < R)
      v = __bfloat162float(w[(((long long)k * R + ii) * R + jj) * C + c]);
    wp[i] = __float2bfloat16_rn(v);
  }
}

}  // namespace

bool stem_s2d4_applicable(const gbconv_desc_s& d, const char** why) {
  if (d.C != 4 && d.C != 8) return *why = "needs C == 4 or 8", false;
  if (d.stride != 2 || d.dil != 1 || d.groups != 1 || d.R != d.S)
    return *why = "needs stride 2, dilation 1, groups 1, square kernel", false;
  if (d.H % 4 || d.W % 32) return *why = "needs H % 4 == 0 and W % 32 == 0", false;
  if (d.OH != d.H / 2 || d.OW != d.W / 2) return *why = "needs an output of H/2 x W/2", false;
  if (d.K != 64) return *why = "needs K == 64", false;
  if (d.has_residual) return *why = "no residual", false;
  const Stem4Geom g = stem4_geom(d);
  if (g.R4 < 1 || g.R4 > 8 || g.a_min < -8) return *why = "kernel size out of range", false;
  if ((long long)d.N * (d.H / 4) * (d.W / 4) >= (1LL << 31))
    return *why = "N*H*W/16 >= 2^31", false;
  return true;
}

size_t stem_s2d4_workspace_bytes(const gbconv_desc_s& d) {
  return ((size_t)d.N * (d.H / 4) * (d.W / 4) * 16 * d.C * 2 + 255) / 256 * 256;
}

size_t stem_s2d4_packed_bytes(const gbconv_desc_s& d) {
  const Stem4Geom g = stem4_geom(d);
  return (size_t)4 * d.K * g.R4 * g.R4 * 16 * d.C * 2;
}

cudaError_t launch_pack_stem4_weights(const gbconv_desc_s& d, const void* w, void* wpack,
                                      cudaStream_t st) {
  const Stem4Geom g = stem4_geom(d);
  const long long total = (long long)4 * d.K * g.R4 * g.R4 * 16 * d.C;
  pack_stem4_weights_kernel<<<grid_for(total), 256, 0, st>>>(
      static_cast<const __nv_bfloat16*>(w), static_cast<__nv_bfloat16*>(wpack), d.K, d.R, d.C,
      d.pad, g.a_min, g.R4);
  gb_count_launch();
  return cudaGetLastError();
}

cudaError_t launch_stem_s2d4(const gbconv_desc_s& d, const void* x, const void* wpack,
                             const float* bias, void* y, void* ws, int* err,
                             unsigned long long wait_ns, cudaStream_t st) {
  const long long rows = (long long)d.N * (d.H / 4) * (d.W / 4) * 4;
  space_to_depth4_kernel<<<grid_for(rows), 256, 0, st>>>(static_cast<const uint4*>(x),
                                                         static_cast<uint4*>(ws), d.N, d.H, d.W,
                                                         d.C);
  gb_count_launch();
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  IgemmSplit sp;
  sp.s2d4_k = d.K;
  // 128-column tiles (the (py = 0) and (py = 1) halves of the 2x2 pixels), two CTAs
  // per SM: measured 81 us against 103 us for 256-column tiles on ResNet-50's stem
  return launch_igemm_bf16(stem4_desc(d), 128, ws, wpack, bias, nullptr, y, err, wait_ns, st, sp);
}

bool stem_s2d_applicable(const gbconv_desc_s& d, const char** why) {
  if (d.C != 8) return *why = "needs C == 8", false;
  if (d.stride != 2 || d.dil != 1 || d.groups != 1 || d.R != d.S)
    return *why = "needs stride 2, dilation 1, groups 1, square kernel", false;
  if (d.H % 2 || d.W % 2 || d.OH != d.H / 2 || d.OW != d.W / 2)
    return *why = "needs even H, W and an output of H/2 x W/2", false;
  if (d.K % 8) return *why = "needs K multiple of 8", false;
  const StemGeom g = stem_geom(d);
  if (g.R2 < 1 || g.R2 > 8) return *why = "kernel size out of range", false;
  if ((long long)d.N * d.OH * d.OW >= (1LL << 31)) return *why = "N*OH*OW >= 2^31", false;
  return true;
}

size_t stem_s2d_workspace_bytes(const gbconv_desc_s& d) {
  return ((size_t)d.N * (d.H / 2) * (d.W / 2) * 32 * 2 + 255) / 256 * 256;
}

size_t stem_s2d_packed_bytes(const gbconv_desc_s& d) {
  const StemGeom g = stem_geom(d);
  return (size_t)d.K * g.R2 * g.R2 * 64 * 2;
}

cudaError_t launch_pack_stem_weights(const gbconv_desc_s& d, const void* w, void* wpack,
                                     cudaStream_t st) {
  const StemGeom g = stem_geom(d);
  const long long total = (long long)d.K * g.R2 * g.R2 * 64;
  pack_stem_weights_kernel<<<grid_for(total), 256, 0, st>>>(
      static_cast<const __nv_bfloat16*>(w), static_cast<__nv_bfloat16*>(wpack), d.K, d.R, d.pad,
      g.a_min, g.R2);
  gb_count_launch();
  return cudaGetLastError();
}

cudaError_t launch_stem_s2d(const gbconv_desc_s& d, const void* x, const void* wpack,
                            const float* bias, const void* res, void* y, void* ws, int* err,
                            unsigned long long wait_ns, cudaStream_t st) {
  const long long pixels = (long long)d.N * (d.H / 2) * (d.W / 2);
  space_to_depth8_kernel<<<grid_for(pixels), 256, 0, st>>>(static_cast<const uint4*>(x),
                                                           static_cast<uint4*>(ws), d.N, d.H, d.W);
  gb_count_launch();
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const gbconv_desc_s e2 = stem_desc(d);
  const int bn = d.K <= 64 ? 64 : (d.K <= 128 ? 128 : 256);
  return launch_igemm_bf16(e2, bn, ws, wpack, bias, res, y, err, wait_ns, st);
}
