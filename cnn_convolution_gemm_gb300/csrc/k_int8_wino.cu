// int8 Winograd F(2x2, 3x3) with float intermediates, exact.
//
// The MegEngine Beta report (native int8 inference, ARM without dotprod)
// keeps the Winograd-domain values in a float format instead of restricting
// the int8 weights to 6 bits so that the int16/int32 intermediates cannot
// overflow.  Here the float quantities are made to stay integers below 2^24,
// so the result equals the direct int8 convolution bit for bit:
//   * transforms with the halves of F(2,3) moved into G:
//       B^T = [[1,0,-1,0],[0,1,1,0],[0,-1,1,0],[0,1,0,-1]],
//       2G  = [[2,0,0],[1,1,1],[1,-1,1],[0,0,2]],  A^T = [[1,1,1,0],[0,1,-1,-1]];
//   * V = B^T d B of an int8 4x4 patch is an integer, |V| <= 512: exact in fp16;
//   * 4U = (2G) g (2G)^T of an int8 3x3 filter is an integer, |4U| <= 1152,
//     split at prepack into 4U = 32 Uh + Ul with Ul in [0, 31], |Uh| <= 36
//     (both exact in fp16);
//   * the 16 Winograd-domain GEMMs (tcgen05, fp16 operands, fp32 accumulate)
//     produce Ml = sum_c Ul V and Mh = sum_c Uh V, whose magnitudes stay below
//     2^24 for up to 896 channels, so fp32 holds them exactly;
//   * 4y = A^T (32 Mh + Ml) A in int32, y = (4y) / 4 exactly, then the int8
//     epilogue: + int32 bias, fp32 requant (round to nearest even), clamp, ReLU.
#include <cuda_fp16.h>

#include <algorithm>

#include "internal.h"

namespace {

constexpr int MAXC = 896;  // channels (rounded up to 16) for which the fp32 sums stay exact

struct Geo {
  int TH, TW, Cp;
  long long T;
};

Geo geo(const gbconv_desc_s& d) {
  Geo g;
  g.TH = (d.OH + 1) / 2;
  g.TW = (d.OW + 1) / 2;
  g.Cp = (d.C + 15) / 16 * 16;
  g.T = (long long)d.N * g.TH * g.TW;
  return g;
}

int grid_for(long long n) { return (int)std::min<long long>((n + 255) / 256, 152LL * 32); }

// int8 w [K][3][3][C] -> fp16 [16][2K][Cp]: rows k hold Ul, rows K + k hold Uh
__global__ void i8w_filter_kernel(const int8_t* __restrict__ w, __half* __restrict__ u, int K,
                                  int C, int Cp) {
  const long long total = (long long)K * Cp;
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < total;
       i += (long long)gridDim.x * blockDim.x) {
    const int c = (int)(i % Cp);
    const int k = (int)(i / Cp);
    int g[3][3];
#pragma unroll
    for (int r = 0; r < 3; ++r)
#pragma unroll
      for (int s = 0; s < 3; ++s) g[r][s] = c < C ? (int)w[(((long long)k * 3 + r) * 3 + s) * C + c] : 0;
    // t = (2G) g: rows 2g0, g0 + g1 + g2, g0 - g1 + g2, 2g2
    int t[4][3];
#pragma unroll
    for (int s = 0; s < 3; ++s) {
      t[0][s] = 2 * g[0][s];
      t[1][s] = g[0][s] + g[1][s] + g[2][s];
      t[2][s] = g[0][s] - g[1][s] + g[2][s];
      t[3][s] = 2 * g[2][s];
    }
#pragma unroll
    for (int a = 0; a < 4; ++a) {
      const int u4[4] = {2 * t[a][0], t[a][0] + t[a][1] + t[a][2], t[a][0] - t[a][1] + t[a][2],
                         2 * t[a][2]};
#pragma unroll
      for (int b = 0; b < 4; ++b) {
        const int lo = u4[b] & 31;        // in [0, 31]
        const int hi = (u4[b] - lo) / 32;  // exact
        const long long xi = a * 4 + b;
        u[(xi * 2 * K + k) * Cp + c] = __int2half_rn(lo);
        u[(xi * 2 * K + K + k) * Cp + c] = __int2half_rn(hi);
      }
    }
  }
}

// V[xi][t][c] = (B^T d B)[xi] of tile t's 4x4 int8 patch, fp16; 4 channels per thread
__global__ void i8w_input_kernel(const int8_t* __restrict__ x, __half* __restrict__ v, int H,
                                 int W, int C, int Cp, int pad, int TH, int TW, long long T) {
  const int C4 = Cp / 4;
  const long long total = T * C4;
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < total;
       i += (long long)gridDim.x * blockDim.x) {
    const int c4 = (int)(i % C4);
    const long long t = i / C4;
    const int tw = (int)(t % TW);
    const long long r1 = t / TW;
    const int th = (int)(r1 % TH);
    const long long n = r1 / TH;
    const int h0 = 2 * th - pad, w0 = 2 * tw - pad, c = 4 * c4;
    int d[4][4][4];  // [row][col][channel]
#pragma unroll
    for (int a = 0; a < 4; ++a)
#pragma unroll
      for (int b = 0; b < 4; ++b) {
        const int hh = h0 + a, ww = w0 + b;
        char4 q = make_char4(0, 0, 0, 0);
        if (hh >= 0 && hh < H && ww >= 0 && ww < W && c < C)
          q = *reinterpret_cast<const char4*>(x + ((n * H + hh) * W + ww) * C + c);
        d[a][b][0] = q.x;
        d[a][b][1] = q.y;
        d[a][b][2] = q.z;
        d[a][b][3] = q.w;
      }
    // rows: e = B^T d; then V = e B (the same combination along columns)
    int e[4][4][4];
#pragma unroll
    for (int b = 0; b < 4; ++b)
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        e[0][b][q] = d[0][b][q] - d[2][b][q];
        e[1][b][q] = d[1][b][q] + d[2][b][q];
        e[2][b][q] = d[2][b][q] - d[1][b][q];
        e[3][b][q] = d[1][b][q] - d[3][b][q];
      }
#pragma unroll
    for (int a = 0; a < 4; ++a) {
      int vv[4][4];  // [column][channel]
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        vv[0][q] = e[a][0][q] - e[a][2][q];
        vv[1][q] = e[a][1][q] + e[a][2][q];
        vv[2][q] = e[a][2][q] - e[a][1][q];
        vv[3][q] = e[a][1][q] - e[a][3][q];
      }
#pragma unroll
      for (int b = 0; b < 4; ++b) {
        __half2 p0 = __halves2half2(__int2half_rn(vv[b][0]), __int2half_rn(vv[b][1]));
        __half2 p1 = __halves2half2(__int2half_rn(vv[b][2]), __int2half_rn(vv[b][3]));
        uint2 o;
        o.x = *reinterpret_cast<uint32_t*>(&p0);
        o.y = *reinterpret_cast<uint32_t*>(&p1);
        *reinterpret_cast<uint2*>(v + ((long long)(a * 4 + b) * T + t) * Cp + c) = o;
      }
    }
  }
}

// M[xi][t][2K] (Ml in columns k, Mh in K + k) -> 4y = A^T (32 Mh + Ml) A -> int8
__global__ void i8w_output_kernel(const float* __restrict__ m, int8_t* __restrict__ y,
                                  const int32_t* __restrict__ bias,
                                  const float* __restrict__ scale, int relu, int K, long long T,
                                  int TH, int TW, int OH, int OW) {
  const long long total = T * K;
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < total;
       i += (long long)gridDim.x * blockDim.x) {
    const int k = (int)(i % K);
    const long long t = i / K;
    int m4[4][4];
#pragma unroll
    for (int xi = 0; xi < 16; ++xi) {
      const float* row = m + ((long long)xi * T + t) * 2 * K;
      // exact: both sums are integers below 2^24
      m4[xi / 4][xi % 4] = 32 * __float2int_rn(row[K + k]) + __float2int_rn(row[k]);
    }
    int e[2][4];
#pragma unroll
    for (int b = 0; b < 4; ++b) {
      e[0][b] = m4[0][b] + m4[1][b] + m4[2][b];
      e[1][b] = m4[1][b] - m4[2][b] - m4[3][b];
    }
    const int tw = (int)(t % TW);
    const long long r1 = t / TW;
    const int th = (int)(r1 % TH);
    const long long n = r1 / TH;
    const int bk = bias ? bias[k] : 0;
    const float sk = scale[k];
#pragma unroll
    for (int a = 0; a < 2; ++a) {
      const int y4[2] = {e[a][0] + e[a][1] + e[a][2], e[a][1] - e[a][2] - e[a][3]};
#pragma unroll
      for (int b = 0; b < 2; ++b) {
        const int oh = 2 * th + a, ow = 2 * tw + b;
        if (oh >= OH || ow >= OW) continue;
        const int tv = y4[b] / 4 + bk;  // 4y is a multiple of 4
        int q = __float2int_rn(__fmul_rn(__int2float_rn(tv), sk));
        q = q > 127 ? 127 : (q < -128 ? -128 : q);
        if (relu && q < 0) q = 0;
        y[((n * OH + oh) * OW + ow) * K + k] = (int8_t)q;
      }
    }
  }
}

}  // namespace

bool int8_wino_applicable(const gbconv_desc_s& d, const char** why) {
  if (d.R != 3 || d.S != 3 || d.stride != 1 || d.dil != 1 || d.groups != 1)
    return *why = "needs 3x3, stride 1, dilation 1, groups 1", false;
  if (d.C % 16 || d.K % 4) return *why = "needs C % 16 == 0 and K % 4 == 0", false;
  if (geo(d).Cp > MAXC) return *why = "more than 896 channels: the float sums would round", false;
  if (d.has_residual) return *why = "no residual in the int8 epilogue", false;
  if (geo(d).T >= (1LL << 31)) return *why = "too many tiles", false;
  return true;
}

size_t int8_wino_packed_bytes(const gbconv_desc_s& d) {
  return (size_t)16 * 2 * d.K * geo(d).Cp * 2;
}

size_t int8_wino_workspace_bytes(const gbconv_desc_s& d) {
  const Geo g = geo(d);
  const size_t v = ((size_t)16 * g.T * g.Cp * 2 + 255) / 256 * 256;
  return v + (size_t)16 * g.T * 2 * d.K * 4;
}

cudaError_t launch_pack_int8_wino(const gbconv_desc_s& d, const void* w, void* wpack,
                                  cudaStream_t st) {
  const Geo g = geo(d);
  i8w_filter_kernel<<<grid_for((long long)d.K * g.Cp), 256, 0, st>>>(
      static_cast<const int8_t*>(w), static_cast<__half*>(wpack), d.K, d.C, g.Cp);
  gb_count_launch();
  return cudaGetLastError();
}

cudaError_t launch_int8_wino(const gbconv_desc_s& d, const void* x, const void* wpack,
                             const int32_t* bias, void* y, void* ws, int* err,
                             unsigned long long wait_ns, cudaStream_t st) {
  const Geo g = geo(d);
  __half* v = static_cast<__half*>(ws);
  float* m = reinterpret_cast<float*>(static_cast<char*>(ws) +
                                      ((size_t)16 * g.T * g.Cp * 2 + 255) / 256 * 256);
  i8w_input_kernel<<<grid_for(g.T * (g.Cp / 4)), 256, 0, st>>>(
      static_cast<const int8_t*>(x), v, d.H, d.W, d.C, g.Cp, d.pad, g.TH, g.TW, g.T);
  gb_count_launch();
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const int n2 = 2 * d.K;
  e = launch_batched_gemm_tc(16, (int)g.T, n2, g.Cp, v, wpack, m, 0,
                             n2 <= 64 ? 64 : (n2 <= 128 ? 128 : 256), err, wait_ns, st);
  if (e != cudaSuccess) return e;
  i8w_output_kernel<<<grid_for(g.T * d.K), 256, 0, st>>>(
      m, static_cast<int8_t*>(y), bias, d.scale, d.act == CONV_ACT_RELU ? 1 : 0, d.K, g.T, g.TH,
      g.TW, d.OH, d.OW);
  gb_count_launch();
  return cudaGetLastError();
}
