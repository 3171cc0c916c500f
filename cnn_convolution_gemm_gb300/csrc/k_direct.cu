// Direct convolution on CUDA cores: the nested loop of the razer666.cn post
// "卷积总结" (section "最原始的卷积实现") with stride, dilation, padding and
// groups, one thread per output element.  It is the general fallback and a
// Fast-Run candidate ("Direct" in the MegEngine report's "Fast-Run" section);
// it covers every shape, layout and dtype the descriptor allows.
#include <cuda_bf16.h>

#include <algorithm>

#include "internal.h"

namespace {

struct DirectParams {
  int N, C, H, W, K, R, S, stride, pad, dil, OH, OW, Cg, Kg;
  int act;
  int nhwc;
  int shuf;  // > 1: input channel c is read from (c mod shuf) * (C / shuf) + c div shuf
};

__device__ __forceinline__ int in_channel(const DirectParams& p, int c) {
  return p.shuf > 1 ? (c % p.shuf) * (p.C / p.shuf) + c / p.shuf : c;
}

__device__ __forceinline__ float to_f(float v) { return v; }
__device__ __forceinline__ float to_f(__nv_bfloat16 v) { return __bfloat162float(v); }
template <typename T>
__device__ __forceinline__ T from_f(float v);
template <>
__device__ __forceinline__ float from_f<float>(float v) {
  return v;
}
template <>
__device__ __forceinline__ __nv_bfloat16 from_f<__nv_bfloat16>(float v) {
  return __float2bfloat16_rn(v);
}

// p.nhwc: 1 NHWC, 0 NCHW, 2 NC32HW32 (int8 only)
__device__ __forceinline__ void decompose(long long i, const DirectParams& p, int& n, int& k,
                                          int& oh, int& ow) {
  if (p.nhwc == 2) {
    const int klo = (int)(i % 32);
    i /= 32;
    ow = (int)(i % p.OW);
    i /= p.OW;
    oh = (int)(i % p.OH);
    i /= p.OH;
    k = (int)(i % (p.K / 32)) * 32 + klo;
    n = (int)(i / (p.K / 32));
  } else if (p.nhwc) {
    k = (int)(i % p.K);
    i /= p.K;
    ow = (int)(i % p.OW);
    i /= p.OW;
    oh = (int)(i % p.OH);
    n = (int)(i / p.OH);
  } else {
    ow = (int)(i % p.OW);
    i /= p.OW;
    oh = (int)(i % p.OH);
    i /= p.OH;
    k = (int)(i % p.K);
    n = (int)(i / p.K);
  }
}

template <typename T>
__global__ void direct_conv_kernel(DirectParams p, const T* __restrict__ x,
                                   const T* __restrict__ w, const float* __restrict__ bias,
                                   const T* __restrict__ res, T* __restrict__ y) {
  const long long total = (long long)p.N * p.K * p.OH * p.OW;
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < total;
       i += (long long)gridDim.x * blockDim.x) {
    int n, k, oh, ow;
    decompose(i, p, n, k, oh, ow);
    const int g = k / p.Kg;
    float acc = 0.f;
    for (int r = 0; r < p.R; ++r) {
      const int ih = oh * p.stride - p.pad + r * p.dil;
      if (ih < 0 || ih >= p.H) continue;
      for (int s = 0; s < p.S; ++s) {
        const int iw = ow * p.stride - p.pad + s * p.dil;
        if (iw < 0 || iw >= p.W) continue;
        for (int cc = 0; cc < p.Cg; ++cc) {
          const int c = in_channel(p, g * p.Cg + cc);
          float xv, wv;
          if (p.nhwc) {
            xv = to_f(x[(((long long)n * p.H + ih) * p.W + iw) * p.C + c]);
            wv = to_f(w[(((long long)k * p.R + r) * p.S + s) * p.Cg + cc]);
          } else {
            xv = to_f(x[(((long long)n * p.C + c) * p.H + ih) * p.W + iw]);
            wv = to_f(w[(((long long)k * p.Cg + cc) * p.R + r) * p.S + s]);
          }
          acc = fmaf(xv, wv, acc);
        }
      }
    }
    if (bias) acc += bias[k];
    if (res) acc += to_f(res[i]);
    if (p.act == 1) acc = fmaxf(acc, 0.f);
    if (p.act == 2) acc = fminf(fmaxf(acc, 0.f), 6.f);
    y[i] = from_f<T>(acc);
  }
}

// int8: exact int32 accumulate, then the fp32 requant
// q = clamp(rne(fp32(acc + bias) * scale[k]), -128, 127), then ReLU.
__global__ void direct_conv_int8_kernel(DirectParams p, const int8_t* __restrict__ x,
                                        const int8_t* __restrict__ w,
                                        const int32_t* __restrict__ bias,
                                        const float* __restrict__ scale,
                                        int8_t* __restrict__ y) {
  const long long total = (long long)p.N * p.K * p.OH * p.OW;
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < total;
       i += (long long)gridDim.x * blockDim.x) {
    int n, k, oh, ow;
    decompose(i, p, n, k, oh, ow);
    const int g = k / p.Kg;
    int acc = 0;
    for (int r = 0; r < p.R; ++r) {
      const int ih = oh * p.stride - p.pad + r * p.dil;
      if (ih < 0 || ih >= p.H) continue;
      for (int s = 0; s < p.S; ++s) {
        const int iw = ow * p.stride - p.pad + s * p.dil;
        if (iw < 0 || iw >= p.W) continue;
        for (int cc = 0; cc < p.Cg; ++cc) {
          const int c = in_channel(p, g * p.Cg + cc);
          const long long xi =
              p.nhwc == 2 ? ((((long long)n * (p.C / 32) + c / 32) * p.H + ih) * p.W + iw) * 32 +
                                (c & 31)
                          : (((long long)n * p.H + ih) * p.W + iw) * p.C + c;
          acc += (int)x[xi] * (int)w[(((long long)k * p.R + r) * p.S + s) * p.Cg + cc];
        }
      }
    }
    if (bias) acc += bias[k];
    const float q = __fmul_rn(__int2float_rn(acc), scale[k]);
    int v = __float2int_rn(q);
    v = v > 127 ? 127 : (v < -128 ? -128 : v);
    if (p.act == 1 && v < 0) v = 0;
    y[i] = (int8_t)v;
  }
}

}  // namespace

cudaError_t launch_direct(const gbconv_desc_s& d, const void* x, const void* w, const void* bias,
                          const void* res, void* y, cudaStream_t st) {
  DirectParams p{d.N, d.C, d.H, d.W, d.K, d.R, d.S, d.stride, d.pad, d.dil, d.OH, d.OW,
                 d.C / d.groups, d.K / d.groups, d.act,
                 d.layout == CONV_NHWC ? 1 : (d.layout == CONV_NC32HW32 ? 2 : 0),
                 d.shuffle_groups};
  const long long total = (long long)d.N * d.K * d.OH * d.OW;
  const int block = 256;
  const int grid = (int)std::min<long long>(gb_ceil_div_ll(total, block), 148LL * 64);
  switch (d.dtype) {
    case CONV_BF16:
      direct_conv_kernel<__nv_bfloat16><<<grid, block, 0, st>>>(
          p, static_cast<const __nv_bfloat16*>(x), static_cast<const __nv_bfloat16*>(w),
          static_cast<const float*>(bias), static_cast<const __nv_bfloat16*>(res),
          static_cast<__nv_bfloat16*>(y));
      gb_count_launch();
      break;
    case CONV_F32:
      direct_conv_kernel<float><<<grid, block, 0, st>>>(
          p, static_cast<const float*>(x), static_cast<const float*>(w),
          static_cast<const float*>(bias), static_cast<const float*>(res),
          static_cast<float*>(y));
      gb_count_launch();
      break;
    case CONV_INT8:
      direct_conv_int8_kernel<<<grid, block, 0, st>>>(
          p, static_cast<const int8_t*>(x), static_cast<const int8_t*>(w),
          static_cast<const int32_t*>(bias), d.scale, static_cast<int8_t*>(y));
      gb_count_launch();
      break;
  }
  return cudaGetLastError();
}
