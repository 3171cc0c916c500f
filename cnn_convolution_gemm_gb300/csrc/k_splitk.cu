// Split-K completion for the bf16 implicit GEMM: when a layer's output tiles
// fill only a fraction of the SMs but its reduction is long (a fully connected
// layer run as a 1x1 convolution, the 7x7 stages of a ResNet at small batch),
// the GEMM cuts the reduction into ksplit ranges and writes each range's fp32
// products to part[ksplit][M][K]; this kernel sums them and applies the layer's
// epilogue (the MegEngine report's Im2col+MatMul with the reduction split, the
// Momenta talk's bias / residual / activation fused after the product).
#include <cuda_bf16.h>

#include <algorithm>

#include "internal.h"

namespace {

constexpr int kBlock = 256;

// One thread per 8 consecutive output channels of one pixel (K % 8 == 0, so a
// vector never crosses a row): ksplit pairs of 16-byte partial loads, summed in
// split order, then + bias, + residual, activation, rounded to nearest bf16.
__global__ void splitk_reduce_bf16_kernel(const float4* __restrict__ part, int ksplit,
                                          long long vecs, int K, const float* __restrict__ bias,
                                          const uint4* __restrict__ res, uint4* __restrict__ y,
                                          int act) {
  const long long plane = vecs * 2;  // float4s per split range
  for (long long v = blockIdx.x * (long long)blockDim.x + threadIdx.x; v < vecs;
       v += (long long)gridDim.x * blockDim.x) {
    float a[8];
    {
      const float4 p0 = __ldg(part + 2 * v), p1 = __ldg(part + 2 * v + 1);
      a[0] = p0.x; a[1] = p0.y; a[2] = p0.z; a[3] = p0.w;
      a[4] = p1.x; a[5] = p1.y; a[6] = p1.z; a[7] = p1.w;
    }
    for (int s = 1; s < ksplit; ++s) {
      const float4 p0 = __ldg(part + s * plane + 2 * v), p1 = __ldg(part + s * plane + 2 * v + 1);
      a[0] += p0.x; a[1] += p0.y; a[2] += p0.z; a[3] += p0.w;
      a[4] += p1.x; a[5] += p1.y; a[6] += p1.z; a[7] += p1.w;
    }
    if (bias) {
      const int k = (int)((v * 8) % K);
#pragma unroll
      for (int j = 0; j < 8; ++j) a[j] += __ldg(bias + k + j);
    }
    if (res) {
      const uint4 r = __ldg(res + v);
      const __nv_bfloat162* rb = reinterpret_cast<const __nv_bfloat162*>(&r);
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float2 f = __bfloat1622float2(rb[j]);
        a[2 * j] += f.x;
        a[2 * j + 1] += f.y;
      }
    }
    if (act != CONV_ACT_NONE) {
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        a[j] = fmaxf(a[j], 0.f);
        if (act == CONV_ACT_RELU6) a[j] = fminf(a[j], 6.f);
      }
    }
    uint4 o;
    __nv_bfloat162* ob = reinterpret_cast<__nv_bfloat162*>(&o);
#pragma unroll
    for (int j = 0; j < 4; ++j) ob[j] = __floats2bfloat162_rn(a[2 * j], a[2 * j + 1]);
    y[v] = o;
  }
}

}  // namespace

cudaError_t launch_splitk_reduce_bf16(const gbconv_desc_s& d, int ksplit, const void* part,
                                      const float* bias, const void* res, void* y,
                                      cudaStream_t st) {
  if (ksplit < 1 || d.K % 8) return cudaErrorInvalidValue;
  const long long vecs = (long long)d.N * d.OH * d.OW * (d.K / 8);
  const int grid = (int)std::min<long long>(gb_ceil_div_ll(vecs, kBlock), 8LL * gb_num_sms());
  splitk_reduce_bf16_kernel<<<grid, kBlock, 0, st>>>(
      static_cast<const float4*>(part), ksplit, vecs, d.K, bias, static_cast<const uint4*>(res),
      static_cast<uint4*>(y), d.act);
  gb_count_launch();
  return cudaGetLastError();
}
