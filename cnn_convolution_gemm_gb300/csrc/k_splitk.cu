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
#include "ptx.cuh"

namespace {

constexpr int kBlock = 128;

// One thread per 4 consecutive output channels of one pixel (K % 8 == 0, so a
// vector never crosses a row; small outputs such as a batch's FC logits still
// spread over the SMs): ksplit 16-byte partial loads summed in split order,
// then + bias, + residual, activation, rounded to nearest bf16.
__global__ void splitk_reduce_bf16_kernel(const float4* __restrict__ part, int ksplit,
                                          long long vecs, int K, const float* __restrict__ bias,
                                          const uint2* __restrict__ res, uint2* __restrict__ y,
                                          int act) {
  gb::allow_dependents();  // the next layer's GEMM sets up meanwhile
  for (long long v = blockIdx.x * (long long)blockDim.x + threadIdx.x; v < vecs;
       v += (long long)gridDim.x * blockDim.x) {
    float4 a = __ldg(part + v);
#pragma unroll 4
    for (int s = 1; s < ksplit; ++s) {
      const float4 q = __ldg(part + s * vecs + v);
      a.x += q.x;
      a.y += q.y;
      a.z += q.z;
      a.w += q.w;
    }
    if (bias) {
      const int k = (int)((v * 4) % K);
      a.x += __ldg(bias + k);
      a.y += __ldg(bias + k + 1);
      a.z += __ldg(bias + k + 2);
      a.w += __ldg(bias + k + 3);
    }
    if (res) {
      const uint2 r = __ldg(res + v);
      const float2 r0 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&r.x));
      const float2 r1 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&r.y));
      a.x += r0.x;
      a.y += r0.y;
      a.z += r1.x;
      a.w += r1.y;
    }
    if (act != CONV_ACT_NONE) {
      const float hi = act == CONV_ACT_RELU6 ? 6.f : INFINITY;
      a.x = fminf(fmaxf(a.x, 0.f), hi);
      a.y = fminf(fmaxf(a.y, 0.f), hi);
      a.z = fminf(fmaxf(a.z, 0.f), hi);
      a.w = fminf(fmaxf(a.w, 0.f), hi);
    }
    __nv_bfloat162 o0 = __floats2bfloat162_rn(a.x, a.y), o1 = __floats2bfloat162_rn(a.z, a.w);
    y[v] = make_uint2(*reinterpret_cast<uint32_t*>(&o0), *reinterpret_cast<uint32_t*>(&o1));
  }
}

}  // namespace

cudaError_t launch_splitk_reduce_bf16(const gbconv_desc_s& d, int ksplit, const void* part,
                                      const float* bias, const void* res, void* y,
                                      cudaStream_t st) {
  if (ksplit < 1 || d.K % 8) return cudaErrorInvalidValue;
  const long long vecs = (long long)d.N * d.OH * d.OW * (d.K / 4);
  const int grid = (int)std::min<long long>(gb_ceil_div_ll(vecs, kBlock), 16LL * gb_num_sms());
  splitk_reduce_bf16_kernel<<<grid, kBlock, 0, st>>>(
      static_cast<const float4*>(part), ksplit, vecs, d.K, bias, static_cast<const uint2*>(res),
      static_cast<uint2*>(y), d.act);
  gb_count_launch();
  return cudaGetLastError();
}
