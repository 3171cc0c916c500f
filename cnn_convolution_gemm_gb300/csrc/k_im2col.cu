// Explicit (materialised) im2col + GEMM: the baseline the MegEngine report's
// "Im2col+MatMul" section improves on.  The im2col matrix [N*OH*OW][R*S*C]
// (each row the receptive field of one output pixel, zeros for padding) is
// written to the workspace, then multiplied by the weights with the same
// tcgen05 kernel, run as a 1x1 convolution over R*S*C input channels.  Kept as
// a Fast-Run candidate and as the comparator that measures what fusing the
// im2col into the operand load saves.
#include <cuda_bf16.h>

#include <algorithm>

#include "internal.h"

namespace {

// one 16-byte vector (8 channels) of one (pixel, tap) per thread
__global__ void im2col_kernel(const __nv_bfloat16* __restrict__ x, __nv_bfloat16* __restrict__ col,
                              int H, int W, int C, int S, int RS, int stride, int pad, int dil,
                              int OH, int OW, long long M) {
  const int cv = C / 8;
  const long long total = M * RS * cv;
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < total;
       i += (long long)gridDim.x * blockDim.x) {
    const int c8 = (int)(i % cv);
    long long t = i / cv;
    const int rs = (int)(t % RS);
    const long long m = t / RS;
    const int ow = (int)(m % OW);
    const long long nh = m / OW;
    const int oh = (int)(nh % OH);
    const long long n = nh / OH;
    const int ih = oh * stride - pad + (rs / S) * dil;
    const int iw = ow * stride - pad + (rs % S) * dil;
    uint4 v = make_uint4(0, 0, 0, 0);
    if (ih >= 0 && ih < H && iw >= 0 && iw < W)
      v = *reinterpret_cast<const uint4*>(x + ((n * H + ih) * W + iw) * C + c8 * 8);
    reinterpret_cast<uint4*>(col)[i] = v;
  }
}

gbconv_desc_s as_gemm(const gbconv_desc_s& d) {
  gbconv_desc_s g = d;  // 1x1 convolution over the im2col matrix
  g.N = 1;
  g.H = d.N * d.OH * d.OW;
  g.W = 1;
  g.C = d.R * d.S * d.C;
  g.R = g.S = 1;
  g.stride = 1;
  g.pad = 0;
  g.dil = 1;
  g.OH = g.H;
  g.OW = 1;
  return g;
}

}  // namespace

size_t im2col_workspace_bytes(const gbconv_desc_s& d) {
  return (size_t)d.N * d.OH * d.OW * d.R * d.S * d.C * 2;
}

size_t im2col_packed_bytes(const gbconv_desc_s& d) {
  return (size_t)d.K * gb_ceil_div(d.R * d.S * d.C, 64) * 64 * 2;
}

cudaError_t launch_pack_im2col_weights(const gbconv_desc_s& d, const void* w, void* wpack,
                                       cudaStream_t st) {
  // [K][R][S][C] is already [K][R*S*C]: pack it as the 1x1 weights of the GEMM
  return launch_pack_igemm_weights(as_gemm(d), w, wpack, st);
}

cudaError_t launch_im2col_gemm(const gbconv_desc_s& d, const void* x, const void* wpack,
                               const float* bias, const void* res, void* y, void* ws, int* err,
                               unsigned long long wait_ns, cudaStream_t st) {
  const long long M = (long long)d.N * d.OH * d.OW;
  const long long total = M * d.R * d.S * (d.C / 8);
  const int grid = (int)std::min<long long>(gb_ceil_div_ll(total, 256), 148LL * 32);
  im2col_kernel<<<grid, 256, 0, st>>>(static_cast<const __nv_bfloat16*>(x),
                                      static_cast<__nv_bfloat16*>(ws), d.H, d.W, d.C, d.S,
                                      d.R * d.S, d.stride, d.pad, d.dil, d.OH, d.OW, M);
  gb_count_launch();
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const gbconv_desc_s g = as_gemm(d);
  const int bn = d.K > 128 ? 256 : (d.K > 64 ? 128 : 64);
  return launch_igemm_bf16(g, bn, ws, wpack, bias, res, y, err, wait_ns, st);
}
