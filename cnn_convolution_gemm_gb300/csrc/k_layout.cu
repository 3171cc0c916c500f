// Layout conversion (the MegEngine report's "Inference Layout": NCHW at the
// boundary, a channel-innermost layout with the channel axis padded to the
// vector width on the device), pooling for the ResNet-50 forward pass, and a
// deterministic random fill for Fast-Run scratch tensors.
#include <cuda_bf16.h>

#include <algorithm>

#include "internal.h"
#include "ptx.cuh"

namespace {

constexpr int kBlock = 256;

int grid_for(long long work) {
  return (int)std::min<long long>(gb_ceil_div_ll(work, kBlock), 148LL * 32);
}

// One thread per output pixel: blockIdx.y walks the image rows (n, h), the
// threads of a block the columns w, so no index needs a division.  A thread
// reads C strided values (coalesced across the warp along w) and writes C_out
// contiguous bf16 values (one 8-byte store when C_out == 4).
__global__ void nchw_f32_to_nhwc_bf16_kernel(const float* __restrict__ x,
                                             __nv_bfloat16* __restrict__ y, int N, int C, int H,
                                             int W, int C_out) {
  const int w = blockIdx.x * blockDim.x + threadIdx.x;
  if (w >= W) return;
  const long long hw = (long long)H * W;
  for (int nh = blockIdx.y; nh < N * H; nh += gridDim.y) {
    const int n = nh / H, h = nh - n * H;
    const float* src = x + (long long)n * C * hw + (long long)h * W + w;
    __nv_bfloat16* dst = y + ((long long)nh * W + w) * C_out;
    if (C_out == 4) {
      float v[4];
#pragma unroll
      for (int c = 0; c < 4; ++c) v[c] = c < C ? __ldg(src + c * hw) : 0.f;
      __nv_bfloat162 lo = __floats2bfloat162_rn(v[0], v[1]), hi = __floats2bfloat162_rn(v[2], v[3]);
      *reinterpret_cast<uint2*>(dst) =
          make_uint2(*reinterpret_cast<uint32_t*>(&lo), *reinterpret_cast<uint32_t*>(&hi));
      continue;
    }
    int c = 0;
    for (; c + 1 < C_out; c += 2) {
      const float a = c < C ? __ldg(src + c * hw) : 0.f;
      const float b = c + 1 < C ? __ldg(src + (c + 1) * hw) : 0.f;
      *reinterpret_cast<__nv_bfloat162*>(dst + c) = __floats2bfloat162_rn(a, b);
    }
    if (c < C_out) dst[c] = __float2bfloat16_rn(c < C ? __ldg(src + c * hw) : 0.f);
  }
}

__global__ void nhwc_bf16_to_nchw_f32_kernel(const __nv_bfloat16* __restrict__ x,
                                             float* __restrict__ y, int N, int C, int H, int W,
                                             int C_in) {
  const long long total = (long long)N * C * H * W;
  const long long hw = (long long)H * W;
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < total;
       i += (long long)gridDim.x * blockDim.x) {
    const long long p = i % hw;
    const long long c = (i / hw) % C;
    const long long n = i / (hw * C);
    y[i] = __bfloat162float(x[(n * hw + p) * C_in + c]);
  }
}

// Max pooling, NHWC bf16, 8 channels (16 bytes) per thread: blockIdx.y walks
// the output rows (n, oh), the threads of a block x cover (ow, 8-channel group)
// of the row with ow outermost, so a warp reads contiguous pixels.
__global__ void maxpool_nhwc_bf16_kernel(const __nv_bfloat16* __restrict__ x,
                                         __nv_bfloat16* __restrict__ y, int N, int C, int H,
                                         int W, int k, int stride, int pad, int OH, int OW) {
  const int cv = C / 8;
  const int item = blockIdx.x * blockDim.x + threadIdx.x;
  if (item >= OW * cv) return;
  const int ow = item / cv, c8 = item - ow * cv;
  for (int row = blockIdx.y; row < N * OH; row += gridDim.y) {
    const int n = row / OH, oh = row - n * OH;
    const long long i = (long long)row * OW * cv + item;  // output vector index
    float m[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) m[j] = -INFINITY;
    for (int r = 0; r < k; ++r) {
      const int ih = oh * stride - pad + r;
      if (ih < 0 || ih >= H) continue;
      for (int s = 0; s < k; ++s) {
        const int iw = ow * stride - pad + s;
        if (iw < 0 || iw >= W) continue;
        const uint4 v =
            *reinterpret_cast<const uint4*>(x + (((long long)n * H + ih) * W + iw) * C + c8 * 8);
        const __nv_bfloat162* b = reinterpret_cast<const __nv_bfloat162*>(&v);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const float2 f = __bfloat1622float2(b[j]);
          m[2 * j] = fmaxf(m[2 * j], f.x);
          m[2 * j + 1] = fmaxf(m[2 * j + 1], f.y);
        }
      }
    }
    uint4 o;
    __nv_bfloat162* ob = reinterpret_cast<__nv_bfloat162*>(&o);
#pragma unroll
    for (int j = 0; j < 4; ++j) ob[j] = __floats2bfloat162_rn(m[2 * j], m[2 * j + 1]);
    *reinterpret_cast<uint4*>(y + i * 8) = o;
  }
}

// Global average pooling: one thread per (n, 8-channel vector), fp32 sum.
__global__ void avgpool_nhwc_bf16_kernel(const __nv_bfloat16* __restrict__ x,
                                         __nv_bfloat16* __restrict__ y, int N, int C, int HW) {
  const int cv = C / 8;
  const long long total = (long long)N * cv;
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < total;
       i += (long long)gridDim.x * blockDim.x) {
    const int c8 = (int)(i % cv);
    const long long n = i / cv;
    float s[8] = {0, 0, 0, 0, 0, 0, 0, 0};
    for (int p = 0; p < HW; ++p) {
      const uint4 v = *reinterpret_cast<const uint4*>(x + (n * HW + p) * C + c8 * 8);
      const __nv_bfloat162* b = reinterpret_cast<const __nv_bfloat162*>(&v);
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float2 f = __bfloat1622float2(b[j]);
        s[2 * j] += f.x;
        s[2 * j + 1] += f.y;
      }
    }
    const float inv = 1.0f / (float)HW;
    uint4 o;
    __nv_bfloat162* ob = reinterpret_cast<__nv_bfloat162*>(&o);
#pragma unroll
    for (int j = 0; j < 4; ++j) ob[j] = __floats2bfloat162_rn(s[2 * j] * inv, s[2 * j + 1] * inv);
    *reinterpret_cast<uint4*>(y + n * C + c8 * 8) = o;
  }
}

__device__ __forceinline__ uint32_t hash32(uint32_t v) {
  v ^= v >> 16;
  v *= 0x7feb352dU;
  v ^= v >> 15;
  v *= 0x846ca68bU;
  v ^= v >> 16;
  return v;
}

// Values in [-1, 1) for float types, [-64, 63] for int8.
__global__ void fill_random_kernel(uint8_t* p, long long n, int elem_bytes, uint32_t seed) {
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n;
       i += (long long)gridDim.x * blockDim.x) {
    const uint32_t h = hash32((uint32_t)i * 2654435761u ^ seed);
    if (elem_bytes == 4) {
      reinterpret_cast<float*>(p)[i] = (float)(h >> 8) * (1.0f / 8388608.0f) - 1.0f;
    } else if (elem_bytes == 2) {
      reinterpret_cast<__nv_bfloat16*>(p)[i] =
          __float2bfloat16_rn((float)(h >> 8) * (1.0f / 8388608.0f) - 1.0f);
    } else {
      reinterpret_cast<int8_t*>(p)[i] = (int8_t)((int)(h >> 25) - 64);
    }
  }
}

}  // namespace

cudaError_t launch_nchw_f32_to_nhwc_bf16(const float* x, void* y, int N, int C, int H, int W,
                                         int C_out, cudaStream_t st) {
  if ((long long)N * H >= (1LL << 31)) return cudaErrorInvalidValue;
  const dim3 grid((unsigned)gb_ceil_div(W, 128), (unsigned)std::min(N * H, 65535));
  nchw_f32_to_nhwc_bf16_kernel<<<grid, 128, 0, st>>>(x, static_cast<__nv_bfloat16*>(y), N, C, H,
                                                     W, C_out);
  gb_count_launch();
  return cudaGetLastError();
}

cudaError_t launch_nhwc_bf16_to_nchw_f32(const void* x, float* y, int N, int C, int H, int W,
                                         int C_in, cudaStream_t st) {
  nhwc_bf16_to_nchw_f32_kernel<<<grid_for((long long)N * C * H * W), kBlock, 0, st>>>(
      static_cast<const __nv_bfloat16*>(x), y, N, C, H, W, C_in);
  gb_count_launch();
  return cudaGetLastError();
}

cudaError_t launch_maxpool_nhwc_bf16(const void* x, void* y, int N, int C, int H, int W, int k,
                                     int stride, int pad, cudaStream_t st) {
  const int OH = (H + 2 * pad - k) / stride + 1, OW = (W + 2 * pad - k) / stride + 1;
  if ((long long)N * OH >= (1LL << 31) || (long long)OW * (C / 8) >= (1LL << 31))
    return cudaErrorInvalidValue;
  const dim3 grid((unsigned)gb_ceil_div(OW * (C / 8), kBlock), (unsigned)std::min(N * OH, 65535));
  maxpool_nhwc_bf16_kernel<<<grid, kBlock, 0, st>>>(
      static_cast<const __nv_bfloat16*>(x), static_cast<__nv_bfloat16*>(y), N, C, H, W, k, stride,
      pad, OH, OW);
  gb_count_launch();
  return cudaGetLastError();
}

cudaError_t launch_avgpool_nhwc_bf16(const void* x, void* y, int N, int C, int H, int W,
                                     cudaStream_t st) {
  avgpool_nhwc_bf16_kernel<<<grid_for((long long)N * (C / 8)), kBlock, 0, st>>>(
      static_cast<const __nv_bfloat16*>(x), static_cast<__nv_bfloat16*>(y), N, C, H * W);
  gb_count_launch();
  return cudaGetLastError();
}

cudaError_t launch_fill_random(void* p, size_t bytes, int elem_bytes, uint32_t seed,
                               cudaStream_t st) {
  const long long n = (long long)(bytes / elem_bytes);
  fill_random_kernel<<<grid_for(n), kBlock, 0, st>>>(static_cast<uint8_t*>(p), n, elem_bytes,
                                                     seed);
  gb_count_launch();
  return cudaGetLastError();
}

namespace {
// NCHW int8 [N][C][H][W] <-> NC32HW32 int8 [N][ceil(C/32)][H][W][32]; one byte
// per thread, indexed by the NC32HW32 element (channels past C read as 0 going
// in, are skipped going out)
__global__ void nc32_convert_kernel(const int8_t* __restrict__ x, int8_t* __restrict__ y, int N,
                                    int C, long long HW, int to_nc32) {
  const int CB = (C + 31) / 32;
  const long long total = (long long)N * CB * HW * 32;
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < total;
       i += (long long)gridDim.x * blockDim.x) {
    const int cl = (int)(i % 32);
    const long long t = i / 32;
    const long long hw = t % HW;
    const long long nb = t / HW;
    const int cb = (int)(nb % CB);
    const long long n = nb / CB;
    const int c = cb * 32 + cl;
    const long long nchw = (n * C + c) * HW + hw;
    if (to_nc32)
      y[i] = c < C ? x[nchw] : (int8_t)0;
    else if (c < C)
      y[nchw] = x[i];
  }
}
}  // namespace

cudaError_t launch_nc32_convert(const void* x, void* y, int N, int C, int H, int W, int to_nc32,
                                cudaStream_t st) {
  const long long total = (long long)N * ((C + 31) / 32) * H * W * 32;
  const int grid = (int)std::min<long long>((total + 255) / 256, 152LL * 32);
  nc32_convert_kernel<<<grid, 256, 0, st>>>(static_cast<const int8_t*>(x),
                                            static_cast<int8_t*>(y), N, C, (long long)H * W,
                                            to_nc32);
  gb_count_launch();
  return cudaGetLastError();
}

namespace {
// One thread waits on an mbarrier that nothing arrives at, through the bounded
// wait every tcgen05 kernel uses: the wait runs out after limit_ns, the thread
// records the timeout in the device error word, and the kernel returns.
__global__ void selftest_wait_timeout_kernel(int* err, unsigned long long limit_ns) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    gb::mbar_init(&bar, 1);
    gb::fence_barrier_init();
    gb::mbar_wait_bounded(&bar, 0, limit_ns, err);
  }
}
}  // namespace

cudaError_t launch_selftest_wait_timeout(int* err, unsigned long long limit_ns, cudaStream_t st) {
  selftest_wait_timeout_kernel<<<1, 32, 0, st>>>(err, limit_ns);
  gb_count_launch();
  return cudaGetLastError();
}
