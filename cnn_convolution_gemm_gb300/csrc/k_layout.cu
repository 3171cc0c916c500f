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

// Four consecutive pixels per thread when rows hold a multiple of four pixels
// and both tensors are 16-byte aligned: one 16-byte load per input plane
// (coalesced across the warp), C_OUT * 8 contiguous bytes stored as 16-byte
// vectors.  Grid-stride over the pixel quads, so every SM keeps several
// thousand bytes of loads in flight; the rounding is the same as above.
template <int C_OUT>
__global__ void nchw_f32_to_nhwc_bf16_quad_kernel(const float* __restrict__ x,
                                                  __nv_bfloat16* __restrict__ y, int C,
                                                  long long hw, long long quads) {
  gb::allow_dependents();
  for (long long q = blockIdx.x * (long long)blockDim.x + threadIdx.x; q < quads;
       q += (long long)gridDim.x * blockDim.x) {
    const long long p = q * 4;
    const long long n = p / hw;
    const float* src = x + n * C * hw + (p - n * hw);
    float v[C_OUT][4];
#pragma unroll
    for (int c = 0; c < C_OUT; ++c) {
      float4 f = make_float4(0.f, 0.f, 0.f, 0.f);
      if (c < C) f = __ldg(reinterpret_cast<const float4*>(src + c * hw));
      v[c][0] = f.x;
      v[c][1] = f.y;
      v[c][2] = f.z;
      v[c][3] = f.w;
    }
    uint32_t o[2 * C_OUT];  // pixel-major, channel pairs
#pragma unroll
    for (int px = 0; px < 4; ++px)
#pragma unroll
      for (int c = 0; c < C_OUT; c += 2) {
        __nv_bfloat162 b = __floats2bfloat162_rn(v[c][px], v[c + 1][px]);
        o[(px * C_OUT + c) / 2] = *reinterpret_cast<uint32_t*>(&b);
      }
    uint4* dst = reinterpret_cast<uint4*>(y + p * C_OUT);
#pragma unroll
    for (int i = 0; i < C_OUT / 2; ++i)
      dst[i] = make_uint4(o[4 * i], o[4 * i + 1], o[4 * i + 2], o[4 * i + 3]);
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

// 3x3 max pooling (ResNet's 3x3 / stride 2), same thread mapping as above with
// the window unrolled: the nine 16-byte loads of a thread are issued together
// (taps outside the image read as -inf), and the maximum is taken on the bf16
// pairs directly (a maximum of bf16 values is one of them, so no widening).
__global__ void maxpool3_nhwc_bf16_kernel(const __nv_bfloat16* __restrict__ x,
                                          __nv_bfloat16* __restrict__ y, int N, int C, int H,
                                          int W, int stride, int pad, int OH, int OW) {
  gb::allow_dependents();
  const int cv = C / 8;
  const int item = blockIdx.x * blockDim.x + threadIdx.x;
  if (item >= OW * cv) return;
  const int ow = item / cv, c8 = item - ow * cv;
  const uint4 ninf = make_uint4(0xFF80FF80u, 0xFF80FF80u, 0xFF80FF80u, 0xFF80FF80u);
  for (int row = blockIdx.y; row < N * OH; row += gridDim.y) {
    const int n = row / OH, oh = row - n * OH;
    uint4 v[9];
#pragma unroll
    for (int r = 0; r < 3; ++r) {
      const int ih = oh * stride - pad + r;
#pragma unroll
      for (int s = 0; s < 3; ++s) {
        const int iw = ow * stride - pad + s;
        v[r * 3 + s] = ninf;
        if (ih >= 0 && ih < H && iw >= 0 && iw < W)
          v[r * 3 + s] = __ldg(reinterpret_cast<const uint4*>(
              x + (((long long)n * H + ih) * W + iw) * C + c8 * 8));
      }
    }
    uint4 m = v[0];
    __nv_bfloat162* mb = reinterpret_cast<__nv_bfloat162*>(&m);
#pragma unroll
    for (int t = 1; t < 9; ++t) {
      const __nv_bfloat162* b = reinterpret_cast<const __nv_bfloat162*>(&v[t]);
#pragma unroll
      for (int j = 0; j < 4; ++j) mb[j] = __hmax2(mb[j], b[j]);
    }
    reinterpret_cast<uint4*>(y)[(long long)row * OW * cv + item] = m;
  }
}

// Global average pooling.  A block covers one image and 32 consecutive
// 8-channel vectors; its 8 warps take every 8th pixel (a warp reads 512
// contiguous bytes per pixel), each thread keeps fp32 sums of its 8 channels,
// and the 8 partial sums meet in shared memory, added in warp order.
constexpr int kPoolParts = 8;
__global__ void __launch_bounds__(32 * kPoolParts)
    avgpool_nhwc_bf16_kernel(const __nv_bfloat16* __restrict__ x, __nv_bfloat16* __restrict__ y,
                             int C, int HW, int groups_per_image) {
  __shared__ float4 part[kPoolParts][32][2];
  gb::allow_dependents();
  const int cv = C / 8;
  const int n = blockIdx.x / groups_per_image;
  const int c8 = (blockIdx.x - n * groups_per_image) * 32 + (threadIdx.x & 31);
  const int slice = threadIdx.x >> 5;
  float s[8] = {0, 0, 0, 0, 0, 0, 0, 0};
  if (c8 < cv) {
    const uint4* src = reinterpret_cast<const uint4*>(x + (long long)n * HW * C) + c8;
#pragma unroll 4
    for (int p = slice; p < HW; p += kPoolParts) {
      const uint4 v = __ldg(src + (long long)p * cv);
      const __nv_bfloat162* b = reinterpret_cast<const __nv_bfloat162*>(&v);
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float2 f = __bfloat1622float2(b[j]);
        s[2 * j] += f.x;
        s[2 * j + 1] += f.y;
      }
    }
  }
  part[slice][threadIdx.x & 31][0] = make_float4(s[0], s[1], s[2], s[3]);
  part[slice][threadIdx.x & 31][1] = make_float4(s[4], s[5], s[6], s[7]);
  __syncthreads();
  if (slice != 0 || c8 >= cv) return;
  float t[8] = {0, 0, 0, 0, 0, 0, 0, 0};
  for (int q = 0; q < kPoolParts; ++q) {
    const float4 a = part[q][threadIdx.x][0], b = part[q][threadIdx.x][1];
    t[0] += a.x; t[1] += a.y; t[2] += a.z; t[3] += a.w;
    t[4] += b.x; t[5] += b.y; t[6] += b.z; t[7] += b.w;
  }
  const float inv = 1.0f / (float)HW;
  uint4 o;
  __nv_bfloat162* ob = reinterpret_cast<__nv_bfloat162*>(&o);
#pragma unroll
  for (int j = 0; j < 4; ++j) ob[j] = __floats2bfloat162_rn(t[2 * j] * inv, t[2 * j + 1] * inv);
  *reinterpret_cast<uint4*>(y + (long long)n * C + c8 * 8) = o;
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
  const long long hw = (long long)H * W;
  if (W % 4 == 0 && C <= C_out && (C_out == 4 || C_out == 8) &&
      ((reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(y)) & 15) == 0) {
    const long long quads = (long long)N * hw / 4;
    const int grid = (int)std::min<long long>(gb_ceil_div_ll(quads, kBlock), 8LL * gb_num_sms());
    if (C_out == 4)
      nchw_f32_to_nhwc_bf16_quad_kernel<4><<<grid, kBlock, 0, st>>>(
          x, static_cast<__nv_bfloat16*>(y), C, hw, quads);
    else
      nchw_f32_to_nhwc_bf16_quad_kernel<8><<<grid, kBlock, 0, st>>>(
          x, static_cast<__nv_bfloat16*>(y), C, hw, quads);
    gb_count_launch();
    return cudaGetLastError();
  }
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
  if (k == 3)
    maxpool3_nhwc_bf16_kernel<<<grid, kBlock, 0, st>>>(static_cast<const __nv_bfloat16*>(x),
                                                       static_cast<__nv_bfloat16*>(y), N, C, H, W,
                                                       stride, pad, OH, OW);
  else
    maxpool_nhwc_bf16_kernel<<<grid, kBlock, 0, st>>>(
        static_cast<const __nv_bfloat16*>(x), static_cast<__nv_bfloat16*>(y), N, C, H, W, k,
        stride, pad, OH, OW);
  gb_count_launch();
  return cudaGetLastError();
}

cudaError_t launch_avgpool_nhwc_bf16(const void* x, void* y, int N, int C, int H, int W,
                                     cudaStream_t st) {
  const int groups = gb_ceil_div(C / 8, 32);
  if ((long long)N * groups >= (1LL << 31) || (long long)H * W >= (1LL << 31))
    return cudaErrorInvalidValue;
  avgpool_nhwc_bf16_kernel<<<N * groups, 32 * kPoolParts, 0, st>>>(
      static_cast<const __nv_bfloat16*>(x), static_cast<__nv_bfloat16*>(y), C, H * W, groups);
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
// Agreement of two outputs of the same convolution (Fast-Run's check of a
// candidate against the reference algorithm).  out[0] = max |a - b| and
// out[1] = max |b| as fp32 bit patterns (non-negative floats order like their
// bits, so an unsigned max is a float max); out[2] = elements of a that are
// not finite or, for int8, differ from b.
__global__ void compare_outputs_kernel(const void* __restrict__ a, const void* __restrict__ b,
                                       long long n, int dtype, unsigned* __restrict__ out) {
  unsigned md = 0, mb = 0, bad = 0;
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n;
       i += (long long)gridDim.x * blockDim.x) {
    float va, vb;
    if (dtype == CONV_BF16) {
      va = __bfloat162float(static_cast<const __nv_bfloat16*>(a)[i]);
      vb = __bfloat162float(static_cast<const __nv_bfloat16*>(b)[i]);
    } else if (dtype == CONV_F32) {
      va = static_cast<const float*>(a)[i];
      vb = static_cast<const float*>(b)[i];
    } else {
      va = (float)static_cast<const int8_t*>(a)[i];
      vb = (float)static_cast<const int8_t*>(b)[i];
      if (va != vb) ++bad;
    }
    const float dv = fabsf(va - vb);
    if (!(dv <= 3.0e38f)) {  // NaN or infinity
      ++bad;
      continue;
    }
    md = max(md, __float_as_uint(dv));
    if (fabsf(vb) <= 3.0e38f) mb = max(mb, __float_as_uint(fabsf(vb)));
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    md = max(md, __shfl_xor_sync(0xffffffffu, md, o));
    mb = max(mb, __shfl_xor_sync(0xffffffffu, mb, o));
    bad += __shfl_xor_sync(0xffffffffu, bad, o);
  }
  if ((threadIdx.x & 31) == 0) {
    atomicMax(out, md);
    atomicMax(out + 1, mb);
    if (bad) atomicAdd(out + 2, bad);
  }
}

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

cudaError_t launch_compare_outputs(const void* a, const void* b, long long n, int dtype,
                                   unsigned* out3, cudaStream_t st) {
  cudaError_t e = cudaMemsetAsync(out3, 0, 3 * sizeof(unsigned), st);
  if (e != cudaSuccess) return e;
  compare_outputs_kernel<<<grid_for(n), kBlock, 0, st>>>(a, b, n, dtype, out3);
  gb_count_launch();
  return cudaGetLastError();
}
