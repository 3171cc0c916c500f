// int8 quantized convolution: exact int32 accumulation, fused bias + per-channel
// fp32 requantisation + ReLU (the 96x.com.cn MegEngine Beta report, section
// "推理：高效原生 int8 实现": native int8 inference on the tensor cores).
//
// sm_103a exposes no int8 kind of tcgen05.mma, so the contraction runs on the
// warp-level tensor-core instruction mma.sync.m16n8k32 with s8 operands and
// s32 accumulators, which is exact for every shape here (the largest
// accumulator, 512 channels x 9 taps x 127^2 = 74.3M, is far below 2^31).
//
// Implicit GEMM as in the bf16 kernel: M = N*OH*OW output pixels, N = K,
// reduction over (r, s, 64-channel block).  A 128 x 64-byte im2col tile and a
// BN x 64-byte weight tile are copied per stage with cp.async (zero-fill for
// padding and channel tails), 4 stages deep; fragments come from ldmatrix on a
// 16-byte-chunk XOR swizzle (conflict-free for 64-byte rows).
//
// Epilogue per output (n, k):  t = acc + bias[k];
//   q = clamp(rne(fp32(t) * scale[k]), -128, 127);  ReLU -> max(q, 0).
// fp32 conversion and multiply are round-to-nearest-even (__int2float_rn,
// __fmul_rn), the integer rounding is half-to-even (__float2int_rn).
#include <stdint.h>

#include <algorithm>

#include "internal.h"

namespace {

constexpr int BM = 128, BK = 64, STAGES = 4, THREADS = 256;

struct I8Params {
  int N, H, W, C, K, R, S, stride, pad, dil, OH, OW;
  int cblocks, kiters, Kw;
  long long M;
  int relu;
  const int32_t* bias;
  const float* scale;
};

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, bool valid) {
  const int n = valid ? 16 : 0;
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(n)
               : "memory");
}
__device__ __forceinline__ void cp_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                        uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

__device__ __forceinline__ void mma_s8(int32_t (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                       uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k32.row.col.s32.s8.s8.s32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
      "{%8, %9}, {%0, %1, %2, %3};"
      : "+r"(d[0]), "+r"(d[1]), "+r"(d[2]), "+r"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// byte offset of 16-byte chunk `c` of row `r` in a tile of 64-byte rows
__device__ __forceinline__ uint32_t swz(int r, int c) {
  return (uint32_t)(r * 64 + ((c ^ ((r >> 1) & 3)) << 4));
}

__device__ __forceinline__ int8_t requant(int32_t acc, int32_t b, float sc, int relu) {
  const float q = __fmul_rn(__int2float_rn(acc + b), sc);
  int v = __float2int_rn(q);
  v = v > 127 ? 127 : (v < -128 ? -128 : v);
  if (relu && v < 0) v = 0;
  return (int8_t)v;
}

template <int BN>
__global__ void __launch_bounds__(THREADS)
    igemm_int8_kernel(const I8Params p, const int8_t* __restrict__ x,
                      const int8_t* __restrict__ wp, int8_t* __restrict__ y) {
  constexpr int A_BYTES = BM * BK, B_BYTES = BN * BK, STAGE = A_BYTES + B_BYTES;
  constexpr int WN = BN / 2;       // warp tile N (warps: 4 along M x 2 along N)
  constexpr int NT = WN / 8;       // n8 tiles per warp
  extern __shared__ __align__(128) uint8_t smem[];
  const uint32_t sbase = (uint32_t)__cvta_generic_to_shared(smem);

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int wm = warp & 3, wn = warp >> 2;
  const long long m0 = (long long)blockIdx.x * BM;
  const int n0 = blockIdx.y * BN;
  const int ohow = p.OH * p.OW;

  // per-thread A rows: 512 chunks per stage, 2 per thread
  int a_row[2], a_chunk[2], a_img[2], a_ih0[2], a_iw0[2];
  bool a_ok[2];
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const int q = tid + i * THREADS;
    a_row[i] = q >> 2;
    a_chunk[i] = q & 3;
    const long long m = m0 + a_row[i];
    a_ok[i] = m < p.M;
    const long long mm = a_ok[i] ? m : 0;
    a_img[i] = (int)(mm / ohow);
    const int rem = (int)(mm % ohow);
    a_ih0[i] = (rem / p.OW) * p.stride - p.pad;
    a_iw0[i] = (rem % p.OW) * p.stride - p.pad;
  }

  auto load_stage = [&](int it, int slot) {
    const int cb = it % p.cblocks;
    const int rs = it / p.cblocks;
    const int r = rs / p.S, s = rs % p.S;
    const uint32_t sa = sbase + slot * STAGE, sb = sa + A_BYTES;
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const int ih = a_ih0[i] + r * p.dil, iw = a_iw0[i] + s * p.dil;
      const int c = cb * BK + a_chunk[i] * 16;
      const bool ok = a_ok[i] && ih >= 0 && ih < p.H && iw >= 0 && iw < p.W && c < p.C;
      const int8_t* src =
          ok ? x + (((size_t)a_img[i] * p.H + ih) * p.W + iw) * p.C + c : x;
      cp_async16(sa + swz(a_row[i], a_chunk[i]), src, ok);
    }
#pragma unroll
    for (int i = 0; i < (BN * 4) / THREADS; ++i) {
      const int q = tid + i * THREADS;
      const int row = q >> 2, ch = q & 3;
      const bool ok = n0 + row < p.K;
      const int8_t* src = ok ? wp + (size_t)(n0 + row) * p.Kw + rs * (p.cblocks * BK) + cb * BK +
                                   ch * 16
                             : wp;
      cp_async16(sb + swz(row, ch), src, ok);
    }
  };

  int32_t acc[2][NT][4];
#pragma unroll
  for (int i = 0; i < 2; ++i)
#pragma unroll
    for (int j = 0; j < NT; ++j)
#pragma unroll
      for (int k = 0; k < 4; ++k) acc[i][j][k] = 0;

#pragma unroll
  for (int st = 0; st < STAGES - 1; ++st) {
    if (st < p.kiters) load_stage(st, st);
    cp_commit();
  }

  for (int it = 0; it < p.kiters; ++it) {
    cp_wait<STAGES - 2>();
    __syncthreads();
    const int nxt = it + STAGES - 1;
    if (nxt < p.kiters) load_stage(nxt, nxt % STAGES);
    cp_commit();

    const uint32_t sa = sbase + (it % STAGES) * STAGE, sb = sa + A_BYTES;
#pragma unroll
    for (int kk = 0; kk < 2; ++kk) {  // two k32 halves of the 64-byte step
      uint32_t af[2][4];
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        const int row = wm * 32 + i * 16 + (lane & 15);
        const int ch = kk * 2 + (lane >> 4);
        ldsm_x4(sa + swz(row, ch), af[i][0], af[i][1], af[i][2], af[i][3]);
      }
#pragma unroll
      for (int j = 0; j < NT; j += 2) {
        const int row = wn * WN + j * 8 + (lane & 7) + ((lane >> 4) << 3);
        const int ch = kk * 2 + ((lane >> 3) & 1);
        uint32_t b0, b1, b2, b3;
        ldsm_x4(sb + swz(row, ch), b0, b1, b2, b3);
#pragma unroll
        for (int i = 0; i < 2; ++i) {
          mma_s8(acc[i][j], af[i], b0, b1);
          mma_s8(acc[i][j + 1], af[i], b2, b3);
        }
      }
    }
  }
  cp_wait<0>();

  // epilogue: bias + requant + ReLU, int8 stores of adjacent channel pairs
#pragma unroll
  for (int j = 0; j < NT; ++j) {
    const int n = n0 + wn * WN + j * 8 + (lane & 3) * 2;
    if (n >= p.K) continue;
    const int32_t b0 = p.bias ? p.bias[n] : 0, b1 = p.bias ? p.bias[n + 1] : 0;
    const float s0 = p.scale[n], s1 = p.scale[n + 1];
#pragma unroll
    for (int i = 0; i < 2; ++i)
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const long long m = m0 + wm * 32 + i * 16 + (lane >> 2) + h * 8;
        if (m >= p.M) continue;
        char2 v;
        v.x = requant(acc[i][j][2 * h], b0, s0, p.relu);
        v.y = requant(acc[i][j][2 * h + 1], b1, s1, p.relu);
        *reinterpret_cast<char2*>(y + (size_t)m * p.K + n) = v;
      }
  }
}

__global__ void pack_int8_weights_kernel(const int8_t* __restrict__ w, int8_t* __restrict__ wp,
                                         int K, int RS, int C, int Cp) {
  const long long total = (long long)K * RS * Cp;
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < total;
       i += (long long)gridDim.x * blockDim.x) {
    const int c = (int)(i % Cp);
    const long long krs = i / Cp;
    wp[i] = c < C ? w[krs * C + c] : (int8_t)0;
  }
}

}  // namespace

cudaError_t launch_igemm_int8(const gbconv_desc_s& d, const void* x, const void* wpack,
                              const int32_t* bias, void* y, cudaStream_t st) {
  const int Cp = gb_ceil_div(d.C, BK) * BK;
  I8Params p{d.N, d.H, d.W, d.C, d.K, d.R, d.S, d.stride, d.pad, d.dil, d.OH, d.OW,
             Cp / BK, d.R * d.S * (Cp / BK), d.R * d.S * Cp,
             (long long)d.N * d.OH * d.OW, d.act == CONV_ACT_RELU ? 1 : 0, bias, d.scale};
  const long long mt = gb_ceil_div_ll(p.M, BM);
  if (mt > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  auto xb = static_cast<const int8_t*>(x);
  auto wb = static_cast<const int8_t*>(wpack);
  auto yb = static_cast<int8_t*>(y);
  if (d.K > 64) {
    constexpr int smem = STAGES * (BM * BK + 128 * BK);
    cudaError_t e = gb_set_smem_once(reinterpret_cast<const void*>(igemm_int8_kernel<128>), smem);
    if (e != cudaSuccess) return e;
    dim3 grid((unsigned)mt, gb_ceil_div(d.K, 128));
    igemm_int8_kernel<128><<<grid, THREADS, smem, st>>>(p, xb, wb, yb);
    gb_count_launch();
  } else {
    constexpr int smem = STAGES * (BM * BK + 64 * BK);
    cudaError_t e = gb_set_smem_once(reinterpret_cast<const void*>(igemm_int8_kernel<64>), smem);
    if (e != cudaSuccess) return e;
    dim3 grid((unsigned)mt, gb_ceil_div(d.K, 64));
    igemm_int8_kernel<64><<<grid, THREADS, smem, st>>>(p, xb, wb, yb);
    gb_count_launch();
  }
  return cudaGetLastError();
}

cudaError_t launch_pack_int8_weights(const gbconv_desc_s& d, const void* w, void* wpack,
                                     cudaStream_t st) {
  const int Cp = gb_ceil_div(d.C, BK) * BK;
  const long long total = (long long)d.K * d.R * d.S * Cp;
  const int grid = (int)std::min<long long>(gb_ceil_div_ll(total, 256), 65535LL * 8);
  pack_int8_weights_kernel<<<grid, 256, 0, st>>>(static_cast<const int8_t*>(w),
                                                 static_cast<int8_t*>(wpack), d.K, d.R * d.S, d.C,
                                                 Cp);
  gb_count_launch();
  return cudaGetLastError();
}
