// Winograd minimal filtering F(m x m, 3 x 3), m in {2, 6}, for 3x3 stride-1
// convolutions (the aminer.cn MegEngine report, section "Winograd": transform
// the input tiles and the weights, batched matrix product, output transform).
//
//   U[xi][k][c]  = (G g_kc G^T)[xi]                   filter transform (prepack)
//   V[xi][t][c]  = (B^T d_tc B)[xi]                   input transform, fp32 math
//   M[xi][t][k]  = sum_c V[xi][t][c] * U[xi][k][c]    alpha^2 GEMMs on tcgen05
//   Y_tk         = A^T M_tk A  (+ bias, residual, act) output transform, fp32
//
// alpha = m + 2.  Tiles of alpha x alpha inputs start at (-pad, -pad) with step m;
// inputs outside the image are zero and outputs past OH x OW are dropped.
//
// The transform matrices come from the Toom-Cook construction with the
// interpolation points {0, 1, -1, inf} (F2) and {0, 1, -1, 2, -2, 1/2, -1/2,
// inf} (F6) of the Lavin & Gray paper the report cites; rows of B^T and G are
// rescaled against each other (any diagonal scaling D: G -> D G, B^T -> D^-1 B^T
// leaves the product unchanged) so that B^T's rows have absolute sums <= 15,
// which keeps V inside the fp16 range for activations up to ~290.
//
// GEMM operand precision: bf16 for F2; fp16 for F6, whose transforms amplify
// rounding error too much for bf16's 8-bit significand.  M is fp32.
//
// The report blocks the tiles so one block's transformed data stays in L1
// ("输入转换时，分块 feature map 的全部 tiles"); here the batch is processed in
// chunks of images whose V and M together fit in a slice of the 129 MB L2, so
// the transformed tiles are produced and consumed through L2 instead of making
// a full round trip through HBM.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <algorithm>

#include "internal.h"

namespace {

// ---- transform tables ---------------------------------------------------------

struct F2T {
  static constexpr int m = 2, a = 4;
  __host__ __device__ static constexpr float BT(int i, int j) {
    constexpr float t[4][4] = {
      {1, 0, -1, 0}, {0, 1, 1, 0}, {0, -1, 1, 0}, {0, -1, 0, 1}};
    return t[i][j];
  }
  __host__ __device__ static constexpr float G(int i, int j) {
    constexpr float t[4][3] = {{1, 0, 0}, {0.5f, 0.5f, 0.5f}, {0.5f, -0.5f, 0.5f}, {0, 0, 1}};
    return t[i][j];
  }
  __host__ __device__ static constexpr float AT(int i, int j) {
    constexpr float t[2][4] = {{1, 1, 1, 0}, {0, 1, -1, 1}};
    return t[i][j];
  }
};

struct F6T {
  static constexpr int m = 6, a = 8;
  __host__ __device__ static constexpr float BT(int i, int j) {
    constexpr float t[8][8] = {
      {1, 0, -5.25f, 0, 5.25f, 0, -1, 0},
      {0, 1, 1, -4.25f, -4.25f, 1, 1, 0},
      {0, -1, 1, 4.25f, -4.25f, -1, 1, 0},
      {0, 0.5f, 0.25f, -2.5f, -1.25f, 2, 1, 0},
      {0, -0.5f, 0.25f, 2.5f, -1.25f, -2, 1, 0},
      {0, 2, 4, -2.5f, -5, 0.5f, 1, 0},
      {0, -2, 4, 2.5f, -5, -0.5f, 1, 0},
      {0, -1, 0, 5.25f, 0, -5.25f, 0, 1}};
    return t[i][j];
  }
  __host__ __device__ static constexpr float G(int i, int j) {
    constexpr float t[8][3] = {
      {1, 0, 0},
      {-2.0f / 9, -2.0f / 9, -2.0f / 9},
      {-2.0f / 9, 2.0f / 9, -2.0f / 9},
      {1.0f / 90, 1.0f / 45, 2.0f / 45},
      {1.0f / 90, -1.0f / 45, 2.0f / 45},
      {32.0f / 45, 16.0f / 45, 8.0f / 45},
      {32.0f / 45, -16.0f / 45, 8.0f / 45},
      {0, 0, 1}};
    return t[i][j];
  }
  __host__ __device__ static constexpr float AT(int i, int j) {
    constexpr float t[6][8] = {
      {1, 1, 1, 1, 1, 1, 1, 0},
      {0, 1, -1, 2, -2, 0.5f, -0.5f, 0},
      {0, 1, 1, 4, 4, 0.25f, 0.25f, 0},
      {0, 1, -1, 8, -8, 0.125f, -0.125f, 0},
      {0, 1, 1, 16, 16, 0.0625f, 0.0625f, 0},
      {0, 1, -1, 32, -32, 0.03125f, -0.03125f, 1}};
    return t[i][j];
  }
};

// y += c * x with the multiply folded away for 0 / +-1 (tables are constexpr,
// loops fully unrolled, so the branches resolve at compile time).
__device__ __forceinline__ float madd(float acc, float c, float x) {
  if (c == 0.f) return acc;
  if (c == 1.f) return acc + x;
  if (c == -1.f) return acc - x;
  return fmaf(c, x, acc);
}

template <bool F16>
struct OpT;
template <>
struct OpT<true> {
  using T2 = __half2;
  static __device__ __forceinline__ T2 make(float a, float b) { return __floats2half2_rn(a, b); }
  static __device__ __forceinline__ __half one(float a) { return __float2half_rn(a); }
};
template <>
struct OpT<false> {
  using T2 = __nv_bfloat162;
  static __device__ __forceinline__ T2 make(float a, float b) {
    return __floats2bfloat162_rn(a, b);
  }
  static __device__ __forceinline__ __nv_bfloat16 one(float a) { return __float2bfloat16_rn(a); }
};

struct WinoParams {
  int N, C, H, W, K, OH, OW, pad, th, tw, act;
  int n0, nb;  // chunk: images [n0, n0 + nb)
};

// ---- filter transform: U[xi][k][c] = (G g G^T)[xi] ------------------------------

template <typename TT, bool F16>
__global__ void filter_transform_kernel(const __nv_bfloat16* __restrict__ w, void* __restrict__ U,
                                        int K, int C) {
  constexpr int A = TT::a;
  const long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x;
  if (i >= (long long)K * C) return;
  const int c = (int)(i % C), k = (int)(i / C);
  float g[3][3];
#pragma unroll
  for (int r = 0; r < 3; ++r)
#pragma unroll
    for (int s = 0; s < 3; ++s) g[r][s] = __bfloat162float(w[((size_t)k * 9 + r * 3 + s) * C + c]);
  float tg[A][3];  // G g
#pragma unroll
  for (int a = 0; a < A; ++a)
#pragma unroll
    for (int s = 0; s < 3; ++s) {
      float v = 0.f;
#pragma unroll
      for (int r = 0; r < 3; ++r) v = madd(v, TT::G(a, r), g[r][s]);
      tg[a][s] = v;
    }
  using Op = OpT<F16>;
  auto* out = reinterpret_cast<decltype(Op::one(0.f))*>(U);
#pragma unroll
  for (int a = 0; a < A; ++a)
#pragma unroll
    for (int b = 0; b < A; ++b) {
      float v = 0.f;
#pragma unroll
      for (int s = 0; s < 3; ++s) v = madd(v, TT::G(b, s), tg[a][s]);
      out[((size_t)(a * A + b) * K + k) * C + c] = Op::one(v);
    }
}

// ---- input transform: V[xi][t][c] = (B^T d B)[xi], two channels per thread -------

template <typename TT, bool F16>
__global__ void __launch_bounds__(128)
    input_transform_kernel(const WinoParams p, const __nv_bfloat16* __restrict__ x,
                           void* __restrict__ V) {
  constexpr int A = TT::a, Mo = TT::m;
  const int cp_per = p.C / 2;
  const long long T = (long long)p.nb * p.th * p.tw;
  const long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x;
  if (i >= T * cp_per) return;
  const int cp = (int)(i % cp_per);
  const long long t = i / cp_per;
  const int tj = (int)(t % p.tw);
  const int ti = (int)((t / p.tw) % p.th);
  const int n = p.n0 + (int)(t / ((long long)p.tw * p.th));
  const int h0 = ti * Mo - p.pad, w0 = tj * Mo - p.pad;
  const __nv_bfloat16* xn = x + (size_t)n * p.H * p.W * p.C + 2 * cp;

  // tmp = B^T d, built column by column
  float2 tmp[A][A];
#pragma unroll
  for (int l = 0; l < A; ++l) {
    float2 col[A];
    const int iw = w0 + l;
#pragma unroll
    for (int k = 0; k < A; ++k) {
      const int ih = h0 + k;
      if (ih >= 0 && ih < p.H && iw >= 0 && iw < p.W) {
        const __nv_bfloat162 v =
            *reinterpret_cast<const __nv_bfloat162*>(xn + ((size_t)ih * p.W + iw) * p.C);
        col[k] = __bfloat1622float2(v);
      } else {
        col[k] = make_float2(0.f, 0.f);
      }
    }
#pragma unroll
    for (int a = 0; a < A; ++a) {
      float2 v = make_float2(0.f, 0.f);
#pragma unroll
      for (int k = 0; k < A; ++k) {
        v.x = madd(v.x, TT::BT(a, k), col[k].x);
        v.y = madd(v.y, TT::BT(a, k), col[k].y);
      }
      tmp[a][l] = v;
    }
  }
  using Op = OpT<F16>;
  using T2 = typename Op::T2;
  T2* out = reinterpret_cast<T2*>(V);
#pragma unroll
  for (int a = 0; a < A; ++a)
#pragma unroll
    for (int b = 0; b < A; ++b) {
      float2 v = make_float2(0.f, 0.f);
#pragma unroll
      for (int l = 0; l < A; ++l) {
        v.x = madd(v.x, TT::BT(b, l), tmp[a][l].x);
        v.y = madd(v.y, TT::BT(b, l), tmp[a][l].y);
      }
      out[((size_t)(a * A + b) * T + t) * cp_per + cp] = Op::make(v.x, v.y);
    }
}

// ---- output transform: Y = A^T M A (+ bias, residual, act), two channels/thread --

template <typename TT>
__global__ void __launch_bounds__(128)
    output_transform_kernel(const WinoParams p, const float* __restrict__ Mws,
                            const float* __restrict__ bias, const __nv_bfloat16* __restrict__ res,
                            __nv_bfloat16* __restrict__ y) {
  constexpr int A = TT::a, Mo = TT::m;
  const int kp_per = p.K / 2;
  const long long T = (long long)p.nb * p.th * p.tw;
  const long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x;
  if (i >= T * kp_per) return;
  const int kp = (int)(i % kp_per);
  const long long t = i / kp_per;
  const int tj = (int)(t % p.tw);
  const int ti = (int)((t / p.tw) % p.th);
  const int n = p.n0 + (int)(t / ((long long)p.tw * p.th));
  const float2* M2 = reinterpret_cast<const float2*>(Mws);

  // tmp[a][l] = sum_xi1 A^T[a][xi1] M[xi1][l]
  float2 tmp[Mo][A];
#pragma unroll
  for (int a = 0; a < Mo; ++a)
#pragma unroll
    for (int l = 0; l < A; ++l) tmp[a][l] = make_float2(0.f, 0.f);
#pragma unroll
  for (int r = 0; r < A; ++r) {
    float2 row[A];
#pragma unroll
    for (int l = 0; l < A; ++l) row[l] = M2[((size_t)(r * A + l) * T + t) * kp_per + kp];
#pragma unroll
    for (int a = 0; a < Mo; ++a)
#pragma unroll
      for (int l = 0; l < A; ++l) {
        tmp[a][l].x = madd(tmp[a][l].x, TT::AT(a, r), row[l].x);
        tmp[a][l].y = madd(tmp[a][l].y, TT::AT(a, r), row[l].y);
      }
  }
  const float b0 = bias ? bias[2 * kp] : 0.f, b1 = bias ? bias[2 * kp + 1] : 0.f;
#pragma unroll
  for (int a = 0; a < Mo; ++a) {
    const int oh = ti * Mo + a;
    if (oh >= p.OH) break;
#pragma unroll
    for (int b = 0; b < Mo; ++b) {
      const int ow = tj * Mo + b;
      if (ow >= p.OW) break;
      float2 v = make_float2(b0, b1);
#pragma unroll
      for (int l = 0; l < A; ++l) {
        v.x = madd(v.x, TT::AT(b, l), tmp[a][l].x);
        v.y = madd(v.y, TT::AT(b, l), tmp[a][l].y);
      }
      const size_t off = (((size_t)n * p.OH + oh) * p.OW + ow) * p.K + 2 * kp;
      if (res) {
        const float2 rv = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(res + off));
        v.x += rv.x;
        v.y += rv.y;
      }
      if (p.act >= 1) {
        v.x = fmaxf(v.x, 0.f);
        v.y = fmaxf(v.y, 0.f);
      }
      if (p.act == 2) {
        v.x = fminf(v.x, 6.f);
        v.y = fminf(v.y, 6.f);
      }
      *reinterpret_cast<__nv_bfloat162*>(y + off) = __floats2bfloat162_rn(v.x, v.y);
    }
  }
}

constexpr size_t kChunkBudget = 48ull << 20;  // V + M bytes per chunk (L2-resident)

int tiles_h(const gbconv_desc_s& d, int m) { return gb_ceil_div(d.OH, m); }
int tiles_w(const gbconv_desc_s& d, int m) { return gb_ceil_div(d.OW, m); }

size_t bytes_per_image(const gbconv_desc_s& d, int m) {
  const size_t a2 = (size_t)(m + 2) * (m + 2);
  const size_t tiles = (size_t)tiles_h(d, m) * tiles_w(d, m);
  return tiles * a2 * ((size_t)d.C * 2 + (size_t)d.K * 4);
}

int images_per_chunk(const gbconv_desc_s& d, int m) {
  const size_t per = bytes_per_image(d, m);
  size_t nb = per ? kChunkBudget / per : 1;
  if (nb < 1) nb = 1;
  if (nb > (size_t)d.N) nb = d.N;
  return (int)nb;
}

template <typename TT, bool F16>
cudaError_t run_winograd(const gbconv_desc_s& d, const void* x, const void* wpack,
                         const float* bias, const void* res, void* y, void* ws, int* err,
                         unsigned long long wait_ns, cudaStream_t st) {
  constexpr int Mo = TT::m, A = TT::a;
  WinoParams p{d.N, d.C, d.H, d.W, d.K, d.OH, d.OW, d.pad, tiles_h(d, Mo), tiles_w(d, Mo), d.act,
               0, 0};
  const int nb_max = images_per_chunk(d, Mo);
  const long long Tmax = (long long)nb_max * p.th * p.tw;
  void* V = ws;
  float* Mws = reinterpret_cast<float*>(static_cast<char*>(ws) +
                                        ((size_t)A * A * Tmax * d.C * 2 + 255) / 256 * 256);
  const int block_n = d.K > 128 ? 256 : (d.K > 64 ? 128 : 64);
  for (int n0 = 0; n0 < d.N; n0 += nb_max) {
    p.n0 = n0;
    p.nb = std::min(nb_max, d.N - n0);
    const long long T = (long long)p.nb * p.th * p.tw;
    const long long in_threads = T * (d.C / 2);
    input_transform_kernel<TT, F16><<<(unsigned)gb_ceil_div_ll(in_threads, 128), 128, 0, st>>>(
        p, static_cast<const __nv_bfloat16*>(x), V);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    e = launch_batched_gemm_tc(A * A, (int)T, d.K, d.C, V, wpack, Mws, F16 ? 0 : 1, block_n, err,
                               wait_ns, st);
    if (e != cudaSuccess) return e;
    const long long out_threads = T * (d.K / 2);
    output_transform_kernel<TT><<<(unsigned)gb_ceil_div_ll(out_threads, 128), 128, 0, st>>>(
        p, Mws, bias, static_cast<const __nv_bfloat16*>(res), static_cast<__nv_bfloat16*>(y));
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace

size_t winograd_packed_bytes(const gbconv_desc_s& d, int m) {
  return (size_t)(m + 2) * (m + 2) * d.K * d.C * 2;
}

size_t winograd_workspace_bytes(const gbconv_desc_s& d, int m) {
  const int A = m + 2;
  const long long Tmax = (long long)images_per_chunk(d, m) * tiles_h(d, m) * tiles_w(d, m);
  const size_t v = ((size_t)A * A * Tmax * d.C * 2 + 255) / 256 * 256;
  return v + (size_t)A * A * Tmax * d.K * 4;
}

cudaError_t launch_winograd_filter_transform(const gbconv_desc_s& d, int m, const void* w,
                                             void* wpack, cudaStream_t st) {
  const long long n = (long long)d.K * d.C;
  const unsigned grid = (unsigned)gb_ceil_div_ll(n, 128);
  auto wb = static_cast<const __nv_bfloat16*>(w);
  if (m == 2)
    filter_transform_kernel<F2T, false><<<grid, 128, 0, st>>>(wb, wpack, d.K, d.C);
  else
    filter_transform_kernel<F6T, true><<<grid, 128, 0, st>>>(wb, wpack, d.K, d.C);
  return cudaGetLastError();
}

cudaError_t launch_winograd(const gbconv_desc_s& d, int m, const void* x, const void* wpack,
                            const float* bias, const void* res, void* y, void* ws, int* err,
                            unsigned long long wait_ns, cudaStream_t st) {
  if (m == 2) return run_winograd<F2T, false>(d, x, wpack, bias, res, y, ws, err, wait_ns, st);
  return run_winograd<F6T, true>(d, x, wpack, bias, res, y, ws, err, wait_ns, st);
}
