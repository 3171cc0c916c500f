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
#include "ptx.cuh"

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

// ---- input transform: V[xi][t][c] = (B^T d B)[xi] ---------------------------------
//
// A CTA transforms one strip: image n, tile row ti, up to TWC tiles along the
// row starting at tile tj0, 64 channels.  One 4-D TMA load brings the strip's
// alpha input rows x (TWC*m + 2) columns x 64 channels into shared memory, with
// zeros outside the image (the padding).  A thread then owns one (tile,
// channel): column transform of the 8 x 8 (4 x 4) patch into registers, row
// transform, and alpha^2 two-byte stores of V (a warp writes 32 consecutive
// channels of one V row).

constexpr int WCB = 64;   // channels per strip
constexpr int TWC = 16;   // tiles per strip along the row (max)

template <typename TT>
struct InCfg {
  static constexpr int IW = TWC * TT::m + 2;                // strip columns
  static constexpr int BYTES = TT::a * IW * WCB * 2;        // strip bytes
  static constexpr int SMEM = BYTES + 64 + 128;
};

template <typename TT, bool F16>
__global__ void __launch_bounds__(256)
    input_transform_kernel(const __grid_constant__ CUtensorMap tm_x, const WinoParams p,
                           void* __restrict__ V, int* err, unsigned long long wait_ns) {
  constexpr int A = TT::a, Mo = TT::m;
  using Cf = InCfg<TT>;
  extern __shared__ __align__(128) uint8_t smem[];
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + Cf::BYTES);
  const int tblocks = (p.tw + TWC - 1) / TWC;
  int b = blockIdx.x;
  const int cblk = b % (p.C / WCB + (p.C % WCB ? 1 : 0));
  b /= (p.C / WCB + (p.C % WCB ? 1 : 0));
  const int tjb = b % tblocks;
  b /= tblocks;
  const int ti = b % p.th;
  const int nl = b / p.th;  // image within the chunk
  const int n = p.n0 + nl;
  if (threadIdx.x == 0) {
    gb::mbar_init(bar, 1);
    gb::fence_barrier_init();
    gb::mbar_arrive_expect_tx(bar, Cf::BYTES);
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4, %5}], [%6];" ::"r"(gb::smem_u32(smem)),
        "l"(reinterpret_cast<uint64_t>(&tm_x)), "r"(cblk * WCB), "r"(tjb * TWC * Mo - p.pad),
        "r"(ti * Mo - p.pad), "r"(n), "r"(gb::smem_u32(bar))
        : "memory");
  }
  __syncthreads();
  const bool ok = gb::mbar_wait_bounded(bar, 0, wait_ns, err);
  if (!__syncthreads_and(ok)) return;  // the load either landed or the wait ran out
  const __nv_bfloat16* strip = reinterpret_cast<const __nv_bfloat16*>(smem);
  const long long T = (long long)p.nb * p.th * p.tw;
  using Op = OpT<F16>;
  auto* out = reinterpret_cast<decltype(Op::one(0.f))*>(V);
  for (int item = threadIdx.x; item < TWC * WCB; item += blockDim.x) {
    const int c = item % WCB;
    const int j = item / WCB;
    const int tj = tjb * TWC + j;
    const int cg = cblk * WCB + c;
    if (tj >= p.tw || cg >= p.C) continue;
    // V = B^T d B accumulated one input row at a time:
    //   u[i][b] = sum_l d[i][l] BT[b][l];   V[a][b] += BT[a][i] u[i][b]
    float acc[A][A];
#pragma unroll
    for (int a = 0; a < A; ++a)
#pragma unroll
      for (int bb = 0; bb < A; ++bb) acc[a][bb] = 0.f;
#pragma unroll
    for (int i = 0; i < A; ++i) {
      asm volatile("" ::: "memory");  // keep one row of loads live at a time
      float row[A];
#pragma unroll
      for (int l = 0; l < A; ++l)
        row[l] = __bfloat162float(strip[((size_t)i * Cf::IW + j * Mo + l) * WCB + c]);
      float u[A];
#pragma unroll
      for (int bb = 0; bb < A; ++bb) {
        float v = 0.f;
#pragma unroll
        for (int l = 0; l < A; ++l) v = madd(v, TT::BT(bb, l), row[l]);
        u[bb] = v;
      }
#pragma unroll
      for (int a = 0; a < A; ++a)
#pragma unroll
        for (int bb = 0; bb < A; ++bb) acc[a][bb] = madd(acc[a][bb], TT::BT(a, i), u[bb]);
    }
    const long long tg = ((long long)nl * p.th + ti) * p.tw + tj;
    auto* o = out + (size_t)tg * p.C + cg;  // V[0][tg][cg]; one xi plane is T*C apart
    const size_t plane = (size_t)T * p.C;
#pragma unroll
    for (int a = 0; a < A; ++a) {
      asm volatile("" ::: "memory");
#pragma unroll
      for (int bb = 0; bb < A; ++bb) {
        *o = Op::one(acc[a][bb]);
        o += plane;
      }
    }
  }
}

// ---- output transform: Y = A^T M A (+ bias, residual, act), one channel per thread

template <typename TT>
__global__ void __launch_bounds__(256)
    output_transform_kernel(const WinoParams p, const float* __restrict__ Mws,
                            const float* __restrict__ bias, const __nv_bfloat16* __restrict__ res,
                            __nv_bfloat16* __restrict__ y) {
  constexpr int A = TT::a, Mo = TT::m;
  const long long T = (long long)p.nb * p.th * p.tw;
  const long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x;
  if (i >= T * p.K) return;
  const int k = (int)(i % p.K);
  const long long t = i / p.K;
  const int tj = (int)(t % p.tw);
  const int ti = (int)((t / p.tw) % p.th);
  const int n = p.n0 + (int)(t / ((long long)p.tw * p.th));

  // tmp[a][l] = sum_xi1 A^T[a][xi1] M[xi1][l]
  float tmp[Mo][A];
#pragma unroll
  for (int a = 0; a < Mo; ++a)
#pragma unroll
    for (int l = 0; l < A; ++l) tmp[a][l] = 0.f;
#pragma unroll
  for (int r = 0; r < A; ++r) {
    float row[A];
#pragma unroll
    for (int l = 0; l < A; ++l) row[l] = __ldg(Mws + ((size_t)(r * A + l) * T + t) * p.K + k);
#pragma unroll
    for (int a = 0; a < Mo; ++a)
#pragma unroll
      for (int l = 0; l < A; ++l) tmp[a][l] = madd(tmp[a][l], TT::AT(a, r), row[l]);
  }
  const float bk = bias ? __ldg(bias + k) : 0.f;
#pragma unroll
  for (int a = 0; a < Mo; ++a) {
    const int oh = ti * Mo + a;
    if (oh >= p.OH) break;
#pragma unroll
    for (int b = 0; b < Mo; ++b) {
      const int ow = tj * Mo + b;
      if (ow >= p.OW) break;
      float v = bk;
#pragma unroll
      for (int l = 0; l < A; ++l) v = madd(v, TT::AT(b, l), tmp[a][l]);
      const size_t off = (((size_t)n * p.OH + oh) * p.OW + ow) * p.K + k;
      if (res) v += __bfloat162float(res[off]);
      if (p.act >= 1) v = fmaxf(v, 0.f);
      if (p.act == 2) v = fminf(v, 6.f);
      y[off] = __float2bfloat16_rn(v);
    }
  }
}

constexpr size_t kChunkBudget = 64ull << 20;  // V + M bytes per chunk (L2-resident)

int tiles_h(const gbconv_desc_s& d, int m) { return gb_ceil_div(d.OH, m); }
int tiles_w(const gbconv_desc_s& d, int m) { return gb_ceil_div(d.OW, m); }

size_t bytes_per_image(const gbconv_desc_s& d, int m) {
  const size_t a2 = (size_t)(m + 2) * (m + 2);
  const size_t tiles = (size_t)tiles_h(d, m) * tiles_w(d, m);
  return tiles * a2 * ((size_t)d.C * 2 + (size_t)d.K * 4);
}

// Images per chunk: within the L2 budget, the count whose tile total fills the
// GEMM's 128-row tiles best (ties: the larger chunk).
int images_per_chunk(const gbconv_desc_s& d, int m) {
  const size_t per = bytes_per_image(d, m);
  long long nbmax = per ? (long long)(kChunkBudget / per) : 1;
  if (nbmax < 1) nbmax = 1;
  if (nbmax > d.N) nbmax = d.N;
  const long long tiles_img = (long long)tiles_h(d, m) * tiles_w(d, m);
  long long best = 1;
  double best_eff = 0.0;
  for (long long nb = 1; nb <= nbmax; ++nb) {
    const long long T = nb * tiles_img;
    const double eff = (double)T / (double)(gb_ceil_div_ll(T, 128) * 128);
    if (eff >= best_eff - 1e-9) {
      best_eff = eff;
      best = nb;
    }
  }
  return (int)best;
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
  // input strips: 4-D tiled map over x, box {64 ch, TWC*m + 2 cols, alpha rows, 1}
  CUtensorMap tmx;
  {
    cuuint64_t dims[4] = {(cuuint64_t)d.C, (cuuint64_t)d.W, (cuuint64_t)d.H, (cuuint64_t)d.N};
    cuuint64_t strides[3] = {(cuuint64_t)d.C * 2, (cuuint64_t)d.W * d.C * 2,
                             (cuuint64_t)d.H * d.W * d.C * 2};
    cuuint32_t box[4] = {WCB, (cuuint32_t)InCfg<TT>::IW, (cuuint32_t)A, 1};
    cuuint32_t estr[4] = {1, 1, 1, 1};
    if (gb_encode_tiled(&tmx, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(x), dims,
                        strides, box, estr, CU_TENSOR_MAP_SWIZZLE_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
    cudaError_t e = gb_set_smem_once(reinterpret_cast<const void*>(input_transform_kernel<TT, F16>),
                                     InCfg<TT>::SMEM);
    if (e != cudaSuccess) return e;
  }
  for (int n0 = 0; n0 < d.N; n0 += nb_max) {
    p.n0 = n0;
    p.nb = std::min(nb_max, d.N - n0);
    const long long T = (long long)p.nb * p.th * p.tw;
    const int strips = p.nb * p.th * gb_ceil_div(p.tw, TWC) * gb_ceil_div(d.C, WCB);
    input_transform_kernel<TT, F16><<<strips, 256, InCfg<TT>::SMEM, st>>>(tmx, p, V, err,
                                                                            wait_ns);
    gb_count_launch();
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    e = launch_batched_gemm_tc(A * A, (int)T, d.K, d.C, V, wpack, Mws, F16 ? 0 : 1, block_n, err,
                               wait_ns, st);
    if (e != cudaSuccess) return e;
    const long long out_threads = T * d.K;
    output_transform_kernel<TT><<<(unsigned)gb_ceil_div_ll(out_threads, 256), 256, 0, st>>>(
        p, Mws, bias, static_cast<const __nv_bfloat16*>(res), static_cast<__nv_bfloat16*>(y));
    gb_count_launch();
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
  gb_count_launch();
  return cudaGetLastError();
}

cudaError_t launch_winograd(const gbconv_desc_s& d, int m, const void* x, const void* wpack,
                            const float* bias, const void* res, void* y, void* ws, int* err,
                            unsigned long long wait_ns, cudaStream_t st) {
  if (m == 2) return run_winograd<F2T, false>(d, x, wpack, bias, res, y, ws, err, wait_ns, st);
  return run_winograd<F6T, true>(d, x, wpack, bias, res, y, ws, err, wait_ns, st);
}
