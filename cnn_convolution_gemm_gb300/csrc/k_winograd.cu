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

// ---- F(2x2,3x3): the batched GEMM with the output transform in its epilogue ----
//
// One CTA work unit: 128 consecutive Winograd tiles (rows of V) x 64 output
// channels.  Its 16 products M_xi,nu = V_xi,nu . U_xi,nu^T (128 x 64 each, fp32,
// reduced over C) are computed in four groups, one per row xi of the 4 x 4
// transformed tile.  A group's four accumulators take 4 x 64 TMEM columns; two
// groups alternate in the 512 columns, so the epilogue drains one while the
// MMAs fill the other.  The epilogue adds every product into the 2 x 2 outputs
// of its tiles (the output transform Y = A^T M A, term by term):
//   Y[i][j] += AT[i][xi] * AT[j][nu] * M_xi,nu
// in registers, and after the fourth group adds bias and residual, applies the
// activation and writes bf16 y.  The fp32 products never leave the SM, which
// is the MegEngine report's point (section "Winograd"): the transformed data
// of a block of tiles is consumed on chip, without a re-pack through memory.
//
// Warps: 0 TMA producer, 1 MMA issuer (one thread each), 2..9 epilogue.  An
// epilogue warp reads TMEM lane quarter (warp % 4) -- 32 tiles -- and one half
// (32) of the unit's 64 channels: 2 x 2 x 32 fp32 accumulators per thread.
namespace wf {
constexpr int BM = 128;                       // tiles per unit (TMEM lanes)
constexpr int BN = 64;                        // output channels per unit
constexpr int BK = 64;                        // channels per k-step (128-byte rows)
constexpr int A_BYTES = BM * BK * 2;          // V tile, 16 KB
constexpr int B_BYTES = BN * BK * 2;          // U tile, 8 KB
constexpr int STAGE = A_BYTES + B_BYTES;
constexpr int STAGES = 8;
constexpr int GROUP_COLS = 4 * BN;            // one row xi: four 64-column products
constexpr int TMEM_COLS = 2 * GROUP_COLS;     // two groups in flight
constexpr int THREADS = 320;
constexpr int SMEM = STAGES * STAGE + 256 + 1024;
}  // namespace wf

struct Wino2Params {
  int C, K, OH, OW, th, tw, act;
  int n0;        // first image of the chunk
  int T;         // tiles in the chunk (rows of V)
  int cblocks;   // k-steps per product: ceil(C / 64)
  int m_tiles, n_tiles;
  const float* bias;
  const __nv_bfloat16* res;
  __nv_bfloat16* y;
  int* err;
  unsigned long long wait_ns;
};

__global__ void __launch_bounds__(wf::THREADS, 1)
    wino2_fused_kernel(const __grid_constant__ CUtensorMap tm_v,
                       const __grid_constant__ CUtensorMap tm_u, const Wino2Params p) {
  using TT = F2T;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* sA = smem;
  uint8_t* sB = smem + wf::STAGES * wf::A_BYTES;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + wf::STAGES * wf::STAGE);
  uint64_t* full = bars;
  uint64_t* empty = bars + wf::STAGES;
  uint64_t* tfull = bars + 2 * wf::STAGES;
  uint64_t* tempty = tfull + 2;
  uint64_t* mma_done = tempty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(mma_done + 1);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < wf::STAGES; ++s) {
      gb::mbar_init(&full[s], 1);
      gb::mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      gb::mbar_init(&tfull[b], 1);
      gb::mbar_init(&tempty[b], 8);  // one arrival per epilogue warp
    }
    gb::mbar_init(mma_done, 1);
    gb::fence_barrier_init();
    gb::tma_prefetch_desc(&tm_v);
    gb::tma_prefetch_desc(&tm_u);
  }
  if (warp == 0) {
    gb::tmem_alloc(tmem_slot, wf::TMEM_COLS);
    gb::tmem_relinquish();
  }
  gb::tc_fence_before();
  __syncthreads();
  gb::tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const int units = p.m_tiles * p.n_tiles;

  if (warp == 0) {
    if (lane == 0) {
      // ---- producer: for each product, its V tile and U tile per k-step ----
      int stage = 0;
      uint32_t phase = 0;
      long long issued = 0;
      bool ok = true;
      // k-step pairs (an even channel-block count): the MMA thread frees a
      // pair of stages with one commit on the second one's barrier
      const int gmask = (p.cblocks % 2 == 0) ? 1 : 0;
      for (int u = blockIdx.x; u < units && ok; u += gridDim.x) {
        const int mt = u / p.n_tiles, nt = u % p.n_tiles;
        for (int a = 0; a < 16 && ok; ++a)
          for (int cb = 0; cb < p.cblocks; ++cb) {
            if (!gb::mbar_wait_bounded(&empty[stage | gmask], phase ^ 1, p.wait_ns, p.err)) {
              ok = false;
              break;
            }
            gb::mbar_arrive_expect_tx(&full[stage], wf::STAGE);
            gb::tma_load_3d(sA + stage * wf::A_BYTES, &tm_v, &full[stage], cb * wf::BK,
                            mt * wf::BM, a);
            gb::tma_load_3d(sB + stage * wf::B_BYTES, &tm_u, &full[stage], cb * wf::BK,
                            nt * wf::BN, a);
            ++issued;
            if (++stage == wf::STAGES) {
              stage = 0;
              phase ^= 1;
            }
          }
      }
      // no copy into shared memory may be in flight when the block exits
      long long pending = issued < wf::STAGES ? issued : wf::STAGES;
      int st = stage;
      uint32_t ph = phase;
      for (long long i = 0; i < pending; ++i) {
        if (--st < 0) {
          st = wf::STAGES - 1;
          ph ^= 1;
        }
        gb::mbar_wait_bounded(&full[st], ph, p.wait_ns, p.err);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ---- MMA issuer: group xi's four products into one TMEM group ----
      constexpr uint32_t IDESC = gb::idesc_f16(wf::BM, wf::BN, 1);
      static_assert(wf::STAGES % 2 == 0, "stage pairs");
      const bool paired = p.cblocks % 2 == 0;  // the producer's rule
      int stage = 0;
      uint32_t phase = 0;
      uint32_t grp = 0;
      bool ok = true;
      for (int u = blockIdx.x; u < units && ok; u += gridDim.x) {
        for (int xi = 0; xi < 4 && ok; ++xi, ++grp) {
          const uint32_t buf = grp & 1, gph = (grp >> 1) & 1;
          if (!gb::mbar_wait_bounded(&tempty[buf], gph ^ 1, p.wait_ns, p.err)) {
            ok = false;
            break;
          }
          gb::tc_fence_after();
          for (int nu = 0; nu < 4 && ok; ++nu) {
            const uint32_t d = tmem_base + buf * wf::GROUP_COLS + nu * wf::BN;
            if (paired) {
              // two k-steps per round of waits and one commit: with N = 64 MMAs
              // the issuing thread, not the tensor pipe, sets the pace
              for (int cb = 0; cb < p.cblocks; cb += 2) {
                const uint64_t ad0 = gb::sw128_kmajor_desc(gb::smem_u32(sA + stage * wf::A_BYTES));
                const uint64_t bd0 = gb::sw128_kmajor_desc(gb::smem_u32(sB + stage * wf::B_BYTES));
                const uint64_t ad1 = gb::sw128_kmajor_desc(gb::smem_u32(sA + (stage + 1) * wf::A_BYTES));
                const uint64_t bd1 = gb::sw128_kmajor_desc(gb::smem_u32(sB + (stage + 1) * wf::B_BYTES));
                if (!gb::mbar_wait_bounded(&full[stage], phase, p.wait_ns, p.err) ||
                    !gb::mbar_wait_bounded(&full[stage + 1], phase, p.wait_ns, p.err)) {
                  ok = false;
                  break;
                }
                gb::tc_fence_after();
#pragma unroll
                for (int k = 0; k < 4; ++k)  // descriptors count 16-byte units
                  gb::tc_mma_f16(d, ad0 + (uint64_t)(k * 2), bd0 + (uint64_t)(k * 2), IDESC,
                                 (cb > 0 || k > 0) ? 1u : 0u);
#pragma unroll
                for (int k = 0; k < 4; ++k)
                  gb::tc_mma_f16(d, ad1 + (uint64_t)(k * 2), bd1 + (uint64_t)(k * 2), IDESC, 1u);
                gb::tc_commit(&empty[stage + 1]);  // frees both stages
                stage += 2;
                if (stage == wf::STAGES) {
                  stage = 0;
                  phase ^= 1;
                }
              }
              continue;
            }
            for (int cb = 0; cb < p.cblocks; ++cb) {
              if (!gb::mbar_wait_bounded(&full[stage], phase, p.wait_ns, p.err)) {
                ok = false;
                break;
              }
              gb::tc_fence_after();
              const uint64_t ad = gb::sw128_kmajor_desc(gb::smem_u32(sA + stage * wf::A_BYTES));
              const uint64_t bd = gb::sw128_kmajor_desc(gb::smem_u32(sB + stage * wf::B_BYTES));
#pragma unroll
              for (int k = 0; k < 4; ++k)
                gb::tc_mma_f16(d, ad + (uint64_t)(k * 2), bd + (uint64_t)(k * 2), IDESC,
                               (cb > 0 || k > 0) ? 1u : 0u);
              gb::tc_commit(&empty[stage]);
              if (++stage == wf::STAGES) {
                stage = 0;
                phase ^= 1;
              }
            }
          }
          if (ok) gb::tc_commit(&tfull[buf]);
        }
      }
      gb::tc_commit(mma_done);
      gb::mbar_wait_bounded(mma_done, 0, p.wait_ns, p.err);
    }
  } else {
    // ---- epilogue: output transform, bias, residual, activation, bf16 ----
    const int q = warp & 3;          // TMEM lane quarter this warp may read
    const int h = (warp - 2) >> 2;   // which 32 of the unit's 64 channels
    uint32_t grp = 0;
    bool ok = true;
    for (int u = blockIdx.x; u < units && ok; u += gridDim.x) {
      const int mt = u / p.n_tiles, nt = u % p.n_tiles;
      float Y[4][32];  // [i * 2 + j][channel]
#pragma unroll
      for (int o = 0; o < 4; ++o)
#pragma unroll
        for (int c = 0; c < 32; ++c) Y[o][c] = 0.f;
#pragma unroll
      for (int xi = 0; xi < 4; ++xi) {
        const uint32_t buf = grp & 1, gph = (grp >> 1) & 1;
        ++grp;
        if (!ok || !gb::mbar_wait_bounded(&tfull[buf], gph, p.wait_ns, p.err)) {
          ok = false;
          continue;
        }
        gb::tc_fence_after();
        const uint32_t tcol =
            tmem_base + ((uint32_t)(q * 32) << 16) + buf * wf::GROUP_COLS + h * 32;
#pragma unroll
        for (int piece = 0; piece < 4; ++piece) {
          uint32_t v[4][8];
#pragma unroll
          for (int nu = 0; nu < 4; ++nu) gb::tmem_ld_x8(tcol + nu * wf::BN + piece * 8, v[nu]);
          gb::tmem_ld_wait();
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            // Z_j = sum_nu AT[j][nu] M_xi,nu, then Y[i][j] += AT[i][xi] Z_j
            float z[2];
#pragma unroll
            for (int j = 0; j < 2; ++j) {
              float a = 0.f;
#pragma unroll
              for (int nu = 0; nu < 4; ++nu) a = madd(a, TT::AT(j, nu), __uint_as_float(v[nu][e]));
              z[j] = a;
            }
#pragma unroll
            for (int i = 0; i < 2; ++i)
#pragma unroll
              for (int j = 0; j < 2; ++j)
                Y[i * 2 + j][piece * 8 + e] = madd(Y[i * 2 + j][piece * 8 + e], TT::AT(i, xi), z[j]);
          }
        }
        gb::tc_fence_before();
        __syncwarp();
        if (lane == 0) gb::mbar_arrive(&tempty[buf]);  // this group's columns are free
      }
      if (!ok) break;
      // outputs of tile t: pixels (2 ti + i, 2 tj + j) of image n, channels kb..kb+31
      const int t = mt * wf::BM + q * 32 + lane;
      if (t >= p.T) continue;
      const int tj = t % p.tw, ti = (t / p.tw) % p.th;
      const int n = p.n0 + t / (p.tw * p.th);
      const int kb = nt * wf::BN + h * 32;
#pragma unroll
      for (int i = 0; i < 2; ++i)
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          const int oh = 2 * ti + i, ow = 2 * tj + j;
          if (oh >= p.OH || ow >= p.OW) continue;
          const size_t pix = (((size_t)n * p.OH + oh) * p.OW + ow) * p.K;
#pragma unroll
          for (int c8 = 0; c8 < 4; ++c8) {
            const int k = kb + c8 * 8;
            if (k >= p.K) break;  // K % 8 == 0
            float o8[8];
#pragma unroll
            for (int e = 0; e < 8; ++e)
              o8[e] = Y[i * 2 + j][c8 * 8 + e] + (p.bias ? __ldg(p.bias + k + e) : 0.f);
            if (p.res) {
              const uint4 r = __ldg(reinterpret_cast<const uint4*>(p.res + pix + k));
              const uint32_t rw[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&rw[e]));
                o8[2 * e] += f.x;
                o8[2 * e + 1] += f.y;
              }
            }
            uint32_t pk[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              float a0 = o8[2 * e], a1 = o8[2 * e + 1];
              if (p.act >= 1) {
                a0 = fmaxf(a0, 0.f);
                a1 = fmaxf(a1, 0.f);
              }
              if (p.act == 2) {
                a0 = fminf(a0, 6.f);
                a1 = fminf(a1, 6.f);
              }
              __nv_bfloat162 b2 = __floats2bfloat162_rn(a0, a1);
              pk[e] = *reinterpret_cast<uint32_t*>(&b2);
            }
            *reinterpret_cast<uint4*>(p.y + pix + k) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
          }
        }
    }
  }
  gb::tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    gb::tc_fence_after();
    gb::tmem_dealloc(tmem_base, wf::TMEM_COLS);
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

// ---- F(2x2,3x3) fused: input transform into an L2-resident V chunk, then the
// GEMM with the output transform in its epilogue (no M buffer) -------------------

constexpr size_t kVBudget = 48ull << 20;  // V bytes per chunk (L2-resident)

size_t v_bytes_per_image(const gbconv_desc_s& d) {
  return (size_t)16 * tiles_h(d, 2) * tiles_w(d, 2) * d.C * 2;
}

// Images per chunk: among counts whose V fits the budget, the one with the
// fewest GEMM waves per image (a chunk's units = 128-tile rows x 64-channel
// columns, over the SMs; ties: the larger chunk), capped at the batch.  The
// count is min(constant, N), so a batch's scratch never shrinks as it grows.
int images_per_chunk_fused(const gbconv_desc_s& d) {
  const size_t per = v_bytes_per_image(d);
  long long nbmax = per ? (long long)(kVBudget / per) : 1;
  if (nbmax < 1) nbmax = 1;
  nbmax = std::min<long long>(nbmax, 4096);
  const long long tiles_img = (long long)tiles_h(d, 2) * tiles_w(d, 2);
  const long long n_tiles = gb_ceil_div(d.K, wf::BN), sms = gb_num_sms();
  long long best = 1;
  double best_cost = 1e300;
  for (long long nb = 1; nb <= nbmax; ++nb) {
    const long long units = gb_ceil_div_ll(nb * tiles_img, wf::BM) * n_tiles;
    const double cost = (double)gb_ceil_div_ll(units, sms) / (double)nb;
    if (cost <= best_cost * (1 + 1e-12)) {
      best_cost = cost;
      best = nb;
    }
  }
  return (int)std::min<long long>(best, d.N);
}

cudaError_t run_winograd2_fused(const gbconv_desc_s& d, const void* x, const void* wpack,
                                const float* bias, const void* res, void* y, void* ws, int* err,
                                unsigned long long wait_ns, cudaStream_t st) {
  using TT = F2T;
  WinoParams p{d.N, d.C, d.H, d.W, d.K, d.OH, d.OW, d.pad, tiles_h(d, 2), tiles_w(d, 2), d.act,
               0, 0};
  const int nb_max = images_per_chunk_fused(d);
  CUtensorMap tmx;  // input strips, as for the unfused transform
  {
    cuuint64_t dims[4] = {(cuuint64_t)d.C, (cuuint64_t)d.W, (cuuint64_t)d.H, (cuuint64_t)d.N};
    cuuint64_t strides[3] = {(cuuint64_t)d.C * 2, (cuuint64_t)d.W * d.C * 2,
                             (cuuint64_t)d.H * d.W * d.C * 2};
    cuuint32_t box[4] = {WCB, (cuuint32_t)InCfg<TT>::IW, (cuuint32_t)TT::a, 1};
    cuuint32_t estr[4] = {1, 1, 1, 1};
    if (gb_encode_tiled(&tmx, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(x), dims,
                        strides, box, estr, CU_TENSOR_MAP_SWIZZLE_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  CUtensorMap tmu;  // U [16][K][C]: 64-channel x 64-row boxes
  {
    cuuint64_t dims[3] = {(cuuint64_t)d.C, (cuuint64_t)d.K, 16};
    cuuint64_t strides[2] = {(cuuint64_t)d.C * 2, (cuuint64_t)d.K * d.C * 2};
    cuuint32_t box[3] = {wf::BK, wf::BN, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    if (gb_encode_tiled(&tmu, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(wpack), dims,
                        strides, box, estr, CU_TENSOR_MAP_SWIZZLE_128B) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  cudaError_t e = gb_set_smem_once(reinterpret_cast<const void*>(input_transform_kernel<TT, false>),
                                   InCfg<TT>::SMEM);
  if (e != cudaSuccess) return e;
  e = gb_set_smem_once(reinterpret_cast<const void*>(wino2_fused_kernel), wf::SMEM);
  if (e != cudaSuccess) return e;
  for (int n0 = 0; n0 < d.N; n0 += nb_max) {
    p.n0 = n0;
    p.nb = std::min(nb_max, d.N - n0);
    const long long T = (long long)p.nb * p.th * p.tw;
    const int strips = p.nb * p.th * gb_ceil_div(p.tw, TWC) * gb_ceil_div(d.C, WCB);
    input_transform_kernel<TT, false><<<strips, 256, InCfg<TT>::SMEM, st>>>(tmx, p, ws, err,
                                                                            wait_ns);
    gb_count_launch();
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    CUtensorMap tmv;  // V [16][T][C] of this chunk: 64-channel x 128-tile boxes
    {
      cuuint64_t dims[3] = {(cuuint64_t)d.C, (cuuint64_t)T, 16};
      cuuint64_t strides[2] = {(cuuint64_t)d.C * 2, (cuuint64_t)T * d.C * 2};
      cuuint32_t box[3] = {wf::BK, wf::BM, 1};
      cuuint32_t estr[3] = {1, 1, 1};
      if (gb_encode_tiled(&tmv, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, ws, dims, strides, box, estr,
                          CU_TENSOR_MAP_SWIZZLE_128B) != CUDA_SUCCESS)
        return cudaErrorInvalidValue;
    }
    Wino2Params q{};
    q.C = d.C;
    q.K = d.K;
    q.OH = d.OH;
    q.OW = d.OW;
    q.th = p.th;
    q.tw = p.tw;
    q.act = d.act;
    q.n0 = n0;
    q.T = (int)T;
    q.cblocks = gb_ceil_div(d.C, wf::BK);
    q.m_tiles = (int)gb_ceil_div_ll(T, wf::BM);
    q.n_tiles = gb_ceil_div(d.K, wf::BN);
    q.bias = bias;
    q.res = static_cast<const __nv_bfloat16*>(res);
    q.y = static_cast<__nv_bfloat16*>(y);
    q.err = err;
    q.wait_ns = wait_ns;
    const int units = q.m_tiles * q.n_tiles;
    const int grid = std::min(units, gb_num_sms());
    wino2_fused_kernel<<<grid, wf::THREADS, wf::SMEM, st>>>(tmv, tmu, q);
    gb_count_launch();
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
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
  if (m == 2) return (size_t)images_per_chunk_fused(d) * v_bytes_per_image(d);
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
  if (m == 2) return run_winograd2_fused(d, x, wpack, bias, res, y, ws, err, wait_ns, st);
  return run_winograd<F6T, true>(d, x, wpack, bias, res, y, ws, err, wait_ns, st);
}
