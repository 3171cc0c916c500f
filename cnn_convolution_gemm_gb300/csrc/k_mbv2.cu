// Fused MobileNetV2 inverted-residual block, stride 1, bf16 NHWC:
//   t1 = ReLU6(x * W_expand + b_expand)            1x1, C_in -> E channels
//   t2 = ReLU6(depthwise3x3(t1, pad 1) + b_dw)     E channels
//   y  = t2 * W_project + b_project (+ x)          1x1, E -> C_out channels
//
// The Momenta talk (Graph層面 / 優化2) counts the block's traffic: run as three
// layers, the two E-channel intermediates are written and read back through
// HBM (four passes of N*H*W*E values), while the block's own input and output
// are 6x smaller.  This kernel keeps t1 and t2 on chip: a persistent CTA takes
// 14x14 output tiles; per tile
//   1. TMA brings the 16x16 input halo (256 pixels x C_in channels, zeros
//      outside the image) into shared memory, laid out as 8-row x 16-byte core
//      matrices (the next tile's halo is loaded while this one is computed);
//   2. the expand is two M=128 tcgen05 MMAs per 16-channel k-step, N = E,
//      accumulating in TMEM.  Its bias rides in the MMA: two padded input
//      channels hold 1 for pixels inside the image and 0 outside, and their
//      weights are the bias split into two bf16 terms (hi + lo, 16 significant
//      bits), so the accumulator is x.W + b inside the image and exactly 0
//      outside — the depthwise conv's zero padding of t1;
//   3. each thread reads one halo pixel's E accumulators back, applies ReLU6
//      and stores bf16 to shared memory;
//   4. the depthwise 3x3 runs on CUDA cores (a thread owns 4 channels x 2
//      columns x 14 rows; each t1 value is loaded once and added into up to
//      three output rows with fma.rn.f32.bf16) and writes ReLU6(.) as bf16
//      straight into the project GEMM's A-operand layout;
//   5. the project is M=128 MMAs over K = E (N = C_out padded to 32), then bias,
//      the optional residual and a bf16 store of the 14x14 x C_out tile.
// t1 and t2 are rounded to bf16 exactly where the three-layer chain stores
// them, so the result matches the chain up to the order of fp32 additions.
#include <cuda_bf16.h>

#include <algorithm>

#include "internal.h"
#include "ptx.cuh"

namespace {

constexpr int TS = 14;            // output tile side
constexpr int HS = TS + 2;        // halo tile side
constexpr int NPIX = HS * HS;     // 256 halo pixels = two M=128 tiles
constexpr int KX = 32;            // expand reduction: C_in, two bias channels, zero padding
constexpr int XCHUNK = NPIX * 16; // one 8-channel chunk of the halo tile: 256 rows x 16 B
constexpr int X_BYTES = (KX / 8) * XCHUNK;
constexpr int NP = 32;            // project N (C_out padded)
constexpr int THREADS = 256;
constexpr int TMEM_COLS = 512;

template <int E>
struct Cfg {
  static_assert(E % 16 == 0 && E <= 160, "E: multiple of 16, at most 160");
  static constexpr int T1_PITCH = E * 2 + 16;         // bytes per halo pixel of t1
  static constexpr int T2_CHUNK = NPIX * 16 + 16;     // 8-channel chunk of t2 (+16: bank spread)
  static constexpr int WE_BYTES = (KX / 8) * E * 16;  // [4][E][8] bf16
  static constexpr int WP_BYTES = (E / 8) * NP * 16;  // [E/8][32][8] bf16
  static constexpr int WD_BYTES = 9 * E * 2;          // [9][E] bf16
  static constexpr int PACKED = WE_BYTES + WP_BYTES + WD_BYTES;
  static constexpr int OFF_X = 0;
  static constexpr int OFF_T1 = OFF_X + 2 * X_BYTES;
  static constexpr int OFF_T2 = OFF_T1 + NPIX * T1_PITCH;
  static constexpr int OFF_WE = OFF_T2 + (E / 8) * T2_CHUNK;
  static constexpr int OFF_WP = OFF_WE + WE_BYTES;
  static constexpr int OFF_B = OFF_WP + WP_BYTES;     // b_project[NP] fp32
  static constexpr int OFF_BAR = OFF_B + NP * 4;
  static constexpr int SMEM = OFF_BAR + 64 + 1024;    // barriers, TMEM slot, 1 KB alignment
  // TMEM columns: expand M-tile mt at mt * ECOL, project M-tile mt at PCOL + mt * NP
  static constexpr int ECOL = (E + 31) / 32 * 32;
  static constexpr int PCOL = 2 * ECOL;
  static_assert(PCOL + 2 * NP <= TMEM_COLS, "TMEM columns");
  static constexpr int ITEMS = (E / 4) * (TS / 2);    // depthwise work items
  static_assert(ITEMS <= THREADS, "one depthwise item per thread");
};

struct Mbv2Params {
  int N, H, W, cin, cout, res;
  int ntw, nth, ntiles;
  int* err;
  unsigned long long wait_ns;
};

// a * b + c for bf16 a, b (bit patterns) and fp32 c: the product of two bf16
// values is exact in fp32, so this is the fp32 FMA of the widened operands
__device__ __forceinline__ float fma_bf16(unsigned short a, unsigned short b, float c) {
  float d;
  asm("fma.rn.f32.bf16 %0, %1, %2, %3;" : "=f"(d) : "h"(a), "h"(b), "f"(c));
  return d;
}
// the two bf16 halves of a packed word (lo: the element at the lower address)
__device__ __forceinline__ void halves(uint32_t u, unsigned short& lo, unsigned short& hi) {
  asm("mov.b32 {%0, %1}, %2;" : "=h"(lo), "=h"(hi) : "r"(u));
}
// two fp32 -> bf16x2 (round to nearest even), lo in the low half
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}
// ReLU6 then bf16: the conversion clamps negatives to zero, then a packed min
// with 6 (exact in bf16); clamping after the monotone rounding equals clamping
// before it
__device__ __forceinline__ uint32_t relu6_bf16(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.relu.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  const __nv_bfloat162 six = __float2bfloat162_rn(6.f);
  __nv_bfloat162 h = __hmin2(*reinterpret_cast<__nv_bfloat162*>(&r), six);
  return *reinterpret_cast<uint32_t*>(&h);
}
__device__ __forceinline__ uint2 lds64(uint32_t addr) {
  uint2 v;
  asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(addr));
  return v;
}
__device__ __forceinline__ void sts64(uint32_t addr, uint32_t a, uint32_t b) {
  asm volatile("st.shared.v2.u32 [%0], {%1, %2};" ::"r"(addr), "r"(a), "r"(b) : "memory");
}
__device__ __forceinline__ void sts128(uint32_t addr, uint32_t a, uint32_t b, uint32_t c,
                                       uint32_t d) {
  asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c),
               "r"(d)
               : "memory");
}

// Depthwise 3x3 + bias + ReLU6 for one work item: channels 4g..4g+3 of output
// columns 2jp, 2jp+1, all 14 rows of the tile.  Input row rho of the halo feeds
// output row rho - i through filter row i; each t1 value is loaded once and
// added (fma.rn.f32.bf16 on the packed words: no widening instructions) into
// the accumulators of the (up to three) output rows it reaches;
// output row o lives in slot o % 3 and is stored once row o + 2 has been added.
// The result goes to t2 in the project GEMM's K-major core-matrix layout:
// channel chunk c/8 at chunk * T2_CHUNK, pixel m at m * 16, (c % 8) * 2 within.
template <int E>
__device__ __forceinline__ void dw_tile(uint32_t t1, uint32_t t2, int g, int jp,
                                        const unsigned short (&wf)[9][4],
                                        const float (&bz)[4]) {
  using C = Cfg<E>;
  const uint32_t src = t1 + (uint32_t)(2 * jp) * C::T1_PITCH + (uint32_t)g * 8;
  const uint32_t dst = t2 + (uint32_t)(g >> 1) * C::T2_CHUNK + (uint32_t)(g & 1) * 8 +
                       (uint32_t)(2 * jp) * 16;
  float acc[3][2][4];  // [slot][output column][channel]
#pragma unroll
  for (int rho = 0; rho < HS; ++rho) {
    unsigned short xh[4][4];  // bf16 t1 values of this row: [column][channel]
#pragma unroll
    for (int cc = 0; cc < 4; ++cc) {
      const uint2 v = lds64(src + rho * (HS * C::T1_PITCH) + cc * C::T1_PITCH);
      halves(v.x, xh[cc][0], xh[cc][1]);
      halves(v.y, xh[cc][2], xh[cc][3]);
    }
#pragma unroll
    for (int i = 0; i < 3; ++i) {
      if (rho < i || rho - i >= TS) continue;
      float(&a)[2][4] = acc[(rho - i) % 3];
#pragma unroll
      for (int s = 0; s < 3; ++s)
#pragma unroll
        for (int o = 0; o < 2; ++o)
#pragma unroll
          for (int q = 0; q < 4; ++q)
            a[o][q] = fma_bf16(xh[o + s][q], wf[i * 3 + s][q],
                               (i == 0 && s == 0) ? bz[q] : a[o][q]);
    }
    if (rho < 2) continue;
    const int orow = rho - 2;
    const float(&a)[2][4] = acc[orow % 3];
#pragma unroll
    for (int o = 0; o < 2; ++o)
      sts64(dst + (uint32_t)(orow * TS + o) * 16, relu6_bf16(a[o][0], a[o][1]),
            relu6_bf16(a[o][2], a[o][3]));
  }
}

template <int E>
__global__ void __launch_bounds__(THREADS, 1)
    mbv2_block_kernel(const __grid_constant__ CUtensorMap tm_x, const Mbv2Params p,
                      const uint8_t* __restrict__ wpack, const float* __restrict__ b_dw,
                      const float* __restrict__ b_proj,
                      const __nv_bfloat16* __restrict__ x, __nv_bfloat16* __restrict__ y) {
  using C = Cfg<E>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint64_t* xfull = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);  // [2] halo landed
  uint64_t* ebar = xfull + 2;  // expand MMAs done
  uint64_t* pbar = xfull + 3;  // project MMAs done
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(xfull + 4);
  float* sb_proj = reinterpret_cast<float*>(smem + C::OFF_B);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t s_x = gb::smem_u32(smem + C::OFF_X);
  const uint32_t s_t1 = gb::smem_u32(smem + C::OFF_T1);
  const uint32_t s_t2 = gb::smem_u32(smem + C::OFF_T2);
  const uint32_t s_we = gb::smem_u32(smem + C::OFF_WE);
  const uint32_t s_wp = gb::smem_u32(smem + C::OFF_WP);
  const int xchunks = p.cin / 8;  // chunks loaded by TMA; chunk xchunks holds the bias channels

  if (tid == 0) {
    gb::mbar_init(&xfull[0], 1);
    gb::mbar_init(&xfull[1], 1);
    gb::mbar_init(ebar, 1);
    gb::mbar_init(pbar, 1);
    gb::fence_barrier_init();
    gb::tma_prefetch_desc(&tm_x);
  }
  if (warp == 0) {
    gb::tmem_alloc(tmem_slot, TMEM_COLS);
    gb::tmem_relinquish();
  }
  // packed weights (already in core-matrix order) and biases into shared
  // memory; both halo buffers zeroed so channel chunks past C_in read as zeros
  {
    const uint4* src = reinterpret_cast<const uint4*>(wpack);
    uint4* dwe = reinterpret_cast<uint4*>(smem + C::OFF_WE);
    for (int i = tid; i < (C::WE_BYTES + C::WP_BYTES) / 16; i += THREADS) dwe[i] = __ldg(src + i);
    uint4* dx = reinterpret_cast<uint4*>(smem + C::OFF_X);
    for (int i = tid; i < 2 * X_BYTES / 16; i += THREADS) dx[i] = make_uint4(0, 0, 0, 0);
    for (int i = tid; i < NP; i += THREADS)
      sb_proj[i] = (b_proj && i < p.cout) ? __ldg(b_proj + i) : 0.f;
  }
  // this thread's depthwise item and its weights (fixed for the whole launch)
  const int dg = tid % (E / 4), djp = tid / (E / 4);
  const bool dw_item = tid < C::ITEMS;
  unsigned short wf[9][4];  // bf16 weights [tap][channel]
  float bz[4];
  if (dw_item) {
    const __nv_bfloat16* wd =
        reinterpret_cast<const __nv_bfloat16*>(wpack + C::WE_BYTES + C::WP_BYTES);
#pragma unroll
    for (int k = 0; k < 9; ++k) {
      const uint2 v = __ldg(reinterpret_cast<const uint2*>(wd + k * E + dg * 4));
      halves(v.x, wf[k][0], wf[k][1]);
      halves(v.y, wf[k][2], wf[k][3]);
    }
    const int c = dg * 4;
    for (int q = 0; q < 4; ++q) bz[q] = b_dw ? __ldg(b_dw + c + q) : 0.f;
  }
  gb::fence_proxy_async_smem();  // generic writes (weights, zeros) before async-proxy use
  gb::tc_fence_before();
  __syncthreads();
  gb::tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  auto tile_coords = [&](int t, int& n, int& h0, int& w0) {
    const int tw = t % p.ntw;
    t /= p.ntw;
    h0 = (t % p.nth) * TS;
    n = t / p.nth;
    w0 = tw * TS;
  };
  // thread 0: halo of tile t into buffer b (one 8-channel box per chunk)
  int xissued0 = 0, xissued1 = 0, xdone0 = 0, xdone1 = 0;  // loads per buffer (thread 0)
  auto issue_x = [&](int t, int b) {
    int n, h0, w0;
    tile_coords(t, n, h0, w0);
    gb::mbar_arrive_expect_tx(&xfull[b], xchunks * XCHUNK);
    for (int k = 0; k < xchunks; ++k)
      asm volatile(
          "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
          " [%0], [%1, {%2, %3, %4, %5}], [%6];" ::"r"(s_x + b * X_BYTES + k * XCHUNK),
          "l"(reinterpret_cast<uint64_t>(&tm_x)), "r"(k * 8), "r"(w0 - 1), "r"(h0 - 1), "r"(n),
          "r"(gb::smem_u32(&xfull[b]))
          : "memory");
    if (b) ++xissued1; else ++xissued0;
  };
  if (tid == 0 && (int)blockIdx.x < p.ntiles) issue_x(blockIdx.x, 0);

  constexpr uint32_t IDESC_E = gb::idesc_f16(128, E, 1);
  constexpr uint32_t IDESC_P = gb::idesc_f16(128, NP, 1);
  uint32_t ephase = 0, pphase = 0;
  bool e_pending = false, p_pending = false;  // MMAs issued and not yet waited for
  const int q = warp & 3, mt = warp >> 2;    // TMEM lane quarter and M-tile of this warp
  const uint32_t lane_off = (uint32_t)(q * 32) << 16;

  // project epilogue of a finished tile: output pixel m = oh * 14 + ow
  auto project_epilogue = [&](int n, int h0, int w0) {
    const int m = mt * 128 + q * 32 + lane;
    const int oh = m / TS, ow = m % TS;
    const int hh = h0 + oh, ww = w0 + ow;
    const bool store = m < TS * TS && hh < p.H && ww < p.W;
    uint32_t r[32];
    const uint32_t tl = tmem_base + lane_off + C::PCOL + mt * NP;
    gb::tmem_ld_x16(tl, *reinterpret_cast<uint32_t(*)[16]>(&r[0]));
    gb::tmem_ld_x16(tl + 16, *reinterpret_cast<uint32_t(*)[16]>(&r[16]));
    gb::tmem_ld_wait();
    if (store) {
      const size_t off = (((size_t)n * p.H + hh) * p.W + ww) * p.cout;
      uint4* yo = reinterpret_cast<uint4*>(y + off);
      const uint4* xr = reinterpret_cast<const uint4*>(x + off);  // residual: C_in == C_out
#pragma unroll
      for (int c8 = 0; c8 < NP / 8; ++c8) {
        if (c8 * 8 >= p.cout) break;
        float v[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) v[i] = __uint_as_float(r[c8 * 8 + i]) + sb_proj[c8 * 8 + i];
        if (p.res) {
          const uint4 rv = __ldg(xr + c8);
          const uint32_t rw[4] = {rv.x, rv.y, rv.z, rv.w};
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            v[2 * i] += __uint_as_float(rw[i] << 16);
            v[2 * i + 1] += __uint_as_float(rw[i] & 0xffff0000u);
          }
        }
        yo[c8] = make_uint4(pack_bf16(v[0], v[1]), pack_bf16(v[2], v[3]), pack_bf16(v[4], v[5]),
                            pack_bf16(v[6], v[7]));
      }
    }
    gb::tc_fence_before();
  };

  // Software pipeline over the CTA's tiles: the project MMAs of tile i run
  // while tile i+1's halo wait and expand MMAs are issued, and tile i's project
  // epilogue overlaps tile i+1's expand MMAs.
  int it = 0, pn = 0, ph0 = 0, pw0 = 0;  // coordinates of the tile whose project is in flight
  bool ok = true;
  for (int t = blockIdx.x; t < p.ntiles; t += gridDim.x, ++it) {
    const int buf = it & 1;
    int n, h0, w0;
    tile_coords(t, n, h0, w0);
    // the other buffer's last tile finished its expand MMA: load the next halo there
    if (tid == 0 && t + (int)gridDim.x < p.ntiles) issue_x(t + gridDim.x, buf ^ 1);
    {  // bias channels C_in, C_in+1 of halo pixel tid: 1 inside the image, 0 outside
      const int hh = h0 - 1 + (tid >> 4), ww = w0 - 1 + (tid & 15);
      const bool inside = hh >= 0 && hh < p.H && ww >= 0 && ww < p.W;
      *reinterpret_cast<uint32_t*>(smem + C::OFF_X + buf * X_BYTES + xchunks * XCHUNK + tid * 16) =
          inside ? 0x3F803F80u : 0u;  // two bf16 ones
      gb::fence_proxy_async_smem();
    }
    ok = gb::mbar_wait_bounded(&xfull[buf], (uint32_t)((it >> 1) & 1), p.wait_ns, p.err);
    if (!__syncthreads_and(ok)) break;
    if (tid == 0) {
      if (buf) ++xdone1; else ++xdone0;
    }

    // 2. expand: D[mt] = X[mt] (128 x 32) * WE^T (32 x E)
    if (tid == 0) {
      gb::tc_fence_after();
#pragma unroll
      for (int m2 = 0; m2 < 2; ++m2)
#pragma unroll
        for (int ks = 0; ks < KX / 16; ++ks)
          gb::tc_mma_f16(
              tmem_base + m2 * C::ECOL,
              gb::noswz_kmajor_desc(s_x + buf * X_BYTES + m2 * 2048 + ks * 2 * XCHUNK, XCHUNK, 128),
              gb::noswz_kmajor_desc(s_we + ks * 2 * (E * 16), E * 16, 128), IDESC_E, ks > 0);
      gb::tc_commit(ebar);
    }
    e_pending = true;

    // previous tile's project epilogue while the expand runs
    if (p_pending) {
      ok = gb::mbar_wait_bounded(pbar, pphase, p.wait_ns, p.err);
      if (!__syncthreads_and(ok)) break;
      p_pending = false;
      pphase ^= 1;
      gb::tc_fence_after();
      project_epilogue(pn, ph0, pw0);
    }

    ok = gb::mbar_wait_bounded(ebar, ephase, p.wait_ns, p.err);
    if (!__syncthreads_and(ok)) break;
    e_pending = false;
    ephase ^= 1;
    gb::tc_fence_after();

    // 3. expand epilogue: halo pixel pix -> t1 row (the accumulator is already
    //    0 outside the image)
    {
      const int pix = mt * 128 + q * 32 + lane;
      const uint32_t tl = tmem_base + lane_off + mt * C::ECOL;
      const uint32_t row = s_t1 + (uint32_t)pix * C::T1_PITCH;
      constexpr int G = 3;  // 16-column chunks per TMEM wait
      static_assert((E / 16) % G == 0, "chunk grouping");
#pragma unroll 1
      for (int j0 = 0; j0 < E / 16; j0 += G) {
        uint32_t r[G][16];
#pragma unroll
        for (int g2 = 0; g2 < G; ++g2) gb::tmem_ld_x16(tl + (j0 + g2) * 16, r[g2]);
        gb::tmem_ld_wait();
#pragma unroll
        for (int g2 = 0; g2 < G; ++g2) {
          uint32_t o[8];
#pragma unroll
          for (int i = 0; i < 8; ++i)
            o[i] = relu6_bf16(__uint_as_float(r[g2][2 * i]), __uint_as_float(r[g2][2 * i + 1]));
          const uint32_t a = row + (j0 + g2) * 32;
          sts128(a, o[0], o[1], o[2], o[3]);
          sts128(a + 16, o[4], o[5], o[6], o[7]);
        }
      }
    }
    gb::tc_fence_before();
    __syncthreads();

    // 4. depthwise into t2 (the previous tile's project MMAs, t2's last reader, are done)
    if (dw_item) dw_tile<E>(s_t1, s_t2, dg, djp, wf, bz);
    gb::fence_proxy_async_smem();  // t2's generic writes before the MMA reads them
    gb::tc_fence_before();
    __syncthreads();

    // 5. project: D[mt] = T2[mt] (128 x E) * WP^T (E x 32); its epilogue runs
    //    next iteration (or after the loop)
    if (tid == 0) {
      gb::tc_fence_after();
#pragma unroll
      for (int m2 = 0; m2 < 2; ++m2)
#pragma unroll
        for (int ks = 0; ks < E / 16; ++ks)
          gb::tc_mma_f16(tmem_base + C::PCOL + m2 * NP,
                         gb::noswz_kmajor_desc(s_t2 + m2 * 2048 + ks * 2 * C::T2_CHUNK,
                                               C::T2_CHUNK, 128),
                         gb::noswz_kmajor_desc(s_wp + ks * 2 * (NP * 16), NP * 16, 128), IDESC_P,
                         ks > 0);
      gb::tc_commit(pbar);
    }
    p_pending = true;
    pn = n;
    ph0 = h0;
    pw0 = w0;
  }
  if (ok && p_pending) {  // the last tile's project epilogue
    ok = gb::mbar_wait_bounded(pbar, pphase, p.wait_ns, p.err);
    if (__syncthreads_and(ok)) {
      p_pending = false;
      gb::tc_fence_after();
      project_epilogue(pn, ph0, pw0);
    }
  }

  // Teardown.  On normal exit every halo load was consumed and every MMA waited
  // for.  After a timeout, let in-flight copies and MMAs finish (bounded)
  // before the shared memory and TMEM are released.
  if (tid == 0) {
    if (xissued0 > xdone0)
      gb::mbar_wait_bounded(&xfull[0], (uint32_t)((xissued0 - 1) & 1), p.wait_ns, p.err);
    if (xissued1 > xdone1)
      gb::mbar_wait_bounded(&xfull[1], (uint32_t)((xissued1 - 1) & 1), p.wait_ns, p.err);
    if (e_pending) gb::mbar_wait_bounded(ebar, ephase, p.wait_ns, p.err);
    if (p_pending) gb::mbar_wait_bounded(pbar, pphase, p.wait_ns, p.err);
  }
  gb::tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    gb::tc_fence_after();
    gb::tmem_dealloc(tmem_base, TMEM_COLS);
  }
}

// wpack = [WE: 4 chunks][E][8] | [WP: E/8 chunks][32][8] | [WD: 9][E], bf16
//   WE[k][e][i] = w_expand[e][c] for c = 8k + i < C_in; at c = C_in and C_in + 1 the
//   bias b_expand[e] as hi = bf16(b) and lo = bf16(b - hi); 0 beyond.
//   WP[j][r][i] = w_project[r][8j + i] (0 for r >= C_out), WD[tap][e] = w_dw[e][tap]
template <int E>
__global__ void pack_mbv2_kernel(const __nv_bfloat16* __restrict__ we,
                                 const float* __restrict__ be,
                                 const __nv_bfloat16* __restrict__ wd,
                                 const __nv_bfloat16* __restrict__ wp, int cin, int cout,
                                 __nv_bfloat16* __restrict__ out) {
  using C = Cfg<E>;
  const int nwe = C::WE_BYTES / 2, nwp = C::WP_BYTES / 2, nwd = C::WD_BYTES / 2;
  const __nv_bfloat16 z = __float2bfloat16_rn(0.f);
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < nwe + nwp + nwd;
       i += gridDim.x * blockDim.x) {
    __nv_bfloat16 v;
    if (i < nwe) {
      const int k = i / (E * 8), e = (i / 8) % E, c = k * 8 + i % 8;
      const float b = be ? be[e] : 0.f;
      const __nv_bfloat16 bhi = __float2bfloat16_rn(b);
      if (c < cin)
        v = we[e * cin + c];
      else if (c == cin)  // bias, high part
        v = bhi;
      else if (c == cin + 1)  // bias, low part: b - hi rounded
        v = __float2bfloat16_rn(b - __bfloat162float(bhi));
      else
        v = z;
    } else if (i < nwe + nwp) {
      const int j = (i - nwe) / (NP * 8), r = ((i - nwe) / 8) % NP, c = j * 8 + (i - nwe) % 8;
      v = r < cout ? wp[r * E + c] : z;
    } else {
      const int tap = (i - nwe - nwp) / E, e = (i - nwe - nwp) % E;
      v = wd[e * 9 + tap];
    }
    out[i] = v;
  }
}

}  // namespace

bool mbv2_block_supported(int cin, int E, int cout) {
  // C_in + 2 bias channels must fit the padded reduction
  return E == 144 && cin % 8 == 0 && cin >= 8 && cin + 2 <= KX && cout % 8 == 0 && cout >= 8 &&
         cout <= NP;
}

size_t mbv2_block_packed_bytes(int E) { return E == 144 ? (size_t)Cfg<144>::PACKED : 0; }

cudaError_t launch_pack_mbv2(int cin, int E, int cout, const void* we, const float* be,
                             const void* wd, const void* wp, void* out, cudaStream_t st) {
  if (E != 144) return cudaErrorInvalidValue;
  pack_mbv2_kernel<144><<<32, 256, 0, st>>>(static_cast<const __nv_bfloat16*>(we), be,
                                            static_cast<const __nv_bfloat16*>(wd),
                                            static_cast<const __nv_bfloat16*>(wp), cin, cout,
                                            static_cast<__nv_bfloat16*>(out));
  gb_count_launch();
  return cudaGetLastError();
}

cudaError_t launch_mbv2_block(int N, int H, int W, int cin, int E, int cout, const void* x,
                              const void* wpack, const float* b_dw, const float* b_proj,
                              int has_res, void* y, int* err,
                              unsigned long long wait_ns, cudaStream_t st) {
  if (E != 144) return cudaErrorInvalidValue;
  using C = Cfg<144>;
  Mbv2Params p{};
  p.N = N;
  p.H = H;
  p.W = W;
  p.cin = cin;
  p.cout = cout;
  p.res = has_res ? 1 : 0;
  p.ntw = gb_ceil_div(W, TS);
  p.nth = gb_ceil_div(H, TS);
  const long long ntiles = (long long)N * p.ntw * p.nth;
  if (ntiles >= (1LL << 31)) return cudaErrorInvalidValue;
  p.ntiles = (int)ntiles;
  p.err = err;
  p.wait_ns = wait_ns;
  CUtensorMap tm;
  cuuint64_t dims[4] = {(cuuint64_t)cin, (cuuint64_t)W, (cuuint64_t)H, (cuuint64_t)N};
  cuuint64_t strides[3] = {(cuuint64_t)cin * 2, (cuuint64_t)W * cin * 2,
                           (cuuint64_t)H * W * cin * 2};
  cuuint32_t box[4] = {8, HS, HS, 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  if (gb_encode_tiled(&tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(x), dims,
                      strides, box, estr, CU_TENSOR_MAP_SWIZZLE_NONE) != CUDA_SUCCESS)
    return cudaErrorInvalidValue;
  cudaError_t e = gb_set_smem_once(reinterpret_cast<const void*>(mbv2_block_kernel<144>), C::SMEM);
  if (e != cudaSuccess) return e;
  const int grid = std::min(p.ntiles, gb_num_sms());
  mbv2_block_kernel<144><<<grid, THREADS, C::SMEM, st>>>(
      tm, p, static_cast<const uint8_t*>(wpack), b_dw, b_proj,
      static_cast<const __nv_bfloat16*>(x), static_cast<__nv_bfloat16*>(y));
  gb_count_launch();
  return cudaGetLastError();
}
