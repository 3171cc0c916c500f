// Implicit-GEMM convolution on the 5th-generation tensor cores (tcgen05).
//
// The aminer.cn MegEngine report (section "Im2col+MatMul") unrolls input
// patches into an im2col matrix [n, fh*fw*ic, oh*ow] and multiplies it by the
// weight matrix; it then blocks the im2col matrix along oh*ow so a block stays
// on chip, and fuses the "PACK" of the GEMM panels into the im2col step so the
// unrolled data is written once instead of twice ("融合 PACK").  Here the
// im2col matrix is never written at all: each 128-pixel block of the output
// (flattened over n, oh, ow) is one GEMM M-tile, and for every filter tap
// (r, s) and 64-channel slice a TMA load in im2col mode copies the matching
// 128 x 64 input patch straight from the NHWC activation tensor into shared
// memory, already in the 128-byte-swizzled K-major layout the tensor core
// reads.  Zero padding comes from TMA's out-of-bounds fill.
//
//   GEMM:  Y[M = N*OH*OW][K] = A[M][R*S*Cp] * Wp[K][R*S*Cp]^T
//   A[m][(r*S+s)*Cp + c] = x[n, oh*st - pad + r*dil, ow*st - pad + s*dil, c]
//
// Warp roles (192 threads, persistent over output tiles):
//   warp 0      TMA producer (one elected lane) -> STAGES-deep smem ring
//   warp 1      MMA issuer (one lane): tcgen05.mma 128 x BN x 16, fp32 in TMEM
//   warps 2..5  epilogue: tcgen05.ld -> + bias (+ residual) -> activation ->
//               bf16 ("Graph層面" of the Momenta talk: bias and ReLU fused into
//               the matrix product), staged per warp in a 128-byte-swizzled
//               32 x 64 shared-memory box and written by a TMA store, so the
//               output (and the residual, read row-coalesced into the same
//               box) moves in full 128-byte lines
// The accumulator is double-buffered in TMEM (2 x BN columns) so the
// epilogue of tile i overlaps the MMAs of tile i+1.
//
// Pair mode (PAIR, BN = 256): the grid is made of clusters of two CTAs on two
// SMs, and each work unit is a 256-row x 256-column tile.  Each CTA loads its
// own 128 rows of A and one half (128 rows) of B, so every SM moves and its
// tensor core reads 32 KB of shared memory per 64-wide k-step instead of 48 KB
// (a single SM's 128 x 256 MMA needs more shared-memory bandwidth than the SM
// has).  The even CTA's MMA thread issues tcgen05.mma.cta_group::2 (M = 256)
// over both CTAs' operands; its commits are multicast to both CTAs' barriers;
// both CTAs' loads complete on the even CTA's stage barrier; each CTA's
// epilogue drains the accumulator rows of its own A half from its own TMEM.
#include <cuda_bf16.h>

#include <algorithm>
#include <type_traits>

#include "internal.h"
#include "ptx.cuh"

namespace {

constexpr int BM = 128;  // output pixels per tile (TMEM lanes)
constexpr int BK = 64;   // channels per k-step: 64 bf16 = one 128-byte swizzle row

struct IgemmParams {
  int H, W, C, K, S, stride, pad, dil, OH, OW;
  int cblocks;  // Cp / 64
  int kiters;   // R * S * cblocks
  int Kw;       // packed weight row length R*S*Cp
  long long M;  // N*OH*OW
  int m_tiles, n_tiles;
  int act;
  const float* bias;
  const __nv_bfloat16* res;
  __nv_bfloat16* y;
  int* err;
  unsigned long long wait_ns;
  // batched-GEMM mode: `batch` independent [M x Kred] x [K x Kred]^T products
  int batch;
  int ab_type;  // 0 = fp16 operands, 1 = bf16
  float* out_f32;
  // narrow-channel mode (C == 8): each 64-wide k-step holds 8 filter taps x 8
  // channels, loaded as 8 im2col boxes of 128 pixels x 16 bytes
  int narrow;
  int taps;  // R * S
  // split-K (conv mode): the reduction is cut into ksplit ranges of kchunk
  // k-steps; range b writes fp32 partial sums to part[b][M][K] (no epilogue)
  int ksplit, kchunk;
  float* part;
  // tail rebalancing: work units from tail_start on cover the last partial
  // wave's tiles as 2^tail_shift narrower (BN >> tail_shift column) units each
  int tail_start;
  int tail_shift;  // 1 or 2 (a shift, not a divisor: decode runs in every role's loop)
  // k-steps whose MMAs the issuing thread starts after one round of waits, with
  // one commit for the group (1 or 2; 2 needs a ring of at least 6 stages, an
  // even number of them, and even k-step counts).  Each barrier wait in that
  // thread costs about 200 cycles that the tensor pipe sees as idle time
  // whenever a k-step's MMAs are short: 4 MMAs of N = 64 or 128 took 506
  // cycles per k-step with a wait each, 380 in pairs (N = 256: 512 either way,
  // the MMAs' own time).  A 4-stage ring in pairs is only two loads deep: the
  // 256-column single-CTA layer ran 13 % slower so.
  int kgroup;
  // exact int8 output (see IgemmSplit): y8[M][i8_kout]
  int8_t* i8_y;
  const int32_t* i8_bias;
  const float* i8_scale;
  int i8_kout, i8_relu, i8_nc32;
  // chunked accumulation (exact int8): every kch k-steps the MMAs start a new
  // BN-column accumulator block, i8_nch blocks per tile (0: lo/hi split weights)
  int i8_nch;
  int kch;        // k-steps per accumulator block (the whole reduction otherwise)
  int acc_cols;   // TMEM columns per tile accumulator (BN, or i8_nch * BN)
  int nacc;       // tile accumulators in TMEM (2: the epilogue overlaps the next tile)
  uint32_t tmem_cols;  // columns allocated (a power of two >= 32)
  // tf32 mode: fp32 residual [M][K] (the fp32 output goes through tm_y)
  const float* res_f32;
  // L2 warm-up (conv mode): while a unit's epilogue runs, each epilogue lane
  // touches the input pixel under the middle filter tap of its output pixel in
  // the unit this CTA takes after the next one (pf_x null: off)
  const uint8_t* pf_x;
  long long pf_pix;  // bytes between pixels of x
  int pf_row;        // bytes of a pixel's channels
  int pf_dh, pf_dw;  // middle tap offset, rows and columns (times the dilation)
  // space-to-depth-by-4 stem output (see IgemmSplit): column c of the GEMM is
  // channel c % s2d4_k of output pixel (2 bh + py, 2 bw + px), (py, px) = the
  // bits of c / s2d4_k; stored through the 5-D map in the tm_y slot
  int s2d4_k;
};

enum { MODE_CONV = 0, MODE_BATCHED = 1 };

// LIGHT: a shallow ring (for short reductions) so two CTAs fit on one SM and
// the epilogue, which bounds memory-bound layers, gets twice the warps.
// PAIR: each CTA holds half of B (see the pair mode above).
template <int BN, bool LIGHT = false, bool PAIR = false>
struct Cfg {
  static constexpr int A_BYTES = BM * BK * 2;
  static constexpr int B_BYTES = (PAIR ? BN / 2 : BN) * BK * 2;
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr int STAGES =
      PAIR ? 6 : (LIGHT ? (BN >= 128 ? 2 : 3) : ((BN >= 256) ? 4 : (BN >= 128 ? 6 : 8)));
  static constexpr uint32_t TMEM_COLS = 2 * BN;  // double-buffered fp32 accumulator
  // epilogue staging: per epilogue warp two 32-row x 64-column bf16 boxes
  // (128-byte swizzle), written by the warp and stored by TMA
  static constexpr int EPI_BOX = 32 * 128;
  static constexpr int EPI_BYTES = 4 * 2 * EPI_BOX + 4 * 256;  // + per-warp bias slice
  static constexpr int BAR_BYTES = 256;
  static constexpr int SMEM = STAGES * STAGE_BYTES + EPI_BYTES + BAR_BYTES + 1024;
};

// rings whose k-steps may be consumed in pairs (see IgemmParams::kgroup)
template <class C>
constexpr bool kGroupable = C::STAGES % 2 == 0 && C::STAGES >= 6;

// Two fp32 values in one 64-bit register pair (channels n, n + 1) for the packed
// fp32 add of the bf16 epilogue.
typedef unsigned long long f32x2;
__device__ __forceinline__ f32x2 f2_pack(float lo, float hi) {
  f32x2 r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
// two IEEE fp32 additions (each rounded to nearest even) in one instruction
__device__ __forceinline__ f32x2 f2_add(f32x2 a, f32x2 b) {
  f32x2 d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
// a bf16x2 word -> its two values in fp32 (exact: a bf16 is the top half of an fp32)
__device__ __forceinline__ f32x2 bf16x2_to_f2(uint32_t u) {
  return f2_pack(__uint_as_float(u << 16), __uint_as_float(u & 0xffff0000u));
}
// activation, then rounding to a bf16x2 word (lo channel in the low half): the
// conversion's relu clamps negatives to zero, ReLU6 then takes a packed min
// with 6 (exact in bf16); activation and the monotone rounding commute
template <int ACT>
__device__ __forceinline__ uint32_t act_to_bf16x2(f32x2 v) {
  float lo, hi;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
  uint32_t r;
  if (ACT == 0) {
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
  }
  asm("cvt.rn.relu.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  if (ACT == 2) {
    const __nv_bfloat162 six = __float2bfloat162_rn(6.f);
    __nv_bfloat162 h = __hmin2(*reinterpret_cast<__nv_bfloat162*>(&r), six);
    r = *reinterpret_cast<uint32_t*>(&h);
  }
  return r;
}

// One 32-row x 64-column bf16 epilogue sub-block of a warp: fp32 accumulator
// (r) + bias (sbias, 64 values) (+ the residual already staged in the box),
// activation, bf16, written to the 128-byte-swizzled staging box.  Per channel
// pair: each add an IEEE fp32 add (packed two per instruction), then the
// activation and the bf16 rounding in one conversion.
template <int ACT>
__device__ __forceinline__ void epi_bf16_subblock(const uint32_t (&r)[64], const float* sbias,
                                                  uint8_t* box, int lane, bool has_res) {
#pragma unroll
  for (int c16 = 0; c16 < 4; ++c16) {
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      uint8_t* chunk = box + lane * 128 + (((c16 * 2 + h) ^ (lane & 7)) << 4);
      uint4 rv = make_uint4(0, 0, 0, 0);
      if (has_res) rv = *reinterpret_cast<const uint4*>(chunk);
      const uint32_t rw[4] = {rv.x, rv.y, rv.z, rv.w};
      const float4 b0 = reinterpret_cast<const float4*>(sbias)[c16 * 4 + h * 2];
      const float4 b1 = reinterpret_cast<const float4*>(sbias)[c16 * 4 + h * 2 + 1];
      const f32x2 bp[4] = {f2_pack(b0.x, b0.y), f2_pack(b0.z, b0.w), f2_pack(b1.x, b1.y),
                           f2_pack(b1.z, b1.w)};
      uint32_t pk[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int i = c16 * 16 + h * 8 + 2 * k;
        f32x2 v = f2_add(f2_pack(__uint_as_float(r[i]), __uint_as_float(r[i + 1])), bp[k]);
        if (has_res) v = f2_add(v, bf16x2_to_f2(rw[k]));
        pk[k] = act_to_bf16x2<ACT>(v);
      }
      *reinterpret_cast<uint4*>(chunk) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
    }
  }
}

__device__ __forceinline__ float act_apply(float v, int act) {
  if (act == 1) return fmaxf(v, 0.0f);
  if (act == 2) return fminf(fmaxf(v, 0.0f), 6.0f);
  return v;
}

// TF32: fp32 NHWC tensors, kind::tf32 MMAs; a 128-byte swizzle row then holds
// 32 channels (BKE) instead of 64 and each MMA still advances 32 bytes of K.
// tm_wt: the weights with a box as wide as a tail unit (its B rows only: a
// narrow unit that loaded the whole tile's box ran at the load path's speed,
// as slow as a full-width unit); tm_w again when there is no tail.
template <int BN, int MODE, bool LIGHT = false, bool TF32 = false, bool PAIR = false>
__global__ void __launch_bounds__(192, 1)
    igemm_bf16_tc_kernel(const __grid_constant__ CUtensorMap tm_x,
                         const __grid_constant__ CUtensorMap tm_w,
                         const __grid_constant__ CUtensorMap tm_wt,
                         const __grid_constant__ CUtensorMap tm_y,
                         const __grid_constant__ CUtensorMap tm_r, const IgemmParams p) {
  using C = Cfg<BN, LIGHT, PAIR>;
  static_assert(!PAIR || (BN == 256 && MODE == MODE_CONV && !LIGHT && !TF32), "pair mode");
  constexpr int BKE = TF32 ? 32 : BK;  // channels per k-step (one 128-byte row)
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* sA = smem;
  uint8_t* sB = smem + C::STAGES * C::A_BYTES;
  uint8_t* sEpi = smem + C::STAGES * C::STAGE_BYTES;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sEpi + C::EPI_BYTES);
  uint64_t* full = bars;
  uint64_t* empty = bars + C::STAGES;
  uint64_t* tfull = bars + 2 * C::STAGES;
  uint64_t* tempty = tfull + 2;
  uint64_t* mma_done = tempty + 2;
  uint64_t* rbar = mma_done + 1;  // [4 epilogue warps][2 boxes]: residual box landed
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(rbar + 8);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  // pair mode: this CTA's rank in its pair (0 issues the MMAs), and the CTA's
  // work-unit stride over the clusters
  const uint32_t rank = PAIR ? gb::cluster_ctarank() : 0u;
  const int unit0 = PAIR ? (int)(blockIdx.x >> 1) : (int)blockIdx.x;
  const int ustep = PAIR ? (int)(gridDim.x >> 1) : (int)gridDim.x;

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      gb::mbar_init(&full[s], 1);
      gb::mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      gb::mbar_init(&tfull[b], 1);
      // pair mode: one arrival per epilogue warp of each CTA (on the even CTA's)
      gb::mbar_init(&tempty[b], PAIR ? 8 : 128);
    }
    gb::mbar_init(mma_done, 1);
    for (int i = 0; i < 8; ++i) gb::mbar_init(&rbar[i], 1);
    gb::fence_barrier_init();
    gb::tma_prefetch_desc(&tm_x);
    gb::tma_prefetch_desc(&tm_w);
    if (MODE == MODE_CONV && p.tail_start < p.m_tiles * p.n_tiles * p.ksplit)
      gb::tma_prefetch_desc(&tm_wt);
    if (MODE == MODE_CONV) gb::tma_prefetch_desc(&tm_y);
    if (MODE == MODE_CONV && p.res) gb::tma_prefetch_desc(&tm_r);
  }
  if (warp == 0) {
    if constexpr (PAIR) {
      gb::tmem_alloc_pair(tmem_slot, C::TMEM_COLS);
      gb::tmem_relinquish_pair();
    } else {
      gb::tmem_alloc(tmem_slot, p.tmem_cols);
      gb::tmem_relinquish();
    }
  }
  gb::tc_fence_before();
  __syncthreads();
  // pair mode: both CTAs' barriers are initialised before either signals the other's
  if constexpr (PAIR) gb::cluster_sync();
  gb::tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  // Programmatic dependent launch: the next kernel on the stream may start its
  // own set-up (this one's above) while this grid drains.  This grid touches
  // global memory only after the kernel before it has completed: the producer
  // waits for it before its first unit's k-steps (the unit's coordinates,
  // integer divisions on one thread, go before the wait), the epilogue warps
  // before their first load or store; the MMA thread touches shared memory and
  // TMEM only.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

  const int tiles_per_batch = p.m_tiles * p.n_tiles;
  const int num_tiles = tiles_per_batch * (MODE == MODE_BATCHED ? p.batch : p.ksplit);
  const int ohow = p.OH * p.OW;
  // work unit u -> tile t, first output column offset within the tile, width
  const int num_units =
      p.tail_start < num_tiles ? p.tail_start + ((num_tiles - p.tail_start) << p.tail_shift)
                               : num_tiles;
  // the 128-row M tile this CTA covers in tile tt of a batch (pair mode: the
  // unit's 256 rows are two M tiles, the even CTA's first)
  auto m_tile = [&](int tt) {
    return PAIR ? (tt / p.n_tiles) * 2 + (int)rank : tt / p.n_tiles;
  };
  auto decode = [&](int u, int& t, int& noff, int& width) {
    if (u < p.tail_start) {
      t = u;
      noff = 0;
      width = BN;
    } else {
      const int h = u - p.tail_start;
      t = p.tail_start + (h >> p.tail_shift);
      width = BN >> p.tail_shift;
      noff = (h & ((1 << p.tail_shift) - 1)) * width;
    }
  };

  if (warp == 0) {
    if (lane == 0) {
      // ---------------- TMA producer ----------------
      int stage = 0;
      uint32_t phase = 0;
      long long issued = 0;
      bool ok = true;
      // pair mode: the even CTA's stage barriers, where both CTAs' loads complete
      const uint32_t full_pair = PAIR ? gb::mapa_shared(gb::smem_u32(full), 0) : 0u;
      const int gmask = (kGroupable<C> && p.kgroup == 2) ? 1 : 0;
      for (int u = unit0; u < num_units && ok; u += ustep) {
        int t, noff, width;
        decode(u, t, noff, width);
        const int bt = t / tiles_per_batch;
        const int tt = t % tiles_per_batch;
        const int mt = m_tile(tt), nt = tt % p.n_tiles;
        const int m0 = mt * BM;  // M < 2^31 (checked on the host): 32-bit index math
        int img = 0, h0 = 0, w0 = 0;
        if (MODE == MODE_CONV) {
          img = m0 / ohow;
          const int rem = m0 - img * ohow;
          const int oh = rem / p.OW;
          h0 = oh * p.stride - p.pad;
          w0 = (rem - oh * p.OW) * p.stride - p.pad;
        }
        const int kbeg = MODE == MODE_CONV ? bt * p.kchunk : 0;
        const int kend = MODE == MODE_CONV ? min(p.kiters, kbeg + p.kchunk) : p.kiters;
        int cb = kbeg % p.cblocks, s = (kbeg / p.cblocks) % p.S, r = (kbeg / p.cblocks) / p.S;
        // pair mode: both CTAs' A tiles and B halves land on the even CTA's
        // barrier, which alone expects their bytes; a B half is one box of
        // width / 2 rows (BN / 2, or a tail unit's through tm_wt)
        const int n0 = nt * BN + noff + (PAIR ? (int)rank * (width / 2) : 0);
        const CUtensorMap* const bmap = width == BN ? &tm_w : &tm_wt;
        const uint32_t stage_tx =
            (uint32_t)(C::A_BYTES + (PAIR ? width / 2 : width) * (BK * 2));  // 128-byte rows
        if (u == unit0) asm volatile("griddepcontrol.wait;" ::: "memory");  // once, see above
        for (int it = kbeg; it < kend; ++it) {
          // Everything the copies need is computed before the wait, so they go
          // out as soon as the stage is free: with the operands in L2 the ring's
          // depth only just covers the load latency, and a delay here is a
          // delay of the MMAs.  The B column of k-step it is it * BKE (taps,
          // then channel blocks, in packed-weight order).
          const int xc = cb * BKE, kcol = it * BKE;
          const uint16_t offw = (uint16_t)(s * p.dil), offh = (uint16_t)(r * p.dil);
          uint8_t* const a_dst = sA + stage * C::A_BYTES;
          uint8_t* const b_dst = sB + stage * C::B_BYTES;
          // grouped k-steps: the commit of a group frees all its stages on the
          // barrier of its last one
          if (!gb::mbar_wait_bounded(&empty[stage | gmask], phase ^ 1, p.wait_ns, p.err)) {
            ok = false;
            break;
          }
          if constexpr (PAIR) {
            if (rank == 0) gb::mbar_arrive_expect_tx(&full[stage], 2 * stage_tx);
            const uint32_t fb = full_pair + stage * 8;
            gb::tma_load_im2col_4d_pair(a_dst, &tm_x, fb, xc, w0, h0, img, offw, offh);
            gb::tma_load_2d_pair(b_dst, bmap, fb, kcol, n0);
          } else {
          gb::mbar_arrive_expect_tx(&full[stage], MODE == MODE_CONV ? stage_tx : C::STAGE_BYTES);
          if (MODE == MODE_CONV && p.narrow) {
#pragma unroll 1
            for (int t = 0; t < 8; ++t) {
              int tap = it * 8 + t;
              if (tap >= p.taps) tap = 0;  // its packed weights are zero
              const int tr = tap / p.S, ts = tap % p.S;
              gb::tma_load_im2col_4d(sA + stage * C::A_BYTES + t * (BM * 16), &tm_x, &full[stage],
                                     0, w0, h0, img, (uint16_t)(ts * p.dil),
                                     (uint16_t)(tr * p.dil));
            }
            gb::tma_load_2d(sB + stage * C::B_BYTES, bmap, &full[stage], it * BK,
                            nt * BN + noff);
          } else if (MODE == MODE_CONV) {
            gb::tma_load_im2col_4d(a_dst, &tm_x, &full[stage], xc, w0, h0, img, offw, offh);
            gb::tma_load_2d(b_dst, bmap, &full[stage], kcol, n0);
          } else {
            gb::tma_load_3d(sA + stage * C::A_BYTES, &tm_x, &full[stage], cb * BK, (int)m0, bt);
            gb::tma_load_3d(sB + stage * C::B_BYTES, &tm_w, &full[stage], cb * BK, nt * BN, bt);
          }
          }
          ++issued;
          if (++stage == C::STAGES) {
            stage = 0;
            phase ^= 1;
          }
          // next (channel block, filter column, filter row), without branches:
          // nested data-dependent branches here measured 4% slower on the
          // 256-column SM-pair layer
          ++cb;
          const bool wrap_c = cb == p.cblocks;
          cb = wrap_c ? 0 : cb;
          s += wrap_c ? 1 : 0;
          const bool wrap_s = s == p.S;
          s = wrap_s ? 0 : s;
          r += wrap_s ? 1 : 0;
        }
      }
      // Drain: wait until the last loads this thread issued have landed, so no
      // copy into shared memory is in flight when the block exits (pair mode:
      // the even CTA's barriers count both CTAs' bytes, so it drains for both,
      // before the cluster barrier that precedes either CTA's exit).
      long long pending = issued < C::STAGES ? issued : C::STAGES;
      if (PAIR && rank != 0) pending = 0;
      int st = stage;
      uint32_t ph = phase;
      for (long long i = 0; i < pending; ++i) {
        if (--st < 0) {
          st = C::STAGES - 1;
          ph ^= 1;
        }
        gb::mbar_wait_bounded(&full[st], ph, p.wait_ns, p.err);
      }
    }
  } else if (warp == 1) {
    if (lane == 0 && rank == 0) {
      // ---------------- MMA issuer ----------------
      // The loop is compiled once per (narrow-channel, chunked-accumulation,
      // k-step group) combination and chosen once: a run-time choice made per
      // MMA between two descriptor forms measured 4% slower on the 256-column
      // SM-pair layer.
      constexpr int MM = PAIR ? 2 * BM : BM;  // pair: M spans both CTAs' A tiles
      const uint32_t IDESC = gb::idesc_f16(MM, BN, TF32 ? 2 : (MODE == MODE_CONV ? 1 : p.ab_type));
      auto issue = [&](auto narrow_tag, auto chunked_tag, auto group_tag) {
        constexpr bool NARROW = MODE == MODE_CONV && decltype(narrow_tag)::value;
        constexpr bool CHUNKED = decltype(chunked_tag)::value;
        constexpr int G = decltype(group_tag)::value;  // stages per round of waits
        int stage = 0;
        uint32_t phase = 0;
        int acc = 0;
        uint32_t acc_phase = 0;
        for (int u = unit0; u < num_units; u += ustep) {
          int t, noff, width;
          decode(u, t, noff, width);
          const uint32_t idesc_u = width == BN ? IDESC : gb::idesc_f16(MM, width, TF32 ? 2 : 1);
          if (!gb::mbar_wait_bounded(&tempty[acc], acc_phase ^ 1, p.wait_ns, p.err)) return;
          gb::tc_fence_after();
          uint32_t d = tmem_base + acc * p.acc_cols;
          const int bt = t / tiles_per_batch;
          const int kbeg = MODE == MODE_CONV ? bt * p.kchunk : 0;
          const int kend = MODE == MODE_CONV ? min(p.kiters, kbeg + p.kchunk) : p.kiters;
          int kin = 0;  // k-steps into the current accumulator block
          for (int it = kbeg; it < kend; it += G) {
            // G consecutive stages (a group starts on a stage that is a multiple
            // of G, so it does not wrap): their descriptors, then one round of
            // waits.  The descriptors are built once per stage and an MMA's are
            // these plus a constant (the start address counts 16-byte units),
            // which keeps the issuing thread's work per MMA small (it bounds
            // MMAs of N <= 128)
            uint64_t ad[G], bd[G];
#pragma unroll
            for (int g = 0; g < G; ++g) {
              const uint32_t a0 = gb::smem_u32(sA + (stage + g) * C::A_BYTES);
              ad[g] = NARROW ? gb::noswz_kmajor_desc(a0, BM * 16, 128) : gb::sw128_kmajor_desc(a0);
              bd[g] = gb::sw128_kmajor_desc(gb::smem_u32(sB + (stage + g) * C::B_BYTES));
            }
#pragma unroll
            for (int g = 0; g < G; ++g)
              if (!gb::mbar_wait_bounded(&full[stage + g], phase, p.wait_ns, p.err)) return;
            gb::tc_fence_after();
#pragma unroll
            for (int g = 0; g < G; ++g) {
              if (CHUNKED && kin == p.kch) {  // chunked accumulation: the next BN-column block
                kin = 0;
                d += BN;
              }
#pragma unroll
              for (int k = 0; k < 4; ++k) {  // 4 MMAs of 32 bytes of K per 128-byte row
                // narrow mode: two taps (2 x 2 KB boxes) per 16-wide k; core matrices
                // are 128 bytes apart along M and one box (2 KB) apart along K
                const uint64_t adesc = ad[g] + (uint64_t)(NARROW ? k * 2 * (BM * 16) / 16 : k * 2);
                const uint64_t bdesc = bd[g] + (uint64_t)(k * 2);
                const uint32_t accum = (kin > 0 || k > 0) ? 1u : 0u;
                if constexpr (TF32)
                  gb::tc_mma_tf32(d, adesc, bdesc, idesc_u, accum);
                else if constexpr (PAIR)
                  gb::tc_mma_f16_pair(d, adesc, bdesc, idesc_u, accum);
                else
                  gb::tc_mma_f16(d, adesc, bdesc, idesc_u, accum);
              }
              ++kin;
            }
            // the group's stages are free once its MMAs complete (the producer
            // waits on the last stage's barrier for each of them)
            if constexpr (PAIR)
              gb::tc_commit_pair_multicast(&empty[stage + G - 1], 0x3);  // both CTAs' stages
            else
              gb::tc_commit(&empty[stage + G - 1]);
            stage += G;
            if (stage == C::STAGES) {
              stage = 0;
              phase ^= 1;
            }
          }
          if constexpr (PAIR)
            gb::tc_commit_pair_multicast(&tfull[acc], 0x3);
          else
            gb::tc_commit(&tfull[acc]);
          if (++acc == p.nacc) {
            acc = 0;
            acc_phase ^= 1;
          }
        }
      };
      using T = std::true_type;
      using F = std::false_type;
      using G1 = std::integral_constant<int, 1>;
      using G2 = std::integral_constant<int, 2>;
      const bool chunked = p.kch < p.kiters;
      auto run_group = [&](auto narrow_tag, auto chunked_tag) {
        if constexpr (kGroupable<C>) {
          if (p.kgroup == 2) {
            issue(narrow_tag, chunked_tag, G2{});
            return;
          }
        }
        issue(narrow_tag, chunked_tag, G1{});
      };
      if (MODE == MODE_CONV && p.narrow) {
        if (chunked) run_group(T{}, T{});
        else run_group(T{}, F{});
      } else {
        if (chunked) run_group(F{}, T{});
        else run_group(F{}, F{});
      }
      // All MMAs issued by this thread have completed once mma_done fires.
      if constexpr (PAIR)
        gb::tc_commit_pair_multicast(mma_done, 0x1);
      else
        gb::tc_commit(mma_done);
      gb::mbar_wait_bounded(mma_done, 0, p.wait_ns, p.err);
    }
  } else {
    // ---------------- epilogue (warps 2..5) ----------------
    const int q = warp & 3;  // TMEM lane quarter this warp may access
    int acc = 0;
    uint32_t acc_phase = 0;
    uint32_t epi_count = 0;  // staging boxes used by this warp (alternating pair)
    uint32_t rphase = 0;     // bit b: parity of the next completion of box b's barrier
    // number of 64-column sub-blocks of work unit u that hold output columns
    auto nsub = [&](int u) {
      int t, noff, width;
      decode(u, t, noff, width);
      const int ntt = (t % tiles_per_batch) % p.n_tiles;
      const int rem = p.K - (ntt * BN + noff);
      const int s64 = rem > 0 ? (rem + 63) / 64 : 0;
      return s64 < width / 64 ? s64 : width / 64;
    };
    // work unit uu's first output column and this warp's first row in it: the
    // decode's divisions cost hundreds of cycles on this one warp, so the bf16
    // path takes them once per unit, for the next unit, before the accumulator
    // wait (not once per 64-column sub-block)
    auto unit_pos = [&](int uu, int& ncol, int& mrow) {
      int t2, noff2, w2;
      decode(uu, t2, noff2, w2);
      const int tt2 = t2 % tiles_per_batch;
      ncol = (tt2 % p.n_tiles) * BN + noff2;
      mrow = m_tile(tt2) * BM + q * 32;
    };
    // residual box (64 columns x 32 rows) of sub-block j of the unit at (ncol, mrow) -> box b
    auto fetch_res = [&](int ncol, int mrow, int j, int b) {
      uint64_t* bar = &rbar[q * 2 + b];
      gb::mbar_arrive_expect_tx(bar, C::EPI_BOX);
      asm volatile(
          "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
          " [%0], [%1, {%2, %3}], [%4];" ::"r"(gb::smem_u32(sEpi + (q * 2 + b) * C::EPI_BOX)),
          "l"(reinterpret_cast<uint64_t>(&tm_r)), "r"(ncol + j * 64), "r"(mrow),
          "r"(gb::smem_u32(bar))
          : "memory");
    };
    const bool has_res = MODE == MODE_CONV && p.res != nullptr && p.part == nullptr;
    // bias of output columns (2 lane, 2 lane + 1) of sub-block j of the unit
    // whose first column is ncol (bf16 epilogue; s2d4: bias of channel c % K)
    auto bias_pair = [&](int ncol, int j) {
      const int nc = ncol + j * 64 + 2 * lane;
      const int bc = p.s2d4_k ? nc % p.s2d4_k : nc;
      float2 bv = make_float2(0.f, 0.f);
      if (p.bias && nc < p.K) bv = make_float2(__ldg(p.bias + bc), __ldg(p.bias + bc + 1));
      return bv;
    };
    asm volatile("griddepcontrol.wait;" ::: "memory");  // see the producer
    int ncol_n = 0, mrow_n = 0;  // the next unit's position (here: the first unit's)
    if (unit0 < num_units) unit_pos(unit0, ncol_n, mrow_n);
    float2 bias_next = make_float2(0.f, 0.f);
    if (!TF32 && MODE == MODE_CONV && !p.i8_y && !p.part && unit0 < num_units)
      bias_next = bias_pair(ncol_n, 0);
    int pending = -1;  // box with a residual load not yet waited for
    if (has_res && unit0 < num_units) {
      if (lane == 0) fetch_res(ncol_n, mrow_n, 0, 0);
      pending = 0;
    }
    // pair mode: the even CTA's accumulator-free barriers
    const uint32_t tempty_pair = PAIR ? gb::mapa_shared(gb::smem_u32(tempty), 0) : 0u;
    for (int u = unit0; u < num_units; u += ustep) {
      int t, noff, width;
      decode(u, t, noff, width);
      const int bt = t / tiles_per_batch;
      const int tt = t % tiles_per_batch;
      const int mt = m_tile(tt), nt = tt % p.n_tiles;
      const int ncol = ncol_n, mrow = mrow_n;  // this unit's position
      const int un = u + ustep;                // the next unit
      if (un < num_units) unit_pos(un, ncol_n, mrow_n);
      if (!gb::mbar_wait_bounded(&tfull[acc], acc_phase, p.wait_ns, p.err)) break;
      gb::tc_fence_after();
      if (MODE == MODE_CONV && !LIGHT && p.pf_x != nullptr && u + 2 * ustep < num_units) {
        // The first k-steps of a unit read its pixels from DRAM (later taps hit
        // L2), and a wave's units all start at once: touching them a unit ahead
        // spreads those reads over the previous unit.  Plain prefetches from
        // these warps leave the TMA unit and the producer thread alone.  Not in
        // the shallow two-CTA kernels: their epilogue is the bound (ResNet-50
        // measured 4 % slower with it there).
        int t2, n2, w2;
        decode(u + 2 * ustep, t2, n2, w2);
        const int tt2 = t2 % tiles_per_batch;
        if (n2 == 0 && tt2 % p.n_tiles == 0) {  // other column units share the rows
          const long long m2 = (long long)m_tile(tt2) * BM + q * 32 + lane;
          if (m2 < p.M) {
            const int img2 = (int)(m2 / ohow);
            const int rem2 = (int)(m2 - (long long)img2 * ohow);
            const int oh2 = rem2 / p.OW, ow2 = rem2 - oh2 * p.OW;
            const int ih = oh2 * p.stride - p.pad + p.pf_dh, iw = ow2 * p.stride - p.pad + p.pf_dw;
            if (ih >= 0 && ih < p.H && iw >= 0 && iw < p.W) {
              const uint8_t* a = p.pf_x + (((long long)img2 * p.H + ih) * p.W + iw) * p.pf_pix;
              for (int l = 0; l < p.pf_row; l += 128)
                asm volatile("prefetch.global.L2 [%0];" ::"l"(a + l));
            }
          }
        }
      }
      const long long m = (long long)mt * BM + q * 32 + lane;
      const bool row_ok = m < p.M;
      const uint32_t tbase = tmem_base + ((uint32_t)(q * 32) << 16) + acc * p.acc_cols;
      if constexpr (TF32) {
        // fp32 NHWC output: 32-column sub-blocks -> + bias (+ residual) ->
        // activation -> a 128-byte-swizzled 32 x 32 fp32 box per warp -> TMA store
        const long long m_warp = (long long)mt * BM + q * 32;
        const int remk = p.K - (nt * BN + noff);
        int ns32 = remk > 0 ? (remk + 31) / 32 : 0;
        if (ns32 > width / 32) ns32 = width / 32;
        float* sbias = reinterpret_cast<float*>(sEpi + 4 * 2 * C::EPI_BOX + q * 256);
#pragma unroll 1
        for (int j = 0; j < ns32; ++j) {
          const int nb0 = nt * BN + noff + j * 32;
          uint8_t* box = sEpi + (q * 2 + (epi_count & 1)) * C::EPI_BOX;
          if (lane == 0) gb::bulk_wait_read<1>();  // the store that last used this box
          __syncwarp();
          uint32_t r[32];
          gb::tmem_ld_x16(tbase + j * 32, *reinterpret_cast<uint32_t(*)[16]>(&r[0]));
          gb::tmem_ld_x16(tbase + j * 32 + 16, *reinterpret_cast<uint32_t(*)[16]>(&r[16]));
          sbias[lane] = (p.bias && nb0 + lane < p.K) ? __ldg(p.bias + nb0 + lane) : 0.f;
          __syncwarp();
          gb::tmem_ld_wait();
          float v[32];
#pragma unroll
          for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]) + sbias[i];
          if (p.res_f32 && row_ok) {
            const float4* rp = reinterpret_cast<const float4*>(p.res_f32 + m * p.K + nb0);
#pragma unroll
            for (int h = 0; h < 8; ++h) {
              if (nb0 + 4 * h >= p.K) break;
              const float4 rv = __ldg(rp + h);
              v[4 * h] += rv.x;
              v[4 * h + 1] += rv.y;
              v[4 * h + 2] += rv.z;
              v[4 * h + 3] += rv.w;
            }
          }
#pragma unroll
          for (int h = 0; h < 8; ++h)
            *reinterpret_cast<float4*>(box + lane * 128 + ((h ^ (lane & 7)) << 4)) =
                make_float4(act_apply(v[4 * h], p.act), act_apply(v[4 * h + 1], p.act),
                            act_apply(v[4 * h + 2], p.act), act_apply(v[4 * h + 3], p.act));
          gb::fence_proxy_async_smem();  // staging writes -> visible to the TMA engine
          __syncwarp();
          if (lane == 0) {
            gb::tma_store_2d(&tm_y, box, nb0, (int)m_warp);
            gb::bulk_commit();
          }
          ++epi_count;
        }
      } else if (MODE == MODE_CONV && p.i8_y && p.i8_nch > 0) {
        // exact int8, chunked accumulation: output channel column j of the unit
        // has i8_nch partial sums, one per BN-column accumulator block, each an
        // exact integer in fp32 (at most 1024 products of int8 values); their
        // int32 sum + bias is requantised to int8 (the MegEngine Beta report's
        // native int8 epilogue).  This group's 64 biases and scales are staged in
        // the warp's (here unused) staging box and read back as broadcasts.
        int32_t* sbi = reinterpret_cast<int32_t*>(sEpi + q * 2 * C::EPI_BOX);
        float* ssc = reinterpret_cast<float*>(sbi + 64);
#pragma unroll 1
        for (int g = 0; g < width / 64; ++g) {
          const int k0 = nt * BN + noff + g * 64;  // first output channel of the group
          if (k0 >= p.i8_kout) break;
          __syncwarp();  // the previous group's reads of the slice are done
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const int kk = k0 + h * 32 + lane;
            const bool in = kk < p.i8_kout;
            sbi[h * 32 + lane] = (in && p.i8_bias) ? __ldg(p.i8_bias + kk) : 0;
            ssc[h * 32 + lane] = in ? __ldg(p.i8_scale + kk) : 0.f;
          }
          __syncwarp();
#pragma unroll 1
          for (int c8 = 0; c8 < 8; ++c8) {
            const int kb = k0 + c8 * 8;
            if (kb >= p.i8_kout) break;  // i8_kout % 16 == 0
            int tv[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) tv[i] = sbi[c8 * 8 + i];
            // two blocks' loads in flight per wait (the block count is
            // warp-uniform, so every lane takes the same loads)
#pragma unroll 1
            for (int c0 = 0; c0 < p.i8_nch; c0 += 2) {
              uint32_t v0[8], v1[8];
              const bool two = c0 + 1 < p.i8_nch;
              gb::tmem_ld_x8(tbase + c0 * BN + g * 64 + c8 * 8, v0);
              if (two) gb::tmem_ld_x8(tbase + (c0 + 1) * BN + g * 64 + c8 * 8, v1);
              gb::tmem_ld_wait();
#pragma unroll
              for (int i = 0; i < 8; ++i)
                tv[i] += __float2int_rn(__uint_as_float(v0[i])) +
                         (two ? __float2int_rn(__uint_as_float(v1[i])) : 0);
            }
            uint32_t pk[2] = {0u, 0u};
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              int qv = __float2int_rn(__fmul_rn(__int2float_rn(tv[i]), ssc[c8 * 8 + i]));
              qv = qv > 127 ? 127 : (qv < -128 ? -128 : qv);
              if (p.i8_relu && qv < 0) qv = 0;
              pk[i >> 2] |= (uint32_t)(qv & 0xff) << (8 * (i & 3));
            }
            if (row_ok) {
              // NHWC: row m, channel kb; NC32HW32: block kb/32 of image m / (OH*OW)
              long long off = m * p.i8_kout + kb;
              if (p.i8_nc32) {
                const long long ohw = (long long)p.OH * p.OW, img = m / ohw;
                off = ((img * (p.i8_kout / 32) + kb / 32) * ohw + (m - img * ohw)) * 32 + (kb & 31);
              }
              *reinterpret_cast<uint2*>(p.i8_y + off) = make_uint2(pk[0], pk[1]);
            }
          }
        }
      } else if (MODE == MODE_CONV && p.i8_y) {
        // exact int8: each 128-column group of the tile holds 64 sums against
        // the low weight nibbles, then 64 against the high parts, all exact
        // integers in fp32; t = 16 * hi + lo + bias, requantised to int8 (the
        // MegEngine Beta report's native int8 epilogue)
        // this group's 64 biases and scales, staged once in the warp's (here
        // unused) staging box and read back as broadcasts
        int32_t* sbi = reinterpret_cast<int32_t*>(sEpi + q * 2 * C::EPI_BOX);
        float* ssc = reinterpret_cast<float*>(sbi + 64);
#pragma unroll 1
        for (int g = 0; g < width / 128; ++g) {
          const int k0 = (nt * BN + noff + g * 128) / 2;  // first output channel of the group
          if (k0 >= p.i8_kout) break;
          __syncwarp();  // the previous group's reads of the slice are done
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const int kk = k0 + h * 32 + lane;
            sbi[h * 32 + lane] = p.i8_bias ? __ldg(p.i8_bias + kk) : 0;
            ssc[h * 32 + lane] = __ldg(p.i8_scale + kk);
          }
          __syncwarp();
#pragma unroll 1
          for (int c16 = 0; c16 < 4; ++c16) {
            uint32_t lo[16], hi[16];
            gb::tmem_ld_x16(tbase + g * 128 + c16 * 16, lo);
            gb::tmem_ld_x16(tbase + g * 128 + 64 + c16 * 16, hi);
            gb::tmem_ld_wait();
            const int kb = k0 + c16 * 16;
            uint32_t pk[4] = {0u, 0u, 0u, 0u};
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const int tv = 16 * __float2int_rn(__uint_as_float(hi[i])) +
                             __float2int_rn(__uint_as_float(lo[i])) + sbi[c16 * 16 + i];
              int qv = __float2int_rn(__fmul_rn(__int2float_rn(tv), ssc[c16 * 16 + i]));
              qv = qv > 127 ? 127 : (qv < -128 ? -128 : qv);
              if (p.i8_relu && qv < 0) qv = 0;
              pk[i >> 2] |= (uint32_t)(qv & 0xff) << (8 * (i & 3));
            }
            if (row_ok) {
              // NHWC: row m, channel kb; NC32HW32: block kb/32 of image m / (OH*OW)
              long long off = m * p.i8_kout + kb;
              if (p.i8_nc32) {
                const long long ohw = (long long)p.OH * p.OW, img = m / ohw;
                off = ((img * (p.i8_kout / 32) + kb / 32) * ohw + (m - img * ohw)) * 32 + (kb & 31);
              }
              *reinterpret_cast<uint4*>(p.i8_y + off) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
            }
          }
        }
      } else if (MODE == MODE_BATCHED || p.part) {
        // fp32 outputs (batched products, split-K partials): 32-column boxes of
        // 32 rows staged with the 128-byte swizzle and written by TMA stores
        // through the fp32 map passed in the tm_r slot
        const long long m_warp = (long long)mt * BM + q * 32;
#pragma unroll 1
        for (int j = 0; j < BN / 32; ++j) {
          const int nb0 = nt * BN + j * 32;
          if (nb0 >= p.K) break;
          uint8_t* box = sEpi + (q * 2 + (epi_count & 1)) * C::EPI_BOX;
          if (lane == 0) gb::bulk_wait_read<1>();
          __syncwarp();
          uint32_t r[32];
          gb::tmem_ld_x16(tbase + j * 32, *reinterpret_cast<uint32_t(*)[16]>(&r[0]));
          gb::tmem_ld_x16(tbase + j * 32 + 16, *reinterpret_cast<uint32_t(*)[16]>(&r[16]));
          gb::tmem_ld_wait();
#pragma unroll
          for (int h = 0; h < 8; ++h)
            *reinterpret_cast<uint4*>(box + lane * 128 + ((h ^ (lane & 7)) << 4)) =
                make_uint4(r[4 * h], r[4 * h + 1], r[4 * h + 2], r[4 * h + 3]);
          gb::fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            gb::tma_store_3d(&tm_r, box, nb0, (int)m_warp, bt);
            gb::bulk_commit();
          }
          ++epi_count;
        }
        (void)row_ok;
      } else {
        // 64-column sub-blocks: TMEM -> registers (+ bias, residual, act) ->
        // swizzled staging box in shared memory -> TMA store of 32 rows x 64 cols
        const long long m_warp = (long long)mt * BM + q * 32;
        const int ns = nsub(u);
#pragma unroll 1
        for (int j = 0; j < ns; ++j) {
          const int cur = epi_count & 1;
          uint8_t* box = sEpi + (q * 2 + cur) * C::EPI_BOX;
          const int nb0 = ncol + j * 64;
          // the sub-block after this one: (this unit, j + 1) or (the next unit, 0)
          const bool same = j + 1 < ns;
          const bool has_nx = same || un < num_units;
          const int ncol_x = same ? ncol : ncol_n, jx = same ? j + 1 : 0;
          if (has_res) {
            // prefetch the next sub-block's residual into the other box once the
            // store that last read that box is done with it
            if (has_nx && lane == 0) {
              gb::bulk_wait_read<0>();
              fetch_res(ncol_x, same ? mrow : mrow_n, jx, cur ^ 1);
            }
            if (!gb::mbar_wait_bounded(&rbar[q * 2 + cur], (rphase >> cur) & 1, p.wait_ns, p.err))
              break;
            rphase ^= 1u << cur;
            pending = has_nx ? (cur ^ 1) : -1;
          } else {
            if (lane == 0) gb::bulk_wait_read<1>();  // the store that last used this box
            __syncwarp();
          }
          uint32_t r[64];
#pragma unroll
          for (int c16 = 0; c16 < 4; ++c16) {
            uint32_t (&rr)[16] = *reinterpret_cast<uint32_t(*)[16]>(&r[c16 * 16]);
            gb::tmem_ld_x16(tbase + j * 64 + c16 * 16, rr);  // accumulator column = nb0 - tile n0
          }
          // this sub-block's 64 bias values (loaded one sub-block ahead, two per
          // lane) staged for broadcast reads; then the next sub-block's are loaded
          float* sbias = reinterpret_cast<float*>(sEpi + 4 * 2 * C::EPI_BOX + q * 256);
          reinterpret_cast<float2*>(sbias)[lane] = bias_next;
          if (has_nx) bias_next = bias_pair(ncol_x, jx);
          __syncwarp();
          gb::tmem_ld_wait();
          if (p.act == 0)
            epi_bf16_subblock<0>(r, sbias, box, lane, has_res);
          else if (p.act == 1)
            epi_bf16_subblock<1>(r, sbias, box, lane, has_res);
          else
            epi_bf16_subblock<2>(r, sbias, box, lane, has_res);
          gb::fence_proxy_async_smem();  // staging writes -> visible to the TMA engine
          __syncwarp();
          if (lane == 0) {
            if (p.s2d4_k) {
              // rows are 4x4 blocks (n, bh, bw), bw fastest; 8-row pieces of the
              // box (8 divides the block-grid width, so a piece stays in one block
              // row and starts on a swizzle-atom boundary) go to output pixels
              // (2 bh + py, 2 bw + px) for bw = bw0 .. bw0 + 7
              const int g = nb0 / p.s2d4_k;
#pragma unroll 1
              for (int r8 = 0; r8 < 4; ++r8) {
                const long long row = m_warp + r8 * 8;
                if (row >= p.M) break;
                gb::tma_store_5d(&tm_y, box + r8 * 1024, 0, g & 1, (int)(row % p.OW), g >> 1,
                                 (int)(row / p.OW));
              }
            } else {
              gb::tma_store_2d(&tm_y, box, nb0, (int)m_warp);
            }
            gb::bulk_commit();
          }
          ++epi_count;
        }
        (void)row_ok;
      }
      gb::tc_fence_before();
      if constexpr (PAIR) {
        __syncwarp();  // every lane's accumulator reads are complete
        if (lane == 0) {
          if (rank == 0)
            gb::mbar_arrive(&tempty[acc]);
          else
            gb::mbar_arrive_cluster(tempty_pair + acc * 8);
        }
      } else {
        gb::mbar_arrive(&tempty[acc]);
      }
      if (++acc == p.nacc) {
        acc = 0;
        acc_phase ^= 1;
      }
    }
    if (lane == 0) {
      gb::bulk_wait_all();  // TMA stores done before exit
      // after a wait ran out, a residual load may still be landing
      if (pending >= 0)
        gb::mbar_wait_bounded(&rbar[q * 2 + pending], (rphase >> pending) & 1, p.wait_ns, p.err);
    }
  }

  gb::tc_fence_before();
  __syncthreads();
  // pair mode: neither CTA frees its TMEM or exits while the even CTA's MMAs,
  // commits or drain may still touch the other's shared memory or TMEM
  if constexpr (PAIR) gb::cluster_sync();
  if (warp == 0) {
    gb::tc_fence_after();
    if constexpr (PAIR)
      gb::tmem_dealloc_pair(tmem_base, C::TMEM_COLS);
    else
      gb::tmem_dealloc(tmem_base, p.tmem_cols);
  }
}

// ---- row-strip implicit GEMM (one input strip per tile, taps by descriptor offset) ----
//
// For stride-1 convolutions over at most 64 channels into at most 64 output
// channels (ResNet-50's 56x56 stage), the im2col loads of the general kernel
// fetch every input pixel once per filter tap.  Here an output row is padded
// to a "virtual" row of Wv pixels (the smallest power of two >= OW + S - 1),
// a 128-row tile is RT = 128 / Wv whole output rows, and ONE tiled TMA load
// brings the RT + R - 1 input rows the tile needs (Wv pixels each, starting at
// column -pad, zeros outside the image) into shared memory with the 128-byte
// swizzle.  Output pixel (i, x) of the tile under filter tap (r, s) reads strip
// row (r + i) * Wv + x + s = m + r * Wv + s for tile row m = i * Wv + x: the A
// operand of tap (r, s) is the strip itself, its start moved by r * Wv + s
// rows (the tensor core applies the 128-byte swizzle to absolute shared-memory
// addresses, so any 128-byte row is a valid start).  Virtual pixels x >= OW
// are computed and dropped by the output map's bounds.  The R*S weight tiles
// (64 output channels x 64 input channels each) stay resident for the whole
// launch.  L2 -> SM bytes per tile: one strip instead of R*S im2col boxes.
namespace strip {
constexpr int STAGES = 3;
constexpr int SLOT = 32 * 1024;          // strip bytes (Wv x rows x 128 B) at most
constexpr int MAXTAPS = 9;
constexpr int W_BYTES = MAXTAPS * 64 * 128;
constexpr int EPI_BOX = 32 * 128;
constexpr int SMEM = W_BYTES + STAGES * SLOT + 4 * 2 * EPI_BOX + 4 * 256 + 256 + 1024;
}  // namespace strip

struct StripParams {
  int OH, OW, K, S, taps, Wv, RT, tiles_per_img, m_tiles, strip_bytes, act;
  const float* bias;
  int* err;
  unsigned long long wait_ns;
  // exact int8 output (i8_y set; bias / act above unused): the sums are exact
  // integers (at most 9 x 64 products of int8 values, below 2^24 in size);
  // + i8_bias in int32, requantised with i8_scale (fp32, round to nearest
  // even), clamped to int8, optional ReLU, stored NHWC or NC32HW32
  int8_t* i8_y;
  const int32_t* i8_bias;
  const float* i8_scale;
  int i8_relu, i8_nc32;
};

template <int ACT>
__global__ void __launch_bounds__(192, 1)
    igemm_strip_kernel(const __grid_constant__ CUtensorMap tm_x,
                       const __grid_constant__ CUtensorMap tm_w,
                       const __grid_constant__ CUtensorMap tm_y, const StripParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* sW = smem;
  uint8_t* sS = smem + strip::W_BYTES;
  uint8_t* sEpi = sS + strip::STAGES * strip::SLOT;
  float* sBias = reinterpret_cast<float*>(sEpi + 4 * 2 * strip::EPI_BOX);
  uint64_t* bars = reinterpret_cast<uint64_t*>(sBias + 4 * 64);
  uint64_t* full = bars;
  uint64_t* empty = bars + strip::STAGES;
  uint64_t* tfull = bars + 2 * strip::STAGES;
  uint64_t* tempty = tfull + 2;
  uint64_t* wbar = tempty + 2;
  uint64_t* mma_done = wbar + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(mma_done + 1);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < strip::STAGES; ++s) {
      gb::mbar_init(&full[s], 1);
      gb::mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      gb::mbar_init(&tfull[b], 1);
      gb::mbar_init(&tempty[b], 128);
    }
    gb::mbar_init(wbar, 1);
    gb::mbar_init(mma_done, 1);
    gb::fence_barrier_init();
    gb::tma_prefetch_desc(&tm_x);
    gb::tma_prefetch_desc(&tm_w);
    gb::tma_prefetch_desc(&tm_y);
  }
  if (warp == 0) {
    gb::tmem_alloc(tmem_slot, 128);  // two 64-column accumulators
    gb::tmem_relinquish();
  }
  gb::tc_fence_before();
  __syncthreads();
  gb::tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  // dependent launch as in the general kernel: the producer and the epilogue
  // warps wait for the previous grid before their first global access, the
  // MMA thread not at all
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  // tile t: image t / tiles_per_img, output rows oh0 .. oh0 + RT - 1
  auto tile_pos = [&](int t, int& n, int& oh0) {
    n = t / p.tiles_per_img;
    oh0 = (t - n * p.tiles_per_img) * p.RT;
  };

  if (warp == 0) {
    if (lane == 0) {
      // ---- producer: the weight tiles once, then one input strip per tile ----
      gb::mbar_arrive_expect_tx(wbar, p.taps * 64 * 128);
      asm volatile("griddepcontrol.wait;" ::: "memory");
      for (int tap = 0; tap < p.taps; ++tap)
        gb::tma_load_2d(sW + tap * 64 * 128, &tm_w, wbar, tap * 64, 0);
      int stage = 0;
      uint32_t phase = 0;
      long long issued = 0;
      const int pad = (p.S - 1) / 2;
      for (int t = blockIdx.x; t < p.m_tiles; t += gridDim.x) {
        if (!gb::mbar_wait_bounded(&empty[stage], phase ^ 1, p.wait_ns, p.err)) break;
        int n, oh0;
        tile_pos(t, n, oh0);
        gb::mbar_arrive_expect_tx(&full[stage], p.strip_bytes);
        gb::tma_load_4d(sS + stage * strip::SLOT, &tm_x, &full[stage], 0, -pad, oh0 - pad, n);
        ++issued;
        if (++stage == strip::STAGES) {
          stage = 0;
          phase ^= 1;
        }
      }
      // no copy into shared memory may be in flight when the block exits
      gb::mbar_wait_bounded(wbar, 0, p.wait_ns, p.err);
      long long pending = issued < strip::STAGES ? issued : strip::STAGES;
      int st = stage;
      uint32_t ph = phase;
      for (long long i = 0; i < pending; ++i) {
        if (--st < 0) {
          st = strip::STAGES - 1;
          ph ^= 1;
        }
        gb::mbar_wait_bounded(&full[st], ph, p.wait_ns, p.err);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ---- MMA issuer: per tile, every tap's product from the one strip ----
      constexpr uint32_t IDESC = gb::idesc_f16(128, 64, 1);
      bool ok = gb::mbar_wait_bounded(wbar, 0, p.wait_ns, p.err);
      gb::tc_fence_after();
      // One tile's 36 (or fewer) MMAs are issued from fully unrolled tap loops,
      // each descriptor its base plus a constant: with N = 64 an MMA takes 48
      // cycles, and the issuing thread is the bound (run-time tap loops that
      // built every descriptor measured 91 cycles per MMA, 3,290 per 3x3 tile).
      const uint64_t bdesc0 = gb::sw128_kmajor_desc(gb::smem_u32(sW));
      const uint32_t row_units = (uint32_t)p.Wv * 8;  // one strip row of Wv pixels, in 16-byte units
      auto run = [&](auto r_tag, auto s_tag) {
        constexpr int R = decltype(r_tag)::value, S = decltype(s_tag)::value;
        int stage = 0;
        uint32_t phase = 0;
        int acc = 0;
        uint32_t acc_phase = 0;
        for (int t = blockIdx.x; t < p.m_tiles && ok; t += gridDim.x) {
          const uint32_t d = tmem_base + acc * 64;
          const uint64_t adesc0 = gb::sw128_kmajor_desc(gb::smem_u32(sS + stage * strip::SLOT));
          if (!gb::mbar_wait_bounded(&tempty[acc], acc_phase ^ 1, p.wait_ns, p.err)) break;
          if (!gb::mbar_wait_bounded(&full[stage], phase, p.wait_ns, p.err)) break;
          gb::tc_fence_after();
          // taps in filter order: row r of the strip is r * Wv pixels (128 bytes
          // each) down, column sx one pixel along; each tap's weights are 64
          // rows; K advances 32 bytes per MMA (descriptor units of 16 bytes)
#pragma unroll
          for (int r = 0; r < R; ++r) {
            const uint64_t arow = adesc0 + (uint64_t)(r * row_units);
#pragma unroll
            for (int sx = 0; sx < S; ++sx)
#pragma unroll
              for (int k = 0; k < 4; ++k)
                gb::tc_mma_f16(d, arow + (uint64_t)(sx * 8 + k * 2),
                               bdesc0 + (uint64_t)((r * S + sx) * 64 * 8 + k * 2), IDESC,
                               (r | sx | k) ? 1u : 0u);
          }
          gb::tc_commit(&empty[stage]);
          gb::tc_commit(&tfull[acc]);
          if (++stage == strip::STAGES) {
            stage = 0;
            phase ^= 1;
          }
          if (++acc == 2) {
            acc = 0;
            acc_phase ^= 1;
          }
        }
      };
      // a 3x3 or 1x1 filter (checked on the host)
      using I1 = std::integral_constant<int, 1>;
      using I3 = std::integral_constant<int, 3>;
      if (p.taps == 9) run(I3{}, I3{});
      else run(I1{}, I1{});
      gb::tc_commit(mma_done);
      gb::mbar_wait_bounded(mma_done, 0, p.wait_ns, p.err);
    }
  } else {
    // ---- epilogue: bias, activation, bf16, 4-D TMA store (virtual pixels clipped) ----
    const int q = warp & 3;
    float* sbias = sBias + q * 64;
    asm volatile("griddepcontrol.wait;" ::: "memory");
    {
      const int c = 2 * lane;  // the 64 biases (channels >= K read as 0)
      sbias[c] = (p.bias && c < p.K) ? __ldg(p.bias + c) : 0.f;
      sbias[c + 1] = (p.bias && c + 1 < p.K) ? __ldg(p.bias + c + 1) : 0.f;
      __syncwarp();
    }
    // int8 output: the 64 int32 biases and fp32 scales, in this warp's (then
    // unused) staging boxes, read back as broadcasts
    int32_t* sbi = reinterpret_cast<int32_t*>(sEpi + q * 2 * strip::EPI_BOX);
    float* ssc = reinterpret_cast<float*>(sbi + 64);
    if (p.i8_y) {
      for (int c = lane; c < 64; c += 32) {
        sbi[c] = (p.i8_bias && c < p.K) ? __ldg(p.i8_bias + c) : 0;
        ssc[c] = c < p.K ? __ldg(p.i8_scale + c) : 0.f;
      }
      __syncwarp();
    }
    int acc = 0;
    uint32_t acc_phase = 0;
    uint32_t epi_count = 0;
    for (int t = blockIdx.x; t < p.m_tiles; t += gridDim.x) {
      if (!gb::mbar_wait_bounded(&tfull[acc], acc_phase, p.wait_ns, p.err)) break;
      gb::tc_fence_after();
      uint8_t* box = sEpi + (q * 2 + (epi_count & 1)) * strip::EPI_BOX;
      if (!p.i8_y) {
        if (lane == 0) gb::bulk_wait_read<1>();  // the store that last used this box
        __syncwarp();
      }
      uint32_t r[64];
      const uint32_t tb = tmem_base + ((uint32_t)(q * 32) << 16) + acc * 64;
#pragma unroll
      for (int c16 = 0; c16 < 4; ++c16)
        gb::tmem_ld_x16(tb + c16 * 16, *reinterpret_cast<uint32_t(*)[16]>(&r[c16 * 16]));
      gb::tmem_ld_wait();
      gb::tc_fence_before();
      gb::mbar_arrive(&tempty[acc]);
      if (p.i8_y) {
        // this lane's output pixel (tile row q * 32 + lane); virtual pixels
        // (ow >= OW) and rows past the image are dropped
        int n, oh0;
        tile_pos(t, n, oh0);
        const int row = q * 32 + lane, rr = row / p.Wv;
        const int oh = oh0 + rr, ow = row - rr * p.Wv;
        if (ow < p.OW && oh < p.OH) {
          const long long pix = ((long long)n * p.OH + oh) * p.OW + ow;
#pragma unroll
          for (int c16 = 0; c16 < 4; ++c16) {
            if (c16 * 16 >= p.K) break;  // K % 16 == 0
            uint32_t pk[4] = {0u, 0u, 0u, 0u};
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const int c = c16 * 16 + i;
              const int tv = __float2int_rn(__uint_as_float(r[c])) + sbi[c];
              int qv = __float2int_rn(__fmul_rn(__int2float_rn(tv), ssc[c]));
              qv = qv > 127 ? 127 : (qv < -128 ? -128 : qv);
              if (p.i8_relu && qv < 0) qv = 0;
              pk[i >> 2] |= (uint32_t)(qv & 0xff) << (8 * (i & 3));
            }
            // NHWC: pixel-major; NC32HW32: 32-channel blocks of the image
            const long long off =
                p.i8_nc32 ? (((long long)n * (p.K / 32) + c16 / 2) * p.OH * p.OW +
                             (long long)oh * p.OW + ow) * 32 + (c16 & 1) * 16
                          : pix * p.K + c16 * 16;
            *reinterpret_cast<uint4*>(p.i8_y + off) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
          }
        }
      } else {
        epi_bf16_subblock<ACT>(r, sbias, box, lane, false);
        gb::fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          int n, oh0;
          tile_pos(t, n, oh0);
          const int row = q * 32;  // this warp's first tile row
          gb::tma_store_4d(&tm_y, box, 0, row % p.Wv, oh0 + row / p.Wv, n);
          gb::bulk_commit();
        }
      }
      ++epi_count;
      if (++acc == 2) {
        acc = 0;
        acc_phase ^= 1;
      }
    }
    if (lane == 0) gb::bulk_wait_all();
  }
  gb::tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    gb::tc_fence_after();
    gb::tmem_dealloc(tmem_base, 128);
  }
}

// wp[k][rs][c] (rs < RS, c < Cp) = w[k][rs][c] for rs < RS_valid and c < C, else 0
__global__ void pack_igemm_weights_kernel(const __nv_bfloat16* __restrict__ w,
                                          __nv_bfloat16* __restrict__ wp, int K, int RS, int C,
                                          int Cp, int RS_valid) {
  const long long total = (long long)K * RS * Cp;
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < total;
       i += (long long)gridDim.x * blockDim.x) {
    const int c = (int)(i % Cp);
    const long long krs = i / Cp;
    const int rs = (int)(krs % RS);
    const long long k = krs / RS;
    wp[i] = (c < C && rs < RS_valid) ? w[(k * RS_valid + rs) * C + c] : __float2bfloat16(0.0f);
  }
}

// Clusters of two CTAs of the pair-mode kernel that fit on the device at once
// (a cluster needs two SMs of one GPU processing cluster); 0 if none.
template <int BN>
int pair_max_clusters(int smem) {
  static int cached[8] = {-1, -1, -1, -1, -1, -1, -1, -1};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 8) return 0;
  if (cached[dev] > 0) return cached[dev];
  // the query needs the kernel's dynamic shared-memory limit raised first
  auto* kern = igemm_bf16_tc_kernel<BN, MODE_CONV, false, false, true>;
  if (gb_set_smem_once(reinterpret_cast<const void*>(kern), smem) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(gb_num_sms() & ~1));
  cfg.blockDim = dim3(192);
  cfg.dynamicSmemBytes = (size_t)smem;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess) n = 0;
  cudaGetLastError();  // clear a failed query
  if (n > 0) cached[dev] = n;  // a failure is not remembered
  return n;
}

template <int BN, bool LIGHT, bool TF32 = false, bool PAIR = false>
cudaError_t launch_bn(const gbconv_desc_s& d, const void* x, const void* wpack, const float* bias,
                      const void* res, void* y, int* err, unsigned long long wait_ns,
                      cudaStream_t st, const IgemmSplit& split) {
  using Cf = Cfg<BN, LIGHT, PAIR>;
  constexpr int BKE = TF32 ? 32 : BK;  // channels per k-step
  constexpr int ES = TF32 ? 4 : 2;     // element bytes
  const CUtensorMapDataType DT =
      TF32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  const bool narrow = !TF32 && d.C == 8;
  const int Cp = gb_ceil_div(d.C, BKE) * BKE;
  IgemmParams p{};
  p.narrow = narrow ? 1 : 0;
  p.taps = d.R * d.S;
  {
    const long long xcs_pf = d.x_cstride ? d.x_cstride : d.C;
    // only for an input of a quarter of L2 or more: a smaller one (the
    // previous layer's output, say) is most likely still in L2 (ResNet-50
    // measured 1 % slower with the prefetch on its 3-13 MB inputs)
    const bool big = (long long)d.N * d.H * d.W * xcs_pf * ES >= gb_l2_bytes() / 4;
    p.pf_x = (narrow || !big) ? nullptr : static_cast<const uint8_t*>(x);  // off for split-K below
    p.pf_pix = xcs_pf * ES;
    p.pf_row = d.C * ES;
    p.pf_dh = (d.R / 2) * d.dil;
    p.pf_dw = (d.S / 2) * d.dil;
  }
  p.H = d.H;
  p.W = d.W;
  p.C = d.C;
  p.K = d.K;
  p.S = d.S;
  p.stride = d.stride;
  p.pad = d.pad;
  p.dil = d.dil;
  p.OH = d.OH;
  p.OW = d.OW;
  p.cblocks = narrow ? 1 : Cp / BKE;
  p.kiters = narrow ? gb_ceil_div(d.R * d.S, 8) : d.R * d.S * p.cblocks;
  p.Kw = narrow ? p.kiters * BK : d.R * d.S * Cp;
  p.M = (long long)d.N * d.OH * d.OW;
  p.m_tiles = (int)gb_ceil_div_ll(p.M, BM);
  if (PAIR) p.m_tiles = gb_ceil_div(p.m_tiles, 2);  // 256-row units
  p.n_tiles = gb_ceil_div(d.K, BN);
  p.act = d.act;
  p.bias = bias;
  p.res = TF32 ? nullptr : static_cast<const __nv_bfloat16*>(res);
  p.res_f32 = TF32 ? static_cast<const float*>(res) : nullptr;
  p.y = static_cast<__nv_bfloat16*>(y);
  p.err = err;
  p.wait_ns = wait_ns;
  p.ksplit = split.ksplit > 1 ? split.ksplit : 1;
  p.kchunk = split.ksplit > 1 ? split.kchunk : p.kiters;
  if (p.ksplit > 1) p.pf_x = nullptr;  // a range of the channels only
  p.part = split.part;
  p.i8_y = split.i8_y;
  p.i8_bias = split.i8_bias;
  p.i8_scale = split.i8_scale;
  p.i8_kout = split.i8_kout;
  p.i8_relu = split.i8_relu;
  p.i8_nc32 = split.i8_nc32;
  // accumulator layout: one BN-column block per tile, or split.i8_nch blocks of
  // at most i8_kch k-steps each (exact int8, chunked); two tile accumulators
  // when they fit so the epilogue overlaps the next tile's MMAs.  A CTA never
  // takes more than its share of the SM's 512 TMEM columns (LIGHT: two CTAs).
  p.i8_nch = p.i8_y ? split.i8_nch : 0;
  p.kch = p.i8_nch > 0 ? split.i8_kch : (1 << 30);
  // k-step pairs: every unit's k-range (kiters, or kchunk-long ranges) even
  p.kgroup = (kGroupable<Cf> && p.kiters % 2 == 0 && (p.ksplit == 1 || p.kchunk % 2 == 0)) ? 2 : 1;
  if (p.i8_y) {
    if (p.ksplit != 1 || p.i8_kout % 16) return cudaErrorInvalidValue;
    if (p.i8_nch == 0 && (BN % 128 != 0 || p.i8_kout * 2 != d.K)) return cudaErrorInvalidValue;
    if (p.i8_nch > 0 && (p.i8_kout != d.K || p.kch < 1 || gb_ceil_div(p.kiters, p.kch) != p.i8_nch))
      return cudaErrorInvalidValue;
  }
  p.acc_cols = p.i8_nch > 0 ? p.i8_nch * BN : BN;
  {
    const int budget = LIGHT ? 256 : 512;
    p.nacc = 2 * p.acc_cols <= budget ? 2 : 1;
    if (p.nacc * p.acc_cols > budget) return cudaErrorInvalidValue;
    uint32_t cols = 32;
    while (cols < (uint32_t)(p.nacc * p.acc_cols)) cols <<= 1;
    p.tmem_cols = cols;
  }
  p.s2d4_k = split.s2d4_k;
  if (p.s2d4_k && (TF32 || res || p.i8_y || p.ksplit != 1 || p.s2d4_k != 64 ||
                   d.K != 4 * p.s2d4_k || d.OW % 8))
    return cudaErrorInvalidValue;
  if (PAIR && (narrow || p.ksplit != 1 || p.part || p.i8_y || p.s2d4_k)) return cudaErrorInvalidValue;

  CUtensorMap tmx, tmw;
  {
    cuuint64_t dims[4] = {(cuuint64_t)d.C, (cuuint64_t)d.W, (cuuint64_t)d.H, (cuuint64_t)d.N};
    const cuuint64_t xcs = d.x_cstride ? d.x_cstride : d.C;  // elements between pixels
    cuuint64_t strides[3] = {xcs * ES, (cuuint64_t)d.W * xcs * ES,
                             (cuuint64_t)d.H * d.W * xcs * ES};
    // Bounding box of the first filter tap's pixel: from -pad to
    // (dim - 1) + pad - dil*(R-1) (R == S is required).
    int lower[2] = {-d.pad, -d.pad};
    const int pad_hi = d.pad + d.pad_hi_delta;  // padding after (equal to pad unless rewritten)
    int upper[2] = {pad_hi - d.dil * (d.S - 1), pad_hi - d.dil * (d.R - 1)};
    cuuint32_t estr[4] = {1, (cuuint32_t)d.stride, (cuuint32_t)d.stride, 1};
    CUresult r = gb_encode_im2col(&tmx, DT, 4, const_cast<void*>(x),
                                  dims, strides, lower, upper, narrow ? 8 : BKE, BM, estr,
                                  narrow ? CU_TENSOR_MAP_SWIZZLE_NONE : CU_TENSOR_MAP_SWIZZLE_128B);
    if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
  }
  {
    cuuint64_t dims[2] = {(cuuint64_t)p.Kw, (cuuint64_t)d.K};
    cuuint64_t strides[1] = {(cuuint64_t)p.Kw * ES};
    cuuint32_t box[2] = {BKE, PAIR ? (cuuint32_t)(BN / 2) : (cuuint32_t)BN};  // pair: a B half
    cuuint32_t estr[2] = {1, 1};
    CUresult r = gb_encode_tiled(&tmw, DT, 2, const_cast<void*>(wpack), dims, strides, box, estr,
                                 CU_TENSOR_MAP_SWIZZLE_128B);
    if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
  }
  CUtensorMap tmy;  // output [M][K]: bf16 64-column (fp32: 32-column) x 32-row boxes,
                    // 128-byte swizzle
  {
    cuuint64_t dims[2] = {(cuuint64_t)d.K, (cuuint64_t)p.M};
    cuuint64_t strides[1] = {(cuuint64_t)(d.y_kstride ? d.y_kstride : d.K) * ES};
    cuuint32_t box[2] = {TF32 ? 32u : 64u, 32};
    cuuint32_t estr[2] = {1, 1};
    if (p.s2d4_k) {
      // the stride-2 conv's NHWC output [N][2 OH][2 OW][k] seen as
      // (k, px, bw, py, (n, bh)): pixel (2 bh + py, 2 bw + px); 8-row boxes
      const cuuint64_t kb = (cuuint64_t)p.s2d4_k * 2;  // bytes per output pixel
      cuuint64_t dims5[5] = {(cuuint64_t)p.s2d4_k, 2, (cuuint64_t)d.OW, 2,
                             (cuuint64_t)d.N * d.OH};
      cuuint64_t strides5[4] = {kb, 2 * kb, 2 * (cuuint64_t)d.OW * kb,
                                4 * (cuuint64_t)d.OW * kb};
      cuuint32_t box5[5] = {64, 1, 8, 1, 1};
      cuuint32_t estr5[5] = {1, 1, 1, 1, 1};
      if (gb_encode_tiled(&tmy, DT, 5, y, dims5, strides5, box5, estr5,
                          CU_TENSOR_MAP_SWIZZLE_128B) != CUDA_SUCCESS)
        return cudaErrorInvalidValue;
    } else if (gb_encode_tiled(&tmy, DT, 2, y, dims, strides, box, estr,
                               CU_TENSOR_MAP_SWIZZLE_128B) != CUDA_SUCCESS) {
      return cudaErrorInvalidValue;
    }
  }
  CUtensorMap tmr = tmy;  // residual (same shape and boxes as the output), or the
                          // fp32 partial-sum map in split-K mode
  if (p.part) {
    cuuint64_t dims[3] = {(cuuint64_t)d.K, (cuuint64_t)p.M, (cuuint64_t)p.ksplit};
    cuuint64_t strides[2] = {(cuuint64_t)d.K * 4, (cuuint64_t)p.M * d.K * 4};
    cuuint32_t box[3] = {32, 32, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    if (gb_encode_tiled(&tmr, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, p.part, dims, strides, box,
                        estr, CU_TENSOR_MAP_SWIZZLE_128B) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  } else if (res && !TF32) {
    cuuint64_t dims[2] = {(cuuint64_t)d.K, (cuuint64_t)p.M};
    cuuint64_t strides[1] = {(cuuint64_t)(d.y_kstride ? d.y_kstride : d.K) * 2};
    cuuint32_t box[2] = {64, 32};
    cuuint32_t estr[2] = {1, 1};
    if (gb_encode_tiled(&tmr, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(res), dims,
                        strides, box, estr, CU_TENSOR_MAP_SWIZZLE_128B) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  auto* kern = igemm_bf16_tc_kernel<BN, MODE_CONV, LIGHT, TF32, PAIR>;
  cudaError_t e = gb_set_smem_once(reinterpret_cast<const void*>(kern), Cf::SMEM);
  if (e != cudaSuccess) return e;
  const int tiles = p.m_tiles * p.n_tiles * p.ksplit;
  // persistent grid: one work unit per CTA (pair mode: per cluster of two) at a time
  int slots = gb_num_sms() * (LIGHT ? 2 : 1);
  if constexpr (PAIR) {
    slots = pair_max_clusters<BN>(Cf::SMEM);
    if (slots <= 0) return cudaErrorInvalidConfiguration;
  }
  const int grid = tiles < slots ? tiles : slots;
  // a last wave that would leave most SMs idle runs as units of a half or a
  // quarter of the tile's width, the narrowest whose count still fits one wave
  // (at least 64 columns: the epilogue's sub-block; the exact int8 lo/hi path
  // needs a whole 128-column group per unit)
  p.tail_start = tiles;
  p.tail_shift = 1;
  if (p.ksplit == 1 && tiles > grid) {
    const int rem = tiles % grid;
    const int min_width = (p.i8_y && p.i8_nch == 0) ? 128 : 64;
    for (int sh = (BN / min_width >= 4) ? 2 : 1; sh >= 1 && (BN / min_width) >= 2 && rem > 0; --sh) {
      if ((rem << sh) <= grid) {
        p.tail_start = tiles - rem;
        p.tail_shift = sh;
        break;
      }
    }
  }
  CUtensorMap tmwt = tmw;  // B boxes of a tail unit's width
  if (p.tail_start < tiles) {
    const int wt = BN >> p.tail_shift;
    cuuint64_t dims[2] = {(cuuint64_t)p.Kw, (cuuint64_t)d.K};
    cuuint64_t strides[1] = {(cuuint64_t)p.Kw * ES};
    cuuint32_t box[2] = {BKE, (cuuint32_t)(PAIR ? wt / 2 : wt)};
    cuuint32_t estr[2] = {1, 1};
    if (gb_encode_tiled(&tmwt, DT, 2, const_cast<void*>(wpack), dims, strides, box, estr,
                        CU_TENSOR_MAP_SWIZZLE_128B) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(PAIR ? 2 * grid : grid));
  cfg.blockDim = dim3(192);
  cfg.dynamicSmemBytes = Cf::SMEM;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = 2;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = PAIR ? 2 : 1;
  cudaError_t le = cudaLaunchKernelEx(&cfg, kern, tmx, tmw, tmwt, tmy, tmr, p);
  if (le != cudaSuccess) return le;
  gb_count_launch();
  return cudaGetLastError();
}

// out[b][m][n] = sum_k A[b][m][k] * B[b][n][k], fp32 out, fp16/bf16 operands.
template <int BN>
cudaError_t launch_batched_bn(int batch, int M, int N, int Kred, const void* A, const void* Bm,
                              float* out, int ab_type, int* err, unsigned long long wait_ns,
                              cudaStream_t st) {
  using Cf = Cfg<BN>;
  IgemmParams p{};
  p.K = N;
  p.cblocks = gb_ceil_div(Kred, BK);
  p.kiters = p.cblocks;
  p.M = M;
  p.m_tiles = gb_ceil_div(M, BM);
  p.n_tiles = gb_ceil_div(N, BN);
  p.batch = batch;
  p.ab_type = ab_type;
  p.out_f32 = out;
  p.err = err;
  p.wait_ns = wait_ns;
  p.OH = p.OW = 1;
  p.tail_start = 1 << 30;
  p.kch = 1 << 30;
  p.kgroup = (kGroupable<Cf> && p.kiters % 2 == 0) ? 2 : 1;
  p.acc_cols = BN;
  p.nacc = 2;
  p.tmem_cols = 2 * BN;
  const CUtensorMapDataType dt =
      ab_type ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  CUtensorMap tma, tmb;
  {
    cuuint64_t dims[3] = {(cuuint64_t)Kred, (cuuint64_t)M, (cuuint64_t)batch};
    cuuint64_t strides[2] = {(cuuint64_t)Kred * 2, (cuuint64_t)M * Kred * 2};
    cuuint32_t box[3] = {BK, BM, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    if (gb_encode_tiled(&tma, dt, 3, const_cast<void*>(A), dims, strides, box, estr,
                        CU_TENSOR_MAP_SWIZZLE_128B) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  {
    cuuint64_t dims[3] = {(cuuint64_t)Kred, (cuuint64_t)N, (cuuint64_t)batch};
    cuuint64_t strides[2] = {(cuuint64_t)Kred * 2, (cuuint64_t)N * Kred * 2};
    cuuint32_t box[3] = {BK, BN, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    if (gb_encode_tiled(&tmb, dt, 3, const_cast<void*>(Bm), dims, strides, box, estr,
                        CU_TENSOR_MAP_SWIZZLE_128B) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  cudaError_t e = gb_set_smem_once(
      reinterpret_cast<const void*>(igemm_bf16_tc_kernel<BN, MODE_BATCHED>), Cf::SMEM);
  if (e != cudaSuccess) return e;
  const long long tiles = (long long)p.m_tiles * p.n_tiles * batch;
  const int grid = tiles < gb_num_sms() ? (int)tiles : gb_num_sms();
  CUtensorMap tmo;  // fp32 products out[b][m][n], 32 x 32 boxes
  {
    cuuint64_t dims[3] = {(cuuint64_t)N, (cuuint64_t)M, (cuuint64_t)batch};
    cuuint64_t strides[2] = {(cuuint64_t)N * 4, (cuuint64_t)M * N * 4};
    cuuint32_t box[3] = {32, 32, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    if (gb_encode_tiled(&tmo, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, out, dims, strides, box, estr,
                        CU_TENSOR_MAP_SWIZZLE_128B) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  igemm_bf16_tc_kernel<BN, MODE_BATCHED><<<grid, 192, Cf::SMEM, st>>>(tma, tmb, tmb, tma, tmo, p);
  gb_count_launch();
  return cudaGetLastError();
}

}  // namespace

int igemm_block_n(int algo) {
  switch (algo) {
    case CONV_ALGO_IGEMM_N64: return 64;
    case CONV_ALGO_IGEMM_N128: return 128;
    case CONV_ALGO_IGEMM_N256: return 256;
    case CONV_ALGO_IGEMM_2SM: return 256;
    default: return 0;
  }
}

cudaError_t launch_igemm_bf16(const gbconv_desc_s& d, int block_n, const void* x,
                              const void* wpack, const float* bias, const void* res, void* y,
                              int* err, unsigned long long wait_ns, cudaStream_t st,
                              const IgemmSplit& split) {
  if (d.dtype == CONV_F32) {  // fp32 tensors: kind::tf32, 32 channels per k-step
    const int kt = d.R * d.S * gb_ceil_div(d.C, 32);
    const bool lt = kt <= 8;
    switch (block_n) {
      case 64:
        return lt ? launch_bn<64, true, true>(d, x, wpack, bias, res, y, err, wait_ns, st, split)
                  : launch_bn<64, false, true>(d, x, wpack, bias, res, y, err, wait_ns, st, split);
      case 128:
        return lt ? launch_bn<128, true, true>(d, x, wpack, bias, res, y, err, wait_ns, st, split)
                  : launch_bn<128, false, true>(d, x, wpack, bias, res, y, err, wait_ns, st,
                                                split);
      case 256:
        return launch_bn<256, false, true>(d, x, wpack, bias, res, y, err, wait_ns, st, split);
      default: return cudaErrorInvalidValue;
    }
  }
  // short reductions (up to 16 k-steps: 1x1 layers up to 1024 channels, 3x3 up
  // to 64 + 64) are bound by the epilogue and by latency, not by the operand
  // pipeline: run two shallow CTAs per SM (measured on ResNet-50 at batch 64:
  // 52.2k images/s with the cut at 8 k-steps, 53.5-54.1k at 9 to 72)
  const int kiters = d.C == 8 ? gb_ceil_div(d.R * d.S, 8) : d.R * d.S * gb_ceil_div(d.C, BK);
  const int kper = split.ksplit > 1 ? split.kchunk : kiters;
  // (the space-to-depth stem's 9 or 18 k-steps per tile leave its epilogue, which
  // scatters 8-row pieces, as the bound: two CTAs per SM as well)
  const bool light = d.C != 8 && (kper <= 16 || (split.s2d4_k && kper <= 18));
  switch (block_n) {
    case 64:
      return light ? launch_bn<64, true>(d, x, wpack, bias, res, y, err, wait_ns, st, split)
                   : launch_bn<64, false>(d, x, wpack, bias, res, y, err, wait_ns, st, split);
    case 128:
      return light ? launch_bn<128, true>(d, x, wpack, bias, res, y, err, wait_ns, st, split)
                   : launch_bn<128, false>(d, x, wpack, bias, res, y, err, wait_ns, st, split);
    case 256: return launch_bn<256, false>(d, x, wpack, bias, res, y, err, wait_ns, st, split);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_igemm_bf16_pair(const gbconv_desc_s& d, const void* x, const void* wpack,
                                   const float* bias, const void* res, void* y, int* err,
                                   unsigned long long wait_ns, cudaStream_t st) {
  if (d.dtype != CONV_BF16 || d.C == 8 || d.x_cstride || d.y_kstride)
    return cudaErrorInvalidValue;
  return launch_bn<256, false, false, true>(d, x, wpack, bias, res, y, err, wait_ns, st,
                                            IgemmSplit());
}

int igemm_kiters(const gbconv_desc_s& d) {
  return d.C == 8 ? gb_ceil_div(d.R * d.S, 8) : d.R * d.S * gb_ceil_div(d.C, BK);
}

cudaError_t launch_batched_gemm_tc(int batch, int M, int N, int Kred, const void* A,
                                   const void* B, float* out, int ab_type, int block_n, int* err,
                                   unsigned long long wait_ns, cudaStream_t st) {
  if (N % 8 || Kred % 8 || batch <= 0 || M <= 0) return cudaErrorInvalidValue;
  switch (block_n) {
    case 64: return launch_batched_bn<64>(batch, M, N, Kred, A, B, out, ab_type, err, wait_ns, st);
    case 128:
      return launch_batched_bn<128>(batch, M, N, Kred, A, B, out, ab_type, err, wait_ns, st);
    case 256:
      return launch_batched_bn<256>(batch, M, N, Kred, A, B, out, ab_type, err, wait_ns, st);
    default: return cudaErrorInvalidValue;
  }
}

namespace {
// fp32 weights [K][R][S][C] -> [K][R*S][Cp], Cp = C rounded up to 32, zero padded
__global__ void pack_tf32_weights_kernel(const float* __restrict__ w, float* __restrict__ wp,
                                         int K, int RS, int C, int Cp) {
  const long long total = (long long)K * RS * Cp;
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < total;
       i += (long long)gridDim.x * blockDim.x) {
    const int c = (int)(i % Cp);
    const long long krs = i / Cp;
    wp[i] = c < C ? w[krs * C + c] : 0.f;
  }
}
}  // namespace

size_t igemm_tf32_packed_bytes(const gbconv_desc_s& d) {
  return (size_t)d.K * d.R * d.S * gb_ceil_div(d.C, 32) * 32 * 4;
}

cudaError_t launch_pack_tf32_weights(const gbconv_desc_s& d, const void* w, void* wpack,
                                     cudaStream_t st) {
  const int Cp = gb_ceil_div(d.C, 32) * 32;
  const long long total = (long long)d.K * d.R * d.S * Cp;
  const int grid = (int)std::min<long long>((total + 255) / 256, 152LL * 16);
  pack_tf32_weights_kernel<<<grid, 256, 0, st>>>(static_cast<const float*>(w),
                                                  static_cast<float*>(wpack), d.K, d.R * d.S,
                                                  d.C, Cp);
  gb_count_launch();
  return cudaGetLastError();
}

cudaError_t launch_pack_igemm_weights(const gbconv_desc_s& d, const void* w, void* wpack,
                                      cudaStream_t st) {
  if (d.C == 8) {  // narrow mode: [K][taps rounded up to 8][8], zero taps at the end
    const int taps8 = gb_ceil_div(d.R * d.S, 8) * 8;
    const long long total = (long long)d.K * taps8 * 8;
    const int grid = (int)std::min<long long>(gb_ceil_div_ll(total, 256), 65535LL * 8);
    pack_igemm_weights_kernel<<<grid, 256, 0, st>>>(static_cast<const __nv_bfloat16*>(w),
                                                    static_cast<__nv_bfloat16*>(wpack), d.K,
                                                    taps8, 8, 8, d.R * d.S);
    gb_count_launch();
    return cudaGetLastError();
  }
  const int Cp = gb_ceil_div(d.C, BK) * BK;
  const long long total = (long long)d.K * d.R * d.S * Cp;
  const int block = 256;
  const int grid = (int)std::min<long long>(gb_ceil_div_ll(total, block), 65535LL * 8);
  pack_igemm_weights_kernel<<<grid, block, 0, st>>>(static_cast<const __nv_bfloat16*>(w),
                                                    static_cast<__nv_bfloat16*>(wpack), d.K,
                                                    d.R * d.S, d.C, Cp, d.R * d.S);
  gb_count_launch();
  return cudaGetLastError();
}

// The row-strip geometry of d: virtual row width Wv and rows per tile RT (0 when
// the strip kernel does not apply).
static void strip_geometry(const gbconv_desc_s& d, int& Wv, int& RT) {
  Wv = RT = 0;
  const int need = d.OW + d.S - 1;
  int w = 8;
  while (w < need) w *= 2;
  if (w > 128) return;
  const int rows = 128 / w + d.R - 1;
  if ((long long)w * rows * 128 > strip::SLOT) return;
  Wv = w;
  RT = 128 / w;
}

bool igemm_strip_applicable(const gbconv_desc_s& d, const char** why) {
  const char* dummy;
  if (!why) why = &dummy;
  if (d.dtype != CONV_BF16 || d.layout != CONV_NHWC) return *why = "needs bf16 NHWC", false;
  if (d.groups != 1 || d.stride != 1 || d.dil != 1)
    return *why = "needs groups 1, stride 1, dilation 1", false;
  if (d.C < 16 || d.C > 64 || d.C % 8 || d.K > 64 || d.K % 8)
    return *why = "needs 16 <= C <= 64 and K <= 64, multiples of 8", false;
  // (the kernel's tap loops are compiled for these two filter sizes)
  if (!((d.R == 1 && d.S == 1) || (d.R == 3 && d.S == 3)) || d.pad != (d.S - 1) / 2)
    return *why = "needs a 1x1 or 3x3 filter with 'same' padding", false;
  if (d.has_residual) return *why = "no residual", false;
  int Wv, RT;
  strip_geometry(d, Wv, RT);
  if (!Wv) return *why = "output row too wide for one strip", false;
  return true;
}

cudaError_t launch_igemm_strip(const gbconv_desc_s& d, const void* x, const void* wpack,
                               const float* bias, void* y, int* err, unsigned long long wait_ns,
                               cudaStream_t st, const IgemmSplit* i8) {
  int Wv, RT;
  strip_geometry(d, Wv, RT);
  if (!Wv || !igemm_strip_applicable(d, nullptr)) return cudaErrorInvalidValue;
  StripParams p{};
  p.OH = d.OH;
  p.OW = d.OW;
  p.K = d.K;
  p.S = d.S;
  p.taps = d.R * d.S;
  p.Wv = Wv;
  p.RT = RT;
  p.tiles_per_img = gb_ceil_div(d.OH, RT);
  p.m_tiles = d.N * p.tiles_per_img;
  const int rows = RT + d.R - 1;
  p.strip_bytes = Wv * rows * 128;
  p.act = d.act;
  p.bias = bias;
  p.err = err;
  p.wait_ns = wait_ns;
  if (i8) {  // exact int8 output (see StripParams)
    if (!i8->i8_y || !i8->i8_scale || d.K % 16 || (i8->i8_nc32 && d.K % 32))
      return cudaErrorInvalidValue;
    p.i8_y = i8->i8_y;
    p.i8_bias = i8->i8_bias;
    p.i8_scale = i8->i8_scale;
    p.i8_relu = i8->i8_relu;
    p.i8_nc32 = i8->i8_nc32;
    p.act = 0;
  }
  CUtensorMap tmx, tmw, tmy;
  {  // x: (C, W, H, N), box {64 channels, Wv pixels, rows, 1}
    cuuint64_t dims[4] = {(cuuint64_t)d.C, (cuuint64_t)d.W, (cuuint64_t)d.H, (cuuint64_t)d.N};
    cuuint64_t strides[3] = {(cuuint64_t)d.C * 2, (cuuint64_t)d.W * d.C * 2,
                             (cuuint64_t)d.H * d.W * d.C * 2};
    cuuint32_t box[4] = {64, (cuuint32_t)Wv, (cuuint32_t)rows, 1};
    cuuint32_t estr[4] = {1, 1, 1, 1};
    if (gb_encode_tiled(&tmx, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(x), dims,
                        strides, box, estr, CU_TENSOR_MAP_SWIZZLE_128B) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  {  // packed weights [K][taps][64]: one {64, 64} box per tap
    const int Kw = d.R * d.S * 64;
    cuuint64_t dims[2] = {(cuuint64_t)Kw, (cuuint64_t)d.K};
    cuuint64_t strides[1] = {(cuuint64_t)Kw * 2};
    cuuint32_t box[2] = {64, 64};
    cuuint32_t estr[2] = {1, 1};
    if (gb_encode_tiled(&tmw, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(wpack), dims,
                        strides, box, estr, CU_TENSOR_MAP_SWIZZLE_128B) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  if (i8) {
    tmy = tmx;  // int8 output: plain stores, the bf16 output map is not used
  } else {  // y: (K, OW, OH, N); a warp's 32 tile rows are min(Wv, 32) pixels of
     // max(1, 32 / Wv) output rows
    cuuint64_t dims[4] = {(cuuint64_t)d.K, (cuuint64_t)d.OW, (cuuint64_t)d.OH, (cuuint64_t)d.N};
    cuuint64_t strides[3] = {(cuuint64_t)d.K * 2, (cuuint64_t)d.OW * d.K * 2,
                             (cuuint64_t)d.OH * d.OW * d.K * 2};
    cuuint32_t box[4] = {64, (cuuint32_t)(Wv < 32 ? Wv : 32), (cuuint32_t)(Wv < 32 ? 32 / Wv : 1),
                         1};
    cuuint32_t estr[4] = {1, 1, 1, 1};
    if (gb_encode_tiled(&tmy, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, y, dims, strides, box, estr,
                        CU_TENSOR_MAP_SWIZZLE_128B) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  auto* kern = p.act == 0 ? igemm_strip_kernel<0>
                          : (p.act == 1 ? igemm_strip_kernel<1> : igemm_strip_kernel<2>);
  cudaError_t e = gb_set_smem_once(reinterpret_cast<const void*>(kern), strip::SMEM);
  if (e != cudaSuccess) return e;
  const int grid = std::min(p.m_tiles, gb_num_sms());
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3(192);
  cfg.dynamicSmemBytes = strip::SMEM;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, kern, tmx, tmw, tmy, p);
  if (e != cudaSuccess) return e;
  gb_count_launch();
  return cudaGetLastError();
}
