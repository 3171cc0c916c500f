// Exact int8 convolution on the tcgen05 tensor cores, bf16 as the carrier.
//
// sm_103a's tcgen05.mma has no int8 kind.  Every int8 value (|v| <= 128) is
// exact in bf16 and every product of two of them (|p| <= 16384) is exact in the
// fp32 accumulator, and a sum of integers stays exact in fp32 while its
// magnitude is at most 2^24.  So the reduction is cut into chunks of at most
// 1024 products per output (16 k-steps of 64 channels: |sum| <= 1024 * 128^2 =
// 2^24), each chunk's sums are accumulated on the bf16 tcgen05 pipeline, and the
// chunks are added in int32 before the int8 epilogue of the MegEngine Beta
// report's native int8 inference: + int32 bias, fp32 requantisation
// q = clamp(rne(fp32(acc + bias) * scale[k]), -128, 127), ReLU.
//
// Steps per call: int8 -> bf16 copy of the activations (workspace), then one
// of three plans.  Two algorithm ids share this file and Fast-Run times both:
// int8_igemm_tc (split weights, else split-K) and int8_igemm_tc_chunked
// (chunked accumulation, else split-K).
//
// Split weights (int8_igemm_tc, when K % 64 == 0, R*S*C <= 8704 and the grid
// fills at least half the SMs): each weight is cut at prepack into
// w = 16 * wh + wl, wl = w & 15 in [0, 15] and wh in [-8, 7].  Products x * wl
// are at most 128 * 15 = 1920 and x * wh at most 128 * 8 = 1024 in magnitude,
// so an fp32 accumulator stays exact over 8704 products (8704 * 1920 < 2^24):
// every ResNet int8 layer (at most 4608) needs no split of the reduction.  One
// implicit GEMM over 2K columns (per 64 output channels: 64 low-part columns,
// 64 high-part columns) finishes in its own epilogue -- t = 16 * hi + lo +
// bias, requant, ReLU, int8 store -- at twice the tensor work, with wide
// (256-column) tiles that read each activation tile once per 128 channels.
//
// Chunked accumulation (int8_igemm_tc_chunked, when K % 16 == 0 and the grid
// fills at least half the SMs): one implicit GEMM over the plain bf16 weights
// whose MMAs start a fresh TMEM accumulator block every kch <= 16 k-steps (at
// most 1024 products, so each block's sums are exact integers in fp32); its
// epilogue converts the blocks to int32, adds them and the bias, requantises
// and stores int8.  The tensor cores do exactly the direct-equivalent work,
// but the blocks share the SM's 512 TMEM columns, so deep reductions get
// narrower tiles.  A reduction of at most 16 k-steps is a single block.
//
// Split-K (smaller grids, either id): the GEMM's split-K mode writes each
// chunk's exact fp32 partial sums to the workspace and a reduction pass sums
// them in int32 and requantises, so the chunks also spread over otherwise idle
// SMs.
#include <cuda_bf16.h>
#include <stdint.h>

#include <algorithm>

#include "internal.h"
#include "ptx.cuh"

namespace {

constexpr int KCHUNK_MAX = 16;  // k-steps of 64 products per exact fp32 chunk

// Chunked accumulation inside one GEMM (see the file comment): the reduction's
// k-steps are cut into nch blocks of kch <= 16, each accumulated in its own
// TMEM block of BN columns.  BN is the widest tile (up to what K needs) whose
// nch blocks fit TMEM twice (so the epilogue overlaps the next tile), else once.
struct Chunked {
  int block_n = 0, nch = 0, kch = 0;
  long long tiles = 0;
};

Chunked chunked_plan(const gbconv_desc_s& d) {
  Chunked c;
  const int kiters = igemm_kiters(d);
  c.nch = gb_ceil_div(kiters, KCHUNK_MAX);
  c.kch = gb_ceil_div(kiters, c.nch);
  c.nch = gb_ceil_div(kiters, c.kch);
  const int widest = d.K > 128 ? 256 : (d.K > 64 ? 128 : 64);
  int bn = widest;
  while (bn > 64 && 2 * c.nch * bn > 512) bn /= 2;
  if (c.nch * bn > 512) return Chunked{};  // more than 8 blocks: not this path
  c.block_n = bn;
  c.tiles = gb_ceil_div_ll((long long)d.N * d.OH * d.OW, 128) * gb_ceil_div(d.K, bn);
  return c;
}

// The chunked GEMM applies (K a multiple of 16, at most 8 accumulator blocks)
// and its tile grid fills at least half the SMs; smaller grids keep split-K,
// which spreads the reduction over more CTAs.
bool use_chunked(const gbconv_desc_s& d) {
  if (d.K % 16) return false;
  const Chunked c = chunked_plan(d);
  return c.block_n > 0 && 2 * c.tiles >= gb_num_sms();
}

constexpr int SPLITW_MAX = 8704;  // products per output that stay exact with split weights

// the split-weight path applies (see the file comment) and its unsplit tile
// grid fills at least half the SMs; smaller grids keep split-K, which spreads the
// reduction (measured on the ResNet-50 stage shapes at batch 32: 256@14 with 98
// tiles runs faster split-weight, 512@7 with 52 tiles faster split-K)
bool split_weights(const gbconv_desc_s& d) {
  if (d.K % 64 || (long long)d.R * d.S * (gb_ceil_div(d.C, 64) * 64) > SPLITW_MAX) return false;
  const long long m_tiles = gb_ceil_div_ll((long long)d.N * d.OH * d.OW, 128);
  const int n_tiles = d.K == 64 ? 1 : 2 * d.K / 256;
  return 2 * m_tiles * n_tiles >= gb_num_sms();
}

// bf16 has 8 significant bits: every int8 value converts exactly.  Output NHWC
// bf16, 16 channels per thread; the int8 input is NHWC, or NC32HW32 (nc32 = 1:
// the same 16 channels are one 16-byte half of a 32-channel block vector).
__global__ void int8_to_bf16_kernel(const int8_t* __restrict__ x, __nv_bfloat16* __restrict__ y,
                                    long long n16, int C, long long HW, int nc32) {
  gb::allow_dependents();  // the GEMM that reads y sets up meanwhile
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n16;
       i += (long long)gridDim.x * blockDim.x) {
    long long src = i;  // in 16-byte units
    if (nc32) {
      const int j = (int)(i % (C / 16));  // 16-channel group of the pixel
      const long long pix = i / (C / 16), n = pix / HW;
      src = ((n * (C / 32) + j / 2) * HW + (pix - n * HW)) * 2 + (j & 1);
    }
    const int4 v = reinterpret_cast<const int4*>(x)[src];
    const int8_t* b = reinterpret_cast<const int8_t*>(&v);
    uint4 o[2];
    uint32_t* ou = reinterpret_cast<uint32_t*>(o);
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      __nv_bfloat162 h = __floats2bfloat162_rn((float)b[2 * j], (float)b[2 * j + 1]);
      ou[j] = *reinterpret_cast<uint32_t*>(&h);
    }
    reinterpret_cast<uint4*>(y)[2 * i] = o[0];
    reinterpret_cast<uint4*>(y)[2 * i + 1] = o[1];
  }
}

// int8 [K][RS][C] -> bf16 [K][RS][Cp], zero padded channels
__global__ void pack_int8_as_bf16_kernel(const int8_t* __restrict__ w,
                                         __nv_bfloat16* __restrict__ wp, int K, int RS, int C,
                                         int Cp) {
  const long long total = (long long)K * RS * Cp;
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < total;
       i += (long long)gridDim.x * blockDim.x) {
    const int c = (int)(i % Cp);
    const long long krs = i / Cp;
    wp[i] = __float2bfloat16_rn(c < C ? (float)w[krs * C + c] : 0.f);
  }
}

// int8 [K][RS][C] -> bf16 [2K][RS][Cp]: per 64 output channels, 64 rows of low
// nibbles (w & 15) then 64 rows of high parts ((w - (w & 15)) / 16), zero
// padded channels
__global__ void pack_int8_split_kernel(const int8_t* __restrict__ w,
                                       __nv_bfloat16* __restrict__ wp, int K, int RS, int C,
                                       int Cp) {
  const long long total = (long long)2 * K * RS * Cp;
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < total;
       i += (long long)gridDim.x * blockDim.x) {
    const int c = (int)(i % Cp);
    const long long rowrs = i / Cp;
    const int rs = (int)(rowrs % RS);
    const int row = (int)(rowrs / RS);
    const int k = (row >> 7) * 64 + (row & 63);  // output channel of this row
    const bool high = (row & 64) != 0;
    float v = 0.f;
    if (c < C) {
      const int wv = w[((long long)k * RS + rs) * C + c];
      const int lo = wv & 15;
      v = high ? (float)((wv - lo) / 16) : (float)lo;
    }
    wp[i] = __float2bfloat16_rn(v);  // |v| <= 15: exact
  }
}

// y[m][n] = requant(sum_b part[b][m][n] + bias[n]); 4 channels per thread
// (y in NHWC, or NC32HW32 when nc32 = 1; ohw = OH * OW)
__global__ void reduce_requant_kernel(const float* __restrict__ part, int ksplit, long long MK,
                                      int K, const int32_t* __restrict__ bias,
                                      const float* __restrict__ scale, int relu,
                                      int8_t* __restrict__ y, long long ohw, int nc32) {
  const long long n4 = MK / 4;
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n4;
       i += (long long)gridDim.x * blockDim.x) {
    int acc[4] = {0, 0, 0, 0};
    for (int b = 0; b < ksplit; ++b) {
      const float4 v = reinterpret_cast<const float4*>(part + (size_t)b * MK)[i];
      acc[0] += __float2int_rn(v.x);  // exact: each partial is an integer below 2^24
      acc[1] += __float2int_rn(v.y);
      acc[2] += __float2int_rn(v.z);
      acc[3] += __float2int_rn(v.w);
    }
    const int n0 = (int)((i * 4) % K);
    char4 o;
    int8_t* ob = reinterpret_cast<int8_t*>(&o);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int t = acc[j] + (bias ? bias[n0 + j] : 0);
      int q = __float2int_rn(__fmul_rn(__int2float_rn(t), scale[n0 + j]));
      q = q > 127 ? 127 : (q < -128 ? -128 : q);
      if (relu && q < 0) q = 0;
      ob[j] = (int8_t)q;
    }
    long long dst = i;  // in 4-byte units
    if (nc32) {
      const long long m = (i * 4) / K, img = m / ohw;
      dst = (((img * (K / 32) + n0 / 32) * ohw + (m - img * ohw)) * 32 + (n0 & 31)) / 4;
    }
    reinterpret_cast<char4*>(y)[dst] = o;
  }
}

struct Plan {
  int block_n, kiters, ksplit, kchunk;
  size_t x_bytes, part_bytes;
};

Plan make_plan(const gbconv_desc_s& d) {
  Plan p{};
  p.block_n = d.K > 128 ? 256 : (d.K > 64 ? 128 : 64);
  p.kiters = igemm_kiters(d);
  const long long M = (long long)d.N * d.OH * d.OW;
  const long long tiles = gb_ceil_div_ll(M, 128) * gb_ceil_div(d.K, p.block_n);
  int ks = gb_ceil_div(p.kiters, KCHUNK_MAX);  // exactness bound
  // more ranges when the tile grid alone would leave SMs idle
  while ((long long)ks * tiles < gb_num_sms() && gb_ceil_div(p.kiters, ks + 1) >= 4) ++ks;
  p.kchunk = gb_ceil_div(p.kiters, ks);
  p.ksplit = gb_ceil_div(p.kiters, p.kchunk);
  p.x_bytes = ((size_t)d.N * d.H * d.W * d.C * 2 + 255) / 256 * 256;
  p.part_bytes = (size_t)p.ksplit * M * d.K * 4;
  return p;
}

int grid_for(long long n) { return (int)std::min<long long>(gb_ceil_div_ll(n, 256), 148LL * 32); }

// the plan algorithm `algo` (int8_igemm_tc or its chunked variant) runs on d
enum class I8Plan { SplitWeights, Chunked, SplitK };

I8Plan plan_for(const gbconv_desc_s& d, int algo) {
  if (algo == CONV_ALGO_INT8_TC_CHUNK) return use_chunked(d) ? I8Plan::Chunked : I8Plan::SplitK;
  return split_weights(d) ? I8Plan::SplitWeights : I8Plan::SplitK;
}

}  // namespace

size_t int8_tc_workspace_bytes(const gbconv_desc_s& d, int algo) {
  const Plan p = make_plan(d);
  return plan_for(d, algo) == I8Plan::SplitK ? p.x_bytes + p.part_bytes : p.x_bytes;
}

size_t int8_tc_packed_bytes(const gbconv_desc_s& d, int algo) {
  return (size_t)(plan_for(d, algo) == I8Plan::SplitWeights ? 2 : 1) * d.K * d.R * d.S *
         gb_ceil_div(d.C, 64) * 64 * 2;
}

cudaError_t launch_pack_int8_tc_weights(const gbconv_desc_s& d, int algo, const void* w,
                                        void* wpack, cudaStream_t st) {
  const int Cp = gb_ceil_div(d.C, 64) * 64;
  if (plan_for(d, algo) == I8Plan::SplitWeights) {
    const long long total = (long long)2 * d.K * d.R * d.S * Cp;
    pack_int8_split_kernel<<<grid_for(total), 256, 0, st>>>(
        static_cast<const int8_t*>(w), static_cast<__nv_bfloat16*>(wpack), d.K, d.R * d.S, d.C,
        Cp);
    gb_count_launch();
    return cudaGetLastError();
  }
  const long long total = (long long)d.K * d.R * d.S * Cp;
  pack_int8_as_bf16_kernel<<<grid_for(total), 256, 0, st>>>(
      static_cast<const int8_t*>(w), static_cast<__nv_bfloat16*>(wpack), d.K, d.R * d.S, d.C, Cp);
  gb_count_launch();
  return cudaGetLastError();
}

cudaError_t launch_int8_tc(const gbconv_desc_s& d, int algo, const void* x, const void* wpack,
                           const int32_t* bias, void* y, void* ws, int* err,
                           unsigned long long wait_ns, cudaStream_t st) {
  const Plan pl = make_plan(d);
  const I8Plan plan = plan_for(d, algo);
  __nv_bfloat16* xb = static_cast<__nv_bfloat16*>(ws);
  float* part = reinterpret_cast<float*>(static_cast<char*>(ws) + pl.x_bytes);
  const long long n16 = (long long)d.N * d.H * d.W * d.C / 16;
  const int nc32 = d.layout == CONV_NC32HW32 ? 1 : 0;
  int8_to_bf16_kernel<<<grid_for(n16), 256, 0, st>>>(static_cast<const int8_t*>(x), xb, n16, d.C,
                                                     (long long)d.H * d.W, nc32);
  gb_count_launch();
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  gbconv_desc_s db = d;  // the same convolution over the bf16 copy
  db.dtype = CONV_BF16;
  db.act = CONV_ACT_NONE;
  db.has_residual = 0;
  if (plan != I8Plan::SplitK) {  // one GEMM, int8 written by its epilogue
    IgemmSplit sp;
    sp.i8_y = static_cast<int8_t*>(y);
    sp.i8_bias = bias;
    sp.i8_scale = d.scale;
    sp.i8_kout = d.K;
    sp.i8_relu = d.act == CONV_ACT_RELU ? 1 : 0;
    sp.i8_nc32 = nc32;
    if (plan == I8Plan::SplitWeights) {  // 2K columns: low and high weight parts
      db.K = 2 * d.K;
      return launch_igemm_bf16(db, d.K == 64 ? 128 : 256, xb, wpack, nullptr, nullptr, y, err,
                               wait_ns, st, sp);
    }
    const Chunked c = chunked_plan(d);
    sp.i8_nch = c.nch;
    sp.i8_kch = c.kch;
    // one accumulator block over at most 64 channels into at most 64, stride 1,
    // a 1x1 or 3x3 filter: the row-strip kernel (one input strip per tile, the
    // taps by shared-memory offset) over the NHWC bf16 copy, same packed weights
    gbconv_desc_s ds = db;
    ds.layout = CONV_NHWC;
    if (c.nch == 1 && igemm_strip_applicable(ds, nullptr))
      return launch_igemm_strip(ds, xb, wpack, nullptr, nullptr, err, wait_ns, st, &sp);
    return launch_igemm_bf16(db, c.block_n, xb, wpack, nullptr, nullptr, y, err, wait_ns, st,
                             sp);
  }
  IgemmSplit sp;
  sp.ksplit = pl.ksplit;
  sp.kchunk = pl.kchunk;
  sp.part = part;
  e = launch_igemm_bf16(db, pl.block_n, xb, wpack, nullptr, nullptr, y, err, wait_ns, st, sp);
  if (e != cudaSuccess) return e;
  const long long MK = (long long)d.N * d.OH * d.OW * d.K;
  reduce_requant_kernel<<<grid_for(MK / 4), 256, 0, st>>>(part, pl.ksplit, MK, d.K, bias, d.scale,
                                                          d.act == CONV_ACT_RELU ? 1 : 0,
                                                          static_cast<int8_t*>(y),
                                                          (long long)d.OH * d.OW, nc32);
  gb_count_launch();
  return cudaGetLastError();
}
