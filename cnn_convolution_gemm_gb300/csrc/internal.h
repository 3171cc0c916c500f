// Internal declarations shared by the library's translation units.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "gbconv.h"

struct gbconv_desc_s {
  int N, C, H, W, K, R, S, stride, pad, dil, groups;
  conv_dtype_t dtype;
  conv_layout_t layout;
  int act;
  int has_residual;
  const float* scale;  // int8 requant scale [K] (device)
  int OH, OW;
  int pad_hi_delta;    // padding after minus padding before (internal rewrites only; 0 = symmetric)
  int shuffle_groups;  // > 1: the input is read channel-shuffled with this many groups
  // channel strides of strided views (one group of a grouped conv): elements
  // between pixels of x and of y / residual; 0 = contiguous (C, K)
  int x_cstride, y_kstride;
};

// Device-side error word codes (written by kernels, read by conv_sync_status).
enum : int { DEV_ERR_NONE = 0, DEV_ERR_TIMEOUT = 1, DEV_ERR_INTERNAL = 2 };

// Thread-local error detail; returns st for convenience.
conv_status_t gb_fail(conv_status_t st, const char* fmt, ...);
// Clears the thread-local error detail and returns CONV_OK (every entry point's
// success return).
conv_status_t gb_ok();
// CONV_OK if algorithm `algo` is built and applies to d (the check conv_fwd
// makes), else CONV_ERR_BAD_PARAM / CONV_ERR_UNSUPPORTED with the reason.
conv_status_t gb_check_algo(const gbconv_desc_s& d, int algo);
// Device error word of the current device (a __device__ int, address cached).
int* gb_device_error_word();
// Number of SMs of the current device (cached).
int gb_num_sms();
// L2 size of the current device in bytes (cached).
long long gb_l2_bytes();
// Called after each kernel launch: counts the kernels the library enqueues.
void gb_count_launch();
// Diagnostic: a kernel whose bounded wait on an mbarrier nothing arrives at runs
// out after limit_ns and records DEV_ERR_TIMEOUT in err.
cudaError_t launch_selftest_wait_timeout(int* err, unsigned long long limit_ns, cudaStream_t st);
// Raise a kernel's dynamic shared-memory limit, once per (kernel, device): the
// attribute call costs host time on every launch otherwise.
cudaError_t gb_set_smem_once(const void* func, int bytes);
// Wait limit for device-side bounded waits, in nanoseconds (GBCONV_WAIT_LIMIT_MS).
unsigned long long gb_wait_limit_ns();

// Driver entry points for TMA descriptors (resolved once through the runtime).
CUresult gb_encode_tiled(CUtensorMap* map, CUtensorMapDataType dt, cuuint32_t rank, void* addr,
                         const cuuint64_t* dims, const cuuint64_t* strides, const cuuint32_t* box,
                         const cuuint32_t* estr, CUtensorMapSwizzle swz);
CUresult gb_encode_im2col(CUtensorMap* map, CUtensorMapDataType dt, cuuint32_t rank, void* addr,
                          const cuuint64_t* dims, const cuuint64_t* strides, const int* lower,
                          const int* upper, cuuint32_t channels, cuuint32_t pixels,
                          const cuuint32_t* estr, CUtensorMapSwizzle swz);

static inline int gb_ceil_div(int a, int b) { return (a + b - 1) / b; }
static inline long long gb_ceil_div_ll(long long a, long long b) { return (a + b - 1) / b; }

// ---- launchers (each returns cudaSuccess or the launch error) --------------

// Direct loop on CUDA cores (any groups / stride / dilation).  Weights in the
// user layout (NHWC: [K][R][S][Cg]; NCHW: [K][Cg][R][S]).
cudaError_t launch_direct(const gbconv_desc_s& d, const void* x, const void* w, const void* bias,
                          const void* res, void* y, cudaStream_t st);

// Implicit GEMM on tcgen05 (bf16 NHWC, groups 1).  wpack: [K][R*S][Cp] bf16,
// Cp = C rounded up to 64, zero padded.
int igemm_block_n(int algo);
// Split-K request: ksplit > 1 cuts the reduction into ranges of kchunk k-steps
// (64 channels of one filter tap each) and writes fp32 partial sums to
// part[ksplit][N*OH*OW][K] instead of running the epilogue.
//
// Exact int8 output mode (i8_y set): the GEMM's N = 2 * i8_kout columns hold, per
// 64 output channels, 64 columns of sums against the low weight nibbles
// (w & 15) then 64 against the high parts (w - (w & 15)) / 16; the epilogue
// forms t = 16 * hi + lo + i8_bias[k] in int32, requantises with i8_scale[k]
// (fp32, round to nearest even), clamps to int8, optional ReLU, and stores
// int8 [M][i8_kout].  Needs BN a multiple of 128 and no split.
struct IgemmSplit {
  int ksplit = 1;
  int kchunk = 0;
  float* part = nullptr;
  int8_t* i8_y = nullptr;
  const int32_t* i8_bias = nullptr;
  const float* i8_scale = nullptr;
  int i8_kout = 0;
  int i8_relu = 0;
  int i8_nc32 = 0;  // int8 output in NC32HW32 (else NHWC)
  // Chunked exact int8 (i8_nch >= 1; 0 selects the lo/hi split weights above):
  // the GEMM's N = i8_kout columns over plain weights; every i8_kch k-steps
  // (64 products each, at most 16: 1024 * 128 * 128 = 2^24) the MMAs start a
  // new TMEM accumulator block, ceil(kiters / i8_kch) == i8_nch blocks in all,
  // and the epilogue sums the blocks' exact integer partial sums in int32.
  int i8_nch = 0;
  int i8_kch = 0;
  // space-to-depth-by-4 stem: the GEMM runs over the 4x4-block grid and its
  // 4K columns are (py, px, k) of the 2x2 output pixels of each block; the
  // epilogue writes them to the stride-2 conv's NHWC output [N][2BH][2BW][K]
  // (s2d4_k = K; 0: off)
  int s2d4_k = 0;
};
int igemm_kiters(const gbconv_desc_s& d);
// Row-strip implicit GEMM (stride 1, C and K <= 64, a 1x1 or 3x3 filter with
// 'same' padding, no residual): one tiled input strip per 128-row tile, the
// taps' A operands by shared-memory offset, weights resident.  wpack: the
// implicit GEMM's packed layout [K][R*S][64].  i8 (optional): exact int8
// output instead of y (its i8_y, i8_bias, i8_scale, i8_relu, i8_nc32; K % 16,
// and K % 32 for NC32HW32), over the bf16 copy of an int8 input.
bool igemm_strip_applicable(const gbconv_desc_s& d, const char** why);
cudaError_t launch_igemm_strip(const gbconv_desc_s& d, const void* x, const void* wpack,
                               const float* bias, void* y, int* err, unsigned long long wait_ns,
                               cudaStream_t st, const IgemmSplit* i8 = nullptr);
// The 256 x 256-tile implicit GEMM over clusters of two CTAs (tcgen05
// cta_group::2): bf16 NHWC, groups 1, C != 8; same packed weights as the
// single-SM tiles.
cudaError_t launch_igemm_bf16_pair(const gbconv_desc_s& d, const void* x, const void* wpack,
                                   const float* bias, const void* res, void* y, int* err,
                                   unsigned long long wait_ns, cudaStream_t st);
// Sums part[ksplit][N*OH*OW][K] (fp32, the split-K GEMM's products) and applies
// d's epilogue (+ bias, + residual, act) into bf16 NHWC y.  K % 8 == 0; part, res
// and y 16-byte aligned.
cudaError_t launch_splitk_reduce_bf16(const gbconv_desc_s& d, int ksplit, const void* part,
                                      const float* bias, const void* res, void* y,
                                      cudaStream_t st);
cudaError_t launch_igemm_bf16(const gbconv_desc_s& d, int block_n, const void* x,
                              const void* wpack, const float* bias, const void* res, void* y,
                              int* err, unsigned long long wait_ns, cudaStream_t st,
                              const IgemmSplit& split = IgemmSplit());
cudaError_t launch_pack_igemm_weights(const gbconv_desc_s& d, const void* w, void* wpack,
                                      cudaStream_t st);
// Batched GEMM on the same tcgen05 pipeline: out[b][m][n] (fp32) =
// sum_k A[b][m][k] * B[b][n][k]; A, B K-major fp16 (ab_type 0) or bf16 (1);
// N and Kred multiples of 8.
cudaError_t launch_batched_gemm_tc(int batch, int M, int N, int Kred, const void* A,
                                   const void* B, float* out, int ab_type, int block_n, int* err,
                                   unsigned long long wait_ns, cudaStream_t st);

// Depthwise 3x3 (bf16 NHWC).  w: packed tap-major [9][C] bf16.
cudaError_t launch_dwconv3x3(const gbconv_desc_s& d, const void* x, const void* w,
                             const float* bias, const void* res, void* y, int* err,
                             unsigned long long wait_ns, cudaStream_t st);
// [C][3][3] -> tap-major [9][C] bf16.
cudaError_t launch_pack_dw_weights(const gbconv_desc_s& d, const void* w, void* wpack,
                                   cudaStream_t st);

// int8 implicit GEMM (mma.sync s8, exact int32 accumulate).  wpack: [K][R*S][Cp] int8.
cudaError_t launch_igemm_int8(const gbconv_desc_s& d, const void* x, const void* wpack,
                              const int32_t* bias, void* y, cudaStream_t st);
cudaError_t launch_pack_int8_weights(const gbconv_desc_s& d, const void* w, void* wpack,
                                     cudaStream_t st);

// int8 on tcgen05 with bf16 as the carrier (exact split-K, see k_int8_tc.cu).
// wpack: [K][R*S][Cp] bf16.
// algo: CONV_ALGO_INT8_TC (split weights, else split-K) or CONV_ALGO_INT8_TC_CHUNK
// (chunked accumulation, else split-K).
size_t int8_tc_workspace_bytes(const gbconv_desc_s& d, int algo);
size_t int8_tc_packed_bytes(const gbconv_desc_s& d, int algo);
cudaError_t launch_pack_int8_tc_weights(const gbconv_desc_s& d, int algo, const void* w,
                                        void* wpack, cudaStream_t st);
cudaError_t launch_int8_tc(const gbconv_desc_s& d, int algo, const void* x, const void* wpack,
                           const int32_t* bias, void* y, void* ws, int* err,
                           unsigned long long wait_ns, cudaStream_t st);

// Explicit im2col matrix in the workspace, then the tcgen05 GEMM (1x1 path).
size_t im2col_workspace_bytes(const gbconv_desc_s& d);
size_t im2col_packed_bytes(const gbconv_desc_s& d);
cudaError_t launch_pack_im2col_weights(const gbconv_desc_s& d, const void* w, void* wpack,
                                       cudaStream_t st);
cudaError_t launch_im2col_gemm(const gbconv_desc_s& d, const void* x, const void* wpack,
                               const float* bias, const void* res, void* y, void* ws, int* err,
                               unsigned long long wait_ns, cudaStream_t st);

// Winograd F(m x m, 3 x 3), m in {2, 6}.
size_t winograd_packed_bytes(const gbconv_desc_s& d, int m);
size_t winograd_workspace_bytes(const gbconv_desc_s& d, int m);
cudaError_t launch_winograd_filter_transform(const gbconv_desc_s& d, int m, const void* w,
                                             void* wpack, cudaStream_t st);
cudaError_t launch_winograd(const gbconv_desc_s& d, int m, const void* x, const void* wpack,
                            const float* bias, const void* res, void* y, void* ws, int* err,
                            unsigned long long wait_ns, cudaStream_t st);

// Layout conversion and pooling.
cudaError_t launch_nchw_f32_to_nhwc_bf16(const float* x, void* y, int N, int C, int H, int W,
                                         int C_out, cudaStream_t st);
cudaError_t launch_nhwc_bf16_to_nchw_f32(const void* x, float* y, int N, int C, int H, int W,
                                         int C_in, cudaStream_t st);
cudaError_t launch_maxpool_nhwc_bf16(const void* x, void* y, int N, int C, int H, int W, int k,
                                     int stride, int pad, cudaStream_t st);
cudaError_t launch_avgpool_nhwc_bf16(const void* x, void* y, int N, int C, int H, int W,
                                     cudaStream_t st);
// Compare two outputs of n elements of dtype (conv_dtype_t): out3[0] = max |a - b|,
// out3[1] = max |b| (fp32 bit patterns), out3[2] = non-finite elements of a
// (int8: also elements that differ).  out3: device, 3 unsigned, zeroed here.
cudaError_t launch_compare_outputs(const void* a, const void* b, long long n, int dtype,
                                   unsigned* out3, cudaStream_t st);
// Fill a buffer with deterministic pseudo-random values (Fast-Run scratch).
cudaError_t launch_fill_random(void* p, size_t bytes, int elem_bytes, uint32_t seed,
                               cudaStream_t st);

// Fused MobileNetV2 block (stride 1): expand 1x1 + ReLU6, depthwise 3x3 + ReLU6,
// project 1x1 (+ residual) in one kernel.
bool mbv2_block_supported(int cin, int E, int cout);
size_t mbv2_block_packed_bytes(int E);
// The expand bias is packed into wpack (it rides in the expand MMA).
cudaError_t launch_pack_mbv2(int cin, int E, int cout, const void* we, const float* be,
                             const void* wd, const void* wp, void* out, cudaStream_t st);
cudaError_t launch_mbv2_block(int N, int H, int W, int cin, int E, int cout, const void* x,
                              const void* wpack, const float* b_dw, const float* b_proj,
                              int has_res, void* y, int* err, unsigned long long wait_ns,
                              cudaStream_t st);

// Stride-2 convolutions over 8 channels as space-to-depth (32 channels) + a
// stride-1 implicit GEMM with asymmetric padding; workspace = the rewritten input.
bool stem_s2d4_applicable(const gbconv_desc_s& d, const char** why);
size_t stem_s2d4_workspace_bytes(const gbconv_desc_s& d);
size_t stem_s2d4_packed_bytes(const gbconv_desc_s& d);
cudaError_t launch_pack_stem4_weights(const gbconv_desc_s& d, const void* w, void* wpack,
                                      cudaStream_t st);
cudaError_t launch_stem_s2d4(const gbconv_desc_s& d, const void* x, const void* wpack,
                             const float* bias, void* y, void* ws, int* err,
                             unsigned long long wait_ns, cudaStream_t st);
bool stem_s2d_applicable(const gbconv_desc_s& d, const char** why);
size_t stem_s2d_workspace_bytes(const gbconv_desc_s& d);
size_t stem_s2d_packed_bytes(const gbconv_desc_s& d);
cudaError_t launch_pack_stem_weights(const gbconv_desc_s& d, const void* w, void* wpack,
                                     cudaStream_t st);
cudaError_t launch_stem_s2d(const gbconv_desc_s& d, const void* x, const void* wpack,
                            const float* bias, const void* res, void* y, void* ws, int* err,
                            unsigned long long wait_ns, cudaStream_t st);

// NCHW int8 <-> NC32HW32 int8 (to_nc32: 1 = NCHW -> NC32HW32, 0 = back).
cudaError_t launch_nc32_convert(const void* x, void* y, int N, int C, int H, int W, int to_nc32,
                                cudaStream_t st);

// Implicit GEMM over fp32 NHWC tensors on kind::tf32 (launch_igemm_bf16 with a
// CONV_F32 desc).  wpack: [K][R*S][Cp] fp32, Cp = C rounded up to 32.
size_t igemm_tf32_packed_bytes(const gbconv_desc_s& d);
cudaError_t launch_pack_tf32_weights(const gbconv_desc_s& d, const void* w, void* wpack,
                                     cudaStream_t st);

// Exact int8 Winograd F(2x2,3x3) with float intermediates: wpack [16][2K][Cp]
// fp16 (the split 4U), workspace V [16][T][Cp] fp16 + M [16][T][2K] fp32.
bool int8_wino_applicable(const gbconv_desc_s& d, const char** why);
size_t int8_wino_packed_bytes(const gbconv_desc_s& d);
size_t int8_wino_workspace_bytes(const gbconv_desc_s& d);
cudaError_t launch_pack_int8_wino(const gbconv_desc_s& d, const void* w, void* wpack,
                                  cudaStream_t st);
cudaError_t launch_int8_wino(const gbconv_desc_s& d, const void* x, const void* wpack,
                             const int32_t* bias, void* y, void* ws, int* err,
                             unsigned long long wait_ns, cudaStream_t st);
