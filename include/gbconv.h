/*
 * gbconv — 2D convolution forward for CNN inference on GB300 (sm_103a).
 *
 * A C ABI over hand-written CUDA kernels.  Plain pointers and sizes only.
 * All tensor pointers are caller-owned DEVICE memory unless a function says
 * otherwise; the library never frees them.  Every call that launches work is
 * stream-ordered on the given stream (a cudaStream_t passed as void*; NULL is
 * the legacy default stream) and returns as soon as the work is enqueued.
 *
 * Passages cited below are from the four pages this library implements:
 *   [MegEngine]  aminer.cn report on MegEngine's CPU convolution work
 *                (sections "Inference Layout", "Im2col+MatMul", "Winograd",
 *                "Fast-Run");
 *   [Momenta]    getit01.com "Paper Reading | 讓深度學習更高效運行的兩個視角"
 *                (roofline, FLOP/traffic accounting, depthwise, fusion);
 *   [Beta]       96x.com.cn MegEngine Beta report (native int8 inference);
 *   [卷积总结]   razer666.cn convolution-internals post (direct loop,
 *                im2col -> GEMM).
 *
 * Error behaviour: every function returns a conv_status_t.  Host-side
 * validation failures return before anything is enqueued.  Errors detected by
 * a kernel on the device (a bounded wait that ran out, an internal check) are
 * recorded in a device-side error word and reported by conv_sync_status().
 * conv_last_error_detail() gives a human-readable reason for the last failure
 * on the calling thread.
 */
#ifndef GBCONV_H_
#define GBCONV_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct gbconv_desc_s* conv_desc_t;

typedef enum {
  CONV_OK = 0,
  CONV_ERR_BAD_PARAM = 1,      /* invalid argument (null, negative size, ...)          */
  CONV_ERR_UNSUPPORTED = 2,    /* the algorithm does not apply to this descriptor      */
  CONV_ERR_ALIGNMENT = 3,      /* a pointer is not 16-byte aligned (TMA requirement)   */
  CONV_ERR_WORKSPACE = 4,      /* workspace missing or smaller than conv_workspace_size */
  CONV_ERR_CUDA = 5,           /* a CUDA runtime/driver call failed                    */
  CONV_ERR_TIMEOUT = 6,        /* a device-side bounded wait ran out                   */
  CONV_ERR_INTERNAL = 7,       /* a device-side consistency check failed               */
  CONV_ERR_FASTRUN_FILE = 8,   /* Fast-Run map file unreadable, corrupt or mismatched  */
  CONV_ERR_NOT_FOUND = 9       /* no Fast-Run entry for this descriptor                */
} conv_status_t;

/* Element type of x, w and y.  CONV_BF16: bfloat16 tensors, fp32 bias,
 * fp32 accumulation.  CONV_F32: fp32 tensors and bias.  CONV_INT8: int8
 * tensors, int32 bias, exact int32 accumulation, fp32 per-channel requant. */
typedef enum { CONV_BF16 = 0, CONV_F32 = 1, CONV_INT8 = 2 } conv_dtype_t;

/* Activation layout ([MegEngine] "Inference Layout").  NHWC is the device
 * layout of every fast kernel; NCHW is accepted for CONV_F32 only. */
/* NC32HW32 (int8 only): channel blocks of 32, element (n, c, h, w) at
 * (((n * C/32 + c/32) * H + h) * W + w) * 32 + c % 32 — the GPU counterpart of
 * the pages' NCHWX layouts ([MegEngine] "Inference Layout"; [Beta] NCHW44):
 * each pixel's 32 channels of a block are one 32-byte vector.  Needs C and K
 * multiples of 32; weights stay [K][R][S][C]. */
typedef enum { CONV_NHWC = 0, CONV_NCHW = 1, CONV_NC32HW32 = 2 } conv_layout_t;

typedef enum { CONV_ACT_NONE = 0, CONV_ACT_RELU = 1, CONV_ACT_RELU6 = 2 } conv_act_t;

/* Algorithm ids ([MegEngine] "Fast-Run": Im2col, Direct and Winograd are the
 * candidate implementations).  Ids are stable. */
typedef int conv_algo_t;
#define CONV_ALGO_AUTO (-1)        /* Fast-Run map entry if present, else the heuristic */
#define CONV_ALGO_DIRECT 0         /* CUDA-core direct loop, any shape ([卷积总结])      */
#define CONV_ALGO_IGEMM_N64 1      /* implicit GEMM on tcgen05, 128x64 output tiles     */
#define CONV_ALGO_IGEMM_N128 2     /* implicit GEMM on tcgen05, 128x128 output tiles    */
#define CONV_ALGO_IGEMM_N256 3     /* implicit GEMM on tcgen05, 128x256 output tiles    */
#define CONV_ALGO_WINO_F2 4        /* Winograd F(2x2,3x3)                               */
#define CONV_ALGO_WINO_F6 5        /* Winograd F(6x6,3x3)                               */
#define CONV_ALGO_DEPTHWISE 6      /* depthwise 3x3 (groups == C == K)                  */
#define CONV_ALGO_INT8_MMA 7       /* int8 implicit GEMM on mma.sync, exact int32 acc.  */
#define CONV_ALGO_INT8_TC 8        /* int8 on tcgen05, exact: weights split into 4-bit
                                      parts over 2K GEMM columns (workspace)            */
#define CONV_ALGO_IM2COL_GEMM 9    /* materialised im2col matrix + GEMM (workspace)     */
#define CONV_ALGO_STEM_S2D 10      /* stride-2 conv over 8 channels (the image stem) as
                                      space-to-depth + stride-1 implicit GEMM (workspace) */
#define CONV_ALGO_IGEMM_TF32 11    /* implicit GEMM over fp32 NHWC tensors on kind::tf32
                                      (inputs read with tf32's 10-bit mantissa)          */
#define CONV_ALGO_INT8_WINO_F2 12  /* int8 Winograd F(2x2,3x3) with float intermediates
                                      ([Beta]), exact: integer transforms, split filter
                                      transform, fp32 sums below 2^24 (C <= 896; workspace) */
#define CONV_ALGO_STEM_S2D4 13     /* stride-2 conv over 4 or 8 channels as a 4x4
                                      space-to-depth + implicit GEMM whose columns are
                                      the 2x2 output pixels of each block (K == 64;
                                      workspace)                                         */
#define CONV_ALGO_IGEMM_2SM 14     /* implicit GEMM with 256 x 256 tiles split over a pair
                                      of SMs (tcgen05 cta_group::2; groups 1, C != 8)   */
#define CONV_ALGO_INT8_TC_CHUNK 15 /* int8 on tcgen05, exact by chunked accumulation: a
                                      fresh TMEM accumulator every <= 16 k-steps, the
                                      blocks summed in int32 by the epilogue (1x the
                                      tensor work; workspace)                           */
#define CONV_ALGO_IGEMM_STRIP 16   /* implicit GEMM for stride-1 layers over <= 64 channels
                                      into <= 64 (1x1 or 3x3, 'same' padding, no
                                      residual): each 128-row tile loads ONE input-row
                                      strip and takes every filter tap from it by a
                                      shared-memory offset ([MegEngine] "Im2col+MatMul":
                                      the unrolled rows are never fetched twice)        */
#define CONV_ALGO_COUNT 17

/* ---- descriptor --------------------------------------------------------- */

/* Create a convolution descriptor.
 * Defines y[n,oh,ow,k] = act(b[k] + sum_{c in group(k), r, s}
 *     w[k,r,s,c] * x[n, oh*stride - pad + r*dilation, ow*stride - pad + s*dilation, c]
 *     (+ residual[n,oh,ow,k])), x = 0 outside the image: the direct loop of
 * [卷积总结] "最原始的卷积实现" with the stride, dilation and padding it names,
 * cross-correlation (no kernel flip) as in its "稀疏连接" example.
 * OH = (H + 2*pad - dilation*(R-1) - 1)/stride + 1, likewise OW.
 * Requirements: all sizes > 0, C % groups == 0, K % groups == 0, OH, OW > 0.
 * The descriptor is owned by the caller and freed with conv_desc_destroy.
 * Defaults: layout NHWC, no activation, no residual, no requant scale. */
conv_status_t conv_desc_create(conv_desc_t* out, int N, int C, int H, int W, int K, int R, int S,
                               int stride, int pad, int dilation, int groups, conv_dtype_t dtype);
conv_status_t conv_desc_destroy(conv_desc_t desc);
/* Activation layout of x, y and residual (weights follow: NHWC -> w is
 * [K][R][S][C/groups], NCHW -> w is [K][C/groups][R][S]). NCHW: CONV_F32 only. */
conv_status_t conv_desc_set_layout(conv_desc_t desc, conv_layout_t layout);
/* Fused epilogue ([Momenta] "Graph層面": bias and ReLU fused into the matrix
 * product).  act: conv_act_t; has_residual: conv_fwd reads a residual tensor
 * shaped like y and adds it before the activation.  INT8 supports
 * act in {NONE, RELU} and no residual. */
conv_status_t conv_desc_set_epilogue(conv_desc_t desc, int act, int has_residual);
/* Read the input channel-shuffled ([Momenta] Graph層面: "shuffle-channel +
 * depthwise" fused): with g groups, channel c of the shuffled input is channel
 * (c mod g) * (C / g) + c div g of x — ShuffleNet's shuffle (view C as g x C/g,
 * transpose) applied while loading, so the shuffled tensor is never written.
 * g = 1 turns it off.  Needs C % g == 0.  Honoured by CONV_ALGO_DEPTHWISE (C <=
 * 256, no residual) and CONV_ALGO_DIRECT; other algorithms do not apply. */
conv_status_t conv_desc_set_input_shuffle(conv_desc_t desc, int groups);
/* INT8 only: per-output-channel requant scale, fp32 [K], DEVICE pointer that
 * must stay valid while the descriptor is used.  Output int8 value:
 * q = clamp(round_half_even(fp32(acc + bias[k]) * scale[k]), -128, 127), then
 * the activation.  ([Beta] "推理：高效原生 int8 实现"; the pages print no
 * formula, this is the library's definition.) */
conv_status_t conv_desc_set_requant(conv_desc_t desc, const float* scale_dev);
/* Output spatial size. */
conv_status_t conv_desc_get_output_dims(conv_desc_t desc, int* OH, int* OW);

/* ---- algorithms --------------------------------------------------------- */

/* Number of algorithm ids (CONV_ALGO_COUNT). */
conv_status_t conv_algo_count(conv_desc_t desc, int* count);
/* Info for algorithm index i in [0, count): its id, a static name string and
 * whether it applies to the descriptor (1) or not (0). */
conv_status_t conv_algo_info(conv_desc_t desc, int i, conv_algo_t* algo, const char** name,
                             int* applicable);
/* The algorithm CONV_ALGO_AUTO resolves to (Fast-Run map, else heuristic). */
conv_status_t conv_algo_resolve(conv_desc_t desc, conv_algo_t* algo);
/* Bytes of device workspace conv_fwd needs for (desc, algo); 0 if none.
 * For the implicit-GEMM algorithms (CONV_ALGO_IGEMM_N64/128/256, groups 1) this
 * is the split-K buffer: when the layer's output tiles (128 rows x the tile
 * width) fill at most half the device's SMs and its reduction has 16 or more
 * k-steps, the reduction is cut into ranges whose fp32 partial products
 * (ksplit x N*OH*OW x K floats) are summed by a second kernel with the bias,
 * residual and activation ([MegEngine] "Im2col+MatMul", the reduction axis of
 * the product split).  There the workspace is optional: a conv_fwd given less
 * runs the same algorithm unsplit.  The size depends on the device's SM count. */
conv_status_t conv_workspace_size(conv_desc_t desc, conv_algo_t algo, size_t* bytes);
/* Bytes of the packed weight buffer for (desc, algo). */
conv_status_t conv_weights_packed_size(conv_desc_t desc, conv_algo_t algo, size_t* bytes);
/* Pack weights once per layer ([MegEngine] "Winograd": the weights are
 * transformed ahead; for implicit GEMM the reduction axis is padded to the
 * tile).  w: device, layout per conv_desc_set_layout, dtype of the desc.
 * wpack: device, conv_weights_packed_size bytes, 16-byte aligned, caller-owned.
 * Stream-ordered. */
conv_status_t conv_weights_prepack(conv_desc_t desc, conv_algo_t algo, const void* w,
                                   void* wpack, void* stream);

/* ---- forward ------------------------------------------------------------ */

/* y = conv(x, w) + bias (+ residual), activation; per conv_desc_create.
 * x, y, residual: device, layout of the desc, dtype of the desc, 16-byte
 * aligned.  wpack: output of conv_weights_prepack for the SAME algo (after
 * CONV_ALGO_AUTO resolution; use conv_algo_resolve).  bias: device fp32 [K]
 * (int32 [K] for INT8) or NULL for zero.  residual: NULL unless the desc has
 * has_residual.  ws: device workspace of at least conv_workspace_size bytes
 * (NULL if 0).  Returns CONV_ERR_UNSUPPORTED if algo does not apply.
 * Stream-ordered; x, wpack, bias, residual must stay valid until the work
 * completes. */
conv_status_t conv_fwd(conv_desc_t desc, const void* x, const void* wpack, const void* bias,
                       const void* residual, void* y, conv_algo_t algo, void* ws,
                       size_t ws_bytes, void* stream);

/* Winograd forward (algo CONV_ALGO_WINO_F2 or CONV_ALGO_WINO_F6) that
 * allocates nothing and takes no workspace.  The pages have no counterpart:
 * this entry point exists for callers that cannot allocate device memory when
 * they run a layer — a plugin inside a host framework whose memory manager
 * owns all device allocations, a latency-critical path where a cudaMalloc or a
 * growing allocator pool would stall or synchronize the GPU, or a deployment
 * whose memory budget is fixed at load time.  They pass inputs and outputs only
 * (same meaning, layout and alignment rules as conv_fwd; wpack from
 * conv_weights_prepack with the same algo).
 * Scratch: a fixed 24 MiB array in device global memory.  It is created on a
 * device when the library's module holding it is loaded there: under CUDA's
 * default lazy module loading that is the first conv_fwd_noalloc call on that
 * device (with CUDA_MODULE_LOADING=EAGER, when the library initialises its
 * modules on the device); from then on it stays until the process exits.  The
 * batch is processed in slices of as many images as fit; if a single image
 * needs more, the call returns CONV_ERR_WORKSPACE before launching anything.
 * All calls on a device share the array: calls that can overlap on the GPU
 * race on it, so order them (one stream, or events).  The first call on a
 * device looks up the array's device address with that device current; make
 * it before any stream capture.  The descriptor must admit the algorithm under
 * conv_fwd's rules (an input shuffle, for one, does not); other algorithms
 * and descriptors return CONV_ERR_UNSUPPORTED.  Stream-ordered. */
conv_status_t conv_fwd_noalloc(conv_desc_t desc, const void* x, const void* wpack,
                               const void* bias, const void* residual, void* y,
                               conv_algo_t algo, void* stream);

/* ---- forward pass on host tensors ---------------------------------------- */

/* conv_fwd with the activations in HOST memory: x_host (and residual_host when
 * the descriptor has a residual) are copied to the device, convolved, and the
 * result copied back to y_host.  The batch is cut into chunks of n_chunk
 * images (n_chunk <= 0 or >= N: one chunk) and the copies run on two streams
 * the library owns, so chunk i+1's input copy and chunk i-1's output copy
 * overlap chunk i's convolution, which runs on `stream`.  Images are
 * independent, so the result equals conv_fwd on the whole batch.
 *   x_host, residual_host, y_host: the same layouts and sizes as conv_fwd's
 *     device tensors, in host memory (page-locked memory lets the copies
 *     overlap; pageable memory works but serialises them).
 *   wpack, bias: DEVICE pointers, as for conv_fwd (weights stay resident).
 *   algo: as for conv_fwd (AUTO resolves on the whole-batch descriptor).  An
 *     algorithm whose packed-weight layout depends on the batch size (the int8
 *     split-weight choice) runs the batch as one chunk.
 *   scratch: device memory of conv_fwd_host_scratch_size() bytes, 256-byte
 *     aligned, caller-owned: two input, two output (and two residual) chunk
 *     buffers plus the algorithm's workspace for one chunk.
 * Stream-ordered: the call enqueues and returns; y_host is complete when
 * `stream` reaches the point after the call (e.g. after
 * cudaStreamSynchronize(stream) or conv_sync_status(stream)).  Host threads
 * calling it at the same time are serialised while they enqueue.
 * Errors: CONV_ERR_BAD_PARAM (NULL tensor, residual mismatch), the algorithm's
 * CONV_ERR_UNSUPPORTED, CONV_ERR_WORKSPACE (scratch too small),
 * CONV_ERR_ALIGNMENT, CONV_ERR_CUDA. */
conv_status_t conv_fwd_host_scratch_size(conv_desc_t desc, conv_algo_t algo, int n_chunk,
                                         size_t* bytes);
conv_status_t conv_fwd_host(conv_desc_t desc, const void* x_host, const void* wpack,
                            const void* bias, const void* residual_host, void* y_host,
                            conv_algo_t algo, int n_chunk, void* scratch, size_t scratch_bytes,
                            void* stream);

/* ---- fused MobileNetV2 block ([Momenta] "Graph層面" and "優化2") ----------- */

/* The inverted-residual block of MobileNetV2 at stride 1 as ONE kernel:
 *   t1 = ReLU6(conv1x1(x, w_expand) + b_expand)          C_in -> E channels
 *   t2 = ReLU6(depthwise3x3(t1, pad 1) + b_dw)           E channels
 *   y  = conv1x1(t2, w_project) + b_project (+ x)        E -> C_out channels
 * The Momenta talk's fusion argument: run as three layers, the two E-channel
 * intermediates make four passes through memory; here they stay in shared
 * memory per 14x14 output tile (halo recomputed), so HBM sees x, y and the
 * weights only.  t1 and t2 are rounded to bf16 where the three-layer chain
 * stores them; b_expand enters the expand's fp32 accumulation as two bf16 terms
 * (16 significant bits).  Supported: E = 144, C_in in {8, 16, 24}, C_out a
 * multiple of 8 in [8, 32] (the 24 -> 144 -> 24 blocks); has_residual needs
 * C_in == C_out.  Anything else returns CONV_ERR_UNSUPPORTED. */
/* Bytes of the packed weight buffer. */
conv_status_t conv_mbv2_block_packed_size(int C_in, int E, int C_out, size_t* bytes);
/* Pack the weights and the expand bias once.  w_expand: device bf16 [E][C_in]
 * (the [K][1][1][C] layout of conv_desc NHWC weights); b_expand: device fp32
 * [E] or NULL for zero; w_dw: device bf16 [E][3][3]; w_project: device bf16
 * [C_out][E].  wpack: device, conv_mbv2_block_packed_size bytes, 16-byte
 * aligned, caller-owned.  Stream-ordered. */
conv_status_t conv_mbv2_block_prepack(int C_in, int E, int C_out, const void* w_expand,
                                      const float* b_expand, const void* w_dw,
                                      const void* w_project, void* wpack, void* stream);
/* x: device bf16 NHWC [N][H][W][C_in]; y: device bf16 NHWC [N][H][W][C_out]
 * (both 16-byte aligned, not overlapping); wpack from conv_mbv2_block_prepack
 * with the same channel counts; b_dw, b_project: device fp32 [E], [C_out] or
 * NULL for zero (4-byte aligned).  Device-side waits are bounded; a timeout is
 * reported by conv_sync_status.  Stream-ordered. */
conv_status_t conv_mbv2_block_fwd(int N, int H, int W, int C_in, int E, int C_out, const void* x,
                                  const void* wpack, const float* b_dw, const float* b_project,
                                  int has_residual, void* y, void* stream);

/* ---- Fast-Run ([MegEngine] "Fast-Run") ----------------------------------- */

/* Selection phase: time every applicable algorithm for this descriptor on the
 * current device (scratch buffers allocated and freed inside the call;
 * synchronizes the stream), keep the fastest in the process-wide map under
 * the descriptor's key, and return it.  How candidates are measured:
 *   - each one's output on seeded random inputs is first compared with the
 *     direct kernel's; one whose normalized max error exceeds the library's
 *     parity bar (bf16 1e-2, Winograd F(6x6,3x3) 3e-2, fp32 5e-3; int8: any
 *     difference) is rejected and cannot win;
 *   - before every timed run the L2 is flushed by a 256 MB write outside the
 *     timed events (as a layer's input arrives from HBM inside a network);
 *   - candidates are timed round-robin over 21 repetitions (one probe first;
 *     a candidate over 5x the fastest probe keeps that single figure);
 *   - the minimum median wins; an exact tie goes to the lower algorithm id.
 * times_ms (optional, CONV_ALGO_COUNT entries) receives each algorithm's median
 * time in ms, -1 where not applicable, -2 where the output check rejected it.
 * Execution phase: CONV_ALGO_AUTO looks the map up.
 * Environment: GBCONV_LOG=1 prints every candidate's time and the decision
 * (and each map load and conv_algo_resolve) on stderr; GBCONV_FASTRUN_FILE=path
 * loads the map from path, if present, before the first lookup and saves the
 * map there after every selection. */
conv_status_t conv_fastrun_select(conv_desc_t desc, void* stream, conv_algo_t* best,
                                  float* times_ms);
/* Map lookup only; CONV_ERR_NOT_FOUND if the descriptor was never selected. */
conv_status_t conv_fastrun_lookup(conv_desc_t desc, conv_algo_t* algo);
/* Persist / restore the map (text file; entries keyed by descriptor, device
 * name, SM count and library version; entries for another device or version
 * are skipped on load).  A corrupt file returns CONV_ERR_FASTRUN_FILE and
 * leaves the map unchanged. */
conv_status_t conv_fastrun_save(const char* path);
conv_status_t conv_fastrun_load(const char* path);
conv_status_t conv_fastrun_clear(void);

/* ---- layout conversion and pooling -------------------------------------- */

/* NCHW fp32 -> NHWC bf16 (round to nearest even), C_out >= C channels with
 * the extra channels zero ([MegEngine] "Inference Layout": padding the
 * channel axis to the vector width).  Stream-ordered. */
conv_status_t conv_nchw_f32_to_nhwc_bf16(const float* x, void* y, int N, int C, int H, int W,
                                         int C_out, void* stream);
/* NHWC bf16 (C_in >= C channels, first C used) -> NCHW fp32. */
conv_status_t conv_nhwc_bf16_to_nchw_f32(const void* x, float* y, int N, int C, int H, int W,
                                         int C_in, void* stream);
/* NCHW int8 -> NC32HW32 int8 with ceil(C/32) channel blocks, channels past C
 * zero; and back (the first C channels).  Stream-ordered. */
conv_status_t conv_nchw_i8_to_nc32hw32(const void* x, void* y, int N, int C, int H, int W,
                                       void* stream);
conv_status_t conv_nc32hw32_to_nchw_i8(const void* x, void* y, int N, int C, int H, int W,
                                       void* stream);
/* Max pooling, NHWC bf16, window k x k, stride, pad (outside = -inf). */
conv_status_t conv_maxpool2d_nhwc_bf16(const void* x, void* y, int N, int C, int H, int W, int k,
                                       int stride, int pad, void* stream);
/* Global average pooling, NHWC bf16 [N][H][W][C] -> bf16 [N][C]. */
conv_status_t conv_global_avgpool_nhwc_bf16(const void* x, void* y, int N, int C, int H, int W,
                                            void* stream);

/* ---- status ------------------------------------------------------------- */

/* Synchronizes the stream, then reads and clears the device error word:
 * CONV_OK, CONV_ERR_TIMEOUT or CONV_ERR_INTERNAL (or CONV_ERR_CUDA if the
 * synchronization itself failed). */
conv_status_t conv_sync_status(void* stream);
/* Diagnostic of the failure path: enqueues a one-thread kernel that waits on an
 * mbarrier nothing arrives at, through the same bounded wait every tensor-core
 * kernel uses, with a limit of limit_us microseconds (0 < limit_us <= 10 s).
 * The wait runs out, the kernel records a timeout in the device error word and
 * returns (the context stays usable); the next conv_sync_status(stream) then
 * returns CONV_ERR_TIMEOUT and clears the word.  Stream-ordered. */
conv_status_t conv_selftest_wait_timeout(unsigned int limit_us, void* stream);
const char* conv_status_string(conv_status_t status);
/* Reason for the last non-OK status returned on this thread ("" if none). */
const char* conv_last_error_detail(void);
/* Library version string. */
const char* conv_version(void);
/* Number of kernels this library has enqueued, on any stream and from any host
 * thread, since it was loaded: forward, prepack and layout kernels alike.  The
 * difference across a call is the number of kernels that call launched (also
 * while a stream is being captured into a CUDA graph, where it is the number of
 * kernel nodes the call added).  count must not be NULL. */
conv_status_t conv_launch_count(unsigned long long* count);

#ifdef __cplusplus
}
#endif
#endif /* GBCONV_H_ */
