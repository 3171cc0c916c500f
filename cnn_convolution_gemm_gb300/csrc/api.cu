// C-ABI entry points: descriptors, algorithm table, dispatch, Fast-Run map,
// device error word and TMA descriptor encoding.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <map>
#include <mutex>
#include <string>
#include <vector>

#include "internal.h"

#define GBCONV_VERSION "gbconv-0.1"

// ---------------------------------------------------------------------------
// errors

static thread_local char g_detail[512];

conv_status_t gb_fail(conv_status_t st, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_detail, sizeof(g_detail), fmt, ap);
  va_end(ap);
  return st;
}

conv_status_t gb_ok() {
  g_detail[0] = 0;
  return CONV_OK;
}

static conv_status_t ok_status() { return gb_ok(); }

static conv_status_t cuda_fail(cudaError_t e, const char* what) {
  return gb_fail(CONV_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

// Device error word: one int per device in global memory, written by kernels
// with atomicCAS(0 -> code) when a bounded wait runs out or a check fails.
__device__ int g_device_error_word;

static constexpr int kMaxDevices = 64;
static std::mutex g_dev_mu;
static int* g_err_ptr[kMaxDevices];
static int g_num_sms[kMaxDevices];
static long long g_l2_bytes[kMaxDevices];

static int current_device() {
  int dev = 0;
  cudaGetDevice(&dev);
  return dev;
}

int* gb_device_error_word() {
  const int dev = current_device();
  if (dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lk(g_dev_mu);
  if (!g_err_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_device_error_word) != cudaSuccess) return nullptr;
    g_err_ptr[dev] = static_cast<int*>(p);
  }
  return g_err_ptr[dev];
}

int gb_num_sms() {
  const int dev = current_device();
  if (dev < 0 || dev >= kMaxDevices) return 1;
  std::lock_guard<std::mutex> lk(g_dev_mu);
  if (!g_num_sms[dev]) {
    int n = 0;
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    g_num_sms[dev] = n > 0 ? n : 1;
  }
  return g_num_sms[dev];
}

long long gb_l2_bytes() {
  const int dev = current_device();
  if (dev < 0 || dev >= kMaxDevices) return 0;
  std::lock_guard<std::mutex> lk(g_dev_mu);
  if (!g_l2_bytes[dev]) {
    int n = 0;
    cudaDeviceGetAttribute(&n, cudaDevAttrL2CacheSize, dev);
    g_l2_bytes[dev] = n > 0 ? n : 1;
  }
  return g_l2_bytes[dev];
}

cudaError_t gb_set_smem_once(const void* func, int bytes) {
  const int dev = current_device();
  static std::mutex mu;
  static std::map<std::pair<const void*, int>, int> done;  // (kernel, device) -> bytes set
  std::lock_guard<std::mutex> lk(mu);
  auto it = done.find({func, dev});
  if (it != done.end() && it->second >= bytes) return cudaSuccess;
  cudaError_t e = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess) done[{func, dev}] = bytes;
  return e;
}

unsigned long long gb_wait_limit_ns() {
  static unsigned long long v = [] {
    const char* e = getenv("GBCONV_WAIT_LIMIT_MS");
    long long ms = e ? atoll(e) : 2000;
    if (ms <= 0) ms = 2000;
    return (unsigned long long)ms * 1000000ull;
  }();
  return v;
}

// ---------------------------------------------------------------------------
// TMA descriptor encoding through driver entry points (no -lcuda needed).

typedef CUresult (*PFN_encodeTiled)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                    const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                    const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                    CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
typedef CUresult (*PFN_encodeIm2col)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                     const cuuint64_t*, const cuuint64_t*, const int*,
                                     const int*, cuuint32_t, cuuint32_t, const cuuint32_t*,
                                     CUtensorMapInterleave, CUtensorMapSwizzle,
                                     CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static void* driver_fn(const char* name) {
  void* fn = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion(name, &fn, 12000, cudaEnableDefault, &q) != cudaSuccess ||
      q != cudaDriverEntryPointSuccess)
    return nullptr;
  return fn;
}

CUresult gb_encode_tiled(CUtensorMap* map, CUtensorMapDataType dt, cuuint32_t rank, void* addr,
                         const cuuint64_t* dims, const cuuint64_t* strides, const cuuint32_t* box,
                         const cuuint32_t* estr, CUtensorMapSwizzle swz) {
  static PFN_encodeTiled fn = (PFN_encodeTiled)driver_fn("cuTensorMapEncodeTiled");
  if (!fn) return CUDA_ERROR_NOT_FOUND;
  return fn(map, dt, rank, addr, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swz,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
}

CUresult gb_encode_im2col(CUtensorMap* map, CUtensorMapDataType dt, cuuint32_t rank, void* addr,
                          const cuuint64_t* dims, const cuuint64_t* strides, const int* lower,
                          const int* upper, cuuint32_t channels, cuuint32_t pixels,
                          const cuuint32_t* estr, CUtensorMapSwizzle swz) {
  static PFN_encodeIm2col fn = (PFN_encodeIm2col)driver_fn("cuTensorMapEncodeIm2col");
  if (!fn) return CUDA_ERROR_NOT_FOUND;
  return fn(map, dt, rank, addr, dims, strides, lower, upper, channels, pixels, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
}

// ---------------------------------------------------------------------------
// descriptor

static int out_dim(int in, int k, int stride, int pad, int dil) {
  return (int)(((long long)in + 2LL * pad - (long long)dil * (k - 1) - 1) / stride + 1);
}

extern "C" conv_status_t conv_desc_create(conv_desc_t* out, int N, int C, int H, int W, int K,
                                          int R, int S, int stride, int pad, int dilation,
                                          int groups, conv_dtype_t dtype) {
  if (!out) return gb_fail(CONV_ERR_BAD_PARAM, "out is NULL");
  *out = nullptr;
  if (N <= 0 || C <= 0 || H <= 0 || W <= 0 || K <= 0 || R <= 0 || S <= 0)
    return gb_fail(CONV_ERR_BAD_PARAM, "sizes must be positive");
  if (stride <= 0 || dilation <= 0 || pad < 0 || groups <= 0)
    return gb_fail(CONV_ERR_BAD_PARAM, "stride/dilation/groups must be > 0 and pad >= 0");
  if (C % groups || K % groups)
    return gb_fail(CONV_ERR_BAD_PARAM, "C and K must be multiples of groups");
  if (dtype != CONV_BF16 && dtype != CONV_F32 && dtype != CONV_INT8)
    return gb_fail(CONV_ERR_BAD_PARAM, "unknown dtype %d", (int)dtype);
  const int OH = out_dim(H, R, stride, pad, dilation), OW = out_dim(W, S, stride, pad, dilation);
  if (OH <= 0 || OW <= 0) return gb_fail(CONV_ERR_BAD_PARAM, "empty output (OH=%d OW=%d)", OH, OW);
  if ((long long)N * H * W * C >= (1LL << 40) || (long long)N * OH * OW * K >= (1LL << 40))
    return gb_fail(CONV_ERR_BAD_PARAM, "tensor too large");
  gbconv_desc_s* d = new (std::nothrow) gbconv_desc_s{};
  if (!d) return gb_fail(CONV_ERR_BAD_PARAM, "out of host memory");
  d->N = N; d->C = C; d->H = H; d->W = W; d->K = K; d->R = R; d->S = S;
  d->stride = stride; d->pad = pad; d->dil = dilation; d->groups = groups;
  d->dtype = dtype;
  d->layout = CONV_NHWC;
  d->act = CONV_ACT_NONE;
  d->has_residual = 0;
  d->scale = nullptr;
  d->OH = OH;
  d->OW = OW;
  *out = d;
  return ok_status();
}

extern "C" conv_status_t conv_desc_destroy(conv_desc_t desc) {
  delete desc;
  return ok_status();
}

extern "C" conv_status_t conv_desc_set_layout(conv_desc_t d, conv_layout_t layout) {
  if (!d) return gb_fail(CONV_ERR_BAD_PARAM, "desc is NULL");
  if (layout != CONV_NHWC && layout != CONV_NCHW && layout != CONV_NC32HW32)
    return gb_fail(CONV_ERR_BAD_PARAM, "unknown layout");
  if (layout == CONV_NCHW && d->dtype != CONV_F32)
    return gb_fail(CONV_ERR_UNSUPPORTED, "NCHW is accepted for CONV_F32 only");
  if (layout == CONV_NC32HW32 &&
      (d->dtype != CONV_INT8 || d->C % 32 || d->K % 32 || d->groups != 1))
    return gb_fail(CONV_ERR_UNSUPPORTED,
                   "NC32HW32 is accepted for CONV_INT8 with C, K multiples of 32, groups 1");
  d->layout = layout;
  return ok_status();
}

extern "C" conv_status_t conv_desc_set_epilogue(conv_desc_t d, int act, int has_residual) {
  if (!d) return gb_fail(CONV_ERR_BAD_PARAM, "desc is NULL");
  if (act < 0 || act > 2) return gb_fail(CONV_ERR_BAD_PARAM, "act must be 0, 1 or 2");
  if (d->dtype == CONV_INT8 && (act == CONV_ACT_RELU6 || has_residual))
    return gb_fail(CONV_ERR_UNSUPPORTED, "int8 epilogue supports act NONE/RELU, no residual");
  d->act = act;
  d->has_residual = has_residual ? 1 : 0;
  return ok_status();
}

extern "C" conv_status_t conv_desc_set_input_shuffle(conv_desc_t d, int groups) {
  if (!d) return gb_fail(CONV_ERR_BAD_PARAM, "desc is NULL");
  if (groups < 1 || d->C % groups)
    return gb_fail(CONV_ERR_BAD_PARAM, "shuffle groups must divide C");
  d->shuffle_groups = groups > 1 ? groups : 0;
  return ok_status();
}

extern "C" conv_status_t conv_desc_set_requant(conv_desc_t d, const float* scale_dev) {
  if (!d) return gb_fail(CONV_ERR_BAD_PARAM, "desc is NULL");
  if (d->dtype != CONV_INT8) return gb_fail(CONV_ERR_UNSUPPORTED, "requant is for CONV_INT8");
  d->scale = scale_dev;
  return ok_status();
}

extern "C" conv_status_t conv_desc_get_output_dims(conv_desc_t d, int* OH, int* OW) {
  if (!d || !OH || !OW) return gb_fail(CONV_ERR_BAD_PARAM, "NULL argument");
  *OH = d->OH;
  *OW = d->OW;
  return ok_status();
}

// ---------------------------------------------------------------------------
// algorithm table

static const char* const kAlgoNames[CONV_ALGO_COUNT] = {
    "direct", "igemm_tc_n64", "igemm_tc_n128", "igemm_tc_n256",
    "winograd_f2x2_3x3", "winograd_f6x6_3x3", "depthwise3x3", "int8_igemm_mma",
    "int8_igemm_tc", "im2col_gemm", "stem_s2d_igemm", "igemm_tf32",
    "int8_winograd_f2x2_3x3", "stem_s2d4_igemm", "igemm_tc_2sm_n256", "int8_igemm_tc_chunked",
    "igemm_tc_strip_n64"};

static bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Whether algo applies; on false, *why says which requirement failed.
static bool applicable(const gbconv_desc_s& d, int algo, const char** why) {
  const char* dummy;
  if (!why) why = &dummy;
  *why = "";
  const bool nhwc = d.layout == CONV_NHWC;
  if (d.shuffle_groups > 1 && algo != CONV_ALGO_DIRECT && algo != CONV_ALGO_DEPTHWISE)
    return *why = "an input shuffle is honoured by depthwise3x3 and direct only", false;
  switch (algo) {
    case CONV_ALGO_DIRECT:
      if (d.dtype == CONV_INT8 && !d.scale) return *why = "int8 needs a requant scale", false;
      return true;
    case CONV_ALGO_IGEMM_2SM:
      if (d.groups != 1) return *why = "needs groups == 1", false;
      if (d.C == 8) return *why = "8-channel inputs take the narrow tile mode", false;
      [[fallthrough]];
    case CONV_ALGO_IGEMM_N64:
    case CONV_ALGO_IGEMM_N128:
    case CONV_ALGO_IGEMM_N256: {
      if (d.dtype != CONV_BF16 || !nhwc) return *why = "needs bf16 NHWC", false;
      if (d.R != d.S) return *why = "needs a square kernel", false;
      // grouped convs run one GEMM per group over strided channel views
      const int Cg = d.C / d.groups, Kg = d.K / d.groups;
      if (Cg % 8 || Kg % 8) return *why = "needs C/groups and K/groups multiples of 8", false;
      if (d.stride > 8) return *why = "stride > 8", false;
      if (d.pad > 128 || d.pad - d.dil * (d.R - 1) < -128)
        return *why = "padding/dilation outside the TMA im2col range", false;
      if ((long long)d.N * d.OH * d.OW >= (1LL << 31)) return *why = "N*OH*OW >= 2^31", false;
      if ((long long)d.H * d.W * d.C * 2 >= (1LL << 40)) return *why = "image too large", false;
      const int bn = igemm_block_n(algo);
      if (bn == 256 && Kg <= 128) return *why = "K/groups <= 128: use a narrower tile", false;
      if (bn == 128 && Kg <= 64) return *why = "K/groups <= 64: use a narrower tile", false;
      return true;
    }
    case CONV_ALGO_IGEMM_STRIP:
      if ((long long)d.N * d.OH * d.OW >= (1LL << 31)) return *why = "N*OH*OW >= 2^31", false;
      return igemm_strip_applicable(d, why);
    case CONV_ALGO_WINO_F2:
    case CONV_ALGO_WINO_F6:
      if (d.dtype != CONV_BF16 || !nhwc) return *why = "needs bf16 NHWC", false;
      if (d.R != 3 || d.S != 3 || d.stride != 1 || d.dil != 1 || d.groups != 1)
        return *why = "needs 3x3, stride 1, dilation 1, groups 1", false;
      if (d.C % 8 || d.K % 8) return *why = "needs C and K multiples of 8", false;
      return true;
    case CONV_ALGO_DEPTHWISE:
      if (d.dtype != CONV_BF16 || !nhwc) return *why = "needs bf16 NHWC", false;
      if (!(d.groups == d.C && d.K == d.C)) return *why = "needs groups == C == K", false;
      if (d.R != 3 || d.S != 3 || d.dil != 1 || d.stride > 2)
        return *why = "needs 3x3, dilation 1, stride 1 or 2", false;
      if (d.C % 8) return *why = "needs C multiple of 8", false;
      if (d.shuffle_groups > 1 && (d.C > 256 || d.has_residual))
        return *why = "an input shuffle needs C <= 256 and no residual", false;
      return true;
    case CONV_ALGO_INT8_MMA:
      if (d.dtype != CONV_INT8 || !nhwc) return *why = "needs int8 NHWC", false;
      if (!d.scale) return *why = "int8 needs a requant scale", false;
      if (d.groups != 1) return *why = "needs groups == 1", false;
      if (d.C % 16 || d.K % 16) return *why = "needs C and K multiples of 16", false;
      return true;
    case CONV_ALGO_INT8_TC:
    case CONV_ALGO_INT8_TC_CHUNK:
      if (d.dtype != CONV_INT8 || !(nhwc || d.layout == CONV_NC32HW32))
        return *why = "needs int8 NHWC or NC32HW32", false;
      if (!d.scale) return *why = "int8 needs a requant scale", false;
      if (d.groups != 1 || d.R != d.S) return *why = "needs groups == 1, square kernel", false;
      if (d.C % 16 || d.K % 8) return *why = "needs C % 16 == 0 and K % 8 == 0", false;
      if (d.stride > 8 || d.pad > 128 || d.pad - d.dil * (d.R - 1) < -128)
        return *why = "stride/padding outside the TMA im2col range", false;
      if ((long long)d.N * d.OH * d.OW >= (1LL << 31)) return *why = "N*OH*OW >= 2^31", false;
      return true;
    case CONV_ALGO_IM2COL_GEMM:
      if (d.dtype != CONV_BF16 || !nhwc) return *why = "needs bf16 NHWC", false;
      if (d.groups != 1) return *why = "needs groups == 1", false;
      if (d.C % 8 || d.K % 8) return *why = "needs C and K multiples of 8", false;
      if ((long long)d.N * d.OH * d.OW >= (1LL << 31)) return *why = "N*OH*OW >= 2^31", false;
      if (im2col_workspace_bytes(d) > (8ull << 30))
        return *why = "im2col matrix above 8 GiB", false;
      return true;
    case CONV_ALGO_STEM_S2D:
      if (d.dtype != CONV_BF16 || !nhwc) return *why = "needs bf16 NHWC", false;
      return stem_s2d_applicable(d, why);
    case CONV_ALGO_STEM_S2D4:
      if (d.dtype != CONV_BF16 || !nhwc) return *why = "needs bf16 NHWC", false;
      return stem_s2d4_applicable(d, why);
    case CONV_ALGO_INT8_WINO_F2:
      if (d.dtype != CONV_INT8 || !nhwc) return *why = "needs int8 NHWC", false;
      if (!d.scale) return *why = "int8 needs a requant scale", false;
      return int8_wino_applicable(d, why);
    case CONV_ALGO_IGEMM_TF32:
      if (d.dtype != CONV_F32 || !nhwc) return *why = "needs fp32 NHWC", false;
      if (d.groups != 1 || d.R != d.S) return *why = "needs groups == 1, square kernel", false;
      if (d.C % 4 || d.K % 4) return *why = "needs C and K multiples of 4", false;
      if (d.stride > 8 || d.pad > 128 || d.pad - d.dil * (d.R - 1) < -128)
        return *why = "stride/padding outside the TMA im2col range", false;
      if ((long long)d.N * d.OH * d.OW >= (1LL << 31)) return *why = "N*OH*OW >= 2^31", false;
      return true;
    default:
      return *why = "unknown algorithm", false;
  }
}

static bool implemented(int algo);

extern "C" conv_status_t conv_algo_count(conv_desc_t d, int* count) {
  if (!d || !count) return gb_fail(CONV_ERR_BAD_PARAM, "NULL argument");
  *count = CONV_ALGO_COUNT;
  return ok_status();
}

extern "C" conv_status_t conv_algo_info(conv_desc_t d, int i, conv_algo_t* algo,
                                        const char** name, int* is_applicable) {
  if (!d) return gb_fail(CONV_ERR_BAD_PARAM, "desc is NULL");
  if (i < 0 || i >= CONV_ALGO_COUNT) return gb_fail(CONV_ERR_BAD_PARAM, "index out of range");
  if (algo) *algo = i;
  if (name) *name = kAlgoNames[i];
  if (is_applicable) *is_applicable = implemented(i) && applicable(*d, i, nullptr) ? 1 : 0;
  return ok_status();
}

// Heuristic preference when no Fast-Run entry exists.  The MegEngine report's
// table of preferences ("Fast-Run" section) is missing from the page, and its
// text prefers Winograd for 3x3 stride-1 layers on CPUs.  On this GPU the
// implicit GEMM measures 3-4x faster than either Winograd variant on the 3x3
// layers timed, so the order is: the int8 kernels for int8, the depthwise
// kernel for depthwise layers, the space-to-depth stems for narrow stride-2
// convs, tf32 for fp32 tensors, the widest applicable implicit-GEMM tile, and
// direct for what nothing else covers.  Fast-Run still times every candidate.
static int heuristic(const gbconv_desc_s& d) {
  if (d.dtype == CONV_INT8) {
    if (implemented(CONV_ALGO_INT8_TC) && applicable(d, CONV_ALGO_INT8_TC, nullptr))
      return CONV_ALGO_INT8_TC;
    return implemented(CONV_ALGO_INT8_MMA) && applicable(d, CONV_ALGO_INT8_MMA, nullptr)
               ? CONV_ALGO_INT8_MMA
               : CONV_ALGO_DIRECT;
  }
  if (implemented(CONV_ALGO_DEPTHWISE) && applicable(d, CONV_ALGO_DEPTHWISE, nullptr))
    return CONV_ALGO_DEPTHWISE;
  // narrow stride-2 stems: the space-to-depth rewrites
  for (int a : {CONV_ALGO_STEM_S2D4, CONV_ALGO_STEM_S2D})
    if (implemented(a) && applicable(d, a, nullptr)) return a;
  if (d.dtype == CONV_F32)
    return implemented(CONV_ALGO_IGEMM_TF32) && applicable(d, CONV_ALGO_IGEMM_TF32, nullptr)
               ? CONV_ALGO_IGEMM_TF32
               : CONV_ALGO_DIRECT;
  const int order[] = {CONV_ALGO_IGEMM_N256, CONV_ALGO_IGEMM_N128, CONV_ALGO_IGEMM_N64};
  for (int a : order)
    if (implemented(a) && applicable(d, a, nullptr)) return a;
  return CONV_ALGO_DIRECT;
}

// ---------------------------------------------------------------------------
// Fast-Run map: key = descriptor + dtype/layout/epilogue; the file adds the
// device name, SM count and library version.

static std::mutex g_map_mu;
static std::map<std::string, int> g_fastrun;

static std::string desc_key(const gbconv_desc_s& d) {
  char buf[256];
  snprintf(buf, sizeof(buf), "N%d_C%d_H%d_W%d_K%d_R%d_S%d_st%d_p%d_d%d_g%d_t%d_l%d_a%d_r%d_q%d%s",
           d.N, d.C, d.H, d.W, d.K, d.R, d.S, d.stride, d.pad, d.dil, d.groups, (int)d.dtype,
           (int)d.layout, d.act, d.has_residual, d.scale ? 1 : 0,
           d.shuffle_groups > 1 ? ("_sh" + std::to_string(d.shuffle_groups)).c_str() : "");
  return buf;
}

static int lookup_map(const gbconv_desc_s& d) {
  std::lock_guard<std::mutex> lk(g_map_mu);
  auto it = g_fastrun.find(desc_key(d));
  return it == g_fastrun.end() ? -1 : it->second;
}

static void fastrun_autoload();
static bool log_enabled();

static int resolve(const gbconv_desc_s& d, int algo) {
  if (algo != CONV_ALGO_AUTO) return algo;
  fastrun_autoload();
  const int a = lookup_map(d);
  if (a >= 0 && implemented(a) && applicable(d, a, nullptr)) return a;
  return heuristic(d);
}

extern "C" conv_status_t conv_algo_resolve(conv_desc_t d, conv_algo_t* algo) {
  if (!d || !algo) return gb_fail(CONV_ERR_BAD_PARAM, "NULL argument");
  *algo = resolve(*d, CONV_ALGO_AUTO);
  if (log_enabled()) {
    const int m = lookup_map(*d);
    fprintf(stderr, "[gbconv] resolve %s -> %s (%s)\n", desc_key(*d).c_str(), kAlgoNames[*algo],
            m == *algo ? "fastrun map" : "heuristic");
  }
  return ok_status();
}

// ---------------------------------------------------------------------------
// sizes and packing

static size_t elem_bytes(conv_dtype_t t) { return t == CONV_F32 ? 4 : (t == CONV_BF16 ? 2 : 1); }

static size_t user_weight_bytes(const gbconv_desc_s& d) {
  return (size_t)d.K * (d.C / d.groups) * d.R * d.S * elem_bytes(d.dtype);
}

static conv_status_t check_algo(const gbconv_desc_s& d, int algo) {
  if (algo < 0 || algo >= CONV_ALGO_COUNT)
    return gb_fail(CONV_ERR_BAD_PARAM, "algorithm id %d out of range", algo);
  if (!implemented(algo)) return gb_fail(CONV_ERR_UNSUPPORTED, "%s not built", kAlgoNames[algo]);
  const char* why = "";
  if (!applicable(d, algo, &why))
    return gb_fail(CONV_ERR_UNSUPPORTED, "%s does not apply: %s", kAlgoNames[algo], why);
  return CONV_OK;
}

conv_status_t gb_check_algo(const gbconv_desc_s& d, int algo) { return check_algo(d, algo); }

// Split-K for the bf16 implicit GEMMs (groups == 1): when the output tiles
// (128 rows x the algorithm's BN columns) fill at most half the SMs and the
// reduction has at least 16 k-steps, cut it into ranges of at least 4 k-steps,
// as many as the idle SMs allow, each written as fp32 partial products, then
// summed with the epilogue by a second kernel.  The plan depends only on the
// layer and the device, so the workspace size and the forward call agree;
// a forward given less workspace than the plan needs runs unsplit.
struct IgemmSplitPlan {
  int ksplit = 1, kchunk = 0;
  size_t bytes = 0;
};
static IgemmSplitPlan igemm_split_plan(const gbconv_desc_s& d, int a) {
  IgemmSplitPlan pl;
  if (d.groups != 1 || d.dtype != CONV_BF16 || d.x_cstride || d.y_kstride) return pl;
  const long long M = (long long)d.N * d.OH * d.OW;
  const long long tiles = gb_ceil_div_ll(M, 128) * gb_ceil_div(d.K, igemm_block_n(a));
  const int kiters = igemm_kiters(d);
  const int sms = gb_num_sms();
  if (kiters < 16 || tiles * 2 > sms) return pl;
  const int ks = (int)std::min<long long>(sms / tiles, kiters / 4);
  if (ks < 2) return pl;
  pl.kchunk = gb_ceil_div(kiters, ks);
  pl.ksplit = gb_ceil_div(kiters, pl.kchunk);
  pl.bytes = (size_t)pl.ksplit * M * d.K * 4;
  return pl;
}

extern "C" conv_status_t conv_workspace_size(conv_desc_t d, conv_algo_t algo, size_t* bytes) {
  if (!d || !bytes) return gb_fail(CONV_ERR_BAD_PARAM, "NULL argument");
  const int a = resolve(*d, algo);
  conv_status_t st = check_algo(*d, a);
  if (st != CONV_OK) return st;
  *bytes = 0;
  if (a == CONV_ALGO_WINO_F2 || a == CONV_ALGO_WINO_F6)
    *bytes = winograd_workspace_bytes(*d, a == CONV_ALGO_WINO_F2 ? 2 : 6);
  if (a == CONV_ALGO_INT8_TC || a == CONV_ALGO_INT8_TC_CHUNK) *bytes = int8_tc_workspace_bytes(*d, a);
  if (a == CONV_ALGO_IM2COL_GEMM) *bytes = im2col_workspace_bytes(*d);
  if (a == CONV_ALGO_STEM_S2D) *bytes = stem_s2d_workspace_bytes(*d);
  if (a == CONV_ALGO_STEM_S2D4) *bytes = stem_s2d4_workspace_bytes(*d);
  if (a == CONV_ALGO_INT8_WINO_F2) *bytes = int8_wino_workspace_bytes(*d);
  if (a == CONV_ALGO_IGEMM_N64 || a == CONV_ALGO_IGEMM_N128 || a == CONV_ALGO_IGEMM_N256)
    *bytes = igemm_split_plan(*d, a).bytes;
  return ok_status();
}

// One group of a (possibly) grouped conv as a plain conv over strided channel
// views: x channels [g*Cg, (g+1)*Cg) with pixel stride C, y / residual
// channels [g*Kg, (g+1)*Kg) with pixel stride K.
static gbconv_desc_s group_view(const gbconv_desc_s& d) {
  gbconv_desc_s e = d;
  e.C = d.C / d.groups;
  e.K = d.K / d.groups;
  e.groups = 1;
  e.x_cstride = d.C;
  e.y_kstride = d.K;
  return e;
}

// packed implicit-GEMM weights of one group (the layout launch_pack_igemm_weights writes)
static size_t igemm_group_packed_bytes(const gbconv_desc_s& e) {
  return e.C == 8 ? (size_t)e.K * gb_ceil_div(e.R * e.S, 8) * 64 * 2  // 8 taps x 8 ch
                  : (size_t)e.K * e.R * e.S * gb_ceil_div(e.C, 64) * 64 * 2;
}

extern "C" conv_status_t conv_weights_packed_size(conv_desc_t d, conv_algo_t algo,
                                                  size_t* bytes) {
  if (!d || !bytes) return gb_fail(CONV_ERR_BAD_PARAM, "NULL argument");
  const int a = resolve(*d, algo);
  conv_status_t st = check_algo(*d, a);
  if (st != CONV_OK) return st;
  const size_t Cp64 = (size_t)gb_ceil_div(d->C, 64) * 64;
  switch (a) {
    case CONV_ALGO_IGEMM_N64:
    case CONV_ALGO_IGEMM_N128:
    case CONV_ALGO_IGEMM_N256:
    case CONV_ALGO_IGEMM_2SM:
    case CONV_ALGO_IGEMM_STRIP:
      *bytes = igemm_group_packed_bytes(group_view(*d)) * d->groups;
      break;
    case CONV_ALGO_INT8_MMA: *bytes = (size_t)d->K * d->R * d->S * Cp64; break;
    case CONV_ALGO_INT8_TC:
    case CONV_ALGO_INT8_TC_CHUNK: *bytes = int8_tc_packed_bytes(*d, a); break;
    case CONV_ALGO_IM2COL_GEMM: *bytes = im2col_packed_bytes(*d); break;
    case CONV_ALGO_STEM_S2D: *bytes = stem_s2d_packed_bytes(*d); break;
    case CONV_ALGO_STEM_S2D4: *bytes = stem_s2d4_packed_bytes(*d); break;
    case CONV_ALGO_IGEMM_TF32: *bytes = igemm_tf32_packed_bytes(*d); break;
    case CONV_ALGO_INT8_WINO_F2: *bytes = int8_wino_packed_bytes(*d); break;
    case CONV_ALGO_WINO_F2: *bytes = winograd_packed_bytes(*d, 2); break;
    case CONV_ALGO_WINO_F6: *bytes = winograd_packed_bytes(*d, 6); break;
    default: *bytes = user_weight_bytes(*d); break;
  }
  return ok_status();
}

extern "C" conv_status_t conv_weights_prepack(conv_desc_t d, conv_algo_t algo, const void* w,
                                              void* wpack, void* stream) {
  if (!d || !w || !wpack) return gb_fail(CONV_ERR_BAD_PARAM, "NULL argument");
  const int a = resolve(*d, algo);
  conv_status_t st = check_algo(*d, a);
  if (st != CONV_OK) return st;
  if (!aligned16(wpack)) return gb_fail(CONV_ERR_ALIGNMENT, "wpack not 16-byte aligned");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaSuccess;
  switch (a) {
    case CONV_ALGO_IGEMM_N64:
    case CONV_ALGO_IGEMM_N128:
    case CONV_ALGO_IGEMM_N256:
    case CONV_ALGO_IGEMM_2SM:
    case CONV_ALGO_IGEMM_STRIP: {  // per group: weights [Kg][R][S][Cg] -> the group's slice
      const gbconv_desc_s v = group_view(*d);
      const size_t in_g = (size_t)v.K * v.R * v.S * v.C * 2, out_g = igemm_group_packed_bytes(v);
      for (int g = 0; g < d->groups && e == cudaSuccess; ++g)
        e = launch_pack_igemm_weights(v, static_cast<const char*>(w) + g * in_g,
                                      static_cast<char*>(wpack) + g * out_g, s);
      break;
    }
    case CONV_ALGO_INT8_MMA: e = launch_pack_int8_weights(*d, w, wpack, s); break;
    case CONV_ALGO_INT8_TC:
    case CONV_ALGO_INT8_TC_CHUNK: e = launch_pack_int8_tc_weights(*d, a, w, wpack, s); break;
    case CONV_ALGO_IM2COL_GEMM: e = launch_pack_im2col_weights(*d, w, wpack, s); break;
    case CONV_ALGO_STEM_S2D: e = launch_pack_stem_weights(*d, w, wpack, s); break;
    case CONV_ALGO_STEM_S2D4: e = launch_pack_stem4_weights(*d, w, wpack, s); break;
    case CONV_ALGO_IGEMM_TF32: e = launch_pack_tf32_weights(*d, w, wpack, s); break;
    case CONV_ALGO_INT8_WINO_F2: e = launch_pack_int8_wino(*d, w, wpack, s); break;
    case CONV_ALGO_DEPTHWISE: e = launch_pack_dw_weights(*d, w, wpack, s); break;
    case CONV_ALGO_WINO_F2: e = launch_winograd_filter_transform(*d, 2, w, wpack, s); break;
    case CONV_ALGO_WINO_F6: e = launch_winograd_filter_transform(*d, 6, w, wpack, s); break;
    default:
      e = cudaMemcpyAsync(wpack, w, user_weight_bytes(*d), cudaMemcpyDeviceToDevice, s);
      break;
  }
  if (e != cudaSuccess) return cuda_fail(e, "weight prepack");
  return ok_status();
}

// ---------------------------------------------------------------------------
// forward

static conv_status_t fwd_impl(const gbconv_desc_s& d, const void* x, const void* wpack,
                              const void* bias, const void* res, void* y, int a, void* ws,
                              size_t ws_bytes, cudaStream_t s) {
  int* err = gb_device_error_word();
  const unsigned long long wait_ns = gb_wait_limit_ns();
  cudaError_t e = cudaSuccess;
  switch (a) {
    case CONV_ALGO_DIRECT: e = launch_direct(d, x, wpack, bias, res, y, s); break;
    case CONV_ALGO_IGEMM_N64:
    case CONV_ALGO_IGEMM_N128:
    case CONV_ALGO_IGEMM_N256: {  // one launch per group over strided channel views
      const IgemmSplitPlan pl = igemm_split_plan(d, a);
      if (pl.ksplit > 1 && ws && ws_bytes >= pl.bytes && aligned16(ws)) {
        IgemmSplit sp;
        sp.ksplit = pl.ksplit;
        sp.kchunk = pl.kchunk;
        sp.part = static_cast<float*>(ws);
        e = launch_igemm_bf16(d, igemm_block_n(a), x, wpack, nullptr, nullptr, y, err, wait_ns, s,
                              sp);
        if (e == cudaSuccess)
          e = launch_splitk_reduce_bf16(d, pl.ksplit, ws, static_cast<const float*>(bias), res, y,
                                        s);
        break;
      }
      const gbconv_desc_s v = group_view(d);
      const size_t wg = igemm_group_packed_bytes(v);
      for (int g = 0; g < d.groups && e == cudaSuccess; ++g)
        e = launch_igemm_bf16(
            v, igemm_block_n(a), static_cast<const __nv_bfloat16*>(x) + (size_t)g * v.C,
            static_cast<const char*>(wpack) + g * wg,
            bias ? static_cast<const float*>(bias) + (size_t)g * v.K : nullptr,
            res ? static_cast<const __nv_bfloat16*>(res) + (size_t)g * v.K : nullptr,
            static_cast<__nv_bfloat16*>(y) + (size_t)g * v.K, err, wait_ns, s);
      break;
    }
    case CONV_ALGO_IGEMM_2SM:
      e = launch_igemm_bf16_pair(d, x, wpack, static_cast<const float*>(bias), res, y, err,
                                 wait_ns, s);
      break;
    case CONV_ALGO_IGEMM_STRIP:
      e = launch_igemm_strip(d, x, wpack, static_cast<const float*>(bias), y, err, wait_ns, s);
      break;
    case CONV_ALGO_DEPTHWISE:
      e = launch_dwconv3x3(d, x, wpack, static_cast<const float*>(bias), res, y, err, wait_ns, s);
      break;
    case CONV_ALGO_INT8_MMA:
      e = launch_igemm_int8(d, x, wpack, static_cast<const int32_t*>(bias), y, s);
      break;
    case CONV_ALGO_IM2COL_GEMM: {
      const size_t need = im2col_workspace_bytes(d);
      if (!ws || ws_bytes < need)
        return gb_fail(CONV_ERR_WORKSPACE, "workspace of %zu bytes needed", need);
      if (reinterpret_cast<uintptr_t>(ws) & 15u)
        return gb_fail(CONV_ERR_ALIGNMENT, "workspace must be 16-byte aligned");
      e = launch_im2col_gemm(d, x, wpack, static_cast<const float*>(bias), res, y, ws, err,
                             wait_ns, s);
      break;
    }
    case CONV_ALGO_INT8_WINO_F2: {
      const size_t need = int8_wino_workspace_bytes(d);
      if (!ws || ws_bytes < need)
        return gb_fail(CONV_ERR_WORKSPACE, "workspace of %zu bytes needed", need);
      if (reinterpret_cast<uintptr_t>(ws) & 255u)
        return gb_fail(CONV_ERR_ALIGNMENT, "workspace must be 256-byte aligned");
      e = launch_int8_wino(d, x, wpack, static_cast<const int32_t*>(bias), y, ws, err, wait_ns,
                           s);
      break;
    }
    case CONV_ALGO_IGEMM_TF32:
      e = launch_igemm_bf16(d, d.K <= 64 ? 64 : (d.K <= 128 ? 128 : 256), x, wpack,
                            static_cast<const float*>(bias), res, y, err, wait_ns, s);
      break;
    case CONV_ALGO_STEM_S2D: {
      const size_t need = stem_s2d_workspace_bytes(d);
      if (!ws || ws_bytes < need)
        return gb_fail(CONV_ERR_WORKSPACE, "workspace of %zu bytes needed", need);
      if (reinterpret_cast<uintptr_t>(ws) & 255u)
        return gb_fail(CONV_ERR_ALIGNMENT, "workspace must be 256-byte aligned");
      e = launch_stem_s2d(d, x, wpack, static_cast<const float*>(bias), res, y, ws, err, wait_ns,
                          s);
      break;
    }
    case CONV_ALGO_STEM_S2D4: {
      const size_t need = stem_s2d4_workspace_bytes(d);
      if (!ws || ws_bytes < need)
        return gb_fail(CONV_ERR_WORKSPACE, "workspace of %zu bytes needed", need);
      if (reinterpret_cast<uintptr_t>(ws) & 255u)
        return gb_fail(CONV_ERR_ALIGNMENT, "workspace must be 256-byte aligned");
      e = launch_stem_s2d4(d, x, wpack, static_cast<const float*>(bias), y, ws, err, wait_ns, s);
      break;
    }
    case CONV_ALGO_INT8_TC:
    case CONV_ALGO_INT8_TC_CHUNK: {
      const size_t need = int8_tc_workspace_bytes(d, a);
      if (!ws || ws_bytes < need)
        return gb_fail(CONV_ERR_WORKSPACE, "workspace of %zu bytes needed", need);
      if (reinterpret_cast<uintptr_t>(ws) & 255u)
        return gb_fail(CONV_ERR_ALIGNMENT, "workspace must be 256-byte aligned");
      e = launch_int8_tc(d, a, x, wpack, static_cast<const int32_t*>(bias), y, ws, err, wait_ns,
                         s);
      break;
    }
    case CONV_ALGO_WINO_F2:
    case CONV_ALGO_WINO_F6: {
      const int m = a == CONV_ALGO_WINO_F2 ? 2 : 6;
      const size_t need = winograd_workspace_bytes(d, m);
      if (need && (!ws || ws_bytes < need))
        return gb_fail(CONV_ERR_WORKSPACE, "workspace of %zu bytes needed", need);
      e = launch_winograd(d, m, x, wpack, static_cast<const float*>(bias), res, y, ws, err,
                          wait_ns, s);
      break;
    }
    default: return gb_fail(CONV_ERR_UNSUPPORTED, "algorithm %d", a);
  }
  if (e != cudaSuccess) return cuda_fail(e, kAlgoNames[a]);
  return ok_status();
}

extern "C" conv_status_t conv_fwd(conv_desc_t d, const void* x, const void* wpack,
                                  const void* bias, const void* residual, void* y,
                                  conv_algo_t algo, void* ws, size_t ws_bytes, void* stream) {
  if (!d || !x || !wpack || !y) return gb_fail(CONV_ERR_BAD_PARAM, "NULL tensor argument");
  if (d->has_residual && !residual)
    return gb_fail(CONV_ERR_BAD_PARAM, "descriptor has a residual but residual is NULL");
  if (!d->has_residual && residual)
    return gb_fail(CONV_ERR_BAD_PARAM, "residual given but the descriptor has none");
  const int a = resolve(*d, algo);
  conv_status_t st = check_algo(*d, a);
  if (st != CONV_OK) return st;
  if (!aligned16(x) || !aligned16(y) || !aligned16(wpack) || (residual && !aligned16(residual)) ||
      (bias && (reinterpret_cast<uintptr_t>(bias) & 3u)))
    return gb_fail(CONV_ERR_ALIGNMENT, "tensors must be 16-byte aligned (bias 4-byte)");
  if (d->dtype == CONV_INT8 && !d->scale)
    return gb_fail(CONV_ERR_BAD_PARAM, "int8 descriptor has no requant scale");
  return fwd_impl(*d, x, wpack, bias, residual, y, a, ws, ws_bytes,
                  static_cast<cudaStream_t>(stream));
}

// ---------------------------------------------------------------------------
// forward pass on host tensors: chunked copies overlapping the convolution

// bytes of one image of the input (or output) tensor in the descriptor's layout
static size_t image_bytes(const gbconv_desc_s& d, bool input) {
  const size_t c = input ? d.C : d.K;
  const size_t hw = input ? (size_t)d.H * d.W : (size_t)d.OH * d.OW;
  const size_t cp = d.layout == CONV_NC32HW32 ? (c + 31) / 32 * 32 : c;
  return cp * hw * elem_bytes(d.dtype);
}

static size_t round256(size_t b) { return (b + 255) / 256 * 256; }

struct HostPlan {
  int a, n_chunk;
  size_t xb, yb, rb, ws;  // per-chunk buffer bytes (rounded) and the chunk workspace
  size_t total;
};

// the algorithm and chunking for conv_fwd_host; chunks fall back to the whole
// batch when the packed weights of a chunk-sized problem would differ
static conv_status_t host_plan(const gbconv_desc_s& d, conv_algo_t algo, int n_chunk,
                               HostPlan* hp) {
  const int a = resolve(d, algo);
  conv_status_t st = check_algo(d, a);
  if (st != CONV_OK) return st;
  int nc = (n_chunk <= 0 || n_chunk > d.N) ? d.N : n_chunk;
  if (nc < d.N) {
    gbconv_desc_s e = d;
    e.N = nc;
    size_t pf = 0, pc = 0;
    if (!applicable(e, a, nullptr) ||
        conv_weights_packed_size(const_cast<gbconv_desc_s*>(&d), a, &pf) != CONV_OK ||
        conv_weights_packed_size(&e, a, &pc) != CONV_OK || pf != pc)
      nc = d.N;
  }
  gbconv_desc_s e = d;
  e.N = nc;
  size_t ws = 0;
  st = conv_workspace_size(&e, a, &ws);
  if (st != CONV_OK) return st;
  hp->a = a;
  hp->n_chunk = nc;
  hp->xb = round256(image_bytes(d, true) * nc);
  hp->yb = round256(image_bytes(d, false) * nc);
  hp->rb = d.has_residual ? hp->yb : 0;
  hp->ws = round256(ws);
  hp->total = 2 * (hp->xb + hp->yb + hp->rb) + hp->ws;
  return ok_status();
}

extern "C" conv_status_t conv_fwd_host_scratch_size(conv_desc_t d, conv_algo_t algo, int n_chunk,
                                                    size_t* bytes) {
  if (!d || !bytes) return gb_fail(CONV_ERR_BAD_PARAM, "NULL argument");
  HostPlan hp;
  conv_status_t st = host_plan(*d, algo, n_chunk, &hp);
  if (st != CONV_OK) return st;
  *bytes = hp.total;
  return ok_status();
}

namespace {
// the copy streams and the events that order chunks (one set per device)
struct HostPipe {
  cudaStream_t s_in = nullptr, s_out = nullptr;
  cudaEvent_t start = nullptr, in[2] = {}, cv[2] = {}, out[2] = {};
};
std::mutex g_pipe_mu;
std::map<int, HostPipe> g_pipes;

cudaError_t host_pipe(HostPipe** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  HostPipe& p = g_pipes[dev];
  if (!p.s_in) {
    if ((e = cudaStreamCreateWithFlags(&p.s_in, cudaStreamNonBlocking)) != cudaSuccess) return e;
    if ((e = cudaStreamCreateWithFlags(&p.s_out, cudaStreamNonBlocking)) != cudaSuccess) return e;
    cudaEvent_t* evs[] = {&p.start, &p.in[0], &p.in[1], &p.cv[0], &p.cv[1], &p.out[0], &p.out[1]};
    for (cudaEvent_t* ev : evs)
      if ((e = cudaEventCreateWithFlags(ev, cudaEventDisableTiming)) != cudaSuccess) return e;
  }
  *out = &p;
  return cudaSuccess;
}
}  // namespace

extern "C" conv_status_t conv_fwd_host(conv_desc_t d, const void* x_host, const void* wpack,
                                       const void* bias, const void* residual_host, void* y_host,
                                       conv_algo_t algo, int n_chunk, void* scratch,
                                       size_t scratch_bytes, void* stream) {
  if (!d || !x_host || !wpack || !y_host || !scratch)
    return gb_fail(CONV_ERR_BAD_PARAM, "NULL argument");
  if (d->has_residual != (residual_host != nullptr))
    return gb_fail(CONV_ERR_BAD_PARAM, "residual_host must be given exactly when the "
                                       "descriptor has a residual");
  if (d->dtype == CONV_INT8 && !d->scale)
    return gb_fail(CONV_ERR_BAD_PARAM, "int8 descriptor has no requant scale");
  if (reinterpret_cast<uintptr_t>(scratch) & 255u)
    return gb_fail(CONV_ERR_ALIGNMENT, "scratch must be 256-byte aligned");
  if (!aligned16(wpack) || (bias && (reinterpret_cast<uintptr_t>(bias) & 3u)))
    return gb_fail(CONV_ERR_ALIGNMENT, "wpack must be 16-byte aligned (bias 4-byte)");
  HostPlan hp;
  conv_status_t st = host_plan(*d, algo, n_chunk, &hp);
  if (st != CONV_OK) return st;
  if (scratch_bytes < hp.total)
    return gb_fail(CONV_ERR_WORKSPACE, "scratch of %zu bytes needed", hp.total);
  char* base = static_cast<char*>(scratch);
  char* xbuf[2] = {base, base + hp.xb};
  char* ybuf[2] = {base + 2 * hp.xb, base + 2 * hp.xb + hp.yb};
  char* rbuf[2] = {base + 2 * (hp.xb + hp.yb), base + 2 * (hp.xb + hp.yb) + hp.rb};
  char* ws = base + 2 * (hp.xb + hp.yb + hp.rb);
  const size_t xi = image_bytes(*d, true), yi = image_bytes(*d, false);
  cudaStream_t s = static_cast<cudaStream_t>(stream);

  std::lock_guard<std::mutex> lk(g_pipe_mu);
  HostPipe* pp = nullptr;
  cudaError_t e = host_pipe(&pp);
  if (e != cudaSuccess) return cuda_fail(e, "conv_fwd_host streams");
  HostPipe& p = *pp;
  // the copies start after whatever `stream` holds before this call
  if ((e = cudaEventRecord(p.start, s)) != cudaSuccess ||
      (e = cudaStreamWaitEvent(p.s_in, p.start, 0)) != cudaSuccess ||
      (e = cudaStreamWaitEvent(p.s_out, p.start, 0)) != cudaSuccess)
    return cuda_fail(e, "conv_fwd_host ordering");
  const int nch = gb_ceil_div(d->N, hp.n_chunk);
  for (int i = 0; i < nch; ++i) {
    const int slot = i & 1;
    const int n0 = i * hp.n_chunk, nc = std::min(hp.n_chunk, d->N - n0);
    // input copies: slot free once the convolution of chunk i - 2 has read it
    if (i >= 2 && (e = cudaStreamWaitEvent(p.s_in, p.cv[slot], 0)) != cudaSuccess) break;
    if ((e = cudaMemcpyAsync(xbuf[slot], static_cast<const char*>(x_host) + n0 * xi, nc * xi,
                             cudaMemcpyHostToDevice, p.s_in)) != cudaSuccess)
      break;
    if (residual_host &&
        (e = cudaMemcpyAsync(rbuf[slot], static_cast<const char*>(residual_host) + n0 * yi,
                             nc * yi, cudaMemcpyHostToDevice, p.s_in)) != cudaSuccess)
      break;
    if ((e = cudaEventRecord(p.in[slot], p.s_in)) != cudaSuccess) break;
    // the convolution of chunk i on `stream`: after its input landed and after
    // the output copy of chunk i - 2 has drained the output slot
    if ((e = cudaStreamWaitEvent(s, p.in[slot], 0)) != cudaSuccess) break;
    if (i >= 2 && (e = cudaStreamWaitEvent(s, p.out[slot], 0)) != cudaSuccess) break;
    gbconv_desc_s c = *d;
    c.N = nc;
    st = fwd_impl(c, xbuf[slot], wpack, bias, residual_host ? rbuf[slot] : nullptr, ybuf[slot],
                  hp.a, ws, hp.ws, s);
    if (st != CONV_OK) return st;
    if ((e = cudaEventRecord(p.cv[slot], s)) != cudaSuccess) break;
    // output copy of chunk i
    if ((e = cudaStreamWaitEvent(p.s_out, p.cv[slot], 0)) != cudaSuccess) break;
    if ((e = cudaMemcpyAsync(static_cast<char*>(y_host) + n0 * yi, ybuf[slot], nc * yi,
                             cudaMemcpyDeviceToHost, p.s_out)) != cudaSuccess)
      break;
    if ((e = cudaEventRecord(p.out[slot], p.s_out)) != cudaSuccess) break;
  }
  if (e != cudaSuccess) return cuda_fail(e, "conv_fwd_host");
  // `stream` continues after every output copy (the last one of each slot)
  for (int slot = 0; slot < 2 && slot < nch; ++slot)
    if ((e = cudaStreamWaitEvent(s, p.out[slot], 0)) != cudaSuccess)
      return cuda_fail(e, "conv_fwd_host ordering");
  return ok_status();
}


// ---------------------------------------------------------------------------
// fused MobileNetV2 block

static conv_status_t mbv2_check(int C_in, int E, int C_out) {
  if (C_in <= 0 || E <= 0 || C_out <= 0) return gb_fail(CONV_ERR_BAD_PARAM, "bad channel counts");
  if (!mbv2_block_supported(C_in, E, C_out))
    return gb_fail(CONV_ERR_UNSUPPORTED,
                   "fused block supports E = 144, C_in in {8, 16, 24}, C_out a multiple of 8 "
                   "in [8, 32]");
  return CONV_OK;
}

extern "C" conv_status_t conv_mbv2_block_packed_size(int C_in, int E, int C_out, size_t* bytes) {
  if (!bytes) return gb_fail(CONV_ERR_BAD_PARAM, "NULL argument");
  conv_status_t st = mbv2_check(C_in, E, C_out);
  if (st != CONV_OK) return st;
  *bytes = mbv2_block_packed_bytes(E);
  return ok_status();
}

extern "C" conv_status_t conv_mbv2_block_prepack(int C_in, int E, int C_out, const void* w_expand,
                                                 const float* b_expand, const void* w_dw,
                                                 const void* w_project, void* wpack,
                                                 void* stream) {
  if (!w_expand || !w_dw || !w_project || !wpack)
    return gb_fail(CONV_ERR_BAD_PARAM, "NULL argument");
  conv_status_t st = mbv2_check(C_in, E, C_out);
  if (st != CONV_OK) return st;
  if (!aligned16(wpack)) return gb_fail(CONV_ERR_ALIGNMENT, "wpack not 16-byte aligned");
  if ((reinterpret_cast<uintptr_t>(w_expand) | reinterpret_cast<uintptr_t>(w_dw) |
       reinterpret_cast<uintptr_t>(w_project)) & 1u)
    return gb_fail(CONV_ERR_ALIGNMENT, "bf16 weights must be 2-byte aligned");
  if (reinterpret_cast<uintptr_t>(b_expand) & 3u)
    return gb_fail(CONV_ERR_ALIGNMENT, "b_expand must be 4-byte aligned");
  cudaError_t e = launch_pack_mbv2(C_in, E, C_out, w_expand, b_expand, w_dw, w_project, wpack,
                                   static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? ok_status() : cuda_fail(e, "mbv2 prepack");
}

extern "C" conv_status_t conv_mbv2_block_fwd(int N, int H, int W, int C_in, int E, int C_out,
                                             const void* x, const void* wpack, const float* b_dw,
                                             const float* b_project, int has_residual, void* y,
                                             void* stream) {
  if (!x || !wpack || !y) return gb_fail(CONV_ERR_BAD_PARAM, "NULL tensor argument");
  if (N <= 0 || H <= 0 || W <= 0) return gb_fail(CONV_ERR_BAD_PARAM, "bad sizes");
  conv_status_t st = mbv2_check(C_in, E, C_out);
  if (st != CONV_OK) return st;
  if (has_residual && C_in != C_out)
    return gb_fail(CONV_ERR_BAD_PARAM, "the residual needs C_in == C_out");
  if (!aligned16(x) || !aligned16(y) || !aligned16(wpack) ||
      ((reinterpret_cast<uintptr_t>(b_dw) | reinterpret_cast<uintptr_t>(b_project)) & 3u))
    return gb_fail(CONV_ERR_ALIGNMENT, "tensors must be 16-byte aligned (biases 4-byte)");
  cudaError_t e = launch_mbv2_block(N, H, W, C_in, E, C_out, x, wpack, b_dw, b_project,
                                    has_residual, y, gb_device_error_word(), gb_wait_limit_ns(),
                                    static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? ok_status() : cuda_fail(e, "mbv2 block");
}

// ---------------------------------------------------------------------------
// Fast-Run selection: time every applicable algorithm on scratch tensors.
//
// The MegEngine report's Fast-Run searches every implemented operator on the
// target device and keeps the best in a map.  Here each candidate is measured
// the way the layer runs in a network pass: its output is first checked
// against the direct kernel's (so a candidate that computes something else
// cannot win), then every timed run starts with the L2 flushed (a 256 MB write
// outside the timed events: a layer's input in a network arrives from HBM, and
// a warm 129 MB L2 would favour memory-bound candidates), and the candidates
// take turns round-robin across the repetitions so a slow drift of the clocks
// lands on all of them alike.  The minimum median wins; an exact tie goes to
// the lower id.

namespace {
struct DevBuf {
  void* p = nullptr;
  DevBuf() = default;
  DevBuf(const DevBuf&) = delete;
  DevBuf& operator=(const DevBuf&) = delete;
  DevBuf(DevBuf&& o) noexcept : p(o.p) { o.p = nullptr; }
  ~DevBuf() {
    if (p) cudaFree(p);
  }
  cudaError_t alloc(size_t n) { return cudaMalloc(&p, n ? n : 16); }
};

constexpr size_t kFastRunFlushBytes = 256ull << 20;  // twice the L2
constexpr int kFastRunReps = 21;

// normalized max error a candidate may show against the direct kernel: the
// parity bars of the library's tests (int8: exact)
float fastrun_tolerance(const gbconv_desc_s& d, int a) {
  if (d.dtype == CONV_INT8) return 0.f;
  if (d.dtype == CONV_F32) return 5e-3f;
  return a == CONV_ALGO_WINO_F6 ? 3e-2f : 1e-2f;
}
}  // namespace

// GBCONV_LOG=1: Fast-Run decisions, map loads and AUTO resolutions on stderr.
static bool log_enabled() {
  static const bool on = [] {
    const char* e = getenv("GBCONV_LOG");
    return e && *e && strcmp(e, "0") != 0;
  }();
  return on;
}

// GBCONV_FASTRUN_FILE=path: the map is loaded from path (if it exists) before
// the first lookup, and saved there after every selection.
static const char* fastrun_file() {
  static const char* f = [] {
    const char* e = getenv("GBCONV_FASTRUN_FILE");
    return (e && *e) ? e : nullptr;
  }();
  return f;
}

static void fastrun_autoload() {
  static std::once_flag once;
  std::call_once(once, [] {
    const char* f = fastrun_file();
    if (!f) return;
    FILE* t = fopen(f, "r");
    if (!t) return;  // not written yet
    fclose(t);
    const conv_status_t st = conv_fastrun_load(f);
    if (log_enabled())
      fprintf(stderr, "[gbconv] fastrun map %s: %s\n", f,
              st == CONV_OK ? "loaded" : conv_last_error_detail());
  });
}

extern "C" conv_status_t conv_fastrun_select(conv_desc_t d, void* stream, conv_algo_t* best,
                                             float* times_ms) {
  if (!d || !best) return gb_fail(CONV_ERR_BAD_PARAM, "NULL argument");
  fastrun_autoload();
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const size_t eb = elem_bytes(d->dtype);
  const size_t xb = (size_t)d->N * d->C * d->H * d->W * eb;
  const long long ny = (long long)d->N * d->K * d->OH * d->OW;
  const size_t yb = (size_t)ny * eb;
  const size_t bb = (size_t)d->K * 4;
  DevBuf x, y, yref, res, bias, w, scale, flush, cmp;
  cudaError_t e;
  if ((e = x.alloc(xb)) != cudaSuccess || (e = y.alloc(yb)) != cudaSuccess ||
      (e = yref.alloc(yb)) != cudaSuccess || (e = bias.alloc(bb)) != cudaSuccess ||
      (e = w.alloc(user_weight_bytes(*d))) != cudaSuccess ||
      (e = flush.alloc(kFastRunFlushBytes)) != cudaSuccess ||
      (e = cmp.alloc(3 * sizeof(unsigned))) != cudaSuccess)
    return cuda_fail(e, "fastrun scratch");
  if (d->has_residual && (e = res.alloc(yb)) != cudaSuccess) return cuda_fail(e, "fastrun");
  gbconv_desc_s dd = *d;
  std::vector<float> sc;
  if (d->dtype == CONV_INT8) {
    if ((e = scale.alloc((size_t)d->K * 4)) != cudaSuccess) return cuda_fail(e, "fastrun");
    sc.assign(d->K, 1e-4f);
    cudaMemcpyAsync(scale.p, sc.data(), sc.size() * 4, cudaMemcpyHostToDevice, s);
    dd.scale = static_cast<const float*>(scale.p);
  }
  const int esz = d->dtype == CONV_F32 ? 4 : (d->dtype == CONV_BF16 ? 2 : 1);
  launch_fill_random(x.p, xb, esz, 1u, s);
  launch_fill_random(w.p, user_weight_bytes(*d), esz, 2u, s);
  cudaMemsetAsync(bias.p, 0, bb, s);
  if (res.p) launch_fill_random(res.p, yb, esz, 3u, s);
  auto flush_l2 = [&] { return cudaMemsetAsync(flush.p, 0, kFastRunFlushBytes, s); };

  float tms[CONV_ALGO_COUNT];
  float err_of[CONV_ALGO_COUNT];
  for (int a = 0; a < CONV_ALGO_COUNT; ++a) tms[a] = -1.f, err_of[a] = -1.f;

  // the reference output: the direct kernel (applies to every descriptor)
  bool have_ref = false;
  {
    DevBuf wp;
    size_t pb = 0;
    if (applicable(dd, CONV_ALGO_DIRECT, nullptr) &&
        conv_weights_packed_size(&dd, CONV_ALGO_DIRECT, &pb) == CONV_OK &&
        wp.alloc(pb) == cudaSuccess &&
        conv_weights_prepack(&dd, CONV_ALGO_DIRECT, w.p, wp.p, s) == CONV_OK &&
        fwd_impl(dd, x.p, wp.p, bias.p, res.p, yref.p, CONV_ALGO_DIRECT, nullptr, 0, s) == CONV_OK)
      have_ref = cudaStreamSynchronize(s) == cudaSuccess;
    cudaGetLastError();
  }

  struct Cand {
    int a;
    DevBuf wp, ws;
    size_t wsb = 0;
    std::vector<float> t;
  };
  std::vector<Cand> cands;
  for (int a = 0; a < CONV_ALGO_COUNT; ++a) {
    if (!implemented(a) || !applicable(dd, a, nullptr)) continue;
    Cand c;
    c.a = a;
    size_t pb = 0;
    if (conv_weights_packed_size(&dd, a, &pb) != CONV_OK) continue;
    if (conv_workspace_size(&dd, a, &c.wsb) != CONV_OK) continue;
    if (c.wp.alloc(pb) != cudaSuccess || c.ws.alloc(c.wsb) != cudaSuccess) {
      cudaGetLastError();
      continue;
    }
    if (conv_weights_prepack(&dd, a, w.p, c.wp.p, s) != CONV_OK) continue;
    // first run: loads the kernels and produces the output that is checked
    if (fwd_impl(dd, x.p, c.wp.p, bias.p, res.p, y.p, a, c.ws.p, c.wsb, s) != CONV_OK) continue;
    if (have_ref && a != CONV_ALGO_DIRECT) {
      unsigned h[3] = {0, 0, 0};
      if (launch_compare_outputs(y.p, yref.p, ny, (int)dd.dtype, static_cast<unsigned*>(cmp.p),
                                 s) != cudaSuccess ||
          cudaMemcpyAsync(h, cmp.p, sizeof(h), cudaMemcpyDeviceToHost, s) != cudaSuccess ||
          cudaStreamSynchronize(s) != cudaSuccess) {
        cudaGetLastError();
        continue;
      }
      float md, mb;
      memcpy(&md, &h[0], 4);
      memcpy(&mb, &h[1], 4);
      const float rel = mb > 0.f ? md / mb : md;
      err_of[a] = rel;
      const float tol = fastrun_tolerance(dd, a);
      if (h[2] != 0 || !(rel <= tol)) {
        tms[a] = -2.f;  // rejected: its output disagrees with the direct kernel's
        if (log_enabled())
          fprintf(stderr, "[gbconv] fastrun %s: %s rejected (error %.3g > %.3g, %u bad)\n",
                  desc_key(*d).c_str(), kAlgoNames[a], rel, tol, h[2]);
        continue;
      }
    }
    cands.push_back(std::move(c));
  }

  cudaEvent_t e0, e1;
  cudaEventCreate(&e0);
  cudaEventCreate(&e1);
  auto time_once = [&](Cand& c, float* ms) {
    if (flush_l2() != cudaSuccess) return false;
    cudaEventRecord(e0, s);
    const bool ok = fwd_impl(dd, x.p, c.wp.p, bias.p, res.p, y.p, c.a, c.ws.p, c.wsb, s) == CONV_OK;
    cudaEventRecord(e1, s);
    if (cudaEventSynchronize(e1) != cudaSuccess) return false;
    cudaEventElapsedTime(ms, e0, e1);
    return ok;
  };
  // one probe each; a candidate over 5x the fastest probe keeps that one figure
  std::vector<float> probe(cands.size(), -1.f);
  float best_probe = 0.f;
  for (size_t i = 0; i < cands.size(); ++i)
    if (time_once(cands[i], &probe[i]) && (best_probe == 0.f || probe[i] < best_probe))
      best_probe = probe[i];
  std::vector<size_t> live;
  for (size_t i = 0; i < cands.size(); ++i) {
    if (probe[i] < 0.f) continue;
    if (probe[i] > 5.f * best_probe)
      tms[cands[i].a] = probe[i];
    else
      live.push_back(i);
  }
  // repetitions, interleaved: rep r starts at candidate r mod count
  bool ok = true;
  for (int r = 0; r < kFastRunReps && ok && !live.empty(); ++r)
    for (size_t j = 0; j < live.size() && ok; ++j) {
      Cand& c = cands[live[(j + r) % live.size()]];
      float ms = 0.f;
      ok = time_once(c, &ms);
      c.t.push_back(ms);
    }
  cudaEventDestroy(e0);
  cudaEventDestroy(e1);
  if (ok)
    for (size_t i : live) {
      std::vector<float> t = cands[i].t;
      std::sort(t.begin(), t.end());
      tms[cands[i].a] = t[t.size() / 2];
    }
  int best_a = -1;
  for (int a = 0; a < CONV_ALGO_COUNT; ++a)
    if (tms[a] >= 0.f && (best_a < 0 || tms[a] < tms[best_a])) best_a = a;
  int* err = gb_device_error_word();
  int code = 0;
  if (err) {
    cudaMemcpy(&code, err, 4, cudaMemcpyDeviceToHost);
    if (code) cudaMemset(err, 0, 4);
  }
  if (code) return gb_fail(code == DEV_ERR_TIMEOUT ? CONV_ERR_TIMEOUT : CONV_ERR_INTERNAL,
                           "device error during Fast-Run timing");
  if (!ok) return gb_fail(CONV_ERR_CUDA, "Fast-Run timing failed");
  if (best_a < 0) return gb_fail(CONV_ERR_UNSUPPORTED, "no applicable algorithm ran");
  {
    std::lock_guard<std::mutex> lk(g_map_mu);
    g_fastrun[desc_key(*d)] = best_a;
  }
  if (log_enabled()) {
    std::string line = "[gbconv] fastrun " + desc_key(*d) + ":";
    char buf[160];
    for (int a = 0; a < CONV_ALGO_COUNT; ++a) {
      if (tms[a] == -1.f) continue;
      if (tms[a] == -2.f)
        snprintf(buf, sizeof(buf), " %s=rejected", kAlgoNames[a]);
      else if (err_of[a] >= 0.f)
        snprintf(buf, sizeof(buf), " %s=%.4fms(err %.1e)", kAlgoNames[a], tms[a], err_of[a]);
      else
        snprintf(buf, sizeof(buf), " %s=%.4fms", kAlgoNames[a], tms[a]);
      line += buf;
    }
    fprintf(stderr, "%s -> %s\n", line.c_str(), kAlgoNames[best_a]);
  }
  if (const char* f = fastrun_file()) {
    const conv_status_t st = conv_fastrun_save(f);
    if (st != CONV_OK) return st;
  }
  *best = best_a;
  if (times_ms) memcpy(times_ms, tms, sizeof(tms));
  return ok_status();
}

extern "C" conv_status_t conv_fastrun_lookup(conv_desc_t d, conv_algo_t* algo) {
  if (!d || !algo) return gb_fail(CONV_ERR_BAD_PARAM, "NULL argument");
  fastrun_autoload();
  const int a = lookup_map(*d);
  if (a < 0) return gb_fail(CONV_ERR_NOT_FOUND, "no Fast-Run entry");
  *algo = a;
  return ok_status();
}

static std::string device_tag() {
  int dev = 0;
  cudaDeviceProp prop;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaGetDeviceProperties(&prop, dev) != cudaSuccess) {
    cudaGetLastError();
    return "nodevice";
  }
  std::string name = prop.name;
  for (char& c : name)
    if (c == ' ' || c == '\t') c = '_';
  return name + "_sm" + std::to_string(prop.multiProcessorCount);
}

extern "C" conv_status_t conv_fastrun_save(const char* path) {
  if (!path) return gb_fail(CONV_ERR_BAD_PARAM, "path is NULL");
  FILE* f = fopen(path, "w");
  if (!f) return gb_fail(CONV_ERR_FASTRUN_FILE, "cannot open %s for writing", path);
  const std::string tag = device_tag();
  std::lock_guard<std::mutex> lk(g_map_mu);
  fprintf(f, "# gbconv fastrun map\nversion %s\n", GBCONV_VERSION);
  for (auto& kv : g_fastrun)
    fprintf(f, "entry %s %s %s\n", tag.c_str(), kv.first.c_str(), kAlgoNames[kv.second]);
  fprintf(f, "end %zu\n", g_fastrun.size());
  const bool bad = ferror(f) != 0;
  fclose(f);
  if (bad) return gb_fail(CONV_ERR_FASTRUN_FILE, "write error on %s", path);
  return ok_status();
}

extern "C" conv_status_t conv_fastrun_load(const char* path) {
  if (!path) return gb_fail(CONV_ERR_BAD_PARAM, "path is NULL");
  FILE* f = fopen(path, "r");
  if (!f) return gb_fail(CONV_ERR_FASTRUN_FILE, "cannot open %s", path);
  const std::string tag = device_tag();
  std::map<std::string, int> fresh;
  char line[1024];
  bool saw_version = false, saw_end = false, version_ok = false;
  size_t entries = 0, declared = 0;
  bool corrupt = false;
  while (fgets(line, sizeof(line), f)) {
    if (line[0] == '#' || line[0] == '\n') continue;
    char a[256], b[512], c[128];
    if (!saw_version) {
      if (sscanf(line, "version %255s", a) != 1) { corrupt = true; break; }
      saw_version = true;
      version_ok = strcmp(a, GBCONV_VERSION) == 0;
      continue;
    }
    if (sscanf(line, "end %zu", &declared) == 1) { saw_end = true; break; }
    if (sscanf(line, "entry %255s %511s %127s", a, b, c) != 3) { corrupt = true; break; }
    ++entries;
    int id = -1;
    for (int i = 0; i < CONV_ALGO_COUNT; ++i)
      if (strcmp(c, kAlgoNames[i]) == 0) id = i;
    if (id < 0) { corrupt = true; break; }
    if (version_ok && tag == a) fresh[b] = id;  // other devices/versions are skipped
  }
  fclose(f);
  if (corrupt || !saw_version || !saw_end || declared != entries)
    return gb_fail(CONV_ERR_FASTRUN_FILE, "corrupt Fast-Run file %s", path);
  std::lock_guard<std::mutex> lk(g_map_mu);
  for (auto& kv : fresh) g_fastrun[kv.first] = kv.second;
  if (log_enabled())
    fprintf(stderr, "[gbconv] fastrun load %s: %zu entries for %s, %zu skipped (other device or "
            "version)\n", path, fresh.size(), tag.c_str(), entries - fresh.size());
  return ok_status();
}

extern "C" conv_status_t conv_fastrun_clear(void) {
  std::lock_guard<std::mutex> lk(g_map_mu);
  g_fastrun.clear();
  return ok_status();
}

// ---------------------------------------------------------------------------
// layout conversion and pooling

extern "C" conv_status_t conv_nchw_f32_to_nhwc_bf16(const float* x, void* y, int N, int C, int H,
                                                    int W, int C_out, void* stream) {
  if (!x || !y) return gb_fail(CONV_ERR_BAD_PARAM, "NULL argument");
  if (N <= 0 || C <= 0 || H <= 0 || W <= 0 || C_out < C)
    return gb_fail(CONV_ERR_BAD_PARAM, "bad sizes");
  cudaError_t e =
      launch_nchw_f32_to_nhwc_bf16(x, y, N, C, H, W, C_out, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? ok_status() : cuda_fail(e, "nchw->nhwc");
}

extern "C" conv_status_t conv_nhwc_bf16_to_nchw_f32(const void* x, float* y, int N, int C, int H,
                                                    int W, int C_in, void* stream) {
  if (!x || !y) return gb_fail(CONV_ERR_BAD_PARAM, "NULL argument");
  if (N <= 0 || C <= 0 || H <= 0 || W <= 0 || C_in < C)
    return gb_fail(CONV_ERR_BAD_PARAM, "bad sizes");
  cudaError_t e =
      launch_nhwc_bf16_to_nchw_f32(x, y, N, C, H, W, C_in, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? ok_status() : cuda_fail(e, "nhwc->nchw");
}

extern "C" conv_status_t conv_nchw_i8_to_nc32hw32(const void* x, void* y, int N, int C, int H,
                                                  int W, void* stream) {
  if (!x || !y) return gb_fail(CONV_ERR_BAD_PARAM, "NULL argument");
  if (N <= 0 || C <= 0 || H <= 0 || W <= 0) return gb_fail(CONV_ERR_BAD_PARAM, "bad sizes");
  cudaError_t e = launch_nc32_convert(x, y, N, C, H, W, 1, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? ok_status() : cuda_fail(e, "nchw->nc32hw32");
}

extern "C" conv_status_t conv_nc32hw32_to_nchw_i8(const void* x, void* y, int N, int C, int H,
                                                  int W, void* stream) {
  if (!x || !y) return gb_fail(CONV_ERR_BAD_PARAM, "NULL argument");
  if (N <= 0 || C <= 0 || H <= 0 || W <= 0) return gb_fail(CONV_ERR_BAD_PARAM, "bad sizes");
  cudaError_t e = launch_nc32_convert(x, y, N, C, H, W, 0, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? ok_status() : cuda_fail(e, "nc32hw32->nchw");
}

extern "C" conv_status_t conv_maxpool2d_nhwc_bf16(const void* x, void* y, int N, int C, int H,
                                                  int W, int k, int stride, int pad,
                                                  void* stream) {
  if (!x || !y) return gb_fail(CONV_ERR_BAD_PARAM, "NULL argument");
  if (N <= 0 || C <= 0 || H <= 0 || W <= 0 || k <= 0 || stride <= 0 || pad < 0 || pad >= k)
    return gb_fail(CONV_ERR_BAD_PARAM, "bad sizes");
  if (C % 8 || !aligned16(x) || !aligned16(y))
    return gb_fail(CONV_ERR_ALIGNMENT, "needs C % 8 == 0 and 16-byte aligned tensors");
  cudaError_t e =
      launch_maxpool_nhwc_bf16(x, y, N, C, H, W, k, stride, pad, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? ok_status() : cuda_fail(e, "maxpool");
}

extern "C" conv_status_t conv_global_avgpool_nhwc_bf16(const void* x, void* y, int N, int C,
                                                       int H, int W, void* stream) {
  if (!x || !y) return gb_fail(CONV_ERR_BAD_PARAM, "NULL argument");
  if (N <= 0 || C <= 0 || H <= 0 || W <= 0) return gb_fail(CONV_ERR_BAD_PARAM, "bad sizes");
  if (C % 8 || !aligned16(x) || !aligned16(y))
    return gb_fail(CONV_ERR_ALIGNMENT, "needs C % 8 == 0 and 16-byte aligned tensors");
  cudaError_t e = launch_avgpool_nhwc_bf16(x, y, N, C, H, W, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? ok_status() : cuda_fail(e, "avgpool");
}

// ---------------------------------------------------------------------------
// status

extern "C" conv_status_t conv_selftest_wait_timeout(unsigned int limit_us, void* stream) {
  if (limit_us == 0 || limit_us > 10u * 1000u * 1000u)
    return gb_fail(CONV_ERR_BAD_PARAM, "limit_us must be in (0, 10 s]");
  int* err = gb_device_error_word();
  if (!err) return gb_fail(CONV_ERR_CUDA, "device error word unavailable");
  cudaError_t e = launch_selftest_wait_timeout(err, (unsigned long long)limit_us * 1000ull,
                                               static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "self-test launch");
  return ok_status();
}

extern "C" conv_status_t conv_sync_status(void* stream) {
  cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "stream synchronize");
  int* err = gb_device_error_word();
  if (!err) return gb_fail(CONV_ERR_CUDA, "device error word unavailable");
  int code = 0;
  e = cudaMemcpy(&code, err, sizeof(int), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(e, "read device error word");
  if (code) {
    cudaMemset(err, 0, sizeof(int));
    return gb_fail(code == DEV_ERR_TIMEOUT ? CONV_ERR_TIMEOUT : CONV_ERR_INTERNAL,
                   "device error word = %d", code);
  }
  return ok_status();
}

extern "C" const char* conv_status_string(conv_status_t s) {
  switch (s) {
    case CONV_OK: return "CONV_OK";
    case CONV_ERR_BAD_PARAM: return "CONV_ERR_BAD_PARAM";
    case CONV_ERR_UNSUPPORTED: return "CONV_ERR_UNSUPPORTED";
    case CONV_ERR_ALIGNMENT: return "CONV_ERR_ALIGNMENT";
    case CONV_ERR_WORKSPACE: return "CONV_ERR_WORKSPACE";
    case CONV_ERR_CUDA: return "CONV_ERR_CUDA";
    case CONV_ERR_TIMEOUT: return "CONV_ERR_TIMEOUT";
    case CONV_ERR_INTERNAL: return "CONV_ERR_INTERNAL";
    case CONV_ERR_FASTRUN_FILE: return "CONV_ERR_FASTRUN_FILE";
    case CONV_ERR_NOT_FOUND: return "CONV_ERR_NOT_FOUND";
    default: return "CONV_ERR_UNKNOWN";
  }
}

extern "C" const char* conv_last_error_detail(void) { return g_detail; }

static std::atomic<unsigned long long> g_launches{0};

void gb_count_launch() { g_launches.fetch_add(1, std::memory_order_relaxed); }

extern "C" conv_status_t conv_launch_count(unsigned long long* count) {
  if (!count) return gb_fail(CONV_ERR_BAD_PARAM, "count is NULL");
  *count = g_launches.load(std::memory_order_relaxed);
  return ok_status();
}

extern "C" const char* conv_version(void) { return GBCONV_VERSION; }

// Algorithms whose kernels are built into this library.
static bool implemented(int algo) {
  switch (algo) {
    case CONV_ALGO_DIRECT:
    case CONV_ALGO_IGEMM_N64:
    case CONV_ALGO_IGEMM_N128:
    case CONV_ALGO_IGEMM_N256:
    case CONV_ALGO_IGEMM_2SM:
    case CONV_ALGO_DEPTHWISE:
    case CONV_ALGO_WINO_F2:
    case CONV_ALGO_WINO_F6:
    case CONV_ALGO_INT8_MMA:
    case CONV_ALGO_INT8_TC:
    case CONV_ALGO_IM2COL_GEMM:
    case CONV_ALGO_STEM_S2D:
    case CONV_ALGO_STEM_S2D4:
    case CONV_ALGO_IGEMM_TF32:
    case CONV_ALGO_INT8_WINO_F2:
    case CONV_ALGO_INT8_TC_CHUNK:
    case CONV_ALGO_IGEMM_STRIP:
      return true;
    default:
      return false;
  }
}
