// Allocation-free Winograd forward: the same kernels as conv_fwd's Winograd
// algorithms, with their scratch (the transformed input tiles V and the fp32
// products M) taken from a fixed array in device global memory instead of a
// caller-provided workspace.
//
// Who needs this: callers that must not allocate device memory at call time —
// a plugin inside a host framework whose memory manager owns every device
// allocation, code on a latency-critical path where a cudaMalloc (or a
// caching-allocator pool growing) would stall or synchronize the device, or a
// deployment with a fixed memory budget decided at load time.  They pass only
// inputs and outputs.
//
// Limits and sharing:
//   * the scratch array is kNoAllocScratchBytes (24 MiB) per GPU that loads the
//     library and is held until the process exits;
//   * the batch is processed in slices of as many images as fit in it; a shape
//     whose single image needs more is rejected with CONV_ERR_WORKSPACE before
//     anything is launched;
//   * every call on a device shares the one array and it keeps the last
//     call's contents; nothing in it needs clearing, since every byte a call
//     reads was written earlier in the same call;
//   * calls that can overlap on the GPU (different streams without ordering
//     between them) race on the array: order them on one stream or with events;
//   * the first call on a device looks up the array's device address
//     (cudaGetSymbolAddress) with that device current; make that first call
//     before any stream capture.
#include <mutex>

#include "internal.h"

static constexpr size_t kNoAllocScratchBytes = 24u << 20;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

namespace {
constexpr int kMaxDev = 64;
std::mutex g_setup_mu;
void* g_scratch_addr[kMaxDev];

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Device address of the scratch array on the current device (set-up once per
// device).  Host code must not use the symbol itself as a pointer.
conv_status_t scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return gb_fail(CONV_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
  if (dev < 0 || dev >= kMaxDev) return gb_fail(CONV_ERR_CUDA, "device index %d too large", dev);
  std::lock_guard<std::mutex> lk(g_setup_mu);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess || !p)
      return gb_fail(CONV_ERR_CUDA, "cudaGetSymbolAddress(scratch): %s", cudaGetErrorString(e));
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return CONV_OK;
}
}  // namespace

extern "C" conv_status_t conv_fwd_noalloc(conv_desc_t d, const void* x, const void* wpack,
                                          const void* bias, const void* residual, void* y,
                                          conv_algo_t algo, void* stream) {
  if (!d || !x || !wpack || !y) return gb_fail(CONV_ERR_BAD_PARAM, "NULL tensor argument");
  if (algo != CONV_ALGO_WINO_F2 && algo != CONV_ALGO_WINO_F6)
    return gb_fail(CONV_ERR_UNSUPPORTED, "conv_fwd_noalloc runs the Winograd algorithms only");
  if (d->dtype != CONV_BF16 || d->layout != CONV_NHWC || d->R != 3 || d->S != 3 ||
      d->stride != 1 || d->dil != 1 || d->groups != 1 || d->C % 8 || d->K % 8)
    return gb_fail(CONV_ERR_UNSUPPORTED,
                   "Winograd needs bf16 NHWC, 3x3, stride 1, dilation 1, groups 1, C and K "
                   "multiples of 8");
  if (d->has_residual != (residual != nullptr))
    return gb_fail(CONV_ERR_BAD_PARAM, "residual must be given exactly when the descriptor has one");
  if (!aligned16(x) || !aligned16(y) || !aligned16(wpack) || (residual && !aligned16(residual)) ||
      (bias && (reinterpret_cast<uintptr_t>(bias) & 3u)))
    return gb_fail(CONV_ERR_ALIGNMENT, "tensors must be 16-byte aligned (bias 4-byte)");
  const int m = algo == CONV_ALGO_WINO_F2 ? 2 : 6;

  // images per slice that fit in the fixed scratch
  gbconv_desc_s sub = *d;
  sub.N = 1;
  const size_t one = winograd_workspace_bytes(sub, m);
  if (one > kNoAllocScratchBytes)
    return gb_fail(CONV_ERR_WORKSPACE,
                   "one image needs %zu bytes of Winograd scratch; the static scratch holds %zu",
                   one, kNoAllocScratchBytes);
  int nb = 1;
  while (nb < d->N) {
    sub.N = nb + 1;
    if (winograd_workspace_bytes(sub, m) > kNoAllocScratchBytes) break;
    ++nb;
  }

  void* scratch = nullptr;
  conv_status_t st = scratch_address(&scratch);
  if (st != CONV_OK) return st;
  int* err = gb_device_error_word();
  const unsigned long long wait_ns = gb_wait_limit_ns();
  const size_t x_img = (size_t)d->H * d->W * d->C * 2;
  const size_t y_img = (size_t)d->OH * d->OW * d->K * 2;
  for (int n0 = 0; n0 < d->N; n0 += nb) {
    sub.N = d->N - n0 < nb ? d->N - n0 : nb;
    const char* xs = static_cast<const char*>(x) + n0 * x_img;
    char* ys = static_cast<char*>(y) + n0 * y_img;
    const char* rs = residual ? static_cast<const char*>(residual) + n0 * y_img : nullptr;
    cudaError_t e = launch_winograd(sub, m, xs, wpack, static_cast<const float*>(bias), rs, ys,
                                    scratch, err, wait_ns, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess)
      return gb_fail(CONV_ERR_CUDA, "conv_fwd_noalloc: %s", cudaGetErrorString(e));
  }
  return CONV_OK;
}
