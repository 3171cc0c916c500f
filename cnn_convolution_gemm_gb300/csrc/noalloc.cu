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
//   * the scratch array is kNoAllocScratchBytes (24 MiB) per GPU; it comes into
//     being when this file's module is loaded on the device (under lazy module
//     loading, the CUDA default, at the first call there) and is held until
//     the process exits;
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
  // the same applicability rules as conv_fwd (shape, dtype, layout, input shuffle)
  conv_status_t st = gb_check_algo(*d, algo);
  if (st != CONV_OK) return st;
  if (d->has_residual != (residual != nullptr))
    return gb_fail(CONV_ERR_BAD_PARAM, "residual must be given exactly when the descriptor has one");
  if (!aligned16(x) || !aligned16(y) || !aligned16(wpack) || (residual && !aligned16(residual)) ||
      (bias && (reinterpret_cast<uintptr_t>(bias) & 3u)))
    return gb_fail(CONV_ERR_ALIGNMENT, "tensors must be 16-byte aligned (bias 4-byte)");
  const int m = algo == CONV_ALGO_WINO_F2 ? 2 : 6;

  // Images per slice: the largest count whose scratch fits the fixed array.  The
  // scratch a batch needs never decreases as the batch grows (its chunk size
  // only grows with the batch), so the fitting counts form a prefix of [1, N]:
  // binary search.  Every slice, the last and shorter one included, then fits.
  gbconv_desc_s sub = *d;
  auto fits = [&](int nb) {
    sub.N = nb;
    return winograd_workspace_bytes(sub, m) <= kNoAllocScratchBytes;
  };
  if (!fits(1)) {
    sub.N = 1;
    return gb_fail(CONV_ERR_WORKSPACE,
                   "one image needs %zu bytes of Winograd scratch; the static scratch holds %zu",
                   winograd_workspace_bytes(sub, m), kNoAllocScratchBytes);
  }
  int lo = 1, hi = d->N;  // fits(lo) holds; find the largest such count
  while (lo < hi) {
    const int mid = lo + (hi - lo + 1) / 2;
    if (fits(mid))
      lo = mid;
    else
      hi = mid - 1;
  }
  const int nb = lo;

  void* scratch = nullptr;
  st = scratch_address(&scratch);
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
  return gb_ok();
}
