// Launchers of algorithms whose kernels are not built into this version of
// the library.  The algorithm table marks them as not implemented, so these
// are never reached through the public API.
#include "internal.h"

cudaError_t launch_dwconv3x3(const gbconv_desc_s&, const void*, const void*, const float*,
                             const void*, void*, cudaStream_t) {
  return cudaErrorNotSupported;
}
cudaError_t launch_igemm_int8(const gbconv_desc_s&, const void*, const void*, const int32_t*,
                              void*, cudaStream_t) {
  return cudaErrorNotSupported;
}
cudaError_t launch_pack_int8_weights(const gbconv_desc_s&, const void*, void*, cudaStream_t) {
  return cudaErrorNotSupported;
}
size_t winograd_packed_bytes(const gbconv_desc_s&, int) { return 0; }
size_t winograd_workspace_bytes(const gbconv_desc_s&, int) { return 0; }
cudaError_t launch_winograd_filter_transform(const gbconv_desc_s&, int, const void*, void*,
                                             cudaStream_t) {
  return cudaErrorNotSupported;
}
cudaError_t launch_winograd(const gbconv_desc_s&, int, const void*, const void*, const float*,
                            const void*, void*, void*, int*, unsigned long long, cudaStream_t) {
  return cudaErrorNotSupported;
}
