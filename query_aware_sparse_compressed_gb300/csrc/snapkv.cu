// snapkv_compress (placeholder until the tensor-core kernels land).
#include "common.cuh"
#include "internal.h"

namespace qasc {

SnapLayout snap_layout(const qasc_shape& s, const qasc_snap_params& p) {
  SnapLayout L;
  L.c_out = p.c < s.n ? p.c : s.n;
  L.total = 256;
  return L;
}

cudaError_t configure_snapkv_kernels(const DeviceInfo&) { return cudaSuccess; }

int launch_snapkv(const qasc_shape&, const qasc_snap_params&, const SnapLayout&, const uint16_t*, const uint16_t*,
                  const uint16_t*, int32_t*, uint16_t*, uint16_t*, uint8_t*, const DeviceInfo&, cudaStream_t) {
  return -1;
}

}  // namespace qasc
