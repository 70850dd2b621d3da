// ibp_codec.cu -- placeholder launchers (replaced by the IBP kernels).
#include <cuda_runtime.h>
#include "internal.h"
namespace lbb {
cudaError_t ibp_launch_build_meta(const void*, unsigned long long, uint32_t, unsigned long long,
                                  double, int, void*, void*, cudaStream_t) {
  return cudaErrorNotSupported;
}
cudaError_t ibp_launch_compress(const void*, uint32_t, const void*, unsigned long long, void*,
                                unsigned long long, unsigned long long*, void*, cudaStream_t) {
  return cudaErrorNotSupported;
}
cudaError_t ibp_launch_decompress(const void*, uint32_t, const void*, unsigned long long, void*,
                                  unsigned long long, void*, cudaStream_t) {
  return cudaErrorNotSupported;
}
}  // namespace lbb
