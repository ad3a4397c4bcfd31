// Large-M preshuffled-weight GEMM (placeholder until the tcgen05 kernel lands).
#include "fg_internal.cuh"

namespace fg {

bool large_supported(int) { return false; }

cudaError_t launch_large(int, const CUtensorMap&, const LargeParams&, int, cudaStream_t) {
  return cudaErrorNotSupported;
}

}  // namespace fg
