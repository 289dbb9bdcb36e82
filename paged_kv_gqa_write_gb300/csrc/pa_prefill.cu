// pa_prefill.cu -- causal chunked-prefill attention (tcgen05 kernel: in progress).
#include "pa_launch.cuh"

namespace pa {

cudaError_t launch_prefill(const CUtensorMap&, const CUtensorMap&, const CUtensorMap&,
                           const PrefillParams&, int, cudaStream_t) {
  return cudaErrorNotSupported;
}

}  // namespace pa
