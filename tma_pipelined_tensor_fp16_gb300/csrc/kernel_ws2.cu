// kernel_ws2.cu -- the CTA-pair GEMM (kernel_ws2.cuh) with the static
// persistent schedule: one cluster per TPC walking its WorkIter sequence.
#include "kernel_ws2.cuh"

namespace tg {

cudaError_t launch_pair(const LaunchSpec& s, cudaStream_t stream)
{
    if (s.grid & 1) return cudaErrorInvalidValue;
    if (s.variant == VAR_DYNAMIC_2CTA) return launch_pair_dynamic(s, stream);
    if (s.variant != VAR_PERSISTENT_2CTA) return cudaErrorInvalidValue;
    return launch_pair_width<false>(s, stream);
}

}  // namespace tg
