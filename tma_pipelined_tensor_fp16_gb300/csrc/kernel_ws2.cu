// kernel_ws2.cu -- the CTA-pair GEMM (kernel_ws2.cuh): the launch dispatch
// over tile schedule and stage K extent, and the instantiation for the static
// persistent schedule with stages of one 64-wide K block.
#include "kernel_ws2.cuh"

namespace tg {

template cudaError_t launch_pair_width<false, 1>(const LaunchSpec&, cudaStream_t);

cudaError_t launch_pair(const LaunchSpec& s, cudaStream_t stream)
{
    if ((s.grid & 1) || (s.p.ksub != 1 && s.p.ksub != 2)) return cudaErrorInvalidValue;
    const bool k2 = s.p.ksub == 2;
    if (s.variant == VAR_DYNAMIC_2CTA)
        return k2 ? launch_pair_width<true, 2>(s, stream) : launch_pair_width<true, 1>(s, stream);
    if (s.variant == VAR_PERSISTENT_2CTA)
        return k2 ? launch_pair_width<false, 2>(s, stream) : launch_pair_width<false, 1>(s, stream);
    return cudaErrorInvalidValue;
}

}  // namespace tg
