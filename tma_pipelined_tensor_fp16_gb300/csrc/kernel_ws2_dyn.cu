// kernel_ws2_dyn.cu -- the CTA-pair GEMM (kernel_ws2.cuh) with the dynamic
// schedule: a grid of one cluster per tile, in which running clusters cancel
// clusters that have not started and take over their tiles (cluster launch
// control).  A translation unit of its own so that both schedules compile in
// parallel.
#include "kernel_ws2.cuh"

namespace tg {

cudaError_t launch_pair_dynamic(const LaunchSpec& s, cudaStream_t stream)
{
    if (s.variant != VAR_DYNAMIC_2CTA || (s.grid & 1)) return cudaErrorInvalidValue;
    return launch_pair_width<true>(s, stream);
}

}  // namespace tg
