// kernel_ws2_dyn.cu -- the CTA-pair GEMM (kernel_ws2.cuh) with the dynamic
// schedule (a grid of one cluster per tile, in which running clusters cancel
// clusters that have not started and take over their tiles: cluster launch
// control) and stages of one 64-wide K block.
#include "kernel_ws2.cuh"

namespace tg {

template cudaError_t launch_pair_width<true, 1>(const LaunchSpec&, cudaStream_t);

}  // namespace tg
