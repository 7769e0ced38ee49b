// kernel_ws2_x2.cu -- the CTA-pair GEMM (kernel_ws2.cuh) with two pairs per cluster
// sharing A, on the dynamic schedule (cluster launch control), with
// stages of one 64-wide K block.
#include "kernel_ws2.cuh"

namespace tg {

template cudaError_t launch_pair_width<true, 1, 2>(const LaunchSpec&, cudaStream_t);

}  // namespace tg
