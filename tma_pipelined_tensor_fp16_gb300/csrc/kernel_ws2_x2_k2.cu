// kernel_ws2_x2_k2.cu -- the CTA-pair GEMM (kernel_ws2.cuh) with two pairs per cluster
// sharing A, on the dynamic schedule (cluster launch control), with
// stages of K = 128 (two 64-wide swizzle groups).
#include "kernel_ws2.cuh"

namespace tg {

template cudaError_t launch_pair_width<true, 2, 2>(const LaunchSpec&, cudaStream_t);

}  // namespace tg
