// kernel_ws2_dyn_k2.cu -- the CTA-pair GEMM (kernel_ws2.cuh) with the dynamic
// schedule (cluster launch control) and stages of K = 128 (two 64-wide
// swizzle groups).
#include "kernel_ws2.cuh"

namespace tg {

template cudaError_t launch_pair_width<true, 2>(const LaunchSpec&, cudaStream_t);

}  // namespace tg
