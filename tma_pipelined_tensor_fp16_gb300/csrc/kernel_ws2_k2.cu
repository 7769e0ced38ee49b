// kernel_ws2_k2.cu -- the CTA-pair GEMM (kernel_ws2.cuh) with the static
// persistent schedule and stages of K = 128 (two 64-wide swizzle groups).
#include "kernel_ws2.cuh"

namespace tg {

template cudaError_t launch_pair_width<false, 2>(const LaunchSpec&, cudaStream_t);

}  // namespace tg
