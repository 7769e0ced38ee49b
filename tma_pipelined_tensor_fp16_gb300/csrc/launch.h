// launch.h -- host-side entry points of the kernel translation units.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include "gemm_common.h"

namespace tg {

// Variant numbers (same values as the public gemm_variant enum).
enum : int {
    VAR_AUTO = 0,
    VAR_SYNC_TILED = 1,
    VAR_TMA_SERIAL = 2,
    VAR_PIPELINED = 3,
    VAR_WS_PIPELINED = 4,
    VAR_PERSISTENT = 5,
    VAR_PERSISTENT_LOCKSTEP = 6,
    VAR_PERSISTENT_2CTA = 7
};

struct LaunchSpec {
    int variant;
    int block_n;
    bool f16out;
    int grid;
    int threads;
    unsigned smem_bytes;
    const CUtensorMap* tmA;
    const CUtensorMap* tmB;
    const CUtensorMap* tmC;
    Params p;
};

// Lock-step variants: VAR_SYNC_TILED, VAR_TMA_SERIAL, VAR_PIPELINED,
// VAR_PERSISTENT_LOCKSTEP.
cudaError_t launch_ladder(const LaunchSpec& s, cudaStream_t stream);

// Warp-specialised variants: VAR_WS_PIPELINED, VAR_PERSISTENT.
cudaError_t launch_ws(const LaunchSpec& s, cudaStream_t stream);

// Warp-specialised persistent GEMM on CTA pairs: VAR_PERSISTENT_2CTA.
cudaError_t launch_pair(const LaunchSpec& s, cudaStream_t stream);

}  // namespace tg
