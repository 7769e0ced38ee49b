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
    VAR_PERSISTENT_2CTA = 7,
    VAR_DYNAMIC_2CTA = 8
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
    const CUtensorMap* tmB2;  // CTA-pair kernel: B with half-height boxes (narrow
                              // tail tiles); nullptr = the same as tmB
    Params p;
};

// Lock-step variants: VAR_SYNC_TILED, VAR_TMA_SERIAL, VAR_PIPELINED,
// VAR_PERSISTENT_LOCKSTEP.
cudaError_t launch_ladder(const LaunchSpec& s, cudaStream_t stream);

// Warp-specialised variants: VAR_WS_PIPELINED, VAR_PERSISTENT.
cudaError_t launch_ws(const LaunchSpec& s, cudaStream_t stream);

// Warp-specialised GEMM on CTA pairs: VAR_PERSISTENT_2CTA (static schedule)
// and VAR_DYNAMIC_2CTA (cluster launch control), with stages of p.ksub K
// blocks of 64.
cudaError_t launch_pair(const LaunchSpec& s, cudaStream_t stream);

// Raise `kernel`'s dynamic shared-memory limit to at least `bytes`, calling
// the runtime only when a larger limit than any set before for that kernel is
// needed (the limit belongs to the kernel, for the whole process).
bool smem_limit_known(const void* kernel, unsigned bytes);
void smem_limit_record(const void* kernel, unsigned bytes);

template <typename KernelT>
cudaError_t ensure_smem_limit(KernelT kernel, unsigned bytes)
{
    const void* key = reinterpret_cast<const void*>(kernel);
    if (smem_limit_known(key, bytes)) return cudaSuccess;
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(bytes));
    if (e == cudaSuccess) smem_limit_record(key, bytes);
    return e;
}

// Launch a warp-specialised GEMM kernel as a programmatic dependent of the
// work before it on `stream`: its CTAs may be scheduled while that work drains
// and run their set-up (barriers, TMEM allocation) meanwhile.  The kernel
// executes griddep_wait() before its first global-memory access, so it still
// reads A and B and writes C only after everything earlier on the stream has
// completed; it calls griddep_launch_dependents() after its set-up.
template <typename KernelT, typename... Maps>
cudaError_t launch_programmatic(KernelT kernel, const LaunchSpec& s, int threads,
                                cudaStream_t stream, const Maps&... extra_maps)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(s.grid));
    cfg.blockDim = dim3(static_cast<unsigned>(threads));
    cfg.dynamicSmemBytes = s.smem_bytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, *s.tmA, *s.tmB, *s.tmC, extra_maps..., s.p);
}

}  // namespace tg
