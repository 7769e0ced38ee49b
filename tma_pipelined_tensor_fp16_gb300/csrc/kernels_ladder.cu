// kernels_ladder.cu -- the lock-step rungs of the ablation ladder ("GEMM II --
// pipelining with TMA", Steps 3-6).  All four keep every thread of the CTA in
// step: one thread issues the copies and the MMAs, everyone waits on the same
// barriers.  They differ only in WHEN and BY WHOM the tiles move:
//
//   k_sync_tiled   Step 3 baseline: all threads copy GMEM -> SMEM with plain
//                  loads/stores (writing the 128-byte-swizzled layout
//                  themselves), thread barrier, one thread issues the MMA,
//                  everyone waits for it, repeat.  Epilogue TMEM -> reg -> GMEM.
//   k_tma_serial   Step 4: one thread fires two TMA tile loads and announces
//                  the byte budget with arrive.expect_tx; all wait on that
//                  mbarrier; MMA; wait; repeat.  TMA-store epilogue.
//   k_pipelined    Step 5: a PIPE_DEPTH ring with one TMA barrier per stage and
//                  one MMA barrier; prologue prefetch of the first min(D, K
//                  tiles) stages, steady-state wait / MMA / wait / refill, and
//                  the drain given by the "next k < K tiles" guard.
//   k_pipelined<PERSIST>
//                  Step 6: the same K loop inside a persistent CTA (grid = SM
//                  count) that walks the grouped raster, keeps its TMEM
//                  allocation across tiles and uses the TMA-store epilogue.
//
// Phase bookkeeping.  Within one tile the pages' rule holds (the MMA barrier
// flips every iteration, a stage's barrier flips once per trip around the
// ring).  Across tiles the pages reset both phases to 0; that is only right
// when every barrier completed an even number of phases in the previous tile,
// which fails e.g. for K tiles = 79 (the MMA barrier) or PIPE_DEPTH = 3 with
// 128 K tiles.  These kernels therefore carry the parities across tiles: one
// parity bit per stage (the tilus tutorial's per-stage phase) and one for the
// MMA barrier, while the stage index restarts at 0 for each tile.
#include "device_common.cuh"
#include "launch.h"

namespace tg {

namespace {

struct CtaSmem {
    uint8_t* gen;   // generic pointer to the 1024-aligned base
    uint32_t base;  // shared-window address of the same byte
};

__device__ __forceinline__ CtaSmem cta_smem()
{
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = align1024(raw);
    return CtaSmem{smem_raw + (base - raw), base};
}

__device__ __forceinline__ uint32_t bar_addr(uint32_t bars, int slot)
{
    return bars + static_cast<uint32_t>(slot) * 8u;
}

// Four MMAs (K = 16 each) cover one 64-wide K block of the stage's tiles.
template <int BN>
__device__ __forceinline__ void issue_kblock_mmas(uint32_t d_tmem, uint32_t a_tile,
                                                  uint32_t b_tile, bool first_kblock)
{
    constexpr uint32_t idesc = idesc_f16_f32(BLK_M, BN);
    const uint64_t adesc = sw128_kmajor_desc(a_tile);
    const uint64_t bdesc = sw128_kmajor_desc(b_tile);
#pragma unroll
    for (int kk = 0; kk < BLK_K / MMA_K; ++kk) {
        // +32 bytes per K=16 step inside the 128-byte swizzle row (encoded >> 4)
        mma_f16_ss(d_tmem, adesc + static_cast<uint64_t>(kk * 2), bdesc + static_cast<uint64_t>(kk * 2),
                   idesc, (first_kblock && kk == 0) ? 0u : 1u);
    }
}

// Teardown drain by the issuing thread: every tcgen05 op it issued has
// completed once this returns (or the bound ran out).
__device__ __forceinline__ void drain_mmas(const Watchdog& wd, uint32_t drain_bar)
{
    mma_commit(drain_bar);
    wd.drain(drain_bar, 0);
}

}  // namespace

// ------------------------------------------------------------- Step 3 baseline

template <int BN, bool F16OUT>
__global__ void __launch_bounds__(128) k_sync_tiled(const __grid_constant__ CUtensorMap tmC,
                                                    const Params p)
{
    const CtaSmem sm = cta_smem();
    const SmemLayout L = smem_layout(1, BN, 0);
    const uint32_t sA = sm.base + L.a;
    const uint32_t sB = sm.base + L.b;
    const uint32_t bars = sm.base + L.bars;
    const uint32_t mma_bar = bar_addr(bars, BAR_MMA);
    const uint32_t drain_bar = bar_addr(bars, BAR_DRAIN);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm.gen + L.bars + TMEM_SLOT_OFFSET);
    const int tid = static_cast<int>(threadIdx.x);
    const int warp = tid >> 5;
    const uint32_t lane = lane_id();
    Watchdog wd = make_watchdog(p);

    int mt, nt;
    raster_tile(static_cast<int>(blockIdx.x), p.tiles_m, p.tiles_n, p.group_m, mt, nt);
    const int m0 = mt * BLK_M, n0 = nt * BN;

    if (warp == 0) {
        tmem_alloc(smem_u32(tmem_slot), BN);
        tmem_relinquish_alloc_permit();
    }
    if (tid == 0) {
        mbar_init(mma_bar, 1);
        mbar_init(drain_bar, 1);
        fence_mbar_init();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = *tmem_slot;

    const __half* A = static_cast<const __half*>(p.A);
    const __half* B = static_cast<const __half*>(p.B);
    uint32_t mma_phase = 0;
    for (int kb = 0; kb < p.k_blocks; ++kb) {
        const int k0 = kb * BLK_K;
        // All threads copy: 16-byte chunks, zero outside the matrix (K is a
        // multiple of 8, so a chunk is wholly inside or wholly outside).
#pragma unroll
        for (int i = 0; i < (BLK_M * 8) / 128; ++i) {
            const int idx = tid + i * 128;
            const int r = idx >> 3, c = idx & 7;
            const int gm = m0 + r, gk = k0 + c * 8;
            uint4 v = make_uint4(0, 0, 0, 0);
            if (gm < p.M && gk < p.K)
                v = __ldg(reinterpret_cast<const uint4*>(A + static_cast<size_t>(gm) * p.K + gk));
            st_shared_v4(sA + sw128_offset(r, c * 16), v.x, v.y, v.z, v.w);
        }
#pragma unroll
        for (int i = 0; i < (BN * 8) / 128; ++i) {
            const int idx = tid + i * 128;
            const int r = idx >> 3, c = idx & 7;
            const int gn = n0 + r, gk = k0 + c * 8;
            uint4 v = make_uint4(0, 0, 0, 0);
            if (gn < p.N && gk < p.K)
                v = __ldg(reinterpret_cast<const uint4*>(B + static_cast<size_t>(gn) * p.K + gk));
            st_shared_v4(sB + sw128_offset(r, c * 16), v.x, v.y, v.z, v.w);
        }
        // the tensor core reads shared memory through the async proxy
        fence_proxy_async_smem();
        __syncthreads();
        if (tid == 0 && !wd.aborted) {
            tc_fence_after_sync();
            issue_kblock_mmas<BN>(tmem, sA, sB, kb == 0);
            mma_commit(mma_bar);
        }
        wd.wait(mma_bar, mma_phase, WAIT_MMA, static_cast<int>(blockIdx.x), kb);
        mma_phase ^= 1u;
    }

    tc_fence_after_sync();
    epilogue_direct_store<BN, F16OUT>(tmem, warp, lane, p.C, p.M, p.N, m0, n0, !wd.aborted);

    if (tid == 0) drain_mmas(wd, drain_bar);
    tc_fence_before_sync();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after_sync();
        tmem_dealloc(tmem, BN);
    }
}

// ---------------------------------------------------------------- Step 4

template <int BN, bool F16OUT>
__global__ void __launch_bounds__(128) k_tma_serial(const __grid_constant__ CUtensorMap tmA,
                                                    const __grid_constant__ CUtensorMap tmB,
                                                    const __grid_constant__ CUtensorMap tmC,
                                                    const Params p)
{
    const CtaSmem sm = cta_smem();
    const SmemLayout L = smem_layout(1, BN, NUM_STAGING);
    const uint32_t sA = sm.base + L.a;
    const uint32_t sB = sm.base + L.b;
    const uint32_t staging = sm.base + L.staging;
    const uint32_t bars = sm.base + L.bars;
    const uint32_t tma_bar = bar_addr(bars, BAR_FULL);
    const uint32_t mma_bar = bar_addr(bars, BAR_MMA);
    const uint32_t drain_bar = bar_addr(bars, BAR_DRAIN);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm.gen + L.bars + TMEM_SLOT_OFFSET);
    const int tid = static_cast<int>(threadIdx.x);
    const int warp = tid >> 5;
    const uint32_t lane = lane_id();
    Watchdog wd = make_watchdog(p);
    const uint32_t tx = stage_tx_bytes(BN);

    int mt, nt;
    raster_tile(static_cast<int>(blockIdx.x), p.tiles_m, p.tiles_n, p.group_m, mt, nt);
    const int m0 = mt * BLK_M, n0 = nt * BN;

    if (warp == 0) {
        tmem_alloc(smem_u32(tmem_slot), BN);
        tmem_relinquish_alloc_permit();
    }
    if (tid == 0) {
        prefetch_tensormap(&tmA);
        prefetch_tensormap(&tmB);
        prefetch_tensormap(&tmC);
        mbar_init(tma_bar, 1);
        mbar_init(mma_bar, 1);
        mbar_init(drain_bar, 1);
        fence_mbar_init();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = *tmem_slot;

    uint32_t tma_phase = 0, mma_phase = 0;
    bool load_pending = false;      // (issuing thread) a load not yet waited on
    uint32_t pending_parity = 0;    // ... and the parity of its phase
    for (int kb = 0; kb < p.k_blocks; ++kb) {
        if (tid == 0 && !wd.aborted) {
            // exactly one thread announces the byte budget and fires both copies
            mbar_arrive_expect_tx(tma_bar, tx);
            tma_load_2d(sA, &tmA, tma_bar, kb * BLK_K, m0);
            tma_load_2d(sB, &tmB, tma_bar, kb * BLK_K, n0);
            load_pending = true;
            pending_parity = tma_phase;
        }
        if (wd.wait(tma_bar, tma_phase, WAIT_FULL, static_cast<int>(blockIdx.x), kb))
            load_pending = false;
        tma_phase ^= 1u;
        if (tid == 0 && !wd.aborted) {
            tc_fence_after_sync();
            issue_kblock_mmas<BN>(tmem, sA, sB, kb == 0);
            mma_commit(mma_bar);
        }
        wd.wait(mma_bar, mma_phase, WAIT_MMA, static_cast<int>(blockIdx.x), kb);
        mma_phase ^= 1u;
    }

    tc_fence_after_sync();
    uint32_t sub_count = 0;
    epilogue_tma_store<BN, F16OUT>(tmem, warp, lane, staging, &tmC, m0, n0, p.M, p.N,
                                   sub_count, !wd.aborted);

    if (tid == 0) {
        if (load_pending) wd.drain(tma_bar, pending_parity);
        drain_mmas(wd, drain_bar);
    }
    // each warp's stores have read their staging before the CTA exits
    if (lane == 0) bulk_wait_group<0>();
    tc_fence_before_sync();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after_sync();
        tmem_dealloc(tmem, BN);
    }
}

// ---------------------------------------------------------- Steps 5 and 6

template <int BN, bool F16OUT, bool PERSIST>
__global__ void __launch_bounds__(128) k_pipelined(const __grid_constant__ CUtensorMap tmA,
                                                   const __grid_constant__ CUtensorMap tmB,
                                                   const __grid_constant__ CUtensorMap tmC,
                                                   const Params p)
{
    const int D = p.pipe_depth;
    const CtaSmem sm = cta_smem();
    const SmemLayout L = smem_layout(D, BN, NUM_STAGING);
    const uint32_t sA = sm.base + L.a;
    const uint32_t sB = sm.base + L.b;
    const uint32_t staging = sm.base + L.staging;
    const uint32_t bars = sm.base + L.bars;
    const uint32_t mma_bar = bar_addr(bars, BAR_MMA);
    const uint32_t drain_bar = bar_addr(bars, BAR_DRAIN);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm.gen + L.bars + TMEM_SLOT_OFFSET);
    const int tid = static_cast<int>(threadIdx.x);
    const int warp = tid >> 5;
    const uint32_t lane = lane_id();
    Watchdog wd = make_watchdog(p);
    const uint32_t tx = stage_tx_bytes(BN);

    if (warp == 0) {
        // allocated once, kept for every tile this CTA processes
        tmem_alloc(smem_u32(tmem_slot), BN);
        tmem_relinquish_alloc_permit();
    }
    if (tid == 0) {
        prefetch_tensormap(&tmA);
        prefetch_tensormap(&tmB);
        prefetch_tensormap(&tmC);
        for (int s = 0; s < D; ++s) mbar_init(bar_addr(bars, BAR_FULL + s), 1);
        mbar_init(mma_bar, 1);
        mbar_init(drain_bar, 1);
        fence_mbar_init();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = *tmem_slot;

    uint32_t tma_parity = 0;    // bit s: parity of the phase stage s waits for next
    uint32_t mma_phase = 0;
    uint32_t pending = 0;       // (issuing thread) stages with a load not yet waited on
    uint32_t pending_parity = 0;  // ... and the parity of that load's phase, per stage
    uint32_t sub_count = 0;
    const int tile_step = PERSIST ? static_cast<int>(gridDim.x) : p.num_tiles;
    const int KB = p.k_blocks;

    for (int t = static_cast<int>(blockIdx.x); t < p.num_tiles; t += tile_step) {
        int mt, nt;
        raster_tile(t, p.tiles_m, p.tiles_n, p.group_m, mt, nt);
        const int m0 = mt * BLK_M, n0 = nt * BN;

        // prologue: prime the ring, never past the last K tile
        const int n_pro = KB < D ? KB : D;
        if (tid == 0 && !wd.aborted) {
            for (int s = 0; s < n_pro; ++s) {
                const uint32_t fb = bar_addr(bars, BAR_FULL + s);
                mbar_arrive_expect_tx(fb, tx);
                tma_load_2d(sA + s * A_TILE_BYTES, &tmA, fb, s * BLK_K, m0);
                tma_load_2d(sB + s * b_tile_bytes(BN), &tmB, fb, s * BLK_K, n0);
                pending |= 1u << s;
                pending_parity = (pending_parity & ~(1u << s)) | (tma_parity & (1u << s));
            }
        }
        // steady state; the refill guard drains the ring at the end
        for (int kb = 0; kb < KB; ++kb) {
            const int s = kb % D;
            const uint32_t fb = bar_addr(bars, BAR_FULL + s);
            if (wd.wait(fb, (tma_parity >> s) & 1u, WAIT_FULL, t, kb)) pending &= ~(1u << s);
            tma_parity ^= 1u << s;
            if (tid == 0 && !wd.aborted) {
                tc_fence_after_sync();
                issue_kblock_mmas<BN>(tmem, sA + s * A_TILE_BYTES, sB + s * b_tile_bytes(BN),
                                      kb == 0);
                mma_commit(mma_bar);
            }
            wd.wait(mma_bar, mma_phase, WAIT_MMA, t, kb);
            mma_phase ^= 1u;
            const int next_k = kb + D;
            if (next_k < KB && tid == 0 && !wd.aborted) {
                mbar_arrive_expect_tx(fb, tx);
                tma_load_2d(sA + s * A_TILE_BYTES, &tmA, fb, next_k * BLK_K, m0);
                tma_load_2d(sB + s * b_tile_bytes(BN), &tmB, fb, next_k * BLK_K, n0);
                pending |= 1u << s;
                pending_parity = (pending_parity & ~(1u << s)) | (tma_parity & (1u << s));
            }
        }

        tc_fence_after_sync();
        epilogue_tma_store<BN, F16OUT>(tmem, warp, lane, staging, &tmC, m0, n0, p.M, p.N,
                                       sub_count, !wd.aborted);
        // every TMEM read is done before the next tile's first MMA overwrites it
        tc_fence_before_sync();
        __syncthreads();
    }

    if (tid == 0) {
        for (int s = 0; s < D; ++s)
            if (pending & (1u << s))
                wd.drain(bar_addr(bars, BAR_FULL + s), (pending_parity >> s) & 1u);
        drain_mmas(wd, drain_bar);
    }
    // each warp's stores have read their staging before the CTA exits
    if (lane == 0) bulk_wait_group<0>();
    tc_fence_before_sync();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after_sync();
        tmem_dealloc(tmem, BN);
    }
}

// ------------------------------------------------------------------ launch

namespace {

template <typename KernelT, typename... Args>
cudaError_t launch_one(KernelT kernel, const LaunchSpec& s, cudaStream_t stream, Args... args)
{
    cudaError_t e = ensure_smem_limit(kernel, s.smem_bytes);
    if (e != cudaSuccess) return e;
    kernel<<<s.grid, s.threads, s.smem_bytes, stream>>>(args...);
    return cudaGetLastError();
}

template <int BN, bool F16OUT>
cudaError_t launch_bn(const LaunchSpec& s, cudaStream_t stream)
{
    switch (s.variant) {
    case VAR_SYNC_TILED:
        return launch_one(k_sync_tiled<BN, F16OUT>, s, stream, *s.tmC, s.p);
    case VAR_TMA_SERIAL:
        return launch_one(k_tma_serial<BN, F16OUT>, s, stream, *s.tmA, *s.tmB, *s.tmC, s.p);
    case VAR_PIPELINED:
        return launch_one(k_pipelined<BN, F16OUT, false>, s, stream, *s.tmA, *s.tmB, *s.tmC, s.p);
    case VAR_PERSISTENT_LOCKSTEP:
        return launch_one(k_pipelined<BN, F16OUT, true>, s, stream, *s.tmA, *s.tmB, *s.tmC, s.p);
    default:
        return cudaErrorInvalidValue;
    }
}

}  // namespace

cudaError_t launch_ladder(const LaunchSpec& s, cudaStream_t stream)
{
    switch (s.block_n) {
    case 64:
        return s.f16out ? launch_bn<64, true>(s, stream) : launch_bn<64, false>(s, stream);
    case 128:
        return s.f16out ? launch_bn<128, true>(s, stream) : launch_bn<128, false>(s, stream);
    case 256:
        return s.f16out ? launch_bn<256, true>(s, stream) : launch_bn<256, false>(s, stream);
    default:
        return cudaErrorInvalidValue;
    }
}

}  // namespace tg
