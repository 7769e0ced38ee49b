// kernel_ws.cu -- the warp-specialised rungs of the ladder: the CTA's threads
// split into roles that talk only through mbarriers, so the copy engine, the
// tensor core and the epilogue run at the same time ("GEMM II -- pipelining
// with TMA", closing section: split the lock-step team into producer and
// consumer roles; tilus "Multi-Stage Software Pipelining", What's Next: a
// producer warp and consumers joined by a producer/consumer barrier pair; "B200
// Tma Pipeline Designer", Case 1: the consumer waits on tma2mma[stage], the
// producer waits on mma2tma[stage] before overwriting).
//
//   warp 0             TMA producer: the warp waits empty[s]; lane 0 issues
//                      arrive.expect_tx(full[s]) and two bulk tensor loads
//                      into stage s ("one elected thread" of the pages).
//   warp 1             MMA issuer: the warp waits full[s]; lane 0 issues four
//                      tcgen05.mma into the TMEM accumulator and
//                      tcgen05.commit -> empty[s]; after the last K block,
//                      commit -> tmem_full[acc].
//   warps 2..5         epilogue: wait tmem_full[acc], TMEM -> regs -> swizzled
//                      staging -> TMA store, arrive tmem_empty[acc].
//
// A pipeline stage spans p.ksub (1, 2 or 4) K blocks of 64, each in a
// sub-slot of its own (sub-slot stage * ksub + s): one barrier round trip per
// ksub x 4 MMAs, and each row of an operand tile is read as ksub adjacent
// 128-byte pieces ("05 Async Data Movement - TMA", Using 3D TMA to Move
// Multiple Swizzle Atoms, loaded here as ksub 2-D boxes).  A block of the last
// stage that lies past K arrives zero-filled and is not multiplied.
//
// PERSIST = false: one output tile per CTA, one accumulator (grid = tiles).
// PERSIST = true : grid = SM count; each CTA walks the grouped raster
// (t = blockIdx.x, + gridDim.x, ...), TMEM is allocated once for two
// accumulators so the epilogue of tile i overlaps the main loop of tile i+1,
// and the ring position {stage, phase} runs on continuously across tiles (the
// tilus tutorial's single per-role phase that flips on wrap-around), so no
// phase is ever reset.  A persistent CTA's work is a sequence of WorkUnits:
// whole tiles, then (when the tile count leaves a partial last wave) its
// share of the stream-K part, finished through the fix-up in
// device_common.cuh.
#include "device_common.cuh"
#include "launch.h"

namespace tg {

namespace {

struct CtaSmem {
    uint8_t* gen;
    uint32_t base;
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

}  // namespace

constexpr int WS_THREADS = 192;
constexpr int EPI_FIRST_WARP = 2;
constexpr uint32_t EPI_BAR_ID = 1;

template <int BN, bool F16OUT, bool PERSIST>
__global__ void __launch_bounds__(WS_THREADS, 1) k_ws(const __grid_constant__ CUtensorMap tmA,
                                                      const __grid_constant__ CUtensorMap tmB,
                                                      const __grid_constant__ CUtensorMap tmC,
                                                      const Params p)
{
    constexpr int ACC = PERSIST ? 2 : 1;
    constexpr uint32_t TMEM_COLS = ACC * BN;  // 64..512, a power of two
    const int D = p.pipe_depth;
    const int KS = p.ksub == 2 || p.ksub == 4 ? p.ksub : 1;  // K blocks of 64 per stage
    const CtaSmem sm = cta_smem();
    const int a_rows = p.a_rows == 64 ? 64 : BLK_M;
    const uint32_t a_slot = a_slot_bytes(a_rows);
    const SmemLayout L = smem_layout(D * KS, BN, NUM_STAGING, a_rows);
    const uint32_t sA = sm.base + L.a;
    const uint32_t sB = sm.base + L.b;
    const uint32_t staging = sm.base + L.staging;
    const uint32_t bars = sm.base + L.bars;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm.gen + L.bars + TMEM_SLOT_OFFSET);
    const int tid = static_cast<int>(threadIdx.x);
    const int warp = tid >> 5;
    const uint32_t lane = lane_id();
    Watchdog wd = make_watchdog(p);
    const int workers = PERSIST ? static_cast<int>(gridDim.x) : p.num_tiles;
    const int KB = (p.k_blocks + KS - 1) / KS;  // stages per tile
    WorkIter units0;
    units0.init(static_cast<int>(blockIdx.x), workers, PERSIST ? p.dp_tiles : p.num_tiles,
                PERSIST ? p.sk_tiles : 0, KB, p.sk_kb_per_worker);

    if (warp == 0 && lane == 0) {
        prefetch_tensormap(&tmA);
        prefetch_tensormap(&tmB);
        prefetch_tensormap(&tmC);
        for (int s = 0; s < D; ++s) {
            mbar_init(bar_addr(bars, BAR_FULL + s), 1);   // producer's expect_tx arrival
            mbar_init(bar_addr(bars, BAR_EMPTY + s), 1);  // MMA issuer's commit
        }
        for (int a = 0; a < ACC; ++a) {
            mbar_init(bar_addr(bars, BAR_TMEM_FULL + a), 1);     // MMA issuer's commit
            mbar_init(bar_addr(bars, BAR_TMEM_EMPTY + a), 128);  // every epilogue thread
        }
        mbar_init(bar_addr(bars, BAR_DRAIN), 1);
        mbar_init(bar_addr(bars, BAR_STALL), 1);
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_slot), TMEM_COLS);
        tmem_relinquish_alloc_permit();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    // global memory only after the work before this launch has completed
    griddep_wait();
    griddep_launch_dependents();
    const uint32_t tmem_base = *tmem_slot;
    if (tid == 0) {
        trace_header(p, TRACE_H_START, globaltimer_ns());
        trace_header(p, TRACE_H_SMID, sm_id());
    }

    // The producer and MMA roles run as whole warps: every lane walks the
    // loop and waits on each barrier, lane 0 issues the copies or the MMAs,
    // and the warp reconverges after every stage (a role run by lane 0 alone,
    // the other lanes parked at a warp barrier, measured up to 9% slower).
    if (warp == 0) {
        // ---------------------------------------------------- TMA producer
        // every box's full bytes, including those of a block past K
        const uint32_t tx = stage_tx_bytes(BN, a_rows) * static_cast<uint32_t>(KS);
        const uint64_t pol_a = (p.l2_policy == 2) ? policy_evict_first() : policy_evict_last();
        const uint64_t pol_b = (p.l2_policy == 1) ? policy_evict_first() : policy_evict_last();
        const bool tr = p.trace && lane == 0;
        if (p.debug_stall) wd.wait(bar_addr(bars, BAR_STALL), 0, WAIT_STALL, -1, -1);
        int stage = 0;
        uint32_t phase = 0;
        int issued = 0;
        int end_stage = 0;       // ring position just after the last issued load
        uint32_t end_phase = 0;
        WorkIter units = units0;
        WorkUnit u;
        int ui = 0;
        while (units.next(u)) {
            const int t = u.tile;
            if (tr)
                trace_unit(p, ui, TRACE_U_TILE,
                           (static_cast<unsigned long long>(t) << 32) |
                               static_cast<unsigned>(u.kb1 - u.kb0));
            unsigned long long empty_wait_ns = 0;
            int mt, nt;
            raster_tile(t, p.tiles_m, p.tiles_n, p.group_m, mt, nt);
            const int m0 = mt * BLK_M, n0 = nt * BN;
            for (int ki = 0; ki < u.kb1 - u.kb0; ++ki) {
                const int kb = kblock_at(ki, ui, u.kb0, u.kb1, p.k_snake);
                // a fresh barrier passes a wait on parity 1 at once: the first
                // trip around the ring does not wait
                const unsigned long long tw0 = tr ? globaltimer_ns() : 0ull;
                const bool ok =
                    wd.wait(bar_addr(bars, BAR_EMPTY + stage), phase ^ 1u, WAIT_EMPTY, t, kb);
                if (tr) empty_wait_ns += globaltimer_ns() - tw0;
                if (lane == 0 && ok) {
                    const uint32_t fb = bar_addr(bars, BAR_FULL + stage);
                    mbar_arrive_expect_tx(fb, tx);
                    for (int s = 0; s < KS; ++s) {
                        const int slot = stage * KS + s;
                        const int kx = (kb * KS + s) * BLK_K;
                        if (p.l2_policy == 0) {
                            tma_load_2d(sA + slot * a_slot, &tmA, fb, kx, m0);
                            tma_load_2d(sB + slot * b_tile_bytes(BN), &tmB, fb, kx, n0);
                        } else {
                            tma_load_2d_hint(sA + slot * a_slot, &tmA, fb, kx, m0, pol_a);
                            tma_load_2d_hint(sB + slot * b_tile_bytes(BN), &tmB, fb, kx, n0,
                                             pol_b);
                        }
                    }
                    ++issued;
                }
                if (tr && ki == 0) trace_unit(p, ui, TRACE_U_LOAD_FIRST, globaltimer_ns());
                if (tr && ki == u.kb1 - u.kb0 - 1)
                    trace_unit(p, ui, TRACE_U_LOAD_LAST, globaltimer_ns());
                __syncwarp();
                if (++stage == D) {
                    stage = 0;
                    phase ^= 1u;
                }
                if (!wd.aborted) {
                    end_stage = stage;
                    end_phase = phase;
                }
            }
            if (tr) trace_unit(p, ui, TRACE_U_EMPTY_WAIT, empty_wait_ns);
            ++ui;
        }
        // drain: the last min(D, issued) loads have landed before exit
        if (lane == 0 && wd.aborted) {
            int st = end_stage;
            uint32_t ph = end_phase;
            for (int i = 0; i < D && i < issued; ++i) {
                if (st == 0) {
                    st = D - 1;
                    ph ^= 1u;
                } else {
                    --st;
                }
                wd.drain(bar_addr(bars, BAR_FULL + st), ph);
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // --------------------------------------------------------- MMA issuer
        constexpr uint32_t idesc = idesc_f16_f32(BLK_M, BN);
        const bool tr = p.trace && lane == 0;
        int stage = 0;
        uint32_t phase = 0;
        int acc = 0;
        uint32_t acc_phase = 0;
        int mui = 0;
        WorkIter units = units0;
        WorkUnit u;
        while (units.next(u)) {
            const int t = u.tile;
            // the epilogue has drained this accumulator (fresh: passes)
            wd.wait(bar_addr(bars, BAR_TMEM_EMPTY + acc), acc_phase ^ 1u, WAIT_TMEM_EMPTY, t, -1);
            tc_fence_after_sync();
            if (tr) trace_unit(p, mui, TRACE_U_ACC_FREE, globaltimer_ns());
            unsigned long long full_wait_ns = 0;
            const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * BN);
            for (int ki = 0; ki < u.kb1 - u.kb0; ++ki) {
                const int kb = kblock_at(ki, mui, u.kb0, u.kb1, p.k_snake);
                const unsigned long long tw0 = tr ? globaltimer_ns() : 0ull;
                const bool ok = wd.wait(bar_addr(bars, BAR_FULL + stage), phase, WAIT_FULL, t, kb);
                if (tr) full_wait_ns += globaltimer_ns() - tw0;
                if (lane == 0 && ok) {
                    tc_fence_after_sync();
                    if (tr && ki == 0) trace_unit(p, mui, TRACE_U_MMA_FIRST, globaltimer_ns());
                    for (int s = 0; s < KS; ++s) {
                        // a block of the last stage may lie past K
                        if (s > 0 && kb * KS + s >= p.k_blocks) break;
                        const int slot = stage * KS + s;
                        const uint64_t adesc = sw128_kmajor_desc(sA + slot * a_slot);
                        const uint64_t bdesc = sw128_kmajor_desc(sB + slot * b_tile_bytes(BN));
#pragma unroll
                        for (int kk = 0; kk < BLK_K / MMA_K; ++kk)
                            mma_f16_ss(d_tmem, adesc + static_cast<uint64_t>(kk * 2),
                                       bdesc + static_cast<uint64_t>(kk * 2), idesc,
                                       (ki == 0 && s == 0 && kk == 0) ? 0u : 1u);
                    }
                    // frees the stage once these MMAs have read it
                    mma_commit(bar_addr(bars, BAR_EMPTY + stage));
                }
                __syncwarp();
                if (++stage == D) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
            if (lane == 0 && !wd.aborted) mma_commit(bar_addr(bars, BAR_TMEM_FULL + acc));
            if (tr) {
                trace_unit(p, mui, TRACE_U_MMA_LAST, globaltimer_ns());
                trace_unit(p, mui, TRACE_U_FULL_WAIT, full_wait_ns);
            }
            __syncwarp();
            ++mui;
            if (ACC == 2) {
                acc ^= 1;
                if (acc == 0) acc_phase ^= 1u;
            } else {
                acc_phase ^= 1u;
            }
        }
        // every MMA has completed before TMEM is released
        if (lane == 0) {
            mma_commit(bar_addr(bars, BAR_DRAIN));
            wd.drain(bar_addr(bars, BAR_DRAIN), 0);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------ epilogue
        const int q = warp & 3;  // TMEM lane quarter this warp may access
        const bool issuer = (tid == EPI_FIRST_WARP * 32);
        int acc = 0;
        uint32_t acc_phase = 0;
        uint32_t sub_count = 0;
        WorkIter units = units0;
        WorkUnit u;
        volatile uint32_t* ticket_smem =
            reinterpret_cast<volatile uint32_t*>(sm.gen + L.bars + TICKET_SLOT_OFFSET);
        int eui = 0;
        while (units.next(u)) {
            const int t = u.tile;
            int mt, nt;
            raster_tile(t, p.tiles_m, p.tiles_n, p.group_m, mt, nt);
            wd.wait(bar_addr(bars, BAR_TMEM_FULL + acc), acc_phase, WAIT_TMEM_FULL, t, -1);
            tc_fence_after_sync();
            if (issuer) trace_unit(p, eui, TRACE_U_EPI_START, globaltimer_ns());
            const uint32_t tmem_acc = tmem_base + static_cast<uint32_t>(acc * BN);
            const uint32_t empty_bar = bar_addr(bars, BAR_TMEM_EMPTY + acc);
            if (u.ncontrib == 1) {
                epilogue_tma_store<BN, F16OUT>(tmem_acc, q, lane, staging, &tmC, mt * BLK_M,
                                               nt * BN, p.M, p.N, sub_count, !wd.aborted);
                tc_fence_before_sync();
                mbar_arrive(empty_bar);
            } else {
                const size_t slot_elems = static_cast<size_t>(BLK_M) * BN;
                float* slot0 = p.sk_partials +
                               static_cast<size_t>(u.sk_index) * p.sk_max_contrib * slot_elems;
                sk_epilogue<BN, F16OUT>(tmem_acc, q, lane, issuer, staging, &tmC, mt * BLK_M,
                                        nt * BN, p.M, p.N, sub_count, EPI_BAR_ID, wd.aborted,
                                        slot0, slot_elems, u.contrib, u.ncontrib,
                                        p.sk_tickets + u.sk_index, p.epoch, ticket_smem, [&] {
                                            tc_fence_before_sync();
                                            mbar_arrive(empty_bar);
                                        });
            }
            if (issuer) trace_unit(p, eui, TRACE_U_EPI_END, globaltimer_ns());
            ++eui;
            if (ACC == 2) {
                acc ^= 1;
                if (acc == 0) acc_phase ^= 1u;
            } else {
                acc_phase ^= 1u;
            }
        }
        // each warp's stores have read their staging before the CTA exits
        if (lane == 0) bulk_wait_group<0>();
        if (issuer) trace_header(p, TRACE_H_UNITS, static_cast<unsigned long long>(eui));
    }

    tc_fence_before_sync();
    __syncthreads();
    if (tid == 0) trace_header(p, TRACE_H_END, globaltimer_ns());
    if (warp == 1) {
        tc_fence_after_sync();
        tmem_dealloc(tmem_base, TMEM_COLS);
    }
}

namespace {

template <typename KernelT>
cudaError_t launch_kernel(KernelT kernel, const LaunchSpec& s, cudaStream_t stream)
{
    cudaError_t e = ensure_smem_limit(kernel, s.smem_bytes);
    if (e != cudaSuccess) return e;
    return launch_programmatic(kernel, s, WS_THREADS, stream);
}

template <int BN, bool F16OUT>
cudaError_t launch_bn(const LaunchSpec& s, cudaStream_t stream)
{
    if (s.variant == VAR_PERSISTENT) return launch_kernel(k_ws<BN, F16OUT, true>, s, stream);
    if (s.variant == VAR_WS_PIPELINED) return launch_kernel(k_ws<BN, F16OUT, false>, s, stream);
    return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t launch_ws(const LaunchSpec& s, cudaStream_t stream)
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
