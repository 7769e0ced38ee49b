// kernel_ws2.cuh -- the persistent, warp-specialised GEMM on CTA pairs: a
// cluster of two CTAs on the two SMs of a TPC computes one 256 x PAIR_BN
// output tile with tcgen05.mma.cta_group::2 issued by the pair's leader.
// Template flags: DYN (tile schedule, below) and KS (K blocks of 64 per
// pipeline stage: 1, or 2 for stages of K = 128).  Each (DYN, KS) combination
// is instantiated by a translation unit of its own: kernel_ws2.cu,
// kernel_ws2_k2.cu, kernel_ws2_dyn.cu, kernel_ws2_dyn_k2.cu.
//
// Why pairs: with one CTA per tile the 128 x 256 tile leaves room for only
// four 48 KB stages beside the output staging.  In a pair each CTA keeps its
// own 128 rows of A and half of B (128 rows) per 64-wide K block -- 32 KB --
// so six such stages fit (or three of K = 128), and every byte of B fetched
// from L2 feeds 256 rows of A instead of 128.
//
// No TMA multicast is used: each CTA loads its own tiles into its own shared
// memory.  Both CTAs' copies signal the LEADER's full[s] barrier (the
// .cta_group::2 form of the bulk tensor copy), which the leader's producer
// arms with the pair's whole byte budget; the leader's MMA commits are
// multicast to both CTAs' empty[s] / tmem_full[a] barriers; both CTAs'
// epilogue warps arrive on the leader's tmem_empty[a].
//
// Roles per CTA (192 threads):
//   warp 0          TMA producer (both CTAs): the warp waits, lane 0 copies
//   warp 1          MMA issuer (leader only): the warp waits, lane 0 issues;
//                   warp 1 of each CTA allocates TMEM
//   warps 2..5      epilogue of this CTA's 128 rows of the pair tile
// The ring position {stage, phase} and the accumulator position run on
// continuously across tiles.
//
// Tile schedules (template flag DYN):
//   static   a grid of one cluster per TPC; cluster c takes the tiles of the
//            WorkIter sequence (c, c + clusters, ..., then stream-K units).
//   dynamic  a grid of one cluster per tile.  A running cluster takes its own
//            tile, then keeps cancelling clusters that have not started yet
//            (clusterlaunchcontrol.try_cancel) and takes their tiles, so
//            clusters that finish early take more tiles and no cluster waits
//            on a fixed share.  The leader's producer issues one request at
//            the start of each tile; the response is multicast into both
//            CTAs' response ring (CLC_SLOTS slots), where every reader -- both
//            producers, the MMA issuer and the eight epilogue warps -- decodes
//            it and releases the slot to the leader's empty barrier.  A
//            response that cancelled nothing ends the cluster.  "GEMM II --
//            pipelining with TMA" (Step 6, the persistent scheduler) names
//            cluster launch control as the upgrade of its precomputed tile
//            assignment: hardware work-stealing for uneven tile costs.

#pragma once

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

__device__ __forceinline__ uint32_t clc_resp(uint32_t bars, int slot)
{
    return bars + CLC_RESP_OFFSET + static_cast<uint32_t>(slot) * CLC_RESP_BYTES;
}

// Readers of every cancellation response, per CTA pair: the producer, the MMA
// issuer and the four epilogue warps of the leader; the producer and the four
// epilogue warps of the peer.
constexpr int CLC_READERS_PER_PAIR = 11;

// One reader's take of response `use` (slot use % CLC_SLOTS): wait for it,
// decode it, re-arm this CTA's full barrier of the slot for the slot's next
// use when `arm` (one reader per CTA, its producer), and release the slot to
// the cluster's rank-0 CTA.  Returns the work unit (pair tile) of the
// cancelled cluster, or -1 when nothing was cancelled (every cluster has
// started) or the run aborted.
__device__ __forceinline__ int clc_read(uint32_t bars, int use, Watchdog& wd, bool arm)
{
    const int slot = use % CLC_SLOTS;
    const uint32_t full = bar_addr(bars, BAR_CLC_FULL + slot);
    if (!wd.wait(full, static_cast<uint32_t>(use / CLC_SLOTS) & 1u, WAIT_CLC_FULL, -1, use))
        return -1;
    uint32_t cta_x = 0;
    const bool cancelled = clc_decode(clc_resp(bars, slot), cta_x);
    if (arm) mbar_arrive_expect_tx(full, CLC_RESP_BYTES);
    // Relaxed: the slot's only access here is the load just decoded, whose
    // value this thread has already consumed.  A release fence would also
    // wait for the MMA issuer's queued tensor-core work at every tile start
    // (measured 1.1 us per tile of drained MMA pipe at 8192^3).
    mbar_arrive_cluster_relaxed(map_shared_rank(bar_addr(bars, BAR_CLC_EMPTY + slot), 0));
    return cancelled ? static_cast<int>(cta_x / 2u) : -1;
}

// The tile sequence of one cluster as each of its roles walks it: the static
// WorkIter sequence, or (DYN) the cluster's own tile followed by the tile of
// every cluster that its cancellation requests took over.
template <bool DYN>
struct PairTiles {
    WorkIter it;  // static schedule
    int own;      // dynamic: this cluster's own unit
    int use;      // dynamic: responses read so far; -1 before the own unit
    int KB;
    int dp;       // dynamic: units below dp are whole tiles
    int splits;   // dynamic: K ranges per tile of the split tail (< 2: none)

    // Next unit for a single-thread reader (`arm` as in clc_read).
    __device__ __forceinline__ bool next(WorkUnit& u, uint32_t bars, Watchdog& wd, bool arm)
    {
        if constexpr (!DYN) {
            return it.next(u);
        } else {
            int t = own;
            if (use >= 0) t = clc_read(bars, use, wd, arm);
            ++use;
            return take(u, t);
        }
    }

    // Next unit for a whole warp: lane 0 reads the response (re-arming the
    // slot when `arm`), the tile is broadcast to the other lanes.
    __device__ __forceinline__ bool next_warp(WorkUnit& u, uint32_t bars, Watchdog& wd,
                                              uint32_t lane, bool arm = false)
    {
        if constexpr (!DYN) {
            return it.next(u);
        } else {
            int t = own;
            if (use >= 0) {
                t = lane == 0 ? clc_read(bars, use, wd, arm) : -1;
                t = __shfl_sync(0xffffffffu, t, 0);
            }
            ++use;
            return take(u, t);
        }
    }

    __device__ __forceinline__ bool take(WorkUnit& u, int t) const
    {
        if (t < 0) return false;
        dynamic_unit(t, dp, splits, KB, u);
        return true;
    }
};

}  // namespace

constexpr int PAIR_THREADS = 192;
constexpr int PAIR_BM = 2 * BLK_M;   // 256 output rows per pair tile
constexpr uint32_t PAIR_EPI_BAR_ID = 1;

__host__ __device__ constexpr uint32_t pow2_at_least(uint32_t x)
{
    uint32_t r = 32;
    while (r < x) r <<= 1;
    return r;
}

// PAIR_BN: output columns per pair tile (a multiple of 32 up to 256; each CTA
// holds PAIR_BN / 2 rows of B per stage).
template <int PAIR_BN, bool F16OUT, bool DYN, int KS>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(PAIR_THREADS, 1)
    k_ws2(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
          const __grid_constant__ CUtensorMap tmC, const __grid_constant__ CUtensorMap tmB2,
          const Params p)
{
    static_assert(PAIR_BN % 32 == 0 && PAIR_BN >= 64 && PAIR_BN <= 256, "pair tile width");
    static_assert(!F16OUT || PAIR_BN % 64 == 0 || PAIR_BN % 64 == 32,
                  "fp16 output: 64-column sub-tiles plus at most one 32-column remainder");
    constexpr int HALF_BN = PAIR_BN / 2;  // B rows held by each CTA
    // Half-width tiles (the last p.tail_halves tiles of the dynamic schedule,
    // each run as two units; see dynamic_unit): PAIR_BN / 2 columns,
    // HALF_BN / 2 rows of B per CTA through tmB2, for the widths whose half
    // the epilogue stores in whole sub-tiles.
    constexpr int NARROW_BN = PAIR_BN / 2;
    constexpr bool NARROW_OK =
        DYN && (F16OUT ? (NARROW_BN % 64 == 0 || NARROW_BN % 64 == 32)
                                  : NARROW_BN % 32 == 0);
    constexpr int ACC = 2;
    // two accumulators of PAIR_BN columns, rounded up to a legal allocation
    constexpr uint32_t TMEM_COLS = pow2_at_least(ACC * PAIR_BN);
    const int D = p.pipe_depth;
    const CtaSmem sm = cta_smem();
    // A stage holds KS K blocks of 64, each in a sub-slot of its own (sub-slot
    // stage * KS + s).  KS = 2 is the K = 128 stage of "05 Async Data Movement
    // - TMA" (Using 3D TMA to Move Multiple Swizzle Atoms): the 128-wide slice
    // is split into two 64-wide groups, each a 128-byte swizzle row.  The page
    // writes both groups with one 3-D copy; here each group is its own 2-D box,
    // which lands the same bytes and keeps the zero fill past a ragged K edge
    // (a 3-D view of a row-major matrix would read the next row there).
    static_assert(KS == 1 || KS == 2, "K blocks of 64 per stage");
    const SmemLayout L = smem_layout(D * KS, HALF_BN, NUM_STAGING);
    const uint32_t sA = sm.base + L.a;
    const uint32_t sB = sm.base + L.b;
    const uint32_t staging = sm.base + L.staging;
    const uint32_t bars = sm.base + L.bars;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm.gen + L.bars + TMEM_SLOT_OFFSET);
    const int tid = static_cast<int>(threadIdx.x);
    const int warp = tid >> 5;
    const uint32_t lane = lane_id();
    const uint32_t rank = cluster_ctarank();
    const uint32_t pr = rank;                  // rank in the pair: 0 = leader
    const uint32_t leader_rank = 0;
    const bool leader = pr == 0;
    Watchdog wd = make_watchdog(p);
    // One work unit (a pair tile, or a K range of one) per cluster at a time.
    const int cluster = static_cast<int>(blockIdx.x) / 2;
    const int nclusters = static_cast<int>(gridDim.x) / 2;
    const int KB = (p.k_blocks + KS - 1) / KS;  // stages per tile
    PairTiles<DYN> tiles0;
    tiles0.it.init(cluster, nclusters, p.dp_tiles, p.sk_tiles, KB, p.sk_kb_per_worker);
    tiles0.own = cluster;
    tiles0.use = -1;
    tiles0.KB = KB;
    tiles0.dp = DYN && p.sk_tiles > 0      ? p.dp_tiles
                : NARROW_OK && p.tail_halves > 0 ? p.num_tiles - p.tail_halves
                                                 : 0x7FFFFFFF;
    tiles0.splits = DYN && p.sk_tiles > 0 ? p.sk_max_contrib
                    : NARROW_OK && p.tail_halves > 0 ? 0
                                                     : 1;

    if (warp == 0 && lane == 0) {
        prefetch_tensormap(&tmA);
        prefetch_tensormap(&tmB);
        prefetch_tensormap(&tmC);
        if (NARROW_OK && p.tail_halves > 0) prefetch_tensormap(&tmB2);
        for (int s = 0; s < D; ++s) {
            mbar_init(bar_addr(bars, BAR_FULL + s), 1);   // leader: its producer's expect_tx
            mbar_init(bar_addr(bars, BAR_EMPTY + s), 1);   // the leader's multicast commit
        }
        for (int a = 0; a < ACC; ++a) {
            mbar_init(bar_addr(bars, BAR_TMEM_FULL + a), 1);   // the leader's multicast commit
            mbar_init(bar_addr(bars, BAR_TMEM_EMPTY + a), 8);  // leader: 4 epilogue warps x 2 CTAs
        }
        if constexpr (DYN) {
            for (int j = 0; j < CLC_SLOTS; ++j) {
                mbar_init(bar_addr(bars, BAR_CLC_FULL + j), 1);  // this CTA's producer arms it
                mbar_init(bar_addr(bars, BAR_CLC_EMPTY + j), CLC_READERS_PER_PAIR);  // rank 0's
            }
        }
        mbar_init(bar_addr(bars, BAR_DRAIN), 1);
        mbar_init(bar_addr(bars, BAR_STALL), 1);
        fence_mbar_init();
        if constexpr (DYN) {
            // the first use of every response slot expects its 16 bytes
            for (int j = 0; j < CLC_SLOTS; ++j)
                mbar_arrive_expect_tx(bar_addr(bars, BAR_CLC_FULL + j), CLC_RESP_BYTES);
        }
    }
    if (warp == 1) {
        tmem_alloc_pair(smem_u32(tmem_slot), TMEM_COLS);
        tmem_relinquish_alloc_permit_pair();
    }
    // every CTA's barriers exist before any CTA of the cluster touches another's
    tc_fence_before_sync();
    cluster_sync_all();
    tc_fence_after_sync();
    // Everything above touches only shared memory, TMEM and the kernel's
    // parameters; global memory (A, B, C, the status record, the trace) is
    // accessed only after the work before this launch has completed.
    griddep_wait();
    griddep_launch_dependents();
    const uint32_t tmem_base = *tmem_slot;
    if (tid == 0) {
        trace_header(p, TRACE_H_START, globaltimer_ns());
        trace_header(p, TRACE_H_SMID, sm_id());
    }

    // The producer and MMA roles run as whole warps: every lane walks the
    // loop and waits on each barrier, lane 0 issues the copies or the MMAs,
    // and the warp reconverges after every stage.  With the other 31 lanes
    // parked at a warp barrier while lane 0 ran the main loop alone, the same
    // kernel measured 9% slower at 8192^3 on GB300 (1693 vs 1852 TFLOP/s).
    if (warp == 0) {
        // ---------------------------------------------------- TMA producer
        // both CTAs' A and B, all KS blocks (a block past K arrives zero-filled)
        const uint32_t pair_tx = 2u * stage_tx_bytes(HALF_BN) * static_cast<uint32_t>(KS);
        const uint32_t narrow_tx = 2u * stage_tx_bytes(HALF_BN / 2) * static_cast<uint32_t>(KS);
        const uint64_t pol_a = (p.l2_policy == 2) ? policy_evict_first() : policy_evict_last();
        const uint64_t pol_b = (p.l2_policy == 1) ? policy_evict_first() : policy_evict_last();
        const bool tr = p.trace && lane == 0;
        if (p.debug_stall) wd.wait(bar_addr(bars, BAR_STALL), 0, WAIT_STALL, -1, -1);
        int stage = 0;
        uint32_t phase = 0;
        int armed = 0;
        int end_stage = 0;       // ring position just after the last armed stage
        uint32_t end_phase = 0;
        int requests = 0;        // dynamic schedule: cancellation requests issued
        PairTiles<DYN> tiles = tiles0;
        WorkUnit u;
        int ui = 0;
        while (tiles.next_warp(u, bars, wd, lane, true)) {
            const int t = u.tile;
            if constexpr (DYN) {
                // Ask for the tile after this one now; its response is read
                // when this tile's loads have all been issued.
                if (rank == 0 && lane == 0 && !wd.aborted) {
                    const int slot = requests % CLC_SLOTS;
                    const uint32_t free_parity =
                        (static_cast<uint32_t>(requests / CLC_SLOTS) & 1u) ^ 1u;
                    if (wd.wait(bar_addr(bars, BAR_CLC_EMPTY + slot), free_parity,
                                WAIT_CLC_EMPTY, t, -1)) {
                        clc_try_cancel_multicast(clc_resp(bars, slot),
                                                 bar_addr(bars, BAR_CLC_FULL + slot));
                        ++requests;
                    }
                }
                __syncwarp();
            }
            if (tr)
                trace_unit(p, ui, TRACE_U_TILE,
                           (static_cast<unsigned long long>(t) << 32) |
                               static_cast<unsigned>(u.kb1 - u.kb0));
            unsigned long long empty_wait_ns = 0;
            int mt, nt;
            raster_tile(t, p.tiles_m, p.tiles_n, p.group_m, mt, nt);
            const bool narrow = NARROW_OK && u.half != 0;
            const int m0 = mt * PAIR_BM + static_cast<int>(pr) * BLK_M;
            const int nb = narrow ? nt * PAIR_BN + (u.half - 1) * NARROW_BN +
                                        static_cast<int>(pr) * (HALF_BN / 2)
                                  : nt * PAIR_BN + static_cast<int>(pr) * HALF_BN;
            const CUtensorMap* mapB = narrow ? &tmB2 : &tmB;
            for (int ki = 0; ki < u.kb1 - u.kb0; ++ki) {
                const int kb = kblock_at(ki, DYN ? t / p.snake_span : ui, u.kb0, u.kb1,
                                         p.k_snake);
                const unsigned long long tw0 = tr ? globaltimer_ns() : 0ull;
                const bool ok =
                    wd.wait(bar_addr(bars, BAR_EMPTY + stage), phase ^ 1u, WAIT_EMPTY, t, kb);
                if (tr) empty_wait_ns += globaltimer_ns() - tw0;
                if (lane == 0 && ok) {
                    const uint32_t fb_local = bar_addr(bars, BAR_FULL + stage);
                    const uint32_t fb_leader = map_shared_rank(fb_local, leader_rank);
                    if (leader) {
                        mbar_arrive_expect_tx(fb_local, narrow ? narrow_tx : pair_tx);
                        ++armed;
                    }
#pragma unroll
                    for (int s = 0; s < KS; ++s) {
                        const int slot = stage * KS + s;
                        const int kx = (kb * KS + s) * BLK_K;
                        if (p.l2_policy == 0) {
                            tma_load_2d_pair(sA + slot * A_TILE_BYTES, &tmA, fb_leader, kx, m0);
                            tma_load_2d_pair(sB + slot * b_tile_bytes(HALF_BN), mapB, fb_leader,
                                             kx, nb);
                        } else {
                            tma_load_2d_pair_hint(sA + slot * A_TILE_BYTES, &tmA, fb_leader, kx,
                                                  m0, pol_a);
                            tma_load_2d_pair_hint(sB + slot * b_tile_bytes(HALF_BN), mapB,
                                                  fb_leader, kx, nb, pol_b);
                        }
                    }
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
        if (lane == 0 && wd.aborted) {
            // Let copies already in flight land before the CTA can exit: the
            // leader drains the phases it armed, the peer waits one
            // budget-bounded grace period (its copies signal the leader).
            if (leader) {
                int st = end_stage;
                uint32_t ph = end_phase;
                for (int i = 0; i < D && i < armed; ++i) {
                    if (st == 0) {
                        st = D - 1;
                        ph ^= 1u;
                    } else {
                        --st;
                    }
                    wd.drain(bar_addr(bars, BAR_FULL + st), ph);
                }
                if constexpr (DYN) {
                    // the last cancellation request may still be in flight
                    if (requests > 0) {
                        const int r = requests - 1;
                        wd.drain(bar_addr(bars, BAR_CLC_FULL + r % CLC_SLOTS),
                                 static_cast<uint32_t>(r / CLC_SLOTS) & 1u);
                    }
                }
            } else {
                const uint64_t t0 = globaltimer_ns();
                while (globaltimer_ns() - t0 < 200000ull) {
                }
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        if (leader) {
            // ----------------------------------------------- MMA issuer (leader)
            constexpr uint32_t idesc_full = idesc_f16_f32(PAIR_BM, PAIR_BN);
            constexpr uint32_t idesc_narrow = idesc_f16_f32(PAIR_BM, NARROW_BN);
            const bool tr = p.trace && lane == 0;
            int stage = 0;
            uint32_t phase = 0;
            int acc = 0;
            uint32_t acc_phase = 0;
            int mui = 0;
            PairTiles<DYN> tiles = tiles0;
            WorkUnit u;
            while (tiles.next_warp(u, bars, wd, lane)) {
                const int t = u.tile;
                wd.wait(bar_addr(bars, BAR_TMEM_EMPTY + acc), acc_phase ^ 1u, WAIT_TMEM_EMPTY,
                        t, -1);
                tc_fence_after_sync();
                if (tr) trace_unit(p, mui, TRACE_U_ACC_FREE, globaltimer_ns());
                unsigned long long full_wait_ns = 0;
                const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * PAIR_BN);
                const uint32_t idesc = (NARROW_OK && u.half != 0) ? idesc_narrow : idesc_full;
                for (int ki = 0; ki < u.kb1 - u.kb0; ++ki) {
                    const int kb = kblock_at(ki, DYN ? t / p.snake_span : mui, u.kb0, u.kb1,
                                             p.k_snake);
                    const unsigned long long tw0 = tr ? globaltimer_ns() : 0ull;
                    const bool ok =
                        wd.wait(bar_addr(bars, BAR_FULL + stage), phase, WAIT_FULL, t, kb);
                    if (tr) full_wait_ns += globaltimer_ns() - tw0;
                    if (lane == 0 && ok) {
                        tc_fence_after_sync();
                        if (tr && ki == 0) trace_unit(p, mui, TRACE_U_MMA_FIRST, globaltimer_ns());
#pragma unroll
                        for (int s = 0; s < KS; ++s) {
                            // the second block of the last stage may lie past K
                            if (s > 0 && kb * KS + s >= p.k_blocks) break;
                            const int slot = stage * KS + s;
                            const uint64_t adesc = sw128_kmajor_desc(sA + slot * A_TILE_BYTES);
                            const uint64_t bdesc =
                                sw128_kmajor_desc(sB + slot * b_tile_bytes(HALF_BN));
#pragma unroll
                            for (int kk = 0; kk < BLK_K / MMA_K; ++kk)
                                mma_f16_ss_pair(d_tmem, adesc + static_cast<uint64_t>(kk * 2),
                                                bdesc + static_cast<uint64_t>(kk * 2), idesc,
                                                (ki == 0 && s == 0 && kk == 0) ? 0u : 1u);
                        }
                        // frees stage `stage` in both CTAs once these MMAs have read it
                        mma_commit_pair_multicast(bar_addr(bars, BAR_EMPTY + stage), 0x3);
                    }
                    __syncwarp();
                    if (++stage == D) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (lane == 0 && !wd.aborted)
                    mma_commit_pair_multicast(bar_addr(bars, BAR_TMEM_FULL + acc), 0x3);
                if (tr) {
                    trace_unit(p, mui, TRACE_U_MMA_LAST, globaltimer_ns());
                    trace_unit(p, mui, TRACE_U_FULL_WAIT, full_wait_ns);
                }
                __syncwarp();
                ++mui;
                acc ^= 1;
                if (acc == 0) acc_phase ^= 1u;
            }
            // every pair MMA has completed before TMEM is released
            if (lane == 0) {
                mma_commit_pair_multicast(bar_addr(bars, BAR_DRAIN),
                                          static_cast<uint16_t>(1u << rank));
                wd.drain(bar_addr(bars, BAR_DRAIN), 0);
            }
        }
        __syncwarp();
    } else {
        // -------------------------------------------------------- epilogue
        const int q = warp & 3;
        const bool issuer = (tid == 2 * 32);
        int acc = 0;
        uint32_t acc_phase = 0;
        uint32_t sub_count = 0;
        PairTiles<DYN> tiles = tiles0;
        WorkUnit u;
        volatile uint32_t* ticket_smem =
            reinterpret_cast<volatile uint32_t*>(sm.gen + L.bars + TICKET_SLOT_OFFSET);
        int eui = 0;
        while (tiles.next_warp(u, bars, wd, lane)) {
            const int t = u.tile;
            int mt, nt;
            raster_tile(t, p.tiles_m, p.tiles_n, p.group_m, mt, nt);
            const int m0 = mt * PAIR_BM + static_cast<int>(pr) * BLK_M;
            wd.wait(bar_addr(bars, BAR_TMEM_FULL + acc), acc_phase, WAIT_TMEM_FULL, t, -1);
            tc_fence_after_sync();
            if (issuer) trace_unit(p, eui, TRACE_U_EPI_START, globaltimer_ns());
            const uint32_t tmem_acc = tmem_base + static_cast<uint32_t>(acc * PAIR_BN);
            const uint32_t empty_leader =
                map_shared_rank(bar_addr(bars, BAR_TMEM_EMPTY + acc), leader_rank);
            auto release = [&] {
                tc_fence_before_sync();
                __syncwarp();
                if (lane == 0) mbar_arrive_cluster(empty_leader);
            };
            if (NARROW_OK && u.half != 0) {
                if constexpr (NARROW_OK)
                    epilogue_tma_store<NARROW_BN, F16OUT>(
                        tmem_acc, q, lane, staging, &tmC, m0,
                        nt * PAIR_BN + (u.half - 1) * NARROW_BN, p.M, p.N, sub_count,
                        !wd.aborted, p.C);
                release();
            } else if (u.ncontrib == 1) {
                epilogue_tma_store<PAIR_BN, F16OUT>(tmem_acc, q, lane, staging, &tmC, m0,
                                                    nt * PAIR_BN, p.M, p.N, sub_count,
                                                    !wd.aborted, p.C);
                release();
            } else {
                // each CTA fixes up its own 128 rows of the pair tile
                const size_t slot_elems = static_cast<size_t>(BLK_M) * PAIR_BN;
                float* slot0 = p.sk_partials +
                               (static_cast<size_t>(u.sk_index) * p.sk_max_contrib * 2 + pr) *
                                   slot_elems;
                sk_epilogue<PAIR_BN, F16OUT>(tmem_acc, q, lane, issuer, staging, &tmC, m0,
                                             nt * PAIR_BN, p.M, p.N, sub_count, PAIR_EPI_BAR_ID,
                                             wd.aborted, slot0, 2 * slot_elems, u.contrib,
                                             u.ncontrib, p.sk_tickets + u.sk_index * 2 + pr,
                                             p.epoch, ticket_smem, release, p.C);
            }
            if (issuer) trace_unit(p, eui, TRACE_U_EPI_END, globaltimer_ns());
            ++eui;
            acc ^= 1;
            if (acc == 0) acc_phase ^= 1u;
        }
        // each warp's stores have read their staging before the CTA exits
        if (lane == 0) bulk_wait_group<0>();
        if (issuer) trace_header(p, TRACE_H_UNITS, static_cast<unsigned long long>(eui));
        __syncwarp();
    }

    // nothing of either CTA is touched remotely after this point
    tc_fence_before_sync();
    cluster_sync_all();
    if (tid == 0) trace_header(p, TRACE_H_END, globaltimer_ns());
    if (warp == 1) {
        tc_fence_after_sync();
        tmem_dealloc_pair(tmem_base, TMEM_COLS);
    }
}

template <typename KernelT>
cudaError_t launch_pair_kernel(KernelT kernel, const LaunchSpec& s, cudaStream_t stream)
{
    cudaError_t e = ensure_smem_limit(kernel, s.smem_bytes);
    if (e != cudaSuccess) return e;
    return launch_programmatic(kernel, s, PAIR_THREADS, stream, s.tmB2 ? *s.tmB2 : *s.tmB);
}

// Launch k_ws2<block_n, f16out, DYN, KS> for one of the built pair tile
// widths.  Each (DYN, KS) combination is instantiated by a translation unit
// of its own (kernel_ws2.cu, kernel_ws2_k2.cu, kernel_ws2_dyn.cu,
// kernel_ws2_dyn_k2.cu), so that they compile in parallel.
template <bool DYN, int KS>
cudaError_t launch_pair_width(const LaunchSpec& s, cudaStream_t stream)
{
    if (s.f16out) {
        switch (s.block_n) {
        case 128: return launch_pair_kernel(k_ws2<128, true, DYN, KS>, s, stream);
        case 160: return launch_pair_kernel(k_ws2<160, true, DYN, KS>, s, stream);
        case 192: return launch_pair_kernel(k_ws2<192, true, DYN, KS>, s, stream);
        case 224: return launch_pair_kernel(k_ws2<224, true, DYN, KS>, s, stream);
        case 256: return launch_pair_kernel(k_ws2<256, true, DYN, KS>, s, stream);
        default: return cudaErrorInvalidValue;
        }
    }
    switch (s.block_n) {
    case 128: return launch_pair_kernel(k_ws2<128, false, DYN, KS>, s, stream);
    case 160: return launch_pair_kernel(k_ws2<160, false, DYN, KS>, s, stream);
    case 192: return launch_pair_kernel(k_ws2<192, false, DYN, KS>, s, stream);
    case 224: return launch_pair_kernel(k_ws2<224, false, DYN, KS>, s, stream);
    case 256: return launch_pair_kernel(k_ws2<256, false, DYN, KS>, s, stream);
    default: return cudaErrorInvalidValue;
    }
}

extern template cudaError_t launch_pair_width<false, 1>(const LaunchSpec&, cudaStream_t);
extern template cudaError_t launch_pair_width<false, 2>(const LaunchSpec&, cudaStream_t);
extern template cudaError_t launch_pair_width<true, 1>(const LaunchSpec&, cudaStream_t);
extern template cudaError_t launch_pair_width<true, 2>(const LaunchSpec&, cudaStream_t);

}  // namespace tg
