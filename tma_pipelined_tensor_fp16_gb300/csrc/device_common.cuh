// device_common.cuh -- device-side pieces shared by every GEMM variant: the
// bounded mbarrier wait (watchdog), the TMEM -> swizzled SMEM -> TMA-store
// epilogue and the plain masked-store epilogue.
#pragma once

#include <cuda_fp16.h>

#include "gemm_common.h"
#include "ptx.cuh"

namespace tg {

// ------------------------------------------------------------ bounded waits
//
// Every wait on an mbarrier is bounded.  A wait that has not completed within
// `budget_ns` records a timeout in the plan's status record and marks the run
// aborted (abort_epoch = this run's epoch); waits in every other CTA of the
// same run notice the abort within a few polls and give up too.  An aborted
// thread skips all further waits, copies, MMAs and stores but keeps executing
// the same sequence of thread barriers as its peers, so no CTA can be left
// parked on a barrier: the kernel always reaches its teardown, frees TMEM and
// exits, and the host reads the code after synchronising.

struct Watchdog {
    DevStatus* st;
    int epoch;
    unsigned long long budget_ns;
    bool aborted;

    __device__ __forceinline__ void record(int where, int tile, int kb)
    {
        if (atomicCAS(&st->code, DEV_OK, DEV_TIMEOUT) == DEV_OK) {
            st->where = where;
            st->block = static_cast<int>(blockIdx.x);
            st->tile = tile;
            st->kblock = kb;
        }
        atomicExch(&st->abort_epoch, epoch);
        __threadfence();
        aborted = true;
    }

    __device__ __forceinline__ bool peer_aborted() const
    {
        return *reinterpret_cast<volatile int*>(&st->abort_epoch) == epoch;
    }

    // Returns true if the phase of `bar` with parity `parity` completed.
    __device__ __forceinline__ bool wait(uint32_t bar, uint32_t parity, int where, int tile,
                                         int kb)
    {
        if (aborted) return false;
        if (mbar_try_wait(bar, parity)) return true;
        const uint64_t t0 = globaltimer_ns();
        uint32_t polls = 0;
        while (true) {
            if (mbar_try_wait(bar, parity)) return true;
            if ((++polls & 31u) == 0) {
                if (peer_aborted()) {
                    aborted = true;
                    return false;
                }
                if (globaltimer_ns() - t0 > budget_ns) {
                    record(where, tile, kb);
                    return false;
                }
            }
        }
    }

    // Teardown drain: wait for a phase with a short bound, recording nothing
    // (the run is already known to be aborted, or the phase is complete).
    __device__ __forceinline__ void drain(uint32_t bar, uint32_t parity) const
    {
        if (mbar_try_wait(bar, parity)) return;
        const uint64_t t0 = globaltimer_ns();
        while (!mbar_try_wait(bar, parity)) {
            if (globaltimer_ns() - t0 > budget_ns) return;
        }
    }
};

__device__ __forceinline__ Watchdog make_watchdog(const Params& p)
{
    Watchdog w;
    w.st = p.status;
    w.epoch = p.epoch;
    w.budget_ns = p.budget_ns;
    w.aborted = false;
    return w;
}

// ----------------------------------------------------------------- epilogue
//
// "GEMM II -- pipelining with TMA", the TMA-store epilogue: TMEM -> registers
// (tcgen05.ld + wait.ld), narrow to the output dtype, registers -> shared
// staging, fence.proxy_async so the TMA proxy sees the thread writes, then
// one thread issues the bulk tensor store and commits it as a bulk group;
// wait_group(.read) gates reuse of the staging buffer ("05 Async Data
// Movement - TMA", "How to Wait for a TMA Store").
//
// A 128-thread group (4 warps) drains one 128 x BLOCK_N fp32 accumulator.
// Warp q of the group (q = warp index mod 4) may only reach TMEM lanes
// 32q..32q+31, so thread `lane` of warp q owns output row 32q + lane.  The
// tile leaves in sub-tiles of 128 rows x 128 bytes (64 fp16 or 32 fp32
// columns), written into a 128-byte-swizzled staging buffer: the 16-byte
// chunk c of row r lands at chunk c ^ (r mod 8), which is the layout the
// C tensor map's SWIZZLE_128B expects and spreads each 8-thread phase of the
// st.shared.v4 over all 32 banks.

template <int BLOCK_N, bool F16OUT>
struct EpilogueShape {
    static constexpr int SUB_COLS = F16OUT ? 64 : 32;  // columns per 128-byte row
    static constexpr int NUM_SUB = BLOCK_N / SUB_COLS;
};

__device__ __forceinline__ uint32_t pack_half2(uint32_t lo_bits, uint32_t hi_bits)
{
    __half2 h = __floats2half2_rn(__uint_as_float(lo_bits), __uint_as_float(hi_bits));
    return *reinterpret_cast<uint32_t*>(&h);
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c,
                                             uint32_t d)
{
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c),
                 "r"(d)
                 : "memory");
}

// `staging`: shared address of NUM_STAGING buffers of STAGING_BYTES, 1024-B
// aligned.  `sub_count` counts the sub-tiles this group has staged so far (it
// carries across tiles and selects the staging buffer).  `bar_id` is a named
// barrier reserved for the 128 threads.  `issuer` is exactly one thread of the
// group.  Stores are skipped (but every barrier is still executed) when
// `do_store` is false.
template <int BLOCK_N, bool F16OUT>
__device__ __forceinline__ void epilogue_tma_store(uint32_t tmem_acc, int q, uint32_t lane,
                                                   bool issuer, uint32_t staging,
                                                   const CUtensorMap* tmap_c, int m0, int n0,
                                                   int N, uint32_t& sub_count, uint32_t bar_id,
                                                   bool do_store)
{
    using S = EpilogueShape<BLOCK_N, F16OUT>;
    const uint32_t row = static_cast<uint32_t>(q) * 32u + lane;
    const uint32_t taddr = tmem_acc + (static_cast<uint32_t>(q * 32) << 16);
#pragma unroll 1
    for (int j = 0; j < S::NUM_SUB; ++j) {
        const int col0 = n0 + j * S::SUB_COLS;
        if (col0 >= N) break;  // uniform across the group: the rest is past the edge

        uint32_t v[S::SUB_COLS];
        if constexpr (F16OUT) {
            tmem_load_32cols(taddr + j * 64, *reinterpret_cast<uint32_t(*)[32]>(&v[0]));
            tmem_load_32cols(taddr + j * 64 + 32, *reinterpret_cast<uint32_t(*)[32]>(&v[32]));
        } else {
            tmem_load_32cols(taddr + j * 32, *reinterpret_cast<uint32_t(*)[32]>(&v[0]));
        }

        const uint32_t buf = staging + (sub_count & 1u) * STAGING_BYTES;
        if (sub_count >= 2) {
            // the store issued two sub-tiles ago read this buffer
            if (issuer) bulk_wait_group_read<1>();
            named_bar_sync(bar_id, 128);
        }
        const uint32_t row_base = buf + row * 128u;
#pragma unroll
        for (uint32_t c = 0; c < 8; ++c) {
            const uint32_t dst = row_base + ((c ^ (row & 7u)) << 4);
            if constexpr (F16OUT) {
                st_shared_v4(dst, pack_half2(v[8 * c + 0], v[8 * c + 1]),
                             pack_half2(v[8 * c + 2], v[8 * c + 3]),
                             pack_half2(v[8 * c + 4], v[8 * c + 5]),
                             pack_half2(v[8 * c + 6], v[8 * c + 7]));
            } else {
                st_shared_v4(dst, v[4 * c + 0], v[4 * c + 1], v[4 * c + 2], v[4 * c + 3]);
            }
        }
        fence_proxy_async_smem();
        named_bar_sync(bar_id, 128);
        if (issuer && do_store) {
            tma_store_2d(tmap_c, buf, col0, m0);
            bulk_commit_group();
        }
        ++sub_count;
    }
}

// Plain epilogue without staging (the synchronous baseline's path TMEM ->
// registers -> global): each thread writes its own row with masked 16-byte
// stores.  N is a multiple of 16 bytes of output, so a 16-byte chunk is
// either wholly inside or wholly outside the matrix.
template <int BLOCK_N, bool F16OUT>
__device__ __forceinline__ void epilogue_direct_store(uint32_t tmem_acc, int q, uint32_t lane,
                                                      void* C, int M, int N, int m0, int n0,
                                                      bool do_store)
{
    const uint32_t row = static_cast<uint32_t>(q) * 32u + lane;
    const uint32_t taddr = tmem_acc + (static_cast<uint32_t>(q * 32) << 16);
    const int gm = m0 + static_cast<int>(row);
#pragma unroll 1
    for (int j = 0; j < BLOCK_N / 32; ++j) {
        const int col0 = n0 + j * 32;
        if (col0 >= N) break;
        uint32_t v[32];
        tmem_load_32cols(taddr + j * 32, v);
        if (!do_store || gm >= M) continue;
        if constexpr (F16OUT) {
            __half* crow = static_cast<__half*>(C) + static_cast<size_t>(gm) * N;
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const int gn = col0 + 8 * c;
                if (gn < N) {
                    uint4 w;
                    w.x = pack_half2(v[8 * c + 0], v[8 * c + 1]);
                    w.y = pack_half2(v[8 * c + 2], v[8 * c + 3]);
                    w.z = pack_half2(v[8 * c + 4], v[8 * c + 5]);
                    w.w = pack_half2(v[8 * c + 6], v[8 * c + 7]);
                    *reinterpret_cast<uint4*>(crow + gn) = w;
                }
            }
        } else {
            float* crow = static_cast<float*>(C) + static_cast<size_t>(gm) * N;
#pragma unroll
            for (int c = 0; c < 8; ++c) {
                const int gn = col0 + 4 * c;
                if (gn < N) {
                    uint4 w = make_uint4(v[4 * c + 0], v[4 * c + 1], v[4 * c + 2], v[4 * c + 3]);
                    *reinterpret_cast<uint4*>(crow + gn) = w;
                }
            }
        }
    }
}

// Round x up to a multiple of 1024 (shared-memory tile alignment that the
// 128-byte swizzle pattern and the MMA descriptors assume).
__device__ __forceinline__ uint32_t align1024(uint32_t x) { return (x + 1023u) & ~1023u; }

}  // namespace tg
