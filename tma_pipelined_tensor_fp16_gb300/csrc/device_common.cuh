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

// ----------------------------------------------------------------- timeline

__device__ __forceinline__ uint32_t sm_id()
{
    uint32_t r;
    asm volatile("mov.u32 %0, %%smid;" : "=r"(r));
    return r;
}

// Unit `unit` of this CTA, word `word` (no-op when tracing is off or the unit
// is past the buffer's capacity).
__device__ __forceinline__ void trace_unit(const Params& p, int unit, int word,
                                           unsigned long long v)
{
    if (p.trace != nullptr && unit < p.trace_units)
        p.trace[trace_index(static_cast<int>(blockIdx.x), p.trace_units, 1 + unit, word)] = v;
}

__device__ __forceinline__ void trace_header(const Params& p, int word, unsigned long long v)
{
    if (p.trace != nullptr)
        p.trace[trace_index(static_cast<int>(blockIdx.x), p.trace_units, 0, word)] = v;
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
// tile leaves in sub-tiles of 128 bytes per row (64 fp16 or 32 fp32
// columns); each warp writes its 32 rows of a sub-tile into its own
// 128-byte-swizzled staging buffer and stores them with a 32-row TMA box (the
// C tensor map's box is 32 rows high).  The 16-byte chunk c of row r lands at
// chunk c ^ (r mod 8), the layout SWIZZLE_128B expects, which spreads each
// 8-thread phase of the st.shared.v4 over all 32 banks.

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

// Stage one output sub-tile held in registers (`v`: SUB_COLS fp32 values of
// output row `row` of the 128-row group, as raw bits) and TMA-store it at
// (col0, m0).  Each warp stages and stores its own 32 rows (row / 32 is the
// warp's quarter): it writes them into its own pair of 4 KB buffers (32 rows
// x 128 bytes, 128-byte swizzled) at `staging` + quarter * 8 KB, reconverges,
// and its lane 0 issues a 32-row TMA store and commits it as a bulk group.
// No thread outside the warp takes part, so the four warps of the group drain
// and store independently (one 128-row store behind a group barrier per
// sub-tile measured slower).  `sub_count` counts the sub-tiles this thread's
// warp has staged so far (it carries across tiles and selects the buffer); a
// buffer is rewritten only after the store issued from it two sub-tiles ago
// has finished reading it.  The store is skipped when `do_store` is false or
// the warp's rows start at or past M.
template <bool F16OUT>
__device__ __forceinline__ void stage_and_store(const uint32_t* v, uint32_t row,
                                                uint32_t staging, const CUtensorMap* tmap_c,
                                                int col0, int m0, int M, uint32_t& sub_count,
                                                bool do_store)
{
    const uint32_t quarter = row >> 5;
    const uint32_t r = row & 31u;
    const uint32_t buf = staging + quarter * (2u * WARP_STAGING_BYTES) +
                         (sub_count & 1u) * WARP_STAGING_BYTES;
    if (sub_count >= 2) {
        // the store issued two sub-tiles ago read this buffer
        if (r == 0) bulk_wait_group_read<1>();
        __syncwarp();
    }
    const uint32_t row_base = buf + r * 128u;
#pragma unroll
    for (uint32_t c = 0; c < 8; ++c) {
        const uint32_t dst = row_base + ((c ^ (r & 7u)) << 4);
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
    __syncwarp();
    const int wm0 = m0 + static_cast<int>(quarter * 32u);
    if (r == 0 && do_store && wm0 < M) {
        tma_store_2d(tmap_c, buf, col0, wm0);
        bulk_commit_group();
    }
    ++sub_count;
}

// A 32-column remainder of a tile whose width is not a whole number of
// 128-byte sub-tiles (fp16 output, widths 160 and 224): row `gm`, columns
// gn0..gn0+31, written straight from registers with 16-byte stores (N and
// the row are checked; N * 2 is a multiple of 16 bytes, so a chunk of 8
// halves is wholly inside or wholly outside the matrix).
__device__ __forceinline__ void direct_store_row32_f16(const uint32_t* v, void* C, int M, int N,
                                                       int gm, int gn0, bool do_store)
{
    if (!do_store || gm >= M) return;
    __half* crow = static_cast<__half*>(C) + static_cast<size_t>(gm) * N;
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        const int gn = gn0 + 8 * c;
        if (gn < N) {
            uint4 w;
            w.x = pack_half2(v[8 * c + 0], v[8 * c + 1]);
            w.y = pack_half2(v[8 * c + 2], v[8 * c + 3]);
            w.z = pack_half2(v[8 * c + 4], v[8 * c + 5]);
            w.w = pack_half2(v[8 * c + 6], v[8 * c + 7]);
            *reinterpret_cast<uint4*>(crow + gn) = w;
        }
    }
}

// The whole 128 x BLOCK_N accumulator at TMEM column `tmem_acc`, sub-tile by
// sub-tile: TMEM -> registers -> staging -> TMA store.
template <int BLOCK_N, bool F16OUT>
__device__ __forceinline__ void epilogue_tma_store(uint32_t tmem_acc, int q, uint32_t lane,
                                                   uint32_t staging, const CUtensorMap* tmap_c,
                                                   int m0, int n0, int M, int N,
                                                   uint32_t& sub_count, bool do_store,
                                                   void* C = nullptr)
{
    using S = EpilogueShape<BLOCK_N, F16OUT>;
    const uint32_t row = static_cast<uint32_t>(q) * 32u + lane;
    const uint32_t taddr = tmem_acc + (static_cast<uint32_t>(q * 32) << 16);
    if constexpr (BLOCK_N % S::SUB_COLS != 0) {
        static_assert(F16OUT && BLOCK_N % S::SUB_COLS == 32, "32-column remainder");
        const int tail = S::NUM_SUB * S::SUB_COLS;
        if (n0 + tail < N) {
            uint32_t v[32];
            tmem_load_32cols(taddr + tail, v);
            direct_store_row32_f16(v, C, M, N, m0 + static_cast<int>(row), n0 + tail, do_store);
        }
    }
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
        stage_and_store<F16OUT>(v, row, staging, tmap_c, col0, m0, M, sub_count, do_store);
    }
}

// ------------------------------------------------------ stream-K fix-up
//
// A tile of the stream-K part is accumulated by several workers, each over
// its own range of K blocks.  Every contributor writes its fp32 partial tile
// to its own workspace slot, publishes it (fence, then an arrival ticket on
// the tile's counter), and the contributor that draws the last ticket sums
// all partials in contributor order (0, 1, ..., in K order) and stores the
// tile.  The order of the sum never depends on which contributor arrives
// last, so results are identical run to run.  Slot layout: the value of
// (row r, column c) sits at float offset ((c / 4) * 128 + r) * 4 + c % 4, so a
// warp's 16-byte accesses to one column group cover 512 contiguous bytes.

// Fold this run's arrival into the tile's ticket word (epoch << 8 | count)
// and return the arrival rank; a word left by an earlier run starts over.
__device__ __forceinline__ uint32_t sk_take_ticket(unsigned* word, int epoch)
{
    const uint32_t ep = static_cast<uint32_t>(epoch) & 0xFFFFFFu;
    uint32_t cur = *reinterpret_cast<volatile unsigned*>(word);
    while (true) {
        const bool same = (cur >> 8) == ep;
        const uint32_t want = same ? cur + 1u : ((ep << 8) | 1u);
        const uint32_t prev = atomicCAS(word, cur, want);
        if (prev == cur) return same ? (cur & 0xFFu) : 0u;
        cur = prev;
    }
}

// Write this CTA's 128 x BLOCK_N accumulator to a partial slot (rows past the
// matrix are skipped).
template <int BLOCK_N>
__device__ __forceinline__ void sk_write_partial(uint32_t tmem_acc, int q, uint32_t lane,
                                                 float* slot, bool row_valid)
{
    const uint32_t row = static_cast<uint32_t>(q) * 32u + lane;
    const uint32_t taddr = tmem_acc + (static_cast<uint32_t>(q * 32) << 16);
#pragma unroll 1
    for (int j = 0; j < BLOCK_N / 32; ++j) {
        uint32_t v[32];
        tmem_load_32cols(taddr + j * 32, v);
        if (!row_valid) continue;
#pragma unroll
        for (int c = 0; c < 8; ++c) {
            float4* dst = reinterpret_cast<float4*>(slot) + (j * 8 + c) * 128 + row;
            *dst = make_float4(__uint_as_float(v[4 * c + 0]), __uint_as_float(v[4 * c + 1]),
                               __uint_as_float(v[4 * c + 2]), __uint_as_float(v[4 * c + 3]));
        }
    }
}

// Sum the `ncontrib` partial slots (slot0, slot0 + slot_stride, ...) in order
// and store the tile like epilogue_tma_store.  The loads of up to four
// contributors' 16-column groups are issued together before they are added
// (in contributor order), so each thread keeps 16 loads in flight instead of
// one contributor's worth.
template <int BLOCK_N, bool F16OUT>
__device__ __forceinline__ void sk_reduce_store(const float* slot0, size_t slot_stride,
                                                int ncontrib, int q, uint32_t lane,
                                                uint32_t staging, const CUtensorMap* tmap_c,
                                                int m0, int n0, int M, int N,
                                                uint32_t& sub_count, bool do_store,
                                                bool row_valid, void* C = nullptr)
{
    using S = EpilogueShape<BLOCK_N, F16OUT>;
    const uint32_t row = static_cast<uint32_t>(q) * 32u + lane;
    if constexpr (BLOCK_N % S::SUB_COLS != 0) {
        const int tail = S::NUM_SUB * S::SUB_COLS;
        if (n0 + tail < N && row_valid) {
            float acc[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) acc[i] = 0.0f;
            for (int cj = 0; cj < ncontrib; ++cj) {
                const float4* src = reinterpret_cast<const float4*>(slot0 + cj * slot_stride);
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    const float4 x = __ldcg(src + (tail / 4 + c) * 128 + row);
                    acc[4 * c + 0] += x.x;
                    acc[4 * c + 1] += x.y;
                    acc[4 * c + 2] += x.z;
                    acc[4 * c + 3] += x.w;
                }
            }
            direct_store_row32_f16(reinterpret_cast<const uint32_t*>(acc), C, M, N,
                                   m0 + static_cast<int>(row), n0 + tail, do_store);
        }
    }
#pragma unroll 1
    for (int j = 0; j < S::NUM_SUB; ++j) {
        const int col0 = n0 + j * S::SUB_COLS;
        if (col0 >= N) break;
        float acc[S::SUB_COLS];
#pragma unroll
        for (int i = 0; i < S::SUB_COLS; ++i) acc[i] = 0.0f;
        if (row_valid) {
#pragma unroll
            for (int g = 0; g < S::SUB_COLS / 16; ++g) {  // 16-column groups
                const int c4 = j * (S::SUB_COLS / 4) + g * 4;
#pragma unroll 1
                for (int cj0 = 0; cj0 < ncontrib; cj0 += 4) {
                    float4 x[4][4];
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        if (cj0 + u < ncontrib) {
                            const float4* src =
                                reinterpret_cast<const float4*>(slot0 + (cj0 + u) * slot_stride);
#pragma unroll
                            for (int c = 0; c < 4; ++c) x[u][c] = __ldcg(src + (c4 + c) * 128 + row);
                        }
                    }
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        if (cj0 + u < ncontrib) {
#pragma unroll
                            for (int c = 0; c < 4; ++c) {
                                acc[g * 16 + 4 * c + 0] += x[u][c].x;
                                acc[g * 16 + 4 * c + 1] += x[u][c].y;
                                acc[g * 16 + 4 * c + 2] += x[u][c].z;
                                acc[g * 16 + 4 * c + 3] += x[u][c].w;
                            }
                        }
                    }
                }
            }
        }
        stage_and_store<F16OUT>(reinterpret_cast<const uint32_t*>(acc), row, staging, tmap_c,
                                col0, m0, M, sub_count, do_store);
    }
}

// Epilogue of one stream-K unit for a 128-thread group: write the partial,
// release the accumulator (the caller's `release` callback, after the TMEM
// reads), publish, and if this is the last arrival, reduce and store.
// `ticket_smem` is a u32 in shared memory for broadcasting the ticket.
template <int BLOCK_N, bool F16OUT, typename Release>
__device__ __forceinline__ void sk_epilogue(uint32_t tmem_acc, int q, uint32_t lane, bool issuer,
                                            uint32_t staging, const CUtensorMap* tmap_c, int m0,
                                            int n0, int M, int N, uint32_t& sub_count,
                                            uint32_t bar_id, bool aborted, float* slot0,
                                            size_t slot_stride, int contrib, int ncontrib,
                                            unsigned* ticket_word, int epoch,
                                            volatile uint32_t* ticket_smem, Release release,
                                            void* C = nullptr)
{
    const uint32_t row = static_cast<uint32_t>(q) * 32u + lane;
    const bool row_valid = m0 + static_cast<int>(row) < M;
    sk_write_partial<BLOCK_N>(tmem_acc, q, lane, slot0 + contrib * slot_stride,
                              row_valid && !aborted);
    release();
    __threadfence();
    named_bar_sync(bar_id, 128);
    if (issuer) {
        uint32_t t = 0xFFFFFFFFu;  // "not last" when aborted
        if (!aborted) t = sk_take_ticket(ticket_word, epoch);
        __threadfence();
        *ticket_smem = t;
    }
    named_bar_sync(bar_id, 128);
    const uint32_t ticket = *ticket_smem;
    named_bar_sync(bar_id, 128);  // everyone has read the slot before it is reused
    if (ticket == static_cast<uint32_t>(ncontrib - 1)) {
        __threadfence();
        sk_reduce_store<BLOCK_N, F16OUT>(slot0, slot_stride, ncontrib, q, lane, staging, tmap_c,
                                         m0, n0, M, N, sub_count, !aborted, row_valid, C);
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
