// gemm_common.h -- definitions shared by the host runtime and the kernels:
// tile constants, the launch parameter block, the device status record, the
// persistent tile scheduler's raster and the 128-byte swizzle map.
#pragma once

#include <cstdint>

#ifdef __CUDACC__
#define TG_HD __host__ __device__ __forceinline__
#else
#define TG_HD inline
#endif

namespace tg {

// Output tile rows per CTA (one tcgen05.mma covers BLK_M x BLK_N x 16) and the
// K extent of one pipeline stage: 64 fp16 = one 128-byte swizzle row, the
// widest swizzle atom ("05 Async Data Movement - TMA", the 3-D TMA section:
// a 128-byte swizzle holds exactly 64 fp16 along the contiguous dimension).
constexpr int BLK_M = 128;
constexpr int BLK_K = 64;
constexpr int MMA_K = 16;
constexpr int MAX_STAGES = 8;
// Depth of the cluster-launch-control response ring: the producer requests
// the next tile when it starts a tile, while the epilogue still reads the
// tile before last, so up to three responses are live at once.
constexpr int CLC_SLOTS = 4;
constexpr int STAGING_BYTES = 128 * 128;  // one 128-row x 128-byte output sub-tile
constexpr int NUM_STAGING = 2;            // double-buffered output staging
// Each epilogue warp stages its own 32 rows: two buffers of 32 x 128 bytes per
// warp, the four warps' pairs side by side in the NUM_STAGING x STAGING_BYTES
// staging area.
constexpr uint32_t WARP_STAGING_BYTES = 32 * 128;
static_assert(4 * 2 * WARP_STAGING_BYTES == NUM_STAGING * STAGING_BYTES, "staging area");

// Bytes one pipeline stage receives: the A tile plus the B tile, in fp16
// ("GEMM II -- pipelining with TMA", Step 4, the byte_count formula).  The TMA
// engine delivers the whole box even where it hangs past the tensor's edge
// (the out-of-bounds part arrives zero-filled), so the count never shrinks
// for ragged tiles.
TG_HD uint32_t stage_tx_bytes(int block_n, int a_rows = BLK_M)
{
    return static_cast<uint32_t>((a_rows * BLK_K + block_n * BLK_K) * 2);
}

// Error codes written by a kernel to its status record (same values as the
// public gemm_status codes).
enum : int { DEV_OK = 0, DEV_TIMEOUT = 4 };

// Where a bounded wait gave up (recorded for diagnosis).
enum : int {
    WAIT_FULL = 1,        // consumer waiting for a stage's TMA bytes
    WAIT_EMPTY = 2,       // producer waiting for the MMA to free a stage
    WAIT_MMA = 3,         // waiting for an MMA batch to complete
    WAIT_TMEM_FULL = 4,   // epilogue waiting for an accumulator
    WAIT_TMEM_EMPTY = 5,  // MMA issuer waiting for the epilogue to drain TMEM
    WAIT_DRAIN = 6,       // teardown waiting for in-flight copies / MMAs
    WAIT_STALL = 7,       // the stall-test barrier that nothing completes
    WAIT_CLC_FULL = 8,    // waiting for a cluster-launch-control response
    WAIT_CLC_EMPTY = 9    // scheduler waiting for every reader of a response slot
};

// Device-side status record, one per plan (device memory, 32 bytes).
struct DevStatus {
    int code;         // first error code recorded (0 = none)
    int where;        // WAIT_* of the first timeout
    int block;        // blockIdx.x of the first timeout
    int tile;         // tile index being processed
    int kblock;       // k-block index being processed
    int abort_epoch;  // epoch of the most recent run that hit a timeout
    int pad[2];
};

struct Params {
    int M, N, K;
    int tiles_m, tiles_n, num_tiles, k_blocks;
    int group_m;     // raster group height (in M tiles)
    int pipe_depth;  // stages in the shared-memory ring (1..MAX_STAGES)
    const void* A;   // M x K fp16, row-major (used by the thread-copy variant)
    const void* B;   // N x K fp16, row-major (used by the thread-copy variant)
    void* C;         // M x N, row-major, fp16 or fp32 (used by plain-store epilogues)
    DevStatus* status;
    int epoch;                  // run counter, > 0
    unsigned long long budget_ns;  // bound on any single wait
    int debug_stall;            // 1: producer first waits on a barrier nothing completes
    // Stream-K tail (static persistent kernels).  The first dp_tiles tiles of the
    // raster order (a multiple of the worker count) are whole tiles; the last
    // sk_tiles tiles are cut into K-block ranges of sk_kb_per_worker blocks,
    // one range per worker.  sk_tiles = 0: every tile is whole.
    int dp_tiles;
    int sk_tiles;
    int sk_kb_per_worker;
    int sk_max_contrib;         // most workers that can share one tile; the
                                // dynamic pair schedule splits each of its
                                // sk_tiles last tiles into exactly this many
                                // K ranges (a split tail, see dynamic_unit)
    float* sk_partials;         // [sk_tiles][sk_max_contrib][halves][tile rows x cols] fp32
    unsigned* sk_tickets;       // [sk_tiles][halves] arrival tickets (epoch << 8 | count)
    // Optional timeline (warp-specialised kernels): per CTA a header record
    // and `trace_units` unit records of TRACE_WORDS 64-bit words (see
    // TRACE_* below); nullptr = off.
    unsigned long long* trace;
    int trace_units;
    // L2 eviction priority of the operand loads (warp-specialised kernels):
    // 0 = default, 1 = A evict_last / B evict_first, 2 = A evict_first /
    // B evict_last, 3 = both evict_last.
    int l2_policy;
    // Rows of A per stage in the single-CTA warp-specialised kernels (128, or
    // 64 when M <= 64; see a_slot_bytes).
    int a_rows;
    // 1: a persistent worker walks the K blocks of its odd-numbered units
    // backwards, so a unit starts on the operand slices its predecessor (the
    // previous wave, which shares the A rows within a raster group) touched
    // last and that are still in L2.  0: always ascending.
    int k_snake;
    // Dynamic tile schedule: which cluster computes a tile, and in which
    // position of its sequence, depends on timing.  So the K direction of
    // tile t is taken from the tile itself: descending when t / snake_span is
    // odd.  With snake_span equal to the static schedule's cluster count,
    // every tile walks K in the same direction under both schedules.
    int snake_span;
    // K blocks of 64 per pipeline stage in the warp-specialised kernels: 1,
    // 2 or (single-CTA kernel only) 4; a stage of K = 64 * ksub as that many
    // 128-byte swizzle atoms, one barrier round trip per 4 * ksub MMAs.  The
    // lock-step ladder kernels use 1.
    int ksub;
    // Dynamic pair schedule, narrow tail: the last `tail_halves` tiles are
    // each computed as two half-width tiles (see dynamic_unit); 0 = none.
    // Their B rows come through the kernel's second B tensor map, whose box
    // is half as high.
    int tail_halves;
};

// The i-th K block (i = 0, 1, ...) processed for work unit number `unit` of a
// worker, for a unit covering blocks [kb0, kb1).
TG_HD int kblock_at(int i, int unit, int kb0, int kb1, int k_snake)
{
    return (k_snake && (unit & 1)) ? kb1 - 1 - i : kb0 + i;
}

// Timeline record layout.  Header record of a CTA: TRACE_H_START (after
// set-up), TRACE_H_END (before teardown), TRACE_H_SMID, TRACE_H_UNITS (units
// processed).  Unit record: globaltimer stamps (ns) of the unit's milestones.
constexpr int TRACE_WORDS = 10;
enum : int {
    TRACE_H_START = 0, TRACE_H_END = 1, TRACE_H_SMID = 2, TRACE_H_UNITS = 3,
    TRACE_U_TILE = 0,        // (tile << 32) | number of K blocks
    TRACE_U_LOAD_FIRST = 1,  // producer: first stage of the unit issued
    TRACE_U_LOAD_LAST = 2,   // producer: last stage of the unit issued
    TRACE_U_ACC_FREE = 3,    // MMA issuer: accumulator free for this unit
    TRACE_U_MMA_FIRST = 4,   // MMA issuer: first stage landed, first MMA issued
    TRACE_U_MMA_LAST = 5,    // MMA issuer: last MMAs issued and committed
    TRACE_U_EPI_START = 6,   // epilogue: accumulator complete
    TRACE_U_EPI_END = 7,     // epilogue: last store of the unit issued
    TRACE_U_FULL_WAIT = 8,   // MMA issuer: ns spent waiting for loaded stages
    TRACE_U_EMPTY_WAIT = 9   // producer: ns spent waiting for free stages
};

TG_HD size_t trace_index(int cta, int trace_units, int record, int word)
{
    return (static_cast<size_t>(cta) * (trace_units + 1) + record) * TRACE_WORDS + word;
}

// One unit of a persistent worker's work: K blocks [kb0, kb1) of one output
// tile.  sk_index < 0: a whole tile of the data-parallel part; otherwise the
// tile's index inside the stream-K part, this worker's rank `contrib` among
// the `ncontrib` workers that share it (ranks follow the K order).
struct WorkUnit {
    int tile;
    int kb0, kb1;
    int sk_index;
    int contrib, ncontrib;
    int half;  // 0: the whole tile; 1, 2: its left or right half-width tile
};

// Work unit number u of the dynamic pair schedule (one cluster per unit).
// Units below dp are the whole tiles 0..dp-1.  With a split tail, the tiles
// dp, dp+1, ... of the partial last wave are each split into `splits` K
// ranges of the tile's KB stages, one unit per range (units dp + splits * i
// + c, c = 0..splits-1, for tile dp + i), so that the last wave has
// splits times as many, shorter units for the clusters it would leave idle.
//
// A narrow tail (splits == 0, tail tiles dp, dp+1, ...) computes each tail
// tile as two half-width tiles over the whole K instead: units dp + 2 * i + h
// are tile dp + i's left (h = 0) and right (h = 1) halves, so no partial sums
// need combining.
TG_HD void dynamic_unit(int u, int dp, int splits, int KB, WorkUnit& w)
{
    w.half = 0;
    if (u >= dp && splits == 0) {
        w.tile = dp + (u - dp) / 2;
        w.kb0 = 0;
        w.kb1 = KB;
        w.sk_index = -1;
        w.contrib = 0;
        w.ncontrib = 1;
        w.half = 1 + (u - dp) % 2;
        return;
    }
    if (u < dp || splits < 2) {
        w.tile = u;
        w.kb0 = 0;
        w.kb1 = KB;
        w.sk_index = -1;
        w.contrib = 0;
        w.ncontrib = 1;
        return;
    }
    const int v = u - dp;
    const int c = v % splits;
    w.tile = dp + v / splits;
    w.kb0 = (c * KB) / splits;
    w.kb1 = ((c + 1) * KB) / splits;
    w.sk_index = v / splits;
    w.contrib = c;
    w.ncontrib = splits;
}

// The sequence of work units of worker `w` out of `workers`: first the whole
// tiles w, w + workers, ... below dp_tiles, then the worker's contiguous range
// [w*L, (w+1)*L) of the stream-K part's K blocks, taken tile by tile in
// raster order (each tile's blocks in K order).  Every (tile, K block) pair is
// covered by exactly one unit of one worker.
struct WorkIter {
    int workers, dp_tiles, KB, L;
    int dp_next;
    int sk_pos, sk_end;

    TG_HD void init(int w, int nworkers, int dp, int sk, int k_blocks, int kb_per_worker)
    {
        workers = nworkers;
        dp_tiles = dp;
        KB = k_blocks;
        L = kb_per_worker;
        dp_next = w;
        const long long sk_kb = static_cast<long long>(sk) * k_blocks;
        const long long b = static_cast<long long>(w) * kb_per_worker;
        const long long e = b + kb_per_worker;
        sk_pos = static_cast<int>(sk > 0 && b < sk_kb ? b : 0);
        sk_end = static_cast<int>(sk > 0 && b < sk_kb ? (e < sk_kb ? e : sk_kb) : 0);
    }

    TG_HD bool next(WorkUnit& u)
    {
        if (dp_next < dp_tiles) {
            u.tile = dp_next;
            u.kb0 = 0;
            u.kb1 = KB;
            u.sk_index = -1;
            u.contrib = 0;
            u.ncontrib = 1;
            u.half = 0;
            dp_next += workers;
            return true;
        }
        if (sk_pos < sk_end) {
            const int t = sk_pos / KB;
            const int kb0 = sk_pos - t * KB;
            const int left = sk_end - sk_pos;
            const int kb1 = (KB - kb0) < left ? KB : kb0 + left;
            const int first = (t * KB) / L;
            const int last = ((t + 1) * KB - 1) / L;
            u.tile = dp_tiles + t;
            u.kb0 = kb0;
            u.kb1 = kb1;
            u.sk_index = t;
            u.contrib = (sk_pos / L) - first;
            u.ncontrib = last - first + 1;
            u.half = 0;
            sk_pos += kb1 - kb0;
            return true;
        }
        return false;
    }
};

// Grouped raster order of the output tiles ("GEMM II -- pipelining with TMA",
// Step 6, l2_group_size): walking the linear tile index t, `group_m`
// consecutive M-tiles are visited for one N-tile before moving to the next
// N-tile, so tiles handed out together share A row-bands and B column-bands
// in L2.  The last group may be shorter.  Defined for 0 <= t < tiles_m*tiles_n.
TG_HD void raster_tile(int t, int tiles_m, int tiles_n, int group_m, int& m_tile, int& n_tile)
{
    const int per_group = group_m * tiles_n;
    const int gid = t / per_group;
    const int m_first = gid * group_m;
    const int rows = (tiles_m - m_first) < group_m ? (tiles_m - m_first) : group_m;
    const int r = t - gid * per_group;
    m_tile = m_first + r % rows;
    n_tile = r / rows;
}

// Byte offset, inside a 1024-byte-aligned tile of 128-byte rows, of the byte
// at (row, byte_in_row) after the 128-byte swizzle: the 16-byte chunk index is
// XORed with the row's position inside its 8-row atom ("05 Async Data
// Movement - TMA", "How TMA Writes a Swizzled Layout": physical sector =
// logical sector XOR (row mod 8)).
TG_HD uint32_t sw128_offset(uint32_t row, uint32_t byte_in_row)
{
    const uint32_t chunk = (byte_in_row >> 4) & 7u;
    return row * 128u + (((chunk ^ (row & 7u)) << 4) | (byte_in_row & 15u));
}

// Shared-memory layout of one CTA (byte offsets from a 1024-byte-aligned
// base): `stages` A tiles (128 x 128 B), `stages` B tiles (block_n x 128 B),
// `staging` output sub-tile buffers, then the mbarriers and the TMEM address
// slot.  `total` includes 1024 bytes of slack for aligning the base.
struct SmemLayout {
    uint32_t a, b, staging, bars, total;
};

constexpr uint32_t A_TILE_BYTES = BLK_M * BLK_K * 2;  // 16 KB
constexpr uint32_t BAR_AREA_BYTES = 384;

TG_HD uint32_t b_tile_bytes(int block_n) { return static_cast<uint32_t>(block_n * BLK_K * 2); }

// `a_rows`: rows of A one stage holds (128, or 64 when the whole problem has at
// most 64 rows: the MMA still computes 128 rows, and rows 64..127 -- read from
// whatever follows the 64-row slot -- are never stored).
TG_HD uint32_t a_slot_bytes(int a_rows) { return static_cast<uint32_t>(a_rows * BLK_K * 2); }

TG_HD SmemLayout smem_layout(int stages, int block_n, int staging, int a_rows = BLK_M)
{
    SmemLayout L;
    L.a = 0;
    L.b = L.a + static_cast<uint32_t>(stages) * a_slot_bytes(a_rows);
    L.staging = L.b + static_cast<uint32_t>(stages) * b_tile_bytes(block_n);
    L.bars = L.staging + static_cast<uint32_t>(staging) * STAGING_BYTES;
    L.total = L.bars + BAR_AREA_BYTES + 1024;
    return L;
}

// Barrier slots (8-byte mbarriers) inside the barrier area.
enum : int {
    BAR_FULL = 0,                     // [MAX_STAGES]  stage filled by TMA
    BAR_EMPTY = BAR_FULL + MAX_STAGES,  // [MAX_STAGES]  stage released by the MMA
    BAR_TMEM_FULL = BAR_EMPTY + MAX_STAGES,  // [2] accumulator ready for the epilogue
    BAR_TMEM_EMPTY = BAR_TMEM_FULL + 2,      // [2] accumulator drained by the epilogue
    BAR_MMA = BAR_TMEM_EMPTY + 2,            // MMA batch complete (lock-step variants)
    BAR_DRAIN = BAR_MMA + 1,                 // teardown drain of in-flight MMAs
    BAR_STALL = BAR_DRAIN + 1,               // stall test: never completed
    BAR_CLC_FULL = BAR_STALL + 1,            // [CLC_SLOTS] cancellation response landed
    BAR_CLC_EMPTY = BAR_CLC_FULL + CLC_SLOTS,  // [CLC_SLOTS] every reader done (leader)
    BAR_COUNT = BAR_CLC_EMPTY + CLC_SLOTS
};
constexpr uint32_t TMEM_SLOT_OFFSET = BAR_COUNT * 8;     // u32 TMEM base address
constexpr uint32_t TICKET_SLOT_OFFSET = TMEM_SLOT_OFFSET + 4;  // u32 stream-K ticket broadcast
// Cluster-launch-control responses: CLC_SLOTS opaque 16-byte records, 16-byte
// aligned (the barrier area starts on a 1024-byte boundary).
constexpr uint32_t CLC_RESP_OFFSET = 256;
constexpr uint32_t CLC_RESP_BYTES = 16;
static_assert(TICKET_SLOT_OFFSET + 4 <= CLC_RESP_OFFSET, "barrier area too small");
static_assert(CLC_RESP_OFFSET + CLC_SLOTS * CLC_RESP_BYTES <= BAR_AREA_BYTES,
              "barrier area too small for the response ring");

}  // namespace tg
