// api.cu -- host runtime behind the C ABI (include/tmagemm.h): argument
// checks, configuration choice, TMA tensor-map encoding, the device status
// record and the kernel launch.  Control crosses to the device only at the
// launch inside gemm_run.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>
#include <vector>

#include "../../include/tmagemm.h"
#include "gemm_common.h"
#include "launch.h"

using namespace tg;

namespace tg {

namespace {
std::mutex g_smem_mutex;
std::vector<std::pair<const void*, unsigned>> g_smem_limits;
}  // namespace

bool smem_limit_known(const void* kernel, unsigned bytes)
{
    std::lock_guard<std::mutex> lock(g_smem_mutex);
    for (const auto& kv : g_smem_limits)
        if (kv.first == kernel) return bytes <= kv.second;
    return false;
}

void smem_limit_record(const void* kernel, unsigned bytes)
{
    std::lock_guard<std::mutex> lock(g_smem_mutex);
    for (auto& kv : g_smem_limits)
        if (kv.first == kernel) {
            if (bytes > kv.second) kv.second = bytes;
            return;
        }
    g_smem_limits.emplace_back(kernel, bytes);
}

}  // namespace tg

namespace {

thread_local std::string g_err;
thread_local int g_status = GEMM_OK;

int fail(int status, const std::string& msg)
{
    g_status = status;
    g_err = msg;
    return status;
}

int ok()
{
    g_status = GEMM_OK;
    g_err.clear();
    return GEMM_OK;
}

int cuda_fail(const char* what, cudaError_t e)
{
    return fail(GEMM_ERR_CUDA, std::string(what) + ": " + cudaGetErrorName(e) + " (" +
                                   cudaGetErrorString(e) + ")");
}

const char* variant_name(int v)
{
    switch (v) {
    case VAR_SYNC_TILED: return "sync_tiled";
    case VAR_TMA_SERIAL: return "tma_serial";
    case VAR_PIPELINED: return "pipelined";
    case VAR_WS_PIPELINED: return "ws_pipelined";
    case VAR_PERSISTENT: return "persistent";
    case VAR_PERSISTENT_LOCKSTEP: return "persistent_lockstep";
    case VAR_PERSISTENT_2CTA: return "persistent_2cta";
    case VAR_DYNAMIC_2CTA: return "dynamic_2cta";
    default: return "?";
    }
}

bool is_ws(int v)
{
    return v == VAR_WS_PIPELINED || v == VAR_PERSISTENT || v == VAR_PERSISTENT_2CTA ||
           v == VAR_DYNAMIC_2CTA;
}
// One resident CTA per SM that takes tile after tile (statically or by
// cancelling clusters that have not started).
bool is_persistent(int v)
{
    return v == VAR_PERSISTENT || v == VAR_PERSISTENT_LOCKSTEP || v == VAR_PERSISTENT_2CTA ||
           v == VAR_DYNAMIC_2CTA;
}
// 256-row tiles computed by CTA pairs (cta_group::2).
bool is_pair(int v)
{
    return v == VAR_PERSISTENT_2CTA || v == VAR_DYNAMIC_2CTA;
}
// One cluster per work unit, clusters cancelling those not started yet.
bool is_dynamic(int v) { return v == VAR_DYNAMIC_2CTA; }
bool has_ring(int v) { return v != VAR_SYNC_TILED && v != VAR_TMA_SERIAL; }

int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

// Work units one full set of resident clusters takes at a time: the dynamic
// schedule flips a unit's K direction every snake_span units.
int snake_span_of(const gemm_config& c, int sms)
{
    return std::max(1, std::min(sms / 2, c.num_tiles));
}

// Fraction of launched tile slots that do work when `tiles` tiles run in
// waves over `sms` SMs.
double wave_efficiency(int64_t tiles, int sms)
{
    const int64_t waves = ceil_div(tiles, sms);
    return static_cast<double>(tiles) / static_cast<double>(waves * sms);
}

int choose_block_n(int variant, int64_t M, int64_t N, int sms)
{
    if (!is_persistent(variant) && variant != VAR_WS_PIPELINED) return 128;
    const int64_t tm = ceil_div(M, BLK_M);
    if (tm * ceil_div(N, 256) >= sms) return 256;
    // Few tiles: trade tile width (operand reuse per tile) against filling
    // the SMs.  Relative per-tile efficiency of narrower tiles is an estimate.
    const int cand[3] = {256, 128, 64};
    const double tile_eff[3] = {1.0, 0.95, 0.85};
    int best = 256;
    double best_score = -1.0;
    for (int i = 0; i < 3; ++i) {
        const double s = wave_efficiency(tm * ceil_div(N, cand[i]), sms) * tile_eff[i];
        if (s > best_score + 1e-9) {
            best_score = s;
            best = cand[i];
        }
    }
    return best;
}

// Pair tile widths the CTA-pair kernel is built for: multiples of 32 (fp32
// output stores 32-column sub-tiles; fp16 output 64-column sub-tiles plus a
// directly stored 32-column remainder for widths 160 and 224).
bool pair_width_ok(int bn)
{
    // fp16 widths of 160 / 224 store their last 32 columns directly
    return bn == 128 || bn == 160 || bn == 192 || bn == 224 || bn == 256;
}

// Pair tile width for an automatic plan: the fraction of launched tile slots
// that do useful columns (waves over the SM pairs, and the last tile column's
// overhang past N), weighted by the throughput of one tile of each width
// relative to 256 columns, measured on GB300 at 8192^3 and 4096^3 with the
// wave and overhang losses divided out (narrower tiles issue more barrier
// round trips and load more operand bytes per FLOP).  Stages of two K blocks
// (ksub = 2) halve the round trips, and narrow tiles lose less.
int choose_pair_bn(int64_t M, int64_t N, int sms, int ksub)
{
    const int widths[5] = {256, 224, 192, 160, 128};
    const double eff_k64[5] = {1.0, 0.92, 0.79, 0.73, 0.54};
    const double eff_k128[5] = {1.0, 0.94, 0.89, 0.81, 0.70};
    const double* tile_eff = ksub == 2 ? eff_k128 : eff_k64;
    const int64_t slots = sms / 2;
    const int64_t tm = ceil_div(M, 2 * BLK_M);
    int best = 256;
    double best_score = -1.0;
    for (int i = 0; i < 5; ++i) {
        const int bn = widths[i];
        const int64_t tn = ceil_div(N, bn);
        const double cols = static_cast<double>(N) / static_cast<double>(tn * bn);
        const double score = wave_efficiency(tm * tn, static_cast<int>(slots)) * cols * tile_eff[i];
        if (score > best_score + 1e-9) {
            best_score = score;
            best = bn;
        }
    }
    return best;
}

// Default kernel: CTA pairs (256-row tiles, cta_group::2) when M spans more
// than one 128-row tile and there are enough pair tiles (at the narrowest
// width, 128) to occupy every TPC; otherwise single-CTA persistent tiles,
// whose narrower widths keep more SMs busy on small or skinny problems.
// Pairs take the dynamic schedule (cluster launch control) unless the options
// ask for something only the static one has (a grid size, stream-K): measured
// on GB300 it runs each tile about 5 % faster at 8192^3 (the clusters no
// longer start every tile in lock-step) and gives bit-identical results.
int auto_variant(int64_t M, int64_t N, int sms, const gemm_options& opts)
{
    const int64_t pair_tiles = ceil_div(M, 2 * BLK_M) * ceil_div(N, 128);
    if (M > BLK_M && pair_tiles >= sms / 2)
        return (opts.grid == 0 && opts.stream_k != 2) ? VAR_DYNAMIC_2CTA : VAR_PERSISTENT_2CTA;
    return VAR_PERSISTENT;
}

int select_config_impl(int64_t M, int64_t N, int64_t K, int dtype, const gemm_options* o,
                       int sms, int smem_optin, gemm_config* c)
{
    gemm_options opts;
    std::memset(&opts, 0, sizeof(opts));
    if (o) opts = *o;
    if (!c) return fail(GEMM_ERR_INVALID_ARG, "config output pointer is NULL");
    const int64_t LIM = (int64_t(1) << 31) - 1;
    if (M < 1 || N < 1 || K < 1 || M > LIM || N > LIM || K > LIM)
        return fail(GEMM_ERR_INVALID_ARG, "M, N, K must be in [1, 2^31-1]");
    if (dtype != GEMM_OUT_F32 && dtype != GEMM_OUT_F16)
        return fail(GEMM_ERR_INVALID_ARG, "dtype_out must be GEMM_OUT_F32 (0) or GEMM_OUT_F16 (1)");
    if (K % 8 != 0)
        return fail(GEMM_ERR_UNSUPPORTED,
                    "K must be a multiple of 8: the TMA row stride of A and B (K*2 bytes) must be a multiple of 16 bytes");
    const int elt = dtype == GEMM_OUT_F16 ? 2 : 4;
    if ((N * elt) % 16 != 0)
        return fail(GEMM_ERR_UNSUPPORTED,
                    "N * sizeof(output) must be a multiple of 16 bytes (TMA row stride of C)");
    if (opts.variant < 0 || opts.variant > VAR_DYNAMIC_2CTA)
        return fail(GEMM_ERR_INVALID_ARG, "unknown variant");
    if (opts.pipe_depth < 0 || opts.pipe_depth > MAX_STAGES)
        return fail(GEMM_ERR_INVALID_ARG, "pipe_depth must be 0 (auto) or 1..8");
    const bool pair_requested = is_pair(opts.variant);
    if (!pair_requested && opts.block_n != 0 && opts.block_n != 64 && opts.block_n != 128 &&
        opts.block_n != 256)
        return fail(GEMM_ERR_INVALID_ARG, "block_n must be 0 (auto), 64, 128 or 256");
    if (opts.group_m < 0 || opts.grid < 0 || opts.wait_budget_ms < 0)
        return fail(GEMM_ERR_INVALID_ARG, "group_m, grid and wait_budget_ms must be >= 0");
    if (opts.stream_k < 0 || opts.stream_k > 2)
        return fail(GEMM_ERR_INVALID_ARG, "stream_k must be 0 (auto), 1 (off) or 2 (on)");
    if (opts.l2_policy < 0 || opts.l2_policy > 3)
        return fail(GEMM_ERR_INVALID_ARG, "l2_policy must be 0..3");
    if (opts.block_k != 0 && opts.block_k != 64 && opts.block_k != 128 && opts.block_k != 256)
        return fail(GEMM_ERR_INVALID_ARG, "block_k must be 0 (auto), 64, 128 or 256");
    if (opts.k_order < 0 || opts.k_order > 2)
        return fail(GEMM_ERR_INVALID_ARG, "k_order must be 0 (auto), 1 (ascending) or 2 (snake)");
    if (sms < 1 || smem_optin < 1) return fail(GEMM_ERR_INVALID_ARG, "bad device limits");

    const int variant = opts.variant == VAR_AUTO ? auto_variant(M, N, sms, opts) : opts.variant;
    if (opts.debug_stall && !is_ws(variant))
        return fail(GEMM_ERR_INVALID_ARG, "debug_stall needs a warp-specialised variant");
    if (is_dynamic(variant) && opts.grid != 0)
        return fail(GEMM_ERR_INVALID_ARG,
                    "the dynamic variant launches one cluster per work unit: grid must be 0 (auto)");
    // the single-CTA warp-specialised kernel
    const bool single_ws = variant == VAR_PERSISTENT || variant == VAR_WS_PIPELINED;
    if (opts.block_k == 128 && !is_pair(variant) && !single_ws)
        return fail(GEMM_ERR_INVALID_ARG,
                    "block_k = 128 is built for the warp-specialised variants");
    if (opts.block_k == 256 && !single_ws)
        return fail(GEMM_ERR_INVALID_ARG,
                    "block_k = 256 is built for the single-CTA warp-specialised variants");
    // A problem of at most 64 rows keeps 64-row A slots (more stages fit).
    const int a_rows = (M <= 64 && single_ws) ? 64 : BLK_M;
    // K blocks of 64 per stage (two 128-byte swizzle atoms at block_k = 128).
    // Automatic for CTA pairs whose operand rows are 128-byte aligned (K a
    // multiple of 64), unless an explicit ring depth is asked for (a depth
    // sweep is a sweep of 64-wide stages).  Stream-K then splits K in units
    // of these stages.  Measured on GB300, 3
    // stages of 64 KB against 6 of 32 KB: 8192^3 1808 vs 1690 TFLOP/s, 4096^3
    // 1600 vs 1357, 4000x3000x4992 1484 vs 1296 (dynamic schedule).  With
    // rows that start off a 128-byte line (K = 5000, 5064) every box row
    // straddles two lines and the wider stages lose: 1128-1143 vs 1162-1178.
    const bool auto_k128 =
        opts.block_k == 0 && is_pair(variant) && opts.pipe_depth == 0 && K % 64 == 0;
    // Stages of 2 or 4 K blocks are also built for the single-CTA kernel but
    // not chosen automatically.  A read-only stream of the skinny shape's B
    // (16384 x 16384) in the GEMM's pattern measured 5.60 TB/s with 128-byte
    // pieces per row and stage, 5.99 with 256-byte and 6.12 with 512-byte
    // pieces (192 KB of ring each); but the GEMM's ring holds only 128 KB of
    // B beside A's slots and the output staging, and each stage stays taken
    // until its MMAs commit, so 64 x 16384 x 16384 measured 100.3 / 99.3 /
    // 100.3 us with stages of 1 / 2 / 4 blocks.
    const int ksub = opts.block_k == 256                   ? 4
                     : (opts.block_k == 128 || auto_k128) ? 2
                                                          : 1;
    if (is_pair(variant) && opts.block_n != 0 && !pair_width_ok(opts.block_n))
        return fail(GEMM_ERR_INVALID_ARG,
                    "CTA-pair tile width (block_n) must be 128, 160, 192, 224 or 256");
    const int bn = opts.block_n   ? opts.block_n
                   : is_pair(variant) ? choose_pair_bn(M, N, sms, ksub)
                                      : choose_block_n(variant, M, N, sms);
    // Shared memory per CTA holds B tiles of `bn_cta` rows: a CTA of a pair
    // keeps half of the pair tile's B rows.
    const int bn_cta = is_pair(variant) ? bn / 2 : bn;
    const int bm = is_pair(variant) ? 2 * BLK_M : BLK_M;
    const int staging = variant == VAR_SYNC_TILED ? 0 : NUM_STAGING;

    int depth;
    if (!has_ring(variant)) {
        if (opts.pipe_depth > 1)
            return fail(GEMM_ERR_INVALID_ARG, "this variant has a single stage (pipe_depth 0 or 1)");
        depth = 1;
    } else if (opts.pipe_depth) {
        depth = opts.pipe_depth;
        const uint32_t need = smem_layout(depth * ksub, bn_cta, staging, a_rows).total;
        if (need > static_cast<uint32_t>(smem_optin)) {
            char buf[200];
            std::snprintf(buf, sizeof(buf),
                          "pipe_depth %d with a %dx%d tile does not fit: %u bytes of shared memory > %d available",
                          depth, bm, bn, need, smem_optin);
            return fail(GEMM_ERR_UNSUPPORTED, buf);
        }
    } else {
        depth = 0;
        for (int d = MAX_STAGES; d >= 1; --d)
            if (smem_layout(d * ksub, bn_cta, staging, a_rows).total <=
                static_cast<uint32_t>(smem_optin)) {
                depth = d;
                break;
            }
        if (depth == 0) return fail(GEMM_ERR_UNSUPPORTED, "no stage count fits shared memory");
    }

    const int64_t tm = ceil_div(M, bm), tn = ceil_div(N, bn);
    const int64_t tiles = tm * tn;
    if (tiles > LIM) return fail(GEMM_ERR_UNSUPPORTED, "too many output tiles");
    uint32_t smem = smem_layout(depth * ksub, bn_cta, staging, a_rows).total;
    if (is_persistent(variant)) {
        // One resident CTA per SM: ask for more than half of the SM's shared
        // memory so that a second CTA can never be co-scheduled.
        const uint32_t half = static_cast<uint32_t>(smem_optin) / 2u + 1024u;
        if (smem < half) smem = half;
        if (smem > static_cast<uint32_t>(smem_optin)) smem = static_cast<uint32_t>(smem_optin);
    }

    std::memset(c, 0, sizeof(*c));
    c->variant = variant;
    c->block_m = bm;
    c->block_n = bn;
    c->block_k = BLK_K * ksub;
    c->pipe_depth = depth;
    // Raster group height in tiles: 16 tile rows of 256 for CTA pairs
    // (measured back to back against 8: 8192^3 1870 vs 1862, 4096^3 1752 vs
    // 1725, 6144^3 1844 vs 1827 TFLOP/s, 4000x3000x5000 unchanged), 8 rows of
    // 128 for single CTAs.
    c->group_m = opts.group_m ? opts.group_m : (is_pair(variant) ? 16 : 8);
    c->tiles_m = static_cast<int>(tm);
    c->tiles_n = static_cast<int>(tn);
    c->num_tiles = static_cast<int>(tiles);
    c->k_blocks = static_cast<int>(ceil_div(K, BLK_K));
    // Stream-K (persistent warp-specialised variants) decides whether a grid
    // larger than the tile count pays: the extra workers share the K blocks.
    // stream-K splits K in units of pipeline stages (ksub K blocks of 64)
    const int64_t KBLK = ceil_div(ceil_div(K, BLK_K), ksub);
    auto stream_k_worth = [&](int64_t T, int64_t workers) {
        const int64_t rem = T % workers;
        if (rem == 0 || opts.stream_k == 1) return false;
        const int64_t sk = T >= workers ? rem : T;
        const int64_t L = ceil_div(sk * KBLK, workers);
        const int64_t maxc = ceil_div(KBLK, L) + 1;
        if (maxc > 255 || sk * KBLK >= LIM) return false;
        // Only on request: on this power-capped part the idle SMs of a
        // partial last wave let the busy ones clock higher, and spreading the
        // tail over every SM measured slower than leaving it data-parallel for
        // the 4096^3, 8192^3 and 4000x3000x5000 workloads.
        (void)L;
        return opts.stream_k == 2;
    };
    const bool sk_capable = variant == VAR_PERSISTENT || variant == VAR_PERSISTENT_2CTA;
    if (is_dynamic(variant)) {
        // one cluster per pair tile; running clusters cancel the rest
        if (2 * tiles > LIM) return fail(GEMM_ERR_UNSUPPORTED, "too many output tiles");
        c->grid = static_cast<int>(2 * tiles);
    } else if (is_pair(variant)) {
        // clusters of two CTAs, one pair tile per cluster at a time
        int64_t pairs = (opts.grid ? opts.grid : sms) / 2;
        if (pairs < 1) pairs = 1;
        if (pairs > tiles && !stream_k_worth(tiles, pairs)) pairs = tiles;
        c->grid = static_cast<int>(2 * pairs);
    } else if (is_persistent(variant)) {
        int64_t g = opts.grid ? opts.grid : sms;
        if (g > tiles && !(sk_capable && stream_k_worth(tiles, g))) g = tiles;
        c->grid = static_cast<int>(g);
    } else {
        c->grid = static_cast<int>(tiles);
    }
    c->threads = is_ws(variant) ? 192 : 128;
    c->smem_bytes = static_cast<int>(smem);
    {
        int cols = (variant == VAR_PERSISTENT || is_pair(variant)) ? 2 * bn : bn;
        int alloc = 32;
        while (alloc < cols) alloc <<= 1;
        c->tmem_cols = alloc;
    }
    c->tx_bytes = static_cast<int>(is_pair(variant) ? 2 * stage_tx_bytes(bn_cta) * ksub
                                                    : stage_tx_bytes(bn, a_rows) * ksub);
    c->a_rows = a_rows;

    // Stream-K tail: whole waves stay data-parallel; the tiles of a partial
    // last wave are cut into equal K-block ranges, one per worker.
    c->dp_tiles = c->num_tiles;
    if (sk_capable) {
        const int64_t workers = is_pair(variant) ? c->grid / 2 : c->grid;
        const int64_t T = c->num_tiles, KB = KBLK;  // stages per tile
        if (stream_k_worth(T, workers)) {
            const int64_t sk = T >= workers ? T % workers : T;
            const int64_t L = ceil_div(sk * KB, workers);
            const int64_t maxc = ceil_div(KB, L) + 1;
            {
                const int halves = is_pair(variant) ? 2 : 1;
                c->dp_tiles = static_cast<int>(T - sk);
                c->sk_tiles = static_cast<int>(sk);
                c->sk_kb_per_worker = static_cast<int>(L);
                c->sk_max_contrib = static_cast<int>(maxc);
                // one fp32 slot of BLK_M x (tile columns) per contributor and
                // CTA, then one ticket word per tile and CTA
                c->workspace_bytes =
                    sk * maxc * halves * static_cast<long long>(BLK_M) * bn * 4 +
                    ((sk * halves * 4 + 255) / 256) * 256;
            }
        }
    }
    // Narrow tiles for a single partial wave (automatic).  When all the tiles
    // fit in at most half the resident clusters, each is computed as two
    // 256 x 128 tiles, one per cluster, over the whole K: twice as many
    // clusters work and nothing needs summing.  A 128-wide tile of the pair
    // kernel runs at 0.70 of a 256-wide tile's throughput (stages of K = 128),
    // so the wave takes about 0.71 of a tile time instead of 1 (measured:
    // 1024 x 1024 x 4096, 16 tiles, 429 vs 414 TFLOP/s).  Applied to the
    // partial last wave of a longer run (8192^3: 36 tiles after 13 waves) it
    // gave nothing (1878 vs 1883): clusters reach the last wave at times
    // spread over half a tile, so the wave is no shorter.
    if (variant == VAR_DYNAMIC_2CTA && opts.stream_k == 0 && bn == 256 && ksub == 2) {
        const int64_t cl = sms / 2;
        const int64_t T = c->num_tiles;
        if (2 * T <= cl) {  // every tile as two units: 2 T clusters of 2 CTAs
            c->tail_halves = static_cast<int>(T);
            c->grid = static_cast<int>(4 * T);
        }
    }
    // Split tail of the dynamic pair schedule (stream_k = 2).  The tiles of a
    // partial last wave -- all of them when there are fewer tiles than
    // resident clusters -- are each cut into S equal K ranges, S =
    // floor(clusters / those tiles) up to 4, so the clusters that would idle
    // share them; every range keeps at least 4 stages.  The two to four
    // partial tiles meet in the workspace and the last one to arrive sums them
    // in K order and stores the tile.  Opt-in: measured on GB300 the fp32
    // partial round trip through the workspace (latency-bound with four
    // warps per CTA) costs what the shorter wave saves, or more.
    if (variant == VAR_DYNAMIC_2CTA && opts.stream_k == 2) {
        const int64_t cl = sms / 2;
        const int64_t T = c->num_tiles;
        const int64_t rem = T % cl;
        int64_t S = rem ? cl / rem : 0;
        if (S > 4) S = 4;
        while (S >= 2 && KBLK / S < 4) --S;
        if (S >= 2) {
            const int64_t units = T - rem + S * rem;
            if (2 * units > LIM) return fail(GEMM_ERR_UNSUPPORTED, "too many output tiles");
            c->grid = static_cast<int>(2 * units);
            c->dp_tiles = static_cast<int>(T - rem);
            c->sk_tiles = static_cast<int>(rem);
            c->sk_kb_per_worker = 0;
            c->sk_max_contrib = static_cast<int>(S);
            c->workspace_bytes = rem * S * 2 * static_cast<long long>(BLK_M) * bn * 4 +
                                 ((rem * 2 * 4 + 255) / 256) * 256;
        }
    }
    return ok();
}

PFN_cuTensorMapEncodeTiled_v12000 get_encode_fn()
{
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

// 2-D tensor map over a row-major matrix with `rows` rows of `cols` elements
// (row pitch `pitch_bytes`), box = box_cols x box_rows, 128-byte swizzle,
// out-of-bounds elements read as zero.
//
// L2 promotion: 256 bytes when every row starts on a 256-byte boundary (a box
// row of 128 bytes then sits in one 256-byte block, and the promotion brings
// in the row's next K block, which the next stage reads); 128 bytes when rows
// start off such a boundary (there a 256-byte promotion fetches bytes of
// neighbouring blocks that no box asks for).  Measured on GB300: K = 8192
// 1799 vs 1742 TFLOP/s with 256 over 128 bytes; K = 5000 (10,000-byte rows)
// 1222 vs 1174 with 128 over 256 bytes.
int encode_2d(CUtensorMap* map, CUtensorMapDataType dt, const void* base, uint64_t cols,
              uint64_t rows, uint64_t pitch_bytes, uint32_t box_cols, uint32_t box_rows,
              const char* what)
{
    PFN_cuTensorMapEncodeTiled_v12000 enc = get_encode_fn();
    if (!enc) return fail(GEMM_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
    const cuuint64_t dims[2] = {cols, rows};
    const cuuint64_t strides[1] = {pitch_bytes};
    const cuuint32_t box[2] = {box_cols, box_rows};
    const cuuint32_t estr[2] = {1, 1};
    const bool rows_on_256 =
        pitch_bytes % 256 == 0 && reinterpret_cast<uintptr_t>(base) % 256 == 0;
    const CUtensorMapL2promotion promo = rows_on_256
                                             ? CU_TENSOR_MAP_L2_PROMOTION_L2_256B
                                             : CU_TENSOR_MAP_L2_PROMOTION_L2_128B;
    CUresult r = enc(map, dt, 2, const_cast<void*>(base), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, promo,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
        char buf[160];
        std::snprintf(buf, sizeof(buf), "cuTensorMapEncodeTiled(%s) failed with CUresult %d", what,
                      static_cast<int>(r));
        return fail(GEMM_ERR_CUDA, buf);
    }
    return GEMM_OK;
}

}  // namespace

struct gemm_plan {
    int64_t M, N, K;
    int dtype;
    gemm_config cfg;
    int device;
    unsigned long long budget_ns;
    int debug_stall;
    int l2_policy;
    int k_snake;
    int snake_span;  // dynamic schedule: see Params::snake_span
    DevStatus* d_status;
    int epoch;
    // tensor maps for the last (A, B, C) triple
    const void* mapA_ptr;
    const void* mapB_ptr;
    const void* mapC_ptr;
    CUtensorMap tmA, tmB, tmC;
    CUtensorMap tmB2;  // B with half-height boxes, for the narrow tail
    // stream-K workspace: partial tiles, then the ticket words
    void* d_workspace;
    // optional timeline buffer (caller-owned device memory)
    unsigned long long* trace;
    int trace_units;
    // device buffers of gemm_run_host
    void* hA;
    void* hB;
    void* hC;
    // banded host round trip (gemm_run_host with page-locked buffers): one
    // sub-plan per band of rows, copy streams and their events
    gemm_options opts;
    std::vector<gemm_plan*> bands;
    int band_rows;
    cudaStream_t s_in, s_out;
    std::vector<cudaEvent_t> ev_in, ev_done;
    cudaEvent_t ev_start, ev_out;
    std::string desc;
};

extern "C" {

int gemm_select_config(int64_t M, int64_t N, int64_t K, int dtype_out, const gemm_options* opts,
                       int sm_count, int smem_optin, gemm_config* out)
{
    return select_config_impl(M, N, K, dtype_out, opts, sm_count, smem_optin, out);
}

gemm_plan* gemm_create_plan_ex(int64_t M, int64_t N, int64_t K, int dtype_out,
                               const gemm_options* opts)
{
    // Shape/option errors are reported before touching the device.
    gemm_config probe;
    if (select_config_impl(M, N, K, dtype_out, opts, 148, 232448, &probe) != GEMM_OK)
        return nullptr;

    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) {
        fail(GEMM_ERR_NO_DEVICE, std::string("no CUDA device: ") + cudaGetErrorString(e));
        return nullptr;
    }
    int major = 0, minor = 0, sms = 0, smem_optin = 0;
    cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
    cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    e = cudaDeviceGetAttribute(&smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    if (e != cudaSuccess) {
        cuda_fail("cudaDeviceGetAttribute", e);
        return nullptr;
    }
    if (major != 10 || minor != 3) {
        char buf[160];
        std::snprintf(buf, sizeof(buf),
                      "device %d is sm_%d%d; this library is built for sm_103a (GB300) only", dev,
                      major, minor);
        fail(GEMM_ERR_NO_DEVICE, buf);
        return nullptr;
    }
    gemm_plan* p = new gemm_plan();
    p->M = M;
    p->N = N;
    p->K = K;
    p->dtype = dtype_out;
    p->device = dev;
    if (select_config_impl(M, N, K, dtype_out, opts, sms, smem_optin, &p->cfg) != GEMM_OK) {
        delete p;
        return nullptr;
    }
    if (opts) p->opts = *opts;
    const int budget_ms = (opts && opts->wait_budget_ms) ? opts->wait_budget_ms : 2000;
    p->budget_ns = static_cast<unsigned long long>(budget_ms) * 1000000ull;
    p->debug_stall = opts ? opts->debug_stall : 0;
    p->l2_policy = opts ? opts->l2_policy : 0;
    // K snake by default: every other tile of a persistent CTA walks K
    // downwards (measured: 14 % less DRAM traffic at 8192^3, L2 hit rate
    // 73 % -> 80 %).
    p->k_snake = (opts && opts->k_order == 1) ? 0 : 1;
    // The dynamic schedule takes each tile's K direction from the tile index,
    // as the static schedule of a full grid (SM count / 2 clusters) would.
    p->snake_span = snake_span_of(p->cfg, sms);
    e = cudaMalloc(&p->d_status, sizeof(DevStatus));
    if (e == cudaSuccess) e = cudaMemset(p->d_status, 0, sizeof(DevStatus));
    if (e == cudaSuccess && p->cfg.workspace_bytes > 0) {
        e = cudaMalloc(&p->d_workspace, static_cast<size_t>(p->cfg.workspace_bytes));
        if (e == cudaSuccess)
            e = cudaMemset(p->d_workspace, 0, static_cast<size_t>(p->cfg.workspace_bytes));
    }
    if (e != cudaSuccess) {
        cuda_fail("allocating the device status record / stream-K workspace", e);
        if (p->d_status) cudaFree(p->d_status);
        if (p->d_workspace) cudaFree(p->d_workspace);
        delete p;
        return nullptr;
    }
    char buf[320];
    const gemm_config& c = p->cfg;
    std::snprintf(buf, sizeof(buf),
                  "variant=%s tile=%dx%dx%d pipe_depth=%d smem=%d grid=%d threads=%d tiles=%d (%dx%d) "
                  "k_blocks=%d tmem_cols=%d group_m=%d out=%s stream_k=%d/%d(L=%d) tail_halves=%d",
                  variant_name(c.variant), c.block_m, c.block_n, c.block_k, c.pipe_depth,
                  c.smem_bytes, c.grid, c.threads, c.num_tiles, c.tiles_m, c.tiles_n, c.k_blocks,
                  c.tmem_cols, c.group_m, dtype_out == GEMM_OUT_F16 ? "f16" : "f32", c.sk_tiles,
                  c.num_tiles, c.sk_kb_per_worker, c.tail_halves);
    p->desc = buf;
    ok();
    return p;
}

gemm_plan* gemm_create_plan(int64_t M, int64_t N, int64_t K, int dtype_out)
{
    return gemm_create_plan_ex(M, N, K, dtype_out, nullptr);
}

int gemm_run(gemm_plan* plan, const void* A, const void* B, void* C, void* cuda_stream)
{
    if (!plan) return fail(GEMM_ERR_INVALID_ARG, "plan is NULL");
    if (!A || !B || !C) return fail(GEMM_ERR_INVALID_ARG, "A, B and C must be non-NULL");
    if ((reinterpret_cast<uintptr_t>(A) | reinterpret_cast<uintptr_t>(B) |
         reinterpret_cast<uintptr_t>(C)) & 15u)
        return fail(GEMM_ERR_UNSUPPORTED, "A, B and C must be 16-byte aligned (TMA)");
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail("cudaGetDevice", e);
    if (dev != plan->device)
        return fail(GEMM_ERR_INVALID_ARG, "plan was created on another device");
    // Arrival tickets of split tiles are keyed by the run counter, which a
    // graph replay repeats: a replayed ticket word would never rank a last
    // arrival, and the shared tiles would stay unwritten.  A captured launch
    // of the dynamic schedule therefore runs every tile whole; a static
    // stream-K plan refuses capture.
    bool whole_tiles = false;
    if (plan->cfg.sk_tiles > 0) {
        cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
        if (cudaStreamIsCapturing(static_cast<cudaStream_t>(cuda_stream), &cs) == cudaSuccess &&
            cs != cudaStreamCaptureStatusNone) {
            if (!is_dynamic(plan->cfg.variant))
                return fail(GEMM_ERR_UNSUPPORTED,
                            "a plan with stream-K tiles cannot be captured into a CUDA graph");
            whole_tiles = true;
        }
    }

    const gemm_config& c = plan->cfg;
    if (A != plan->mapA_ptr || B != plan->mapB_ptr || C != plan->mapC_ptr) {
        int r = encode_2d(&plan->tmA, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, A, plan->K, plan->M,
                          plan->K * 2, BLK_K, static_cast<uint32_t>(c.a_rows), "A");
        if (r == GEMM_OK)
            r = encode_2d(&plan->tmB, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, B, plan->K, plan->N,
                          plan->K * 2, BLK_K, is_pair(c.variant) ? c.block_n / 2 : c.block_n,
                          "B");
        if (r == GEMM_OK && c.tail_halves > 0)
            r = encode_2d(&plan->tmB2, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, B, plan->K, plan->N,
                          plan->K * 2, BLK_K, static_cast<uint32_t>(c.block_n / 4), "B (narrow)");
        if (r == GEMM_OK) {
            if (plan->dtype == GEMM_OUT_F16)
                r = encode_2d(&plan->tmC, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, C, plan->N, plan->M,
                              plan->N * 2, 64, 32, "C");
            else
                r = encode_2d(&plan->tmC, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, C, plan->N, plan->M,
                              plan->N * 4, 32, 32, "C");
        }
        if (r != GEMM_OK) {
            plan->mapA_ptr = plan->mapB_ptr = plan->mapC_ptr = nullptr;
            return r;
        }
        plan->mapA_ptr = A;
        plan->mapB_ptr = B;
        plan->mapC_ptr = C;
    }

    LaunchSpec s{};  // every field not set below is zero (trace and stream-K off)
    s.variant = c.variant;
    s.block_n = c.block_n;
    s.f16out = plan->dtype == GEMM_OUT_F16;
    s.grid = c.grid;
    s.threads = c.threads;
    s.smem_bytes = static_cast<unsigned>(c.smem_bytes);
    s.tmA = &plan->tmA;
    s.tmB = &plan->tmB;
    s.tmC = &plan->tmC;
    s.tmB2 = c.tail_halves > 0 ? &plan->tmB2 : nullptr;
    Params& p = s.p;
    p.M = static_cast<int>(plan->M);
    p.N = static_cast<int>(plan->N);
    p.K = static_cast<int>(plan->K);
    p.tiles_m = c.tiles_m;
    p.tiles_n = c.tiles_n;
    p.num_tiles = c.num_tiles;
    p.k_blocks = c.k_blocks;
    p.group_m = c.group_m;
    p.pipe_depth = c.pipe_depth;
    p.A = A;
    p.B = B;
    p.C = C;
    p.status = plan->d_status;
    if (++plan->epoch <= 0) plan->epoch = 1;
    p.epoch = plan->epoch;
    p.budget_ns = plan->budget_ns;
    p.debug_stall = plan->debug_stall;
    p.l2_policy = plan->l2_policy;
    p.k_snake = plan->k_snake;
    p.snake_span = plan->snake_span;
    p.ksub = c.block_k / BLK_K;
    p.a_rows = c.a_rows;
    p.dp_tiles = c.dp_tiles;
    p.sk_tiles = c.sk_tiles;
    p.sk_kb_per_worker = c.sk_kb_per_worker;
    p.sk_max_contrib = c.sk_max_contrib;
    p.tail_halves = c.tail_halves;
    p.trace = plan->trace;
    p.trace_units = plan->trace_units;
    if (whole_tiles) {
        s.grid = 2 * c.num_tiles;
        p.dp_tiles = c.num_tiles;
        p.sk_tiles = 0;
        p.sk_max_contrib = 1;
    }
    if (p.sk_tiles > 0) {
        const int halves = is_pair(c.variant) ? 2 : 1;
        const size_t partial_bytes = static_cast<size_t>(c.sk_tiles) * c.sk_max_contrib * halves *
                                     BLK_M * c.block_n * 4;
        p.sk_partials = static_cast<float*>(plan->d_workspace);
        p.sk_tickets = reinterpret_cast<unsigned*>(static_cast<char*>(plan->d_workspace) +
                                                   partial_bytes);
    } else {
        p.sk_partials = nullptr;
        p.sk_tickets = nullptr;
    }

    cudaStream_t stream = static_cast<cudaStream_t>(cuda_stream);
    e = is_pair(c.variant) ? launch_pair(s, stream)
        : is_ws(c.variant) ? launch_ws(s, stream)
                           : launch_ladder(s, stream);
    if (e != cudaSuccess) return cuda_fail("kernel launch", e);
    return ok();
}

int gemm_get_device_status(gemm_plan* plan)
{
    if (!plan) return fail(GEMM_ERR_INVALID_ARG, "plan is NULL");
    DevStatus st;
    cudaError_t e = cudaMemcpy(&st, plan->d_status, sizeof(st), cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return cuda_fail("reading the device status record", e);
    if (st.code == DEV_OK) return ok();
    DevStatus zero;
    std::memset(&zero, 0, sizeof(zero));
    zero.abort_epoch = st.abort_epoch;  // keep: a stale epoch never matches a new run
    cudaMemcpy(plan->d_status, &zero, sizeof(zero), cudaMemcpyHostToDevice);
    char buf[200];
    std::snprintf(buf, sizeof(buf),
                  "kernel wait timed out (where=%d block=%d tile=%d k_block=%d); the run was abandoned",
                  st.where, st.block, st.tile, st.kblock);
    return fail(st.code == DEV_TIMEOUT ? GEMM_ERR_TIMEOUT : GEMM_ERR_CUDA, buf);
}

namespace {

bool host_pinned(const void* p)
{
    cudaPointerAttributes a;
    if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    return a.type == cudaMemoryTypeHost;
}

// Rows per band of the banded host round trip: about eight bands of whole
// 256-row pair tiles, none smaller than 512 rows; 0 = do not band.
int host_band_rows(int64_t M)
{
    if (M < 2048) return 0;
    int64_t rows = ((M + 7) / 8 + 255) / 256 * 256;
    if (rows < 512) rows = 512;
    return rows < M ? static_cast<int>(rows) : 0;
}

// Sub-plans, streams and events of the banded round trip (created once).
int prepare_bands(gemm_plan* plan)
{
    const int rows = host_band_rows(plan->M);
    if (rows == 0) return GEMM_ERR_UNSUPPORTED;
    if (!plan->bands.empty() && plan->band_rows == rows) return GEMM_OK;
    const int64_t nb = (plan->M + rows - 1) / rows;
    std::vector<gemm_plan*> bands;
    for (int64_t i = 0; i < nb; ++i) {
        const int64_t m = (i + 1 < nb) ? rows : plan->M - i * rows;
        gemm_plan* b = gemm_create_plan_ex(m, plan->N, plan->K, plan->dtype, &plan->opts);
        if (!b) {
            for (gemm_plan* x : bands) gemm_destroy(x);
            return gemm_last_status();
        }
        bands.push_back(b);
    }
    cudaError_t e = cudaSuccess;
    if (!plan->s_in) e = cudaStreamCreateWithFlags(&plan->s_in, cudaStreamNonBlocking);
    if (e == cudaSuccess && !plan->s_out)
        e = cudaStreamCreateWithFlags(&plan->s_out, cudaStreamNonBlocking);
    if (e == cudaSuccess && !plan->ev_start)
        e = cudaEventCreateWithFlags(&plan->ev_start, cudaEventDisableTiming);
    if (e == cudaSuccess && !plan->ev_out)
        e = cudaEventCreateWithFlags(&plan->ev_out, cudaEventDisableTiming);
    while (e == cudaSuccess && plan->ev_in.size() < bands.size()) {
        cudaEvent_t a = nullptr, b = nullptr;
        e = cudaEventCreateWithFlags(&a, cudaEventDisableTiming);
        if (e == cudaSuccess) e = cudaEventCreateWithFlags(&b, cudaEventDisableTiming);
        if (a) plan->ev_in.push_back(a);
        if (b) plan->ev_done.push_back(b);
    }
    if (e != cudaSuccess) {
        for (gemm_plan* x : bands) gemm_destroy(x);
        return cuda_fail("creating streams / events for the banded host round trip", e);
    }
    for (gemm_plan* x : plan->bands) gemm_destroy(x);
    plan->bands = bands;
    plan->band_rows = rows;
    return GEMM_OK;
}

}  // namespace

int gemm_run_host(gemm_plan* plan, const void* A, const void* B, void* C, void* cuda_stream)
{
    if (!plan) return fail(GEMM_ERR_INVALID_ARG, "plan is NULL");
    if (!A || !B || !C) return fail(GEMM_ERR_INVALID_ARG, "A, B and C must be non-NULL");
    const size_t eltC = plan->dtype == GEMM_OUT_F16 ? 2 : 4;
    const size_t bytesA = static_cast<size_t>(plan->M) * plan->K * 2;
    const size_t bytesB = static_cast<size_t>(plan->N) * plan->K * 2;
    const size_t bytesC = static_cast<size_t>(plan->M) * plan->N * eltC;
    cudaError_t e = cudaSuccess;
    if (!plan->hA) e = cudaMalloc(&plan->hA, bytesA);
    if (e == cudaSuccess && !plan->hB) e = cudaMalloc(&plan->hB, bytesB);
    if (e == cudaSuccess && !plan->hC) e = cudaMalloc(&plan->hC, bytesC);
    if (e != cudaSuccess) return cuda_fail("allocating device buffers for gemm_run_host", e);
    cudaStream_t stream = static_cast<cudaStream_t>(cuda_stream);

    // Banded pipeline (page-locked buffers only, else copies cannot overlap):
    // B goes in first, then A band by band on one copy stream; the band GEMMs
    // run on the caller's stream as their A band lands; each band of C goes
    // back on a second copy stream as soon as its GEMM is done.
    const bool banded = host_pinned(A) && host_pinned(B) && host_pinned(C) &&
                        prepare_bands(plan) == GEMM_OK;
    if (banded) {
        const size_t nb = plan->bands.size();
        const size_t rows = static_cast<size_t>(plan->band_rows);
        e = cudaEventRecord(plan->ev_start, stream);
        if (e == cudaSuccess) e = cudaStreamWaitEvent(plan->s_in, plan->ev_start, 0);
        if (e == cudaSuccess) e = cudaStreamWaitEvent(plan->s_out, plan->ev_start, 0);
        if (e == cudaSuccess)
            e = cudaMemcpyAsync(plan->hB, B, bytesB, cudaMemcpyHostToDevice, plan->s_in);
        for (size_t i = 0; e == cudaSuccess && i < nb; ++i) {
            const size_t r0 = i * rows;
            const size_t m = (i + 1 < nb) ? rows : static_cast<size_t>(plan->M) - r0;
            const size_t offA = r0 * static_cast<size_t>(plan->K) * 2;
            e = cudaMemcpyAsync(static_cast<char*>(plan->hA) + offA,
                                static_cast<const char*>(A) + offA,
                                m * static_cast<size_t>(plan->K) * 2, cudaMemcpyHostToDevice,
                                plan->s_in);
            if (e == cudaSuccess) e = cudaEventRecord(plan->ev_in[i], plan->s_in);
        }
        if (e != cudaSuccess) return cuda_fail("banded host-to-device copies", e);
        for (size_t i = 0; i < nb; ++i) {
            const size_t r0 = i * rows;
            e = cudaStreamWaitEvent(stream, plan->ev_in[i], 0);
            if (e != cudaSuccess) return cuda_fail("cudaStreamWaitEvent", e);
            const size_t offA = r0 * static_cast<size_t>(plan->K) * 2;
            const size_t offC = r0 * static_cast<size_t>(plan->N) * eltC;
            int r = gemm_run(plan->bands[i], static_cast<char*>(plan->hA) + offA, plan->hB,
                             static_cast<char*>(plan->hC) + offC, cuda_stream);
            if (r != GEMM_OK) return r;
            e = cudaEventRecord(plan->ev_done[i], stream);
            if (e == cudaSuccess) e = cudaStreamWaitEvent(plan->s_out, plan->ev_done[i], 0);
            const size_t m = (i + 1 < nb) ? rows : static_cast<size_t>(plan->M) - r0;
            if (e == cudaSuccess)
                e = cudaMemcpyAsync(static_cast<char*>(C) + offC,
                                    static_cast<char*>(plan->hC) + offC,
                                    m * static_cast<size_t>(plan->N) * eltC,
                                    cudaMemcpyDeviceToHost, plan->s_out);
            if (e != cudaSuccess) return cuda_fail("banded device-to-host copy", e);
        }
        e = cudaEventRecord(plan->ev_out, plan->s_out);
        if (e == cudaSuccess) e = cudaStreamWaitEvent(stream, plan->ev_out, 0);
        if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
        if (e != cudaSuccess) return cuda_fail("cudaStreamSynchronize", e);
        int status = GEMM_OK;
        for (gemm_plan* b : plan->bands) {
            const int r = gemm_get_device_status(b);
            if (r != GEMM_OK && status == GEMM_OK) status = r;
        }
        return status == GEMM_OK ? ok() : fail(status, "a band of the host round trip failed");
    }

    e = cudaMemcpyAsync(plan->hA, A, bytesA, cudaMemcpyHostToDevice, stream);
    if (e == cudaSuccess) e = cudaMemcpyAsync(plan->hB, B, bytesB, cudaMemcpyHostToDevice, stream);
    if (e != cudaSuccess) return cuda_fail("host-to-device copy", e);
    int r = gemm_run(plan, plan->hA, plan->hB, plan->hC, cuda_stream);
    if (r != GEMM_OK) return r;
    e = cudaMemcpyAsync(C, plan->hC, bytesC, cudaMemcpyDeviceToHost, stream);
    if (e != cudaSuccess) return cuda_fail("device-to-host copy", e);
    e = cudaStreamSynchronize(stream);
    if (e != cudaSuccess) return cuda_fail("cudaStreamSynchronize", e);
    return gemm_get_device_status(plan);
}

void gemm_destroy(gemm_plan* plan)
{
    if (!plan) return;
    if (plan->d_status) cudaFree(plan->d_status);
    if (plan->d_workspace) cudaFree(plan->d_workspace);
    if (plan->hA) cudaFree(plan->hA);
    if (plan->hB) cudaFree(plan->hB);
    if (plan->hC) cudaFree(plan->hC);
    for (gemm_plan* b : plan->bands) gemm_destroy(b);
    for (cudaEvent_t ev : plan->ev_in) cudaEventDestroy(ev);
    for (cudaEvent_t ev : plan->ev_done) cudaEventDestroy(ev);
    if (plan->ev_start) cudaEventDestroy(plan->ev_start);
    if (plan->ev_out) cudaEventDestroy(plan->ev_out);
    if (plan->s_in) cudaStreamDestroy(plan->s_in);
    if (plan->s_out) cudaStreamDestroy(plan->s_out);
    delete plan;
}

const char* gemm_last_error(void) { return g_err.c_str(); }

int gemm_last_status(void) { return g_status; }

const char* gemm_plan_describe(const gemm_plan* plan)
{
    return plan ? plan->desc.c_str() : "(null plan)";
}

int gemm_plan_config(const gemm_plan* plan, gemm_config* out)
{
    if (!plan || !out) return fail(GEMM_ERR_INVALID_ARG, "plan or out is NULL");
    *out = plan->cfg;
    return ok();
}

int gemm_schedule_tile(const gemm_config* cfg, int64_t tile, int* m_tile, int* n_tile)
{
    if (!cfg || !m_tile || !n_tile) return fail(GEMM_ERR_INVALID_ARG, "NULL argument");
    if (tile < 0 || tile >= cfg->num_tiles || cfg->group_m < 1)
        return fail(GEMM_ERR_INVALID_ARG, "tile index out of range");
    raster_tile(static_cast<int>(tile), cfg->tiles_m, cfg->tiles_n, cfg->group_m, *m_tile,
                *n_tile);
    return ok();
}

int gemm_set_trace(gemm_plan* plan, void* device_buffer, int units_per_cta)
{
    if (!plan) return fail(GEMM_ERR_INVALID_ARG, "plan is NULL");
    if (device_buffer && units_per_cta < 1)
        return fail(GEMM_ERR_INVALID_ARG, "units_per_cta must be >= 1");
    if (device_buffer && (reinterpret_cast<uintptr_t>(device_buffer) & 7u))
        return fail(GEMM_ERR_INVALID_ARG, "trace buffer must be 8-byte aligned");
    if (device_buffer && plan->cfg.variant != VAR_PERSISTENT && !is_pair(plan->cfg.variant) &&
        plan->cfg.variant != VAR_WS_PIPELINED)
        return fail(GEMM_ERR_UNSUPPORTED, "the timeline is recorded by the warp-specialised variants");
    plan->trace = static_cast<unsigned long long*>(device_buffer);
    plan->trace_units = device_buffer ? units_per_cta : 0;
    return ok();
}

int gemm_schedule_unit(const gemm_config* cfg, int worker, int index, int* tile, int* kb0,
                       int* kb1, int* contrib, int* ncontrib)
{
    if (!cfg || !tile || !kb0 || !kb1 || !contrib || !ncontrib || index < 0)
        return fail(GEMM_ERR_INVALID_ARG, "NULL argument or negative index");
    // workers: clusters (CTA pairs) or CTAs
    const int workers = is_pair(cfg->variant) ? cfg->grid / 2 : cfg->grid;
    if (worker < 0 || worker >= workers) return fail(GEMM_ERR_INVALID_ARG, "worker out of range");
    // the kernels count K in pipeline stages of `ks` K blocks; report blocks
    const int ks = cfg->block_k > BLK_K ? cfg->block_k / BLK_K : 1;
    const int stages = (cfg->k_blocks + ks - 1) / ks;
    const int dp = cfg->dp_tiles;
    if (is_dynamic(cfg->variant)) {
        // the cluster's own unit; the rest is decided while the kernel runs
        if (index > 0) {
            ok();
            return 0;
        }
        WorkUnit u;
        if (cfg->tail_halves > 0)
            dynamic_unit(worker, cfg->num_tiles - cfg->tail_halves, 0, stages, u);
        else
            dynamic_unit(worker, dp, cfg->sk_tiles > 0 ? cfg->sk_max_contrib : 1, stages, u);
        *tile = u.tile;
        *kb0 = u.kb0 * ks;
        *kb1 = u.kb1 * ks < cfg->k_blocks ? u.kb1 * ks : cfg->k_blocks;
        *contrib = u.contrib;
        *ncontrib = u.ncontrib;
        ok();
        return 1;
    }
    WorkIter it;
    it.init(worker, workers, dp, cfg->sk_tiles, stages, cfg->sk_kb_per_worker);
    WorkUnit u;
    for (int i = 0; it.next(u); ++i) {
        if (i == index) {
            *tile = u.tile;
            *kb0 = u.kb0 * ks;
            *kb1 = u.kb1 * ks < cfg->k_blocks ? u.kb1 * ks : cfg->k_blocks;
            *contrib = u.contrib;
            *ncontrib = u.ncontrib;
            ok();
            return 1;
        }
    }
    ok();
    return 0;
}

int64_t gemm_sw128_offset(int64_t row, int64_t byte_in_row)
{
    if (row < 0 || byte_in_row < 0 || byte_in_row >= 128) return -1;
    return static_cast<int64_t>(sw128_offset(static_cast<uint32_t>(row),
                                             static_cast<uint32_t>(byte_in_row)));
}

}  // extern "C"

// ---------------------------------------------------------------------------
// Allocation-free entry point.
//
// Some callers cannot call cudaMalloc: applications whose device memory is
// owned entirely by a framework's caching allocator or a pre-reserved arena
// (a foreign cudaMalloc either fails for lack of memory or is forbidden by
// policy), and latency-critical serving loops that cannot afford the device
// synchronisation cudaMalloc/cudaFree imply.  gemm_create_plan allocates the
// plan's device status record, so those callers use gemm_run_noalloc instead.
// It runs the kernel an automatic plan would (automatic plans never use
// stream-K, the only option that needs a workspace); the kernel's only
// scratch memory, the status record, lives in the file-scope array below,
// which every GPU that loads this library holds until the process exits.

namespace {

constexpr size_t NOALLOC_SCRATCH_BYTES = 256;  // stated maximum scratch size
static_assert(sizeof(DevStatus) <= NOALLOC_SCRATCH_BYTES, "status record must fit");

constexpr int NOALLOC_MAX_DEVICES = 64;
std::mutex g_noalloc_mutex;
void* g_noalloc_ptr[NOALLOC_MAX_DEVICES] = {};
unsigned long long g_noalloc_ctx[NOALLOC_MAX_DEVICES] = {};  // context the address belongs to
int g_noalloc_epoch[NOALLOC_MAX_DEVICES] = {};

// Unique id of the calling thread's current CUDA context, or 0 when there is
// none or the driver cannot say.  A context created after cudaDeviceReset
// gets a new id, so an address looked up in the old one is never reused.
unsigned long long current_context_id()
{
    static PFN_cuCtxGetCurrent_v4000 get_current = nullptr;
    static PFN_cuCtxGetId_v12000 get_id = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 4000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(f);
        f = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &f, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(f);
    });
    CUcontext ctx = nullptr;
    if (!get_current || !get_id || get_current(&ctx) != CUDA_SUCCESS || !ctx) return 0;
    unsigned long long id = 0;
    if (get_id(ctx, &id) != CUDA_SUCCESS) return 0;
    return id;
}

}  // namespace

// Shared by every gemm_run_noalloc call on a device; keeps the last call's
// contents.  Host code must not pass this name to a kernel: on the host it is
// a stand-in symbol, not a device address (see noalloc_scratch_ptr).
static __device__ __align__(256) unsigned char g_noalloc_scratch[NOALLOC_SCRATCH_BYTES];

namespace {

// Device address of g_noalloc_scratch on device `dev` (which is current),
// looked up with cudaGetSymbolAddress once per device and again whenever the
// current context is not the one the cached address was looked up in (a
// cudaDeviceReset by the caller, or a context of the caller's own).
int noalloc_scratch_ptr(int dev, void** out)
{
    if (dev < 0 || dev >= NOALLOC_MAX_DEVICES)
        return fail(GEMM_ERR_UNSUPPORTED, "device index too large for gemm_run_noalloc");
    std::lock_guard<std::mutex> lock(g_noalloc_mutex);
    const unsigned long long ctx = current_context_id();
    if (!g_noalloc_ptr[dev] || ctx == 0 || ctx != g_noalloc_ctx[dev]) {
        void* p = nullptr;
        cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess || !p)
            return cuda_fail("cudaGetSymbolAddress(g_noalloc_scratch)", e);
        g_noalloc_ptr[dev] = p;
        // the lookup has made the device's context current if none was
        g_noalloc_ctx[dev] = current_context_id();
    }
    *out = g_noalloc_ptr[dev];
    return GEMM_OK;
}

}  // namespace

extern "C" int gemm_run_noalloc(int64_t M, int64_t N, int64_t K, int dtype_out, const void* A,
                                const void* B, void* C, void* cuda_stream, int* device_status)
{
    if (device_status) *device_status = GEMM_OK;
    if (!A || !B || !C) return fail(GEMM_ERR_INVALID_ARG, "A, B and C must be non-NULL");
    if ((reinterpret_cast<uintptr_t>(A) | reinterpret_cast<uintptr_t>(B) |
         reinterpret_cast<uintptr_t>(C)) & 15u)
        return fail(GEMM_ERR_UNSUPPORTED, "A, B and C must be 16-byte aligned (TMA)");
    const size_t scratch_needed = sizeof(DevStatus);
    if (scratch_needed > NOALLOC_SCRATCH_BYTES) {
        char buf[160];
        std::snprintf(buf, sizeof(buf),
                      "gemm_run_noalloc needs %zu bytes of scratch; its static array holds %zu",
                      scratch_needed, NOALLOC_SCRATCH_BYTES);
        return fail(GEMM_ERR_UNSUPPORTED, buf);
    }
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return fail(GEMM_ERR_NO_DEVICE, std::string("no CUDA device: ") +
                                                              cudaGetErrorString(e));
    int major = 0, minor = 0, sms = 0, smem_optin = 0;
    cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
    cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    e = cudaDeviceGetAttribute(&smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    if (e != cudaSuccess) return cuda_fail("cudaDeviceGetAttribute", e);
    if (major != 10 || minor != 3)
        return fail(GEMM_ERR_NO_DEVICE, "this library is built for sm_103a (GB300) only");

    gemm_config c;
    int r = select_config_impl(M, N, K, dtype_out, nullptr, sms, smem_optin, &c);
    if (r != GEMM_OK) return r;
    // automatic plans never split K: no workspace
    if (c.sk_tiles != 0 || c.workspace_bytes != 0)
        return fail(GEMM_ERR_UNSUPPORTED, "gemm_run_noalloc: the automatic plan needs a workspace");

    void* scratch = nullptr;
    r = noalloc_scratch_ptr(dev, &scratch);
    if (r != GEMM_OK) return r;

    CUtensorMap tmA, tmB, tmC, tmB2;
    r = encode_2d(&tmA, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, A, K, M, K * 2, BLK_K,
                  static_cast<uint32_t>(c.a_rows), "A");
    if (r == GEMM_OK)
        r = encode_2d(&tmB, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, B, K, N, K * 2, BLK_K,
                      static_cast<uint32_t>(is_pair(c.variant) ? c.block_n / 2 : c.block_n), "B");
    if (r == GEMM_OK && c.tail_halves > 0)
        r = encode_2d(&tmB2, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, B, K, N, K * 2, BLK_K,
                      static_cast<uint32_t>(c.block_n / 4), "B (narrow)");
    if (r == GEMM_OK) {
        if (dtype_out == GEMM_OUT_F16)
            r = encode_2d(&tmC, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, C, N, M, N * 2, 64, 32, "C");
        else
            r = encode_2d(&tmC, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, C, N, M, N * 4, 32, 32, "C");
    }
    if (r != GEMM_OK) return r;

    cudaStream_t stream = static_cast<cudaStream_t>(cuda_stream);
    // The status record must start at zero for this call.
    e = cudaMemsetAsync(scratch, 0, sizeof(DevStatus), stream);
    if (e != cudaSuccess) return cuda_fail("clearing the scratch status record", e);

    LaunchSpec s{};  // every field not set below is zero (trace and stream-K off)
    s.variant = c.variant;
    s.block_n = c.block_n;
    s.f16out = dtype_out == GEMM_OUT_F16;
    s.grid = c.grid;
    s.threads = c.threads;
    s.smem_bytes = static_cast<unsigned>(c.smem_bytes);
    s.tmA = &tmA;
    s.tmB = &tmB;
    s.tmC = &tmC;
    s.tmB2 = c.tail_halves > 0 ? &tmB2 : nullptr;
    Params& p = s.p;
    p.M = static_cast<int>(M);
    p.N = static_cast<int>(N);
    p.K = static_cast<int>(K);
    p.tiles_m = c.tiles_m;
    p.tiles_n = c.tiles_n;
    p.num_tiles = c.num_tiles;
    p.k_blocks = c.k_blocks;
    p.group_m = c.group_m;
    p.pipe_depth = c.pipe_depth;
    p.A = A;
    p.B = B;
    p.C = C;
    p.status = static_cast<DevStatus*>(scratch);
    {
        std::lock_guard<std::mutex> lock(g_noalloc_mutex);
        if (++g_noalloc_epoch[dev] <= 0) g_noalloc_epoch[dev] = 1;
        p.epoch = g_noalloc_epoch[dev];
    }
    p.budget_ns = 2000ull * 1000000ull;
    p.debug_stall = 0;
    p.dp_tiles = c.dp_tiles;
    p.tail_halves = c.tail_halves;
    p.sk_tiles = 0;
    p.sk_kb_per_worker = 0;
    p.sk_max_contrib = 0;
    p.sk_partials = nullptr;
    p.sk_tickets = nullptr;
    p.a_rows = c.a_rows;
    p.k_snake = 1;
    p.snake_span = snake_span_of(c, sms);
    p.ksub = c.block_k / BLK_K;
    e = is_pair(c.variant) ? launch_pair(s, stream) : launch_ws(s, stream);
    if (e != cudaSuccess) return cuda_fail("kernel launch", e);

    if (device_status) {
        e = cudaStreamSynchronize(stream);
        if (e != cudaSuccess) return cuda_fail("cudaStreamSynchronize", e);
        DevStatus st;
        e = cudaMemcpy(&st, scratch, sizeof(st), cudaMemcpyDeviceToHost);
        if (e != cudaSuccess) return cuda_fail("reading the scratch status record", e);
        *device_status = st.code == DEV_OK ? GEMM_OK : GEMM_ERR_TIMEOUT;
        if (st.code != DEV_OK)
            return fail(GEMM_ERR_TIMEOUT, "kernel wait timed out; the run was abandoned");
    }
    return ok();
}
