/* ringsim.h -- host-side model of the stage-ring protocols (C ABI).
 *
 * A discrete-event model of the load/compute handshake that the GEMM kernels
 * implement with mbarriers, TMA copies and tcgen05 MMAs.  It serves two
 * purposes:
 *
 * 1. Protocol checking.  mbarriers are modelled with an arrival count, a
 *    pending transaction-byte count and a completed-phase counter ("05 Async
 *    Data Movement - TMA", How to Wait for a TMA Load: a phase completes only
 *    after both the arrivals and the pending bytes reach zero; a wait on
 *    parity p returns once the phase of parity p has completed).  Stage slots
 *    and accumulators carry the identity and landed byte count of what they
 *    hold, so that a read of bytes that have not landed or of a stale round,
 *    and a write over data still being read, are detected.  Faults of the
 *    kinds the pages warn about can be injected: a wrong byte budget, a budget
 *    announced several times, a missed phase flip, phases reset to 0 at every
 *    persistent tile, a refill issued before the MMA reading the slot is done,
 *    an epilogue that does not wait for its accumulator.  The model reports
 *    deadlock (nothing can progress and nothing is in flight) or the first
 *    hazard.
 *
 * 2. Timing.  With a fixed load time per copy and a fixed MMA time per stage
 *    ("GEMM II -- pipelining with TMA", the interactive pipeline Gantt: serial
 *    vs prefetch, PIPE_DEPTH, K tiles, load : MMA cost) it reports the
 *    makespan, the tensor-pipe idle fraction, whether the MMAs run back to
 *    back and the most loads in flight.
 *
 * Protocols:
 *   RINGSIM_LOCKSTEP   one thread per CTA: prologue loads of the first
 *                      PIPE_DEPTH stages, then per K block wait(tma_bar[s]),
 *                      MMA, wait(mma_bar), refill slot s with block k + D
 *                      ("GEMM II", Step 5; depth 1 is Step 4's serial loop),
 *                      per-stage TMA barriers and one MMA barrier, the TMA
 *                      phase flipped when the ring wraps and the MMA phase
 *                      every iteration.
 *   RINGSIM_WARP_SPEC  the warp-specialised kernels of this library: a
 *                      producer (wait empty[s], arrive.expect_tx(full[s]),
 *                      two copies), an MMA issuer (wait full[s], MMA,
 *                      commit -> empty[s]; at the end of a tile commit ->
 *                      tmem_full[a]) and an epilogue (wait tmem_full[a], read,
 *                      arrive tmem_empty[a]) with `accumulators` TMEM buffers;
 *                      ring position and phases run on across tiles.
 *   RINGSIM_PAIR       the CTA-pair kernel (a cluster of two CTAs): a
 *                      producer in each CTA, the MMA issuer and its barriers
 *                      in the leader.  Both CTAs' copies of a stage signal the
 *                      leader's full[s] (armed once with the pair's bytes);
 *                      the leader's commit frees empty[s] in both CTAs.
 *   RINGSIM_CLC        the response ring of the dynamic tile schedule
 *                      (cluster launch control, which "GEMM II" Step 6 names
 *                      as the successor of its precomputed tile assignment).
 *                      One cluster (a CTA pair) takes `tiles` tiles:
 *                      its own, then one per cancellation response.  The
 *                      rank-0 producer requests at the start of each tile
 *                      (wait clc_empty[j], try_cancel multicast into every
 *                      CTA's slot j, landing `clc_latency` later and
 *                      completing 16 bytes on that CTA's clc_full[j]).  Every
 *                      reader -- each CTA's producer and four epilogue warps,
 *                      the leader's MMA issuer: 11 in all -- reads the
 *                      next response after its tile (wait clc_full[j],
 *                      decode; the producer re-arms its CTA's clc_full[j]
 *                      with 16 bytes for the slot's next use) and arrives on
 *                      the rank-0 CTA's clc_empty[j].  The last response
 *                      cancels nothing and ends every reader.  Role timing:
 *                      a tile's MMAs take k_tiles * mma_time, start
 *                      load_time after its first loads, and may run D =
 *                      depth stages behind the producer; an epilogue warp
 *                      drains a tile in epilogue_time once its MMAs are done;
 *                      `accumulators` tiles may be in flight between them.
 *
 * No GPU is involved; results are deterministic. */
#ifndef RINGSIM_H
#define RINGSIM_H

#ifdef __cplusplus
extern "C" {
#endif

#if defined(_WIN32)
#define RINGSIM_API __declspec(dllexport)
#else
#define RINGSIM_API __attribute__((visibility("default")))
#endif

enum { RINGSIM_LOCKSTEP = 0, RINGSIM_WARP_SPEC = 1, RINGSIM_PAIR = 2, RINGSIM_CLC = 3 };

enum {
    RINGSIM_OK = 0,
    RINGSIM_DEADLOCK = 1,      /* no role can progress and nothing is in flight */
    RINGSIM_EARLY_READ = 2,    /* a stage or accumulator read before its data was complete */
    RINGSIM_OVERWRITE = 3,     /* a stage or accumulator written while still being read */
    RINGSIM_EXTRA_ARRIVAL = 4, /* more arrivals on a barrier phase than it expects */
    RINGSIM_BAD_ARG = 5
};

typedef struct {
    int protocol;          /* RINGSIM_LOCKSTEP, RINGSIM_WARP_SPEC, RINGSIM_PAIR or RINGSIM_CLC */
    int depth;             /* PIPE_DEPTH, 1..64 */
    int k_tiles;           /* K blocks per output tile, >= 1 */
    int tiles;             /* output tiles processed in sequence by one CTA (pair: by each
                              pair; CLC: by the cluster, its own and one per response), >= 1 */
    int accumulators;      /* warp-specialised, pair, CLC: TMEM accumulator buffers, 1 or 2 */
    double load_time;      /* time from a copy's issue to its bytes landing */
    double mma_time;       /* tensor-pipe time of one stage's MMAs */
    double epilogue_time;  /* time to drain one accumulator */
    double issue_latency;  /* time a role spends between a completed wait and its issue */
    long long stage_bytes; /* bytes of one stage of one CTA (two copies of half each: A and B) */
    int chunks;            /* each copy's bytes land in this many equal parts (>= 1) */
    /* fault injection (0 = off) */
    long long bytes_delta;     /* the announced byte budget is stage_bytes + bytes_delta
                                  (pair: the leader's 2 * stage_bytes + bytes_delta) */
    int announce_times;        /* the budget is announced this many times (1 = correct; 0 = 1) */
    int skip_phase_flip;       /* the issuing side never flips its ring phase */
    int reset_phase_per_tile;  /* ring position and phases restart at 0 at every tile */
    int refill_before_mma;     /* lock-step: refill a slot before waiting for its MMA */
    int epilogue_no_wait;      /* warp-specialised: the epilogue skips its accumulator wait */
    int clc_slots;             /* RINGSIM_CLC: response slots, 1..16 (0 = 4) */
    double clc_latency;        /* RINGSIM_CLC: time from a request to its response landing */
    int clc_readers_delta;     /* RINGSIM_CLC fault: clc_empty expects 11 + this arrivals */
    int clc_no_rearm;          /* RINGSIM_CLC fault: the producer never re-arms clc_full */
    int clc_rearm_after_release; /* RINGSIM_CLC: the producer re-arms after its release, issue_latency later */
    int clc_request_late;      /* RINGSIM_CLC: the next request is issued at the end of a tile */
} ringsim_config;

typedef struct {
    int status;                /* RINGSIM_* */
    double makespan;           /* end of the last activity */
    double mma_busy;           /* total tensor-pipe busy time */
    double idle_fraction;      /* 1 - mma_busy / makespan */
    int mma_back_to_back;      /* 1 if every MMA after the first started as the previous ended
                                  (per pair; CLC: not tracked, 0) */
    int max_loads_in_flight;   /* most copies issued and not yet landed at once */
    int stages_consumed;       /* stages whose MMAs were issued */
    int tiles_stored;          /* accumulators drained by the epilogue (CLC: tiles drained
                                  by every epilogue warp) */
    int roles_unique;          /* 1 if every barrier had one arriving and one waiting role
                                  (RINGSIM_CLC: always 1; its responses have many readers) */
    char detail[256];          /* the hazard or deadlock, in words */
    double response_wait;      /* RINGSIM_CLC: time the requesting producer waited for responses */
    double request_wait;       /* RINGSIM_CLC: time the requester waited for a free response slot */
    int responses_read;        /* RINGSIM_CLC: responses read, summed over the readers */
} ringsim_result;

/* Run one configuration.  Returns the result's status (RINGSIM_BAD_ARG, with
 * a message in `detail`, for an invalid configuration). */
RINGSIM_API int ringsim_run(const ringsim_config* cfg, ringsim_result* out);

/* The byte-count handshake of one barrier phase ("05 Async Data Movement -
 * TMA", How to Wait for a TMA Load): a barrier expecting one arrival, one
 * arrive.expect_tx(bytes_a + bytes_b), then the two copies' complete-tx.
 * Writes three states (after expect_tx, after the first copy, after the
 * second), each as {pending arrivals, pending bytes, phase completed 0/1},
 * into `states` (9 values). */
RINGSIM_API void ringsim_byte_trace(long long bytes_a, long long bytes_b, long long* states);

#ifdef __cplusplus
}
#endif

#endif /* RINGSIM_H */
