// ringsim.cpp -- host-side discrete-event model of the stage-ring protocols
// (declared in include/ringsim.h).  Plain C++17, no CUDA.
//
// Time advances only through events: a part of a copy's bytes landing, an
// MMA finishing, a commit reaching its barrier, an epilogue finishing, a role
// waking after its issue latency.  The roles are state machines that take
// every step their barriers allow at the current time.  When no role can
// step and no event is pending while work remains, the configuration has
// deadlocked.
#include "ringsim.h"

#include <algorithm>
#include <cstdio>
#include <cstring>
#include <queue>
#include <string>
#include <vector>

namespace {

enum Role { ROLE_LOCKSTEP = 0, ROLE_PRODUCER = 1, ROLE_MMA = 2, ROLE_EPILOGUE = 3 };

// One mbarrier.  A phase completes when its pending arrivals reach zero and
// its pending transaction bytes reach zero; the arrivals then re-arm for the
// next phase.  Bytes beyond a phase's budget (a budget announced too small)
// drive the count below zero: the phase completes at the crossing, with some
// copies still landing, and the surplus counts against the next phase.  `completed` counts completed phases, so a wait on parity p returns
// once (completed & 1) != p: the phase of parity p has completed ("05 Async
// Data Movement - TMA", How to Wait for a TMA Load).  The roles that arrive
// on it and wait on it are recorded for the one-producer / one-consumer check
// ("B200 Tma Pipeline Designer", Validate).
struct Barrier {
    int expected = 1;
    int pending = 1;
    long long tx = 0;
    unsigned completed = 0;
    int arrive_role = -1, wait_role = -1;
    bool roles_ok = true;

    void note(int& slot, int role)
    {
        if (slot < 0) slot = role;
        else if (slot != role) roles_ok = false;
    }
    void check_complete()
    {
        if (pending == 0 && tx <= 0) {
            ++completed;
            pending = expected;
        }
    }
    // false: an arrival beyond the phase's expected count
    bool arrive(int role)
    {
        note(arrive_role, role);
        if (pending <= 0) return false;
        --pending;
        check_complete();
        return true;
    }
    bool arrive_expect_tx(int role, long long bytes)
    {
        tx += bytes;
        return arrive(role);
    }
    void complete_tx(long long bytes)
    {
        tx -= bytes;
        check_complete();
    }
    bool passed(int role, unsigned parity)
    {
        note(wait_role, role);
        return (completed & 1u) != parity;
    }
};

// What a stage slot holds: the (tile, k) round last copied into it, how many
// of its bytes have landed, its copies still in flight and the issued MMAs
// still reading it.
struct Slot {
    int tile = -1, k = -1;
    long long landed = 0;
    int copies = 0;
    int readers = 0;
};

// An accumulator: the tile accumulated into it, MMAs completed into it, and
// whether the epilogue has drained it.
struct Accum {
    int tile = -1;
    int mmas_done = 0;
    bool draining = false;
    bool drained = true;
};

enum EventKind { EV_BYTES, EV_MMA_DONE, EV_COMMIT, EV_EPI_DONE, EV_WAKE, EV_CLC_RESPONSE, EV_CLC_REARM };

struct Event {
    double t;
    long long seq;
    int kind;
    int slot, tile, k, acc;
    long long bytes;
    bool last;           // EV_BYTES: the copy's last part
    Barrier* bar;        // EV_BYTES, EV_COMMIT
    int role;            // EV_COMMIT: arriving role
    bool operator>(const Event& o) const { return t != o.t ? t > o.t : seq > o.seq; }
};

struct Sim;

// A role: a program counter, the time before which it cannot issue (its
// issue latency after a completed wait), and its loop state.
struct RoleState {
    int pc = 0;
    double ready_at = 0.0;
    bool done = false;
    int tile = 0, k = 0, stage = 0;
    unsigned phase = 0, phase2 = 0;  // ring phase; MMA / accumulator phase
    int acc = 0;
    bool epi_busy = false;
};

struct Sim {
    ringsim_config c{};
    ringsim_result* r = nullptr;
    double now = 0.0;
    long long seq = 0;
    std::priority_queue<Event, std::vector<Event>, std::greater<Event>> events;
    std::vector<Slot> slots;
    std::vector<Accum> accs;
    std::vector<Barrier> full, empty, tmem_full, tmem_empty;
    Barrier mma_bar;
    int loads_in_flight = 0;
    double pipe_free = 0.0;     // the tensor pipe runs one MMA at a time
    double last_mma_end = 0.0;
    bool first_mma = true;
    bool fault = false;

    void fail(int status, const char* what)
    {
        if (fault) return;
        fault = true;
        r->status = status;
        std::snprintf(r->detail, sizeof(r->detail), "t=%.3f: %s", now, what);
    }
    void push(Event e)
    {
        e.seq = seq++;
        events.push(e);
    }
    void wake(RoleState& s, double t)
    {
        s.ready_at = t;
        Event e{};
        e.t = t;
        e.kind = EV_WAKE;
        push(e);
    }
    long long budget() const
    {
        const int times = c.announce_times > 0 ? c.announce_times : 1;
        return (c.stage_bytes + c.bytes_delta) * times;
    }

    // Issue the two copies of round (tile, k) into slot s; their bytes land
    // in `chunks` equal parts over load_time and each part is a complete-tx
    // on `bar`.
    void issue_copies(int s, int tile, int k, Barrier* bar)
    {
        Slot& sl = slots[s];
        if (sl.readers > 0 || sl.copies > 0) {
            char m[200];
            std::snprintf(m, sizeof(m),
                          "slot %d refilled with (tile %d, k %d) while (tile %d, k %d) is still %s",
                          s, tile, k, sl.tile, sl.k, sl.readers ? "read by an MMA" : "landing");
            fail(RINGSIM_OVERWRITE, m);
            return;
        }
        sl.tile = tile;
        sl.k = k;
        sl.landed = 0;
        const int parts = c.chunks < 1 ? 1 : c.chunks;
        const long long half = c.stage_bytes / 2;
        for (int copy = 0; copy < 2; ++copy) {
            const long long bytes = copy == 0 ? half : c.stage_bytes - half;
            ++sl.copies;
            ++loads_in_flight;
            r->max_loads_in_flight = std::max(r->max_loads_in_flight, loads_in_flight);
            for (int i = 0; i < parts; ++i) {
                Event e{};
                e.t = now + c.load_time * static_cast<double>(i + 1) / parts;
                e.kind = EV_BYTES;
                e.slot = s;
                e.tile = tile;
                e.k = k;
                e.bytes = bytes / parts + (i == parts - 1 ? bytes % parts : 0);
                e.last = i == parts - 1;
                e.bar = bar;
                push(e);
            }
        }
    }

    // Announce a round's byte budget on `bar` (once, or `announce_times`
    // times over when that fault is injected) and issue its copies.
    void load(int role, int s, int tile, int k, Barrier* bar)
    {
        if (!bar->arrive_expect_tx(role, budget())) {
            fail(RINGSIM_EXTRA_ARRIVAL, "a second arrival on a full barrier phase");
            return;
        }
        issue_copies(s, tile, k, bar);
    }

    // Start the MMAs of round (tile, k) from slot s into accumulator a (-1:
    // the lock-step kernel's single accumulator); false on a hazard.
    bool start_mma(int s, int tile, int k, int a)
    {
        Slot& sl = slots[s];
        if (sl.tile != tile || sl.k != k || sl.landed != c.stage_bytes) {
            char m[220];
            std::snprintf(m, sizeof(m),
                          "MMA of (tile %d, k %d) reads slot %d holding (tile %d, k %d) with %lld of %lld bytes landed",
                          tile, k, s, sl.tile, sl.k, sl.landed, c.stage_bytes);
            fail(RINGSIM_EARLY_READ, m);
            return false;
        }
        ++sl.readers;
        const double start = std::max(pipe_free, now);
        if (!first_mma && start > last_mma_end + 1e-9) r->mma_back_to_back = 0;
        first_mma = false;
        pipe_free = start + c.mma_time;
        last_mma_end = pipe_free;
        r->mma_busy += c.mma_time;
        ++r->stages_consumed;
        Event e{};
        e.t = pipe_free;
        e.kind = EV_MMA_DONE;
        e.slot = s;
        e.tile = tile;
        e.acc = a;
        push(e);
        return true;
    }

    // tcgen05.commit: one arrival on `bar` once every MMA issued so far has
    // completed.
    void commit(int role, Barrier* bar)
    {
        Event e{};
        e.t = std::max(pipe_free, now);
        e.kind = EV_COMMIT;
        e.bar = bar;
        e.role = role;
        push(e);
    }

    void apply(const Event& e);
    bool step_lockstep(RoleState& s);
    bool step_producer(RoleState& s);
    bool step_mma(RoleState& s);
    bool step_epilogue(RoleState& s);
};

}  // namespace

namespace {

void Sim::apply(const Event& e)
{
    switch (e.kind) {
    case EV_BYTES: {
        Slot& sl = slots[e.slot];
        if (sl.tile == e.tile && sl.k == e.k) sl.landed += e.bytes;
        e.bar->complete_tx(e.bytes);
        if (e.last) {
            --sl.copies;
            --loads_in_flight;
        }
        break;
    }
    case EV_MMA_DONE:
        --slots[e.slot].readers;
        if (e.acc >= 0 && accs[e.acc].tile == e.tile) ++accs[e.acc].mmas_done;
        break;
    case EV_COMMIT:
        if (!e.bar->arrive(e.role)) fail(RINGSIM_EXTRA_ARRIVAL, "a commit arrived on a completed phase");
        break;
    default:  // EV_WAKE, EV_EPI_DONE: only advance time
        break;
    }
}

// "GEMM II -- pipelining with TMA", Step 5 (and Step 6 around it): one thread
// issues the prologue loads of the first PIPE_DEPTH stages, then per K block
// waits for its stage, issues the MMA, waits for the MMA, refills the stage
// with block k + PIPE_DEPTH, and moves the ring position on (the TMA phase
// flips when the ring wraps, the MMA phase every iteration).  The ring
// position and phases run on across tiles unless reset_phase_per_tile.
bool Sim::step_lockstep(RoleState& s)
{
    const int D = c.depth, K = c.k_tiles;
    switch (s.pc) {
    case 0:
        if (s.tile == c.tiles) {
            s.done = true;
            return true;
        }
        if (c.reset_phase_per_tile) {
            s.stage = 0;
            s.phase = 0;
            s.phase2 = 0;
        }
        for (int i = 0; i < std::min(D, K) && !fault; ++i) {
            const int slot = (s.stage + i) % D;
            load(ROLE_LOCKSTEP, slot, s.tile, i, &full[slot]);
        }
        s.k = 0;
        s.pc = 1;
        return true;
    case 1:
        if (!full[s.stage].passed(ROLE_LOCKSTEP, s.phase)) return false;
        s.pc = 2;
        wake(s, now + c.issue_latency);
        return true;
    case 2:
        if (now < s.ready_at) return false;
        if (!start_mma(s.stage, s.tile, s.k, -1)) return true;
        commit(ROLE_LOCKSTEP, &mma_bar);
        if (c.refill_before_mma && s.k + D < K)
            load(ROLE_LOCKSTEP, s.stage, s.tile, s.k + D, &full[s.stage]);
        s.pc = 3;
        return true;
    case 3:
        if (!mma_bar.passed(ROLE_LOCKSTEP, s.phase2)) return false;
        if (!c.skip_phase_flip) s.phase2 ^= 1u;
        s.pc = 4;
        wake(s, now + c.issue_latency);
        return true;
    case 4:
        if (now < s.ready_at) return false;
        if (!c.refill_before_mma && s.k + D < K)
            load(ROLE_LOCKSTEP, s.stage, s.tile, s.k + D, &full[s.stage]);
        if (++s.stage == D) {
            s.stage = 0;
            if (!c.skip_phase_flip) s.phase ^= 1u;
        }
        s.pc = (++s.k == K) ? 5 : 1;
        return true;
    case 5:  // the epilogue drains the accumulator before the next tile
        s.pc = 6;
        wake(s, now + c.epilogue_time);
        return true;
    case 6:
        if (now < s.ready_at) return false;
        ++r->tiles_stored;
        ++s.tile;
        s.pc = 0;
        return true;
    }
    return false;
}

// The warp-specialised producer: wait empty[s] (a fresh barrier passes the
// first trip), announce full[s]'s byte budget, issue the two copies.
bool Sim::step_producer(RoleState& s)
{
    const int D = c.depth, K = c.k_tiles;
    switch (s.pc) {
    case 0:
        if (s.tile == c.tiles) {
            s.done = true;
            return true;
        }
        if (c.reset_phase_per_tile) {
            s.stage = 0;
            s.phase = 0;
        }
        s.k = 0;
        s.pc = 1;
        return true;
    case 1:
        if (!empty[s.stage].passed(ROLE_PRODUCER, s.phase ^ 1u)) return false;
        s.pc = 2;
        wake(s, now + c.issue_latency);
        return true;
    case 2:
        if (now < s.ready_at) return false;
        load(ROLE_PRODUCER, s.stage, s.tile, s.k, &full[s.stage]);
        if (++s.stage == D) {
            s.stage = 0;
            if (!c.skip_phase_flip) s.phase ^= 1u;
        }
        if (++s.k == K) {
            ++s.tile;
            s.pc = 0;
        } else {
            s.pc = 1;
        }
        return true;
    }
    return false;
}

// The warp-specialised MMA issuer: wait for a drained accumulator, then per K
// block wait full[s], issue the MMA and commit it to empty[s]; at the end of
// the tile commit to tmem_full[a].
bool Sim::step_mma(RoleState& s)
{
    const int D = c.depth, K = c.k_tiles, A = c.accumulators;
    switch (s.pc) {
    case 0:
        if (s.tile == c.tiles) {
            s.done = true;
            return true;
        }
        if (c.reset_phase_per_tile) {  // the ring restarts; accumulators run on
            s.stage = 0;
            s.phase = 0;
        }
        s.k = 0;
        s.pc = 1;
        return true;
    case 1: {
        if (!tmem_empty[s.acc].passed(ROLE_MMA, s.phase2 ^ 1u)) return false;
        Accum& a = accs[s.acc];
        if (!a.drained || a.draining) {
            char m[160];
            std::snprintf(m, sizeof(m), "MMA of tile %d starts into accumulator %d before tile %d is drained",
                          s.tile, s.acc, a.tile);
            fail(RINGSIM_OVERWRITE, m);
            return true;
        }
        a.tile = s.tile;
        a.mmas_done = 0;
        a.drained = false;
        s.pc = 2;
        return true;
    }
    case 2:
        if (!full[s.stage].passed(ROLE_MMA, s.phase)) return false;
        s.pc = 3;
        wake(s, now + c.issue_latency);
        return true;
    case 3:
        if (now < s.ready_at) return false;
        if (!start_mma(s.stage, s.tile, s.k, s.acc)) return true;
        commit(ROLE_MMA, &empty[s.stage]);
        if (++s.stage == D) {
            s.stage = 0;
            if (!c.skip_phase_flip) s.phase ^= 1u;
        }
        if (++s.k == K) {
            commit(ROLE_MMA, &tmem_full[s.acc]);
            if (++s.acc == A) {
                s.acc = 0;
                s.phase2 ^= 1u;
            }
            ++s.tile;
            s.pc = 0;
        } else {
            s.pc = 2;
        }
        return true;
    }
    return false;
}

// The warp-specialised epilogue: wait tmem_full[a], drain the accumulator
// for epilogue_time, release it with an arrival on tmem_empty[a].
bool Sim::step_epilogue(RoleState& s)
{
    const int K = c.k_tiles, A = c.accumulators;
    switch (s.pc) {
    case 0:
        if (s.tile == c.tiles) {
            s.done = true;
            return true;
        }
        s.pc = 1;
        return true;
    case 1: {
        if (!c.epilogue_no_wait && !tmem_full[s.acc].passed(ROLE_EPILOGUE, s.phase2)) return false;
        Accum& a = accs[s.acc];
        if (a.tile != s.tile || a.mmas_done != K) {
            char m[160];
            std::snprintf(m, sizeof(m),
                          "epilogue of tile %d reads accumulator %d holding tile %d after %d of %d MMAs",
                          s.tile, s.acc, a.tile, a.mmas_done, K);
            fail(RINGSIM_EARLY_READ, m);
            return true;
        }
        a.draining = true;
        s.pc = 2;
        wake(s, now + c.epilogue_time);
        return true;
    }
    case 2: {
        if (now < s.ready_at) return false;
        Accum& a = accs[s.acc];
        a.draining = false;
        a.drained = true;
        if (!tmem_empty[s.acc].arrive(ROLE_EPILOGUE)) {
            fail(RINGSIM_EXTRA_ARRIVAL, "a second arrival on an accumulator's empty barrier");
            return true;
        }
        ++r->tiles_stored;
        if (++s.acc == A) {
            s.acc = 0;
            s.phase2 ^= 1u;
        }
        ++s.tile;
        s.pc = 0;
        return true;
    }
    }
    return false;
}

const char* role_name(int role)
{
    switch (role) {
    case ROLE_LOCKSTEP: return "the lock-step thread";
    case ROLE_PRODUCER: return "the producer";
    case ROLE_MMA: return "the MMA issuer";
    default: return "the epilogue";
    }
}

}  // namespace

namespace {

// The CTA-pair kernel (RINGSIM_PAIR): a cluster of two CTAs, 0 the leader
// and 1 its peer.  Every CTA has a producer and stage slots; the leader has
// the MMA issuer, full[s] and the accumulators; every CTA has empty[s].  One
// epilogue role stands for the pair's eight epilogue warps.  Role identities
// are counted by kind (producer, MMA issuer, epilogue) for the unique-role
// check.
struct PairSim {
    ringsim_config c{};
    ringsim_result* r = nullptr;
    static constexpr int NP = 1, C = 2;
    int D = 1, A = 2;
    double now = 0.0;
    long long seq = 0;
    std::priority_queue<Event, std::vector<Event>, std::greater<Event>> events;
    std::vector<Slot> slots;                  // [cta * D + s]
    std::vector<Barrier> full, empty;         // [cta * D + s]
    std::vector<Barrier> tmem_full, tmem_empty;  // [pair * A + a]
    std::vector<Accum> accs;                  // [pair * A + a]
    std::vector<double> pipe_free, last_end;  // per pair
    std::vector<char> first;                  // per pair
    int loads_in_flight = 0;
    bool fault = false;

    void fail(int status, const char* what)
    {
        if (fault) return;
        fault = true;
        r->status = status;
        std::snprintf(r->detail, sizeof(r->detail), "t=%.3f: %s", now, what);
    }
    void push(Event e)
    {
        e.seq = seq++;
        events.push(e);
    }
    void wake(RoleState& s, double t)
    {
        s.ready_at = t;
        Event e{};
        e.t = t;
        e.kind = EV_WAKE;
        push(e);
    }

    // A copy of `bytes` of round (tile, k) into CTA d's slot s, signalling
    // the leader of d's pair.
    void copy_into(int d, int s, int tile, int k, long long bytes)
    {
        Slot& sl = slots[d * D + s];
        const bool same = sl.tile == tile && sl.k == k;
        if (sl.readers > 0 || (!same && sl.copies > 0)) {
            char m[200];
            std::snprintf(m, sizeof(m),
                          "CTA %d slot %d written with (tile %d, k %d) while (tile %d, k %d) is still %s",
                          d, s, tile, k, sl.tile, sl.k, sl.readers ? "read by an MMA" : "landing");
            fail(RINGSIM_OVERWRITE, m);
            return;
        }
        if (!same) {
            sl.tile = tile;
            sl.k = k;
            sl.landed = 0;
        }
        ++sl.copies;
        ++loads_in_flight;
        r->max_loads_in_flight = std::max(r->max_loads_in_flight, loads_in_flight);
        const int parts = c.chunks < 1 ? 1 : c.chunks;
        Barrier* bar = &full[(d & ~1) * D + s];
        for (int i = 0; i < parts; ++i) {
            Event e{};
            e.t = now + c.load_time * static_cast<double>(i + 1) / parts;
            e.kind = EV_BYTES;
            e.slot = d * D + s;
            e.tile = tile;
            e.k = k;
            e.bytes = bytes / parts + (i == parts - 1 ? bytes % parts : 0);
            e.last = i == parts - 1;
            e.bar = bar;
            push(e);
        }
    }

    void apply(const Event& e)
    {
        if (e.kind == EV_BYTES) {
            Slot& sl = slots[e.slot];
            if (sl.tile == e.tile && sl.k == e.k) sl.landed += e.bytes;
            e.bar->complete_tx(e.bytes);
            if (e.last) {
                --sl.copies;
                --loads_in_flight;
            }
        } else if (e.kind == EV_MMA_DONE) {
            // e.slot: the pair's leader CTA * D + stage; both CTAs' slots were read
            --slots[e.slot].readers;
            --slots[e.slot + D].readers;
            if (accs[e.acc].tile == e.tile) ++accs[e.acc].mmas_done;
        } else if (e.kind == EV_COMMIT) {
            if (!e.bar->arrive(ROLE_MMA))
                fail(RINGSIM_EXTRA_ARRIVAL, "a commit arrived on a completed phase");
        }
    }

    bool step_producer(RoleState& s, int cta)
    {
        const int K = c.k_tiles;
        const int pr = cta & 1;
        switch (s.pc) {
        case 0:
            if (s.tile == c.tiles) {
                s.done = true;
                return true;
            }
            s.k = 0;
            s.pc = 1;
            return true;
        case 1:
            if (!empty[cta * D + s.stage].passed(ROLE_PRODUCER, s.phase ^ 1u)) return false;
            s.pc = 2;
            wake(s, now + c.issue_latency);
            return true;
        case 2: {
            if (now < s.ready_at) return false;
            if (pr == 0) {
                const int times = c.announce_times > 0 ? c.announce_times : 1;
                const long long budget = (2 * c.stage_bytes + c.bytes_delta) * times;
                if (!full[cta * D + s.stage].arrive_expect_tx(ROLE_PRODUCER, budget)) {
                    fail(RINGSIM_EXTRA_ARRIVAL, "a second arrival on a full barrier phase");
                    return true;
                }
            }
            const long long half = c.stage_bytes / 2;  // A rows, and this CTA's half of B
            copy_into(cta, s.stage, s.tile, s.k, c.stage_bytes - half);  // B
            copy_into(cta, s.stage, s.tile, s.k, half);                   // A
            if (++s.stage == D) {
                s.stage = 0;
                if (!c.skip_phase_flip) s.phase ^= 1u;
            }
            if (++s.k == K) {
                ++s.tile;
                s.pc = 0;
            } else {
                s.pc = 1;
            }
            return true;
        }
        }
        return false;
    }

    bool step_mma(RoleState& s, int pair)
    {
        const int K = c.k_tiles, L = 2 * pair;
        switch (s.pc) {
        case 0:
            if (s.tile == c.tiles) {
                s.done = true;
                return true;
            }
            s.k = 0;
            s.pc = 1;
            return true;
        case 1: {
            if (!tmem_empty[pair * A + s.acc].passed(ROLE_MMA, s.phase2 ^ 1u)) return false;
            Accum& a = accs[pair * A + s.acc];
            if (!a.drained || a.draining) {
                fail(RINGSIM_OVERWRITE, "MMA starts into an accumulator not yet drained");
                return true;
            }
            a.tile = s.tile;
            a.mmas_done = 0;
            a.drained = false;
            s.pc = 2;
            return true;
        }
        case 2:
            if (!full[L * D + s.stage].passed(ROLE_MMA, s.phase)) return false;
            s.pc = 3;
            wake(s, now + c.issue_latency);
            return true;
        case 3: {
            if (now < s.ready_at) return false;
            for (int d = L; d < L + 2; ++d) {
                const Slot& sl = slots[d * D + s.stage];
                if (sl.tile != s.tile || sl.k != s.k || sl.landed != c.stage_bytes) {
                    char m[220];
                    std::snprintf(m, sizeof(m),
                                  "pair %d MMA of (tile %d, k %d) reads CTA %d slot %d holding (tile %d, k %d) "
                                  "with %lld of %lld bytes landed",
                                  pair, s.tile, s.k, d, s.stage, sl.tile, sl.k, sl.landed, c.stage_bytes);
                    fail(RINGSIM_EARLY_READ, m);
                    return true;
                }
            }
            ++slots[L * D + s.stage].readers;
            ++slots[(L + 1) * D + s.stage].readers;
            const double start = std::max(pipe_free[pair], now);
            if (!first[pair] && start > last_end[pair] + 1e-9) r->mma_back_to_back = 0;
            first[pair] = 0;
            pipe_free[pair] = start + c.mma_time;
            last_end[pair] = pipe_free[pair];
            r->mma_busy += c.mma_time;
            ++r->stages_consumed;
            Event done{};
            done.t = pipe_free[pair];
            done.kind = EV_MMA_DONE;
            done.slot = L * D + s.stage;
            done.tile = s.tile;
            done.acc = pair * A + s.acc;
            push(done);
            // the commit frees the stage in both CTAs of the pair
            for (int d = L; d < L + 2; ++d) {
                Event cm{};
                cm.t = pipe_free[pair];
                cm.kind = EV_COMMIT;
                cm.bar = &empty[d * D + s.stage];
                push(cm);
            }
            if (++s.stage == D) {
                s.stage = 0;
                if (!c.skip_phase_flip) s.phase ^= 1u;
            }
            if (++s.k == K) {
                Event cm{};
                cm.t = pipe_free[pair];
                cm.kind = EV_COMMIT;
                cm.bar = &tmem_full[pair * A + s.acc];
                push(cm);
                if (++s.acc == A) {
                    s.acc = 0;
                    s.phase2 ^= 1u;
                }
                ++s.tile;
                s.pc = 0;
            } else {
                s.pc = 2;
            }
            return true;
        }
        }
        return false;
    }

    bool step_epilogue(RoleState& s, int pair)
    {
        const int K = c.k_tiles;
        switch (s.pc) {
        case 0:
            if (s.tile == c.tiles) {
                s.done = true;
                return true;
            }
            s.pc = 1;
            return true;
        case 1: {
            if (!c.epilogue_no_wait &&
                !tmem_full[pair * A + s.acc].passed(ROLE_EPILOGUE, s.phase2))
                return false;
            Accum& a = accs[pair * A + s.acc];
            if (a.tile != s.tile || a.mmas_done != K) {
                fail(RINGSIM_EARLY_READ, "the epilogue reads an accumulator before its MMAs are done");
                return true;
            }
            a.draining = true;
            s.pc = 2;
            wake(s, now + c.epilogue_time);
            return true;
        }
        case 2: {
            if (now < s.ready_at) return false;
            Accum& a = accs[pair * A + s.acc];
            a.draining = false;
            a.drained = true;
            if (!tmem_empty[pair * A + s.acc].arrive(ROLE_EPILOGUE)) {
                fail(RINGSIM_EXTRA_ARRIVAL, "a second arrival on an accumulator's empty barrier");
                return true;
            }
            ++r->tiles_stored;
            if (++s.acc == A) {
                s.acc = 0;
                s.phase2 ^= 1u;
            }
            ++s.tile;
            s.pc = 0;
            return true;
        }
        }
        return false;
    }

    int run()
    {
        D = c.depth;
        A = c.accumulators;
        slots.resize(C * D);
        full.resize(C * D);
        empty.resize(C * D);
        for (Barrier& b : empty) b.expected = b.pending = 1;
        tmem_full.resize(NP * A);
        tmem_empty.resize(NP * A);
        accs.resize(NP * A);
        pipe_free.assign(NP, 0.0);
        last_end.assign(NP, 0.0);
        first.assign(NP, 1);
        r->mma_back_to_back = 1;
        // roles: producers 0..C-1, MMA issuers C..C+NP-1, epilogues after
        std::vector<RoleState> roles(C + 2 * NP);
        auto step = [&](int i) {
            RoleState& s = roles[i];
            if (s.done || fault) return false;
            if (i < C) return step_producer(s, i);
            if (i < C + NP) return step_mma(s, i - C);
            return step_epilogue(s, i - C - NP);
        };
        long long budget_steps =
            400LL * (c.tiles * static_cast<long long>(c.k_tiles) + 16) * C + 1000000;
        while (!fault) {
            bool progressed = true;
            while (progressed && !fault && budget_steps >= 0) {
                progressed = false;
                for (int i = 0; i < static_cast<int>(roles.size()); ++i)
                    while (step(i)) {
                        progressed = true;
                        if (--budget_steps < 0) break;
                    }
            }
            if (fault) break;
            if (budget_steps < 0) {
                fail(RINGSIM_DEADLOCK, "step limit reached");
                break;
            }
            bool all_done = true;
            for (const RoleState& s : roles) all_done = all_done && s.done;
            if (events.empty()) {
                if (!all_done) {
                    // MMA issuers first: their waits name the cause within the detail's length
                    std::string stuck = "deadlock:";
                    const int nroles = static_cast<int>(roles.size());
                    for (int j = 0; j < nroles; ++j) {
                        const int i = (j + C) % nroles;
                        const RoleState& s = roles[i];
                        if (s.done) continue;
                        const Barrier* b;
                        const char* who;
                        const char* which;
                        int idx, owner;
                        unsigned parity;
                        if (i < C) {
                            who = "producer";
                            idx = owner = i;
                            b = &empty[i * D + s.stage];
                            which = "empty";
                            parity = s.phase ^ 1u;
                        } else if (i < C + NP) {
                            who = "MMA issuer";
                            idx = i - C;
                            owner = 2 * idx;
                            if (s.pc == 1) {
                                b = &tmem_empty[idx * A + s.acc];
                                which = "tmem_empty";
                                parity = s.phase2 ^ 1u;
                            } else {
                                b = &full[owner * D + s.stage];
                                which = "full";
                                parity = s.phase;
                            }
                        } else {
                            who = "epilogue";
                            idx = i - C - NP;
                            owner = 2 * idx;
                            b = &tmem_full[idx * A + s.acc];
                            which = "tmem_full";
                            parity = s.phase2;
                        }
                        char m[200];
                        std::snprintf(m, sizeof(m),
                                      " %s %d (tile %d, k %d) waits on CTA %d's %s parity %u "
                                      "(%u done, %d arrivals, %lld bytes pending);",
                                      who, idx, s.tile, s.k, owner, which, parity, b->completed,
                                      b->pending, b->tx);
                        stuck += m;
                    }
                    fail(RINGSIM_DEADLOCK, stuck.c_str());
                }
                break;
            }
            const Event e = events.top();
            events.pop();
            now = std::max(now, e.t);
            apply(e);
        }
        r->makespan = now;
        r->idle_fraction = now > 0 ? 1.0 - r->mma_busy / (now * NP) : 0.0;
        bool unique = true;
        for (const Barrier& b : full) unique = unique && b.roles_ok;
        for (const Barrier& b : empty) unique = unique && b.roles_ok;
        for (const Barrier& b : tmem_full) unique = unique && b.roles_ok;
        for (const Barrier& b : tmem_empty) unique = unique && b.roles_ok;
        r->roles_unique = unique ? 1 : 0;
        return r->status;
    }
};

}  // namespace

namespace {

// The response ring of the dynamic tile schedule (RINGSIM_CLC).  Each CTA c
// has clc_full[c][j] and a response slot j; the rank-0 CTA has clc_empty[j].
// Roles: a producer per CTA (the rank-0 one also requests), an MMA issuer
// per pair (in its leader), four epilogue warps per CTA.  Every role walks
// the same tile sequence: its own tile, then the tile each response names,
// until a response names none.
struct ClcSim {
    ringsim_config c{};
    ringsim_result* r = nullptr;
    static constexpr int NP = 1, C = 2;
    int S = 4, D = 1, A = 2, K = 1;
    double T = 0.0;  // MMA time of one tile
    double now = 0.0;
    long long seq = 0;
    std::priority_queue<Event, std::vector<Event>, std::greater<Event>> events;
    struct RespSlot {
        int use = -1, value = -1, readers_left = 0;
    };
    std::vector<RespSlot> slots;        // [cta * S + j]
    std::vector<Barrier> full;          // [cta * S + j]
    std::vector<Barrier> empty;         // [j], in the rank-0 CTA
    // per role: position in the tile sequence and the current tile's index
    struct Clc {
        int pc = 0;
        int i = 0;          // tiles started
        int tile = 0;       // current tile (-1: done)
        int use = 0;        // responses read
        double ready_at = 0.0;
        double wait_since = -1.0;
        bool done = false;
    };
    std::vector<Clc> roles;
    std::vector<std::vector<double>> prod_start;  // [cta][i]
    std::vector<std::vector<double>> mma_start;   // [pair][i]
    std::vector<int> mma_started, mma_ended;      // [pair]
    std::vector<int> epi_done;                    // [cta * 4 + w]
    int requests = 0;
    bool fault = false;

    static constexpr long long RESP_BYTES = 16;

    void fail(int status, const char* what)
    {
        if (fault) return;
        fault = true;
        r->status = status;
        std::snprintf(r->detail, sizeof(r->detail), "t=%.3f: %s", now, what);
    }
    void push(Event e)
    {
        e.seq = seq++;
        events.push(e);
    }
    void wake(Clc& s, double t)
    {
        s.ready_at = t;
        Event e{};
        e.t = t;
        e.kind = EV_WAKE;
        push(e);
    }
    int readers_in(int cta) const { return 5 + ((cta & 1) == 0 ? 1 : 0); }
    int cta_of_role(int i) const
    {
        if (i < C) return i;
        if (i < C + NP) return 2 * (i - C);
        return (i - C - NP) / 4;
    }

    void apply(const Event& e)
    {
        if (e.kind == EV_CLC_RESPONSE) {
            // the multicast response lands in every CTA's slot
            for (int d = 0; d < C; ++d) {
                RespSlot& sl = slots[d * S + e.slot];
                if (sl.use >= 0 && sl.readers_left > 0) {
                    char m[200];
                    std::snprintf(m, sizeof(m),
                                  "response %d lands in CTA %d slot %d while %d reader(s) of response %d "
                                  "have not read it",
                                  e.k, d, e.slot, sl.readers_left, sl.use);
                    fail(RINGSIM_OVERWRITE, m);
                    return;
                }
                sl.use = e.k;
                sl.value = e.tile;
                sl.readers_left = readers_in(d);
                full[d * S + e.slot].complete_tx(RESP_BYTES);
            }
        } else if (e.kind == EV_CLC_REARM) {
            e.bar->arrive_expect_tx(ROLE_PRODUCER, RESP_BYTES);
        }
    }

    // Request the tile after the current one (rank-0 producer).  False while
    // the slot is still held by readers of its previous response.
    bool request(Clc& s)
    {
        const int j = requests % S;
        const unsigned free_parity = (static_cast<unsigned>(requests / S) & 1u) ^ 1u;
        if (!empty[j].passed(ROLE_PRODUCER, free_parity)) {
            if (s.wait_since < 0) s.wait_since = now;
            return false;
        }
        if (s.wait_since >= 0) {
            r->request_wait += now - s.wait_since;
            s.wait_since = -1.0;
        }
        Event e{};
        e.t = now + c.clc_latency;
        e.kind = EV_CLC_RESPONSE;
        e.slot = j;
        e.k = requests;                                     // response index
        e.tile = requests + 1 < c.tiles ? requests + 1 : -1;  // the cancelled cluster's tile
        push(e);
        ++requests;
        return true;
    }

    // Read this role's next response in CTA `cta`; `arm`: the CTA's producer.
    // False while the response has not landed.
    bool read(Clc& s, int cta, bool arm, bool timed)
    {
        const int j = s.use % S;
        Barrier& b = full[cta * S + j];
        if (!b.passed(arm ? ROLE_PRODUCER : ROLE_EPILOGUE, static_cast<unsigned>(s.use / S) & 1u)) {
            if (timed && s.wait_since < 0) s.wait_since = now;
            return false;
        }
        if (timed && s.wait_since >= 0) {
            r->response_wait += now - s.wait_since;
            s.wait_since = -1.0;
        }
        RespSlot& sl = slots[cta * S + j];
        if (sl.use != s.use) {
            char m[200];
            std::snprintf(m, sizeof(m), "a reader in CTA %d takes slot %d for response %d but it holds response %d",
                          cta, j, s.use, sl.use);
            fail(RINGSIM_EARLY_READ, m);
            return true;
        }
        const int value = sl.value;
        --sl.readers_left;
        ++r->responses_read;
        if (arm && !c.clc_no_rearm && !c.clc_rearm_after_release)
            b.arrive_expect_tx(ROLE_PRODUCER, RESP_BYTES);
        empty[j].arrive(ROLE_EPILOGUE);
        if (arm && !c.clc_no_rearm && c.clc_rearm_after_release) {
            Event e{};
            e.t = now + c.issue_latency;
            e.kind = EV_CLC_REARM;
            e.bar = &b;
            push(e);
        }
        ++s.use;
        s.tile = value;
        ++s.i;
        return true;
    }

    bool step_producer(Clc& s, int cta)
    {
        const bool requester = cta == 0;
        const int p = cta >> 1;
        switch (s.pc) {
        case 0:  // loop head: a tile to load, or done
            if (s.tile < 0) {
                s.done = true;
                return true;
            }
            prod_start[cta].push_back(now);
            s.pc = requester && !c.clc_request_late ? 1 : 2;
            return true;
        case 1:  // request at the start of the tile
            if (!request(s)) return false;
            s.pc = 2;
            return true;
        case 2: {  // issue the tile's loads: the last D wait for the MMAs to free stages
            if (mma_started[p] <= s.i) return false;
            const int ahead = K > D ? K - D : 0;
            wake(s, std::max(now, mma_start[p][s.i] + ahead * c.mma_time));
            s.pc = 3;
            return true;
        }
        case 3:
            if (now < s.ready_at) return false;
            s.pc = requester && c.clc_request_late ? 4 : 5;
            return true;
        case 4:  // late request: at the end of the tile
            if (!request(s)) return false;
            s.pc = 5;
            return true;
        case 5:
            if (!read(s, cta, true, requester)) return false;
            s.pc = 0;
            return true;
        }
        return false;
    }

    bool step_mma(Clc& s, int p)
    {
        switch (s.pc) {
        case 0: {
            if (s.tile < 0) {
                s.done = true;
                return true;
            }
            // the loads of this tile started in every CTA that feeds the pair
            const int lo = 2 * p, hi = 2 * p + 2;
            double first = 0.0;
            for (int d = lo; d < hi; ++d) {
                if (static_cast<int>(prod_start[d].size()) <= s.i) return false;
                first = std::max(first, prod_start[d][s.i]);
            }
            // an accumulator is free: tile i - A drained by all the pair's epilogue warps
            for (int d = 2 * p; d < 2 * p + 2; ++d)
                for (int w = 0; w < 4; ++w)
                    if (epi_done[d * 4 + w] < s.i - A + 1) return false;
            wake(s, std::max(now, first + c.load_time));
            s.pc = 1;
            return true;
        }
        case 1:
            if (now < s.ready_at) return false;
            mma_start[p].push_back(now);
            mma_started[p] = s.i + 1;
            r->mma_busy += T;
            r->stages_consumed += K;
            wake(s, now + T);
            s.pc = 2;
            return true;
        case 2:
            if (now < s.ready_at) return false;
            mma_ended[p] = s.i + 1;
            s.pc = 3;
            return true;
        case 3:
            if (!read(s, 2 * p, false, false)) return false;
            s.pc = 0;
            return true;
        }
        return false;
    }

    bool step_epilogue(Clc& s, int cta, int w)
    {
        const int p = cta >> 1;
        switch (s.pc) {
        case 0:
            if (s.tile < 0) {
                s.done = true;
                return true;
            }
            if (mma_ended[p] <= s.i) return false;
            wake(s, now + c.epilogue_time);
            s.pc = 1;
            return true;
        case 1:
            if (now < s.ready_at) return false;
            epi_done[cta * 4 + w] = s.i + 1;
            s.pc = 2;
            return true;
        case 2:
            if (!read(s, cta, false, false)) return false;
            s.pc = 0;
            return true;
        }
        return false;
    }

    int run()
    {
        S = c.clc_slots > 0 ? c.clc_slots : 4;
        D = c.depth;
        A = c.accumulators;
        K = c.k_tiles;
        T = K * c.mma_time;
        slots.resize(C * S);
        full.resize(C * S);
        empty.resize(S);
        for (Barrier& b : full) b.arrive_expect_tx(ROLE_PRODUCER, RESP_BYTES);  // armed for first use
        for (Barrier& b : empty) b.expected = b.pending = 11 * NP + c.clc_readers_delta;
        roles.resize(C + NP + 4 * C);
        prod_start.resize(C);
        mma_start.resize(NP);
        mma_started.assign(NP, 0);
        mma_ended.assign(NP, 0);
        epi_done.assign(4 * C, 0);
        r->roles_unique = 1;
        auto step = [&](int i) {
            Clc& s = roles[i];
            if (s.done || fault) return false;
            if (i < C) return step_producer(s, i);
            if (i < C + NP) return step_mma(s, i - C);
            const int e = i - C - NP;
            return step_epilogue(s, e / 4, e % 4);
        };
        long long budget_steps = 200LL * (c.tiles + 16) * static_cast<long long>(roles.size()) + 1000000;
        const int nroles = static_cast<int>(roles.size());
        while (!fault) {
            bool progressed = true;
            while (progressed && !fault && budget_steps >= 0) {
                progressed = false;
                for (int i = 0; i < nroles; ++i)
                    while (step(i)) {
                        progressed = true;
                        if (--budget_steps < 0) break;
                    }
            }
            if (fault) break;
            if (budget_steps < 0) {
                fail(RINGSIM_DEADLOCK, "step limit reached");
                break;
            }
            bool all_done = true;
            for (const Clc& s : roles) all_done = all_done && s.done;
            if (events.empty()) {
                if (!all_done) {
                    std::string stuck = "deadlock:";
                    for (int i = 0; i < nroles; ++i) {
                        const Clc& s = roles[i];
                        if (s.done) continue;
                        const char* who = i < C ? "producer" : (i < C + NP ? "MMA issuer" : "epilogue warp");
                        const int cta = cta_of_role(i);
                        const int j = s.use % S;
                        const Barrier& b = full[cta * S + j];
                        char m[200];
                        std::snprintf(m, sizeof(m),
                                      " %s of CTA %d (tile %d, step %d, response %d; clc_full[%d] %u done, "
                                      "%d arrivals, %lld bytes pending; clc_empty[%d] %u done, %d arrivals);",
                                      who, cta, s.i, s.pc, s.use, j, b.completed, b.pending, b.tx,
                                      requests % S, empty[requests % S].completed,
                                      empty[requests % S].pending);
                        stuck += m;
                    }
                    fail(RINGSIM_DEADLOCK, stuck.c_str());
                }
                break;
            }
            const Event e = events.top();
            events.pop();
            now = std::max(now, e.t);
            apply(e);
        }
        r->makespan = now;
        r->idle_fraction = now > 0 ? 1.0 - r->mma_busy / (now * NP) : 0.0;
        r->mma_back_to_back = 0;
        int stored = c.tiles;
        for (int v : epi_done) stored = std::min(stored, v);
        r->tiles_stored = stored;
        return r->status;
    }
};

}  // namespace

extern "C" {

RINGSIM_API int ringsim_run(const ringsim_config* cfg, ringsim_result* out)
{
    if (!out) return RINGSIM_BAD_ARG;
    std::memset(out, 0, sizeof(*out));
    auto bad = [&](const char* why) {
        out->status = RINGSIM_BAD_ARG;
        std::snprintf(out->detail, sizeof(out->detail), "%s", why);
        return RINGSIM_BAD_ARG;
    };
    if (!cfg) return bad("config is NULL");
    const ringsim_config& c = *cfg;
    if (c.protocol < RINGSIM_LOCKSTEP || c.protocol > RINGSIM_CLC)
        return bad("protocol must be RINGSIM_LOCKSTEP, RINGSIM_WARP_SPEC, RINGSIM_PAIR or RINGSIM_CLC");
    if (c.depth < 1 || c.depth > 64) return bad("depth must be 1..64");
    if (c.k_tiles < 1 || c.k_tiles > 65535) return bad("k_tiles must be 1..65535");
    if (c.tiles < 1 || c.tiles > 100000) return bad("tiles must be 1..100000");
    if (c.protocol != RINGSIM_LOCKSTEP && (c.accumulators < 1 || c.accumulators > 2))
        return bad("accumulators must be 1 or 2");
    if (c.protocol == RINGSIM_CLC) {
        if (c.clc_slots < 0 || c.clc_slots > 16) return bad("clc_slots must be 0 (4) or 1..16");
        if (c.clc_latency < 0) return bad("clc_latency must be non-negative");
        if (11 + c.clc_readers_delta < 1)
            return bad("clc_empty must expect at least one arrival");
    }
    if (c.protocol == RINGSIM_PAIR && c.stage_bytes % 4 != 0)
        return bad("stage_bytes must be a multiple of 4 for CTA pairs");
    if (c.stage_bytes < 2 || c.load_time < 0 || c.mma_time < 0 || c.epilogue_time < 0 ||
        c.issue_latency < 0)
        return bad("stage_bytes >= 2 and non-negative times required");
    if ((c.protocol == RINGSIM_PAIR ? 2 : 1) * c.stage_bytes + c.bytes_delta <= 0)
        return bad("the announced byte budget must be positive");

    if (c.protocol == RINGSIM_CLC) {
        ClcSim cs;
        cs.c = c;
        cs.r = out;
        return cs.run();
    }
    if (c.protocol == RINGSIM_PAIR) {
        PairSim ps;
        ps.c = c;
        ps.r = out;
        return ps.run();
    }
    Sim sim;
    sim.c = c;
    sim.r = out;
    out->mma_back_to_back = 1;
    sim.slots.resize(c.depth);
    sim.full.resize(c.depth);
    sim.empty.resize(c.depth);
    const int A = c.protocol == RINGSIM_WARP_SPEC ? c.accumulators : 1;
    sim.accs.resize(A);
    sim.tmem_full.resize(A);
    sim.tmem_empty.resize(A);

    std::vector<RoleState> roles(c.protocol == RINGSIM_LOCKSTEP ? 1 : 3);
    auto step = [&](int i) {
        RoleState& s = roles[i];
        if (s.done || sim.fault) return false;
        if (c.protocol == RINGSIM_LOCKSTEP) return sim.step_lockstep(s);
        if (i == 0) return sim.step_producer(s);
        if (i == 1) return sim.step_mma(s);
        return sim.step_epilogue(s);
    };
    long long budget_steps = 200LL * (c.tiles * static_cast<long long>(c.k_tiles) + 16) + 1000000;
    while (!sim.fault) {
        bool progressed = true;
        while (progressed && !sim.fault) {
            progressed = false;
            for (size_t i = 0; i < roles.size(); ++i)
                while (step(static_cast<int>(i))) {
                    progressed = true;
                    if (--budget_steps < 0) break;
                }
            if (budget_steps < 0) break;
        }
        if (sim.fault) break;
        if (budget_steps < 0) {
            sim.fail(RINGSIM_DEADLOCK, "step limit reached");
            break;
        }
        bool all_done = true;
        for (const RoleState& s : roles) all_done = all_done && s.done;
        if (sim.events.empty()) {
            if (!all_done) {
                // name every stuck role and the barrier it waits on
                std::string stuck;
                for (size_t i = 0; i < roles.size(); ++i) {
                    const RoleState& s = roles[i];
                    if (s.done) continue;
                    const int role = c.protocol == RINGSIM_LOCKSTEP ? ROLE_LOCKSTEP
                                                                      : static_cast<int>(i) + 1;
                    const Barrier* b = nullptr;
                    const char* which = "a barrier";
                    unsigned parity = 0;
                    int index = 0;
                    if (role == ROLE_LOCKSTEP) {
                        if (s.pc == 1) { b = &sim.full[s.stage]; which = "tma_bar"; parity = s.phase; index = s.stage; }
                        else { b = &sim.mma_bar; which = "mma_bar"; parity = s.phase2; }
                    } else if (role == ROLE_PRODUCER) {
                        b = &sim.empty[s.stage]; which = "empty"; parity = s.phase ^ 1u; index = s.stage;
                    } else if (role == ROLE_MMA) {
                        if (s.pc == 1) { b = &sim.tmem_empty[s.acc]; which = "tmem_empty"; parity = s.phase2 ^ 1u; index = s.acc; }
                        else { b = &sim.full[s.stage]; which = "full"; parity = s.phase; index = s.stage; }
                    } else {
                        b = &sim.tmem_full[s.acc]; which = "tmem_full"; parity = s.phase2; index = s.acc;
                    }
                    char m[200];
                    std::snprintf(m, sizeof(m),
                                  "%s%s (tile %d, k %d) waits on %s[%d] parity %u (%u phases done, "
                                  "%d arrivals, %lld bytes pending)",
                                  stuck.empty() ? "deadlock: " : "; ", role_name(role), s.tile, s.k,
                                  which, index, parity, b->completed, b->pending, b->tx);
                    stuck += m;
                }
                sim.fail(RINGSIM_DEADLOCK, stuck.c_str());
            }
            break;
        }
        // one event at a time, so that a role can act between two events of
        // the same instant (a phase released before a later part lands)
        const Event e = sim.events.top();
        sim.events.pop();
        sim.now = std::max(sim.now, e.t);
        sim.apply(e);
    }
    out->makespan = sim.now;
    out->idle_fraction = out->makespan > 0 ? 1.0 - out->mma_busy / out->makespan : 0.0;
    bool unique = true;
    for (const Barrier& b : sim.full) unique = unique && b.roles_ok;
    for (const Barrier& b : sim.empty) unique = unique && b.roles_ok;
    for (const Barrier& b : sim.tmem_full) unique = unique && b.roles_ok;
    for (const Barrier& b : sim.tmem_empty) unique = unique && b.roles_ok;
    unique = unique && sim.mma_bar.roles_ok;
    out->roles_unique = unique ? 1 : 0;
    return out->status;
}

RINGSIM_API void ringsim_byte_trace(long long bytes_a, long long bytes_b, long long* states)
{
    if (!states) return;
    Barrier bar;  // one expected arrival
    const unsigned before = bar.completed;
    auto record = [&](int i) {
        states[3 * i + 0] = bar.completed != before ? 0 : bar.pending;
        states[3 * i + 1] = bar.tx;
        states[3 * i + 2] = bar.completed != before ? 1 : 0;
    };
    bar.arrive_expect_tx(ROLE_PRODUCER, bytes_a + bytes_b);
    record(0);
    bar.complete_tx(bytes_a);
    record(1);
    bar.complete_tx(bytes_b);
    record(2);
}

}  // extern "C"
