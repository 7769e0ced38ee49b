"""CPU checks of the host model of the stage-ring protocols (include/ringsim.h).

* The byte-count handshake of one barrier phase against the values "05 Async
  Data Movement - TMA" prints (tests/golden/p2_byte_count_trace.txt).
* The pipeline Gantt of "GEMM II -- pipelining with TMA" (serial vs prefetch)
  against makespans derived by hand and closed forms where loads are hidden.
* Correct protocols run clean for every ring depth 1..8 and K-block count
  around it (1, D-1, D, D+1, 2D+1), one to three tiles, one or two
  accumulators, each barrier with one arriving and one waiting role ("B200
  Tma Pipeline Designer", Validate).
* Faults injected on the host end as the pages say they do: a byte budget too
  large deadlocks, too small releases early, a budget announced four times
  (elect_sync across a warpgroup) deadlocks, phases reset per persistent tile
  fail when a stage completes an odd number of phases per tile, a refill
  before the MMA is done overwrites, an epilogue that does not wait reads an
  incomplete accumulator.
* The CTA-pair protocol runs clean over the same sweep, and a byte budget
  armed for one CTA instead of the pair releases the stage early.
* The response ring of the dynamic tile schedule (cluster launch control)
  runs clean for one to eight slots, any response latency
  and epilogue time; a reader count too high deadlocks; one reader too few
  overwrites a response still unread, or deadlocks, only after a number of
  tiles per cluster that grows with the slot count (beyond what one cluster
  takes at 8192^3 with four slots); a producer that never re-arms its slot
  deadlocks at the slot's second use; re-arming after the release is
  benign.  Requesting at the
  start of a tile hides a response latency shorter than the tile.
"""
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def rs():
    from tma_pipelined_tensor_fp16_gb300 import ringsim
    ringsim.build()
    return ringsim


def _golden(name):
    vals = {}
    for line in open(os.path.join(ROOT, "tests", "golden", name)):
        line = line.split("#", 1)[0].strip()
        if line:
            k, v = line.split("=", 1)
            vals[k.strip()] = int(v.strip())
    return vals


def test_library_exports_every_declared_function(rs):
    text = open(os.path.join(ROOT, "include", "ringsim.h")).read()
    declared = re.findall(r"^RINGSIM_API\s+[\w\s\*]+?\b(\w+)\s*\(", text, re.M)
    assert sorted(declared) == ["ringsim_byte_trace", "ringsim_run"]
    out = subprocess.run(["nm", "-D", "--defined-only", rs.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    exported = set(re.findall(r"\bT (\w+)$", out, re.M))
    assert set(declared) <= exported


def test_byte_count_handshake_matches_the_page(rs):
    g = _golden("p2_byte_count_trace.txt")
    b = g["tile_bytes"]
    after_expect, after_one, after_both = rs.byte_trace(b, b)
    assert after_expect == (g["after_expect_tx_arrivals"], g["after_expect_tx_bytes"], 0)
    assert after_one == (0, b, 0)  # one copy landed: the phase is still open
    assert after_both == (g["after_tma_completes_arrivals"], g["after_tma_completes_bytes"], 1)


def test_serial_gantt_is_load_then_mma_per_tile(rs):
    for K, L in [(8, 1.2), (5, 0.5), (1, 3.0)]:
        g = rs.gantt("serial", k_tiles=K, load_mma=L)
        assert g["status"] == "ok"
        assert g["makespan"] == pytest.approx(K * (L + 1.0))
        assert g["tensor_idle"] == pytest.approx(L / (L + 1.0))
        assert g["loads_in_flight_max"] == 1
        assert not g["mma_back_to_back"] or K == 1


def test_prefetch_gantt_at_the_widget_defaults(rs):
    # PIPE_DEPTH 2, 8 K tiles, load 1.2 x MMA: loads of tiles 0 and 1 land at
    # 1.2; each later load is issued as the MMA two tiles earlier ends, so
    # tile 2 starts at 2.2 + 1.2 = 3.4 (0.2 late), tile 3 at 4.4, tile 4 at
    # 5.6, ... tile 7 ends at 9.8 (derived by hand step by step).
    g = rs.gantt("prefetch", depth=2, k_tiles=8, load_mma=1.2)
    assert g["status"] == "ok" and g["makespan"] == pytest.approx(9.8)
    assert g["tensor_idle"] == pytest.approx(1.8 / 9.8)
    assert not g["mma_back_to_back"] and g["loads_in_flight_max"] == 2


@pytest.mark.parametrize("D,K,L", [(2, 8, 1.0), (3, 8, 1.2), (4, 16, 2.9), (8, 8, 7.0)])
def test_prefetch_hides_loads_up_to_depth_minus_one_mma_times(rs, D, K, L):
    # a load issued when the MMA of tile k ends is needed D - 1 MMA times
    # later: with L <= (D - 1) * T the MMAs run back to back after the first
    # load, makespan L + K T
    g = rs.gantt("prefetch", depth=D, k_tiles=K, load_mma=L)
    assert g["status"] == "ok" and g["mma_back_to_back"]
    assert g["makespan"] == pytest.approx(L + K)
    assert g["loads_in_flight_max"] == min(D, K)


@pytest.mark.parametrize("protocol", ["lockstep", "warp_spec"])
@pytest.mark.parametrize("D", [1, 2, 3, 4, 5, 6, 7, 8])
def test_correct_protocols_run_clean(rs, protocol, D):
    for K in sorted({1, max(1, D - 1), D, D + 1, 2 * D + 1}):
        for tiles in (1, 2, 3):
            for acc in ((1, 2) if protocol == "warp_spec" else (1,)):
                for chunks in (1, 3):
                    r = rs.run(protocol=protocol, depth=D, k_tiles=K, tiles=tiles,
                               accumulators=acc, chunks=chunks, epilogue_time=0.7,
                               load_time=1.3, mma_time=1.0)
                    where = (protocol, D, K, tiles, acc, chunks, r["detail"])
                    assert r["status_name"] == "ok", where
                    assert r["stages_consumed"] == tiles * K, where
                    assert r["tiles_stored"] == tiles, where
                    assert r["roles_unique"] == 1, where
                    assert r["max_loads_in_flight"] <= 2 * D, where


@pytest.mark.parametrize("protocol", ["lockstep", "warp_spec"])
def test_byte_budget_too_large_deadlocks(rs, protocol):
    r = rs.run(protocol=protocol, bytes_delta=16)
    assert r["status_name"] == "deadlock", r
    assert "bytes pending" in r["detail"]


@pytest.mark.parametrize("protocol", ["lockstep", "warp_spec"])
def test_byte_budget_too_small_releases_early(rs, protocol):
    # budget = only A's half of the stage: the phase completes while B's copy
    # is still landing and the MMA reads a half-filled slot
    r = rs.run(protocol=protocol, bytes_delta=-(128 * 64 * 2), chunks=2)
    assert r["status_name"] == "early read", r


@pytest.mark.parametrize("protocol", ["lockstep", "warp_spec"])
def test_budget_announced_four_times_deadlocks(rs, protocol):
    # elect_sync() elects one lane per warp: four announcements in a
    # 128-thread warpgroup, four times the bytes the copies deliver
    r = rs.run(protocol=protocol, announce_times=4)
    assert r["status_name"] == "deadlock", r


def test_missed_phase_flip_is_caught(rs):
    for protocol in ("lockstep", "warp_spec"):
        r = rs.run(protocol=protocol, depth=2, k_tiles=8, skip_phase_flip=1)
        assert r["status_name"] != "ok", (protocol, r)


def test_phase_reset_per_tile_fails_for_odd_phase_counts(rs):
    # resetting the ring position and phases at every persistent tile is
    # safe only while every stage completes an even number of phases per
    # tile: D = 3 with 128 or 79 K blocks has stage 0 complete 43 or 27; the
    # continuous ring position and phases of this library run clean there
    for protocol in ("lockstep", "warp_spec"):
        for K in (128, 79):
            bad = rs.run(protocol=protocol, depth=3, k_tiles=K, tiles=3, reset_phase_per_tile=1)
            assert bad["status_name"] != "ok", (protocol, K, bad)
            good = rs.run(protocol=protocol, depth=3, k_tiles=K, tiles=3)
            assert good["status_name"] == "ok", (protocol, K, good["detail"])
        even = rs.run(protocol=protocol, depth=2, k_tiles=8, tiles=3, reset_phase_per_tile=1)
        assert even["status_name"] == "ok", (protocol, even["detail"])


def test_refill_before_the_mma_is_done_overwrites(rs):
    r = rs.run(protocol="lockstep", depth=2, k_tiles=8, refill_before_mma=1)
    assert r["status_name"] == "overwrite", r


def test_epilogue_that_does_not_wait_reads_early(rs):
    r = rs.run(protocol="warp_spec", tiles=2, epilogue_no_wait=1)
    assert r["status_name"] == "early read", r


def test_second_accumulator_hides_the_epilogue(rs):
    # loads hidden (L <= (D - 1) T); with two accumulators only the last
    # epilogue is exposed, with one every tile's is
    K, T, L, E, tiles = 8, 1.0, 0.5, 3.0, 4
    two = rs.run(protocol="warp_spec", depth=4, k_tiles=K, tiles=tiles, accumulators=2,
                 load_time=L, mma_time=T, epilogue_time=E)
    one = rs.run(protocol="warp_spec", depth=4, k_tiles=K, tiles=tiles, accumulators=1,
                 load_time=L, mma_time=T, epilogue_time=E)
    assert two["status_name"] == one["status_name"] == "ok"
    assert two["makespan"] == pytest.approx(L + tiles * K * T + E)
    assert one["makespan"] == pytest.approx(L + tiles * K * T + tiles * E)


def test_split_roles_keep_the_tensor_pipe_fed(rs):
    # With an issue latency after every completed wait, the single lock-step
    # thread leaves a gap between MMAs (it waits for each MMA before issuing
    # the next); the MMA issuer of the split roles queues MMAs ahead ("GEMM
    # II": prefetch is not yet true concurrency).
    o = 0.2
    lock = rs.run(protocol="lockstep", depth=4, k_tiles=16, load_time=1.0, issue_latency=o)
    spec = rs.run(protocol="warp_spec", depth=4, k_tiles=16, load_time=1.0, issue_latency=o)
    assert lock["status_name"] == spec["status_name"] == "ok"
    assert not lock["mma_back_to_back"] and spec["mma_back_to_back"]
    assert spec["makespan"] < lock["makespan"]


def test_bad_arguments(rs):
    for kw in (dict(depth=0), dict(k_tiles=0), dict(tiles=0), dict(accumulators=3),
               dict(stage_bytes=1), dict(bytes_delta=-(1 << 20))):
        assert rs.run(**kw)["status_name"] == "bad argument", kw
    with pytest.raises(TypeError):
        rs.run(no_such_option=1)


@pytest.mark.parametrize("D", [1, 2, 3, 4, 6])
def test_pair_protocol_runs_clean(rs, D):
    for K in sorted({1, max(1, D - 1), D, D + 1, 2 * D + 1}):
        for tiles in (1, 3):
            for acc in (1, 2):
                r = rs.run(protocol="pair", depth=D, k_tiles=K, tiles=tiles,
                           accumulators=acc, chunks=3, epilogue_time=0.7, load_time=1.3,
                           mma_time=1.0, issue_latency=0.1)
                where = (D, K, tiles, acc, r["detail"])
                assert r["status_name"] == "ok", where
                assert r["stages_consumed"] == tiles * K, where
                assert r["tiles_stored"] == tiles, where
                assert r["roles_unique"] == 1, where


def test_pair_byte_budget_faults(rs):
    kw = dict(protocol="pair", depth=4, k_tiles=8, tiles=2)
    big = rs.run(bytes_delta=16, **kw)
    assert big["status_name"] == "deadlock" and "16 bytes pending" in big["detail"], big
    # the leader arms its full[s] with one CTA's bytes instead of the pair's
    small = rs.run(bytes_delta=-(128 * 64 + 128 * 64) * 2, chunks=2, **kw)
    assert small["status_name"] == "early read", small
    assert rs.run(epilogue_no_wait=1, **kw)["status_name"] == "early read"
    assert rs.run(skip_phase_flip=1, **kw)["status_name"] != "ok"


def test_pair_bad_arguments(rs):
    for kw in (dict(stage_bytes=6), dict(accumulators=0)):
        assert rs.run(protocol="pair", **kw)["status_name"] == "bad argument", kw


CLC = dict(protocol="clc", depth=4, k_tiles=8, load_time=1.2, mma_time=1.0, tiles=9)


@pytest.mark.parametrize("slots", [1, 2, 4, 8])
def test_clc_ring_runs_clean(rs, slots):
    for tiles in (1, 2, 5, 17):
        for latency in (0.0, 0.5, 3.0, 20.0):
            for epi in (0.0, 2.0, 12.0):
                for acc in (1, 2):
                    r = rs.run(**dict(CLC, clc_slots=slots, tiles=tiles,
                                      clc_latency=latency, epilogue_time=epi, accumulators=acc))
                    where = (slots, tiles, latency, epi, acc, r["detail"])
                    assert r["status_name"] == "ok", where
                    assert r["tiles_stored"] == tiles, where
                    # every reader (11 per pair) reads every response, the last
                    # one included (it cancels nothing and ends the loop)
                    assert r["responses_read"] == 11 * tiles, where
                    assert r["stages_consumed"] == tiles * 8, where


def test_clc_reader_count_too_high_deadlocks(rs):
    r = rs.run(**dict(CLC, clc_readers_delta=1))
    assert r["status_name"] == "deadlock" and "clc_empty" in r["detail"], r


def _first_failing_tile_count(rs, limit, **kw):
    for tiles in range(1, limit + 1):
        r = rs.run(**dict(kw, tiles=tiles))
        if r["status_name"] != "ok":
            return tiles, r
    return None, None


def test_clc_reader_count_too_low_shows_only_after_many_tiles(rs):
    # One reader forgotten: each response's surplus arrival completes the
    # slot's next phase one reader earlier, until the requester overwrites a
    # response that epilogue warps have not read, or the parities fall out
    # of step and it deadlocks.  With more slots this takes more tiles per
    # cluster: with four slots more than a GPU run of 8192^3 gives a cluster
    # (1024 tiles over 76 clusters), so only a long run or this model shows it.
    kw = dict(CLC, epilogue_time=6.0, clc_readers_delta=-1)
    n1, r1 = _first_failing_tile_count(rs, 400, clc_slots=1, **kw)
    n4, r4 = _first_failing_tile_count(rs, 400, clc_slots=4, **kw)
    assert n1 is not None and r1["status_name"] == "overwrite", r1
    assert "have not read it" in r1["detail"]
    assert n4 is not None and r4["status_name"] in ("overwrite", "deadlock"), r4
    assert n4 > 3 * n1 and n4 > 1024 // 76, (n1, n4)


def test_clc_missing_rearm_deadlocks_at_the_second_use(rs):
    assert rs.run(**dict(CLC, clc_no_rearm=1, tiles=4))["status_name"] == "ok"
    r = rs.run(**dict(CLC, clc_no_rearm=1, tiles=5))
    assert r["status_name"] == "deadlock" and "-16 bytes pending" in r["detail"], r


@pytest.mark.parametrize("slots", [1, 4])
def test_clc_rearm_after_release_is_benign(rs, slots):
    # the next response may land before the re-arm: its bytes count against
    # the phase first, and the phase completes with the re-arm's arrival
    r = rs.run(**dict(CLC, clc_slots=slots, clc_rearm_after_release=1, issue_latency=50.0))
    assert r["status_name"] == "ok" and r["tiles_stored"] == 9, r
    assert r["response_wait"] > 0


def test_clc_request_at_tile_start_hides_the_latency(rs):
    ref = rs.run(**dict(CLC, clc_latency=0.0))
    early = rs.run(**dict(CLC, clc_latency=3.0))
    late = rs.run(**dict(CLC, clc_latency=3.0, clc_request_late=1))
    assert ref["status_name"] == early["status_name"] == late["status_name"] == "ok"
    assert early["makespan"] == pytest.approx(ref["makespan"])
    assert early["response_wait"] == 0
    # requested at the end of each tile, every response (the last included)
    # is waited for in full
    assert late["response_wait"] == pytest.approx(9 * 3.0)
    assert late["makespan"] > ref["makespan"]
    # a latency longer than a tile is exposed even when requested early
    slow = rs.run(**dict(CLC, clc_latency=12.0))
    assert slow["response_wait"] > 0 and slow["makespan"] > ref["makespan"]


def test_clc_one_slot_stalls_the_requester(rs):
    # with one slot a request waits for the epilogue warps to read the
    # previous response; two slots already remove the cost here
    kw = dict(CLC, epilogue_time=6.0, clc_latency=2.0)
    one, two, four = (rs.run(clc_slots=n, **kw) for n in (1, 2, 4))
    assert one["status_name"] == two["status_name"] == four["status_name"] == "ok"
    assert one["request_wait"] > two["request_wait"] > 0 and four["request_wait"] == 0
    assert one["makespan"] > two["makespan"] == pytest.approx(four["makespan"])


def test_clc_bad_arguments(rs):
    for kw in (dict(clc_slots=17), dict(clc_slots=-1), dict(clc_latency=-1.0),
               dict(clc_readers_delta=-11)):
        assert rs.run(protocol="clc", **kw)["status_name"] == "bad argument", kw


def test_command_line_tables(rs):
    import sys
    env = dict(os.environ, PYTHONPATH=ROOT)
    out = subprocess.run([sys.executable, "-m", "tma_pipelined_tensor_fp16_gb300.ringsim"],
                         capture_output=True, text=True, check=True, cwd=ROOT, env=env).stdout
    assert "makespan 17.60" in out and "makespan 9.80" in out
    out = subprocess.run([sys.executable, "-m", "tma_pipelined_tensor_fp16_gb300.ringsim", "--clc"],
                         capture_output=True, text=True, check=True, cwd=ROOT, env=env).stdout
    assert out.count(" ok ") == 9
    assert "4 slot(s): first fails at 41 tiles (deadlock)" in out
