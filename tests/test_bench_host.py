"""Host-side arithmetic of bench.py: passes and compulsory bytes per run."""
import bench

CELLS = 16384 * 16384


def info(variant, shape, depth=None, straddle=None):
    if depth is None:
        depth = bench.SHAPES[shape][2] if variant == 2 else 1
    if straddle is None:  # the plan takes the straddling kernel for three-sweep STREAM shapes
        straddle = variant == 2 and depth == 3
    return {"variant": variant, "stream_config": shape, "sweeps_per_pass": depth,
            "straddle": int(straddle)}


def test_single_sweep_shape_moves_8_bytes_per_cell_update():
    assert bench.passes_of(info(2, 3), 100, 0.0, 0) == (100, 0)
    assert bench.algorithmic_bytes(info(2, 3), CELLS, 100, False, 0.0, 0) == 8.0 * CELLS * 100


def test_two_sweep_shape_moves_8_bytes_per_two_cell_updates():
    assert bench.passes_of(info(2, 6), 100, 0.0, 0) == (50, 0)
    assert bench.algorithmic_bytes(info(2, 6), CELLS, 100, False, 0.0, 0) == 8.0 * CELLS * 50
    # an odd count ends with one single sweep
    assert bench.passes_of(info(2, 8), 7, 0.0, 0) == (4, 0)


def test_passes_stop_at_checks_unless_three_sweep_stream():
    # odd interval on a STREAM two-sweep shape: passes of 2 and 1 sweeps
    assert bench.passes_of(info(2, 6), 9, 1e-4, 3) == (6, 1)
    # a depth-2 LOCAL run with an odd interval: passes of 2, 1, 2, 1, ... never past a check
    assert bench.passes_of(info(3, -1, 2), 9, 1e-4, 3) == (6, 1)
    # LOCAL at depth 3 and an interval of 10: 3, 3, 3, 1 per interval
    assert bench.passes_of(info(3, -1, 3), 20, 1e-4, 10) == (8, 1)
    # even interval: pairs, plus the check-only pass when n is a multiple
    assert bench.passes_of(info(2, 6), 2000, 1e-4, 10) == (1000, 1)
    b = bench.algorithmic_bytes(info(2, 6), 4096 * 4096, 2000, True, 1e-4, 10)
    assert b == 4096 * 4096 * (1000 * 12.0 + 8.0)


def test_three_sweep_stream_passes_straddle_checks():
    # interval 10: passes from 0, 3, 6, 9 (check 10 in stage 2), 12, 15, 18
    # (check 20 would be in stage 3, but only two sweeps are left: the pass
    # stops at 20), then the check-only pass
    assert bench.passes_of(info(2, 10), 20, 1e-4, 10) == (7, 1)
    # 30 sweeps take ten passes: checks 10, 20 and 30 in stages 2, 3 and 1
    assert bench.passes_of(info(2, 12), 30, 1e-4, 10) == (10, 1)
    # the 4096^2 Poisson run: 667 passes instead of 800
    assert bench.passes_of(info(2, 12), 2000, 1e-4, 10) == (667, 1)
    b = bench.algorithmic_bytes(dict(info(2, 12), sweeps_done=2000), 4096 * 4096, 2000, True, 1e-4, 10)
    assert b == 4096 * 4096 * (667 * 12.0 + 8.0)
    # a run that did not take the straddling kernel stops its passes at checks
    assert bench.passes_of(info(2, 11, straddle=False), 20, 1e-4, 10) == (8, 1)
    # no straddling where a second check would fall inside the pass
    assert bench.passes_of(info(2, 11), 10, 1e-4, 2) == (5, 1)
    assert bench.passes_of(info(2, 11), 10, 1e-4, 1) == (10, 1)
    # interval 4: 0..3 (check 0), 3..6 (check 4 in stage 2), 6..8 (stops at 8), ...
    assert bench.passes_of(info(2, 11), 8, 1e-4, 4) == (3, 1)


def test_exit_at_a_straddled_check_costs_one_more_pass():
    # exit at check 10 (stage 2 of the pass from 9): 4 passes + the sweep again from 9
    assert bench.passes_of(info(2, 12), 1000, 1e-4, 10, exit_at=10) == (5, 0)
    # exit at 20 (stage 3 of the pass from 18)
    assert bench.passes_of(info(2, 12), 1000, 1e-4, 10, exit_at=20) == (8, 0)
    # exit at 30 (stage 1 of the pass from 30: U_30 is in memory)
    assert bench.passes_of(info(2, 12), 1000, 1e-4, 10, exit_at=30) == (11, 0)


def test_other_variants_take_one_sweep_per_pass():
    assert bench.passes_of(info(1, -1), 10, 0.0, 0) == (10, 0)
    assert bench.passes_of(info(3, -1), 10, 0.0, 0) == (10, 0)
    assert bench.passes_of(info(3, -1, 2), 10, 0.0, 0) == (5, 0)
    assert bench.shape_label(info(3, -1, 2), False) == "k_persistent_local2"
    assert bench.shape_label(info(2, 6), False).startswith(
        "k_persistent_stream<{1 float4/thread, 8-deep ring, 2 sweeps/pass, 256 consumers}")


def test_clock_summary_keeps_the_timed_region(tmp_path):
    # samples after the mark are the timed region; with none there, the last
    # warm-up sample stands in and the record says so
    path = tmp_path / "clocks.csv"
    idle = "0, 120, 2070, 90, 0x0, Not Active, Not Active, Not Active, Not Active\n"
    warm = "0, 2070, 2070, 900, 0x0, Not Active, Not Active, Not Active, Not Active\n"
    busy = "0, 2040, 2070, 950, 0x4, Not Active, Not Active, Not Active, Active\n"
    path.write_text(idle + warm + busy + busy)
    cs = bench.ClockSampler(0)
    cs.path = str(path)
    cs.offset = len(idle + warm)
    got = cs._summary()
    assert got["samples"] == 2 and got["sm_mhz"] == 2040 and got["reasons"] == ["sw_power_cap"]
    assert got["window"] == "timed region"
    cs.offset = len(idle + warm + busy + busy)
    got = cs._summary()
    assert got["samples"] == 1 and got["sm_mhz"] == 2040 and got["window"].startswith("last warm-up")


def test_compaction_settle_wait_is_bounded():
    # the e2e leg's wait for the host's memory compaction to be idle ends
    # within its limit whatever the host is doing, and says whether it saw
    # the idle state (None where /proc/vmstat cannot be read)
    import time
    import bench
    t0 = time.perf_counter()
    waited, idle = bench.wait_compaction_idle(limit_s=1.0, quiet_s=0.2)
    assert time.perf_counter() - t0 < 2.0 and 0.0 <= waited <= 1.5
    assert idle in (True, False, None)
    pages = bench.compaction_pages()
    assert pages is None or pages >= 0


def test_huge_page_wait_is_bounded():
    # the e2e leg's wait for its buffers' huge pages: immediate where there
    # is nothing to wait for, and never past its limit
    import time
    import numpy as np
    import bench
    a = np.zeros(1 << 20, dtype=np.float32)
    assert bench.wait_huge_pages([a], 0.0) == (0.0, None)
    t0 = time.perf_counter()
    waited, reached = bench.wait_huge_pages([a], 1.0, limit_s=0.5)
    assert time.perf_counter() - t0 < 1.5 and waited <= 1.0
    frac = bench.huge_page_fraction([a])
    assert reached == (frac is not None and frac >= 0.999)
