"""Host-side arithmetic of bench.py: passes and compulsory bytes per run."""
import bench

CELLS = 16384 * 16384


def info(variant, shape, depth=None):
    if depth is None:
        depth = bench.SHAPES[shape][2] if variant == 2 else 1
    return {"variant": variant, "stream_config": shape, "sweeps_per_pass": depth}


def test_single_sweep_shape_moves_8_bytes_per_cell_update():
    assert bench.passes_of(info(2, 3), 100, 0.0, 0) == (100, 0)
    assert bench.algorithmic_bytes(info(2, 3), CELLS, 100, False, 0.0, 0) == 8.0 * CELLS * 100


def test_two_sweep_shape_moves_8_bytes_per_two_cell_updates():
    assert bench.passes_of(info(2, 6), 100, 0.0, 0) == (50, 0)
    assert bench.algorithmic_bytes(info(2, 6), CELLS, 100, False, 0.0, 0) == 8.0 * CELLS * 50
    # an odd count ends with one single sweep
    assert bench.passes_of(info(2, 8), 7, 0.0, 0) == (4, 0)


def test_passes_never_straddle_a_check():
    # odd interval on a STREAM two-sweep shape: passes of 2 and 1 sweeps
    assert bench.passes_of(info(2, 6), 9, 1e-4, 3) == (6, 1)
    # a three-sweep shape with an interval of 10: 3, 3, 3, 1
    assert bench.passes_of(info(2, 10), 20, 1e-4, 10) == (8, 1)
    # a depth-2 LOCAL run with an odd interval: passes of 2, 1, 2, 1, ... never past a check
    assert bench.passes_of(info(3, -1, 2), 9, 1e-4, 3) == (6, 1)
    # depth 3 and an interval of 10: 3, 3, 3, 1 per interval
    assert bench.passes_of(info(3, -1, 3), 20, 1e-4, 10) == (8, 1)
    # even interval: pairs, plus the check-only pass when n is a multiple
    assert bench.passes_of(info(2, 6), 2000, 1e-4, 10) == (1000, 1)
    b = bench.algorithmic_bytes(info(2, 6), 4096 * 4096, 2000, True, 1e-4, 10)
    assert b == 4096 * 4096 * (1000 * 12.0 + 8.0)


def test_other_variants_take_one_sweep_per_pass():
    assert bench.passes_of(info(1, -1), 10, 0.0, 0) == (10, 0)
    assert bench.passes_of(info(3, -1), 10, 0.0, 0) == (10, 0)
    assert bench.passes_of(info(3, -1, 2), 10, 0.0, 0) == (5, 0)
    assert bench.shape_label(info(3, -1, 2), False) == "k_persistent_local2"
    assert bench.shape_label(info(2, 6), False).startswith("k_persistent_stream<{1 float4/thread, 8-deep ring, 2 sweeps/pass}")
