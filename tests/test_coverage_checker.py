"""The coverage build's checker (tests/coverage_cases.py) on the CPU: the
mistakes it exists to catch are planted in made-up counter arrays, never in
a kernel."""
import os
import sys

import numpy as np
import pytest

sys.path.insert(0, os.path.dirname(os.path.abspath(__file__)))
import coverage_cases as cc  # noqa: E402


def counts_for(nx, ny, pitch, per):
    c = np.zeros((2, ny + 2, pitch), np.uint32)
    for b in range(2):
        c[b, 1:ny + 1, 4:nx + 4] = per[b]
    return c


def test_a_correct_record_passes():
    cc.verify_counts(counts_for(13, 5, 32, (4, 3)), (0, 0), 13, 5, 7, "ok")
    cc.verify_counts(counts_for(13, 5, 32, (0, 9)), (0, 0), 13, 5, 9, "in place", in_place=True)


@pytest.mark.parametrize("plant", ["double", "missed", "ring", "pad", "status", "total", "lopsided"])
def test_planted_mistakes_fail(plant):
    nx, ny, pitch = 13, 5, 32
    c = counts_for(nx, ny, pitch, (4, 3))
    status = (0, 0)
    stores = 7
    if plant == "double":        # one cell stored twice in a pass
        c[0, 2, 7] += 1
    elif plant == "missed":      # one cell never stored in a pass
        c[1, ny, nx + 3] -= 1
    elif plant == "ring":        # the ring column stored
        c[0, 3, nx + 4] = 1
    elif plant == "pad":         # a pad float stored
        c[1, 0, 1] = 1
    elif plant == "status":      # an access the kernel flagged
        status = (1, 5)
    elif plant == "total":       # one storing pass too many
        stores = 6
    elif plant == "lopsided":    # passes not alternating between the buffers
        c = counts_for(nx, ny, pitch, (7, 0))
    with pytest.raises(AssertionError):
        cc.verify_counts(c, status, nx, ny, stores, plant)
