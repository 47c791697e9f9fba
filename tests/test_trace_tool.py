"""The trace tool's per-slot table (host logic only): earliest times are
stored complemented, unreached slots and stamps are left out or dashed, and
times print in microseconds after the launch start."""
import numpy as np

from block_scaled_fp4_router_gb300.trace import SLOT_COLUMNS, slot_table


def test_slot_table_decodes_stamps():
    t0 = 1_000_000_000
    sl = np.zeros((320, 8), np.uint64)
    mask = (1 << 64) - 1
    # slot 0: expert 5, 3 rows; every stamp set, ns after t0 = 1000 * (c + 1)
    for c in range(7):
        v = t0 + 1000 * (c + 1)
        sl[0, c] = (~v & mask) if c in (0, 4) else v
    sl[0, 7] = (5 << 8) | 3
    # slot 2: expert 9, 1 row; only its gate/up stamps
    sl[2, 0] = ~(t0 + 500) & mask
    sl[2, 1] = t0 + 600
    sl[2, 7] = (9 << 8) | 1
    lines = slot_table(sl, t0)
    assert lines[0].count("|") == len(SLOT_COLUMNS) + 4
    rows = lines[2:]
    assert len(rows) == 2  # slot 1 was never reached
    assert rows[0] == "| 0 | 5 | 3 | 1.0 | 2.0 | 3.0 | 4.0 | 5.0 | 6.0 | 7.0 |"
    assert rows[1] == "| 2 | 9 | 1 | 0.5 | 0.6 | - | - | - | - | - |"
