"""Query rows to compare at full size (test infrastructure).

The persistent kernels hand out (batch, head, 128-row query tile) items in an
order that depends on the problem size, so a full-size check should touch
every tile of every head: ``tile_rows`` returns the first and the last row of
every 128-row tile plus one seeded interior row per tile (and N - 1, the
ragged tail's last row).
"""

import numpy as np


def tile_rows(N, tile=128, seed=0):
    rng = np.random.default_rng(seed)
    rows = []
    for t0 in range(0, N, tile):
        t1 = min(N, t0 + tile)
        rows += [t0, t1 - 1, int(rng.integers(t0, t1))]
    return np.unique(np.array(rows + [N - 1]))
