"""The sampled full-size Y checks reach every output tile (CPU only).

The full-size parity tests compare Y with the oracle on a grid of sampled rows
and columns.  These tests check, on the routing of each full-size workload,
that the grid holds an entry in every 32-row block of every expert (so every
epilogue lane quarter of every 128-row tile and both halves of every 256-row
pair tile) and in every 64-column box of every column tile.
"""
import numpy as np
import pytest

import oracle
from moe_token_dispatch_route_gb300 import workloads
from tests.gpu_util import sample_rows_cols


@pytest.mark.parametrize("name", ["mixtral", "finegrained", "deepseek_v3", "decode"])
def test_sample_grid_covers_every_tile(name):
    wl = workloads.WORKLOADS[name]
    inp = workloads.make_inputs(wl, seed=0, with_weights=False)
    ref = oracle.route(inp["logits"].numpy(), wl.k)
    rows, cols = sample_rows_cols(ref, wl.N, tile_n=256)
    off = ref["offsets"]
    rows = np.array(rows)
    for e in range(wl.E):
        a, b = int(off[e]), int(off[e + 1])
        for r0 in range(a, b, 32):
            assert ((rows >= r0) & (rows < min(r0 + 32, b))).any(), (e, r0)
    cols = np.array(cols)
    for c0 in range(0, wl.N, 64):
        assert ((cols >= c0) & (cols < c0 + 64)).any(), c0
    assert rows.min() >= 0 and rows.max() < wl.S and cols.max() < wl.N
