"""Per-CTA trace records of the fused kernel (moe_set_trace): consistent stamps,
every tile accounted for, every role ticket taken once, results unchanged, and
nothing written when the trace is off."""
import math

import numpy as np
import pytest
import torch

import oracle
from moe_token_dispatch_route_gb300 import binding, workloads
from tests.gpu_util import check_Y

pytestmark = pytest.mark.gpu

F = {name: i for i, name in enumerate(binding.TRACE_FIELDS)}


@pytest.mark.parametrize("tile_m,tile_n", [(128, 0), (256, 0), (256, 512)])
def test_trace_records_are_consistent(tile_m, tile_n):
    wl = workloads.custom("trace", 1200, 256, 8, 2, 512, 2, "zipf")
    inp = workloads.make_inputs(wl, seed=17)
    plan = binding.moe_plan(wl.T, wl.d, wl.E, wl.k, wl.N, num_ranks=wl.R, tile_m=tile_m, tile_n=tile_n)
    bufs = binding.MoeBuffers(plan, "cuda")
    info = plan.info
    assert tile_n == 0 or info["tile_n"] == tile_n
    trace = torch.full((info["sm_count"] * binding.TRACE_WORDS,), -1, dtype=torch.int64, device="cuda")
    binding.moe_set_trace(plan, trace)
    binding.forward(plan, inp["logits"].cuda(), inp["x"].cuda(), inp["W"].cuda(), bufs)
    rc, status = binding.moe_read_status(bufs.status)
    assert rc == 0, status

    g = info["num_ctas"]
    t = trace.view(-1, binding.TRACE_WORDS)[:g].cpu().numpy()
    assert (t[:, F["start"]] > 0).all() and (t[:, F["end"]] >= t[:, F["start"]]).all()
    assert (t[:, F["scatter_end"]] >= t[:, F["start"]]).all()  # every CTA scatters first by default
    assert (t[:, F["scatter_end"]] <= t[:, F["end"]]).all()
    loaded = t[:, F["tiles"]] > 0
    assert (t[loaded, F["first_tile"]] >= t[loaded, F["scatter_end"]]).all()
    assert (t[:, F["issue_end"]] <= t[:, F["end"]]).all()
    assert (t[:, F["flag_wait_ns"]] >= 0).all()

    ref = oracle.route(inp["logits"].numpy(), wl.k)
    counts = np.diff(ref["offsets"])
    n_tiles = math.ceil(wl.N / info["tile_n"])
    row_tiles = sum(math.ceil(c / tile_m) for c in counts)
    per_tile = 2 if tile_m == 256 else 1  # both CTAs of a pair count the pair's tile
    whole = row_tiles * n_tiles
    # single CTAs claim every tile as two halves when the tiles fill at most half the grid
    split = whole if tile_m == 128 and info["half_tiles"] == 1 and 2 * whole <= g else 0
    assert tile_m == 128 or info["half_tiles"] == 0
    assert int(t[:, F["tiles"]].sum()) == (whole + split) * per_tile
    roles = np.sort(t[:, F["role"]])
    if tile_m == 256:
        assert (roles == np.repeat(np.arange(g // 2), 2)).all()
    else:
        assert (roles == np.arange(g)).all()

    rows = oracle.gather(workloads.bf16_bits(inp["x"]), ref["perm"], wl.k)
    check_Y(bufs.Y.cpu().double().numpy(),
            oracle.grouped_gemm(rows, workloads.bf16_bits(inp["W"]), ref["offsets"]))


def test_trace_off_writes_nothing_and_small_buffers_are_refused():
    wl = workloads.custom("trace_off", 300, 128, 4, 2, 256)
    inp = workloads.make_inputs(wl, seed=18)
    plan = binding.moe_plan(wl.T, wl.d, wl.E, wl.k, wl.N)
    bufs = binding.MoeBuffers(plan, "cuda")
    trace = torch.full((plan.info["sm_count"] * binding.TRACE_WORDS,), -1, dtype=torch.int64, device="cuda")
    with pytest.raises(binding.MoeError) as exc:
        binding.moe_set_trace(plan, trace[:8])
    assert exc.value.status == binding.MOE_ERR_INVALID_ARG
    binding.moe_set_trace(plan, trace)
    binding.moe_set_trace(plan, None)
    binding.forward(plan, inp["logits"].cuda(), inp["x"].cuda(), inp["W"].cuda(), bufs)
    torch.cuda.synchronize()
    assert (trace == -1).all()
