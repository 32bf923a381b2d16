"""The fused dispatch + grouped GEMM (moe_dispatch_gemm) against the oracle.

Small cases compare every output; the full-size workloads (in the launch
configuration the benchmark times) compare the receive buffers in full and Y
on sampled rows and columns, plus the property that no output row was left
unwritten (outputs are poisoned with NaN before each run).
"""
import numpy as np
import pytest
import torch

import oracle
from moe_token_dispatch_route_gb300 import binding, workloads
from tests.gpu_util import (check_recv, check_route, check_Y, check_Y_sampled, oracle_grid, run_path,
                            sample_rows_cols)

pytestmark = pytest.mark.gpu


def _full_check(wl, seed=0, **plan_kw):
    inp = workloads.make_inputs(wl, seed=seed)
    plan, bufs, rc, status = run_path(wl, inp, **plan_kw)
    assert rc == 0, status
    L = inp["logits"].numpy()
    ref = oracle.route(L, wl.k)
    check_route(bufs, ref, wl.k)
    xb = workloads.bf16_bits(inp["x"])
    rows = oracle.gather(xb, ref["perm"], wl.k)
    check_recv(bufs, xb, ref, wl.k, wl.R, rows)
    Yref = oracle.grouped_gemm(rows, workloads.bf16_bits(inp["W"]), ref["offsets"])
    check_Y(bufs.Y.cpu().double().numpy(), Yref)
    return plan, bufs


def test_tiny_workload_full_parity():
    _full_check(workloads.WORKLOADS["tiny"])


@pytest.mark.parametrize("T,d,E,k,N,R,bias", [
    (100, 128, 3, 2, 272, 1, "none"),     # ragged rows and a ragged 16-wide column tail
    (300, 64, 4, 1, 16, 1, "none"),       # minimum d and N
    (257, 192, 8, 2, 512, 2, "none"),     # two ranks
    (600, 128, 16, 4, 384, 4, "zipf"),    # skewed load, empty experts, four ranks
    (64, 256, 128, 8, 256, 1, "hot4"),    # decode-like: 4 hot experts, many 1-6 row experts
    (1, 128, 8, 8, 128, 8, "none"),       # one token, k = E, one expert per rank
    (500, 128, 1, 1, 256, 1, "none"),     # one expert: a plain GEMM with 4 row tiles
])
def test_edge_shapes_full_parity(T, d, E, k, N, R, bias):
    _full_check(workloads.custom("edge", T, d, E, k, N, R, bias))


@pytest.mark.parametrize("tile_n", [128, 192, 256])
def test_tile_widths(tile_n):
    _full_check(workloads.custom("tn", 700, 256, 8, 2, 1408 // 2, 1, "zipf"), tile_n=tile_n)


@pytest.mark.parametrize("d", [16, 80, 1040])
@pytest.mark.parametrize("tile_m", [128, 256])
def test_reduction_not_a_multiple_of_64(d, tile_m):
    """d % 64 != 0: the last k-block holds d % 64 columns (1, 1 and 1 K=16 steps past
    the 64-multiples for d = 16, 80, 1040); the MMAs stop at d in both tile shapes."""
    plan, _ = _full_check(workloads.custom("dk", 600, d, 4, 2, 512, 2, "zipf"), tile_m=tile_m)
    assert plan.info["tile_m"] == tile_m


def test_all_rows_to_one_expert():
    wl = workloads.custom("one", 700, 128, 8, 1, 256, 2, "none")
    inp = workloads.make_inputs(wl, seed=3)
    inp["logits"][:, 5] += 100.0
    plan, bufs, rc, status = run_path(wl, inp)
    assert rc == 0, status
    ref = oracle.route(inp["logits"].numpy(), wl.k)
    assert ref["counts"][5] == 700
    check_route(bufs, ref, wl.k)
    xb = workloads.bf16_bits(inp["x"])
    rows = oracle.gather(xb, ref["perm"], wl.k)
    check_recv(bufs, xb, ref, wl.k, wl.R, rows)
    check_Y(bufs.Y.cpu().double().numpy(),
            oracle.grouped_gemm(rows, workloads.bf16_bits(inp["W"]), ref["offsets"]))


def test_role_split_and_grid_do_not_change_bits():
    """Each output element is reduced in the same K order whatever the scatter/GEMM
    split or grid size, so the results agree bit for bit."""
    wl = workloads.custom("split", 900, 256, 8, 2, 512, 2, "none")
    inp = workloads.make_inputs(wl, seed=4)
    outs = []
    for kw in (dict(), dict(producer_ctas=1), dict(producer_ctas=40), dict(num_ctas=16, producer_ctas=3)):
        _, bufs, rc, status = run_path(wl, inp, **kw)
        assert rc == 0, status
        outs.append(bufs.Y.clone())
    for o in outs[1:]:
        assert torch.equal(outs[0], o)


@pytest.mark.parametrize("tile_n", [128, 256])
def test_half_width_tiles_do_not_change_bits(tile_n, monkeypatch):
    """Single-CTA tiles claimed as left and right halves (N = BN/2 MMAs): whole tiles,
    the default (halves only for small schedules) and every tile split give the same
    bits, for fp32 and bf16 Y and for the direct gather; the split run against the oracle."""
    wl = workloads.custom("tsplit", 700, 256, 8, 2, 656, 2, "zipf")  # ragged last column tile
    inp = workloads.make_inputs(wl, seed=30)
    ref = oracle.route(inp["logits"].numpy(), wl.k)
    rows = oracle.gather(workloads.bf16_bits(inp["x"]), ref["perm"], wl.k)
    Yref = oracle.grouped_gemm(rows, workloads.bf16_bits(inp["W"]), ref["offsets"])
    x, W = inp["x"].cuda(), inp["W"].cuda()
    for out_dtype in (binding.MOE_OUT_F32, binding.MOE_OUT_BF16):
        bf16 = out_dtype == binding.MOE_OUT_BF16
        outs = []
        for split in ("0", None, "2"):
            if split is None:
                monkeypatch.delenv("MOE_HALF_TILES", raising=False)
            else:
                monkeypatch.setenv("MOE_HALF_TILES", split)
            plan, bufs, rc, status = run_path(wl, inp, tile_m=128, tile_n=tile_n, out_dtype=out_dtype)
            assert rc == 0, status
            assert plan.info["half_tiles"] == (0 if split == "0" else 2 if split == "2" else 1)
            outs.append(bufs.Y.clone())
            if not bf16:
                bufs.Y.fill_(float("nan"))
                binding.gather_gemm(plan, x, W, bufs)
                rc, status = binding.moe_read_status(bufs.status)
                assert rc == 0, status
                assert torch.equal(outs[-1], bufs.Y)
        for o in outs[1:]:
            assert torch.equal(outs[0].view(torch.int16 if bf16 else torch.int32),
                               o.view(torch.int16 if bf16 else torch.int32))
        if bf16:
            _check_bf16(outs[2].float().cpu().double().numpy(), Yref)
        else:
            check_Y(outs[2].cpu().double().numpy(), Yref)


def test_repeated_calls_reuse_workspace():
    """Epoch-tagged flags: back-to-back calls on one workspace, outputs poisoned
    between calls, every call complete and identical."""
    wl = workloads.custom("rep", 400, 128, 8, 2, 256, 2, "none")
    inp = workloads.make_inputs(wl, seed=5)
    plan = binding.moe_plan(wl.T, wl.d, wl.E, wl.k, wl.N, num_ranks=wl.R)
    bufs = binding.MoeBuffers(plan, "cuda")
    x, W, L = inp["x"].cuda(), inp["W"].cuda(), inp["logits"].cuda()
    first = None
    for i in range(6):
        bufs.Y.fill_(float("nan"))
        for r in bufs.recv:
            r.fill_(float("nan"))
        binding.forward(plan, L, x, W, bufs)
        rc, st = binding.moe_read_status(bufs.status)
        assert rc == 0, st
        if first is None:
            first = bufs.Y.clone()
        else:
            assert torch.equal(first, bufs.Y)
    hdr = bufs.workspace[:64].cpu()
    assert int(hdr[0]) == 6  # epoch of the last call
    assert int(hdr[8]) == 0 and int(hdr[16]) == 0 and int(hdr[24]) == 0  # counters reset


@pytest.mark.parametrize("name", ["mixtral", "finegrained", "deepseek_v3", "decode"])
def test_full_size_workloads(name):
    wl = workloads.WORKLOADS[name]
    inp = workloads.make_inputs(wl, seed=0, w_device="cuda")
    plan, bufs, rc, status = run_path(wl, inp)
    assert rc == 0, status
    ref = oracle.route(inp["logits"].numpy(), wl.k)
    check_route(bufs, ref, wl.k)
    xb = workloads.bf16_bits(inp["x"])
    check_recv(bufs, xb, ref, wl.k, wl.R)
    rows, cols = sample_rows_cols(ref, wl.N, tile_n=plan.info["tile_n"])
    check_Y_sampled(bufs.Y, xb, inp["W"], ref, wl.k, rows, cols)


def test_missing_flag_times_out_without_hanging():
    """Fault injection on the host side of the contract: the scatter CTAs never
    publish one row tile.  The GEMM CTAs' bounded wait gives up after 2 ms and
    the status names the tile; the kernel still finishes."""
    wl = workloads.custom("fault", 300, 128, 4, 2, 256, 1, "none")
    inp = workloads.make_inputs(wl, seed=6)
    plan, bufs, rc, status = run_path(wl, inp, timeout_ns=2_000_000, debug_skip_publish=2)
    assert rc == binding.MOE_ERR_TIMEOUT, status
    assert status[1] == 1  # the m-tile that was never published
    # the workspace stays consistent: a normal plan on the same shape runs clean afterwards
    plan2, bufs2, rc2, st2 = run_path(wl, inp)
    assert rc2 == 0, st2


def test_receive_capacity_overflow_is_reported():
    wl = workloads.custom("cap", 256, 128, 4, 2, 128, 2, "none")
    inp = workloads.make_inputs(wl, seed=7)
    plan, bufs, rc, status = run_path(wl, inp, rank_capacity_rows=16)
    assert rc == binding.MOE_ERR_CAPACITY, status


# ---------------------------------------------------------------- CTA-pair mode
# The plan runs 256-row tiles on CTA pairs (tcgen05 cta_group::2) when experts
# hold many rows; the shape's tile_m fixes the choice either way for these tests.

@pytest.mark.parametrize("T,d,E,k,N,R,bias", [
    (1000, 128, 2, 1, 512, 1, "none"),    # 2 experts of ~500 rows: odd 128-row halves at the tail
    (700, 256, 4, 2, 400, 2, "none"),     # ragged N tail (400 = 256 + 144), two ranks
    (900, 128, 8, 2, 256, 4, "zipf"),     # skewed: some experts empty, some with < 128 rows
    (130, 64, 1, 1, 272, 1, "none"),      # one expert, 130 rows: the odd half holds 2 rows
])
def test_pair_mode_full_parity(T, d, E, k, N, R, bias):
    plan, _ = _full_check(workloads.custom("pair", T, d, E, k, N, R, bias), tile_m=256)
    assert plan.info["tile_m"] == 256


@pytest.mark.parametrize("T,d,E,k,N,R,bias", [
    (1000, 128, 2, 1, 512, 1, "none"),    # one 512-column tile
    (1200, 256, 4, 2, 1408, 1, "none"),   # ragged N: the last tile holds 384 of 512 columns
    (800, 128, 4, 2, 528, 2, "zipf"),     # 528 = 512 + 16: the last tile's boxes lie mostly outside W
    (130, 64, 1, 1, 1024, 1, "none"),     # one expert of 130 rows: the odd half holds 2 rows
])
def test_pair_mode_512_wide_tiles_full_parity_and_bits(T, d, E, k, N, R, bias):
    """512-column pair tiles (two N=256 MMAs per K step into one 512-column
    accumulator) against the oracle, and bit for bit against 256-column pair
    tiles: every output element sees the same MMAs in the same K order."""
    wl = workloads.custom("pair512", T, d, E, k, N, R, bias)
    plan, bufs = _full_check(wl, tile_m=256, tile_n=512)
    assert plan.info["tile_m"] == 256 and plan.info["tile_n"] == 512 and plan.info["stages"] == 4
    plan256, bufs256 = _full_check(wl, tile_m=256, tile_n=256)
    assert plan256.info["tile_n"] == 256
    assert torch.equal(bufs.Y, bufs256.Y)


def test_pair_mode_512_wide_role_split_and_grid_do_not_change_bits():
    wl = workloads.custom("p512split", 2500, 128, 4, 2, 1024, 1, "none")
    inp = workloads.make_inputs(wl, seed=11)
    outs = []
    for kw in (dict(), dict(producer_ctas=2), dict(num_ctas=16, producer_ctas=4), dict(num_ctas=2)):
        _, bufs, rc, status = run_path(wl, inp, tile_m=256, tile_n=512, **kw)
        assert rc == 0, status
        outs.append(bufs.Y.clone())
    for o in outs[1:]:
        assert torch.equal(outs[0], o)


@pytest.mark.parametrize("name", ["mixtral", "finegrained"])
def test_pair_mode_512_wide_full_size(name):
    wl = workloads.WORKLOADS[name]
    inp = workloads.make_inputs(wl, seed=0, w_device="cuda")
    plan, bufs, rc, status = run_path(wl, inp, tile_n=512)
    assert rc == 0, status
    assert plan.info["tile_m"] == 256 and plan.info["tile_n"] == 512
    ref = oracle.route(inp["logits"].numpy(), wl.k)
    xb = workloads.bf16_bits(inp["x"])
    rows, cols = sample_rows_cols(ref, wl.N, tile_n=512)
    check_Y_sampled(bufs.Y, xb, inp["W"], ref, wl.k, rows, cols)


@pytest.mark.parametrize("tile_n", [256, 512])
@pytest.mark.parametrize("T", [257, 280, 320, 321, 356, 384, 385])
def test_pair_mode_last_tile_of_at_most_128_rows(T, tile_n):
    """One expert of T = 256 + r rows: its last pair tile holds r rows.  With r <= 128
    it runs as an M=128 pair MMA, 64 rows per CTA (r = 1, 24, 64, 65, 100, 128); r =
    129 is an ordinary pair tile with a short odd half.  Every row against the oracle."""
    plan, _ = _full_check(workloads.custom("ptail", T, 128, 1, 1, 1024, 1, "none"), tile_m=256, tile_n=tile_n)
    assert plan.info["tile_m"] == 256 and plan.info["tile_n"] == tile_n


@pytest.mark.parametrize("T,E,k,N", [
    (1000, 4, 2, 384),    # 384 = 256 + 128: the last column tile exactly 128 wide
    (1000, 4, 2, 640),    # 640 = 512 + 128
    (1200, 8, 2, 528),    # a 16-wide last tile; ~300-row experts, so M=128 tails (not narrow) too
    (1500, 4, 2, 1408),   # six column tiles, the last 128 wide
])
def test_pair_mode_narrow_last_column_tile(T, E, k, N):
    """256-wide pair tiles whose last column tile holds at most 128 columns (its B boxes
    partly or wholly outside W, zero-filled).  Against the oracle, and (where 512-wide
    tiles exist, N >= 512) bit for bit against 512-wide tiles: each element sees the same
    K order."""
    wl = workloads.custom("narrow", T, 128, E, k, N, 1, "none")
    plan, bufs = _full_check(wl, tile_m=256, tile_n=256)
    assert plan.info["tile_m"] == 256 and plan.info["tile_n"] == 256
    if N >= 512:
        _, bufs512 = _full_check(wl, tile_m=256, tile_n=512)
        assert torch.equal(bufs.Y, bufs512.Y)


def test_pair_and_single_modes_agree():
    wl = workloads.custom("modes", 1200, 256, 4, 2, 512, 2, "none")
    inp = workloads.make_inputs(wl, seed=8)
    outs = {}
    for tile_m in (128, 256):
        plan, bufs, rc, status = run_path(wl, inp, tile_m=tile_m)
        assert rc == 0, status
        assert plan.info["tile_m"] == tile_m
        outs[tile_m] = bufs.Y.cpu().double().numpy()
    # same K order per element; the two MMA shapes may round differently, so compare to tolerance
    err = np.abs(outs[128] - outs[256]).max()
    assert err <= 1e-4 * np.sqrt(np.mean(outs[128] ** 2))


def test_pair_mode_role_split_does_not_change_bits():
    wl = workloads.custom("psplit", 1500, 128, 4, 2, 512, 1, "none")
    inp = workloads.make_inputs(wl, seed=9)
    outs = []
    for kw in (dict(), dict(producer_ctas=2), dict(producer_ctas=60), dict(num_ctas=16, producer_ctas=4)):
        _, bufs, rc, status = run_path(wl, inp, tile_m=256, **kw)
        assert rc == 0, status
        outs.append(bufs.Y.clone())
    for o in outs[1:]:
        assert torch.equal(outs[0], o)


def test_pair_mode_missing_flag_times_out():
    wl = workloads.custom("pfault", 600, 128, 2, 1, 256, 1, "none")
    inp = workloads.make_inputs(wl, seed=10)
    plan, bufs, rc, status = run_path(wl, inp, tile_m=256, timeout_ns=2_000_000, debug_skip_publish=2)
    assert plan.info["tile_m"] == 256
    assert rc == binding.MOE_ERR_TIMEOUT, status
    assert status[1] == 1
    plan2, bufs2, rc2, st2 = run_path(wl, inp)
    assert rc2 == 0, st2


def test_even_waves_same_bits():
    """A single-CTA schedule of about four waves of tiles: only as many CTAs claim as fill
    every wave.  Against the oracle, and bit for bit against a 16-CTA grid (40 waves, where
    every CTA claims)."""
    wl = workloads.custom("waves", 4096, 128, 16, 2, 1024, 1, "zipf")
    inp = workloads.make_inputs(wl, seed=33)
    outs = []
    for kw in (dict(), dict(num_ctas=16)):
        plan, bufs, rc, status = run_path(wl, inp, tile_m=128, tile_n=128, **kw)
        assert rc == 0, status
        outs.append(bufs.Y.clone())
    tiles = int(((bufs.counts.cpu() + 127) // 128).sum()) * (wl.N // 128)
    grid = binding.moe_plan(wl.T, wl.d, wl.E, wl.k, wl.N, tile_m=128, tile_n=128).info["num_ctas"]
    assert 2 * grid < tiles <= 8 * grid  # the default grid runs the even-waves rule
    assert torch.equal(outs[0], outs[1])
    ref = oracle.route(inp["logits"].numpy(), wl.k)
    rows = oracle.gather(workloads.bf16_bits(inp["x"]), ref["perm"], wl.k)
    check_Y(outs[0].cpu().double().numpy(), oracle.grouped_gemm(rows, workloads.bf16_bits(inp["W"]), ref["offsets"]))


# Background scatter (CTA pairs, wide layers): every warp copies only the rows of the first
# experts before the GEMM, warp 3 of every CTA the rest beside it.  MOE_BG_HEAD sets the head
# (pair tiles) at plan time: 0 off; the automatic setting turns it on from 8192 columns.
@pytest.mark.parametrize("head,kw", [
    ("0", {}), ("1", {}), ("12", {}), (None, {}), ("100000", {}),
    ("1", dict(producer_ctas=8)), ("1", dict(num_ctas=16, producer_ctas=4)),
])
def test_background_scatter_does_not_change_bits(head, kw, monkeypatch):
    """Receive rows against the oracle, Y against the oracle and bit for bit against the
    scatter-first run, and the fused combine bit for bit, for heads of one tile (the first
    non-empty expert), several experts, every expert (no background copies) and under
    role splits with fewer scatter CTAs and a small grid."""
    wl = workloads.custom("pbg", 1500, 336, 8, 2, 512, 2, "zipf")  # 2 ranks, last k-block of 16
    inp = workloads.make_inputs(wl, seed=31)
    ref = oracle.route(inp["logits"].numpy(), wl.k)
    xb = workloads.bf16_bits(inp["x"])
    rows = oracle.gather(xb, ref["perm"], wl.k)
    x, W = inp["x"].cuda(), inp["W"].cuda()

    def run(h):
        if h is None:
            monkeypatch.delenv("MOE_BG_HEAD", raising=False)
        else:
            monkeypatch.setenv("MOE_BG_HEAD", h)
        plan, bufs, rc, status = run_path(wl, inp, tile_m=256, **kw)
        assert rc == 0, status
        assert plan.info["background_scatter"] == (0 if h is None else int(h))
        check_recv(bufs, xb, ref, wl.k, wl.R, rows)
        out = torch.full((wl.T, wl.N), float("nan"), device="cuda")
        binding.dispatch_gemm_combine(plan, x, W, bufs, out)
        rc, status = binding.moe_read_status(bufs.status)
        assert rc == 0, status
        check_recv(bufs, xb, ref, wl.k, wl.R, rows)
        return bufs.Y.clone(), out

    Y, out = run(head)
    check_Y(Y.cpu().double().numpy(), oracle.grouped_gemm(rows, workloads.bf16_bits(inp["W"]), ref["offsets"]))
    Y0, out0 = run("0")
    assert torch.equal(Y, Y0)
    assert torch.equal(out, out0)


def test_background_scatter_missing_flag_times_out(monkeypatch):
    """A ready flag of a tile in the background range that never comes: the bounded wait
    reports MOE_ERR_TIMEOUT with that tile, and the next call on the device is clean."""
    monkeypatch.setenv("MOE_BG_HEAD", "1")
    wl = workloads.custom("pbgfault", 600, 128, 2, 1, 256, 1, "none")
    inp = workloads.make_inputs(wl, seed=10)
    ref = oracle.route(inp["logits"].numpy(), wl.k)
    first_bg = int(-(-int(ref["counts"][0]) // 128))  # first 128-row tile of expert 1
    assert first_bg > 0 and int(ref["counts"][1]) > 0
    plan, bufs, rc, status = run_path(wl, inp, tile_m=256, timeout_ns=2_000_000,
                                      debug_skip_publish=first_bg + 1)
    assert plan.info["background_scatter"] == 1
    assert rc == binding.MOE_ERR_TIMEOUT, status
    assert status[1] == first_bg
    monkeypatch.delenv("MOE_BG_HEAD")
    plan2, bufs2, rc2, st2 = run_path(wl, inp)
    assert rc2 == 0, st2


@pytest.mark.parametrize("T,d,E,k,N,R", [
    (1024, 128, 1024, 8, 64, 32),   # the largest E and R the library accepts
    (200, 64, 64, 32, 32, 4),       # the largest k
    (130, 65536, 1, 1, 16, 1),      # the largest d: 1024 k-blocks per tile
])
def test_limits_full_parity(T, d, E, k, N, R):
    _full_check(workloads.custom("limits", T, d, E, k, N, R))


# ------------------------------------------------------------------ bf16 output
# With MOE_OUT_BF16 the fp32 accumulator is rounded once to bf16 (nearest even):
# at most half an ulp, 2^-8 of the value, beyond the fp32 accumulation error.

def _check_bf16(Y_bf16: np.ndarray, Yref: np.ndarray):
    assert np.isfinite(Y_bf16).all(), "unwritten (NaN) or non-finite output"
    rms = float(np.sqrt(np.mean(Yref ** 2)))
    assert (np.abs(Y_bf16 - Yref) <= 2.0 ** -8 * np.abs(Yref) + 1e-4 * rms).all()


@pytest.mark.parametrize("tile_m,tile_n,N", [(128, 256, 400), (128, 128, 400), (256, 0, 400),
                                            (256, 512, 1040),   # 1040 = 2 x 512 + 16
                                            (256, 256, 384)])   # a 128-wide last column tile
def test_bf16_output_full_parity_and_combine(tile_m, tile_n, N):
    wl = workloads.custom("bf16", 1000, 256, 4, 2, N, 2, "none")
    inp = workloads.make_inputs(wl, seed=14)
    plan, bufs, rc, status = run_path(wl, inp, tile_m=tile_m, tile_n=tile_n, out_dtype=binding.MOE_OUT_BF16)
    assert rc == 0, status
    assert bufs.Y.dtype == torch.bfloat16 and plan.info["tile_m"] == tile_m
    ref = oracle.route(inp["logits"].numpy(), wl.k)
    rows = oracle.gather(workloads.bf16_bits(inp["x"]), ref["perm"], wl.k)
    Yref = oracle.grouped_gemm(rows, workloads.bf16_bits(inp["W"]), ref["offsets"])
    _check_bf16(bufs.Y.float().cpu().double().numpy(), Yref)
    # combine reads the bf16 rows: each term carries at most the rounding of its row
    out = torch.full((wl.T, wl.N), float("nan"), device="cuda")
    binding.moe_combine(plan, bufs.Y, bufs.topk_w, bufs.dest, out)
    want = oracle.combine(Yref, ref["topk_w"], ref["dest"])
    bound = oracle.combine(np.abs(Yref), np.abs(ref["topk_w"]), ref["dest"]) * 2.0 ** -8
    rms = float(np.sqrt(np.mean(want ** 2)))
    assert (np.abs(out.cpu().double().numpy() - want) <= bound + 1e-4 * rms).all()


@pytest.mark.parametrize("tile_n", [256, 512])
def test_bf16_output_on_m128_tail_tiles(tile_n):
    """bf16 Y on pair tiles whose experts end in tails of at most 128 rows (about
    300 rows per expert: one 256-row tile and an M=128 tail each)."""
    wl = workloads.custom("bf16tail", 1200, 128, 8, 2, 1024, 2, "none")
    inp = workloads.make_inputs(wl, seed=16)
    plan, bufs, rc, status = run_path(wl, inp, tile_m=256, tile_n=tile_n, out_dtype=binding.MOE_OUT_BF16)
    assert rc == 0, status
    ref = oracle.route(inp["logits"].numpy(), wl.k)
    counts = np.diff(ref["offsets"])
    assert ((counts % 256 > 0) & (counts % 256 <= 128)).sum() >= 4  # tail tiles present
    rows = oracle.gather(workloads.bf16_bits(inp["x"]), ref["perm"], wl.k)
    Yref = oracle.grouped_gemm(rows, workloads.bf16_bits(inp["W"]), ref["offsets"])
    _check_bf16(bufs.Y.float().cpu().double().numpy(), Yref)


def test_bf16_output_mixtral_full_size_sampled():
    wl = workloads.WORKLOADS["mixtral"]
    inp = workloads.make_inputs(wl, seed=0, w_device="cuda")
    plan, bufs, rc, status = run_path(wl, inp, out_dtype=binding.MOE_OUT_BF16)
    assert rc == 0, status
    assert not torch.isnan(bufs.Y).any().item()
    ref = oracle.route(inp["logits"].numpy(), wl.k)
    rows, cols = sample_rows_cols(ref, wl.N, tile_n=plan.info["tile_n"])
    a_rows = oracle.gather(workloads.bf16_bits(inp["x"]), ref["perm"][rows], wl.k)
    cols_t = torch.tensor(cols, device="cuda")
    got = bufs.Y[torch.tensor(rows, device="cuda")][:, cols_t].float().cpu().double().numpy()
    _check_bf16(got, oracle_grid(a_rows, rows, inp["W"], ref, cols))


def test_empty_batch_every_gemm_entry_point():
    """T = 0: every GEMM entry point returns MOE_OK without launching, and the
    outputs (all zero-sized) need no pointers."""
    plan = binding.moe_plan(0, 128, 8, 2, 256)
    ws = torch.zeros(plan.workspace_bytes // 4 + 64, dtype=torch.int32, device="cuda")
    st = torch.zeros(4, dtype=torch.int32, device="cuda")
    W = torch.zeros(8, 128, 256, dtype=torch.bfloat16, device="cuda")
    binding.moe_dispatch_gemm(plan, None, None, None, W, [], None, ws, st)
    binding.moe_gather_gemm(plan, None, None, None, W, None, ws, st)
    binding.moe_grouped_gemm(plan, None, None, W, None, ws, st)
    binding.moe_dispatch_gemm_swiglu(plan, None, None, None, W, [], None, ws, st)
    rc, status = binding.moe_read_status(st)
    assert rc == 0 and status == [0, 0, 0, 0]


def test_misaligned_pointers_are_refused_before_any_launch():
    wl = workloads.custom("align", 256, 128, 4, 2, 256)
    inp = workloads.make_inputs(wl, seed=19)
    plan = binding.moe_plan(wl.T, wl.d, wl.E, wl.k, wl.N)
    bufs = binding.MoeBuffers(plan, "cuda")
    x, W = inp["x"].cuda(), inp["W"].cuda()
    binding.route(plan, inp["logits"].cuda(), bufs)
    Y_flat = torch.empty(wl.S * wl.N + 4, dtype=torch.float32, device="cuda")
    with pytest.raises(binding.MoeError) as exc:  # Y 4 bytes past a 16-byte boundary
        binding.moe_dispatch_gemm(plan, x, bufs.offsets, bufs.perm, W, bufs.recv, Y_flat[1:].data_ptr(),
                                  bufs.workspace, bufs.status)
    assert exc.value.status == binding.MOE_ERR_INVALID_ARG
    ws = torch.zeros(plan.workspace_bytes // 4 + 128, dtype=torch.int32, device="cuda")
    with pytest.raises(binding.MoeError) as exc:  # workspace off its 256-byte alignment
        binding.moe_dispatch_gemm(plan, x, bufs.offsets, bufs.perm, W, bufs.recv, bufs.Y,
                                  ws[4:].data_ptr(), bufs.status)
    assert exc.value.status == binding.MOE_ERR_WORKSPACE
    x_flat = torch.empty(wl.T * wl.d + 8, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(binding.MoeError) as exc:  # x 2 bytes past a 16-byte boundary
        binding.moe_gather_gemm(plan, x_flat[1:].data_ptr(), bufs.offsets, bufs.perm, W, bufs.Y,
                                bufs.workspace, bufs.status)
    assert exc.value.status == binding.MOE_ERR_INVALID_ARG
    # nothing ran: the status word is still clean and a correct call still works
    rc, status = binding.moe_read_status(bufs.status)
    assert rc == 0, status
    binding.dispatch_gemm(plan, x, W, bufs)
    rc, status = binding.moe_read_status(bufs.status)
    assert rc == 0, status


@pytest.mark.parametrize("tile_m", [128, 256])
def test_calls_with_changing_routing_share_a_workspace(tile_m):
    """Three calls on one plan and workspace with different tokens and logits,
    so the experts' row counts (and the tiles whose flags the epoch tags) change
    from call to call; every call matches the oracle."""
    wl = workloads.custom("change", 900, 128, 8, 2, 512, 2, "zipf")
    plan = binding.moe_plan(wl.T, wl.d, wl.E, wl.k, wl.N, num_ranks=wl.R, tile_m=tile_m)
    bufs = binding.MoeBuffers(plan, "cuda")
    W_cpu = workloads.make_weights(wl, seed=30)
    W = W_cpu.cuda()
    for seed in (31, 32, 33):
        inp = workloads.make_inputs(wl, seed=seed, with_weights=False)
        bufs.Y.fill_(float("nan"))
        binding.forward(plan, inp["logits"].cuda(), inp["x"].cuda(), W, bufs)
        rc, status = binding.moe_read_status(bufs.status)
        assert rc == 0, (seed, status)
        ref = oracle.route(inp["logits"].numpy(), wl.k)
        check_route(bufs, ref, wl.k)
        rows = oracle.gather(workloads.bf16_bits(inp["x"]), ref["perm"], wl.k)
        check_Y(bufs.Y.cpu().double().numpy(),
                oracle.grouped_gemm(rows, workloads.bf16_bits(W_cpu), ref["offsets"]))


def test_receive_capacity_exactly_enough_and_one_short():
    wl = workloads.custom("capx", 500, 128, 8, 2, 256, 4, "zipf")
    inp = workloads.make_inputs(wl, seed=34)
    ref = oracle.route(inp["logits"].numpy(), wl.k)
    base = oracle.rank_base(ref["offsets"], wl.R)
    need = int(np.max(np.diff(base)))
    plan, bufs, rc, status = run_path(wl, inp, rank_capacity_rows=need)
    assert rc == 0, status
    check_recv(bufs, workloads.bf16_bits(inp["x"]), ref, wl.k, wl.R)
    plan, bufs, rc, status = run_path(wl, inp, rank_capacity_rows=need - 1)
    assert rc == binding.MOE_ERR_CAPACITY, status
