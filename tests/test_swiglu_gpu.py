"""Gated (SwiGLU) expert FFN on the GPU against the oracle.

* moe_dispatch_gemm_swiglu: the fused dispatch + gated up-projection, whose
  epilogue writes H = silu(gate) * up in bf16;
* moe_grouped_gemm: the grouped GEMM alone on rows already in destination
  order (the down projection);
* the chain route -> up -> down -> combine.

Tolerance of H.  The GPU accumulates gate and up in fp32, applies the
activation in fp32 and rounds once to bf16 (nearest even); the oracle computes
H in fp64.  Rounding to bf16 moves a value by at most half an ulp, 2^-8 of its
magnitude; the fp32 accumulation and activation add a few 1e-6 of the row's
scale, covered by 1e-4 x RMS(H).
"""
import numpy as np
import pytest
import torch

import oracle
from moe_token_dispatch_route_gb300 import binding, workloads
from tests.gpu_util import (TOL_FRO, TOL_MAX_REL_RMS, check_after_bf16_rounding, check_recv, check_route,
                            check_Y, oracle_grid, sample_rows_cols)

pytestmark = pytest.mark.gpu

H_REL = 2.0 ** -8
H_ABS = 1e-4


def check_H(H_dev: torch.Tensor, Href: np.ndarray):
    Hg = H_dev.float().cpu().double().numpy()
    assert Hg.shape == Href.shape
    assert np.isfinite(Hg).all(), "unwritten (NaN) or non-finite H"
    rms = float(np.sqrt(np.mean(Href ** 2)))
    err = np.abs(Hg - Href)
    bound = H_REL * np.abs(Href) + H_ABS * rms
    worst = np.unravel_index(np.argmax(err - bound), err.shape)
    assert (err <= bound).all(), (worst, float(Hg[worst]), float(Href[worst]))


def _run_up(wl, F, inp, W1_dev, **plan_kw):
    plan = binding.moe_plan(wl.T, wl.d, wl.E, wl.k, 2 * F, num_ranks=wl.R, **plan_kw)
    bufs = binding.MoeBuffers(plan, "cuda", out="H")
    bufs.H.fill_(float("nan"))
    for r in bufs.recv:
        r.fill_(float("nan"))
    binding.route(plan, inp["logits"].cuda(), bufs)
    binding.dispatch_gemm_swiglu(plan, inp["x"].cuda(), W1_dev, bufs)
    rc, status = binding.moe_read_status(bufs.status)
    return plan, bufs, rc, status


def _up_check(T, d, E, k, F, R, bias, seed=0, **plan_kw):
    wl = workloads.custom("glu", T, d, E, k, 2 * F, R, bias)
    inp = workloads.make_inputs(wl, seed=seed, with_weights=False)
    W1, _ = workloads.make_ffn_weights(wl, F, seed=seed)
    plan, bufs, rc, status = _run_up(wl, F, inp, W1.cuda(), **plan_kw)
    assert rc == 0, status
    ref = oracle.route(inp["logits"].numpy(), k)
    check_route(bufs, ref, k)
    xb = workloads.bf16_bits(inp["x"])
    rows = oracle.gather(xb, ref["perm"], k)
    check_recv(bufs, xb, ref, k, R, rows)
    G = oracle.grouped_gemm(rows, workloads.bf16_bits(W1), ref["offsets"])
    check_H(bufs.H, oracle.swiglu(G))
    return plan


@pytest.mark.parametrize("T,d,E,k,F,R,bias,tile_n", [
    (300, 128, 4, 2, 144, 1, "none", 0),     # 256-wide tiles: 128 gate + 128 up, ragged F tail
    (257, 64, 8, 2, 64, 2, "none", 0),       # N = 128: 64 + 64, two ranks
    (600, 128, 16, 4, 200, 4, "zipf", 0),    # skewed load, empty experts, tail of 72
    (500, 128, 4, 2, 136, 1, "none", 128),   # forced 128-wide tiles: 3 column tiles (64, 64, 8)
    (64, 256, 128, 8, 96, 1, "hot4", 0),     # decode-like
    (300, 80, 4, 2, 144, 1, "none", 0),      # d = 80: a last k-block of 16 columns
    (200, 1040, 4, 2, 128, 2, "none", 0),    # d = 1040
])
def test_swiglu_up_full_parity(T, d, E, k, F, R, bias, tile_n):
    plan = _up_check(T, d, E, k, F, R, bias, tile_n=tile_n)
    assert plan.info["tile_m"] == 128


@pytest.mark.parametrize("T,d,E,k,F", [
    (1000, 128, 2, 1, 272),   # 3 column tiles of 128 (128, 128, 16); odd halves at the tail
    (130, 64, 1, 1, 128),     # one expert, 130 rows: the odd half holds 2 rows
    (600, 80, 2, 1, 272),     # d = 80: a last k-block of 16 columns
])
def test_swiglu_up_pair_mode(T, d, E, k, F):
    plan = _up_check(T, d, E, k, F, 1, "none", tile_m=256)
    assert plan.info["tile_m"] == 256


@pytest.mark.parametrize("T,d,E,k,F", [
    (1000, 128, 2, 1, 272),   # 512-wide tiles: 256 gate + 256 up columns; 2 column tiles (256, 16)
    (1200, 128, 3, 2, 640),   # 3 column tiles (256, 256, 128)
])
def test_swiglu_up_pair_mode_512_wide_tiles(T, d, E, k, F):
    """Gated up-projection on 512-wide pair tiles: against the oracle, and H bit
    for bit against 256-wide pair tiles (the same MMAs in the same K order)."""
    plan = _up_check(T, d, E, k, F, 1, "none", tile_m=256, tile_n=512)
    assert plan.info["tile_m"] == 256 and plan.info["tile_n"] == 512
    wl = workloads.custom("glu", T, d, E, k, 2 * F, 1, "none")
    inp = workloads.make_inputs(wl, seed=0, with_weights=False)
    W1 = workloads.make_ffn_weights(wl, F, seed=0)[0].cuda()
    H = {}
    for tn in (256, 512):
        _, bufs, rc, status = _run_up(wl, F, inp, W1, tile_m=256, tile_n=tn)
        assert rc == 0, status
        H[tn] = bufs.H.clone()
    assert torch.equal(H[256].view(torch.int16), H[512].view(torch.int16))


def test_swiglu_up_background_scatter_same_bits(monkeypatch):
    """The gated up-projection on CTA pairs with the background scatter (head of one pair
    tile): against the oracle, and H bit for bit against the scatter-first run."""
    monkeypatch.setenv("MOE_BG_HEAD", "1")
    plan = _up_check(1200, 128, 3, 2, 640, 1, "none", tile_m=256)
    assert plan.info["background_scatter"] == 1
    wl = workloads.custom("glu", 1200, 128, 3, 2, 1280, 1, "none")
    inp = workloads.make_inputs(wl, seed=0, with_weights=False)
    W1 = workloads.make_ffn_weights(wl, 640, seed=0)[0].cuda()
    H = {}
    for head in ("1", "0"):
        monkeypatch.setenv("MOE_BG_HEAD", head)
        _, bufs, rc, status = _run_up(wl, 640, inp, W1, tile_m=256)
        assert rc == 0, status
        H[head] = bufs.H.clone()
    assert torch.equal(H["1"].view(torch.int16), H["0"].view(torch.int16))


def test_swiglu_rejects_192_wide_tiles():
    wl = workloads.custom("g192", 100, 64, 4, 2, 384)
    plan = binding.moe_plan(wl.T, wl.d, wl.E, wl.k, wl.N, tile_n=192)
    bufs = binding.MoeBuffers(plan, "cuda", out="H")
    with pytest.raises(binding.MoeError) as exc:
        binding.dispatch_gemm_swiglu(plan, torch.zeros(wl.T, wl.d, dtype=torch.bfloat16, device="cuda"),
                                     torch.zeros(wl.E, wl.d, wl.N, dtype=torch.bfloat16, device="cuda"), bufs)
    assert exc.value.status == binding.MOE_ERR_UNSUPPORTED


# ------------------------------------------------------------ grouped GEMM alone

def _grouped_check(T, d, E, k, N, bias, seed=0, **plan_kw):
    wl = workloads.custom("grp", T, d, E, k, N, 1, bias)
    inp = workloads.make_inputs(wl, seed=seed)
    plan = binding.moe_plan(T, d, E, k, N, **plan_kw)
    bufs = binding.MoeBuffers(plan, "cuda")
    binding.route(plan, inp["logits"].cuda(), bufs)
    A = workloads.make_rows(T * k, d, seed=seed)
    bufs.Y.fill_(float("nan"))
    binding.moe_grouped_gemm(plan, A.cuda(), bufs.offsets, inp["W"].cuda(), bufs.Y, bufs.workspace,
                             bufs.status)
    rc, status = binding.moe_read_status(bufs.status)
    assert rc == 0, status
    ref = oracle.route(inp["logits"].numpy(), k)
    Yref = oracle.grouped_gemm(workloads.bf16_bits(A), workloads.bf16_bits(inp["W"]), ref["offsets"])
    check_Y(bufs.Y.cpu().double().numpy(), Yref)
    return plan


@pytest.mark.parametrize("T,d,E,k,N,bias", [
    (300, 128, 4, 2, 272, "none"),
    (700, 256, 8, 2, 512, "zipf"),
    (64, 256, 128, 8, 256, "hot4"),
    (1, 64, 8, 8, 128, "none"),
    (300, 16, 4, 2, 272, "none"),    # K = 16
    (500, 1040, 8, 2, 256, "zipf"),  # K = 1040
])
def test_grouped_gemm_full_parity(T, d, E, k, N, bias):
    _grouped_check(T, d, E, k, N, bias)


@pytest.mark.parametrize("T,E,N,tile_n", [(1000, 2, 400, 0), (1000, 2, 1040, 512),
                                          (1200, 4, 512, 0), (1200, 4, 512, 512),  # ~300-row experts: M=128 tails
                                          (1000, 2, 1408, 256)])  # a 128-wide last column tile
@pytest.mark.parametrize("d", [128, 80])
def test_grouped_gemm_pair_mode(T, E, N, tile_n, d):
    plan = _grouped_check(T, d, E, 1, N, "none", tile_m=256, tile_n=tile_n)
    assert plan.info["tile_m"] == 256 and (tile_n == 0 or plan.info["tile_n"] == tile_n)


def test_dispatch_and_grouped_calls_share_a_plan():
    """The tensor maps are re-encoded when a plan switches between the dispatch
    and the grouped entry points; the workspace epoch carries across both."""
    wl = workloads.custom("mix", 400, 128, 8, 2, 256, 2, "none")
    inp = workloads.make_inputs(wl, seed=12)
    plan = binding.moe_plan(wl.T, wl.d, wl.E, wl.k, wl.N, num_ranks=wl.R)
    bufs = binding.MoeBuffers(plan, "cuda")
    x, W, L = inp["x"].cuda(), inp["W"].cuda(), inp["logits"].cuda()
    A = workloads.make_rows(wl.S, wl.d, seed=12).cuda()
    ref = oracle.route(inp["logits"].numpy(), wl.k)
    Wb = workloads.bf16_bits(inp["W"])
    Y_disp = oracle.grouped_gemm(oracle.gather(workloads.bf16_bits(inp["x"]), ref["perm"], wl.k), Wb,
                                 ref["offsets"])
    Y_grp = oracle.grouped_gemm(workloads.bf16_bits(A.cpu()), Wb, ref["offsets"])
    binding.route(plan, L, bufs)
    for which in ("dispatch", "grouped", "dispatch", "grouped"):
        bufs.Y.fill_(float("nan"))
        if which == "dispatch":
            binding.dispatch_gemm(plan, x, W, bufs)
        else:
            binding.moe_grouped_gemm(plan, A, bufs.offsets, W, bufs.Y, bufs.workspace, bufs.status)
        rc, status = binding.moe_read_status(bufs.status)
        assert rc == 0, (which, status)
        check_Y(bufs.Y.cpu().double().numpy(), Y_disp if which == "dispatch" else Y_grp)


# ------------------------------------------------------------------ whole FFN

@pytest.mark.parametrize("tile_m", [128, 256])
def test_swiglu_ffn_chain(tile_m):
    """route -> dispatch + gated up-projection -> down projection -> combine,
    against the oracle chain with H rounded to bf16 (the oracle's rounding)."""
    T, d, E, k, F, R = 600, 256, 4, 2, 256, 2  # d = 256: the down projection may pair too
    wl = workloads.custom("ffn", T, d, E, k, 2 * F, R, "none")
    inp = workloads.make_inputs(wl, seed=13, with_weights=False)
    W1, W2 = workloads.make_ffn_weights(wl, F, seed=13)
    up = binding.moe_plan(T, d, E, k, 2 * F, num_ranks=R, tile_m=tile_m)
    bu = binding.MoeBuffers(up, "cuda", out="H")
    down = binding.moe_plan(T, F, E, k, d, tile_m=tile_m)
    bd = binding.MoeBuffers(down, "cuda")
    assert up.info["tile_m"] == down.info["tile_m"] == tile_m
    binding.route(up, inp["logits"].cuda(), bu)
    binding.dispatch_gemm_swiglu(up, inp["x"].cuda(), W1.cuda(), bu)
    binding.moe_grouped_gemm(down, bu.H, bu.offsets, W2.cuda(), bd.Y, bd.workspace, bd.status)
    out = torch.full((T, d), float("nan"), device="cuda")
    binding.moe_combine(down, bd.Y, bu.topk_w, bu.dest, out)
    for st in (bu.status, bd.status):
        rc, status = binding.moe_read_status(st)
        assert rc == 0, status

    ref = oracle.route(inp["logits"].numpy(), k)
    rows = oracle.gather(workloads.bf16_bits(inp["x"]), ref["perm"], k)
    Href = oracle.swiglu(oracle.grouped_gemm(rows, workloads.bf16_bits(W1), ref["offsets"]))
    check_H(bu.H, Href)
    Hb, W2b = oracle.round_bf16(Href), workloads.bf16_bits(W2)
    Y2 = oracle.grouped_gemm(Hb, W2b, ref["offsets"])
    absHW = oracle.grouped_gemm(Hb & 0x7FFF, W2b & 0x7FFF, ref["offsets"])  # |H| . |W2|
    check_after_bf16_rounding(out.cpu().double().numpy(), oracle.combine(Y2, ref["topk_w"], ref["dest"]),
                              oracle.combine(absHW, np.abs(ref["topk_w"]), ref["dest"]))


# -------------------------------------------------- full size, sampled entries

def test_swiglu_mixtral_ffn_full_size_sampled():
    """Mixtral-shaped expert FFN (d = 4096, F = 14336, 8 experts, top-2, 8192
    tokens) in the launch configuration of the benchmark: H and the down
    projection checked at sampled rows and columns, entry by entry."""
    T, d, E, k, F = 8192, 4096, 8, 2, 14336
    wl = workloads.custom("mixtral_ffn", T, d, E, k, 2 * F)
    inp = workloads.make_inputs(wl, seed=0, with_weights=False)
    W1, W2 = workloads.make_ffn_weights(wl, F, seed=0, device="cuda")
    up = binding.moe_plan(T, d, E, k, 2 * F)
    bu = binding.MoeBuffers(up, "cuda", out="H")
    bu.H.fill_(float("nan"))
    binding.route(up, inp["logits"].cuda(), bu)
    binding.dispatch_gemm_swiglu(up, inp["x"].cuda(), W1, bu)
    rc, status = binding.moe_read_status(bu.status)
    assert rc == 0, status
    ref = oracle.route(inp["logits"].numpy(), k)
    check_route(bu, ref, k)
    assert not torch.isnan(bu.H).any().item(), "unwritten (NaN) H"

    rows, fcols = sample_rows_cols(ref, F, tile_n=128, n_random=24)
    a_rows = oracle.gather(workloads.bf16_bits(inp["x"]), ref["perm"][rows], k)
    got = bu.H[torch.tensor(rows, device="cuda")][:, torch.tensor(fcols, device="cuda")]
    got = got.float().cpu().double().numpy()
    G = oracle_grid(a_rows, rows, W1, ref, list(fcols) + [F + f for f in fcols])
    want = oracle.swiglu(G)
    err = np.abs(got - want)
    rms = float(np.sqrt(np.mean(want ** 2)))
    assert (err <= H_REL * np.abs(want) + H_ABS * rms).all()

    # down projection at full size on seeded rows in place of H (no oracle input
    # comes from the library's own output)
    del bu.H
    A = workloads.make_rows(T * k, F, seed=0, device="cuda")
    down = binding.moe_plan(T, F, E, k, d)
    assert down.info["tile_m"] == 256
    ws = torch.zeros(down.workspace_bytes // 4 + 64, dtype=torch.int32, device="cuda")
    status_d = torch.zeros(4, dtype=torch.int32, device="cuda")
    Y2 = torch.full((T * k, d), float("nan"), device="cuda")
    binding.moe_grouped_gemm(down, A, bu.offsets, W2, Y2, ws, status_d)
    rc, status = binding.moe_read_status(status_d)
    assert rc == 0, status
    assert not torch.isnan(Y2).any().item()
    _, dcols = sample_rows_cols(ref, d, tile_n=256, seed=1)  # one column in every 64-column box
    dcols_t = torch.tensor(dcols, device="cuda")
    h_rows = workloads.bf16_bits(A[torch.tensor(rows, device="cuda")])
    got = Y2[torch.tensor(rows, device="cuda")][:, dcols_t].cpu().double().numpy()
    want = oracle_grid(h_rows, rows, W2, ref, dcols)
    err = np.abs(got - want)
    rms = float(np.sqrt(np.mean(want ** 2)))
    assert float(err.max()) <= TOL_MAX_REL_RMS * rms
    assert float(np.linalg.norm(got - want)) <= TOL_FRO * float(np.linalg.norm(want))
