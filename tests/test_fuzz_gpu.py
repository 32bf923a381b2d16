"""Seeded random shapes and plan options through every GEMM entry point, each run
checked in full against the oracle.

For each case: routing and the receive rows bit-exact; Y (fp32, or bf16 with its one
rounding) within the tolerance; the direct gather bit for bit against the dispatch on
the same plan; the grouped GEMM on the
landed rows bit for bit against the dispatch; the combine, separate and fused into the
epilogue, against the oracle's combine.  The cases mix what the hand-written tests
cover one at a time: ragged experts and column tails, d not a multiple of 64, several
ranks, empty experts, CTA pairs with M=128 tails, 512-wide pair tiles, 128/192/256-wide
single tiles, half-width tiles of small schedules, and bf16 Y.  A second set runs the
gated expert FFN (dispatch + SwiGLU up-projection, grouped down projection, combine) on
random shapes against the oracle chain.
"""
import numpy as np
import pytest
import torch

import oracle
from moe_token_dispatch_route_gb300 import binding, workloads
from tests.gpu_util import check_after_bf16_rounding, check_recv, check_route, check_Y, run_path

pytestmark = pytest.mark.gpu

N_CASES = 64
N_FFN_CASES = 16


def _case(i: int) -> dict:
    rng = np.random.default_rng(7000 + i)
    E = int(rng.choice([1, 2, 3, 4, 8, 12, 16, 32, 64, 128]))
    k = int(rng.integers(1, min(E, 8) + 1))
    T = int(rng.integers(1, 1200 // k + 1))  # S = T k <= 1200 rows
    d = 16 * int(rng.integers(1, 33))        # 16 .. 512
    N = 16 * int(rng.integers(1, 49))        # 16 .. 768
    R = int(rng.choice([r for r in (1, 2, 4, 8) if E % r == 0]))
    bias = str(rng.choice(["none", "zipf"] + (["hot4"] if E >= 4 else [])))
    tile_m = int(rng.choice([0, 128] + ([256] if N >= 256 else [])))
    if tile_m == 256:
        tile_n = int(rng.choice([0, 256] + ([512] if N >= 512 else [])))
    elif tile_m == 128:
        tile_n = int(rng.choice([0, 128, 192, 256]))
    else:
        tile_n = 0
    out_dtype = binding.MOE_OUT_BF16 if rng.random() < 0.25 else binding.MOE_OUT_F32
    # CTA pairs: the background scatter's head (pair tiles), or the automatic setting
    bg_head = str(rng.choice(["auto", "0", "1", "4", "16"]))
    return dict(T=T, d=d, E=E, k=k, N=N, R=R, bias=bias, tile_m=tile_m, tile_n=tile_n,
                out_dtype=out_dtype, bg_head=bg_head)


def _check_bf16(Y_bf16: np.ndarray, Yref: np.ndarray):
    """bf16 Y: at most half an ulp (2^-8 of the value) beyond the fp32 accumulation."""
    assert np.isfinite(Y_bf16).all(), "unwritten (NaN) or non-finite output"
    rms = float(np.sqrt(np.mean(Yref ** 2))) if Yref.size else 0.0
    assert (np.abs(Y_bf16 - Yref) <= 2.0 ** -8 * np.abs(Yref) + 1e-4 * rms).all()


def _check_out(Y_dev: torch.Tensor, Yref: np.ndarray, bf16: bool):
    if bf16:
        _check_bf16(Y_dev.float().cpu().double().numpy(), Yref)
    else:
        check_Y(Y_dev.cpu().double().numpy(), Yref)


@pytest.mark.parametrize("i", range(N_CASES))
def test_random_shapes_every_entry_point(i, monkeypatch):
    c = _case(i)
    if c["bg_head"] == "auto":
        monkeypatch.delenv("MOE_BG_HEAD", raising=False)
    else:
        monkeypatch.setenv("MOE_BG_HEAD", c["bg_head"])
    wl = workloads.custom("fuzz", c["T"], c["d"], c["E"], c["k"], c["N"], c["R"], c["bias"])
    inp = workloads.make_inputs(wl, seed=100 + i)
    bf16 = c["out_dtype"] == binding.MOE_OUT_BF16
    plan, bufs, rc, status = run_path(wl, inp, tile_m=c["tile_m"], tile_n=c["tile_n"],
                                      out_dtype=c["out_dtype"])
    assert rc == 0, (c, status)
    if c["tile_m"]:
        assert plan.info["tile_m"] == c["tile_m"], c

    ref = oracle.route(inp["logits"].numpy(), wl.k)
    check_route(bufs, ref, wl.k)
    xb = workloads.bf16_bits(inp["x"])
    rows = oracle.gather(xb, ref["perm"], wl.k)
    check_recv(bufs, xb, ref, wl.k, wl.R, rows)
    Yref = oracle.grouped_gemm(rows, workloads.bf16_bits(inp["W"]), ref["offsets"])
    _check_out(bufs.Y, Yref, bf16)
    Y_dispatch = bufs.Y.clone()
    x, W = inp["x"].cuda(), inp["W"].cuda()

    # the direct gather on the same plan: the same tiles, the same bits
    bufs.Y.fill_(float("nan"))
    binding.gather_gemm(plan, x, W, bufs)
    rc, status = binding.moe_read_status(bufs.status)
    assert rc == 0, (c, status)
    assert torch.equal(bufs.Y, Y_dispatch), c

    # the grouped GEMM on the landed rows, gathered from the rank buffers in destination order
    off = ref["offsets"]
    epr = wl.E // wl.R
    A = torch.cat([bufs.recv[r][: int(off[(r + 1) * epr] - off[r * epr])] for r in range(wl.R)])
    assert A.shape[0] == wl.T * wl.k
    bufs.Y.fill_(float("nan"))
    binding.moe_grouped_gemm(plan, A, bufs.offsets, W, bufs.Y, bufs.workspace, bufs.status)
    rc, status = binding.moe_read_status(bufs.status)
    assert rc == 0, (c, status)
    assert torch.equal(bufs.Y, Y_dispatch), c

    # both combines against the oracle's combine of its own Y and gates
    want = oracle.combine(Yref, ref["topk_w"], ref["dest"])
    if not bf16:
        out = torch.full((wl.T, wl.N), float("nan"), dtype=torch.float32, device="cuda")
        binding.moe_combine(plan, Y_dispatch, bufs.topk_w, bufs.dest, out)
        check_Y(out.cpu().double().numpy(), want)
    out = torch.full((wl.T, wl.N), float("nan"), dtype=torch.float32, device="cuda")
    binding.dispatch_gemm_combine(plan, x, W, bufs, out)
    rc, status = binding.moe_read_status(bufs.status)
    assert rc == 0, (c, status)
    check_Y(out.cpu().double().numpy(), want)


def _ffn_case(i: int) -> dict:
    rng = np.random.default_rng(9000 + i)
    E = int(rng.choice([1, 2, 4, 8, 16, 64]))
    k = int(rng.integers(1, min(E, 8) + 1))
    T = int(rng.integers(1, 800 // k + 1))
    d = 16 * int(rng.integers(1, 25))   # 16 .. 384: the up-projection's K, the down one's N
    F = 16 * int(rng.integers(1, 25))   # 16 .. 384: H width, the down projection's K
    R = int(rng.choice([r for r in (1, 2, 4) if E % r == 0]))
    bias = str(rng.choice(["none", "zipf"]))
    tile_m = int(rng.choice([0, 128] + ([256] if 2 * F >= 256 else [])))
    tile_n = int(rng.choice([0, 256] + ([128] if tile_m != 256 else [])))
    return dict(T=T, d=d, E=E, k=k, F=F, R=R, bias=bias, tile_m=tile_m, tile_n=tile_n)


def _check_H(H_dev: torch.Tensor, Href: np.ndarray):
    """bf16 H: one rounding (2^-8 of the value) beyond the fp32 accumulation and activation."""
    Hg = H_dev.float().cpu().double().numpy()
    assert np.isfinite(Hg).all(), "unwritten (NaN) or non-finite H"
    rms = float(np.sqrt(np.mean(Href ** 2))) if Href.size else 0.0
    assert (np.abs(Hg - Href) <= 2.0 ** -8 * np.abs(Href) + 1e-4 * rms).all()


@pytest.mark.parametrize("i", range(N_FFN_CASES))
def test_random_shapes_gated_ffn_chain(i):
    c = _ffn_case(i)
    T, d, E, k, F, R = c["T"], c["d"], c["E"], c["k"], c["F"], c["R"]
    wl = workloads.custom("fuzzffn", T, d, E, k, 2 * F, R, c["bias"])
    inp = workloads.make_inputs(wl, seed=200 + i, with_weights=False)
    W1, W2 = workloads.make_ffn_weights(wl, F, seed=200 + i)
    up = binding.moe_plan(T, d, E, k, 2 * F, num_ranks=R, tile_m=c["tile_m"], tile_n=c["tile_n"])
    bu = binding.MoeBuffers(up, "cuda", out="H")
    bu.H.fill_(float("nan"))
    down = binding.moe_plan(T, F, E, k, d)
    bd = binding.MoeBuffers(down, "cuda")
    bd.Y.fill_(float("nan"))
    binding.route(up, inp["logits"].cuda(), bu)
    binding.dispatch_gemm_swiglu(up, inp["x"].cuda(), W1.cuda(), bu)
    binding.moe_grouped_gemm(down, bu.H, bu.offsets, W2.cuda(), bd.Y, bd.workspace, bd.status)
    out = torch.full((T, d), float("nan"), device="cuda")
    binding.moe_combine(down, bd.Y, bu.topk_w, bu.dest, out)
    for st in (bu.status, bd.status):
        rc, status = binding.moe_read_status(st)
        assert rc == 0, (c, status)

    ref = oracle.route(inp["logits"].numpy(), k)
    check_route(bu, ref, k)
    rows = oracle.gather(workloads.bf16_bits(inp["x"]), ref["perm"], k)
    Href = oracle.swiglu(oracle.grouped_gemm(rows, workloads.bf16_bits(W1), ref["offsets"]))
    _check_H(bu.H, Href)
    Hb, W2b = oracle.round_bf16(Href), workloads.bf16_bits(W2)
    Y2 = oracle.grouped_gemm(Hb, W2b, ref["offsets"])
    absHW = oracle.grouped_gemm(Hb & 0x7FFF, W2b & 0x7FFF, ref["offsets"])  # |H| . |W2|
    check_after_bf16_rounding(bd.Y.cpu().double().numpy(), Y2, absHW)
    check_after_bf16_rounding(out.cpu().double().numpy(), oracle.combine(Y2, ref["topk_w"], ref["dest"]),
                              oracle.combine(absHW, np.abs(ref["topk_w"]), ref["dest"]))
