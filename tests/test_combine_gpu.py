"""moe_combine (the step after the path) against the oracle's combine of the
oracle's own Y and gates: out[t][n] = sum_j w[t][j] * Y[dest[t*k+j]][n]."""
import numpy as np
import pytest
import torch

import oracle
from moe_token_dispatch_route_gb300 import binding, workloads
from tests.gpu_util import (TOL_FRO, TOL_MAX_REL_RMS, check_recv, check_route, check_Y, oracle_grid, run_path,
                            sample_rows_cols)

pytestmark = pytest.mark.gpu


def _combine_gpu(plan, bufs, T, N):
    out = torch.full((T, N), float("nan"), dtype=torch.float32, device=bufs.Y.device)
    binding.moe_combine(plan, bufs.Y, bufs.topk_w, bufs.dest, out)
    torch.cuda.synchronize()
    return out


@pytest.mark.parametrize("T,d,E,k,N,R", [
    (256, 512, 8, 2, 1024, 1),
    (300, 128, 16, 4, 272, 2),
    (64, 256, 128, 8, 256, 1),
    (900, 128, 4, 1, 512, 1),
])
def test_combine_full_parity(T, d, E, k, N, R):
    wl = workloads.custom("comb", T, d, E, k, N, R)
    inp = workloads.make_inputs(wl, seed=12)
    plan, bufs, rc, st = run_path(wl, inp)
    assert rc == 0, st
    out = _combine_gpu(plan, bufs, T, N).cpu().double().numpy()
    ref = oracle.route(inp["logits"].numpy(), k)
    rows = oracle.gather(workloads.bf16_bits(inp["x"]), ref["perm"], k)
    Yref = oracle.grouped_gemm(rows, workloads.bf16_bits(inp["W"]), ref["offsets"])
    check_Y(out, oracle.combine(Yref, ref["topk_w"], ref["dest"]))


def test_combine_mixtral_sampled():
    wl = workloads.WORKLOADS["mixtral"]
    inp = workloads.make_inputs(wl, seed=0, w_device="cuda")
    plan, bufs, rc, st = run_path(wl, inp)
    assert rc == 0, st
    out = _combine_gpu(plan, bufs, wl.T, wl.N)
    assert not torch.isnan(out).any().item()
    ref = oracle.route(inp["logits"].numpy(), wl.k)
    rng = np.random.default_rng(0)
    toks = sorted(set(rng.integers(0, wl.T, 24).tolist()) | {0, wl.T - 1})
    cols = sorted(set(rng.integers(0, wl.N, 12).tolist()) | {0, wl.N - 1})
    xb = workloads.bf16_bits(inp["x"])
    cols_t = torch.tensor(cols, device="cuda")
    Wc = {}
    got = out[torch.tensor(toks, device="cuda")][:, cols_t].cpu().double().numpy()
    want = np.zeros_like(got)
    for a, t in enumerate(toks):
        for j in range(wl.k):
            s = t * wl.k + j
            row = int(ref["dest"][s])
            e = oracle.expert_of_row(ref["offsets"], row)
            if e not in Wc:
                Wc[e] = workloads.bf16_bits(inp["W"][e][:, cols_t])
            a_row = oracle.gather(xb, ref["perm"][row:row + 1], wl.k)[0]
            for b in range(len(cols)):
                want[a, b] += ref["topk_w"][t, j] * oracle.gemm_entry(a_row, Wc[e], b)
    err = np.abs(got - want)
    rms = float(np.sqrt(np.mean(want ** 2)))
    assert float(err.max()) <= TOL_MAX_REL_RMS * rms
    assert float(np.linalg.norm(got - want)) <= TOL_FRO * float(np.linalg.norm(want))


def test_combine_is_repeatable_bitwise():
    wl = workloads.custom("combrep", 500, 128, 8, 2, 512, 1)
    inp = workloads.make_inputs(wl, seed=13)
    plan, bufs, rc, st = run_path(wl, inp)
    assert rc == 0, st
    a = _combine_gpu(plan, bufs, wl.T, wl.N)
    b = _combine_gpu(plan, bufs, wl.T, wl.N)
    assert torch.equal(a, b)


# ------------------------------------------------------------ combine fused into the GEMM epilogue

def _fused(wl, inp, **plan_kw):
    """route + moe_dispatch_gemm_combine; receive buffers and the output poisoned first
    (every output element must be written by its token's first term)."""
    dev = torch.device("cuda")
    plan = binding.moe_plan(wl.T, wl.d, wl.E, wl.k, wl.N, num_ranks=wl.R, **plan_kw)
    bufs = binding.MoeBuffers(plan, dev)
    for r in bufs.recv:
        r.fill_(float("nan"))
    out = torch.full((wl.T, wl.N), float("nan"), dtype=torch.float32, device=dev)
    W = inp["W"] if inp["W"].device.type == "cuda" else inp["W"].to(dev)
    binding.route(plan, inp["logits"].to(dev), bufs)
    binding.dispatch_gemm_combine(plan, inp["x"].to(dev), W, bufs, out)
    rc, status = binding.moe_read_status(bufs.status)
    return plan, bufs, out, rc, status


@pytest.mark.parametrize("T,d,E,k,N,R,tile_m,tile_n", [
    (256, 512, 8, 2, 1024, 1, 0, 0),        # the tiny workload's shape, single-CTA tiles
    (900, 128, 4, 1, 512, 1, 0, 0),         # k = 1: one reduction per output element
    (1200, 128, 4, 2, 1408, 2, 256, 256),   # CTA pairs: M=128 tails, an N=128 last column tile
    (1000, 128, 2, 2, 1040, 1, 256, 512),   # 512-wide pair tiles with a 16-wide tail
    (600, 80, 8, 2, 272, 1, 128, 128),      # d = 80; 128-wide single tiles, ragged column tail
    (64, 256, 128, 2, 256, 1, 0, 0),        # decode-like: many experts with 1-3 rows
    (600, 128, 16, 4, 384, 4, 0, 0),        # k = 4 (a store and three ordered additions), skewed
    (2000, 128, 8, 4, 640, 1, 256, 256),    # k = 4 on CTA pairs, M=128 tails, narrow last tile
    (64, 256, 128, 8, 256, 1, 0, 0),        # decode-like, k = 8
])
def test_fused_combine_full_parity(T, d, E, k, N, R, tile_m, tile_n):
    wl = workloads.custom("fcomb", T, d, E, k, N, R, "zipf" if k == 4 and tile_m == 0 else "none")
    inp = workloads.make_inputs(wl, seed=16)
    plan, bufs, out, rc, st = _fused(wl, inp, tile_m=tile_m, tile_n=tile_n)
    assert rc == 0, st
    if tile_m:
        assert plan.info["tile_m"] == tile_m
    ref = oracle.route(inp["logits"].numpy(), k)
    check_route(bufs, ref, k)
    xb = workloads.bf16_bits(inp["x"])
    rows = oracle.gather(xb, ref["perm"], k)
    check_recv(bufs, xb, ref, k, R, rows)
    Yref = oracle.grouped_gemm(rows, workloads.bf16_bits(inp["W"]), ref["offsets"])
    check_Y(out.cpu().double().numpy(), oracle.combine(Yref, ref["topk_w"], ref["dest"]))


@pytest.mark.parametrize("k", [2, 4])
def test_fused_combine_is_bitwise_repeatable_across_role_splits_and_grids(k):
    """The terms of a token are summed in ascending expert order whatever the timing:
    every split and grid size (and a second call) gives the same bits."""
    wl = workloads.custom("fcsplit", 1500, 256, 8, k, 640, 2, "none")
    inp = workloads.make_inputs(wl, seed=17)
    for tile_m in (128, 256):
        outs = []
        for kw in (dict(), dict(producer_ctas=2), dict(num_ctas=16, producer_ctas=4), dict(num_ctas=2)):
            for _ in range(2):
                _, _, out, rc, st = _fused(wl, inp, tile_m=tile_m, **kw)
                assert rc == 0, st
                outs.append(out)
        for o in outs[1:]:
            assert torch.equal(outs[0].view(torch.int32), o.view(torch.int32))


@pytest.mark.parametrize("name", ["mixtral", "finegrained", "deepseek_v3", "decode"])
def test_fused_combine_full_size_sampled(name):
    """Each large layer in the benchmark's launch configuration (k = 2, 4, 8, 8): every
    output element written (poisoned first), and sampled tokens whose slots fall in every
    (row tile, column tile) of the GEMM, with all k terms, against the oracle's combine."""
    wl = workloads.WORKLOADS[name]
    inp = workloads.make_inputs(wl, seed=0, w_device="cuda")
    plan, bufs, out, rc, st = _fused(wl, inp)
    assert rc == 0, st
    assert not torch.isnan(out).any().item(), "unwritten output"
    ref = oracle.route(inp["logits"].numpy(), wl.k)
    rows, cols = sample_rows_cols(ref, wl.N, tile_m=plan.info["tile_m"], tile_n=plan.info["tile_n"],
                                  n_random=16)
    toks = sorted({int(ref["perm"][r]) // wl.k for r in rows})
    # both slots of every sampled token, as destination rows, and the oracle's Y there
    slots = np.array([t * wl.k + j for t in toks for j in range(wl.k)])
    drows = [int(ref["dest"][s]) for s in slots]
    a_rows = oracle.gather(workloads.bf16_bits(inp["x"]), ref["perm"][drows], wl.k)
    Ysub = oracle_grid(a_rows, drows, inp["W"], ref, cols)
    want = oracle.combine(Ysub, ref["topk_w"][toks], np.arange(len(slots), dtype=np.int32))
    got = out[torch.tensor(toks, device="cuda")][:, torch.tensor(cols, device="cuda")].cpu().double().numpy()
    err = np.abs(got - want)
    rms = float(np.sqrt(np.mean(want ** 2)))
    assert float(err.max()) <= TOL_MAX_REL_RMS * rms, (float(err.max()), rms)
    assert float(np.linalg.norm(got - want)) <= TOL_FRO * float(np.linalg.norm(want))
