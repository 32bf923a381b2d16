"""moe_combine (the step after the path) against the oracle's combine of the
oracle's own Y and gates: out[t][n] = sum_j w[t][j] * Y[dest[t*k+j]][n]."""
import numpy as np
import pytest
import torch

import oracle
from moe_token_dispatch_route_gb300 import binding, workloads
from tests.gpu_util import TOL_FRO, TOL_MAX_REL_RMS, check_Y, run_path

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
