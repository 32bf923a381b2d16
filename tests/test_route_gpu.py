"""GPU routing (moe_route) against the oracle: bit-exact indices, counts,
offsets, permutation and inverse on every workload and on edge cases."""
import numpy as np
import pytest
import torch

import oracle
from moe_token_dispatch_route_gb300 import binding, workloads
from tests.gpu_util import check_route

pytestmark = pytest.mark.gpu


def _route_only(T, E, k, logits_np):
    plan = binding.moe_plan(T, 64, E, k, 16)
    bufs = binding.MoeBuffers(plan, "cuda")
    for t in (bufs.topk_idx, bufs.perm, bufs.dest, bufs.counts, bufs.offsets):
        t.fill_(-7)
    binding.route(plan, torch.from_numpy(logits_np).cuda(), bufs)
    torch.cuda.synchronize()
    return bufs


@pytest.mark.parametrize("name", ["tiny", "mixtral", "finegrained", "deepseek_v3", "decode"])
def test_route_workloads(name):
    wl = workloads.WORKLOADS[name]
    inp = workloads.make_inputs(wl, seed=0, with_weights=False)
    L = inp["logits"].numpy()
    bufs = _route_only(wl.T, wl.E, wl.k, L)
    check_route(bufs, oracle.route(L, wl.k), wl.k)


def _coarse(rng, T, E):
    L = np.round(rng.standard_normal((T, E)) * 2).astype(np.float32) / np.float32(2)
    z = (L == 0) & (rng.random((T, E)) < 0.5)
    L[z] = np.float32(-0.0)
    return L


@pytest.mark.parametrize("T,E,k", [
    (1, 1, 1), (1, 8, 8), (63, 8, 2), (64, 8, 2), (65, 8, 2), (1000, 3, 2), (777, 64, 4),
    (300, 256, 8), (129, 1024, 32), (2048, 16, 16), (5000, 33, 5), (10, 32, 32),
])
def test_route_edge_shapes_with_ties(T, E, k):
    rng = np.random.default_rng(T * 1000 + E)
    L = _coarse(rng, T, E)  # many exact ties and signed zeros
    bufs = _route_only(T, E, k, L)
    check_route(bufs, oracle.route(L, k), k)


def test_route_all_tokens_one_expert():
    T, E, k = 500, 16, 1
    L = np.zeros((T, E), np.float32)
    L[:, 11] = 3.0
    bufs = _route_only(T, E, k, L)
    check_route(bufs, oracle.route(L, k), k)


def test_route_all_equal_logits():
    T, E, k = 333, 40, 7
    L = np.full((T, E), 0.25, np.float32)
    bufs = _route_only(T, E, k, L)
    ref = oracle.route(L, k)
    check_route(bufs, ref, k)
    assert (bufs.topk_idx.cpu().numpy() == np.arange(k)).all()


def test_route_empty_batch():
    plan = binding.moe_plan(0, 64, 8, 2, 16)
    bufs = binding.MoeBuffers(plan, "cuda")
    bufs.counts.fill_(5)
    bufs.offsets.fill_(5)
    binding.route(plan, torch.empty(0, 8, device="cuda"), bufs)
    torch.cuda.synchronize()
    assert bufs.counts.cpu().tolist() == [0] * 8
    assert bufs.offsets.cpu().tolist() == [0] * 9


def test_route_repeatable_bitwise():
    wl = workloads.WORKLOADS["finegrained"]
    L = workloads.make_inputs(wl, seed=1, with_weights=False)["logits"]
    plan = binding.moe_plan(wl.T, wl.d, wl.E, wl.k, wl.N)
    bufs = binding.MoeBuffers(plan, "cuda")
    Ld = L.cuda()
    outs = []
    for _ in range(3):
        binding.route(plan, Ld, bufs)
        outs.append([t.clone() for t in (bufs.topk_idx, bufs.topk_w, bufs.perm, bufs.offsets)])
    torch.cuda.synchronize()
    for o in outs[1:]:
        for a, b in zip(outs[0], o):
            assert torch.equal(a, b)
