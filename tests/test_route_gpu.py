"""GPU routing (moe_route) against the oracle: bit-exact indices, counts,
offsets, permutation and inverse on every workload and on edge cases."""
import numpy as np
import pytest
import torch

import oracle
from moe_token_dispatch_route_gb300 import binding, workloads
from tests.gpu_util import check_route

pytestmark = pytest.mark.gpu


def _route_only(T, E, k, logits_np, route_flags=0, bias_np=None):
    plan = binding.moe_plan(T, 64, E, k, 16, route_flags=route_flags)
    bufs = binding.MoeBuffers(plan, "cuda")
    for t in (bufs.topk_idx, bufs.perm, bufs.dest, bufs.counts, bufs.offsets):
        t.fill_(-7)
    bias = None if bias_np is None else torch.from_numpy(bias_np).cuda()
    binding.route(plan, torch.from_numpy(logits_np).cuda(), bufs, selection_bias=bias)
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


@pytest.mark.parametrize("flags", [0, binding.MOE_ROUTE_RENORM])
@pytest.mark.parametrize("T,E,k", [(500, 8, 2), (400, 64, 4), (300, 300, 8)])
def test_route_extreme_magnitudes_subnormals_and_signed_zeros(T, E, k, flags):
    """Logits drawn from the extremes of fp32 (largest finite, smallest normal
    and subnormal, both zeros), with many exact ties: the selection order is
    the float order with ties to the lower index, and -0.0 ties with +0.0."""
    big = np.finfo(np.float32).max
    tiny = np.finfo(np.float32).tiny
    sub = np.float32(1e-45)
    pool = np.array([-big, -1e30, -1.5, -tiny, -1e-40, -sub, -0.0, 0.0, sub, 1e-40, tiny, 1.5, 1e30, big],
                    np.float32)
    rng = np.random.default_rng(T + E + k + flags)
    L = pool[rng.integers(0, pool.size, (T, E))]
    bufs = _route_only(T, E, k, L, route_flags=flags)
    check_route(bufs, oracle.route(L, k, renorm=bool(flags & binding.MOE_ROUTE_RENORM)), k)


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


# ---------------------------------------------------- renormalised gates (route flag)

@pytest.mark.parametrize("name", ["tiny", "mixtral", "deepseek_v3", "decode"])
def test_route_renorm_workloads(name):
    wl = workloads.WORKLOADS[name]
    L = workloads.make_inputs(wl, seed=2, with_weights=False)["logits"].numpy()
    bufs = _route_only(wl.T, wl.E, wl.k, L, route_flags=binding.MOE_ROUTE_RENORM)
    check_route(bufs, oracle.route(L, wl.k, renorm=True), wl.k)


@pytest.mark.parametrize("T,E,k", [(1, 1, 1), (100, 8, 1), (777, 64, 4), (129, 1024, 32), (10, 32, 32)])
def test_route_renorm_edge_shapes_with_ties(T, E, k):
    rng = np.random.default_rng(T * 7 + E)
    L = _coarse(rng, T, E)
    bufs = _route_only(T, E, k, L, route_flags=binding.MOE_ROUTE_RENORM)
    check_route(bufs, oracle.route(L, k, renorm=True), k)
    w = bufs.topk_w.cpu().double().numpy()
    if k == 1:
        assert np.all(w == 1.0)  # x / x
    assert np.allclose(w.sum(axis=1), 1.0, rtol=0, atol=1e-5)


# ------------------------------------- selection-only bias and logistic gates

FLAGS = [0, binding.MOE_ROUTE_RENORM, binding.MOE_ROUTE_SIGMOID,
         binding.MOE_ROUTE_SIGMOID | binding.MOE_ROUTE_RENORM]


def _oracle_route(L, k, flags, bias=None):
    return oracle.route(L, k, renorm=bool(flags & binding.MOE_ROUTE_RENORM),
                        sigmoid=bool(flags & binding.MOE_ROUTE_SIGMOID), selection_bias=bias)


@pytest.mark.parametrize("flags", FLAGS)
@pytest.mark.parametrize("name", ["mixtral", "deepseek_v3"])
def test_route_biased_workloads(name, flags):
    wl = workloads.WORKLOADS[name]
    L = workloads.make_inputs(wl, seed=3, with_weights=False)["logits"].numpy()
    b = (np.random.default_rng(31).standard_normal(wl.E) * 0.3).astype(np.float32)
    bufs = _route_only(wl.T, wl.E, wl.k, L, route_flags=flags, bias_np=b)
    check_route(bufs, _oracle_route(L, wl.k, flags, b), wl.k)


@pytest.mark.parametrize("flags", FLAGS)
@pytest.mark.parametrize("T,E,k", [(1, 1, 1), (65, 8, 2), (777, 64, 4), (129, 1024, 32), (10, 32, 32)])
def test_route_biased_edge_shapes_with_ties(T, E, k, flags):
    rng = np.random.default_rng(T * 13 + E)
    L = _coarse(rng, T, E)
    b = (np.round(rng.standard_normal(E) * 2) / 2).astype(np.float32)  # keys tie often
    b[rng.random(E) < 0.2] = np.float32(-0.0)
    bufs = _route_only(T, E, k, L, route_flags=flags, bias_np=b)
    check_route(bufs, _oracle_route(L, k, flags, b), k)


def test_route_bias_steers_tokens_to_cold_experts():
    """A bias on the 4 least-loaded experts of the unbiased routing moves
    tokens onto them; the gates stay those of the unbiased logits."""
    wl = workloads.WORKLOADS["deepseek_v3"]
    L = workloads.make_inputs(wl, seed=4, with_weights=False)["logits"].numpy()
    counts0 = oracle.route(L, wl.k)["counts"]
    cold = np.argsort(counts0, kind="stable")[:4]
    b = np.zeros(wl.E, np.float32)
    b[cold] = 1.5
    flags = binding.MOE_ROUTE_SIGMOID | binding.MOE_ROUTE_RENORM
    bufs = _route_only(wl.T, wl.E, wl.k, L, route_flags=flags, bias_np=b)
    ref = _oracle_route(L, wl.k, flags, b)
    check_route(bufs, ref, wl.k)
    assert np.all(ref["counts"][cold] > counts0[cold])
