"""Direct-gather grouped GEMM (moe_gather_gemm) on the GPU.

The A rows come straight from x (row perm[i] / k for destination row i) into
the GEMM's shared-memory tiles by 16-byte asynchronous copies; no receive buffer
is written.  Each output
element is reduced in the same order as in moe_dispatch_gemm with the same
tile shape, so the two agree bit for bit; both are also checked against the
oracle.
"""
import pytest
import torch

import oracle
from moe_token_dispatch_route_gb300 import binding, workloads
from tests.gpu_util import check_route, check_Y, check_Y_sampled, sample_rows_cols

pytestmark = pytest.mark.gpu


def _both(wl, inp, **plan_kw):
    """Route once, then run the dispatch and the gather entry points on one plan."""
    plan = binding.moe_plan(wl.T, wl.d, wl.E, wl.k, wl.N, num_ranks=wl.R, **plan_kw)
    bufs = binding.MoeBuffers(plan, "cuda")
    x, L = inp["x"].cuda(), inp["logits"].cuda()
    W = inp["W"] if inp["W"].is_cuda else inp["W"].cuda()
    binding.route(plan, L, bufs)
    bufs.Y.fill_(float("nan"))
    binding.gather_gemm(plan, x, W, bufs)
    rc, status = binding.moe_read_status(bufs.status)
    assert rc == 0, status
    Y_gather = bufs.Y.clone()
    bufs.Y.fill_(float("nan"))
    binding.dispatch_gemm(plan, x, W, bufs)
    rc, status = binding.moe_read_status(bufs.status)
    assert rc == 0, status
    return plan, bufs, Y_gather


@pytest.mark.parametrize("T,d,E,k,N,R,bias", [
    (100, 128, 3, 2, 272, 1, "none"),     # ragged rows and column tail
    (300, 64, 4, 1, 16, 1, "none"),       # minimum d and N
    (600, 128, 16, 4, 384, 4, "zipf"),    # skewed load, empty experts, four ranks
    (64, 256, 128, 8, 256, 1, "hot4"),    # decode-like
    (1, 128, 8, 8, 128, 8, "none"),       # one token, k = E
    (500, 128, 1, 1, 256, 1, "none"),     # one expert: a plain GEMM with 4 row tiles
    (700, 256, 8, 2, 704, 1, "none"),
    (300, 16, 4, 2, 256, 1, "none"),      # d = 16: one k-block of one K=16 step
    (400, 80, 8, 2, 384, 2, "zipf"),      # d = 80: a last k-block of 16 columns
    (257, 1040, 8, 2, 256, 1, "none"),    # d = 1040 = 16 * 65
])
def test_gather_matches_dispatch_bitwise_and_oracle(T, d, E, k, N, R, bias):
    wl = workloads.custom("gat", T, d, E, k, N, R, bias)
    inp = workloads.make_inputs(wl, seed=20)
    plan, bufs, Y_gather = _both(wl, inp, tile_m=128)
    assert torch.equal(Y_gather, bufs.Y)
    ref = oracle.route(inp["logits"].numpy(), k)
    check_route(bufs, ref, k)
    rows = oracle.gather(workloads.bf16_bits(inp["x"]), ref["perm"], k)
    Yref = oracle.grouped_gemm(rows, workloads.bf16_bits(inp["W"]), ref["offsets"])
    check_Y(Y_gather.cpu().double().numpy(), Yref)


@pytest.mark.parametrize("tile_n", [128, 192])
def test_gather_other_tile_widths(tile_n):
    wl = workloads.custom("gtn", 700, 256, 8, 2, 704, 1, "zipf")
    inp = workloads.make_inputs(wl, seed=21)
    _, bufs, Y_gather = _both(wl, inp, tile_m=128, tile_n=tile_n)
    assert torch.equal(Y_gather, bufs.Y)


@pytest.mark.parametrize("T,d,E,k,N,tile_n", [
    (1500, 128, 4, 2, 512, 256),     # several 256-row pair tiles per expert, M=128 tails
    (1000, 128, 2, 1, 400, 256),     # ragged column tail
    (1200, 128, 4, 2, 1408, 256),    # an N=128 last column tile
    (1000, 80, 2, 2, 1040, 512),     # 512-wide pair tiles, d = 80
    (130, 64, 1, 1, 256, 256),       # one expert of 130 rows: an M=128 tail after a full half
])
def test_gather_on_cta_pairs_matches_dispatch_bitwise(T, d, E, k, N, tile_n):
    """CTA-pair plans gather on CTA pairs (the peer's stages pass to the leader's stage
    barrier through its relay thread): bit for bit the pair dispatch with the same tiles,
    and the oracle."""
    wl = workloads.custom("gpair", T, d, E, k, N, 1, "none")
    inp = workloads.make_inputs(wl, seed=22)
    plan, bufs, Y_gather = _both(wl, inp, tile_m=256, tile_n=tile_n)
    assert plan.info["tile_m"] == 256
    assert torch.equal(Y_gather, bufs.Y)
    ref = oracle.route(inp["logits"].numpy(), k)
    rows = oracle.gather(workloads.bf16_bits(inp["x"]), ref["perm"], k)
    check_Y(Y_gather.cpu().double().numpy(),
            oracle.grouped_gemm(rows, workloads.bf16_bits(inp["W"]), ref["offsets"]))


def test_gather_repeated_calls_and_grid_sizes():
    wl = workloads.custom("grep", 900, 256, 8, 2, 512, 2, "none")
    inp = workloads.make_inputs(wl, seed=23)
    outs = []
    for kw in (dict(tile_m=128), dict(tile_m=128, num_ctas=16), dict(tile_m=128, num_ctas=3),
               dict(tile_m=256), dict(tile_m=256, num_ctas=6), dict(tile_m=256, num_ctas=2)):
        plan = binding.moe_plan(wl.T, wl.d, wl.E, wl.k, wl.N, num_ranks=wl.R, **kw)
        bufs = binding.MoeBuffers(plan, "cuda")
        x, W, L = inp["x"].cuda(), inp["W"].cuda(), inp["logits"].cuda()
        binding.route(plan, L, bufs)
        for _ in range(3):
            bufs.Y.fill_(float("nan"))
            binding.gather_gemm(plan, x, W, bufs)
            rc, status = binding.moe_read_status(bufs.status)
            assert rc == 0, status
            outs.append(bufs.Y.clone())
    for o in outs[1:4]:
        assert torch.equal(outs[0], o)
    for o in outs[4:]:  # CTA pairs: the same K order per element, the M=256 MMA's own rounding
        assert torch.equal(outs[3], o)


@pytest.mark.parametrize("name", ["mixtral", "finegrained", "deepseek_v3", "decode"])
def test_gather_full_size(name):
    """In the launch configuration of the benchmark (the plan's own choice of tiles,
    CTA pairs on the Mixtral-shaped and fine-grained layers): bit for bit against the
    dispatch on the same plan, and the oracle on a grid covering every tile."""
    wl = workloads.WORKLOADS[name]
    inp = workloads.make_inputs(wl, seed=0, w_device="cuda")
    plan, bufs, Y_gather = _both(wl, inp)
    assert torch.equal(Y_gather, bufs.Y)
    ref = oracle.route(inp["logits"].numpy(), wl.k)
    check_route(bufs, ref, wl.k)
    rows, cols = sample_rows_cols(ref, wl.N, tile_n=plan.info["tile_n"])
    check_Y_sampled(Y_gather, workloads.bf16_bits(inp["x"]), inp["W"], ref, wl.k, rows, cols)
