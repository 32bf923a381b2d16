"""moe_router_logits (the step before the path) against the oracle's router in
the same fixed fp32 order: bit-exact logits, and bit-exact routing downstream."""
import numpy as np
import pytest
import torch

import oracle
from moe_token_dispatch_route_gb300 import binding, workloads
from tests.gpu_util import check_route

pytestmark = pytest.mark.gpu


def _gpu_logits(wl, inp, rows=None):
    plan = binding.moe_plan(wl.T, wl.d, wl.E, wl.k, wl.N, num_ranks=wl.R)
    x = inp["x"].cuda()
    Wr = inp["W_r"].cuda()
    bias = inp["bias"].cuda() if wl.bias != "none" else None
    L = torch.full((wl.T, wl.E), float("nan"), dtype=torch.float32, device="cuda")
    binding.moe_router_logits(plan, x, Wr, bias, L)
    torch.cuda.synchronize()
    return plan, L


def _oracle_logits(wl, inp, rows=None):
    xb = workloads.bf16_bits(inp["x"])
    if rows is not None:
        xb = np.ascontiguousarray(xb[rows])
    bias = inp["bias"].numpy() if wl.bias != "none" else None
    return oracle.router_logits(xb, workloads.bf16_bits(inp["W_r"]), bias)


def _bits(a):
    return np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)


@pytest.mark.parametrize("T,d,E,bias", [
    (1, 64, 1, "none"), (100, 128, 3, "none"), (257, 256, 8, "none"), (300, 192, 17, "zipf"),
    (64, 512, 128, "hot4"), (70, 64, 1024, "none"), (1000, 2048, 64, "zipf"),
    (333, 128, 24, "none"),    # streamed, narrow shape: 8-expert blocks, 128-element stages
    (700, 64, 40, "zipf"),     # streamed, narrow shape with 64-element stages (d = 64)
    (520, 256, 256, "none"),   # streamed, narrow shape: too few CTAs for the wide one
    (31, 4096, 16, "none"),    # streamed: a single partial row of tokens, a long reduction
    # streamed, wide shape (128 tokens x 32 experts per CTA, grid of at least 152 CTAs):
    (10000, 128, 40, "zipf"),  # the second expert block holds 8 experts, the last token block 16 tokens
    (19457, 64, 32, "none"),   # the last CTA holds 1 token (its second-token rows all past T); one stage
    (4864, 192, 256, "hot4"),  # three stages, fewer than the ring's depth
    # d % 64 != 0: the fallback kernel; d % 32 == 16 ends in a half chunk
    (300, 16, 8, "none"), (257, 80, 24, "zipf"), (500, 1040, 64, "none"), (100, 48, 3, "none"),
])
def test_router_logits_bit_exact(T, d, E, bias):
    wl = workloads.custom("router", T, d, E, 1, 16, 1, bias)
    inp = workloads.make_inputs(wl, seed=14, with_weights=False)
    _, L = _gpu_logits(wl, inp)
    assert np.array_equal(_bits(L.cpu().numpy()), _bits(_oracle_logits(wl, inp)))


@pytest.mark.parametrize("E", [8, 64])
def test_router_logits_unaligned_inputs_take_the_fallback_kernel(E):
    """x at a 4-byte (not 16-byte) offset: the scalar fallback kernel, bit-exact too."""
    wl = workloads.custom("router_unaligned", 200, 256, E, 1, 16, 1, "none")
    inp = workloads.make_inputs(wl, seed=15, with_weights=False)
    plan = binding.moe_plan(wl.T, wl.d, wl.E, wl.k, wl.N)
    raw = torch.empty(wl.T * wl.d + 2, dtype=torch.bfloat16, device="cuda")
    x = raw[2:].view(wl.T, wl.d)
    x.copy_(inp["x"])
    assert x.data_ptr() % 16 == 4
    L = torch.full((wl.T, wl.E), float("nan"), dtype=torch.float32, device="cuda")
    binding.moe_router_logits(plan, x, inp["W_r"].cuda(), None, L)
    torch.cuda.synchronize()
    assert np.array_equal(_bits(L.cpu().numpy()), _bits(_oracle_logits(wl, inp)))


def test_router_logits_mixtral_full():
    wl = workloads.WORKLOADS["mixtral"]
    inp = workloads.make_inputs(wl, seed=0, with_weights=False)
    _, L = _gpu_logits(wl, inp)
    assert np.array_equal(_bits(L.cpu().numpy()), _bits(_oracle_logits(wl, inp)))


def test_router_logits_deepseek_sampled_rows():
    wl = workloads.WORKLOADS["deepseek_v3"]
    inp = workloads.make_inputs(wl, seed=0, with_weights=False)
    _, L = _gpu_logits(wl, inp)
    rows = np.array(sorted(set(range(0, 64)) | set(np.random.default_rng(1).integers(0, wl.T, 64).tolist()) | {wl.T - 1}))
    assert np.array_equal(_bits(L.cpu().numpy()[rows]), _bits(_oracle_logits(wl, inp, rows)))


@pytest.mark.parametrize("name", ["finegrained", "decode"])
def test_gpu_router_then_route_matches_oracle_chain(name):
    wl = workloads.WORKLOADS[name]
    inp = workloads.make_inputs(wl, seed=0, with_weights=False)
    plan, L = _gpu_logits(wl, inp)
    bufs = binding.MoeBuffers(plan, "cuda")
    binding.route(plan, L, bufs)
    torch.cuda.synchronize()
    check_route(bufs, oracle.route(_oracle_logits(wl, inp), wl.k), wl.k)
