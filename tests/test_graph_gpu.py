"""The path inside a CUDA graph: route + fused dispatch/GEMM captured once and
replayed.  Every call is stream-ordered with no host synchronisation, and the
workspace counters return to zero by themselves, so a captured step replays
with the same bits as an eager one and follows new inputs written into the
captured buffers."""
import pytest
import torch

import oracle
from moe_token_dispatch_route_gb300 import binding, workloads
from tests.gpu_util import check_route, check_Y

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("tile_m,tile_n", [(128, 0), (256, 0), (256, 512)])
def test_forward_replays_from_a_cuda_graph(tile_m, tile_n):
    wl = workloads.custom("graph", 1200, 256, 8, 2, 512, 2, "zipf")
    inp = workloads.make_inputs(wl, seed=15)
    plan = binding.moe_plan(wl.T, wl.d, wl.E, wl.k, wl.N, num_ranks=wl.R, tile_m=tile_m, tile_n=tile_n)
    bufs = binding.MoeBuffers(plan, "cuda")
    x, W, L = inp["x"].cuda(), inp["W"].cuda(), inp["logits"].cuda()

    binding.forward(plan, L, x, W, bufs)
    rc, status = binding.moe_read_status(bufs.status)
    assert rc == 0, status
    Y_eager = bufs.Y.clone()

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):  # warm-up on the capture stream's side, as torch asks
        binding.forward(plan, L, x, W, bufs)
    torch.cuda.current_stream().wait_stream(side)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        binding.forward(plan, L, x, W, bufs)
    for _ in range(3):
        bufs.Y.fill_(float("nan"))
        graph.replay()
        torch.cuda.synchronize()
        rc, status = binding.moe_read_status(bufs.status)
        assert rc == 0, status
        assert torch.equal(bufs.Y, Y_eager)

    # new logits and tokens written into the captured buffers: the replay follows them
    inp2 = workloads.make_inputs(wl, seed=16, with_weights=False)
    L.copy_(inp2["logits"].cuda())
    x.copy_(inp2["x"].cuda())
    bufs.Y.fill_(float("nan"))
    graph.replay()
    torch.cuda.synchronize()
    rc, status = binding.moe_read_status(bufs.status)
    assert rc == 0, status
    ref = oracle.route(inp2["logits"].numpy(), wl.k)
    check_route(bufs, ref, wl.k)
    rows = oracle.gather(workloads.bf16_bits(inp2["x"]), ref["perm"], wl.k)
    check_Y(bufs.Y.cpu().double().numpy(),
            oracle.grouped_gemm(rows, workloads.bf16_bits(inp["W"]), ref["offsets"]))
