"""moe_route_noalloc: the routing entry point for callers that are not
allowed to allocate device memory (for example a plugin in a host framework
that owns all device memory).  It keeps its scratch in a static device array
inside the library instead of a caller workspace.

Checked through the C ABI against moe_route (the workspace entry point) on
the same inputs, bit for bit (the two run the same kernels), and against the
CPU oracle (indices, counts, offsets, permutation and inverse bit-exact,
gates within 1e-5), for two calls in a row with different inputs, so that
leftovers of the first call in the shared array cannot go unnoticed.  This
file is collected last on purpose.
"""
import numpy as np
import pytest
import torch

import oracle
from moe_token_dispatch_route_gb300 import binding, workloads
from tests.gpu_util import TOL_GATE

pytestmark = pytest.mark.gpu

KEYS = ("topk_idx", "counts", "offsets", "perm", "dest")


def _outputs(plan, dev):
    s = plan.shape
    S = s.T * s.k
    i32 = dict(dtype=torch.int32, device=dev)
    return {"topk_idx": torch.full((s.T, s.k), -1, **i32),
            "topk_w": torch.full((s.T, s.k), float("nan"), dtype=torch.float32, device=dev),
            "counts": torch.full((s.E,), -1, **i32), "offsets": torch.full((s.E + 1,), -1, **i32),
            "perm": torch.full((S,), -1, **i32), "dest": torch.full((S,), -1, **i32)}


def _args(o):
    return (o["topk_idx"], o["topk_w"], o["counts"], o["offsets"], o["perm"], o["dest"])


@pytest.mark.parametrize("name,route_flags", [("finegrained", 0), ("deepseek_v3", 0),
                                              ("mixtral", binding.MOE_ROUTE_RENORM)])
def test_noalloc_route_matches_workspace_route_twice(name, route_flags):
    dev = torch.device("cuda", torch.cuda.current_device())
    wl = workloads.WORKLOADS[name]
    plan = binding.moe_plan(wl.T, wl.d, wl.E, wl.k, wl.N, num_ranks=wl.R, route_flags=route_flags)
    ws = torch.zeros(plan.workspace_bytes // 4 + 64, dtype=torch.int32, device=dev)
    for call, seed in enumerate((11, 12)):
        logits_h = workloads.make_inputs(wl, seed=seed, with_weights=False)["logits"]
        logits = logits_h.to(dev)
        want = _outputs(plan, dev)
        binding.moe_route(plan, logits, *_args(want), ws)
        got = _outputs(plan, dev)
        binding.moe_route_noalloc(plan, logits, *_args(got))
        torch.cuda.synchronize()
        for key in KEYS:
            assert torch.equal(got[key], want[key]), f"call {call}: {key}"
        # the same kernels on the same logits: the gates agree bit for bit too
        assert torch.equal(got["topk_w"].view(torch.int32), want["topk_w"].view(torch.int32)), \
            f"call {call}: gate weights differ from moe_route"
        ref = oracle.route(logits_h.numpy(), wl.k, renorm=bool(route_flags & binding.MOE_ROUTE_RENORM))
        for key in KEYS:
            g = got[key].cpu().numpy().reshape(ref[key].shape)
            assert np.array_equal(g, ref[key]), f"call {call}: {key} differs from the oracle"
        err = float(np.abs(got["topk_w"].cpu().double().numpy() - ref["topk_w"]).max())
        assert err <= TOL_GATE, f"call {call}: gate weights differ from the oracle by {err}"


def test_noalloc_route_rejects_plans_beyond_its_scratch():
    # ceil(T/64) * E = 1025 * 256 > 262144: refused before any launch
    plan = binding.moe_plan(64 * 1025, 64, 256, 8, 16)
    with pytest.raises(binding.MoeError) as exc:
        binding.moe_route_noalloc(plan, None, None, None, None, None, None, None)
    assert exc.value.status == binding.MOE_ERR_UNSUPPORTED
