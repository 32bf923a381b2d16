"""The C-ABI library without a GPU: it loads, exports every function the
header declares, its structs match the ctypes layout, and host-side
argument validation rejects bad shapes before touching a device."""
import ctypes
import os
import re
import subprocess

import pytest

from moe_token_dispatch_route_gb300 import binding

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "moe.h")


@pytest.fixture(scope="module")
def lib():
    from moe_token_dispatch_route_gb300 import build
    build.build()
    return binding.load_library()


def _declared_functions():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"MOE_API\s+[\w\s\*]+?\b(moe_\w+)\s*\(", text)))


def test_header_declares_the_abi():
    assert _declared_functions() == sorted(binding.EXPORTED)


def test_library_exports_every_declared_symbol(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", binding.LIB_PATH],
                         capture_output=True, text=True, check=True).stdout
    exported = set(re.findall(r"\sT\s(moe_\w+)", out))
    for fn in _declared_functions():
        assert fn in exported, fn
        assert hasattr(lib, fn)


def test_struct_layout_matches_header(tmp_path):
    src = tmp_path / "layout.c"
    src.write_text(
        '#include <stdio.h>\n#include <stddef.h>\n#include "moe.h"\n'
        "int main(void){printf(\"%zu %zu %zu %zu %zu %zu %zu\\n\", sizeof(moe_shape_t),"
        " offsetof(moe_shape_t, timeout_ns), offsetof(moe_shape_t, debug_skip_publish),"
        " sizeof(moe_plan_info_t), offsetof(moe_plan_info_t, workspace_bytes),"
        " offsetof(moe_plan_info_t, half_tiles), offsetof(moe_plan_info_t, background_scatter));"
        "return 0;}\n")
    exe = tmp_path / "layout"
    subprocess.check_call(["gcc", "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe)])
    vals = [int(v) for v in subprocess.check_output([str(exe)]).split()]
    assert vals == [ctypes.sizeof(binding.Shape), binding.Shape.timeout_ns.offset,
                    binding.Shape.debug_skip_publish.offset, ctypes.sizeof(binding.PlanInfo),
                    binding.PlanInfo.workspace_bytes.offset, binding.PlanInfo.half_tiles.offset,
                    binding.PlanInfo.background_scatter.offset]


def _plan_rc(lib, **kw):
    fields = dict(T=64, d=128, E=8, k=2, N=256, num_ranks=1, rank_capacity_rows=0, tile_n=0,
                  producer_ctas=0, num_ctas=0, timeout_ns=0, debug_skip_publish=0, route_flags=0,
                  tile_m=0, out_dtype=0)
    fields.update(kw)
    shape = binding.Shape(**fields)
    h = ctypes.c_void_p()
    ws = ctypes.c_size_t()
    return lib.moe_plan(ctypes.byref(shape), 0, ctypes.byref(h), ctypes.byref(ws))


@pytest.mark.parametrize("kw,expect", [
    (dict(T=-1), binding.MOE_ERR_INVALID_ARG),
    (dict(d=0), binding.MOE_ERR_INVALID_ARG),
    (dict(k=0), binding.MOE_ERR_INVALID_ARG),
    (dict(route_flags=4), binding.MOE_ERR_INVALID_ARG),
    (dict(debug_skip_publish=-2), binding.MOE_ERR_INVALID_ARG),
    (dict(tile_n=512, tile_m=128), binding.MOE_ERR_UNSUPPORTED),   # 512-wide tiles: CTA pairs only
    (dict(tile_n=512, N=256), binding.MOE_ERR_UNSUPPORTED),
    (dict(tile_n=384), binding.MOE_ERR_UNSUPPORTED),
    (dict(E=1025, k=2), binding.MOE_ERR_UNSUPPORTED),
    (dict(E=8, k=9), binding.MOE_ERR_UNSUPPORTED),
    (dict(E=64, k=33), binding.MOE_ERR_UNSUPPORTED),
    (dict(d=100), binding.MOE_ERR_UNSUPPORTED),
    (dict(d=72), binding.MOE_ERR_UNSUPPORTED),                     # d % 16 != 0
    (dict(d=65536 + 16), binding.MOE_ERR_UNSUPPORTED),
    (dict(d=65536 + 64), binding.MOE_ERR_UNSUPPORTED),
    (dict(N=24), binding.MOE_ERR_UNSUPPORTED),
    (dict(num_ranks=3), binding.MOE_ERR_UNSUPPORTED),
    (dict(E=64, num_ranks=64), binding.MOE_ERR_UNSUPPORTED),
    (dict(tile_n=160), binding.MOE_ERR_UNSUPPORTED),
    (dict(out_dtype=2), binding.MOE_ERR_INVALID_ARG),
    (dict(tile_m=64), binding.MOE_ERR_UNSUPPORTED),
    (dict(tile_m=256, N=128), binding.MOE_ERR_UNSUPPORTED),
    (dict(tile_m=256, tile_n=128), binding.MOE_ERR_UNSUPPORTED),
    (dict(T=1 << 30, k=2), binding.MOE_ERR_UNSUPPORTED),
])
def test_plan_rejects_bad_shapes_before_any_device_call(lib, kw, expect):
    assert _plan_rc(lib, **kw) == expect


def test_null_arguments_are_rejected(lib):
    h = ctypes.c_void_p()
    ws = ctypes.c_size_t()
    assert lib.moe_plan(None, 0, ctypes.byref(h), ctypes.byref(ws)) == binding.MOE_ERR_INVALID_ARG
    nulls = [None] * 10
    assert lib.moe_route(*nulls) == binding.MOE_ERR_INVALID_ARG
    assert lib.moe_route_biased(*([None] * 11)) == binding.MOE_ERR_INVALID_ARG
    assert lib.moe_dispatch_gemm(*nulls) == binding.MOE_ERR_INVALID_ARG
    out = (ctypes.c_int32 * 4)()
    assert lib.moe_read_status(None, None, out) == binding.MOE_ERR_INVALID_ARG
    assert lib.moe_plan_destroy(None) == binding.MOE_OK


def test_status_strings(lib):
    for code, name in binding.STATUS_NAMES.items():
        assert lib.moe_status_string(code).decode() == name


def test_valid_shape_without_gpu_reports_cuda_error(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    assert _plan_rc(lib) == binding.MOE_ERR_CUDA
