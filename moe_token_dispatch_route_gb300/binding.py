"""Thin ctypes binding of libmoe_gb300.so (the C ABI in include/moe.h).

Argument marshalling only: tensors are handed over as raw device pointers
together with the current CUDA stream; every step of the path runs in the
library's kernels.  Importing this module does not need a GPU; the first
call loads the library and raises if it has not been built.
"""
from __future__ import annotations

import ctypes
import os
from typing import Sequence

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmoe_gb300.so")
_lib = None

STATUS_NAMES = {
    0: "MOE_OK", 1: "MOE_ERR_INVALID_ARG", 2: "MOE_ERR_UNSUPPORTED", 3: "MOE_ERR_WORKSPACE",
    4: "MOE_ERR_CUDA", 5: "MOE_ERR_TIMEOUT", 6: "MOE_ERR_CAPACITY", 7: "MOE_ERR_DEVICE",
}
MOE_OK = 0
MOE_ERR_INVALID_ARG = 1
MOE_ERR_UNSUPPORTED = 2
MOE_ERR_WORKSPACE = 3
MOE_ERR_CUDA = 4
MOE_ERR_TIMEOUT = 5
MOE_ERR_CAPACITY = 6
MOE_ERR_DEVICE = 7
MOE_ROUTE_RENORM = 1
MOE_ROUTE_SIGMOID = 2
MOE_OUT_F32 = 0
MOE_OUT_BF16 = 1


class MoeError(RuntimeError):
    def __init__(self, status: int, call: str):
        super().__init__(f"{call} returned {STATUS_NAMES.get(status, status)}")
        self.status = status


class Shape(ctypes.Structure):
    _fields_ = [
        ("T", ctypes.c_int32), ("d", ctypes.c_int32), ("E", ctypes.c_int32),
        ("k", ctypes.c_int32), ("N", ctypes.c_int32), ("num_ranks", ctypes.c_int32),
        ("rank_capacity_rows", ctypes.c_int32), ("tile_n", ctypes.c_int32),
        ("producer_ctas", ctypes.c_int32), ("num_ctas", ctypes.c_int32),
        ("timeout_ns", ctypes.c_int64), ("debug_skip_publish", ctypes.c_int32),
        ("route_flags", ctypes.c_int32), ("tile_m", ctypes.c_int32), ("out_dtype", ctypes.c_int32),
    ]


class PlanInfo(ctypes.Structure):
    _fields_ = [
        ("tile_m", ctypes.c_int32), ("tile_n", ctypes.c_int32), ("tile_k", ctypes.c_int32),
        ("stages", ctypes.c_int32), ("num_ctas", ctypes.c_int32), ("producer_ctas", ctypes.c_int32),
        ("sm_count", ctypes.c_int32), ("smem_bytes", ctypes.c_int32), ("max_mtiles", ctypes.c_int32),
        ("route_blocks", ctypes.c_int32), ("workspace_bytes", ctypes.c_int64),
        ("half_tiles", ctypes.c_int32), ("background_scatter", ctypes.c_int32),
    ]

    def as_dict(self) -> dict:
        return {name: getattr(self, name) for name, _ in self._fields_}


EXPORTED = ("moe_plan", "moe_plan_destroy", "moe_plan_info", "moe_route", "moe_dispatch_gemm",
            "moe_read_status", "moe_status_string", "moe_route_noalloc", "moe_combine",
            "moe_router_logits", "moe_route_biased", "moe_dispatch_gemm_swiglu",
            "moe_grouped_gemm", "moe_gather_gemm", "moe_set_trace", "moe_dispatch_gemm_combine")


def load_library(path: str = LIB_PATH):
    """Load libmoe_gb300.so and declare its signatures (raises if it is missing)."""
    global _lib
    if _lib is not None and path == LIB_PATH:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(
            f"{path} is missing: build the CUDA library first (__graft_entry__.build() or "
            "python moe_token_dispatch_route_gb300/build.py); there is no fallback path")
    lib = ctypes.CDLL(path)
    P, I32, VP = ctypes.POINTER, ctypes.c_int32, ctypes.c_void_p
    lib.moe_plan.argtypes = [P(Shape), ctypes.c_int, P(VP), P(ctypes.c_size_t)]
    lib.moe_plan.restype = I32
    lib.moe_plan_destroy.argtypes = [VP]
    lib.moe_plan_destroy.restype = I32
    lib.moe_plan_info.argtypes = [VP, P(PlanInfo)]
    lib.moe_plan_info.restype = I32
    lib.moe_route.argtypes = [VP] * 10
    lib.moe_route.restype = I32
    lib.moe_route_biased.argtypes = [VP] * 11
    lib.moe_route_biased.restype = I32
    lib.moe_dispatch_gemm.argtypes = [VP] * 10
    lib.moe_dispatch_gemm.restype = I32
    lib.moe_dispatch_gemm_combine.argtypes = [VP] * 12
    lib.moe_dispatch_gemm_combine.restype = I32
    lib.moe_dispatch_gemm_swiglu.argtypes = [VP] * 10
    lib.moe_dispatch_gemm_swiglu.restype = I32
    lib.moe_grouped_gemm.argtypes = [VP] * 8
    lib.moe_grouped_gemm.restype = I32
    lib.moe_gather_gemm.argtypes = [VP] * 9
    lib.moe_gather_gemm.restype = I32
    lib.moe_set_trace.argtypes = [VP, VP, ctypes.c_int64]
    lib.moe_set_trace.restype = I32
    lib.moe_read_status.argtypes = [VP, VP, P(I32)]
    lib.moe_read_status.restype = I32
    lib.moe_router_logits.argtypes = [VP] * 6
    lib.moe_router_logits.restype = I32
    lib.moe_combine.argtypes = [VP] * 6
    lib.moe_combine.restype = I32
    lib.moe_route_noalloc.argtypes = [VP] * 9
    lib.moe_route_noalloc.restype = I32
    lib.moe_status_string.argtypes = [I32]
    lib.moe_status_string.restype = ctypes.c_char_p
    if path == LIB_PATH:
        _lib = lib
    return lib


def _ptr(t) -> int | None:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream, device=None) -> int:
    if stream is None:
        return torch.cuda.current_stream(device).cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(rc: int, call: str):
    if rc != MOE_OK:
        raise MoeError(rc, call)


class Plan:
    """Owns a moe_plan_t; `workspace_bytes` and `info` come from the library."""

    def __init__(self, handle: int, workspace_bytes: int, shape: Shape, device: int):
        self.handle = handle
        self.workspace_bytes = workspace_bytes
        self.shape = shape
        self.device = device
        info = PlanInfo()
        _check(load_library().moe_plan_info(handle, ctypes.byref(info)), "moe_plan_info")
        self.info = info.as_dict()

    def __del__(self):
        h, self.handle = getattr(self, "handle", None), None
        if h and _lib is not None:
            _lib.moe_plan_destroy(h)


def moe_plan(T: int, d: int, E: int, k: int, N: int, num_ranks: int = 1,
             rank_capacity_rows: int = 0, tile_n: int = 0, producer_ctas: int = 0,
             num_ctas: int = 0, timeout_ns: int = 0, debug_skip_publish: int = 0,
             route_flags: int = 0, tile_m: int = 0, out_dtype: int = MOE_OUT_F32,
             device: int | None = None) -> Plan:
    lib = load_library()
    dev = torch.cuda.current_device() if device is None else int(device)
    shape = Shape(T, d, E, k, N, num_ranks, rank_capacity_rows, tile_n, producer_ctas, num_ctas,
                  timeout_ns, debug_skip_publish, route_flags, tile_m, out_dtype)
    handle = ctypes.c_void_p()
    ws = ctypes.c_size_t()
    _check(lib.moe_plan(ctypes.byref(shape), dev, ctypes.byref(handle), ctypes.byref(ws)), "moe_plan")
    return Plan(handle.value, ws.value, shape, dev)


def moe_route(plan: Plan, logits, topk_idx, topk_w, counts, offsets, perm, dest, workspace,
              stream=None) -> None:
    rc = load_library().moe_route(plan.handle, _ptr(logits), _ptr(topk_idx), _ptr(topk_w),
                                  _ptr(counts), _ptr(offsets), _ptr(perm), _ptr(dest),
                                  _ptr(workspace), _stream(stream, plan.device))
    _check(rc, "moe_route")


def moe_route_biased(plan: Plan, logits, selection_bias, topk_idx, topk_w, counts, offsets, perm,
                     dest, workspace, stream=None) -> None:
    """moe_route ranking experts by logit + selection_bias[e]; gates from the logits."""
    rc = load_library().moe_route_biased(plan.handle, _ptr(logits), _ptr(selection_bias),
                                         _ptr(topk_idx), _ptr(topk_w), _ptr(counts),
                                         _ptr(offsets), _ptr(perm), _ptr(dest), _ptr(workspace),
                                         _stream(stream, plan.device))
    _check(rc, "moe_route_biased")


def moe_route_noalloc(plan: Plan, logits, topk_idx, topk_w, counts, offsets, perm, dest,
                      stream=None) -> None:
    """moe_route without a workspace: the library's static device scratch is used
    instead (for callers that cannot allocate device memory)."""
    rc = load_library().moe_route_noalloc(plan.handle, _ptr(logits), _ptr(topk_idx), _ptr(topk_w),
                                          _ptr(counts), _ptr(offsets), _ptr(perm), _ptr(dest),
                                          _stream(stream, plan.device))
    _check(rc, "moe_route_noalloc")


def moe_dispatch_gemm(plan: Plan, x, offsets, perm, W, recv: Sequence, Y, workspace, dev_status,
                      stream=None) -> None:
    arr = (ctypes.c_void_p * max(1, len(recv)))(*[_ptr(r) for r in recv])
    rc = load_library().moe_dispatch_gemm(plan.handle, _ptr(x), _ptr(offsets), _ptr(perm), _ptr(W),
                                          ctypes.cast(arr, ctypes.c_void_p), _ptr(Y),
                                          _ptr(workspace), _ptr(dev_status),
                                          _stream(stream, plan.device))
    _check(rc, "moe_dispatch_gemm")


def moe_dispatch_gemm_combine(plan: Plan, x, offsets, perm, dest, topk_w, W, recv: Sequence, out, workspace,
                              dev_status, stream=None) -> None:
    """Fused dispatch + grouped GEMM + combine: out[t] = sum_j w[t,j] * (x[t] W[e_j]), summed in
    ascending expert order (no Y)."""
    arr = (ctypes.c_void_p * max(1, len(recv)))(*[_ptr(r) for r in recv])
    rc = load_library().moe_dispatch_gemm_combine(plan.handle, _ptr(x), _ptr(offsets), _ptr(perm), _ptr(dest),
                                                  _ptr(topk_w), _ptr(W), ctypes.cast(arr, ctypes.c_void_p),
                                                  _ptr(out), _ptr(workspace), _ptr(dev_status),
                                                  _stream(stream, plan.device))
    _check(rc, "moe_dispatch_gemm_combine")


def dispatch_gemm_combine(plan: Plan, x, W, bufs: "MoeBuffers", out, stream=None):
    moe_dispatch_gemm_combine(plan, x, bufs.offsets, bufs.perm, bufs.dest, bufs.topk_w, W, bufs.recv, out,
                              bufs.workspace, bufs.status, stream)


def moe_dispatch_gemm_swiglu(plan: Plan, x, offsets, perm, W1, recv: Sequence, H, workspace,
                             dev_status, stream=None) -> None:
    """Fused dispatch + gated up-projection: H = silu(x W1_gate) * (x W1_up), bf16."""
    arr = (ctypes.c_void_p * max(1, len(recv)))(*[_ptr(r) for r in recv])
    rc = load_library().moe_dispatch_gemm_swiglu(plan.handle, _ptr(x), _ptr(offsets), _ptr(perm),
                                                 _ptr(W1), ctypes.cast(arr, ctypes.c_void_p),
                                                 _ptr(H), _ptr(workspace), _ptr(dev_status),
                                                 _stream(stream, plan.device))
    _check(rc, "moe_dispatch_gemm_swiglu")


def moe_grouped_gemm(plan: Plan, A, offsets, W, Y, workspace, dev_status, stream=None) -> None:
    """Per-expert grouped GEMM on rows already in destination order (no scatter)."""
    rc = load_library().moe_grouped_gemm(plan.handle, _ptr(A), _ptr(offsets), _ptr(W), _ptr(Y),
                                         _ptr(workspace), _ptr(dev_status),
                                         _stream(stream, plan.device))
    _check(rc, "moe_grouped_gemm")


def moe_gather_gemm(plan: Plan, x, offsets, perm, W, Y, workspace, dev_status, stream=None) -> None:
    """Grouped GEMM whose A rows are gathered from x by perm (no receive buffers)."""
    rc = load_library().moe_gather_gemm(plan.handle, _ptr(x), _ptr(offsets), _ptr(perm), _ptr(W),
                                        _ptr(Y), _ptr(workspace), _ptr(dev_status),
                                        _stream(stream, plan.device))
    _check(rc, "moe_gather_gemm")


def gather_gemm(plan: Plan, x, W, bufs: "MoeBuffers", stream=None):
    moe_gather_gemm(plan, x, bufs.offsets, bufs.perm, W, bufs.Y, bufs.workspace, bufs.status, stream)


TRACE_WORDS = 8
TRACE_FIELDS = ("start", "scatter_end", "first_tile", "flag_wait_ns", "tiles", "issue_end", "end", "role")


def moe_set_trace(plan: Plan, trace) -> None:
    """Per-CTA timing records of later GEMM launches into `trace` (a device int64
    tensor of at least sm_count * 8 words), or None to stop."""
    nbytes = 0 if trace is None else trace.numel() * trace.element_size()
    _check(load_library().moe_set_trace(plan.handle, _ptr(trace), nbytes), "moe_set_trace")


def moe_router_logits(plan: Plan, x, W_r, bias, logits, stream=None) -> None:
    rc = load_library().moe_router_logits(plan.handle, _ptr(x), _ptr(W_r), _ptr(bias), _ptr(logits),
                                          _stream(stream, plan.device))
    _check(rc, "moe_router_logits")


def moe_combine(plan: Plan, Y, topk_w, dest, out, stream=None) -> None:
    rc = load_library().moe_combine(plan.handle, _ptr(Y), _ptr(topk_w), _ptr(dest), _ptr(out),
                                    _stream(stream, plan.device))
    _check(rc, "moe_combine")


def moe_read_status(dev_status, stream=None) -> tuple[int, list[int]]:
    out = (ctypes.c_int32 * 4)()
    rc = load_library().moe_read_status(_ptr(dev_status), _stream(stream), out)
    return rc, list(out)


class MoeBuffers:
    """Device buffers of one layer shape, allocated with PyTorch (the caller's
    side of the ABI): routing outputs, R receive buffers, the GEMM output, workspace,
    status.  out="Y": fp32 Y [S][N] (moe_dispatch_gemm); out="H": bf16 H [S][N/2]
    (moe_dispatch_gemm_swiglu)."""

    def __init__(self, plan: Plan, device="cuda", out: str = "Y"):
        s = plan.shape
        S = s.T * s.k
        R = s.num_ranks or 1
        cap = s.rank_capacity_rows or S
        dev = torch.device(device)
        i32 = dict(dtype=torch.int32, device=dev)
        self.topk_idx = torch.empty(s.T, s.k, **i32)
        self.topk_w = torch.empty(s.T, s.k, dtype=torch.float32, device=dev)
        self.counts = torch.empty(s.E, **i32)
        self.offsets = torch.empty(s.E + 1, **i32)
        self.perm = torch.empty(S, **i32)
        self.dest = torch.empty(S, **i32)
        self.recv = [torch.empty(max(cap, 1), s.d, dtype=torch.bfloat16, device=dev) for _ in range(R)]
        y_dtype = torch.bfloat16 if s.out_dtype == MOE_OUT_BF16 else torch.float32
        self.Y = torch.empty(S, s.N, dtype=y_dtype, device=dev) if out == "Y" else None
        self.H = torch.empty(S, s.N // 2, dtype=torch.bfloat16, device=dev) if out == "H" else None
        self.workspace = torch.zeros(plan.workspace_bytes // 4 + 64, dtype=torch.int32, device=dev)
        self.status = torch.zeros(4, **i32)


def route(plan: Plan, logits, bufs: MoeBuffers, stream=None, selection_bias=None):
    moe_route_biased(plan, logits, selection_bias, bufs.topk_idx, bufs.topk_w, bufs.counts,
                     bufs.offsets, bufs.perm, bufs.dest, bufs.workspace, stream)


def dispatch_gemm(plan: Plan, x, W, bufs: MoeBuffers, stream=None):
    moe_dispatch_gemm(plan, x, bufs.offsets, bufs.perm, W, bufs.recv, bufs.Y, bufs.workspace,
                      bufs.status, stream)


def dispatch_gemm_swiglu(plan: Plan, x, W1, bufs: MoeBuffers, stream=None):
    moe_dispatch_gemm_swiglu(plan, x, bufs.offsets, bufs.perm, W1, bufs.recv, bufs.H,
                             bufs.workspace, bufs.status, stream)


def forward(plan: Plan, logits, x, W, bufs: MoeBuffers, stream=None):
    """One pass of the whole path: routing, then the fused dispatch + grouped GEMM."""
    route(plan, logits, bufs, stream)
    dispatch_gemm(plan, x, W, bufs, stream)
