"""ctypes front end of the plain C oracle (``moe_oracle.c``).

TEST INFRASTRUCTURE ONLY.  Each function below hands numpy arrays to one C
function of the oracle and returns numpy arrays; no arithmetic of the method
happens here.  See ``moe_oracle.c`` for the definition each step follows.

bf16 tensors travel as their uint16 bit patterns.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moe_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build_oracle(force: bool = False) -> str:
    """Compile moe_oracle.c into liboracle.so next to it (gcc, no FMA contraction)."""
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(
            ["gcc", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared",
             "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build_oracle())
            P = ctypes.c_void_p
            I = ctypes.c_int
            L = ctypes.c_long
            lib.oracle_topk.argtypes = [P, I, I, I, P, P]
            lib.oracle_topk.restype = I
            lib.oracle_topk_renorm_gates.argtypes = [P, I, I, I, P, P]
            lib.oracle_topk_renorm_gates.restype = I
            lib.oracle_select_biased.argtypes = [P, P, I, I, I, P]
            lib.oracle_select_biased.restype = I
            lib.oracle_gates_at.argtypes = [P, P, I, I, I, I, I, P]
            lib.oracle_gates_at.restype = I
            lib.oracle_histogram.argtypes = [P, I, I, I, P, P]
            lib.oracle_histogram.restype = I
            lib.oracle_permutation.argtypes = [P, I, I, I, P, P]
            lib.oracle_permutation.restype = I
            lib.oracle_rank_base.argtypes = [P, I, I, P]
            lib.oracle_rank_base.restype = I
            lib.oracle_gather.argtypes = [P, I, I, I, P, L, P]
            lib.oracle_gather.restype = None
            lib.oracle_grouped_gemm.argtypes = [P, P, P, I, I, I, P]
            lib.oracle_grouped_gemm.restype = I
            lib.oracle_gemm_entry.argtypes = [P, P, I, I, I]
            lib.oracle_gemm_entry.restype = ctypes.c_double
            lib.oracle_router_logits.argtypes = [P, P, P, I, I, I, P]
            lib.oracle_router_logits.restype = None
            lib.oracle_combine.argtypes = [P, P, P, I, I, I, P]
            lib.oracle_combine.restype = None
            lib.oracle_swiglu.argtypes = [P, L, I, P]
            lib.oracle_swiglu.restype = None
            lib.oracle_round_bf16.argtypes = [P, L, P]
            lib.oracle_round_bf16.restype = None
            lib.oracle_expert_of_row.argtypes = [P, I, L]
            lib.oracle_expert_of_row.restype = I
            _lib = lib
    return _lib


def _p(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data_as(ctypes.c_void_p)


def topk(logits: np.ndarray, k: int):
    """Step A1 -> (topk_idx int32 [T,k], topk_w float64 [T,k])."""
    L = np.ascontiguousarray(logits, dtype=np.float32)
    T, E = L.shape
    idx = np.empty((T, k), np.int32)
    w = np.empty((T, k), np.float64)
    rc = _load().oracle_topk(_p(L), T, E, k, _p(idx), _p(w))
    if rc != 0:
        raise ValueError(f"oracle_topk failed ({rc})")
    return idx, w


def renorm_gates(logits: np.ndarray, topk_idx: np.ndarray):
    """Step A1, renormalised variant: softmax over each token's k chosen logits
    -> topk_w float64 [T,k]."""
    L = np.ascontiguousarray(logits, dtype=np.float32)
    idx = np.ascontiguousarray(topk_idx, dtype=np.int32)
    T, E = L.shape
    k = idx.shape[1]
    assert idx.shape[0] == T
    w = np.empty((T, k), np.float64)
    if _load().oracle_topk_renorm_gates(_p(L), T, E, k, _p(idx), _p(w)) != 0:
        raise ValueError("expert index out of range")
    return w


def select_biased(logits: np.ndarray, bias: np.ndarray, k: int):
    """Step A1 ranked by the fp32 key logit + bias[e] -> topk_idx int32 [T,k]."""
    L = np.ascontiguousarray(logits, dtype=np.float32)
    b = np.ascontiguousarray(bias, dtype=np.float32)
    T, E = L.shape
    assert b.shape == (E,)
    idx = np.empty((T, k), np.int32)
    rc = _load().oracle_select_biased(_p(L), _p(b), T, E, k, _p(idx))
    if rc != 0:
        raise ValueError(f"oracle_select_biased failed ({rc})")
    return idx


def gates_at(logits: np.ndarray, topk_idx: np.ndarray, sigmoid: bool = False,
             renorm: bool = False):
    """Gates of the given picks from the logits (softmax over all E, or the
    logistic), optionally divided by their per-token sum -> float64 [T,k]."""
    L = np.ascontiguousarray(logits, dtype=np.float32)
    idx = np.ascontiguousarray(topk_idx, dtype=np.int32)
    T, E = L.shape
    k = idx.shape[1]
    w = np.empty((T, k), np.float64)
    if _load().oracle_gates_at(_p(L), _p(idx), T, E, k, int(sigmoid), int(renorm), _p(w)) != 0:
        raise ValueError("expert index out of range")
    return w


def histogram(topk_idx: np.ndarray, E: int):
    """Step A2 -> (counts int32 [E], offsets int32 [E+1])."""
    idx = np.ascontiguousarray(topk_idx, dtype=np.int32)
    T, k = idx.shape
    counts = np.empty(E, np.int32)
    offsets = np.empty(E + 1, np.int32)
    rc = _load().oracle_histogram(_p(idx), T, k, E, _p(counts), _p(offsets))
    if rc != 0:
        raise ValueError("expert index out of range")
    return counts, offsets


def permutation(topk_idx: np.ndarray, E: int):
    """Step A3 -> (perm int32 [T*k], dest int32 [T*k])."""
    idx = np.ascontiguousarray(topk_idx, dtype=np.int32)
    T, k = idx.shape
    perm = np.empty(T * k, np.int32)
    dest = np.empty(T * k, np.int32)
    rc = _load().oracle_permutation(_p(idx), T, k, E, _p(perm), _p(dest))
    if rc != 0:
        raise ValueError("permutation incomplete")
    return perm, dest


def rank_base(offsets: np.ndarray, R: int):
    """First global destination row of each simulated rank; [R+1] int32."""
    off = np.ascontiguousarray(offsets, dtype=np.int32)
    E = off.shape[0] - 1
    out = np.empty(R + 1, np.int32)
    if _load().oracle_rank_base(_p(off), E, R, _p(out)) != 0:
        raise ValueError("R must divide E")
    return out


def gather(x_bits: np.ndarray, perm: np.ndarray, k: int):
    """Step A4: destination rows (uint16 bf16 bits) in global destination order."""
    x = np.ascontiguousarray(x_bits, dtype=np.uint16)
    T, d = x.shape
    pm = np.ascontiguousarray(perm, dtype=np.int32)
    S = pm.shape[0]
    rows = np.empty((S, d), np.uint16)
    _load().oracle_gather(_p(x), T, d, k, _p(pm), S, _p(rows))
    return rows


def grouped_gemm(rows_bits: np.ndarray, W_bits: np.ndarray, offsets: np.ndarray):
    """Step A5 on every destination row -> Y float64 [S, N]."""
    rows = np.ascontiguousarray(rows_bits, dtype=np.uint16)
    W = np.ascontiguousarray(W_bits, dtype=np.uint16)
    off = np.ascontiguousarray(offsets, dtype=np.int32)
    E, d, N = W.shape
    S = rows.shape[0]
    Y = np.empty((S, N), np.float64)
    if _load().oracle_grouped_gemm(_p(rows), _p(W), _p(off), E, d, N, _p(Y)) != 0:
        raise MemoryError
    return Y


def grouped_gemm_parallel(rows_bits: np.ndarray, W_bits: np.ndarray, offsets: np.ndarray,
                          threads: int):
    """Step A5 with the output rows split into `threads` contiguous ranges, each
    computed by the same C function as grouped_gemm in a thread of its own (ctypes
    releases the GIL for the call).  Every element is the same fp64 sum in the same
    order, so the result equals grouped_gemm's bit for bit; only the wall time
    changes.  Used to time the oracle on all host cores."""
    import concurrent.futures as cf

    rows = np.ascontiguousarray(rows_bits, dtype=np.uint16)
    W = np.ascontiguousarray(W_bits, dtype=np.uint16)
    off = np.ascontiguousarray(offsets, dtype=np.int32)
    E, d, N = W.shape
    S = rows.shape[0]
    Y = np.empty((S, N), np.float64)
    threads = max(1, min(int(threads), S))
    bounds = [S * i // threads for i in range(threads + 1)]
    lib = _load()

    def part(i):
        r0, r1 = bounds[i], bounds[i + 1]
        if r1 <= r0:
            return 0
        # the part's rows and the expert segments clipped to them, shifted to start at 0
        sub_off = np.ascontiguousarray(np.clip(off.astype(np.int64) - r0, 0, r1 - r0), dtype=np.int32)
        sub_rows = rows[r0:r1]
        out = Y[r0:r1]
        return lib.oracle_grouped_gemm(_p(sub_rows), _p(W), _p(sub_off), E, d, N, _p(out))

    with cf.ThreadPoolExecutor(max_workers=threads) as ex:
        rcs = list(ex.map(part, range(threads)))
    if any(rc != 0 for rc in rcs):
        raise MemoryError
    return Y


def gemm_entry(row_bits: np.ndarray, We_bits: np.ndarray, n: int) -> float:
    """One element of step A5: row . We[:, n] in fp64."""
    row = np.ascontiguousarray(row_bits, dtype=np.uint16)
    We = np.ascontiguousarray(We_bits, dtype=np.uint16)
    d, N = We.shape
    assert row.shape == (d,)
    return float(_load().oracle_gemm_entry(_p(row), _p(We), d, N, int(n)))


def expert_of_row(offsets: np.ndarray, row: int) -> int:
    off = np.ascontiguousarray(offsets, dtype=np.int32)
    return int(_load().oracle_expert_of_row(_p(off), off.shape[0] - 1, int(row)))


def route(logits: np.ndarray, k: int, renorm: bool = False, sigmoid: bool = False,
          selection_bias=None):
    """Steps A1-A3 chained: returns a dict of the oracle's routing outputs.
    renorm: each token's gates divided by their sum over the k picks (for the
    softmax: the softmax over the k chosen logits); sigmoid: logistic gates;
    selection_bias: [E] added to the logits for the choice only."""
    E = logits.shape[1]
    idx, w = topk(logits, k)
    if selection_bias is not None:
        idx = select_biased(logits, selection_bias, k)
    if sigmoid or selection_bias is not None:
        w = gates_at(logits, idx, sigmoid=sigmoid, renorm=renorm)
    elif renorm:
        w = renorm_gates(logits, idx)
    counts, offsets = histogram(idx, E)
    perm, dest = permutation(idx, E)
    return {"topk_idx": idx, "topk_w": w, "counts": counts, "offsets": offsets,
            "perm": perm, "dest": dest}


def combine(Y: np.ndarray, topk_w: np.ndarray, dest: np.ndarray):
    """Combine: out[t][n] = sum_j w[t,j] * Y[dest[t*k+j]][n] (fp64) -> [T, N]."""
    Yd = np.ascontiguousarray(Y, dtype=np.float64)
    w = np.ascontiguousarray(topk_w, dtype=np.float64)
    T, k = w.shape
    N = Yd.shape[1]
    ds = np.ascontiguousarray(dest, dtype=np.int32).reshape(-1)
    assert ds.shape[0] == T * k
    out = np.empty((T, N), np.float64)
    _load().oracle_combine(_p(Yd), _p(w), _p(ds), T, k, N, _p(out))
    return out


def swiglu(G: np.ndarray):
    """Gated activation of up-projection rows: G [S, 2F] (gate | up) -> H float64 [S, F]."""
    Gd = np.ascontiguousarray(G, dtype=np.float64)
    S, F2 = Gd.shape
    assert F2 % 2 == 0
    H = np.empty((S, F2 // 2), np.float64)
    _load().oracle_swiglu(_p(Gd), S, F2 // 2, _p(H))
    return H


def round_bf16(v: np.ndarray):
    """Round fp64 values to bf16 (nearest, ties to even) -> uint16 bit patterns."""
    a = np.ascontiguousarray(v, dtype=np.float64)
    out = np.empty(a.shape, np.uint16)
    _load().oracle_round_bf16(_p(a), a.size, _p(out))
    return out


def router_logits(x_bits: np.ndarray, Wr_bits: np.ndarray, bias=None):
    """Router logits in the library's fixed fp32 order: fma over i ascending, then + bias."""
    x = np.ascontiguousarray(x_bits, dtype=np.uint16)
    W = np.ascontiguousarray(Wr_bits, dtype=np.uint16)
    T, d = x.shape
    E = W.shape[1]
    out = np.empty((T, E), np.float32)
    b = None if bias is None else np.ascontiguousarray(bias, dtype=np.float32)
    _load().oracle_router_logits(_p(x), _p(W), None if b is None else _p(b), T, d, E, _p(out))
    return out
