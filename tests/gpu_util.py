"""Helpers of the GPU parity tests: run the CUDA path through the C ABI and
compare it with the CPU oracle.

Parity bar: routing indices, counts, offsets, permutation, inverse and the
receive buffers bit for bit; gate weights within 1e-5 absolute (fp32 expf
against fp64 exp); Y within max|err| <= 1e-2 * RMS(ref) and
||err||_F <= 5e-3 * ||ref||_F against the oracle's fp64 sums.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
from moe_token_dispatch_route_gb300 import binding, workloads

TOL_MAX_REL_RMS = 1e-2
TOL_FRO = 5e-3
TOL_GATE = 1e-5


def run_path(wl, inp, device="cuda", poison=True, **plan_kw):
    """Plan, allocate, poison outputs with NaN, run route + dispatch_gemm."""
    dev = torch.device(device)
    plan = binding.moe_plan(wl.T, wl.d, wl.E, wl.k, wl.N, num_ranks=wl.R, **plan_kw)
    bufs = binding.MoeBuffers(plan, dev)
    if poison:
        bufs.Y.fill_(float("nan"))
        for r in bufs.recv:
            r.fill_(float("nan"))
    x = inp["x"].to(dev)
    W = inp["W"] if inp["W"].device == dev else inp["W"].to(dev)
    logits = inp["logits"].to(dev)
    binding.forward(plan, logits, x, W, bufs)
    rc, status = binding.moe_read_status(bufs.status)
    return plan, bufs, rc, status


def check_route(bufs, ref, k):
    for key in ("topk_idx", "counts", "offsets", "perm", "dest"):
        got = getattr(bufs, key).cpu().numpy().reshape(ref[key].shape)
        assert np.array_equal(got, ref[key]), f"{key} differs from the oracle"
    w = bufs.topk_w.cpu().double().numpy()
    assert np.max(np.abs(w - ref["topk_w"])) <= TOL_GATE


def rank_rows(ref, E, R):
    return oracle.rank_base(ref["offsets"], R)


def check_recv(bufs, x_bits, ref, k, R, rows=None):
    """Each rank buffer's defined rows equal the oracle's gathered rows, bit for bit.
    `rows`: optional precomputed oracle gather (global destination order)."""
    E = ref["offsets"].shape[0] - 1
    base = rank_rows(ref, E, R)
    if rows is None:
        rows = oracle.gather(x_bits, ref["perm"], k)
    for r in range(R):
        n = int(base[r + 1] - base[r])
        got = bufs.recv[r][:n].cpu().view(torch.int16).numpy().view(np.uint16)
        assert np.array_equal(got, rows[base[r]:base[r + 1]]), f"rank {r} receive rows differ"


def check_Y(Y: np.ndarray, Yref: np.ndarray):
    assert Y.shape == Yref.shape
    assert np.isfinite(Y).all(), "unwritten (NaN) or non-finite output"
    err = np.abs(Y - Yref)
    rms = float(np.sqrt(np.mean(Yref ** 2)))
    assert float(err.max()) <= TOL_MAX_REL_RMS * rms, (float(err.max()), rms)
    assert float(np.linalg.norm(Y - Yref)) <= TOL_FRO * float(np.linalg.norm(Yref))
    return float(err.max()), rms


def check_after_bf16_rounding(Y: np.ndarray, Yref: np.ndarray, abs_bound: np.ndarray):
    """A product whose left operand the GPU rounded to bf16 from its fp32 value and the
    oracle from its fp64 one (SwiGLU's H before the down projection).  Where the unrounded
    value sits within fp32 error of a bf16 rounding midpoint the two round one bf16 ulp
    apart, at most 2^-7 of its magnitude; so each element may differ by 2^-7 times
    `abs_bound` (the oracle's |H| . |W| for that element) beyond the fp32 accumulation
    error (1e-4 RMS)."""
    assert Y.shape == Yref.shape
    assert np.isfinite(Y).all(), "unwritten (NaN) or non-finite output"
    rms = float(np.sqrt(np.mean(Yref ** 2))) if Yref.size else 0.0
    bound = 2.0 ** -7 * abs_bound + 1e-4 * rms
    worst = np.unravel_index(np.argmax(np.abs(Y - Yref) - bound), Y.shape) if Y.size else None
    assert (np.abs(Y - Yref) <= bound).all(), (worst, float(Y[worst]), float(Yref[worst]), float(bound[worst]))


def sample_rows_cols(ref, N, tile_m=128, tile_n=256, n_random=48, seed=0, row_block=32, col_block=64):
    """Rows and columns of a sampled check of Y that touches every output tile.

    Rows: every expert's first and last row and the rows on both sides of each
    tile_m boundary, random rows, and one seeded row inside every block of
    `row_block` rows of each expert (32: one per epilogue warp's lane quarter of
    every 128-row tile, so every row tile and both halves of every pair tile).
    Columns: the edges, the tile_n boundaries, random columns, and one seeded
    column inside every `col_block` columns (64: one per B box of every column
    tile).  The check evaluates the whole rows x columns grid, so it holds at
    least one entry of every (row tile, column tile) pair."""
    rng = np.random.default_rng(seed)
    off = ref["offsets"]
    S = int(off[-1])
    rows = set()
    for e in range(len(off) - 1):
        a, b = int(off[e]), int(off[e + 1])
        if b > a:
            rows.update({a, b - 1})
            for t in range(a + tile_m - 1, b, tile_m):
                rows.update({t, min(t + 1, b - 1)})
    rows = sorted(rows)
    if len(rows) > 96:
        rows = sorted(rng.choice(rows, 96, replace=False).tolist())
    rows = set(rows) | set(rng.integers(0, S, n_random).tolist())
    for e in range(len(off) - 1):
        a, b = int(off[e]), int(off[e + 1])
        for r0 in range(a, b, row_block):
            rows.add(int(rng.integers(r0, min(r0 + row_block, b))))
    cols = {0, N - 1, min(N - 1, tile_n - 1), min(N - 1, tile_n), N // 2}
    cols |= set(rng.integers(0, N, 12).tolist())
    for c0 in range(0, N, col_block):
        cols.add(int(rng.integers(c0, min(c0 + col_block, N))))
    return sorted(rows), sorted(cols)


def oracle_grid(a_rows_bits, rows, W_dev: torch.Tensor, ref, cols) -> np.ndarray:
    """The oracle's fp64 Y at rows x cols: one oracle grouped GEMM per expert on that
    expert's sampled rows (a_rows_bits, gathered in the order of `rows`) and the
    columns `cols` of its weights."""
    cols_t = torch.tensor(cols, device=W_dev.device)
    experts = np.array([oracle.expert_of_row(ref["offsets"], r) for r in rows])
    want = np.empty((len(rows), len(cols)), np.float64)
    for e in np.unique(experts):
        sel = np.nonzero(experts == e)[0]
        We = workloads.bf16_bits(W_dev[int(e)][:, cols_t])[None]
        want[sel] = oracle.grouped_gemm(a_rows_bits[sel], We, np.array([0, len(sel)], np.int32))
    return want


def check_Y_sampled(Y_dev: torch.Tensor, x_bits, W_dev: torch.Tensor, ref, k, rows, cols):
    """Oracle entries at the sampled (row, col) grid."""
    assert not torch.isnan(Y_dev).any().item(), "unwritten (NaN) output rows"
    a_rows = oracle.gather(x_bits, ref["perm"][rows], k)
    cols_t = torch.tensor(cols, device=Y_dev.device)
    got = Y_dev[torch.tensor(rows, device=Y_dev.device)][:, cols_t].cpu().double().numpy()
    want = oracle_grid(a_rows, rows, W_dev, ref, cols)
    err = np.abs(got - want)
    rms = float(np.sqrt(np.mean(want ** 2)))
    assert float(err.max()) <= TOL_MAX_REL_RMS * rms, (float(err.max()), rms)
    assert float(np.linalg.norm(got - want)) <= TOL_FRO * float(np.linalg.norm(want))
    return float(err.max()), rms
