"""Pins of the CPU oracle against facts that do not come from the oracle itself.

Each test checks one step of the oracle against an independent statement of
what the step must produce: a hand-worked example, a brute-force computation
by a different algorithm, a closed form, an invariant, or a special case that
reduces to a library routine.  None of these calls the CUDA path.
"""
import collections
import itertools
import math
import os
from fractions import Fraction

import numpy as np
import pytest

HERE = os.path.dirname(os.path.abspath(__file__))


def _bf16_bits_from_f32(a: np.ndarray) -> np.ndarray:
    """Round fp32 -> bf16 bits with round-to-nearest-even (test-side helper)."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32).astype(np.uint64)
    r = ((u >> 16) & 1) + 0x7FFF
    return ((u + r) >> 16).astype(np.uint16)


def _bits_to_f64(b: np.ndarray) -> np.ndarray:
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def _read_golden(name):
    data = {}
    logits = {}
    with open(os.path.join(HERE, "golden", name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, *vals = line.split()
            if key == "logits":
                logits[int(vals[0])] = [float(v) for v in vals[1:]]
            elif key in ("T", "E", "k"):
                data[key] = int(vals[0])
            else:
                data[key] = [int(v) for v in vals]
    data["logits"] = np.array([logits[t] for t in range(data["T"])], np.float32)
    return data


# ---------------------------------------------------------------- A1 .. A3

def test_handworked_example(oracle_mod):
    g = _read_golden("route_handworked.txt")
    r = oracle_mod.route(g["logits"], g["k"])
    assert r["topk_idx"].ravel().tolist() == g["topk_idx"]
    assert r["counts"].tolist() == g["counts"]
    assert r["offsets"].tolist() == g["offsets"]
    assert r["perm"].tolist() == g["perm"]
    assert r["dest"].tolist() == g["dest"]


def _random_logits(rng, T, E, coarse):
    L = rng.standard_normal((T, E)).astype(np.float32)
    if coarse:  # a coarse grid makes exact ties common; include signed zeros
        L = np.round(L * 2.0).astype(np.float32) / np.float32(2.0)
        neg0 = rng.random((T, E)) < 0.1
        L[neg0 & (L == 0)] = np.float32(-0.0)
    return L


@pytest.mark.parametrize("seed", range(6))
def test_topk_matches_full_sort(oracle_mod, seed):
    """Brute force: a full sort of (−logit, index) per token, first k entries."""
    rng = np.random.default_rng(seed)
    T, E = 40, int(rng.integers(1, 13))
    k = int(rng.integers(1, E + 1))
    L = _random_logits(rng, T, E, coarse=seed % 2 == 0)
    idx, _ = oracle_mod.topk(L, k)
    for t in range(T):
        # Python's float compare treats -0.0 == 0.0, as the definition asks
        want = [e for _, e in sorted((-float(L[t, e]), e) for e in range(E))][:k]
        assert idx[t].tolist() == want


def test_topk_invariants(oracle_mod):
    rng = np.random.default_rng(11)
    T, E, k = 300, 64, 6
    L = _random_logits(rng, T, E, coarse=True)
    idx, _ = oracle_mod.topk(L, k)
    for t in range(T):
        chosen = set(idx[t].tolist())
        assert len(chosen) == k
        lo = min(L[t, e] for e in chosen)
        assert all(L[t, e] <= lo for e in range(E) if e not in chosen)
        # slots are in non-increasing logit order
        assert all(L[t, idx[t, j]] >= L[t, idx[t, j + 1]] for j in range(k - 1))


def test_topk_special_cases(oracle_mod):
    # all logits equal -> experts 0..k-1 and uniform gate weights 1/E
    L = np.full((3, 10), 0.37, np.float32)
    idx, w = oracle_mod.topk(L, 4)
    assert (idx == np.arange(4)).all()
    assert np.allclose(w, 0.1, rtol=0, atol=1e-15)
    # k == E -> every expert, sorted by logit, and the weights sum to one
    rng = np.random.default_rng(3)
    L = rng.standard_normal((20, 7)).astype(np.float32)
    idx, w = oracle_mod.topk(L, 7)
    assert (np.sort(idx, axis=1) == np.arange(7)).all()
    assert np.allclose(w.sum(axis=1), 1.0, rtol=0, atol=1e-14)
    # E == 1
    idx, w = oracle_mod.topk(np.array([[5.0], [-3.0]], np.float32), 1)
    assert idx.ravel().tolist() == [0, 0] and np.all(w == 1.0)


def test_gate_weight_two_experts_is_logistic(oracle_mod):
    """With E = 2 the softmax weight of the winner is the logistic 1/(1+e^-(a-b))."""
    a = np.linspace(-4, 4, 17, dtype=np.float32)
    L = np.stack([a, np.zeros_like(a)], axis=1)
    idx, w = oracle_mod.topk(L, 1)
    for t in range(len(a)):
        diff = abs(float(a[t]))
        assert w[t, 0] == pytest.approx(1.0 / (1.0 + math.exp(-diff)), abs=1e-15)


def test_renorm_gates_closed_forms(oracle_mod):
    """Gates renormalised over the k picks (Mixtral-style): k = 1 gives exactly 1;
    k = 2 gives the logistic of the two chosen logits' difference; k = E gives the
    softmax over all experts."""
    rng = np.random.default_rng(21)
    L = rng.standard_normal((40, 9)).astype(np.float32) * 3
    idx, _ = oracle_mod.topk(L, 1)
    assert np.all(oracle_mod.renorm_gates(L, idx) == 1.0)
    idx, _ = oracle_mod.topk(L, 2)
    w = oracle_mod.renorm_gates(L, idx)
    for t in range(L.shape[0]):
        a, b = float(L[t, idx[t, 0]]), float(L[t, idx[t, 1]])
        assert w[t, 0] == pytest.approx(1.0 / (1.0 + math.exp(b - a)), abs=1e-15)
        assert w[t, 1] == pytest.approx(1.0 / (1.0 + math.exp(a - b)), abs=1e-15)
    idx, w_all = oracle_mod.topk(L, 9)
    e = np.exp(L.astype(np.float64) - L.max(axis=1, keepdims=True))
    full = e / e.sum(axis=1, keepdims=True)
    assert np.allclose(oracle_mod.renorm_gates(L, idx), np.take_along_axis(full, idx, axis=1),
                       rtol=0, atol=1e-15)


def test_renorm_gates_ignore_unchosen_logits(oracle_mod):
    """Renormalised gates depend only on the chosen logits: lowering the rest
    changes neither the picks nor the gates, and every token's gates sum to 1
    with ratios exp(L_j - L_0)."""
    rng = np.random.default_rng(22)
    T, E, k = 60, 32, 4
    L = rng.standard_normal((T, E)).astype(np.float32)
    idx, _ = oracle_mod.topk(L, k)
    w = oracle_mod.renorm_gates(L, idx)
    L2 = L.copy()
    mask = np.ones_like(L, bool)
    np.put_along_axis(mask, idx, False, axis=1)
    L2[mask] -= 5.0
    idx2, _ = oracle_mod.topk(L2, k)
    assert np.array_equal(idx, idx2)
    assert np.array_equal(oracle_mod.renorm_gates(L2, idx2), w)
    assert np.allclose(w.sum(axis=1), 1.0, rtol=0, atol=1e-14)
    lo = np.take_along_axis(L, idx, axis=1).astype(np.float64)
    assert np.allclose(w / w[:, :1], np.exp(lo - lo[:, :1]), rtol=1e-14, atol=0)


def test_biased_selection_brute_force(oracle_mod):
    """Selection on fp32(logit + bias): zero bias gives the plain top-k; on tiny
    inputs with many ties the picks equal a stable sort of the keys (numpy's
    fp32 addition, largest key first, lower index first between equals)."""
    rng = np.random.default_rng(23)
    for trial in range(30):
        T, E = int(rng.integers(1, 20)), int(rng.integers(1, 12))
        k = int(rng.integers(1, E + 1))
        L = _random_logits(rng, T, E, coarse=True)
        assert np.array_equal(oracle_mod.select_biased(L, np.zeros(E, np.float32), k),
                              oracle_mod.topk(L, k)[0])
        b = (np.round(rng.standard_normal(E) * 2) / 2).astype(np.float32)
        idx = oracle_mod.select_biased(L, b, k)
        key = L + b[None, :]
        assert key.dtype == np.float32
        for t in range(T):
            order = np.lexsort((np.arange(E), -key[t].astype(np.float64)))
            assert idx[t].tolist() == order[:k].tolist(), (trial, t)


def test_biased_selection_forces_the_biased_experts(oracle_mod):
    """A bias far above the logits' spread makes the biased experts the picks,
    ordered among themselves by logit; the gates ignore the bias."""
    rng = np.random.default_rng(24)
    T, E, k = 50, 16, 3
    L = _random_logits(rng, T, E, coarse=True)
    hot = np.array([13, 2, 7])
    b = np.zeros(E, np.float32)
    b[hot] = 512.0
    idx = oracle_mod.select_biased(L, b, k)
    for t in range(T):
        want = sorted(hot.tolist(), key=lambda e: (-float(L[t, e]), e))
        assert idx[t].tolist() == want
    w = oracle_mod.gates_at(L, idx)
    e = np.exp(L.astype(np.float64) - L.max(axis=1, keepdims=True))
    assert np.allclose(w, np.take_along_axis(e / e.sum(axis=1, keepdims=True), idx, axis=1),
                       rtol=0, atol=1e-15)


def test_gates_at_closed_forms(oracle_mod):
    """Logistic gates: 1/2 at 0 and (1 + tanh(x/2)) / 2 elsewhere; renormalised,
    a single pick gets exactly 1 and k picks sum to 1; softmax gates at the
    plain top-k picks equal oracle_topk's own weights."""
    rng = np.random.default_rng(25)
    L = (rng.standard_normal((30, 12)) * 3).astype(np.float32)
    L[0, :] = 0.0
    idx, w_soft = oracle_mod.topk(L, 4)
    w = oracle_mod.gates_at(L, idx, sigmoid=True)
    assert np.all(w[0] == 0.5)
    x = np.take_along_axis(L, idx, axis=1).astype(np.float64)
    assert np.allclose(w, (1.0 + np.tanh(x / 2)) / 2, rtol=0, atol=1e-15)
    wr = oracle_mod.gates_at(L, idx, sigmoid=True, renorm=True)
    assert np.allclose(wr.sum(axis=1), 1.0, rtol=0, atol=1e-15)
    assert np.allclose(wr * w.sum(axis=1, keepdims=True), w, rtol=1e-14, atol=0)
    assert np.all(oracle_mod.gates_at(L, idx[:, :1], sigmoid=True, renorm=True) == 1.0)
    assert np.allclose(oracle_mod.gates_at(L, idx), w_soft, rtol=0, atol=1e-16)
    assert np.allclose(oracle_mod.gates_at(L, idx, renorm=True), oracle_mod.renorm_gates(L, idx),
                       rtol=0, atol=1e-15)


def test_swiglu_closed_forms(oracle_mod):
    """silu(g) * u: 0 when g = 0 or u = 0; g * u once e^-g is below half an ulp
    of 1; (1 + tanh(g/2)) / 2 * g * u in general; gate and up halves not
    interchangeable."""
    rng = np.random.default_rng(26)
    S, F = 7, 24
    G = rng.standard_normal((S, 2 * F)) * 3
    G[0, :F] = 0.0
    G[1, F:] = 0.0
    G[2, :F] = 50.0
    H = oracle_mod.swiglu(G)
    assert np.all(H[0] == 0.0) and np.all(H[1] == 0.0)
    assert np.array_equal(H[2], 50.0 * G[2, F:])
    g, u = G[:, :F], G[:, F:]
    ref = (1.0 + np.tanh(g / 2)) / 2 * g * u  # 1 + tanh cancels for g << 0: absolute bound
    assert np.all(np.abs(H - ref) <= 1e-15 * np.abs(g * u) + 1e-14 * np.abs(ref))
    h = oracle_mod.swiglu(np.array([[2.0, 3.0]]))[0, 0]
    assert h == pytest.approx(2.0 / (1.0 + math.exp(-2.0)) * 3.0, rel=1e-15)
    assert h != pytest.approx(3.0 / (1.0 + math.exp(-3.0)) * 2.0, rel=1e-3)


def test_round_bf16_ties_and_library(oracle_mod):
    """Round to nearest, ties to even: the halfway points around 1 and 3;
    then fp32-representable values of every magnitude (subnormal, overflow,
    signed zero) against torch's fp32 -> bf16 conversion, which is the same
    rounding done once."""
    torch = pytest.importorskip("torch")
    ties = np.array([1 + 2 ** -8, 1 + 3 * 2 ** -8, -(1 + 2 ** -8), 3 + 2 ** -7, 3 + 3 * 2 ** -7,
                     1 + 2 ** -8 + 2 ** -30])
    want = [0x3F80, 0x3F82, 0xBF80, 0x4040, 0x4042, 0x3F81]
    assert oracle_mod.round_bf16(ties).tolist() == want
    rng = np.random.default_rng(27)
    v32 = (rng.standard_normal(20000) * np.exp(rng.uniform(-95, 86, 20000))).astype(np.float32)
    v32 = np.concatenate([v32, np.array([0.0, -0.0, 2 ** -133, 2 ** -134, 3 * 2 ** -135, 3.39e38],
                                        np.float32)])
    ref = torch.from_numpy(v32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(oracle_mod.round_bf16(v32.astype(np.float64)), ref)


def test_topk_rejects_nan(oracle_mod):
    L = np.array([[0.0, np.nan, 1.0]], np.float32)
    with pytest.raises(ValueError):
        oracle_mod.topk(L, 1)


@pytest.mark.parametrize("seed", range(4))
def test_histogram_and_permutation_brute_force(oracle_mod, seed):
    rng = np.random.default_rng(100 + seed)
    T, E = int(rng.integers(1, 50)), int(rng.integers(1, 17))
    k = int(rng.integers(1, E + 1))
    L = _random_logits(rng, T, E, coarse=True)
    r = oracle_mod.route(L, k)
    idx = r["topk_idx"]
    cnt = collections.Counter(idx.ravel().tolist())
    assert r["counts"].tolist() == [cnt.get(e, 0) for e in range(E)]
    assert r["offsets"].tolist() == [0] + list(itertools.accumulate(cnt.get(e, 0) for e in range(E)))
    assert int(r["counts"].sum()) == T * k
    # the destination order is the sort of (expert, token, slot) triples
    triples = sorted((int(idx[t, j]), t, j) for t in range(T) for j in range(k))
    assert r["perm"].tolist() == [t * k + j for _, t, j in triples]
    # bijection and inverse
    assert sorted(r["perm"].tolist()) == list(range(T * k))
    assert (r["dest"][r["perm"]] == np.arange(T * k)).all()
    assert (r["perm"][r["dest"]] == np.arange(T * k)).all()
    # inside each expert segment, tokens ascend
    for e in range(E):
        seg = r["perm"][r["offsets"][e]:r["offsets"][e + 1]] // k
        assert (np.diff(seg) > 0).all()


def test_all_tokens_on_one_expert(oracle_mod):
    T, E, k = 33, 5, 1
    L = np.zeros((T, E), np.float32)
    L[:, 3] = 1.0
    r = oracle_mod.route(L, k)
    assert r["counts"].tolist() == [0, 0, 0, T, 0]
    assert r["offsets"].tolist() == [0, 0, 0, 0, T, T]
    assert r["perm"].tolist() == list(range(T))


def test_rank_base(oracle_mod):
    off = np.array([0, 2, 6, 7, 8], np.int32)
    assert oracle_mod.rank_base(off, 2).tolist() == [0, 6, 8]
    assert oracle_mod.rank_base(off, 4).tolist() == [0, 2, 6, 7, 8]
    assert oracle_mod.rank_base(off, 1).tolist() == [0, 8]
    with pytest.raises(ValueError):
        oracle_mod.rank_base(off, 3)


# ---------------------------------------------------------------- A4

def test_gather_is_fancy_index(oracle_mod):
    rng = np.random.default_rng(5)
    T, d, E, k = 37, 24, 6, 3
    x = rng.integers(0, 65536, size=(T, d), dtype=np.uint16)
    L = rng.standard_normal((T, E)).astype(np.float32)
    r = oracle_mod.route(L, k)
    rows = oracle_mod.gather(x, r["perm"], k)
    assert np.array_equal(rows, x[r["perm"] // k])


# ---------------------------------------------------------------- A5

def test_gemm_single_expert_is_plain_matmul(oracle_mod):
    """E = 1, k = 1: the grouped GEMM is one plain GEMM (numpy fp64 as cross-check)."""
    rng = np.random.default_rng(7)
    S, d, N = 19, 48, 40
    a = _bf16_bits_from_f32(rng.standard_normal((S, d)).astype(np.float32))
    W = _bf16_bits_from_f32((rng.standard_normal((1, d, N)) / np.sqrt(d)).astype(np.float32))
    off = np.array([0, S], np.int32)
    Y = oracle_mod.grouped_gemm(a, W, off)
    ref = _bits_to_f64(a) @ _bits_to_f64(W[0])
    assert np.allclose(Y, ref, rtol=1e-12, atol=1e-12)


def test_gemm_one_hot_weights_copy_rows(oracle_mod):
    """W_e = identity columns: Y equals the destination rows exactly."""
    rng = np.random.default_rng(8)
    S, d, E = 12, 16, 3
    rows = _bf16_bits_from_f32(rng.standard_normal((S, d)).astype(np.float32))
    eye = _bf16_bits_from_f32(np.eye(d, dtype=np.float32))
    W = np.stack([eye] * E)
    off = np.array([0, 5, 5, S], np.int32)  # expert 1 empty
    Y = oracle_mod.grouped_gemm(rows, W, off)
    assert np.array_equal(Y, _bits_to_f64(rows))


def test_gemm_uses_each_rows_own_expert(oracle_mod):
    """Rows in expert e's segment see W_e and no other: compare per segment."""
    rng = np.random.default_rng(9)
    d, N, E = 32, 24, 4
    off = np.array([0, 3, 3, 10, 14], np.int32)
    S = int(off[-1])
    rows = _bf16_bits_from_f32(rng.standard_normal((S, d)).astype(np.float32))
    W = _bf16_bits_from_f32((rng.standard_normal((E, d, N)) / np.sqrt(d)).astype(np.float32))
    Y = oracle_mod.grouped_gemm(rows, W, off)
    for e in range(E):
        seg = slice(off[e], off[e + 1])
        ref = _bits_to_f64(rows[seg]) @ _bits_to_f64(W[e])
        assert np.allclose(Y[seg], ref, rtol=1e-12, atol=1e-12)
        for row in range(off[e], off[e + 1]):
            assert oracle_mod.expert_of_row(off, row) == e
    # the single-entry helper agrees bit for bit with the full GEMM
    for row, n in [(0, 0), (5, 7), (13, 23)]:
        e = oracle_mod.expert_of_row(off, row)
        assert oracle_mod.gemm_entry(rows[row], W[e], n) == Y[row, n]


def test_gemm_within_fp64_summation_bound(oracle_mod):
    """Exact rational re-sum: |fl(sum) - sum| <= gamma_{d-1} * sum |terms|.

    bf16 x bf16 products are exact in fp64 (8-bit significands), so the only
    error is the d-1 additions: gamma_n = n u / (1 - n u), u = 2^-53.
    """
    rng = np.random.default_rng(10)
    S, d, N = 4, 64, 6
    rows = _bf16_bits_from_f32(rng.standard_normal((S, d)).astype(np.float32) * 3)
    W = _bf16_bits_from_f32(rng.standard_normal((1, d, N)).astype(np.float32))
    Y = oracle_mod.grouped_gemm(rows, W, np.array([0, S], np.int32))
    a = _bits_to_f64(rows)
    w = _bits_to_f64(W[0])
    u = 2.0 ** -53
    gamma = (d - 1) * u / (1 - (d - 1) * u)
    for i in range(S):
        for n in range(N):
            terms = [Fraction(float(a[i, q])) * Fraction(float(w[q, n])) for q in range(d)]
            exact = sum(terms, Fraction(0))
            bound = gamma * float(sum(abs(t) for t in terms))
            assert abs(Fraction(Y[i, n]) - exact) <= Fraction(bound)


# ---------------------------------------------------------------- combine (the step after the path)

def test_combine_single_slot_unit_gate_undoes_the_permutation(oracle_mod):
    rng = np.random.default_rng(20)
    T, E, N = 30, 5, 12
    L = rng.standard_normal((T, E)).astype(np.float32)
    r = oracle_mod.route(L, 1)
    Y = rng.standard_normal((T, N))
    out = oracle_mod.combine(Y, np.ones((T, 1)), r["dest"])
    assert np.array_equal(out, Y[r["dest"]])
    # and the permutation applied to token rows comes back to the token rows
    rows_in_dest_order = Y[r["perm"]]
    assert np.array_equal(oracle_mod.combine(rows_in_dest_order, np.ones((T, 1)), r["dest"]), Y)


def test_combine_matches_fancy_index_sum(oracle_mod):
    """A different implementation: numpy fancy indexing, then a weighted sum over slots."""
    rng = np.random.default_rng(21)
    T, E, k, N = 25, 7, 3, 9
    L = rng.standard_normal((T, E)).astype(np.float32)
    r = oracle_mod.route(L, k)
    Y = rng.standard_normal((T * k, N))
    w = r["topk_w"]
    out = oracle_mod.combine(Y, w, r["dest"])
    ref = (Y[r["dest"].reshape(T, k)] * w[:, :, None]).sum(axis=1)
    assert np.allclose(out, ref, rtol=1e-14, atol=1e-14)


def test_combine_k_equals_e_with_constant_expert_outputs(oracle_mod):
    """k = E and Y row = 1 for every slot: out = sum of all softmax weights = 1."""
    rng = np.random.default_rng(22)
    T, E, N = 10, 6, 4
    L = rng.standard_normal((T, E)).astype(np.float32)
    r = oracle_mod.route(L, E)
    out = oracle_mod.combine(np.ones((T * E, N)), r["topk_w"], r["dest"])
    assert np.allclose(out, 1.0, rtol=0, atol=1e-13)


# ---------------------------------------------------------------- router logits (the step before the path)

def test_router_logits_near_fp64_and_exact_on_small_integers(oracle_mod):
    rng = np.random.default_rng(30)
    T, d, E = 17, 96, 6
    x = _bf16_bits_from_f32(rng.standard_normal((T, d)).astype(np.float32))
    W = _bf16_bits_from_f32((rng.standard_normal((d, E)) / np.sqrt(d)).astype(np.float32))
    L = oracle_mod.router_logits(x, W)
    ref = _bits_to_f64(x) @ _bits_to_f64(W)
    # fp32 sequential sum: error bounded by gamma_d * sum |terms| in fp32 arithmetic
    bound = d * 2.0 ** -24 * (np.abs(_bits_to_f64(x)) @ np.abs(_bits_to_f64(W)))
    assert np.all(np.abs(L - ref) <= bound)
    # small integers: every partial sum is exact, so the result equals the exact dot product
    xi = rng.integers(-8, 9, (T, d)).astype(np.float32)
    Wi = rng.integers(-8, 9, (d, E)).astype(np.float32)
    Li = oracle_mod.router_logits(_bf16_bits_from_f32(xi), _bf16_bits_from_f32(Wi))
    assert np.array_equal(Li, (xi.astype(np.int64) @ Wi.astype(np.int64)).astype(np.float32))


def test_router_logits_order_is_ascending_fma(oracle_mod):
    """Terms 2^24, 1, -2^24: an ascending fp32 sum gives 0 (the 1 is absorbed);
    any other grouping of these three gives 1."""
    x = _bf16_bits_from_f32(np.array([[2.0 ** 12, 1.0, -(2.0 ** 12)]], np.float32))
    W = _bf16_bits_from_f32(np.array([[2.0 ** 12], [1.0], [2.0 ** 12]], np.float32))
    assert oracle_mod.router_logits(x, W)[0, 0] == 0.0
    bias = np.array([0.5], np.float32)
    assert oracle_mod.router_logits(x, W, bias)[0, 0] == 0.5


# ---------------------------------------------------------------- the oracle timed on all host cores

@pytest.mark.parametrize("threads", [2, 5, 8, 64])
def test_grouped_gemm_on_several_cores_is_bitwise_the_single_threaded_one(oracle_mod, threads):
    """The benchmark times the oracle's grouped GEMM split by output rows over the
    host cores.  On the tiny workload (T=256, d=512, E=8, top-2, N=1024) every
    split gives the single-threaded result bit for bit, and both equal a numpy fp64
    product of each expert's rows (a cross-check, within fp64 rounding)."""
    from moe_token_dispatch_route_gb300 import workloads
    wl = workloads.WORKLOADS["tiny"]
    inp = workloads.make_inputs(wl, seed=0)
    ref = oracle_mod.route(inp["logits"].numpy(), wl.k)
    rows = oracle_mod.gather(workloads.bf16_bits(inp["x"]), ref["perm"], wl.k)
    Wb = workloads.bf16_bits(inp["W"])
    one = oracle_mod.grouped_gemm(rows, Wb, ref["offsets"])
    many = oracle_mod.grouped_gemm_parallel(rows, Wb, ref["offsets"], threads)
    assert np.array_equal(one.view(np.uint64), many.view(np.uint64))
    off = ref["offsets"]
    for e in range(wl.E):
        a, b = int(off[e]), int(off[e + 1])
        want = _bits_to_f64(rows[a:b]) @ _bits_to_f64(Wb[e])
        assert np.allclose(many[a:b], want, rtol=1e-12, atol=1e-12)
