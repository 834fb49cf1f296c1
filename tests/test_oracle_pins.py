"""Pins for the float64 oracle, checked against facts fixed outside the oracle.

Sources of truth:
  * the worked example printed on scratchllm.com "Tensor-Parallel MLP
    (Megatron)" (section "The split", Example; stored in
    tests/golden/worked_example.json);
  * the GeLU values and the row-split counterexample printed on that page;
  * closed forms of the tanh GeLU (Taylor series at 0, odd-part identity,
    limits), and its closeness to the exact erf GeLU from Python's math.erf;
  * brute force with Python scalars on tiny inputs;
  * central finite differences for every gradient.

The last test plants plausible mistakes in a copy of the oracle and checks
that the pins catch each of them.
"""

import json
import math
import os

import numpy as np
import pytest

import oracle
from oracle import tpmlp_oracle as orc

GOLD = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "worked_example.json")))


def _rounded(v, d=3):
    # Round half away from zero to d decimals, as the page prints; map -0.0 to 0.0.
    return [float(np.round(x + 0.0, d)) + 0.0 for x in np.ravel(v)]


# ---------------------------------------------------------------- worked example

def worked_example_mismatches(mod=orc):
    """List of (what, got, printed) for every printed value the oracle misses."""
    g = GOLD
    X, A, B, n, d = np.array(g["X"], float), np.array(g["A"], float), np.array(g["B"], float), g["n"], g["decimals"]
    bad = []

    def cmp(what, got, printed):
        if _rounded(got, d) != [float(p) for p in printed]:
            bad.append((what, np.ravel(got).tolist(), printed))

    cmp("XA", X @ A, g["XA"])
    cmp("H", mod.gelu(X @ A), g["H"])
    cmp("Y", mod.mlp(X, A, B), g["Y"])
    shards = mod.shard_mlp(A, B, n)
    Y, parts = mod.tp_mlp(X, shards, return_partials=True)
    for i, s in enumerate(g["shards"]):
        cmp(f"A_{i}", shards[i][0], A[:, s["A_cols"]].ravel())
        cmp(f"B_{i}", shards[i][1], B[s["B_rows"], :].ravel())
        cmp(f"H_{i}", parts[i][0], s["H"])
        cmp(f"Y_{i}", parts[i][1], s["Y"])
    cmp("allreduce", Y, g["allreduce"])
    for x, v in g["gelu_points"].items():
        cmp(f"gelu({x})", mod.gelu(float(x)), [v])
    cmp("gelu(1+1)", mod.gelu(2.0), [g["counterexample"]["gelu_of_sum_1_plus_1"]])
    cmp("gelu(1)+gelu(1)", mod.gelu(1.0) + mod.gelu(1.0), [g["counterexample"]["sum_of_gelus_1_and_1"]])
    return bad


def test_worked_example_matches_printed_values():
    assert worked_example_mismatches() == []


def test_gelu_zero_is_exactly_zero():
    assert oracle.gelu(0.0) == 0.0


def test_row_split_counterexample():
    # GeLU of a sum is not the sum of GeLUs (the reason A is split by columns).
    assert abs(oracle.gelu(2.0) - 2 * oracle.gelu(1.0)) > 0.25


# ---------------------------------------------------------------- GeLU closed forms

def test_gelu_taylor_series_at_zero():
    # GeLU(x) = x/2 + (c/2) x^2 + (c a/2 - c^3/6) x^4 + O(x^6), c = sqrt(2/pi), a = 0.044715,
    # from tanh(u) = u - u^3/3 + ... with u = c (x + a x^3).
    c, a = math.sqrt(2 / math.pi), 0.044715
    for x in [1e-2, 2e-2, 4e-2]:
        g = float(oracle.gelu(x))
        c2 = (g - x / 2) / x**2
        assert abs(c2 - c / 2) < 1e-2 * x  # x^2 coefficient; next term is O(x^2)
        c4 = (g - x / 2 - c / 2 * x**2) / x**4
        assert abs(c4 - (c * a / 2 - c**3 / 6)) < 5 * x**2


def test_gelu_odd_part_identity():
    # tanh is odd, so GeLU(x) - GeLU(-x) = x exactly in real arithmetic.
    x = np.linspace(-9, 9, 4001)
    np.testing.assert_allclose(oracle.gelu(x) - oracle.gelu(-x), x, rtol=0, atol=4e-15 * 9)


def test_gelu_limits():
    assert float(oracle.gelu(30.0)) == 30.0
    assert abs(float(oracle.gelu(-30.0))) < 1e-300


def test_gelu_close_to_exact_erf_gelu():
    # The tanh form approximates x * Phi(x); its largest gap on the real line is below 5e-4.
    xs = np.linspace(-8, 8, 3201)
    exact = np.array([0.5 * x * (1 + math.erf(x / math.sqrt(2))) for x in xs])
    gap = np.max(np.abs(oracle.gelu(xs) - exact))
    assert 1e-4 < gap < 5e-4


def test_gelu_grad_matches_central_differences():
    x = np.linspace(-6, 6, 241)
    h = 1e-5
    fd = (oracle.gelu(x + h) - oracle.gelu(x - h)) / (2 * h)
    np.testing.assert_allclose(oracle.gelu_grad(x), fd, rtol=0, atol=1e-9)
    assert abs(float(oracle.gelu_grad(0.0)) - 0.5) < 1e-15


# ---------------------------------------------------------------- sharding

def test_shard_slices_follow_the_index_rule():
    D, F = 3, 12
    A = np.array([[1000 * r + c for c in range(F)] for r in range(D)], float)
    B = np.array([[1000 * r + c for c in range(D)] for r in range(F)], float)
    for n in [1, 2, 3, 4, 6, 12]:
        Fs = F // n
        for i, (A_i, B_i) in enumerate(oracle.shard_mlp(A, B, n)):
            assert A_i.shape == (D, Fs) and B_i.shape == (Fs, D)
            for r in range(D):
                for c in range(Fs):
                    assert A_i[r, c] == 1000 * r + (i * Fs + c)
            for r in range(Fs):
                for c in range(D):
                    assert B_i[r, c] == 1000 * (i * Fs + r) + c


@pytest.mark.parametrize("n", [0, 5, 7, -2])
def test_shard_rejects_non_divisor(n):
    with pytest.raises(ValueError):
        oracle.shard_mlp(np.zeros((2, 12)), np.zeros((12, 2)), n)


def test_sharded_equals_unsplit_for_every_divisor():
    rng = np.random.default_rng(1)
    T, D, F = 5, 4, 24
    X, A, B = rng.normal(size=(T, D)), rng.normal(size=(D, F)), rng.normal(size=(F, D))
    Y = oracle.mlp(X, A, B)
    for n in [d for d in range(1, F + 1) if F % d == 0]:
        np.testing.assert_allclose(oracle.tp_mlp(X, oracle.shard_mlp(A, B, n)), Y, rtol=1e-13, atol=1e-13)


def _brute_force_mlp(X, A, B):
    T, D = len(X), len(X[0])
    F = len(A[0])
    c = math.sqrt(2 / math.pi)
    Y = [[0.0] * D for _ in range(T)]
    for t in range(T):
        for f in range(F):
            p = 0.0
            for d in range(D):
                p += X[t][d] * A[d][f]
            h = 0.5 * p * (1 + math.tanh(c * (p + 0.044715 * p**3)))
            for d in range(D):
                Y[t][d] += h * B[f][d]
    return Y


def test_brute_force_tiny():
    rng = np.random.default_rng(2)
    T, D, F = 3, 5, 6
    X, A, B = rng.normal(size=(T, D)), rng.normal(size=(D, F)), rng.normal(size=(F, D))
    ref = np.array(_brute_force_mlp(X.tolist(), A.tolist(), B.tolist()))
    for n in [1, 2, 3, 6]:
        np.testing.assert_allclose(oracle.tp_mlp(X, oracle.shard_mlp(A, B, n)), ref, rtol=1e-12, atol=1e-12)


# ---------------------------------------------------------------- backward

def _loss(X, A, B, dY):
    return float(np.sum(oracle.mlp(X, A, B) * dY))


@pytest.mark.parametrize("n", [1, 2, 3])
def test_backward_matches_finite_differences(n):
    rng = np.random.default_rng(3 + n)
    T, D, F = 4, 3, 6
    X, A, B, dY = (rng.normal(size=s) for s in [(T, D), (D, F), (F, D), (T, D)])
    dX, dA, dB = oracle.tp_mlp_backward(X, dY, oracle.shard_mlp(A, B, n))
    h = 1e-6

    def fd(M, idx):
        Mp, Mm = M.copy(), M.copy()
        Mp[idx] += h
        Mm[idx] -= h
        args_p = {"X": X, "A": A, "B": B}
        args_m = dict(args_p)
        key = [k for k, v in args_p.items() if v is M][0]
        args_p[key], args_m[key] = Mp, Mm
        return (_loss(args_p["X"], args_p["A"], args_p["B"], dY) - _loss(args_m["X"], args_m["A"], args_m["B"], dY)) / (2 * h)

    Fs = F // n
    for idx in np.ndindex(T, D):
        assert abs(dX[idx] - fd(X, idx)) < 1e-7
    for r, c in np.ndindex(D, F):
        assert abs(dA[c // Fs][r, c % Fs] - fd(A, (r, c))) < 1e-7
    for r, c in np.ndindex(F, D):
        assert abs(dB[r // Fs][r % Fs, c] - fd(B, (r, c))) < 1e-7


def test_sharded_gradients_reassemble_the_unsplit_ones():
    rng = np.random.default_rng(7)
    T, D, F = 6, 4, 12
    X, A, B, dY = (rng.normal(size=s) for s in [(T, D), (D, F), (F, D), (T, D)])
    dX1, (dA1,), (dB1,) = oracle.tp_mlp_backward(X, dY, oracle.shard_mlp(A, B, 1))
    for n in [2, 3, 4, 6, 12]:
        dX, dA, dB = oracle.tp_mlp_backward(X, dY, oracle.shard_mlp(A, B, n))
        np.testing.assert_allclose(dX, dX1, rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(np.concatenate(dA, axis=1), dA1, rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(np.concatenate(dB, axis=0), dB1, rtol=1e-12, atol=1e-12)


# ---------------------------------------------------------------- sampled entries

def test_sampled_entries_equal_full_results():
    rng = np.random.default_rng(11)
    T, D, F, n = 9, 5, 8, 2
    X, A, B, dY = (rng.normal(size=s) for s in [(T, D), (D, F), (F, D), (T, D)])
    shards = oracle.shard_mlp(A, B, n)
    Y, parts = oracle.tp_mlp(X, shards, return_partials=True)
    dX, dA, dB = oracle.tp_mlp_backward(X, dY, shards)
    rows, cols = [0, 3, 8], [1, 3]
    np.testing.assert_allclose(oracle.tp_mlp_rows(X, shards, rows), Y[rows], rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(oracle.tp_mlp_backward_dx_rows(X, dY, shards, rows), dX[rows], rtol=1e-13, atol=1e-13)
    for i, (A_i, B_i) in enumerate(shards):
        H_r, Y_r = oracle.shard_partial_rows(X, A_i, B_i, rows)
        np.testing.assert_allclose(H_r, parts[i][0][rows], rtol=1e-13, atol=1e-13)
        np.testing.assert_allclose(Y_r, parts[i][1][rows], rtol=1e-13, atol=1e-13)
        np.testing.assert_allclose(oracle.grad_A_cols(X, dY, A_i, B_i, cols), dA[i][:, cols], rtol=1e-13, atol=1e-13)
        np.testing.assert_allclose(oracle.grad_B_rows(X, dY, A_i, cols), dB[i][cols, :], rtol=1e-13, atol=1e-13)


# ---------------------------------------------------------------- planted mistakes

class _Mutant:
    """A copy of the oracle's public functions with one plausible mistake planted."""

    def __init__(self, **over):
        for k in ["gelu", "gelu_grad", "shard_mlp", "mlp", "shard_partial", "tp_mlp"]:
            setattr(self, k, getattr(orc, k))
        self.__dict__.update(over)


def _erf_gelu(x):
    x = np.asarray(x, float)
    return 0.5 * x * (1 + np.vectorize(math.erf)(x / math.sqrt(2)))


def _gelu_no_cubic(x):
    x = np.asarray(x, float)
    return 0.5 * x * (1 + np.tanh(math.sqrt(2 / math.pi) * x))


def _shard_off_by_one(A, B, n):
    s = orc.shard_mlp(A, B, n)
    return [(a, s[(i + 1) % n][1]) for i, (a, _) in enumerate(s)]


def _shard_interleaved(A, B, n):
    A, B = np.asarray(A, float), np.asarray(B, float)
    return [(A[:, i::n], B[i::n, :]) for i in range(n)]


def _tp_mlp_last_only(X, shards, return_partials=False):
    Y, parts = orc.tp_mlp(X, shards, return_partials=True)
    Y = parts[-1][1]
    return (Y, parts) if return_partials else Y


def _mlp_rows_of_B_reversed(X, A, B):
    return orc.gelu(np.asarray(X, float) @ np.asarray(A, float)) @ np.asarray(B, float)[::-1]


@pytest.mark.parametrize(
    "name,mut",
    [
        ("erf GeLU instead of tanh", dict(gelu=_erf_gelu)),
        ("cubic term dropped", dict(gelu=_gelu_no_cubic)),
        ("B rows of the wrong shard", dict(shard_mlp=_shard_off_by_one)),
        ("interleaved instead of contiguous slices", dict(shard_mlp=_shard_interleaved)),
        ("all-reduce drops partials", dict(tp_mlp=_tp_mlp_last_only)),
        ("rows of B reversed", dict(mlp=_mlp_rows_of_B_reversed)),
    ],
)
def test_pins_catch_planted_mistakes(name, mut):
    assert worked_example_mismatches(_Mutant(**mut)) != [], name


def test_gradient_pins_catch_a_wrong_gelu_grad():
    # A gelu' missing its second term must fail the central-difference pin.
    bad = lambda x: 0.5 * (1 + np.tanh(math.sqrt(2 / math.pi) * (x + 0.044715 * x**3)))
    x = np.linspace(-3, 3, 61)
    h = 1e-5
    fd = (oracle.gelu(x + h) - oracle.gelu(x - h)) / (2 * h)
    assert np.max(np.abs(bad(x) - fd)) > 1e-2


# ---------------------------------------------------------------- block tail: layer norm + residual

def test_layer_norm_against_torch_library_routine():
    import torch

    rng = np.random.default_rng(21)
    x = rng.normal(size=(7, 33)) * 3 + 1.5
    ref = torch.nn.functional.layer_norm(torch.from_numpy(x), (33,), eps=1e-5).numpy()
    np.testing.assert_allclose(oracle.layer_norm(x), ref, rtol=1e-12, atol=1e-12)


def test_layer_norm_closed_forms():
    rng = np.random.default_rng(22)
    x = rng.normal(size=(5, 64)) * 2 - 3
    y = oracle.layer_norm(x)
    var = x.var(axis=1)
    np.testing.assert_allclose(y.mean(axis=1), 0, atol=1e-13)
    np.testing.assert_allclose(y.var(axis=1), var / (var + oracle.LN_EPS), rtol=1e-12)
    # without eps the map is invariant to a per-row positive scale and shift
    np.testing.assert_allclose(oracle.layer_norm(4.0 * x + 7.0, eps=0.0), oracle.layer_norm(x, eps=0.0), atol=1e-12)
    # a constant row normalises to zero
    assert np.all(oracle.layer_norm(np.full((2, 8), 3.25)) == 0.0)
    # two elements (a, b): (a - m) / sqrt(((a - b) / 2)^2 + eps)
    a, b = 1.0, 2.0
    h = (b - a) / 2
    np.testing.assert_allclose(oracle.layer_norm([[a, b]]), [[-h / math.sqrt(h * h + 1e-5), h / math.sqrt(h * h + 1e-5)]])


def test_block_mlp_residual_and_composition():
    rng = np.random.default_rng(23)
    T, D, F = 6, 8, 24
    x, A, B = rng.normal(size=(T, D)), rng.normal(size=(D, F)), rng.normal(size=(F, D))
    # with B = 0 the MLP contributes nothing and the block is the identity
    assert np.array_equal(oracle.block_mlp(x, oracle.shard_mlp(A, np.zeros((F, D)), 3)), x)
    # otherwise it is x + the unsplit MLP of the normalised input, for every divisor
    ref = x + oracle.mlp(oracle.layer_norm(x), A, B)
    for n in [1, 2, 3, 4, 6]:
        np.testing.assert_allclose(oracle.block_mlp(x, oracle.shard_mlp(A, B, n)), ref, rtol=1e-13, atol=1e-13)
    rows = [0, 4]
    np.testing.assert_allclose(oracle.block_mlp_rows(x, oracle.shard_mlp(A, B, 2), rows), ref[rows], rtol=1e-13)


def test_layer_norm_backward_against_autograd_and_differences():
    import torch

    rng = np.random.default_rng(24)
    x, g = rng.normal(size=(4, 12)) * 2 + 0.5, rng.normal(size=(4, 12))
    xt = torch.from_numpy(x).requires_grad_(True)
    (torch.nn.functional.layer_norm(xt, (12,), eps=1e-5) * torch.from_numpy(g)).sum().backward()
    np.testing.assert_allclose(oracle.layer_norm_backward(x, g), xt.grad.numpy(), rtol=1e-11, atol=1e-12)
    # central differences of sum(LN(x) * g)
    h = 1e-6
    fd = np.zeros_like(x)
    for t in range(x.shape[0]):
        for k in range(x.shape[1]):
            e = np.zeros_like(x)
            e[t, k] = h
            fd[t, k] = ((oracle.layer_norm(x + e) - oracle.layer_norm(x - e)) * g).sum() / (2 * h)
    np.testing.assert_allclose(oracle.layer_norm_backward(x, g), fd, rtol=1e-6, atol=1e-7)
    # the gradient is orthogonal to the constant direction and to y (shift and, without eps, scale invariance)
    dx = oracle.layer_norm_backward(x, g, eps=0.0)
    np.testing.assert_allclose(dx.sum(axis=1), 0, atol=1e-11)
    np.testing.assert_allclose((dx * x).sum(axis=1), 0, atol=1e-10)


def test_block_backward_against_autograd():
    import torch

    rng = np.random.default_rng(25)
    T, D, F, n = 5, 8, 24, 3
    x, dout = rng.normal(size=(T, D)), rng.normal(size=(T, D))
    A, B = rng.normal(size=(D, F)) * 0.5, rng.normal(size=(F, D)) * 0.5
    xt = torch.from_numpy(x).requires_grad_(True)
    At = torch.from_numpy(A).requires_grad_(True)
    Bt = torch.from_numpy(B).requires_grad_(True)
    xn = torch.nn.functional.layer_norm(xt, (D,), eps=1e-5)
    out = xt + torch.nn.functional.gelu(xn @ At, approximate="tanh") @ Bt
    np.testing.assert_allclose(out.detach().numpy(), oracle.block_mlp(x, oracle.shard_mlp(A, B, n)), rtol=1e-12)
    (out * torch.from_numpy(dout)).sum().backward()
    dx, dA, dB = oracle.block_mlp_backward(x, dout, oracle.shard_mlp(A, B, n))
    np.testing.assert_allclose(dx, xt.grad.numpy(), rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(np.concatenate(dA, axis=1), At.grad.numpy(), rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(np.concatenate(dB, axis=0), Bt.grad.numpy(), rtol=1e-10, atol=1e-12)
    rows = [1, 3]
    np.testing.assert_allclose(oracle.block_mlp_backward_dx_rows(x, dout, oracle.shard_mlp(A, B, n), rows), dx[rows],
                               rtol=1e-12, atol=1e-13)


def test_block_pins_catch_planted_mistakes():
    rng = np.random.default_rng(26)
    x, g = rng.normal(size=(3, 10)) + 1.0, rng.normal(size=(3, 10))
    ref = oracle.layer_norm_backward(x, g)
    y = oracle.layer_norm(x)
    r = 1.0 / np.sqrt(x.var(axis=1, keepdims=True) + 1e-5)
    # dropping the mean-of-g term, or the y-projection term, changes the gradient
    no_mean = r * (g - y * (g * y).mean(axis=1, keepdims=True))
    no_proj = r * (g - g.mean(axis=1, keepdims=True))
    assert np.max(np.abs(no_mean - ref)) > 1e-2 and np.max(np.abs(no_proj - ref)) > 1e-2
    # the unbiased variance gives a different normalisation
    bad = (x - x.mean(axis=1, keepdims=True)) / np.sqrt(x.var(axis=1, ddof=1, keepdims=True) + 1e-5)
    assert np.max(np.abs(bad - y)) > 1e-2


# ---------------------------------------------------------------- sequence-parallel sum

def test_reduce_scatter_brute_force_and_all_reduce_identity():
    rng = np.random.default_rng(27)
    n, T, D = 3, 6, 4
    partials = [rng.normal(size=(T, D)) for _ in range(n)]
    rs = oracle.reduce_scatter(partials, n)
    # brute force with Python scalars: rank j, row r, column c
    for j in range(n):
        for r in range(T // n):
            for c in range(D):
                acc = partials[0][j * (T // n) + r][c]
                for i in range(1, n):
                    acc = acc + partials[i][j * (T // n) + r][c]
                assert rs[j][r, c] == acc
    # all-gather after reduce-scatter is the all-reduce, bit for bit in the same order
    ar = partials[0] + partials[1] + partials[2]
    assert np.array_equal(oracle.all_gather(rs), ar)
    # and all-gather inverts the row split
    X = rng.normal(size=(T, D))
    assert np.array_equal(oracle.all_gather(oracle.split_rows(X, n)), X)
    with pytest.raises(ValueError):
        oracle.split_rows(np.zeros((7, 2)), 3)


def test_sequence_parallel_forward_and_backward_equal_the_unsplit_ones():
    rng = np.random.default_rng(28)
    T, D, F = 8, 6, 12
    X, dY = rng.normal(size=(T, D)), rng.normal(size=(T, D))
    A, B = rng.normal(size=(D, F)) * 0.5, rng.normal(size=(F, D)) * 0.5
    for n in (1, 2, 4):
        shards = oracle.shard_mlp(A, B, n)
        Y = oracle.tp_mlp(X, shards)
        Ys = oracle.tp_mlp_sp(oracle.split_rows(X, n), shards)
        assert len(Ys) == n and all(y.shape == (T // n, D) for y in Ys)
        np.testing.assert_allclose(oracle.all_gather(Ys), oracle.mlp(X, A, B), rtol=1e-13, atol=1e-13)
        for j, Yj in enumerate(Ys):  # rank j owns rows j*T/n.. of the all-reduced output
            np.testing.assert_allclose(Yj, Y[j * (T // n):(j + 1) * (T // n)], rtol=1e-14, atol=1e-14)
        dXs, dA, dB = oracle.tp_mlp_sp_backward(oracle.split_rows(X, n), oracle.split_rows(dY, n), shards)
        dX_ref, dA_ref, dB_ref = oracle.tp_mlp_backward(X, dY, shards)
        np.testing.assert_allclose(oracle.all_gather(dXs), dX_ref, rtol=1e-12, atol=1e-13)
        for i in range(n):
            np.testing.assert_allclose(dA[i], dA_ref[i], rtol=1e-12, atol=1e-13)
            np.testing.assert_allclose(dB[i], dB_ref[i], rtol=1e-12, atol=1e-13)


def test_sequence_parallel_pins_catch_planted_mistakes():
    rng = np.random.default_rng(29)
    n, T, D = 2, 4, 3
    partials = [rng.normal(size=(T, D)) for _ in range(n)]
    rs = oracle.reduce_scatter(partials, n)
    # scattering by columns, or handing rank j the other rank's rows, is caught
    by_cols = [sum(P[:, :2] for P in partials), sum(P[:, 2:] for P in partials)]
    assert by_cols[0].shape != rs[0].shape or not np.allclose(by_cols[0], rs[0])
    swapped = list(reversed(rs))
    assert not np.allclose(oracle.all_gather(swapped), partials[0] + partials[1])
    # a reduce-scatter that drops a partial
    assert not np.allclose(oracle.split_rows(partials[0], n)[0], rs[0])


# ---------------------------------------------------------------- head-split attention

def test_attention_core_against_torch_sdpa():
    import torch

    rng = np.random.default_rng(30)
    batch, s, heads, dh = 2, 5, 3, 4
    Q, K, V = (rng.normal(size=(batch * s, heads * dh)) for _ in range(3))
    O = oracle.attention_core(Q, K, V, batch, heads)

    def bhsd(M):  # [T, H*dh] -> [batch, heads, s, dh]
        return torch.from_numpy(M).reshape(batch, s, heads, dh).permute(0, 2, 1, 3)

    ref = torch.nn.functional.scaled_dot_product_attention(bhsd(Q), bhsd(K), bhsd(V))
    ref = ref.permute(0, 2, 1, 3).reshape(batch * s, heads * dh).numpy()
    np.testing.assert_allclose(O, ref, rtol=1e-12, atol=1e-13)


def test_attention_closed_forms():
    rng = np.random.default_rng(31)
    s, dh = 6, 4
    Q, V = rng.normal(size=(s, dh)), rng.normal(size=(s, dh))
    # identical keys: uniform weights, every output row is the mean of V
    K = np.tile(rng.normal(size=(1, dh)), (s, 1))
    np.testing.assert_allclose(oracle.attention_core(Q, K, V, 1, 1), np.tile(V.mean(axis=0), (s, 1)), rtol=1e-13)
    # identical values: the output is that row whatever the weights
    Vc = np.tile(V[:1], (s, 1))
    np.testing.assert_allclose(oracle.attention_core(Q, rng.normal(size=(s, dh)), Vc, 1, 1), Vc, rtol=1e-13)
    # a one-token sequence attends only to itself
    np.testing.assert_allclose(oracle.attention_core(Q[:1], Q[1:2], V[:1], 1, 1), V[:1], rtol=1e-14)
    # softmax rows sum to one and are shift-invariant; 1/sqrt(d_h) scales the logits
    S = rng.normal(size=(3, 7))
    np.testing.assert_allclose(oracle.softmax_rows(S).sum(axis=1), 1.0, rtol=1e-14)
    np.testing.assert_allclose(oracle.softmax_rows(S + 5.0), oracle.softmax_rows(S), rtol=1e-13)
    q, k, v = rng.normal(size=(2, 16)), rng.normal(size=(2, 16)), rng.normal(size=(2, 16))
    w = np.exp(q @ k.T / 4.0)  # d_h = 16: logits divided by 4
    np.testing.assert_allclose(oracle.attention_core(q, k, v, 1, 1), (w / w.sum(axis=1, keepdims=True)) @ v,
                               rtol=1e-13)
    # sequences of a batch do not see each other
    Q2, K2, V2 = rng.normal(size=(4, dh)), rng.normal(size=(4, dh)), rng.normal(size=(4, dh))
    both = oracle.attention_core(Q2, K2, V2, 2, 1)
    np.testing.assert_allclose(both[2:], oracle.attention_core(Q2[2:], K2[2:], V2[2:], 1, 1), rtol=1e-14)


def test_head_split_attention_equals_unsplit_for_every_divisor():
    rng = np.random.default_rng(32)
    batch, s, D, heads = 2, 4, 12, 6
    X = rng.normal(size=(batch * s, D))
    W = [rng.normal(size=(D, D)) * 0.3 for _ in range(4)]
    ref = oracle.mha(X, batch, *W, heads)
    for n in (1, 2, 3, 6):
        shards = oracle.shard_attention(*W, heads, n)
        Y, parts = oracle.tp_attention(X, batch, shards, heads, return_partials=True)
        np.testing.assert_allclose(Y, ref, rtol=1e-12, atol=1e-13)
        # the ranks' head outputs side by side are the unsplit heads (the all-gather of ai-hpc.org §2)
        O_full = oracle.attention_core(X @ W[0], X @ W[1], X @ W[2], batch, heads)
        np.testing.assert_allclose(np.concatenate([O for O, _ in parts], axis=1), O_full, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(oracle.tp_attention_rows(X, batch, oracle.shard_attention(*W, heads, 2), heads, [1]),
                               ref[s:], rtol=1e-12, atol=1e-13)
    with pytest.raises(ValueError):
        oracle.shard_attention(*W, heads, 4)


def test_attention_pins_catch_planted_mistakes():
    rng = np.random.default_rng(33)
    batch, s, heads, dh = 1, 5, 2, 4
    Q, K, V = (rng.normal(size=(s, heads * dh)) for _ in range(3))
    ref = oracle.attention_core(Q, K, V, batch, heads)
    c = slice(0, dh)
    no_scale = oracle.softmax_rows(Q[:, c] @ K[:, c].T) @ V[:, c]
    wrong_axis = oracle.softmax_rows((Q[:, c] @ K[:, c].T / 2.0).T).T @ V[:, c]
    assert np.max(np.abs(no_scale - ref[:, c])) > 1e-3 and np.max(np.abs(wrong_axis - ref[:, c])) > 1e-3
    # a rank taking every n-th column instead of a contiguous block of heads
    D, n = 8, 2
    W = [rng.normal(size=(D, D)) for _ in range(4)]
    X = rng.normal(size=(3, D))
    good = oracle.tp_attention(X, 1, oracle.shard_attention(*W, 2, n), 2)
    bad_shards = [(W[0][:, i::n], W[1][:, i::n], W[2][:, i::n], W[3][i::n, :]) for i in range(n)]
    bad = oracle.tp_attention(X, 1, bad_shards, 2)
    assert np.max(np.abs(bad - good)) > 1e-3
