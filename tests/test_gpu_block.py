"""GPU parity of the block's FFN half (ai-hpc.org "LLM Lab Notes 06", §2 steps
5-8): layer norm, the split MLP, the residual, and the backward through them,
called through the C ABI and compared with the float64 oracle.

Tolerances are those of the MLP tests (fp32: max|err| <= 1e-4 max|ref|; bf16:
relative Frobenius <= 5e-3 and max <= 2e-2), applied twice: to the block's
output and, so that the residual cannot hide an error in the MLP part, to the
output minus the residual (out - x, dx - dout), which the fp32 output carries
to within 2^-24 of |out|. The layer norm on its own: fp32 within 1e-5, bf16
within one rounding of its fp32 value (2^-8 relative) of the oracle.
"""

import numpy as np
import pytest
import torch

import oracle
from tpmlp_inputs import WORKLOADS, Workload, make_block_inputs, sample_indices

pytestmark = pytest.mark.gpu

EPS = 1e-5


@pytest.fixture(scope="module")
def tp():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__

    __graft_entry__.build()
    import tensor_transformer_mlp_column_gb300 as tp

    torch.cuda.set_device(0)
    return tp


def f64(t) -> np.ndarray:
    return t.detach().to("cpu", torch.float64).numpy()


def check(got, ref, dtype, what=""):
    got, ref = np.asarray(got, np.float64), np.asarray(ref, np.float64)
    err = got - ref
    fro = np.linalg.norm(err) / max(np.linalg.norm(ref), 1e-300)
    mx = np.max(np.abs(err)) / max(np.max(np.abs(ref)), 1e-300)
    if dtype == "f32":
        assert mx <= 1e-4, f"{what}: max err {mx:.3e} of max|ref|"
    else:
        assert fro <= 5e-3 and mx <= 2e-2, f"{what}: rel Frobenius {fro:.3e}, max {mx:.3e}"


# ----------------------------------------------------------------- layer norm

@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("T,D", [(1, 1), (3, 2), (7, 999), (300, 1000), (64, 8192), (5, 25536), (1031, 768)])
def test_layer_norm(tp, dtype, T, D):
    g = torch.Generator().manual_seed(T * 100003 + D)
    x = (torch.randn((T, D), generator=g) * 3.0 + torch.rand((T, 1), generator=g) * 4 - 2).to(dtype)
    ref = oracle.layer_norm(f64(x), EPS)
    y = tp.tpmlp_layer_norm(x.cuda(), EPS)
    if dtype == torch.float32:
        np.testing.assert_allclose(f64(y), ref, rtol=1e-5, atol=1e-5)
    else:
        np.testing.assert_allclose(f64(y), ref, rtol=2.0**-8, atol=1e-5)


def test_layer_norm_degenerate_rows(tp):
    # A constant row (dyadic value, power-of-two length: every fp32 step is
    # exact) normalises to exactly zero; T = 0 is a no-op; in place works.
    x = torch.full((4, 64), 3.25, dtype=torch.float32, device="cuda")
    assert torch.count_nonzero(tp.tpmlp_layer_norm(x, EPS)).item() == 0
    e = torch.empty((0, 16), device="cuda")
    assert tp.tpmlp_layer_norm(e, EPS).shape == (0, 16)
    z = torch.randn((33, 130), device="cuda", dtype=torch.bfloat16)
    ref = oracle.layer_norm(f64(z), EPS)
    tp.tpmlp_layer_norm(z, EPS, y=z)
    np.testing.assert_allclose(f64(z), ref, rtol=2.0**-8, atol=1e-5)


def test_layer_norm_argument_errors(tp):
    x = torch.zeros((4, 8), device="cuda")
    for bad in (0.0, -1.0, float("inf"), float("nan")):
        with pytest.raises(tp.TpmlpError):
            tp.tpmlp_layer_norm(x, bad)
    with pytest.raises(tp.TpmlpError):
        tp.tpmlp_layer_norm(torch.zeros((2, 25537), device="cuda"), EPS)


# ----------------------------------------------------------------- block forward

SMALL = [
    # name, T, D, F, n
    ("ragged", 300, 320, 1536, 3),
    ("narrow_shards", 257, 136, 288, 4),
    ("one_token", 1, 64, 256, 4),
    ("many_shards", 96, 128, 16 * 72, 16),
    ("min_dims", 5, 8, 16, 2),
    ("pair_tiles", 1000, 512, 4096, 4),
    ("pair_ragged", 2000, 1288, 1024, 4),  # the fused sum on CTA pairs, ragged M and N tails
]


def small_workload(name, T, D, F, n, dtype):
    return Workload(name, T, D, F, n, dtype, 1.0, 1.0 / np.sqrt(D), 1.0 / np.sqrt(F), 1.0, True)


def check_block_out(out, x, ref_mlp, dtype, what):
    """out against x + ref_mlp, and out - x against ref_mlp."""
    out, x = f64(out), np.asarray(x, np.float64)
    check(out, x + ref_mlp, dtype, what)
    check(out - x, ref_mlp, dtype, what + " minus residual")


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("case", SMALL, ids=[c[0] for c in SMALL])
def test_block_forward_against_oracle(tp, case, dtype):
    w = small_workload(*case, dtype)
    inp = make_block_inputs(w, seed=31)
    x = f64(inp["x"])
    shards_ref = oracle.shard_mlp(f64(inp["A"]), f64(inp["B"]), w.N)
    xn_ref = oracle.layer_norm(x, EPS)
    mlp_ref = oracle.tp_mlp(xn_ref, shards_ref)
    np.testing.assert_allclose(mlp_ref + x, oracle.block_mlp(x, shards_ref, EPS), rtol=1e-13, atol=1e-13)
    d = {k: v.cuda() for k, v in inp.items()}
    sh = tp.tpmlp_shard(d["A"], d["B"], w.N)
    outs = {}
    for mode in ("faithful", "fused"):
        xn = torch.empty_like(d["x"])
        outs[mode] = tp.tpmlp_block_forward(d["x"], sh, mode, EPS, xn=xn)
        tp.tpmlp_check_status()
        check_block_out(outs[mode], x, mlp_ref, dtype, f"out {mode}")
        tol = 1e-5 if dtype == "f32" else 2.0**-8
        np.testing.assert_allclose(f64(xn), xn_ref, rtol=tol, atol=1e-5)
    # Faithful: bitwise the same as x + allreduce(partials(hidden(LN(x)))), the
    # residual added once to the shard-ordered sum.
    xn = tp.tpmlp_layer_norm(d["x"], EPS)
    Y = tp.tpmlp_allreduce(tp.tpmlp_partials(tp.tpmlp_hidden(xn, sh), sh))
    assert torch.equal(outs["faithful"], d["x"].float() + Y)


def test_block_forward_is_bitwise_reproducible(tp):
    w = small_workload("ragged", 300, 320, 1536, 3, "bf16")
    d = {k: v.cuda() for k, v in make_block_inputs(w, seed=32).items()}
    sh = tp.tpmlp_shard(d["A"], d["B"], w.N)
    for mode in ("faithful", "fused"):
        a = tp.tpmlp_block_forward(d["x"], sh, mode, EPS)
        b = tp.tpmlp_block_forward(d["x"], sh, mode, EPS)
        assert torch.equal(a, b)


@pytest.mark.parametrize("name", ["gpt2_small", "seq512"])
def test_block_workload_forward_full_oracle(tp, name):
    w = WORKLOADS[name]
    inp = make_block_inputs(w, seed=0)
    x = f64(inp["x"])
    shards_ref = oracle.shard_mlp(f64(inp["A"]), f64(inp["B"]), w.N)
    mlp_ref = oracle.tp_mlp(oracle.layer_norm(x, EPS), shards_ref)
    d = {k: v.cuda() for k, v in inp.items()}
    sh = tp.tpmlp_shard(d["A"], d["B"], w.N)
    for mode in ("faithful", "fused"):
        check_block_out(tp.tpmlp_block_forward(d["x"], sh, mode, EPS), x, mlp_ref, w.dtype, f"{name} {mode}")
    tp.tpmlp_check_status()


def test_block_large_forward_sampled_rows(tp):
    # T=16384, D=4096, F=16384, N=8 at full size, the bench's launch configuration.
    w = WORKLOADS["large"]
    inp = make_block_inputs(w, seed=0)
    rows = sample_indices(w.T, 128, seed=7)
    x = f64(inp["x"][rows])
    shards_ref = oracle.shard_mlp(f64(inp["A"]), f64(inp["B"]), w.N)
    mlp_ref = oracle.tp_mlp(oracle.layer_norm(x, EPS), shards_ref)
    d = {k: v.cuda() for k, v in inp.items()}
    sh = tp.tpmlp_shard(d["A"], d["B"], w.N)
    idx = torch.tensor(rows, device="cuda")
    for mode in ("faithful", "fused"):
        out = tp.tpmlp_block_forward(d["x"], sh, mode, EPS)
        check_block_out(out.index_select(0, idx), x, mlp_ref, "bf16", f"large {mode}")
        del out
    tp.tpmlp_check_status()


# ----------------------------------------------------------------- block backward

@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("case", SMALL, ids=[c[0] for c in SMALL])
def test_block_backward_against_oracle(tp, case, dtype):
    w = small_workload(*case, dtype)
    inp = make_block_inputs(w, seed=33, with_dout=True)
    x, dout = f64(inp["x"]), f64(inp["dout"])
    shards_ref = oracle.shard_mlp(f64(inp["A"]), f64(inp["B"]), w.N)
    dx_ref, dA_ref, dB_ref = oracle.block_mlp_backward(x, dout, shards_ref, EPS)
    d = {k: v.cuda() for k, v in inp.items()}
    sh = tp.tpmlp_shard(d["A"], d["B"], w.N)
    for mode in ("faithful", "fused"):
        dx, dA, dB = tp.tpmlp_block_backward(d["x"], d["dout"], sh, mode, EPS)
        tp.tpmlp_check_status()
        check(f64(dx), dx_ref, dtype, f"dx {mode}")
        check(f64(dx) - dout, dx_ref - dout, dtype, f"dx - dout {mode}")
        for i in range(w.N):
            check(f64(dA[i]), dA_ref[i], dtype, f"dA_{i} {mode}")
            check(f64(dB[i]), dB_ref[i], dtype, f"dB_{i} {mode}")


def test_block_backward_matches_mlp_backward_of_the_norm(tp):
    # The weight gradients are the MLP's for X = LN(x) (bitwise, same kernels
    # on the same bf16 operand), and the faithful dx is the layer norm's
    # backward of the MLP's partials.
    w = small_workload("pair_tiles", 1000, 512, 4096, 4, "bf16")
    d = {k: v.cuda() for k, v in make_block_inputs(w, seed=34, with_dout=True).items()}
    sh = tp.tpmlp_shard(d["A"], d["B"], w.N)
    xn = tp.tpmlp_layer_norm(d["x"], EPS)
    _, dA_m, dB_m = tp.tpmlp_backward(xn, d["dout"], sh, "faithful")
    _, dA_b, dB_b = tp.tpmlp_block_backward(d["x"], d["dout"], sh, "faithful", EPS)
    for i in range(w.N):
        assert torch.equal(dA_m[i], dA_b[i]) and torch.equal(dB_m[i], dB_b[i])


def test_block_fwd_bwd_workload_sampled(tp):
    # T=8192, D=8192, F=32768, N=8 at full size: sampled rows of out and dx,
    # sampled columns of every dA_i and rows of every dB_i.
    w = WORKLOADS["fwd_bwd"]
    inp = make_block_inputs(w, seed=0, with_dout=True)
    rows = sample_indices(w.T, 48, seed=8)
    cols = sample_indices(w.Fs, 12, seed=9)
    x_full = f64(inp["x"])
    dout_full = f64(inp["dout"])
    shards_ref = oracle.shard_mlp(f64(inp["A"]), f64(inp["B"]), w.N)
    d = {k: v.cuda() for k, v in inp.items()}
    sh = tp.tpmlp_shard(d["A"], d["B"], w.N)
    idx = torch.tensor(rows, device="cuda")
    cidx = torch.tensor(cols, device="cuda")
    out = tp.tpmlp_block_forward(d["x"], sh, "fused", EPS)
    check_block_out(out.index_select(0, idx), x_full[rows],
                    oracle.tp_mlp(oracle.layer_norm(x_full[rows], EPS), shards_ref), "bf16", "out rows")
    del out
    dx, dA, dB = tp.tpmlp_block_backward(d["x"], d["dout"], sh, "faithful", EPS)
    tp.tpmlp_check_status()
    dx_ref = oracle.block_mlp_backward_dx_rows(x_full, dout_full, shards_ref, rows, EPS)
    check(f64(dx.index_select(0, idx)), dx_ref, "bf16", "dx rows")
    check(f64(dx.index_select(0, idx)) - dout_full[rows], dx_ref - dout_full[rows], "bf16", "dx - dout rows")
    xn_full = oracle.layer_norm(x_full, EPS)
    for i, (A_i, B_i) in enumerate(shards_ref):
        check(f64(dA[i].index_select(1, cidx)), oracle.grad_A_cols(xn_full, dout_full, A_i, B_i, cols), "bf16",
              f"dA_{i} cols")
        check(f64(dB[i].index_select(0, cidx)), oracle.grad_B_rows(xn_full, dout_full, A_i, cols), "bf16",
              f"dB_{i} rows")


def _random_block_shapes(count, seed):
    """Seeded (T, D, F, N) for the bf16 block: D and F/N multiples of 8, D up
    to the register layer norm's 8192-wide backward rows, T ragged."""
    rng = np.random.default_rng(seed)
    out = []
    while len(out) < count:
        n = int(rng.choice([1, 2, 4, 8]))
        fs = 8 * int(rng.integers(1, 97))
        d = 8 * int(rng.integers(1, 161))
        t = int(rng.integers(1, 1801))
        if n * fs <= 6144:
            out.append((t, d, n * fs, n))
    return out


@pytest.mark.parametrize("shape", _random_block_shapes(8, 77), ids=lambda s: "T%dD%dF%dN%d" % s)
def test_block_random_shapes(tp, shape):
    """The block forward (out and out - x) and backward dx on sampled rows, both
    modes, on seeded random shapes, against the float64 oracle."""
    T, D, F, N = shape
    w = Workload("rb", T, D, F, N, "bf16", 1.0, 0.05, 0.05, 1.0, True)
    inp = make_block_inputs(w, seed=T + 3 * D, with_dout=True)
    x, dout = f64(inp["x"]), f64(inp["dout"])
    rows = sorted(set(sample_indices(T, min(T, 40), seed=5)) | {T - 1})
    shards_ref = oracle.shard_mlp(f64(inp["A"]), f64(inp["B"]), N)
    out_ref = oracle.block_mlp_rows(x, shards_ref, rows, EPS)
    dx_ref = oracle.block_mlp_backward_dx_rows(x, dout, shards_ref, rows, EPS)
    d = {k: v.cuda() for k, v in inp.items()}
    sh = tp.tpmlp_shard(d["A"], d["B"], N)
    idx = torch.tensor(rows, device="cuda")
    for mode in ("faithful", "fused"):
        out = f64(tp.tpmlp_block_forward(d["x"], sh, mode, EPS).index_select(0, idx))
        check(out, out_ref, "bf16", f"out {mode} {shape}")
        check(out - x[rows], out_ref - x[rows], "bf16", f"out - x {mode} {shape}")
        dx = f64(tp.tpmlp_block_backward(d["x"], d["dout"], sh, mode, EPS)[0].index_select(0, idx))
        check(dx, dx_ref, "bf16", f"dx {mode} {shape}")
    tp.tpmlp_check_status()
    sh.free()
