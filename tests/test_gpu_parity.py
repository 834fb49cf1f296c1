"""GPU parity: the CUDA library (called through its C ABI) against the float64 oracle.

Tolerances (the same for every output Y, H_i, Y_i, dX, dA_i, dB_i):
  fp32 path:  max|err| <= 1e-4 * max|ref|
  bf16 path:  ||err||_F / ||ref||_F <= 5e-3  and  max|err| <= 2e-2 * max|ref|
  shard slicing: bit-exact.
The bf16 path rounds H_i (and the backward's dP_i) to bf16 before the next
product while the oracle keeps float64; that rounding (relative 2^-9 per
element, independent signs) puts the relative Frobenius error near 1e-3,
inside the budget.
"""

import json
import os

import numpy as np
import pytest
import torch

import oracle
from tpmlp_inputs import WORKLOADS, Workload, make_inputs, sample_indices

pytestmark = pytest.mark.gpu

GOLD = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "worked_example.json")))


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


def errs(got, ref):
    got, ref = np.asarray(got, np.float64), np.asarray(ref, np.float64)
    err = got - ref
    fro = np.linalg.norm(err) / max(np.linalg.norm(ref), 1e-300)
    mx = np.max(np.abs(err)) / max(np.max(np.abs(ref)), 1e-300)
    return fro, mx


def check(got, ref, dtype, what=""):
    fro, mx = errs(got, ref)
    if dtype == "f32":
        assert mx <= 1e-4, f"{what}: max err {mx:.3e} of max|ref|"
    else:
        assert fro <= 5e-3 and mx <= 2e-2, f"{what}: rel Frobenius {fro:.3e}, max {mx:.3e}"


def on_gpu(inp):
    return {k: v.cuda() for k, v in inp.items()}


# ----------------------------------------------------------------- GeLU

@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("n", [1, 7, 4096, 1_000_003])
def test_gelu(tp, dtype, n):
    g = torch.Generator().manual_seed(n)
    x = (torch.randn(n, generator=g) * 4).to(dtype)
    x[0] = 0.0
    ref = oracle.gelu(f64(x))
    y = f64(tp.tpmlp_gelu(x.cuda()))
    assert y[0] == 0.0
    if dtype == torch.float32:
        np.testing.assert_allclose(y, ref, rtol=2e-6, atol=1e-7)
    else:  # one rounding to bf16 (relative 2^-9) plus the fp32 evaluation
        np.testing.assert_allclose(y, ref, rtol=2.0**-8, atol=1e-6)


def test_gelu_extremes(tp):
    # For x <= -8 the oracle's 1 + tanh(u) cancels to exactly 0 in float64 (the
    # true GeLU(-8) is about -3.1e-21), while the kernel's x*sigmoid(2u) keeps
    # the tiny value; both are within 1e-12 of each other there.
    x = torch.tensor([-1e4, -100.0, -30.0, -8.0, -5.0, 5.0, 8.0, 30.0, 100.0, 1e4], dtype=torch.float32)
    y = f64(tp.tpmlp_gelu(x.cuda()))
    np.testing.assert_allclose(y, oracle.gelu(f64(x)), rtol=2e-6, atol=1e-12)
    assert np.all(y[:5] <= 0) and np.all(y[5:] > 0)


# ----------------------------------------------------------------- shard slicing

@pytest.mark.parametrize("D,F,n", [(1024, 4096, 4), (128, 512, 2)], ids=["pair_kernel", "single_cta_kernel"])
def test_gemm_epilogue_gelu_pointwise(tp, D, F, n):
    """The GeLU of the bf16 GEMM epilogue, element by element: with X = I the
    pre-activations P_i = X A_i are exactly A's bf16 entries, swept over
    [-8, 8], so every H_i[t, f] must be GeLU(A[t, i F/n + f]) up to the bf16
    rounding of the result (2^-9 relative) and the hardware tanh's error
    (below 2^-11 |x| / 2 absolute)."""
    T = D
    X = torch.eye(D, dtype=torch.bfloat16)
    g = torch.Generator().manual_seed(3)
    A = ((torch.rand((D, F), generator=g) * 2 - 1) * 8).to(torch.bfloat16)
    A[0, :16] = torch.tensor([0, 1, -1, 2, -2, 3, -3, 4, -4, 6, -6, 8, -8, 0.5, -0.5, 1.5], dtype=torch.bfloat16)
    B = (torch.randn((F, D), generator=g) * 0.02).to(torch.bfloat16)
    sh = tp.tpmlp_shard(A.cuda(), B.cuda(), n)
    H = f64(tp.tpmlp_hidden(X.cuda(), sh))  # [n, T, F/n]
    a = f64(A)
    ref = oracle.gelu(a)
    got = np.concatenate([H[i] for i in range(n)], axis=1)  # back to [T, F]
    assert got.shape == (T, F)
    bound = 2.0**-8 * np.abs(ref) + 2.0**-11 * np.abs(a) + 1e-6
    worst = np.max(np.abs(got - ref) - bound)
    assert worst <= 0, f"GeLU epilogue off by {worst:.3e} beyond the bound"
    pos = a >= 0
    assert np.max(np.abs(got - ref)[pos] / np.maximum(np.abs(ref[pos]), 1e-30)) <= 2.0**-8 + 2.0**-10
    sh.free()


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("D,F,n", [(64, 256, 4), (24, 96, 3), (8, 8, 1), (136, 1152, 16)])
def test_shard_slices_bit_exact(tp, dtype, D, F, n):
    g = torch.Generator().manual_seed(D * F + n)
    A = torch.randn(D, F, generator=g).to(dtype).cuda()
    B = torch.randn(F, D, generator=g).to(dtype).cuda()
    sh = tp.tpmlp_shard(A, B, n)
    Fs = F // n
    for i in range(n):
        A_i, B_i = sh.get(i)
        assert torch.equal(A_i, A[:, i * Fs:(i + 1) * Fs])
        assert torch.equal(B_i, B[i * Fs:(i + 1) * Fs, :])
        if dtype == torch.bfloat16:
            At_i, Bt_i = sh.get_transposed(i)
            assert torch.equal(At_i, A[:, i * Fs:(i + 1) * Fs].t())
            assert torch.equal(Bt_i, B[i * Fs:(i + 1) * Fs, :].t())
    sh.free()


def test_shard_errors_on_gpu(tp):
    A = torch.zeros(64, 256, dtype=torch.bfloat16, device="cuda")
    B = torch.zeros(256, 64, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(tp.TpmlpError) as e:
        tp.tpmlp_shard(A, B, 3)
    assert e.value.code == tp.TPMLP_ERR_DIVISIBILITY


# ----------------------------------------------------------------- all-reduce

@pytest.mark.parametrize("n,count", [(1, 4096), (2, 1000), (4, 1_000_003), (8, 262_144), (13, 4100), (20, 777)])
def test_allreduce_fixed_order(tp, n, count):
    g = torch.Generator().manual_seed(n * 7 + count)
    Yp = torch.randn(n, count, generator=g)
    Y = tp.tpmlp_allreduce(Yp.cuda()).cpu().numpy()
    # Same order in fp32 on the host: ((Y_0 + Y_1) + Y_2) + ...
    ref32 = Yp[0].numpy().copy()
    for i in range(1, n):
        ref32 = (ref32 + Yp[i].numpy()).astype(np.float32)
    assert np.array_equal(Y, ref32)
    np.testing.assert_allclose(Y, f64(Yp).sum(0), rtol=0, atol=1e-5 * n)


def test_allreduce_is_deterministic(tp):
    Yp = torch.randn(8, 1 << 20, device="cuda")
    a = tp.tpmlp_allreduce(Yp)
    b = tp.tpmlp_allreduce(Yp)
    assert torch.equal(a, b)


# ----------------------------------------------------------------- worked example

def test_worked_example_fp32(tp):
    X = torch.tensor(GOLD["X"], dtype=torch.float32, device="cuda")
    A = torch.tensor(GOLD["A"], dtype=torch.float32, device="cuda")
    B = torch.tensor(GOLD["B"], dtype=torch.float32, device="cuda")
    sh = tp.tpmlp_shard(A, B, GOLD["n"])
    H = tp.tpmlp_hidden(X, sh)
    Yp = tp.tpmlp_partials(H, sh)
    for i, s in enumerate(GOLD["shards"]):
        assert np.round(f64(H[i]).ravel(), 3).tolist() == s["H"]
        assert np.round(f64(Yp[i]).ravel(), 3).tolist() == s["Y"]
    for mode in ("faithful", "fused"):
        Y = f64(tp.tpmlp_forward(X, sh, mode)).ravel()
        assert np.round(Y, 3).tolist() == GOLD["Y"]
        np.testing.assert_allclose(Y, oracle.mlp(GOLD["X"], GOLD["A"], GOLD["B"]).ravel(), rtol=1e-6)


# ----------------------------------------------------------------- forward, step by step

SMALL = [
    # name, T, D, F, n  (ragged tails in every dimension; several tiles each)
    ("ragged", 300, 320, 1536, 3),
    ("narrow_shards", 257, 136, 288, 4),
    ("single_shard", 129, 64, 512, 1),
    ("one_token", 1, 64, 256, 4),
    ("many_shards", 96, 128, 16 * 72, 16),
    ("min_dims", 5, 8, 16, 2),
]


def small_workload(name, T, D, F, n, dtype):
    return Workload(name, T, D, F, n, dtype, 1.0, 1.0 / np.sqrt(D), 1.0 / np.sqrt(F), 1.0, True)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("case", SMALL, ids=[c[0] for c in SMALL])
def test_forward_steps_against_oracle(tp, case, dtype):
    w = small_workload(*case, dtype)
    inp = make_inputs(w, seed=11)
    ref = {k: f64(v) for k, v in inp.items()}
    shards_ref = oracle.shard_mlp(ref["A"], ref["B"], w.N)
    Y_ref, parts = oracle.tp_mlp(ref["X"], shards_ref, return_partials=True)
    d = on_gpu(inp)
    sh = tp.tpmlp_shard(d["A"], d["B"], w.N)
    H = tp.tpmlp_hidden(d["X"], sh)
    Yp = tp.tpmlp_partials(H, sh)
    for i, (H_ref, Yi_ref) in enumerate(parts):
        check(f64(H[i]), H_ref, dtype, f"H_{i}")
        check(f64(Yp[i]), Yi_ref, dtype, f"Y_{i}")
    check(f64(tp.tpmlp_allreduce(Yp)), Y_ref, dtype, "allreduce")
    check(f64(tp.tpmlp_fused_sum(H, sh)), Y_ref, dtype, "fused sum")
    for mode in ("faithful", "fused"):
        check(f64(tp.tpmlp_forward(d["X"], sh, mode)), Y_ref, dtype, f"Y {mode}")
    tp.tpmlp_check_status()


def test_faithful_forward_is_bitwise_reproducible(tp):
    w = small_workload("ragged", 300, 320, 1536, 3, "bf16")
    d = on_gpu(make_inputs(w, seed=3))
    sh = tp.tpmlp_shard(d["A"], d["B"], w.N)
    a = tp.tpmlp_forward(d["X"], sh, "faithful")
    b = tp.tpmlp_forward(d["X"], sh, "faithful")
    assert torch.equal(a, b)


def test_reduce_runs_once_per_faithful_forward(tp):
    # The faithful forward equals allreduce(partials(hidden(X))) bit for bit:
    # the partial sums are reduced exactly once, in shard order.
    w = small_workload("ragged", 300, 320, 1536, 3, "bf16")
    d = on_gpu(make_inputs(w, seed=4))
    sh = tp.tpmlp_shard(d["A"], d["B"], w.N)
    Y = tp.tpmlp_forward(d["X"], sh, "faithful")
    Y2 = tp.tpmlp_allreduce(tp.tpmlp_partials(tp.tpmlp_hidden(d["X"], sh), sh))
    assert torch.equal(Y, Y2)


@pytest.mark.parametrize("name", ["tiny_fp32", "gpt2_small", "seq128", "seq256", "seq512"])
def test_workload_forward_full_oracle(tp, name):
    w = WORKLOADS[name]
    inp = make_inputs(w, seed=0)
    ref = {k: f64(v) for k, v in inp.items()}
    Y_ref = oracle.tp_mlp(ref["X"], oracle.shard_mlp(ref["A"], ref["B"], w.N))
    d = on_gpu(inp)
    sh = tp.tpmlp_shard(d["A"], d["B"], w.N)
    for mode in ("faithful", "fused"):
        check(f64(tp.tpmlp_forward(d["X"], sh, mode)), Y_ref, w.dtype, f"{name} {mode}")
    tp.tpmlp_check_status()


def test_large_forward_sampled_rows(tp):
    # T=16384, D=4096, F=16384, N=8 at full size; 256 sampled token rows.
    w = WORKLOADS["large"]
    inp = make_inputs(w, seed=0)
    rows = sample_indices(w.T, 256, seed=99)
    shards_ref = oracle.shard_mlp(f64(inp["A"]), f64(inp["B"]), w.N)
    Y_ref = oracle.tp_mlp_rows(f64(inp["X"]), shards_ref, rows)
    d = on_gpu(inp)
    sh = tp.tpmlp_shard(d["A"], d["B"], w.N)
    idx = torch.tensor(rows, device="cuda")
    for mode in ("faithful", "fused"):
        Y = tp.tpmlp_forward(d["X"], sh, mode)
        check(f64(Y.index_select(0, idx)), Y_ref, "bf16", f"large {mode}")
    tp.tpmlp_check_status()


def _random_shapes(count, seed):
    """Seeded (T, D, F, N) draws over the bf16 path's constraints (D and F/N
    multiples of 8), small and pair-sized alike, ragged in every dimension."""
    rng = np.random.default_rng(seed)
    out = []
    while len(out) < count:
        n = int(rng.choice([1, 2, 3, 4, 5, 8, 16]))
        fs = 8 * int(rng.integers(1, 129))   # 8 .. 1024
        d = 8 * int(rng.integers(1, 193))    # 8 .. 1536
        t = int(rng.integers(1, 2501))
        if n * fs > 8192:
            continue
        out.append((t, d, n * fs, n))
    return out


RANDOM_SHAPES = _random_shapes(12, 2026)


@pytest.mark.parametrize("shape", RANDOM_SHAPES, ids=lambda s: "T%dD%dF%dN%d" % s)
def test_random_shapes_forward_backward(tp, shape):
    """Forward (both modes) on 48 sampled token rows plus the last one, and the
    backward's dX on the same rows, against the float64 oracle."""
    T, D, F, N = shape
    w = Workload("rand", T, D, F, N, "bf16", 1.0, 0.05, 0.05, 1.0, True)
    inp = make_inputs(w, seed=T + D)
    rows = sorted(set(sample_indices(T, min(T, 48), seed=7)) | {T - 1})
    ref = {k: f64(v) for k, v in inp.items()}
    shards_ref = oracle.shard_mlp(ref["A"], ref["B"], N)
    Y_ref = oracle.tp_mlp_rows(ref["X"], shards_ref, rows)
    dX_ref = oracle.tp_mlp_backward_dx_rows(ref["X"], ref["dY"], shards_ref, rows)
    d = on_gpu(inp)
    sh = tp.tpmlp_shard(d["A"], d["B"], N)
    idx = torch.tensor(rows, device="cuda")
    for mode in ("faithful", "fused"):
        check(f64(tp.tpmlp_forward(d["X"], sh, mode).index_select(0, idx)), Y_ref, "bf16", f"Y {mode} {shape}")
        dX, _, _ = tp.tpmlp_backward(d["X"], d["dY"], sh, mode)
        check(f64(dX.index_select(0, idx)), dX_ref, "bf16", f"dX {mode} {shape}")
    tp.tpmlp_check_status()
    sh.free()


# ----------------------------------------------------------------- backward

@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("case", SMALL, ids=[c[0] for c in SMALL])
def test_backward_against_oracle(tp, case, dtype):
    w = small_workload(*case, dtype)
    inp = make_inputs(w, seed=21, with_dy=True)
    ref = {k: f64(v) for k, v in inp.items()}
    dX_ref, dA_ref, dB_ref = oracle.tp_mlp_backward(ref["X"], ref["dY"], oracle.shard_mlp(ref["A"], ref["B"], w.N))
    d = on_gpu(inp)
    sh = tp.tpmlp_shard(d["A"], d["B"], w.N)
    for mode in ("faithful", "fused"):
        dX, dA, dB = tp.tpmlp_backward(d["X"], d["dY"], sh, mode)
        check(f64(dX), dX_ref, dtype, f"dX {mode}")
        for i in range(w.N):
            check(f64(dA[i]), dA_ref[i], dtype, f"dA_{i} {mode}")
            check(f64(dB[i]), dB_ref[i], dtype, f"dB_{i} {mode}")
    tp.tpmlp_check_status()


def test_backward_tiny_fp32_workload(tp):
    w = WORKLOADS["tiny_fp32"]
    inp = make_inputs(w, seed=0, with_dy=True)
    ref = {k: f64(v) for k, v in inp.items()}
    dX_ref, dA_ref, dB_ref = oracle.tp_mlp_backward(ref["X"], ref["dY"], oracle.shard_mlp(ref["A"], ref["B"], w.N))
    d = on_gpu(inp)
    sh = tp.tpmlp_shard(d["A"], d["B"], w.N)
    dX, dA, dB = tp.tpmlp_backward(d["X"], d["dY"], sh, "faithful")
    check(f64(dX), dX_ref, "f32", "dX")
    for i in range(w.N):
        check(f64(dA[i]), dA_ref[i], "f32", f"dA_{i}")
        check(f64(dB[i]), dB_ref[i], "f32", f"dB_{i}")


def _check_sampled_fwd_bwd(tp, w, inp, rows, cols, what):
    """Both modes of tpmlp_forward and tpmlp_backward at the workload's full
    size, against the float64 oracle on sampled token rows of Y and dX,
    sampled columns of every dA_i and the same rows of every dB_i. The oracle
    values are computed once; the GPU outputs of each mode are compared with
    them separately."""
    X, dY = f64(inp["X"]), f64(inp["dY"])
    shards_ref = oracle.shard_mlp(f64(inp["A"]), f64(inp["B"]), w.N)
    Y_ref = oracle.tp_mlp_rows(X, shards_ref, rows)
    dX_ref = oracle.tp_mlp_backward_dx_rows(X, dY, shards_ref, rows)
    dA_ref = [oracle.grad_A_cols(X, dY, A_i, B_i, cols) for A_i, B_i in shards_ref]
    dB_ref = [oracle.grad_B_rows(X, dY, A_i, cols) for A_i, _ in shards_ref]
    d = on_gpu(inp)
    sh = tp.tpmlp_shard(d["A"], d["B"], w.N)
    idx = torch.tensor(rows, device="cuda")
    cidx = torch.tensor(cols, device="cuda")
    for mode in ("faithful", "fused"):
        Y = tp.tpmlp_forward(d["X"], sh, mode)
        check(f64(Y.index_select(0, idx)), Y_ref, "bf16", f"{what} Y rows {mode}")
        del Y
        dX, dA, dB = tp.tpmlp_backward(d["X"], d["dY"], sh, mode)
        tp.tpmlp_check_status()
        check(f64(dX.index_select(0, idx)), dX_ref, "bf16", f"{what} dX rows {mode}")
        for i in range(w.N):
            check(f64(dA[i].index_select(1, cidx)), dA_ref[i], "bf16", f"{what} dA_{i} cols {mode}")
            check(f64(dB[i].index_select(0, cidx)), dB_ref[i], "bf16", f"{what} dB_{i} rows {mode}")
        del dX, dA, dB
    sh.free()


def test_fwd_bwd_workload_sampled(tp):
    # T=8192, D=8192, F=32768, N=8 at full size, in the bench's launch
    # configuration, both modes of the forward and of the backward: 64 sampled
    # rows of Y and dX, 16 sampled columns of every dA_i and rows of every dB_i.
    # The fused products chain K over all eight shards (F = 32768: 512 K blocks
    # of 64 per output tile).
    w = WORKLOADS["fwd_bwd"]
    inp = make_inputs(w, seed=0)
    rows = sample_indices(w.T, 64, seed=5)
    cols = sample_indices(w.Fs, 16, seed=6)
    _check_sampled_fwd_bwd(tp, w, inp, rows, cols, "fwd_bwd")


# Shapes whose shard-ordered sums chain K over 512 blocks of 64 (F = 32768, as
# in the fwd+bwd workload) at a fraction of its size: one with enough 256 x 256
# output tiles for the CTA-pair kernel, one small enough for the single-CTA
# kernel's narrow tiles.
LONG_CHAIN = [("pair_kernel", 2048, 1280, 32768, 8), ("single_cta_kernel", 384, 512, 32768, 8)]


@pytest.mark.parametrize("case", LONG_CHAIN, ids=[c[0] for c in LONG_CHAIN])
def test_long_shard_chain_sampled(tp, case):
    name, T, D, F, N = case
    w = Workload(name, T, D, F, N, "bf16", 1.0, 0.01, 0.01, 1.0, True)
    inp = make_inputs(w, seed=T + 3)
    rows = sorted(set(sample_indices(T, 48, seed=8)) | {0, T - 1})
    cols = sorted(set(sample_indices(w.Fs, 24, seed=9)) | {0, w.Fs - 1})
    _check_sampled_fwd_bwd(tp, w, inp, rows, cols, name)


# ----------------------------------------------------------------- bounded waits

def test_bounded_wait_reports_timeout_and_context_survives(tp):
    tp.tpmlp_check_status()  # clean start
    tp.tpmlp_selftest_wait_timeout(50)
    with pytest.raises(tp.TpmlpError) as e:
        tp.tpmlp_check_status()
    assert e.value.code == tp.TPMLP_ERR_TIMEOUT
    tp.tpmlp_check_status()  # cleared
    x = torch.randn(1000, device="cuda")
    np.testing.assert_allclose(f64(tp.tpmlp_gelu(x)), oracle.gelu(f64(x)), rtol=2e-6, atol=1e-7)


# ----------------------------------------------------------------- saved pre-activations (training mode)

@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("case", SMALL[:3] + [("pair_tiles", 1000, 512, 4096, 4)], ids=lambda c: c[0])
def test_forward_save_and_backward_saved(tp, case, dtype):
    w = small_workload(*case, dtype)
    inp = make_inputs(w, seed=51, with_dy=True)
    ref = {k: f64(v) for k, v in inp.items()}
    shards_ref = oracle.shard_mlp(ref["A"], ref["B"], w.N)
    dX_ref, dA_ref, dB_ref = oracle.tp_mlp_backward(ref["X"], ref["dY"], shards_ref)
    d = on_gpu(inp)
    sh = tp.tpmlp_shard(d["A"], d["B"], w.N)
    for mode in ("faithful", "fused"):
        Y, P = tp.tpmlp_forward_save(d["X"], sh, mode)
        # the same output as the inference forward, bit for bit
        assert torch.equal(Y, tp.tpmlp_forward(d["X"], sh, mode))
        # P_i = X A_i: exact bf16/fp32 products summed in fp32
        for i, (A_i, _) in enumerate(shards_ref):
            P_ref = ref["X"] @ A_i
            assert np.max(np.abs(f64(P[i]) - P_ref)) <= 1e-5 * np.max(np.abs(P_ref)), f"P_{i}"
        P_before = P.clone()
        g_re = tp.tpmlp_backward(d["X"], d["dY"], sh, mode)
        g_sv = tp.tpmlp_backward_saved(d["X"], d["dY"], P, sh, mode)
        assert torch.equal(P, P_before)  # the saved P is only read
        # The recomputing backward keeps P in its workspace unless the dual
        # kernel holds it in tensor memory (bf16, products with enough CTA-pair
        # tiles). With P in the workspace both calls run the same kernels on the
        # same P: identical gradients. The dual kernel keeps GeLU'(P) in fp16,
        # so there both are held to the oracle only.
        p_bytes = w.N * w.T * w.Fs * 4
        dual = (tp.tpmlp_workspace_bytes(w.T, sh, mode, 1) - tp.tpmlp_workspace_bytes(w.T, sh, mode, 2)) < p_bytes
        assert dual == (dtype == "bf16" and case[0] == "pair_tiles"), "dual backward kernel chosen unexpectedly"
        if not dual:
            assert torch.equal(g_re[0], g_sv[0])
            for i in range(w.N):
                assert torch.equal(g_re[1][i], g_sv[1][i]) and torch.equal(g_re[2][i], g_sv[2][i])
        for g, kind in ((g_sv, "saved"), (g_re, "recomputed")):
            check(f64(g[0]), dX_ref, dtype, f"dX {mode} {kind}")
            for i in range(w.N):
                check(f64(g[1][i]), dA_ref[i], dtype, f"dA_{i} {mode} {kind}")
                check(f64(g[2][i]), dB_ref[i], dtype, f"dB_{i} {mode} {kind}")
    tp.tpmlp_check_status()


# ----------------------------------------------------------------- CUDA graphs

def test_forward_replays_from_a_cuda_graph(tp):
    # The calls only enqueue work on the given stream, so a CUDA graph of them
    # replays the same computation: bit-identical to eager calls.
    w = small_workload("graph", 1000, 512, 4096, 4, "bf16")
    d = on_gpu(make_inputs(w, seed=61))
    sh = tp.tpmlp_shard(d["A"], d["B"], w.N)
    for mode in ("faithful", "fused"):
        ws = torch.empty(tp.tpmlp_workspace_bytes(w.T, sh, mode), dtype=torch.uint8, device="cuda")
        Y = torch.empty((w.T, w.D), dtype=torch.float32, device="cuda")
        ref = tp.tpmlp_forward(d["X"], sh, mode)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            tp.tpmlp_forward(d["X"], sh, mode, Y, ws)
        Y.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(Y, ref)
        d["X"].mul_(-1.0)  # new input, same buffers: the replay sees it
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(Y, tp.tpmlp_forward(d["X"], sh, mode))
        d["X"].mul_(-1.0)
    tp.tpmlp_check_status()
