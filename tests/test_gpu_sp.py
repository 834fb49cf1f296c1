"""GPU parity of the sequence-parallel form (duoan.github.io "Tensor
Parallelism in Megatron-LM", "Row split": reduce-scatter / all-gather when the
sequence is split), called through the C ABI.

The simulated collectives are checked bit for bit (the all-gather is a copy;
the reduce-scatter against an fp32 sum in shard order); the forward and
backward against the float64 oracle with the MLP tolerances (fp32: max|err|
<= 1e-4 max|ref|; bf16: relative Frobenius <= 5e-3, max <= 2e-2), and bit for
bit against the unsplit calls on the same inputs, which compute the same
values in the same order.
"""

import numpy as np
import pytest
import torch

import oracle
from tpmlp_inputs import WORKLOADS, Workload, make_inputs, sample_indices

pytestmark = pytest.mark.gpu


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


def slices_of(t, n):
    """n separately allocated copies of t's row slices (each rank's own buffer)."""
    return [c.clone() for c in torch.chunk(t, n, dim=0)]


# ----------------------------------------------------------------- collectives

@pytest.mark.parametrize("n,rows,cols", [(1, 8, 4), (2, 3, 5), (3, 100, 320), (4, 257, 136), (8, 64, 1000),
                                         (16, 6, 128), (5, 7, 3)])
def test_reduce_scatter_fixed_order(tp, n, rows, cols):
    g = torch.Generator().manual_seed(n * 1000 + rows)
    Yp = torch.randn((n, n * rows, cols), generator=g).cuda()
    out = tp.tpmlp_reduce_scatter(Yp)
    acc = Yp[0].clone()
    for i in range(1, n):
        acc = acc + Yp[i]  # fp32, shard order
    full = tp.tpmlp_allreduce(Yp)
    for j in range(n):
        assert torch.equal(out[j], acc[j * rows:(j + 1) * rows])
        assert torch.equal(out[j], full[j * rows:(j + 1) * rows])


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("n,rows,cols", [(1, 4, 8), (2, 3, 5), (3, 100, 320), (8, 2048, 64), (16, 1, 8)])
def test_all_gather_is_a_copy(tp, dtype, n, rows, cols):
    g = torch.Generator().manual_seed(rows * 7 + cols)
    X = torch.randn((n * rows, cols), generator=g).to(dtype).cuda()
    assert torch.equal(tp.tpmlp_all_gather(slices_of(X, n)), X)


def test_collective_argument_errors(tp):
    Yp = torch.zeros((3, 4, 4), device="cuda")
    with pytest.raises(tp.TpmlpError):  # 16 elements per partial do not split into 3 slices
        tp.tpmlp_reduce_scatter(Yp, [torch.empty(5, device="cuda") for _ in range(3)])


# ----------------------------------------------------------------- forward / backward

SMALL = [
    # name, T, D, F, n (T divisible by n)
    ("ragged", 300, 320, 1536, 3),
    ("narrow_shards", 256, 136, 288, 4),
    ("single_shard", 129, 64, 512, 1),
    ("many_shards", 96, 128, 16 * 72, 16),
    ("min_dims", 6, 8, 16, 2),
    ("pair_ragged", 2000, 1288, 1024, 4),  # fused sum on CTA pairs; tiles straddle rank slices
    ("pair_sliced", 2048, 1288, 1024, 4),  # 512-row slices: per-slice TMA stores
]


def small_workload(name, T, D, F, n, dtype):
    return Workload(name, T, D, F, n, dtype, 1.0, 1.0 / np.sqrt(D), 1.0 / np.sqrt(F), 1.0, True)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("case", SMALL, ids=[c[0] for c in SMALL])
def test_sp_forward_backward_against_oracle(tp, case, dtype):
    w = small_workload(*case, dtype)
    inp = make_inputs(w, seed=41)
    n = w.N
    X, dY = f64(inp["X"]), f64(inp["dY"])
    shards_ref = oracle.shard_mlp(f64(inp["A"]), f64(inp["B"]), n)
    Ys_ref = oracle.tp_mlp_sp(oracle.split_rows(X, n), shards_ref)
    dXs_ref, dA_ref, dB_ref = oracle.tp_mlp_sp_backward(oracle.split_rows(X, n), oracle.split_rows(dY, n),
                                                        shards_ref)
    d = {k: v.cuda() for k, v in inp.items()}
    sh = tp.tpmlp_shard(d["A"], d["B"], n)
    Xs, dYs = slices_of(d["X"], n), slices_of(d["dY"], n)
    Ts = w.T // n
    for mode in ("faithful", "fused"):
        Ys = tp.tpmlp_forward_sp(Xs, sh, mode)
        tp.tpmlp_check_status()
        Y = tp.tpmlp_forward(d["X"], sh, mode)
        for j in range(n):
            check(f64(Ys[j]), Ys_ref[j], dtype, f"Y slice {j} {mode}")
            assert torch.equal(Ys[j], Y[j * Ts:(j + 1) * Ts]), f"Y slice {j} {mode} differs from the unsplit forward"
        dXs, dA, dB = tp.tpmlp_backward_sp(Xs, dYs, sh, mode)
        tp.tpmlp_check_status()
        dX_u, dA_u, dB_u = tp.tpmlp_backward(d["X"], d["dY"], sh, mode)
        for j in range(n):
            check(f64(dXs[j]), dXs_ref[j], dtype, f"dX slice {j} {mode}")
            assert torch.equal(dXs[j], dX_u[j * Ts:(j + 1) * Ts])
        for i in range(n):
            check(f64(dA[i]), dA_ref[i], dtype, f"dA_{i} {mode}")
            check(f64(dB[i]), dB_ref[i], dtype, f"dB_{i} {mode}")
            assert torch.equal(dA[i], dA_u[i]) and torch.equal(dB[i], dB_u[i])


def test_sp_rejects_indivisible_token_counts(tp):
    w = small_workload("r", 12, 64, 256, 4, "bf16")
    inp = make_inputs(w, seed=42)
    sh = tp.tpmlp_shard(inp["A"].cuda(), inp["B"].cuda(), 4)
    X = inp["X"].cuda()
    l = tp.lib()
    import ctypes

    xs = (ctypes.c_void_p * 4)(*[X.data_ptr()] * 4)
    ys = (ctypes.c_void_p * 4)(*[X.data_ptr()] * 4)
    ws = torch.empty(1 << 20, dtype=torch.uint8, device="cuda")
    assert l.tpmlp_forward_sp(xs, 10, sh.handle, ys, 0, ws.data_ptr(), 1 << 20, None) == tp.TPMLP_ERR_DIVISIBILITY
    assert tp.tpmlp_sp_workspace_bytes(10, sh) == 0


def test_sp_large_workload_matches_unsplit_and_oracle_rows(tp):
    # T=16384, D=4096, F=16384, N=8 (2048 tokens per rank) at full size.
    w = WORKLOADS["large"]
    inp = make_inputs(w, seed=0)
    n = w.N
    Ts = w.T // n
    d = {k: v.cuda() for k, v in inp.items()}
    sh = tp.tpmlp_shard(d["A"], d["B"], n)
    Xs = slices_of(d["X"], n)
    rows = sample_indices(w.T, 64, seed=12)
    shards_ref = oracle.shard_mlp(f64(inp["A"]), f64(inp["B"]), n)
    Y_rows_ref = oracle.tp_mlp_rows(f64(inp["X"]), shards_ref, rows)
    for mode in ("faithful", "fused"):
        Ys = tp.tpmlp_forward_sp(Xs, sh, mode)
        Y = tp.tpmlp_forward(d["X"], sh, mode)
        tp.tpmlp_check_status()
        for j in range(n):
            assert torch.equal(Ys[j], Y[j * Ts:(j + 1) * Ts])
        got = torch.cat(Ys).index_select(0, torch.tensor(rows, device="cuda"))
        check(f64(got), Y_rows_ref, "bf16", f"large SP rows {mode}")
        del Ys, Y


def test_sp_fwd_bwd_workload_matches_unsplit(tp):
    # T=8192, D=8192, F=32768, N=8 at full size: the SP backward equals the
    # unsplit one bit for bit (whose own parity with the oracle is tested
    # separately on sampled rows and columns).
    w = WORKLOADS["fwd_bwd"]
    inp = make_inputs(w, seed=0)
    n = w.N
    Ts = w.T // n
    d = {k: v.cuda() for k, v in inp.items()}
    del inp
    sh = tp.tpmlp_shard(d["A"], d["B"], n)
    Xs, dYs = slices_of(d["X"], n), slices_of(d["dY"], n)
    for mode in ("faithful", "fused"):
        dXs, dA, dB = tp.tpmlp_backward_sp(Xs, dYs, sh, mode)
        dX, dA_u, dB_u = tp.tpmlp_backward(d["X"], d["dY"], sh, mode)
        tp.tpmlp_check_status()
        for j in range(n):
            assert torch.equal(dXs[j], dX[j * Ts:(j + 1) * Ts])
        for i in range(n):
            assert torch.equal(dA[i], dA_u[i]) and torch.equal(dB[i], dB_u[i])
        del dXs, dA, dB, dX, dA_u, dB_u


def _random_sp_shapes(count, seed):
    """Seeded (T, D, F, N) with T a multiple of N (the rank slices), D and F/N
    multiples of 8, slices of any height (not only multiples of 32)."""
    rng = np.random.default_rng(seed)
    out = []
    while len(out) < count:
        n = int(rng.choice([2, 3, 4, 8]))
        fs = 8 * int(rng.integers(1, 97))
        d = 8 * int(rng.integers(1, 161))
        t = n * int(rng.integers(1, 400))
        if n * fs <= 6144:
            out.append((t, d, n * fs, n))
    return out


@pytest.mark.parametrize("shape", _random_sp_shapes(8, 91), ids=lambda s: "T%dD%dF%dN%d" % s)
def test_sp_random_shapes(tp, shape):
    """Sequence-parallel forward and backward (dX) on seeded random shapes: every
    rank slice bitwise equal to the unsplit call's rows, and sampled rows
    against the float64 oracle, both modes."""
    T, D, F, n = shape
    w = Workload("rs", T, D, F, n, "bf16", 1.0, 0.05, 0.05, 1.0, True)
    inp = make_inputs(w, seed=T + 5 * D)
    rows = sorted(set(sample_indices(T, min(T, 40), seed=9)) | {T - 1})
    shards_ref = oracle.shard_mlp(f64(inp["A"]), f64(inp["B"]), n)
    Y_ref = oracle.tp_mlp_rows(f64(inp["X"]), shards_ref, rows)
    d = {k: v.cuda() for k, v in inp.items()}
    sh = tp.tpmlp_shard(d["A"], d["B"], n)
    Xs, dYs = slices_of(d["X"], n), slices_of(d["dY"], n)
    idx = torch.tensor(rows, device="cuda")
    for mode in ("faithful", "fused"):
        Y = torch.cat(tp.tpmlp_forward_sp(Xs, sh, mode))
        assert torch.equal(Y, tp.tpmlp_forward(d["X"], sh, mode)), f"{mode} {shape}: slices differ from the unsplit rows"
        check(f64(Y.index_select(0, idx)), Y_ref, "bf16", f"Y {mode} {shape}")
        dX = torch.cat(tp.tpmlp_backward_sp(Xs, dYs, sh, mode)[0])
        assert torch.equal(dX, tp.tpmlp_backward(d["X"], d["dY"], sh, mode)[0]), f"dX {mode} {shape}"
    tp.tpmlp_check_status()
    sh.free()
