"""Float64 CPU oracle for the tensor-parallel MLP  Y = GeLU(X A) B.

TEST INFRASTRUCTURE ONLY. This module is the slow, plainly written checker
that the CUDA library is compared against. Only the tests, the smoke check of
the package entry file and the benchmark's CPU-baseline leg may import it; the
library itself never calls it and has no CPU fallback. It shares no code,
constant or helper with the CUDA sources.

Everything is float64 numpy. Matrix products use numpy's matmul as a library
step; nothing is blocked, fused or reordered beyond what the formulas state.

Notation (scratchllm.com "Tensor-Parallel MLP (Megatron)", section "The
problem"): X is [T, D] (one row per token), A is [D, F], B is [F, D], and
there are n shards with F divisible by n.

Every function below is pinned by tests in tests/test_oracle_pins.py against
values printed on the pages, closed forms or brute force; none is "parity
unpinned".
"""

from __future__ import annotations

import math

import numpy as np

# Constants of the GPT-2 GeLU approximation, scratchllm.com "Tensor-Parallel
# MLP (Megatron)", section "GeLU": u = sqrt(2/pi) * (x + 0.044715 x^3).
SQRT_2_OVER_PI = math.sqrt(2.0 / math.pi)
CUBIC_COEF = 0.044715


def _f64(a) -> np.ndarray:
    return np.asarray(a, dtype=np.float64)


def gelu(x):
    """GeLU(x) ~= 1/2 x (1 + tanh u), u = sqrt(2/pi)(x + 0.044715 x^3), elementwise.

    scratchllm.com "Tensor-Parallel MLP (Megatron)", section "GeLU".
    """
    x = _f64(x)
    u = SQRT_2_OVER_PI * (x + CUBIC_COEF * x * x * x)
    return 0.5 * x * (1.0 + np.tanh(u))


def gelu_grad(x):
    """d/dx of the tanh GeLU above, by the product and chain rules.

    With t = tanh(u):  d/dx [1/2 x (1+t)] = 1/2 (1+t) + 1/2 x (1 - t^2) du/dx,
    du/dx = sqrt(2/pi) (1 + 3 * 0.044715 x^2).  (The pages give the forward
    formula only; this is its derivative, needed for the backward pass of the
    column-then-row MLP that duoan.github.io "Tensor Parallelism in
    Megatron-LM" section 3 describes.)
    """
    x = _f64(x)
    u = SQRT_2_OVER_PI * (x + CUBIC_COEF * x * x * x)
    t = np.tanh(u)
    du = SQRT_2_OVER_PI * (1.0 + 3.0 * CUBIC_COEF * x * x)
    return 0.5 * (1.0 + t) + 0.5 * x * (1.0 - t * t) * du


def shard_mlp(A, B, n: int):
    """Split A by columns and B by the matching rows into n pairs (A_i, B_i).

    Shard i gets columns i*F/n .. (i+1)*F/n - 1 of A and the same range of
    rows of B (scratchllm.com "Tensor-Parallel MLP (Megatron)", sections "The
    split" and "Requirements"). F must be divisible by n ("What to implement").
    """
    A = _f64(A)
    B = _f64(B)
    D, F = A.shape
    if B.shape != (F, D):
        raise ValueError(f"B must be [F, D] = [{F}, {D}], got {B.shape}")
    if n <= 0 or F % n != 0:
        raise ValueError(f"F={F} is not divisible by n={n}")
    Fs = F // n
    return [(A[:, i * Fs:(i + 1) * Fs], B[i * Fs:(i + 1) * Fs, :]) for i in range(n)]


def mlp(X, A, B):
    """The unsplit MLP  Y = GeLU(X A) B  (scratchllm.com, section "The problem")."""
    return gelu(_f64(X) @ _f64(A)) @ _f64(B)


def shard_partial(X, A_i, B_i):
    """One shard's work: H_i = GeLU(X A_i) and the partial output Y_i = H_i B_i.

    scratchllm.com "Tensor-Parallel MLP (Megatron)", section "The split"
    (first two bullets). Returns (H_i, Y_i).
    """
    H_i = gelu(_f64(X) @ _f64(A_i))
    return H_i, H_i @ _f64(B_i)


def tp_mlp(X, shards, return_partials: bool = False):
    """Each shard's partial from its own (A_i, B_i), then the sum Y = sum_i Y_i.

    The sum is the simulated all-reduce (scratchllm.com, section "The split",
    third bullet, and "What to implement"), taken in shard order
    ((Y_0 + Y_1) + Y_2) + ... .
    """
    partials = [shard_partial(X, A_i, B_i) for (A_i, B_i) in shards]
    Y = partials[0][1].copy()
    for _, Y_i in partials[1:]:
        Y = Y + Y_i
    if return_partials:
        return Y, partials
    return Y


def tp_mlp_backward(X, dY, shards):
    """Gradients of L = sum(Y * dY) for Y = sum_i GeLU(X A_i) B_i.

    Per shard (the column/row algebra of duoan.github.io "Tensor Parallelism
    in Megatron-LM", sections 2-3; the upstream gradient dY reaches every
    shard unchanged because the forward reduction is a plain sum):
        P_i  = X A_i
        H_i  = GeLU(P_i)
        dH_i = dY B_i^T
        dP_i = dH_i * GeLU'(P_i)
        dB_i = H_i^T dY
        dA_i = X^T dP_i
    and dX = sum_i dP_i A_i^T, summed in shard order (the one reduction the
    backward pass needs). Returns (dX, [dA_i], [dB_i]).
    """
    X = _f64(X)
    dY = _f64(dY)
    dX = None
    dA, dB = [], []
    for A_i, B_i in shards:
        A_i = _f64(A_i)
        B_i = _f64(B_i)
        P_i = X @ A_i
        H_i = gelu(P_i)
        dH_i = dY @ B_i.T
        dP_i = dH_i * gelu_grad(P_i)
        dB.append(H_i.T @ dY)
        dA.append(X.T @ dP_i)
        dX_i = dP_i @ A_i.T
        dX = dX_i if dX is None else dX + dX_i
    return dX, dA, dB


# ---------------------------------------------------------------------------
# Sampled entries, for workloads too large to run whole in float64. Each is
# the same formula restricted to the rows or columns that the sampled outputs
# depend on, so it gives exactly the entries the full functions would.
# ---------------------------------------------------------------------------

def tp_mlp_rows(X, shards, rows):
    """Rows `rows` of tp_mlp(X, shards): each output row needs only its X row."""
    return tp_mlp(_f64(X)[rows], shards)


def shard_partial_rows(X, A_i, B_i, rows):
    """Rows `rows` of (H_i, Y_i) for one shard."""
    return shard_partial(_f64(X)[rows], A_i, B_i)


def tp_mlp_backward_dx_rows(X, dY, shards, rows):
    """Rows `rows` of dX: row t of dX needs only rows t of X and dY."""
    dX, _, _ = tp_mlp_backward(_f64(X)[rows], _f64(dY)[rows], shards)
    return dX


def grad_A_cols(X, dY, A_i, B_i, cols):
    """Columns `cols` of dA_i = X^T (dH_i * GeLU'(P_i)).

    Column j of dA_i needs column j of P_i = X A_i and of dH_i = dY B_i^T,
    i.e. column j of A_i and row j of B_i, over all tokens.
    """
    X = _f64(X)
    dY = _f64(dY)
    P = X @ _f64(A_i)[:, cols]
    dH = dY @ _f64(B_i)[cols, :].T
    return X.T @ (dH * gelu_grad(P))


def grad_B_rows(X, dY, A_i, rows):
    """Rows `rows` of dB_i = H_i^T dY: row j needs column j of H_i = GeLU(X A_i)."""
    H = gelu(_f64(X) @ _f64(A_i)[:, rows])
    return H.T @ _f64(dY)


# ---------------------------------------------------------------------------
# The FFN half of a tensor-parallel transformer block (ai-hpc.org "LLM Lab
# Notes 06", §2 steps 5-7): normalise the block input, run the column/row
# split MLP, and add the residual. The block there calls
# F.layer_norm(x, (hidden,)) with no weight, bias or eps, so the normalisation
# has no affine parameters and PyTorch's default eps.
# ---------------------------------------------------------------------------

LN_EPS = 1e-5


def layer_norm(x, eps: float = LN_EPS):
    """Row-wise (x - mean) / sqrt(var + eps), var the biased variance of the row."""
    x = _f64(x)
    mu = x.mean(axis=-1, keepdims=True)
    var = ((x - mu) ** 2).mean(axis=-1, keepdims=True)
    return (x - mu) / np.sqrt(var + eps)


def block_mlp(x, shards, eps: float = LN_EPS):
    """out = x + sum_i GeLU(LN(x) A_i) B_i: the residual is added to the
    all-reduced sum (ai-hpc.org §2: local_out = AllReduce(mid @ w2); out = x + local_out)."""
    return _f64(x) + tp_mlp(layer_norm(x, eps), shards)


def block_mlp_rows(x, shards, rows, eps: float = LN_EPS):
    """Rows `rows` of block_mlp: every step is row-wise in x."""
    return block_mlp(_f64(x)[rows], shards, eps)


def layer_norm_backward(x, g, eps: float = LN_EPS):
    """The gradient of sum(layer_norm(x) * g) with respect to x, row by row.

    The backward of the block (ai-hpc.org "LLM Lab Notes 06", §2 step 8) passes
    through the normalisation. For one row with y = (x - mu) r,
    r = (var + eps)^(-1/2), differentiating mu and var gives the Jacobian
        dy_j/dx_k = r (delta_jk - 1/D - y_j y_k / D),
    which is symmetric; the gradient is that matrix applied to g, built here
    for each row as written.
    """
    x = _f64(x)
    g = _f64(g)
    D = x.shape[-1]
    y = layer_norm(x, eps)
    mu = x.mean(axis=-1, keepdims=True)
    r = 1.0 / np.sqrt(((x - mu) ** 2).mean(axis=-1, keepdims=True) + eps)
    out = np.empty_like(x)
    eye = np.eye(D)
    for t in range(x.shape[0]):
        J = r[t, 0] * (eye - 1.0 / D - np.outer(y[t], y[t]) / D)
        out[t] = J @ g[t]
    return out


def block_mlp_backward(x, dout, shards, eps: float = LN_EPS):
    """Gradients of L = sum(block_mlp(x) * dout): (dx, [dA_i], [dB_i]).

    The residual passes dout to x unchanged; the MLP sees the normalised input
    and the same upstream gradient, and its input gradient goes back through
    the normalisation.
    """
    x = _f64(x)
    dout = _f64(dout)
    dxn, dA, dB = tp_mlp_backward(layer_norm(x, eps), dout, shards)
    return dout + layer_norm_backward(x, dxn, eps), dA, dB


def block_mlp_backward_dx_rows(x, dout, shards, rows, eps: float = LN_EPS):
    """Rows `rows` of block_mlp_backward's dx: each row needs only its own x and dout rows."""
    dx, _, _ = block_mlp_backward(_f64(x)[rows], _f64(dout)[rows], shards, eps)
    return dx


# ---------------------------------------------------------------------------
# Sequence-parallel form of the sum (duoan.github.io "Tensor Parallelism in
# Megatron-LM", "Row split": the partials are summed by an all-reduce, or by
# reduce-scatter / all-gather when the sequence is split). With n ranks and T
# divisible by n, rank j holds token rows j*T/n .. (j+1)*T/n - 1 of X and of
# the output; the all-gather assembles X from the slices in rank order, and
# the reduce-scatter hands rank j the same rows of the shard-ordered sum.
# ---------------------------------------------------------------------------

def split_rows(M, n: int):
    """Rank j's token slice: rows j*T/n .. (j+1)*T/n - 1 (T divisible by n)."""
    M = _f64(M)
    T = M.shape[0]
    if n <= 0 or T % n != 0:
        raise ValueError(f"T={T} is not divisible by n={n}")
    Ts = T // n
    return [M[j * Ts:(j + 1) * Ts] for j in range(n)]


def all_gather(slices):
    """The full [T, D] tensor from the n rank slices, in rank order."""
    return np.concatenate([_f64(s) for s in slices], axis=0)


def reduce_scatter(partials, n: int):
    """Rank j's slice of ((P_0 + P_1) + ...) + P_{n-1}, summed slice by slice."""
    parts = [split_rows(P, n) for P in partials]
    out = []
    for j in range(n):
        acc = parts[0][j].copy()
        for i in range(1, len(parts)):
            acc = acc + parts[i][j]
        out.append(acc)
    return out


def tp_mlp_sp(X_slices, shards):
    """Sequence-parallel forward: all-gather X, every shard's partial, reduce-scatter."""
    X = all_gather(X_slices)
    partials = [shard_partial(X, A_i, B_i)[1] for (A_i, B_i) in shards]
    return reduce_scatter(partials, len(X_slices))


def tp_mlp_sp_backward(X_slices, dY_slices, shards):
    """Sequence-parallel backward: all-gather X and dY, the shards' gradients,
    and the dX partials reduce-scattered to the ranks: ([dX_j], [dA_i], [dB_i])."""
    X = all_gather(X_slices)
    dY = all_gather(dY_slices)
    dA, dB, dX_parts = [], [], []
    for A_i, B_i in shards:
        A_i = _f64(A_i)
        B_i = _f64(B_i)
        P_i = X @ A_i
        dP_i = (dY @ B_i.T) * gelu_grad(P_i)
        dB.append(gelu(P_i).T @ dY)
        dA.append(X.T @ dP_i)
        dX_parts.append(dP_i @ A_i.T)
    return reduce_scatter(dX_parts, len(X_slices)), dA, dB


# ---------------------------------------------------------------------------
# Head-split attention (duoan.github.io "Tensor Parallelism in Megatron-LM",
# §4 "Attention: Split Heads"; ai-hpc.org "LLM Lab Notes 06" §2 steps 2-3):
# with H heads of size d_h = D / H, rank i owns heads i*H/n .. (i+1)*H/n - 1,
# i.e. columns i*D/n .. (i+1)*D/n - 1 of W^Q, W^K, W^V (column-parallel) and
# the same rows of the output projection W^O (row-parallel). Per head and per
# sequence of the batch, O = softmax(Q K^T / sqrt(d_h)) V with no mask; the
# output projection's partials are summed like the MLP's.
# X is [T, D] with T = batch * seq, sequence b occupying rows b*seq ..
# (b+1)*seq - 1.
# ---------------------------------------------------------------------------

def softmax_rows(S):
    """Row-wise softmax; the row maximum is subtracted first (the value is unchanged)."""
    S = _f64(S)
    E = np.exp(S - S.max(axis=-1, keepdims=True))
    return E / E.sum(axis=-1, keepdims=True)


def attention_core(Q, K, V, batch: int, heads: int):
    """O [T, H*d_h]: for every sequence b and head h, softmax(Q_bh K_bh^T / sqrt(d_h)) V_bh."""
    Q, K, V = _f64(Q), _f64(K), _f64(V)
    T, HD = Q.shape
    if T % batch != 0 or HD % heads != 0:
        raise ValueError("T must be divisible by batch and the width by heads")
    s, dh = T // batch, HD // heads
    O = np.empty_like(Q)
    for b in range(batch):
        r = slice(b * s, (b + 1) * s)
        for h in range(heads):
            c = slice(h * dh, (h + 1) * dh)
            P = softmax_rows(Q[r, c] @ K[r, c].T / math.sqrt(dh))
            O[r, c] = P @ V[r, c]
    return O


def mha(X, batch: int, Wq, Wk, Wv, Wo, heads: int):
    """Unsplit multi-head attention: attention_core(X Wq, X Wk, X Wv) Wo."""
    X = _f64(X)
    return attention_core(X @ _f64(Wq), X @ _f64(Wk), X @ _f64(Wv), batch, heads) @ _f64(Wo)


def shard_attention(Wq, Wk, Wv, Wo, heads: int, n: int):
    """Rank i's (Wq_i, Wk_i, Wv_i, Wo_i): its heads' columns of Wq, Wk, Wv and rows of Wo."""
    Wq, Wk, Wv, Wo = _f64(Wq), _f64(Wk), _f64(Wv), _f64(Wo)
    D = Wq.shape[0]
    if n <= 0 or heads % n != 0 or D % heads != 0:
        raise ValueError(f"heads={heads} must be divisible by n={n} and D={D} by heads")
    Dn = D // n
    c = [slice(i * Dn, (i + 1) * Dn) for i in range(n)]
    return [(Wq[:, c[i]], Wk[:, c[i]], Wv[:, c[i]], Wo[c[i], :]) for i in range(n)]


def attn_shard_partial(X, batch: int, shard, local_heads: int):
    """Rank i's work: O_i = attention over its local heads, and Y_i = O_i Wo_i. Returns (O_i, Y_i)."""
    X = _f64(X)
    Wq, Wk, Wv, Wo = shard
    O = attention_core(X @ Wq, X @ Wk, X @ Wv, batch, local_heads)
    return O, O @ Wo


def tp_attention(X, batch: int, shards, heads: int, return_partials: bool = False):
    """Every rank's partial, then the shard-ordered sum Y = ((Y_0 + Y_1) + ...) + Y_{n-1}."""
    lh = heads // len(shards)
    partials = [attn_shard_partial(X, batch, sh, lh) for sh in shards]
    Y = partials[0][1].copy()
    for _, Y_i in partials[1:]:
        Y = Y + Y_i
    if return_partials:
        return Y, partials
    return Y


def tp_attention_rows(X, batch: int, shards, heads: int, seqs):
    """The rows of tp_attention belonging to sequences `seqs` (each sequence attends only to itself)."""
    X = _f64(X)
    s = X.shape[0] // batch
    rows = np.concatenate([np.arange(b * s, (b + 1) * s) for b in seqs])
    return tp_attention(X[rows], len(seqs), shards, heads)
