"""GPU parity of head-split attention (duoan.github.io "Tensor Parallelism in
Megatron-LM", §4), called through the C ABI and compared with the float64
oracle.

Tolerances are the MLP's: fp32 path max|err| <= 1e-4 max|ref|; bf16 path
relative Frobenius <= 5e-3 and max <= 2e-2 max|ref|, for every rank's head
outputs O_i and for Y. The bf16 path rounds Q, K, V (the projection's output)
and the softmax weights P to bf16 where they become tensor-core operands,
while the oracle keeps float64 throughout. Weight slicing is bit-exact.
"""

import numpy as np
import pytest
import torch

import oracle
from tpmlp_inputs import ATTN_WORKLOADS, AttnWorkload, make_attn_inputs

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


def workload(name, batch, seq, D, heads, n, dtype):
    return AttnWorkload(name, batch, seq, D, heads, n, dtype, 1.0, 1.0 / np.sqrt(D))


SMALL_BF16 = [
    # name, batch, seq, D, heads, n
    ("two_ranks", 2, 128, 256, 4, 2),
    ("ragged_seq", 3, 200, 128, 2, 1),      # a partial query tile and key block
    ("seq512", 1, 512, 512, 8, 4),          # 4 key blocks, two P phases
    ("short_seq", 4, 8, 64, 1, 1),
    ("three_blocks", 2, 384, 128, 2, 2),
    ("phase_tail", 1, 264, 64, 1, 1),       # 5 key chunks: phases of 4 and 1
    ("many_ranks", 2, 64, 1024, 16, 16),
    ("long_seq", 2, 640, 128, 2, 1),        # streaming kernel: 5 key blocks
    ("seq1024", 1, 1024, 256, 4, 2),
    ("long_ragged", 1, 1000, 64, 1, 1),     # streaming kernel, partial last key block
]
SMALL_F32 = [
    ("two_ranks", 2, 16, 64, 4, 2),
    ("dh16", 3, 33, 48, 3, 3),
    ("dh128", 1, 100, 256, 2, 2),
    ("seq512", 2, 512, 64, 1, 1),
    ("seq700", 1, 700, 64, 2, 2),
]


def _random_bf16_cases(count, seed):
    """Seeded (name, batch, seq, D, heads, n) for the bf16 path: head size 64,
    seq any multiple of 8, heads a multiple of the rank count."""
    rng = np.random.default_rng(seed)
    out = []
    while len(out) < count:
        n = int(rng.choice([1, 2, 4, 8]))
        heads = n * int(rng.integers(1, 5))
        seq = 8 * int(rng.integers(1, 161))   # 8 .. 1280
        batch = int(rng.integers(1, 5))
        if batch * seq <= 3000:
            out.append((f"random{len(out)}", batch, seq, 64 * heads, heads, n))
    return out


CASES = ([c + ("bf16",) for c in SMALL_BF16] + [c + ("f32",) for c in SMALL_F32] +
         [c + ("bf16",) for c in _random_bf16_cases(6, 61)])


def oracle_parts(inp, w):
    shards = oracle.shard_attention(f64(inp["Wq"]), f64(inp["Wk"]), f64(inp["Wv"]), f64(inp["Wo"]), w.heads, w.N)
    return oracle.tp_attention(f64(inp["X"]), w.batch, shards, w.heads, return_partials=True)


@pytest.mark.parametrize("case", CASES, ids=[f"{c[0]}-{c[-1]}" for c in CASES])
def test_attention_heads_and_forward_against_oracle(tp, case):
    w = workload(*case)
    inp = make_attn_inputs(w, seed=51)
    Y_ref, parts = oracle_parts(inp, w)
    d = {k: v.cuda() for k, v in inp.items()}
    sh = tp.tpmlp_attn_shard(d["Wq"], d["Wk"], d["Wv"], d["Wo"], w.heads, w.N)
    O = tp.tpmlp_attn_heads(d["X"], w.batch, sh)
    tp.tpmlp_check_status()
    for i, (O_ref, _) in enumerate(parts):
        check(f64(O[i]), O_ref, w.dtype, f"O_{i}")
    outs = {}
    for mode in ("faithful", "fused"):
        outs[mode] = tp.tpmlp_attn_forward(d["X"], w.batch, sh, mode)
        tp.tpmlp_check_status()
        check(f64(outs[mode]), Y_ref, w.dtype, f"Y {mode}")
    assert torch.equal(tp.tpmlp_attn_forward(d["X"], w.batch, sh, "faithful"), outs["faithful"])
    sh.free()


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_attention_weight_layout_bit_exact(tp, dtype):
    D, heads, n = 256, 4, 2
    g = torch.Generator().manual_seed(7)
    W = [torch.randn((D, D), generator=g).to(dtype).cuda() for _ in range(4)]
    sh = tp.tpmlp_attn_shard(*W, heads, n)
    Dn = D // n
    for i in range(n):
        wqkv, wo = sh.get(i)
        cols = slice(i * Dn, (i + 1) * Dn)
        ref_qkv = torch.cat([W[0][:, cols], W[1][:, cols], W[2][:, cols]], dim=1)
        ref_wo = W[3][cols, :]
        if dtype == torch.bfloat16:
            ref_qkv, ref_wo = ref_qkv.t(), ref_wo.t()
        assert torch.equal(wqkv, ref_qkv) and torch.equal(wo, ref_wo)
    sh.free()


@pytest.mark.parametrize("name", ["attn_tiny_fp32", "attn_seq128", "attn_seq256", "attn_seq512", "attn_long1024",
                                  "attn_long4096"])
def test_attention_workload_full_oracle(tp, name):
    w = ATTN_WORKLOADS[name]
    inp = make_attn_inputs(w, seed=0)
    Y_ref, parts = oracle_parts(inp, w)
    d = {k: v.cuda() for k, v in inp.items()}
    sh = tp.tpmlp_attn_shard(d["Wq"], d["Wk"], d["Wv"], d["Wo"], w.heads, w.N)
    O = tp.tpmlp_attn_heads(d["X"], w.batch, sh)
    for i, (O_ref, _) in enumerate(parts):
        check(f64(O[i]), O_ref, w.dtype, f"{name} O_{i}")
    for mode in ("faithful", "fused"):
        check(f64(tp.tpmlp_attn_forward(d["X"], w.batch, sh, mode)), Y_ref, w.dtype, f"{name} Y {mode}")
    tp.tpmlp_check_status()
    sh.free()


def test_attention_argument_errors(tp):
    D = 128
    Wb = [torch.zeros((D, D), dtype=torch.bfloat16, device="cuda") for _ in range(4)]
    with pytest.raises(tp.TpmlpError):  # bf16 head size 32
        tp.tpmlp_attn_shard(*Wb, 4, 2)
    with pytest.raises(tp.TpmlpError):  # heads not divisible by n
        tp.tpmlp_attn_shard(*Wb, 2, 4)
    sh = tp.tpmlp_attn_shard(*Wb, 2, 2)
    X = torch.zeros((2 * 12, D), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(tp.TpmlpError):  # bf16 needs seq % 8 == 0
        tp.tpmlp_attn_forward(X, 2, sh)
    sh.free()
    Wf = [torch.zeros((D, D), dtype=torch.float32, device="cuda") for _ in range(4)]
    shf = tp.tpmlp_attn_shard(*Wf, 2, 2)
    X = torch.zeros((8200, D), dtype=torch.float32, device="cuda")
    with pytest.raises(tp.TpmlpError):  # fp32 seq 8200 > 8192
        tp.tpmlp_attn_forward(X, 1, shf)
    shf.free()


@pytest.mark.parametrize("case", [c + ("bf16",) for c in SMALL_BF16 if c[2] <= 512], ids=lambda c: c[0])
def test_exact_kernel_matches_oracle(tp, case, monkeypatch):
    # TPMLP_ATTN_KERNEL=0 runs the exact kernel (whole score row in tensor
    # memory, up to 512 tokens) instead of the default streaming one; both
    # must meet the same tolerance.
    monkeypatch.setenv("TPMLP_ATTN_KERNEL", "0")
    w = workload(*case)
    inp = make_attn_inputs(w, seed=52)
    Y_ref, parts = oracle_parts(inp, w)
    d = {k: v.cuda() for k, v in inp.items()}
    sh = tp.tpmlp_attn_shard(d["Wq"], d["Wk"], d["Wv"], d["Wo"], w.heads, w.N)
    O = tp.tpmlp_attn_heads(d["X"], w.batch, sh)
    tp.tpmlp_check_status()
    for i, (O_ref, _) in enumerate(parts):
        check(f64(O[i]), O_ref, "bf16", f"exact-kernel O_{i}")
    check(f64(tp.tpmlp_attn_forward(d["X"], w.batch, sh, "fused")), Y_ref, "bf16", "exact-kernel Y")
    sh.free()


def test_streaming_kernel_handles_large_logits(tp, monkeypatch):
    # Logits of tens: the streaming kernel's running maximum rescales earlier
    # blocks by tiny factors. Both kernels see the same bf16 Q, K, V here, so
    # they must agree closely (the oracle's exact Q, K differ from the rounded
    # ones by more than the tolerance once logits are this large), and every
    # output must be finite.
    w = workload("large_logits", 2, 512, 128, 2, 1, "bf16")
    inp = make_attn_inputs(w, seed=53)
    inp["X"] = (inp["X"].float() * 6.0).to(torch.bfloat16)
    d = {k: v.cuda() for k, v in inp.items()}
    sh = tp.tpmlp_attn_shard(d["Wq"], d["Wk"], d["Wv"], d["Wo"], w.heads, w.N)
    monkeypatch.setenv("TPMLP_ATTN_KERNEL", "0")
    O_exact = tp.tpmlp_attn_heads(d["X"], w.batch, sh).float()
    monkeypatch.setenv("TPMLP_ATTN_KERNEL", "1")
    O_strm = tp.tpmlp_attn_heads(d["X"], w.batch, sh).float()
    tp.tpmlp_check_status()
    assert torch.isfinite(O_exact).all() and torch.isfinite(O_strm).all()
    rel = (torch.linalg.norm(O_strm - O_exact) / torch.linalg.norm(O_exact)).item()
    assert rel <= 1e-2, rel
    sh.free()


# The streaming kernel's barriers are used once per key block with parity
# waits; a wait that let a barrier run two phases ahead would hang (and then
# time out) only when one role falls a block behind. Many back-to-back
# launches on long and ragged sequences must all finish without a timeout and
# give the same bits every time (each launch computes the same thing in the
# same order).
@pytest.mark.parametrize("shape", [(1, 4096, 16, 4), (2, 1000, 16, 4), (8, 512, 16, 4)], ids=lambda s: f"b{s[0]}_s{s[1]}")
def test_streaming_kernel_repeated_launches_bit_identical(tp, shape):
    batch, seq, heads, n = shape
    aw = AttnWorkload("rep", batch, seq, 1024, heads, n, "bf16", 1.0, 0.03)
    ai = {k: v.cuda() for k, v in make_attn_inputs(aw, seed=97).items()}
    sh = tp.tpmlp_attn_shard(ai["Wq"], ai["Wk"], ai["Wv"], ai["Wo"], aw.heads, aw.N)
    ref = tp.tpmlp_attn_heads(ai["X"], aw.batch, sh).clone()
    O = torch.empty_like(ref)
    for i in range(200):
        tp.tpmlp_attn_heads(ai["X"], aw.batch, sh, O)
        if i % 50 == 49:
            tp.tpmlp_check_status()
            assert torch.equal(O, ref), f"launch {i} differs"
    tp.tpmlp_check_status()
