"""Launch variants that the environment selects (read once per
process, so each runs in a child process): TPMLP_TC_KERNEL=0 (single-CTA
tiles everywhere) and =1 (the default: CTA pairs for every product with
enough 256 x 256 tiles). Each child checks, against the float64 oracle with
the bf16 tolerances, every epilogue the pair kernel is tested with: GeLU,
fp32 partials and the fused sum (TMA stores), the backward's activation step,
the saved pre-activation, the block's residual, the sequence-parallel slice
outputs and attention's QKV projection with V written transposed. TPMLP_PDL=0
(kernels launched without programmatic dependent launch) must reproduce the
default's results bit for bit. TPMLP_NARROW=0 (no 128 x 64 single-CTA tiles for
a small shard-ordered sum) must match both the oracle and the default."""

import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = r'''
import numpy as np, torch
import oracle
import tensor_transformer_mlp_column_gb300 as tp
from tpmlp_inputs import Workload, make_inputs, make_block_inputs, AttnWorkload, make_attn_inputs

def check(got, ref, what):
    got = np.asarray(got, np.float64); ref = np.asarray(ref, np.float64)
    fro = np.linalg.norm(got - ref) / np.linalg.norm(ref); mx = np.max(np.abs(got - ref)) / np.max(np.abs(ref))
    assert fro <= 5e-3 and mx <= 2e-2, (what, fro, mx)

f64 = lambda t: t.detach().to("cpu", torch.float64).numpy()
torch.cuda.set_device(0)
# T=2048, D=2048, F=4096, N=4: every product has enough 256 x 256 tiles for pairs.
w = Workload("v", 2048, 2048, 4096, 4, "bf16", 1.0, 0.02, 0.02, 1.0, True)
inp = make_inputs(w, seed=71)
X, A, B, dY = (f64(inp[k]) for k in ("X", "A", "B", "dY"))
shards = oracle.shard_mlp(A, B, w.N)
rows = list(range(0, w.T, 17))
Y_ref = oracle.tp_mlp_rows(X, shards, rows)
d = {k: v.cuda() for k, v in inp.items()}
sh = tp.tpmlp_shard(d["A"], d["B"], w.N)
idx = torch.tensor(rows, device="cuda")
for mode in ("faithful", "fused"):
    check(f64(tp.tpmlp_forward(d["X"], sh, mode).index_select(0, idx)), Y_ref, "Y " + mode)
Y, P = tp.tpmlp_forward_save(d["X"], sh, "fused")
check(f64(P[1].index_select(0, idx)), X[rows] @ shards[1][0], "saved P")
dX, dA, dB = tp.tpmlp_backward(d["X"], d["dY"], sh, "fused")
check(f64(dX.index_select(0, idx)), oracle.tp_mlp_backward_dx_rows(X, dY, shards, rows), "dX")
cols = list(range(0, w.Fs, 37))
cidx = torch.tensor(cols, device="cuda")
check(f64(dA[2].index_select(1, cidx)), oracle.grad_A_cols(X, dY, shards[2][0], shards[2][1], cols), "dA_2")
check(f64(dB[3].index_select(0, cidx)), oracle.grad_B_rows(X, dY, shards[3][0], cols), "dB_3")
bi = make_block_inputs(w, seed=72)
x = f64(bi["x"])
out = tp.tpmlp_block_forward(bi["x"].cuda(), tp.tpmlp_shard(bi["A"].cuda(), bi["B"].cuda(), w.N), "fused")
check(f64(out.index_select(0, idx)), oracle.block_mlp_rows(x, oracle.shard_mlp(f64(bi["A"]), f64(bi["B"]), w.N), rows), "block")
Ys = tp.tpmlp_forward_sp([c.clone() for c in torch.chunk(d["X"], w.N)], sh, "fused")
assert torch.equal(torch.cat(Ys), tp.tpmlp_forward(d["X"], sh, "fused")), "sequence-parallel slices"
aw = AttnWorkload("va", 4, 512, 1024, 16, 4, "bf16", 1.0, 0.03)
ai = make_attn_inputs(aw, seed=73)
a64 = {k: f64(v) for k, v in ai.items()}
ash = oracle.shard_attention(a64["Wq"], a64["Wk"], a64["Wv"], a64["Wo"], aw.heads, aw.N)
Ya_ref, parts = oracle.tp_attention(a64["X"], aw.batch, ash, aw.heads, return_partials=True)
ad = {k: v.cuda() for k, v in ai.items()}
sha = tp.tpmlp_attn_shard(ad["Wq"], ad["Wk"], ad["Wv"], ad["Wo"], aw.heads, aw.N)
O = tp.tpmlp_attn_heads(ad["X"], aw.batch, sha)
for i, (O_ref, _) in enumerate(parts):
    check(f64(O[i]), O_ref, f"attention O_{i}")
check(f64(tp.tpmlp_attn_forward(ad["X"], aw.batch, sha, "faithful")), Ya_ref, "attention Y")
tp.tpmlp_check_status()
print("ok")
'''


@pytest.mark.parametrize("family", ["0", "1"], ids=["single_cta", "pair"])
def test_gemm_variant_against_oracle(family):
    import torch

    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__

    __graft_entry__.build()
    env = dict(os.environ, TPMLP_TC_KERNEL=family)
    r = subprocess.run([sys.executable, "-c", CHILD], env=env, cwd=ROOT, capture_output=True, text=True, timeout=900)
    assert r.returncode == 0 and r.stdout.strip().endswith("ok"), r.stdout[-2000:] + r.stderr[-4000:]


# Programmatic dependent launch on (the default) and off (TPMLP_PDL=0, also read
# once per process): every call must give the same bits either way, since each
# kernel waits for its predecessor before its first global access.
PDL_CHILD = r'''
import sys, torch
import tensor_transformer_mlp_column_gb300 as tp
from tpmlp_inputs import Workload, make_inputs, make_block_inputs, AttnWorkload, make_attn_inputs
torch.cuda.set_device(0)
out = {}
for name, T, D, F, N in (("pair", 1000, 1024, 4096, 4), ("single", 96, 128, 512, 2)):
    w = Workload(name, T, D, F, N, "bf16", 1.0, 0.02, 0.02, 1.0, True)
    inp = {k: v.cuda() for k, v in make_inputs(w, seed=81).items()}
    sh = tp.tpmlp_shard(inp["A"], inp["B"], w.N)
    bi = {k: v.cuda() for k, v in make_block_inputs(w, seed=82, with_dout=True).items()}
    shb = tp.tpmlp_shard(bi["A"], bi["B"], w.N)
    for mode in ("faithful", "fused"):
        k = f"{name}_{mode}_"
        out[k + "Y"] = tp.tpmlp_forward(inp["X"], sh, mode)
        dX, dA, dB = tp.tpmlp_backward(inp["X"], inp["dY"], sh, mode)
        out[k + "dX"], out[k + "dA"], out[k + "dB"] = dX, torch.stack(list(dA)), torch.stack(list(dB))
        out[k + "block"] = tp.tpmlp_block_forward(bi["x"], shb, mode)
        out[k + "block_dx"] = tp.tpmlp_block_backward(bi["x"], bi["dout"], shb, mode)[0]
        out[k + "sp"] = torch.cat(tp.tpmlp_forward_sp([c.clone() for c in torch.chunk(inp["X"], w.N)], sh, mode))
aw = AttnWorkload("pa", 2, 256, 512, 8, 2, "bf16", 1.0, 0.03)
ai = {k: v.cuda() for k, v in make_attn_inputs(aw, seed=83).items()}
sha = tp.tpmlp_attn_shard(ai["Wq"], ai["Wk"], ai["Wv"], ai["Wo"], aw.heads, aw.N)
for mode in ("faithful", "fused"):
    out["attn_" + mode] = tp.tpmlp_attn_forward(ai["X"], aw.batch, sha, mode)
torch.cuda.synchronize()
tp.tpmlp_check_status()
torch.save({k: v.cpu() for k, v in out.items()}, sys.argv[1])
print("ok")
'''


def test_dependent_launch_off_gives_identical_bits(tmp_path):
    import torch

    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__

    __graft_entry__.build()
    results = {}
    for flag in ("1", "0"):
        path = str(tmp_path / f"pdl{flag}.pt")
        env = dict(os.environ, TPMLP_PDL=flag)
        r = subprocess.run([sys.executable, "-c", PDL_CHILD, path], env=env, cwd=ROOT, capture_output=True,
                           text=True, timeout=900)
        assert r.returncode == 0 and r.stdout.strip().endswith("ok"), r.stdout[-2000:] + r.stderr[-4000:]
        results[flag] = torch.load(path)
    assert results["1"].keys() == results["0"].keys()
    for k in results["1"]:
        assert torch.equal(results["1"][k], results["0"][k]), f"{k} differs with dependent launch off"


# Narrow single-CTA tiles (128 x 64) for a shard-ordered sum with few output
# tiles, on by default and off with TPMLP_NARROW=0 (each setting in a child
# process of its own):
# both must match the oracle, and each other to within fp32 rounding, since an
# output element is summed over the same K blocks in the same order either way.
NARROW_CHILD = r'''
import sys, numpy as np, torch
import oracle
import tensor_transformer_mlp_column_gb300 as tp
from tpmlp_inputs import Workload, make_inputs, make_block_inputs

def check(got, ref, what):
    got = np.asarray(got, np.float64); ref = np.asarray(ref, np.float64)
    fro = np.linalg.norm(got - ref) / np.linalg.norm(ref); mx = np.max(np.abs(got - ref)) / np.max(np.abs(ref))
    assert fro <= 5e-3 and mx <= 2e-2, (what, fro, mx)

f64 = lambda t: t.detach().to("cpu", torch.float64).numpy()
torch.cuda.set_device(0)
out = {}
# 8 x 16 and 8 x 15 (ragged rows and columns) tiles of 128 x 64, a single round.
for name, T, D, F, N in (("seq128", 1024, 1024, 4096, 4), ("ragged", 1000, 960, 1920, 2)):
    w = Workload(name, T, D, F, N, "bf16", 1.0, 0.02, 0.02)
    inp = make_inputs(w, seed=91)
    shards = oracle.shard_mlp(f64(inp["A"]), f64(inp["B"]), N)
    rows = list(range(0, T, 13))
    idx = torch.tensor(rows, device="cuda")
    d = {k: v.cuda() for k, v in inp.items()}
    sh = tp.tpmlp_shard(d["A"], d["B"], N)
    Y = tp.tpmlp_forward(d["X"], sh, "fused")
    check(f64(Y.index_select(0, idx)), oracle.tp_mlp_rows(f64(inp["X"]), shards, rows), name + " fused")
    out[name + "_Y"] = Y
    bi = make_block_inputs(w, seed=92)
    shb = tp.tpmlp_shard(bi["A"].cuda(), bi["B"].cuda(), N)
    blk = tp.tpmlp_block_forward(bi["x"].cuda(), shb, "fused")
    check(f64(blk.index_select(0, idx)),
          oracle.block_mlp_rows(f64(bi["x"]), oracle.shard_mlp(f64(bi["A"]), f64(bi["B"]), N), rows), name + " block")
    out[name + "_block"] = blk
    if T % N == 0:
        out[name + "_sp"] = torch.cat(tp.tpmlp_forward_sp([c.clone() for c in torch.chunk(d["X"], N)], sh, "fused"))
        assert torch.equal(out[name + "_sp"], Y), name + " sequence-parallel slices"
torch.cuda.synchronize()
tp.tpmlp_check_status()
torch.save({k: v.cpu() for k, v in out.items()}, sys.argv[1])
print("ok")
'''


def test_narrow_single_cta_tiles_against_oracle_and_wide(tmp_path):
    import torch

    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__

    __graft_entry__.build()
    results = {}
    for flag in ("1", "0"):
        path = str(tmp_path / f"narrow{flag}.pt")
        env = dict(os.environ, TPMLP_NARROW=flag)
        r = subprocess.run([sys.executable, "-c", NARROW_CHILD, path], env=env, cwd=ROOT, capture_output=True,
                           text=True, timeout=900)
        assert r.returncode == 0 and r.stdout.strip().endswith("ok"), r.stdout[-2000:] + r.stderr[-4000:]
        results[flag] = torch.load(path)
    assert results["1"].keys() == results["0"].keys()
    for k in results["1"]:
        a, b = results["1"][k].double(), results["0"][k].double()
        assert (a - b).abs().max() <= 1e-5 * b.abs().max(), f"{k}: narrow and wide tiles differ"


# The forward's two products in one persistent launch (the default for
# products small enough) against two launches (TPMLP_FWD_PERSIST=0, read once
# per process, so each setting runs in a child process): every tile sums the
# same K blocks in the same order either way, so the outputs agree bit for
# bit, and both match the oracle. Shapes: GPT-2-small and seq 512 (the
# persistent launch in both modes), a ragged token count (last band partial),
# 8 shards, ragged T, D and F/n together (T=2500, D=1288, F/n=1000), 16
# shards (faithful only: its shard-ordered sum has too few pair tiles), and a
# ragged D whose shard-ordered sum runs in 256 x 128 tiles (T=1700, D=1160;
# the ragged-T and 8-shard shapes take those tiles as well), and a mid-size
# shape of 20 rounds of tiles in faithful mode (T=8192, D=1024, F=4096, N=8).
PERSIST_CHILD = r"""
import sys, numpy as np, torch
import oracle
import tensor_transformer_mlp_column_gb300 as tp
from tpmlp_inputs import Workload, make_inputs

def check(got, ref, what):
    got = np.asarray(got, np.float64); ref = np.asarray(ref, np.float64)
    fro = np.linalg.norm(got - ref) / np.linalg.norm(ref); mx = np.max(np.abs(got - ref)) / np.max(np.abs(ref))
    assert fro <= 5e-3 and mx <= 2e-2, (what, fro, mx)

f64 = lambda t: t.detach().to("cpu", torch.float64).numpy()
torch.cuda.set_device(0)
out = {}
for name, T, D, F, N in (("gpt2", 4096, 768, 3072, 4), ("seq512", 4096, 1024, 4096, 4),
                         ("ragged", 3000, 768, 3072, 4), ("eight", 2048, 1024, 8192, 8),
                         ("ragged_all", 2500, 1288, 4000, 4), ("sixteen", 1024, 1024, 4096, 16),
                         ("ragged_narrow", 1700, 1160, 4096, 4), ("mid", 8192, 1024, 4096, 8)):
    w = Workload(name, T, D, F, N, "bf16", 1.0, 0.02, 0.02)
    inp = make_inputs(w, seed=93)
    shards = oracle.shard_mlp(f64(inp["A"]), f64(inp["B"]), N)
    rows = list(range(0, T, 23))
    idx = torch.tensor(rows, device="cuda")
    d = {k: v.cuda() for k, v in inp.items()}
    sh = tp.tpmlp_shard(d["A"], d["B"], N)
    Y_ref = oracle.tp_mlp_rows(f64(inp["X"]), shards, rows)
    for mode in ("faithful", "fused"):
        Y = tp.tpmlp_forward(d["X"], sh, mode)
        check(f64(Y.index_select(0, idx)), Y_ref, name + " " + mode)
        out[name + "_" + mode] = Y
        out[name + "_" + mode + "_again"] = tp.tpmlp_forward(d["X"], sh, mode)
torch.cuda.synchronize()
tp.tpmlp_check_status()
torch.save({k: v.cpu() for k, v in out.items()}, sys.argv[1])
print("ok")
"""


def test_persistent_forward_matches_two_launches(tmp_path):
    import torch

    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__

    __graft_entry__.build()
    results = {}
    for flag in ("1", "0"):
        path = str(tmp_path / f"persist{flag}.pt")
        env = dict(os.environ, TPMLP_FWD_PERSIST=flag)
        r = subprocess.run([sys.executable, "-c", PERSIST_CHILD, path], env=env, cwd=ROOT, capture_output=True,
                           text=True, timeout=900)
        assert r.returncode == 0 and r.stdout.strip().endswith("ok"), flag + r.stdout[-2000:] + r.stderr[-4000:]
        results[flag] = torch.load(path)
    for k in results["1"]:
        assert torch.equal(results["1"][k], results["0"][k]), f"{k}: one launch and two launches differ"
        if k.endswith("_again"):
            assert torch.equal(results["1"][k], results["1"][k[:-6]]), f"{k}: not reproducible"


# The backward's first step in the dual-accumulator kernel (the default for
# products with CTA-pair tiles) against two products (TPMLP_BWD_DUAL=0, read
# once per process): both match the oracle on every gradient, on ragged T, D
# and F/n and on 16 shards. (They are not bit-identical: the dual kernel keeps
# GeLU'(P) in fp16 between its two phases.)
DUAL_CHILD = r"""
import sys, numpy as np, torch
import oracle
import tensor_transformer_mlp_column_gb300 as tp
from tpmlp_inputs import Workload, make_inputs

def check(got, ref, what):
    got = np.asarray(got, np.float64); ref = np.asarray(ref, np.float64)
    fro = np.linalg.norm(got - ref) / np.linalg.norm(ref); mx = np.max(np.abs(got - ref)) / np.max(np.abs(ref))
    assert fro <= 5e-3 and mx <= 2e-2, (what, fro, mx)

f64 = lambda t: t.detach().to("cpu", torch.float64).numpy()
torch.cuda.set_device(0)
for name, T, D, F, N in (("ragged_all", 2500, 1288, 4000, 4), ("sixteen", 1024, 1024, 4096, 16),
                         ("tall", 6000, 512, 2048, 2)):
    w = Workload(name, T, D, F, N, "bf16", 1.0, 0.03, 0.03, 1.0, True)
    inp = make_inputs(w, seed=95)
    X, A, B, dY = (f64(inp[k]) for k in ("X", "A", "B", "dY"))
    shards = oracle.shard_mlp(A, B, N)
    rows = list(range(0, T, 29))
    cols = list(range(0, w.Fs, 31))
    idx, cidx = torch.tensor(rows, device="cuda"), torch.tensor(cols, device="cuda")
    d = {k: v.cuda() for k, v in inp.items()}
    sh = tp.tpmlp_shard(d["A"], d["B"], N)
    dX_ref = oracle.tp_mlp_backward_dx_rows(X, dY, shards, rows)
    for mode in ("faithful", "fused"):
        dX, dA, dB = tp.tpmlp_backward(d["X"], d["dY"], sh, mode)
        check(f64(dX.index_select(0, idx)), dX_ref, f"{name} {mode} dX")
        for i in (0, N - 1):
            check(f64(dA[i].index_select(1, cidx)), oracle.grad_A_cols(X, dY, shards[i][0], shards[i][1], cols),
                  f"{name} {mode} dA_{i}")
            check(f64(dB[i].index_select(0, cidx)), oracle.grad_B_rows(X, dY, shards[i][0], cols),
                  f"{name} {mode} dB_{i}")
    tp.tpmlp_check_status()
print("ok")
"""


@pytest.mark.parametrize("flag", ["1", "0"], ids=["dual", "two_products"])
def test_dual_and_two_product_backward_against_oracle(flag):
    import torch

    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__

    __graft_entry__.build()
    env = dict(os.environ, TPMLP_BWD_DUAL=flag)
    r = subprocess.run([sys.executable, "-c", DUAL_CHILD], env=env, cwd=ROOT, capture_output=True, text=True,
                       timeout=900)
    assert r.returncode == 0 and r.stdout.strip().endswith("ok"), r.stdout[-2000:] + r.stderr[-4000:]
