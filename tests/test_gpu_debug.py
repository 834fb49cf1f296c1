"""The debug build (libtpmlp_debug.so, TPMLP_DEBUG=1; device-side index
checks): on correct inputs no check fires and every result equals the normal
build's bit for bit (the checks guard accesses, they change no arithmetic);
its self test shows a failing check recorded as TPMLP_ERR_BOUNDS with the
access skipped, the device still usable afterwards. Each build runs in a
child process of its own."""

import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = r'''
import sys, torch
import tensor_transformer_mlp_column_gb300 as tp
from tpmlp_inputs import Workload, make_inputs, make_block_inputs, AttnWorkload, make_attn_inputs
torch.cuda.set_device(0)
debug = tp.tpmlp_build_flags() & 1
assert bool(debug) == (sys.argv[2] == "debug")
out = {}
for name, T, D, F, N, dt in (("pair", 1000, 1024, 4096, 4, "bf16"), ("small", 70, 128, 384, 3, "bf16"),
                             ("f32", 33, 64, 256, 4, "f32")):
    w = Workload(name, T, D, F, N, dt, 1.0, 0.05, 0.05, 1.0, True)
    d = {k: v.cuda() for k, v in make_inputs(w, seed=97).items()}
    sh = tp.tpmlp_shard(d["A"], d["B"], w.N)
    for mode in ("faithful", "fused"):
        k = f"{name}_{mode}_"
        out[k + "Y"] = tp.tpmlp_forward(d["X"], sh, mode)
        dX, dA, dB = tp.tpmlp_backward(d["X"], d["dY"], sh, mode)
        out[k + "dX"], out[k + "dA"], out[k + "dB"] = dX, torch.stack(list(dA)), torch.stack(list(dB))
        Y, P = tp.tpmlp_forward_save(d["X"], sh, mode)
        out[k + "dX_saved"] = tp.tpmlp_backward_saved(d["X"], d["dY"], P, sh, mode)[0]
        tp.tpmlp_check_status()
    if dt == "bf16" and T % N == 0:
        out[name + "_sp"] = torch.cat(tp.tpmlp_forward_sp([c.clone() for c in torch.chunk(d["X"], N)], sh, "fused"))
    bi = {k: v.cuda() for k, v in make_block_inputs(w, seed=98, with_dout=True).items()}
    shb = tp.tpmlp_shard(bi["A"], bi["B"], w.N)
    out[name + "_block"] = tp.tpmlp_block_forward(bi["x"], shb, "faithful")
    out[name + "_block_dx"] = tp.tpmlp_block_backward(bi["x"], bi["dout"], shb, "fused")[0]
    out[name + "_gelu"] = tp.tpmlp_gelu(d["X"])
    tp.tpmlp_check_status()
aw = AttnWorkload("attn", 2, 256, 512, 8, 2, "bf16", 1.0, 0.03)
ai = {k: v.cuda() for k, v in make_attn_inputs(aw, seed=99).items()}
sha = tp.tpmlp_attn_shard(ai["Wq"], ai["Wk"], ai["Wv"], ai["Wo"], aw.heads, aw.N)
for mode in ("faithful", "fused"):
    out["attn_" + mode] = tp.tpmlp_attn_forward(ai["X"], aw.batch, sha, mode)
tp.tpmlp_check_status()
if debug:
    tp.tpmlp_selftest_bounds(5)
    tp.tpmlp_check_status()  # an index inside the array: nothing recorded
    for bad in (40, -1, 32):
        tp.tpmlp_selftest_bounds(bad)
        try:
            tp.tpmlp_check_status()
            raise AssertionError(f"index {bad}: no check failure recorded")
        except tp.TpmlpError as e:
            assert e.code == tp.TPMLP_ERR_BOUNDS, (bad, e)
    # the device is still usable and the word was cleared by the read
    assert torch.equal(tp.tpmlp_forward(d["X"], sh, "fused"), out["f32_fused_Y"])
    tp.tpmlp_check_status()
torch.cuda.synchronize()
torch.save({k: v.cpu() for k, v in out.items()}, sys.argv[1])
print("ok")
'''


def test_debug_build_matches_normal_build_and_reports_failed_checks(tmp_path):
    import torch

    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    from tensor_transformer_mlp_column_gb300 import build_lib

    __graft_entry__.build()
    build_lib.build(debug=True, quiet=True)
    results = {}
    for kind in ("debug", "normal"):
        path = str(tmp_path / f"{kind}.pt")
        env = dict(os.environ)
        env.pop("TPMLP_DEBUG", None)
        if kind == "debug":
            env["TPMLP_DEBUG"] = "1"
        r = subprocess.run([sys.executable, "-c", CHILD, path, kind], env=env, cwd=ROOT, capture_output=True,
                           text=True, timeout=900)
        assert r.returncode == 0 and r.stdout.strip().endswith("ok"), kind + r.stdout[-2000:] + r.stderr[-4000:]
        results[kind] = torch.load(path)
    assert results["debug"].keys() == results["normal"].keys()
    for k in results["normal"]:
        assert torch.equal(results["debug"][k], results["normal"][k]), f"{k}: debug and normal builds differ"
