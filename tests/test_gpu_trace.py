"""Per-step timing (TPMLP_TRACE=1, read once per process, so each case runs in
a child process): every step of a forward and a backward is recorded in the
order it was enqueued, with a positive device time, the steps of a call add up
to no more than the call's own time, a forward captured into a CUDA graph
records nothing, and without the variable nothing is recorded at all."""

import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = r'''
import torch
import tensor_transformer_mlp_column_gb300 as tp
from tpmlp_inputs import Workload, make_inputs
torch.cuda.set_device(0)
assert tp.tpmlp_trace_enabled()
# Large enough for CTA pairs and the dual backward kernel: T=2048, D=1024, F=4096, N=4.
w = Workload("trace", 2048, 1024, 4096, 4, "bf16", 1.0, 0.02, 0.02, 1.0, True)
d = {k: v.cuda() for k, v in make_inputs(w, seed=91).items()}
sh = tp.tpmlp_shard(d["A"], d["B"], w.N)
torch.cuda.synchronize()
tp.tpmlp_trace_read()  # forget set-up
# (both forwards of this shape run both products in one persistent launch)
expect = {
    ("forward", "faithful"): ["forward_persistent", "allreduce"],
    ("forward", "fused"): ["forward_persistent"],
    ("backward", "faithful"): ["bwd_dual_P_dH", "bwd_dB", "bwd_dA", "bwd_dX_partials", "bwd_dx_allreduce"],
    ("backward", "fused"): ["bwd_dual_P_dH", "bwd_dB", "bwd_dA", "bwd_dX_fused_sum"],
}
for (call, mode), names in expect.items():
    for rep in range(2):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        if call == "forward":
            tp.tpmlp_forward(d["X"], sh, mode)
        else:
            tp.tpmlp_backward(d["X"], d["dY"], sh, mode)
        e1.record()
        steps = tp.tpmlp_trace_read()
        total = e0.elapsed_time(e1)
        assert [s for s, _ in steps] == names, (call, mode, steps)
        assert all(ms > 0 for _, ms in steps), steps
        assert sum(ms for _, ms in steps) <= total * 1.02 + 0.01, (steps, total)
# A shard-ordered sum too short for the one-launch form (T=1024): two launches.
w2 = Workload("trace2", 1024, 1024, 4096, 4, "bf16", 1.0, 0.02, 0.02, 1.0, True)
d2 = {k: v.cuda() for k, v in make_inputs(w2, seed=92).items()}
sh2 = tp.tpmlp_shard(d2["A"], d2["B"], w2.N)
torch.cuda.synchronize()
tp.tpmlp_trace_read()
tp.tpmlp_forward(d2["X"], sh2, "fused")
steps = tp.tpmlp_trace_read()
assert [s for s, _ in steps] == ["gemm1_gelu", "gemm2_fused_sum"], steps
assert all(ms > 0 for _, ms in steps), steps
# Graph capture records nothing; replay matches the eager result.
Y = torch.empty(w.T, w.D, device="cuda")
ws = torch.empty(tp.tpmlp_workspace_bytes(w.T, sh, "fused"), dtype=torch.uint8, device="cuda")
s = torch.cuda.Stream()
with torch.cuda.stream(s):
    tp.tpmlp_forward(d["X"], sh, "fused", Y=Y, workspace=ws)
s.synchronize()
tp.tpmlp_trace_read()
g = torch.cuda.CUDAGraph()
with torch.cuda.graph(g, stream=s):
    tp.tpmlp_forward(d["X"], sh, "fused", Y=Y, workspace=ws)
g.replay()
torch.cuda.synchronize()
assert tp.tpmlp_trace_read() == []
assert torch.equal(Y, tp.tpmlp_forward(d["X"], sh, "fused"))
tp.tpmlp_trace_read()
tp.tpmlp_check_status()
print("ok")
'''

OFF = r'''
import torch
import tensor_transformer_mlp_column_gb300 as tp
from tpmlp_inputs import Workload, make_inputs
torch.cuda.set_device(0)
assert not tp.tpmlp_trace_enabled()
w = Workload("trace_off", 512, 256, 1024, 2, "bf16", 1.0, 0.02, 0.02, 1.0, True)
d = {k: v.cuda() for k, v in make_inputs(w, seed=92).items()}
sh = tp.tpmlp_shard(d["A"], d["B"], w.N)
tp.tpmlp_forward(d["X"], sh, "faithful")
tp.tpmlp_backward(d["X"], d["dY"], sh, "fused")
assert tp.tpmlp_trace_read() == []
print("ok")
'''


def _run(code, env):
    import torch

    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__

    __graft_entry__.build()
    r = subprocess.run([sys.executable, "-c", code], env=env, cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0 and r.stdout.strip().endswith("ok"), r.stdout[-2000:] + r.stderr[-4000:]


def test_trace_records_every_step():
    _run(CHILD, dict(os.environ, TPMLP_TRACE="1"))


def test_trace_off_records_nothing():
    env = dict(os.environ)
    env.pop("TPMLP_TRACE", None)
    _run(OFF, env)
