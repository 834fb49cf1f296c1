"""tpmlp_forward_noalloc: the forward for callers that cannot allocate device
memory at call time (their runtime owns all GPU memory through its own pool,
or their loop cannot take cudaMalloc's synchronisation). It uses the library's
fixed 64 MiB scratch array instead of a caller workspace.

Checked through the C ABI against tpmlp_forward (which takes a workspace), on
two calls in a row with different inputs, so the second call runs on scratch
that still holds the first call's data. Same tolerances as the other parity
tests. The second call must also leave the device's free memory exactly as it
found it (the first call may still load kernel code). This file is collected
last on purpose.
"""

import ctypes

import numpy as np
import pytest
import torch

from tpmlp_inputs import Workload, make_inputs

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


def _call_noalloc(tp, X, sh, Y, mode):
    stream = torch.cuda.current_stream().cuda_stream
    return tp.lib().tpmlp_forward_noalloc(X.data_ptr(), X.shape[0], sh.handle, Y.data_ptr(), mode, stream)


def _close(got, ref, dtype):
    got = got.double().cpu().numpy()
    ref = ref.double().cpu().numpy()
    err = got - ref
    fro = np.linalg.norm(err) / np.linalg.norm(ref)
    mx = np.abs(err).max() / np.abs(ref).max()
    if dtype == "f32":
        assert mx <= 1e-4, mx
    else:
        assert fro <= 5e-3 and mx <= 2e-2, (fro, mx)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("mode", [0, 1], ids=["faithful", "fused"])
def test_noalloc_forward_matches_forward_twice(tp, dtype, mode):
    w = Workload("noalloc", 1000, 512, 2048, 4, dtype, 1.0, 0.04, 0.02)
    first = {k: v.cuda() for k, v in make_inputs(w, seed=31).items()}
    second_X = make_inputs(w, seed=32)["X"].cuda()
    sh = tp.tpmlp_shard(first["A"], first["B"], w.N)
    for call, X in enumerate((first["X"], second_X)):  # two calls in a row on the shared scratch
        Y = torch.full((w.T, w.D), float("nan"), dtype=torch.float32, device="cuda")
        torch.cuda.synchronize()
        free_before = torch.cuda.mem_get_info()[0]
        assert _call_noalloc(tp, X, sh, Y, mode) == tp.TPMLP_OK, tp.tpmlp_last_error()
        torch.cuda.synchronize()
        if call == 1:  # nothing allocated or freed on the device by the call itself
            assert torch.cuda.mem_get_info()[0] == free_before
        ref = tp.tpmlp_forward(X, sh, "fused" if mode else "faithful")
        torch.cuda.synchronize()
        assert torch.isfinite(Y).all()
        _close(Y, ref, dtype)
        if mode == 0:  # faithful is bitwise reproducible, whichever scratch it uses
            assert torch.equal(Y, ref)
    tp.tpmlp_check_status()


def test_noalloc_rejects_sizes_beyond_its_scratch(tp):
    w = Workload("big", 4096, 1024, 16384, 8, "bf16", 1.0, 0.02, 0.02)  # H alone is 128 MiB
    d = {k: v.cuda() for k, v in make_inputs(w, seed=1).items()}
    sh = tp.tpmlp_shard(d["A"], d["B"], w.N)
    Y = torch.zeros((w.T, w.D), dtype=torch.float32, device="cuda")
    rc = _call_noalloc(tp, d["X"], sh, Y, 1)
    assert rc == tp.TPMLP_ERR_WORKSPACE
    assert "64 MiB" in tp.tpmlp_last_error()
    torch.cuda.synchronize()
    assert not Y.any()  # nothing was enqueued


@pytest.mark.parametrize("mode", [0, 1], ids=["faithful", "fused"])
def test_noalloc_forward_captures_without_allocating(tp, mode):
    """After a first call (which caches the scratch address), a call captured
    into a CUDA graph in global capture mode: a device allocation or free, or
    any other call the capture forbids, would fail the capture. The replay
    must match tpmlp_forward. (The eager call leaves the caching allocator's
    count of allocated bytes where it was; around the capture that count
    also moves with the graph's own bookkeeping, so it is not compared there.)"""
    w = Workload("noalloc_graph", 1000, 512, 2048, 4, "bf16", 1.0, 0.04, 0.02)
    d = {k: v.cuda() for k, v in make_inputs(w, seed=33).items()}
    sh = tp.tpmlp_shard(d["A"], d["B"], w.N)
    Y = torch.empty((w.T, w.D), dtype=torch.float32, device="cuda")
    s = torch.cuda.Stream()
    torch.cuda.synchronize()
    allocated = torch.cuda.memory_allocated()
    with torch.cuda.stream(s):
        assert _call_noalloc(tp, d["X"], sh, Y, mode) == tp.TPMLP_OK, tp.tpmlp_last_error()
    s.synchronize()
    assert torch.cuda.memory_allocated() == allocated
    Y.fill_(float("nan"))
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s, capture_error_mode="global"):
        assert _call_noalloc(tp, d["X"], sh, Y, mode) == tp.TPMLP_OK, tp.tpmlp_last_error()
    g.replay()
    torch.cuda.synchronize()
    ref = tp.tpmlp_forward(d["X"], sh, "fused" if mode else "faithful")
    torch.cuda.synchronize()
    assert torch.isfinite(Y).all()
    _close(Y, ref, "bf16")
    if mode == 0:
        assert torch.equal(Y, ref)
    tp.tpmlp_check_status()
