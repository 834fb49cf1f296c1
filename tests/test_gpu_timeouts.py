"""Failure detection inside the tensor-core product, without faulting the GPU.

tpmlp_selftest_gemm_withheld_fill runs the GeLU(X A_i) product with one
stage fill never issued, so the MMA issuer of every CTA (or CTA pair) that
reaches it waits on a barrier that never completes. The bounded wait must give
up after the short limit, the kernel must release its resources (drain copies
and MMAs, free tensor memory) and record TPMLP_ERR_TIMEOUT, and the library
must keep working afterwards: the next forward still matches the oracle.
Both kernels are covered: the CTA-pair kernel (a product with many 256 x 256
tiles) and the single-CTA kernel (a small product). The same holds for the
backward's dual-accumulator kernel (a withheld fill) and for the one-launch
forward's band waits (a band of H that is never complete): each gives up,
records TPMLP_ERR_TIMEOUT and leaves the library working.
"""

import numpy as np
import pytest
import torch

import oracle
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


# Each CTA of both cases issues at least three stage fills (K = D in blocks of
# 64, two blocks per stage), so the withheld third fill is reached.
@pytest.mark.parametrize("case", [("pair_kernel", 4096, 1024, 4096, 4), ("single_cta_kernel", 256, 512, 1024, 4)],
                         ids=lambda c: c[0])
def test_withheld_fill_times_out_and_library_recovers(tp, case):
    name, T, D, F, n = case
    w = Workload(name, T, D, F, n, "bf16", 1.0, 1.0 / np.sqrt(D), 1.0 / np.sqrt(F))
    inp = make_inputs(w, seed=41)
    d = {k: v.cuda() for k, v in inp.items()}
    sh = tp.tpmlp_shard(d["A"], d["B"], n)
    H = torch.zeros((n, T, w.Fs), dtype=torch.bfloat16, device="cuda")
    tp.tpmlp_check_status()  # clean start

    tp.tpmlp_selftest_gemm_withheld_fill(d["X"], sh, H, fill=3, limit_ms=100)
    with pytest.raises(tp.TpmlpError) as e:
        tp.tpmlp_check_status()
    assert e.value.code == tp.TPMLP_ERR_TIMEOUT
    tp.tpmlp_check_status()  # the status word was cleared

    # Tensor memory was released and the context is usable: a full forward is right.
    ref = {k: v.to(torch.float64).numpy() for k, v in inp.items()}
    Y_ref = oracle.tp_mlp(ref["X"], oracle.shard_mlp(ref["A"], ref["B"], n))
    for mode in ("faithful", "fused"):
        Y = tp.tpmlp_forward(d["X"], sh, mode).double().cpu().numpy()
        err = Y - Y_ref
        assert np.linalg.norm(err) / np.linalg.norm(Y_ref) <= 5e-3
        assert np.abs(err).max() / np.abs(Y_ref).max() <= 2e-2
    tp.tpmlp_check_status()


def _check_forward_and_backward(tp, inp, d, sh, n):
    ref = {k: v.to(torch.float64).numpy() for k, v in inp.items()}
    shards = oracle.shard_mlp(ref["A"], ref["B"], n)
    Y_ref = oracle.tp_mlp(ref["X"], shards)
    dX_ref = oracle.tp_mlp_backward(ref["X"], ref["dY"], shards)[0]
    for mode in ("faithful", "fused"):
        for got, want in ((tp.tpmlp_forward(d["X"], sh, mode), Y_ref),
                          (tp.tpmlp_backward(d["X"], d["dY"], sh, mode)[0], dX_ref)):
            err = got.double().cpu().numpy() - want
            assert np.linalg.norm(err) / np.linalg.norm(want) <= 5e-3
            assert np.abs(err).max() / np.abs(want).max() <= 2e-2
    tp.tpmlp_check_status()


# GPT-2-small-shaped (T=4096, D=768, F=3072, N=4): both modes of the forward
# run as one persistent launch, and the backward's first step uses the dual
# kernel (each CTA pair fills at least 12 K blocks = 6 stages per tile).
def test_forward_band_wait_times_out_and_library_recovers(tp):
    w = Workload("band", 4096, 768, 3072, 4, "bf16", 1.0, 0.02, 0.02, 1.0, True)
    inp = make_inputs(w, seed=43)
    d = {k: v.cuda() for k, v in inp.items()}
    sh = tp.tpmlp_shard(d["A"], d["B"], w.N)
    tp.tpmlp_check_status()
    for mode in ("faithful", "fused"):
        Y = torch.zeros((w.T, w.D), dtype=torch.float32, device="cuda")
        tp.tpmlp_selftest_forward_band_timeout(d["X"], sh, Y, mode, limit_ms=100)
        with pytest.raises(tp.TpmlpError) as e:
            tp.tpmlp_check_status()
        assert e.value.code == tp.TPMLP_ERR_TIMEOUT
        tp.tpmlp_check_status()
    _check_forward_and_backward(tp, inp, d, sh, w.N)


def test_dual_backward_withheld_fill_times_out_and_library_recovers(tp):
    w = Workload("dual", 4096, 768, 3072, 4, "bf16", 1.0, 0.02, 0.02, 1.0, True)
    inp = make_inputs(w, seed=44)
    d = {k: v.cuda() for k, v in inp.items()}
    sh = tp.tpmlp_shard(d["A"], d["B"], w.N)
    tp.tpmlp_check_status()
    tp.tpmlp_selftest_backward_withheld_fill(d["X"], d["dY"], sh, fill=3, limit_ms=100)
    with pytest.raises(tp.TpmlpError) as e:
        tp.tpmlp_check_status()
    assert e.value.code == tp.TPMLP_ERR_TIMEOUT
    tp.tpmlp_check_status()
    _check_forward_and_backward(tp, inp, d, sh, w.N)
