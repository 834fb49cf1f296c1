"""Failure detection inside the tensor-core product, without faulting the GPU.

tpmlp_selftest_gemm_withheld_fill runs the GeLU(X A_i) product with one
stage fill never issued, so the MMA issuer of every CTA (or CTA pair) that
reaches it waits on a barrier that never completes. The bounded wait must give
up after the short limit, the kernel must release its resources (drain copies
and MMAs, free tensor memory) and record TPMLP_ERR_TIMEOUT, and the library
must keep working afterwards: the next forward still matches the oracle.
Both kernels are covered: the CTA-pair kernel (a product with many 256 x 256
tiles) and the single-CTA kernel (a small product).
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
