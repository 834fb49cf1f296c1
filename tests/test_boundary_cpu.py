"""Host-side checks of the C-ABI library that need no GPU.

The library is built (nvcc cross-compiles for sm_103a without a GPU) and
loaded; every symbol that include/tpmlp.h declares must be exported, and the
argument checks that run before any CUDA call must return their documented
status codes. Fake, never-dereferenced device addresses stand in for buffers.
"""

import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "tpmlp.h")


@pytest.fixture(scope="module")
def tp():
    import __graft_entry__

    __graft_entry__.build()
    import tensor_transformer_mlp_column_gb300 as tp

    return tp


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(tpmlp_[a-z_0-9]+)\s*\(", text)))


def test_header_declares_the_calls_of_the_problem():
    names = declared_functions()
    for required in ["tpmlp_gelu", "tpmlp_shard", "tpmlp_forward", "tpmlp_backward"]:
        assert required in names


def test_library_exports_every_declared_symbol(tp):
    l = tp.lib()
    names = declared_functions()
    missing = [n for n in names if not hasattr(l, n)]
    assert missing == []
    # and the binding knows the signature of each one
    assert sorted(tp.SIGNATURES) == names


def test_version(tp):
    assert tp.tpmlp_version() == (1 << 16)


FAKE = 0x7F0000000000  # 16-byte aligned, never dereferenced


def _shard(tp, A=FAKE, B=FAKE, D=64, F=256, n=4, dt=1):
    h = ctypes.c_void_p()
    rc = tp.lib().tpmlp_shard(A, B, D, F, n, dt, None, ctypes.byref(h))
    return rc, h.value


@pytest.mark.parametrize(
    "kw,code",
    [
        (dict(F=256, n=3), "TPMLP_ERR_DIVISIBILITY"),
        (dict(F=10, n=4, dt=0), "TPMLP_ERR_DIVISIBILITY"),
        (dict(n=0), "TPMLP_ERR_ARG"),
        (dict(n=-1), "TPMLP_ERR_ARG"),
        (dict(D=0), "TPMLP_ERR_ARG"),
        (dict(A=0), "TPMLP_ERR_ARG"),
        (dict(B=0), "TPMLP_ERR_ARG"),
        (dict(dt=7), "TPMLP_ERR_ARG"),
        (dict(A=FAKE + 2), "TPMLP_ERR_ALIGN"),
        (dict(D=60), "TPMLP_ERR_SHAPE"),
        (dict(F=4 * 12, n=4), "TPMLP_ERR_SHAPE"),
        (dict(F=32 * 8, n=32), "TPMLP_ERR_UNSUPPORTED"),
    ],
)
def test_shard_argument_errors(tp, kw, code):
    rc, h = _shard(tp, **kw)
    assert tp.STATUS_NAMES[rc] == code, tp.tpmlp_last_error()
    assert h is None
    assert tp.tpmlp_last_error() != ""


def test_null_out_pointer(tp):
    assert tp.lib().tpmlp_shard(FAKE, FAKE, 64, 256, 4, 1, None, None) == tp.TPMLP_ERR_ARG


def test_calls_reject_null_handles(tp):
    l = tp.lib()
    assert l.tpmlp_forward(FAKE, 4, None, FAKE, 0, FAKE, 1 << 20, None) == tp.TPMLP_ERR_ARG
    assert l.tpmlp_hidden(FAKE, 4, None, FAKE, None) == tp.TPMLP_ERR_ARG
    assert l.tpmlp_partials(FAKE, 4, None, FAKE, None) == tp.TPMLP_ERR_ARG
    assert l.tpmlp_fused_sum(FAKE, 4, None, FAKE, None) == tp.TPMLP_ERR_ARG
    assert l.tpmlp_backward(FAKE, FAKE, 4, None, FAKE, None, None, 0, FAKE, 1 << 20, None) == tp.TPMLP_ERR_ARG
    assert l.tpmlp_shard_info(None, None, None, None, None) == tp.TPMLP_ERR_ARG
    assert l.tpmlp_shard_get(None, 0, None, None) == tp.TPMLP_ERR_ARG
    assert l.tpmlp_workspace_bytes(16, None, 0, 0) == 0
    l.tpmlp_shards_free(None)  # no-op


def test_token_count_outside_its_range(tp):
    # T >= 1 (and at most 2^30) by the header's contract: an empty or negative
    # token count is an argument error, reported before the handle is read.
    l = tp.lib()
    for T in (0, -1, (1 << 30) + 1):
        assert l.tpmlp_forward(FAKE, T, FAKE, FAKE, 0, FAKE, 1 << 20, None) == tp.TPMLP_ERR_ARG
        assert "T = " in tp.tpmlp_last_error()
        assert l.tpmlp_hidden(FAKE, T, FAKE, FAKE, None) == tp.TPMLP_ERR_ARG
        assert l.tpmlp_backward(FAKE, FAKE, T, FAKE, FAKE, None, None, 0, FAKE, 1 << 20, None) == tp.TPMLP_ERR_ARG


def test_gelu_and_allreduce_argument_errors(tp):
    l = tp.lib()
    assert l.tpmlp_gelu(FAKE, FAKE, -1, 0, None) == tp.TPMLP_ERR_ARG
    assert l.tpmlp_gelu(FAKE, FAKE, 0, 0, None) == tp.TPMLP_OK  # empty input enqueues nothing
    assert l.tpmlp_gelu(None, FAKE, 8, 0, None) == tp.TPMLP_ERR_ARG
    assert l.tpmlp_gelu(FAKE + 4, FAKE, 8, 0, None) == tp.TPMLP_ERR_ALIGN
    assert l.tpmlp_gelu(FAKE, FAKE, 8, 5, None) == tp.TPMLP_ERR_ARG
    assert l.tpmlp_allreduce(FAKE, 0, 8, FAKE, None) == tp.TPMLP_ERR_ARG
    assert l.tpmlp_allreduce(FAKE, 2, 0, FAKE, None) == tp.TPMLP_OK
    assert l.tpmlp_allreduce(FAKE, 2, 8, FAKE + 8, None) == tp.TPMLP_ERR_ALIGN
    assert l.tpmlp_selftest_wait_timeout(0, None) == tp.TPMLP_ERR_ARG
    assert l.tpmlp_selftest_gemm_withheld_fill(FAKE, 16, None, FAKE, 1, 10, None) == tp.TPMLP_ERR_ARG


def test_calls_without_a_gpu_report_cuda_or_device_errors(tp):
    # With valid arguments the first CUDA call fails on a GPU-less host; the
    # library must say so with a status code, never crash.
    import torch

    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    rc = tp.lib().tpmlp_gelu(FAKE, FAKE, 8, 0, None)
    assert rc in (tp.TPMLP_ERR_CUDA, tp.TPMLP_ERR_DEVICE)
    assert tp.tpmlp_last_error()


def test_block_call_argument_errors(tp):
    l = tp.lib()
    # layer norm: shape, eps, pointers, alignment (all checked before any CUDA call)
    assert l.tpmlp_layer_norm(FAKE, 4, 0, 0, 1e-5, FAKE, None) == tp.TPMLP_ERR_ARG
    assert l.tpmlp_layer_norm(FAKE, -1, 8, 0, 1e-5, FAKE, None) == tp.TPMLP_ERR_ARG
    assert l.tpmlp_layer_norm(FAKE, 4, 25537, 0, 1e-5, FAKE, None) == tp.TPMLP_ERR_SHAPE
    assert l.tpmlp_layer_norm(FAKE, 4, 8, 9, 1e-5, FAKE, None) == tp.TPMLP_ERR_ARG
    for eps in (0.0, -1e-5, float("inf"), float("nan")):
        assert l.tpmlp_layer_norm(FAKE, 4, 8, 0, eps, FAKE, None) == tp.TPMLP_ERR_ARG
    assert l.tpmlp_layer_norm(FAKE, 0, 8, 0, 1e-5, FAKE, None) == tp.TPMLP_OK  # no rows: nothing enqueued
    assert l.tpmlp_layer_norm(None, 4, 8, 0, 1e-5, FAKE, None) == tp.TPMLP_ERR_ARG
    assert l.tpmlp_layer_norm(FAKE + 4, 4, 8, 0, 1e-5, FAKE, None) == tp.TPMLP_ERR_ALIGN
    # the block calls need a handle
    assert l.tpmlp_block_workspace_bytes(16, None, 0, 0) == 0
    assert l.tpmlp_block_forward(FAKE, 4, None, 1e-5, FAKE, None, 0, FAKE, 1 << 20, None) == tp.TPMLP_ERR_ARG
    assert l.tpmlp_block_backward(FAKE, FAKE, 4, None, 1e-5, FAKE, None, None, 0, FAKE, 1 << 20,
                                  None) == tp.TPMLP_ERR_ARG


def test_sequence_parallel_argument_errors(tp):
    import ctypes

    l = tp.lib()
    P = ctypes.c_void_p
    good = (P * 2)(FAKE, FAKE)
    assert l.tpmlp_all_gather(good, 0, 32, FAKE, None) == tp.TPMLP_ERR_ARG
    assert l.tpmlp_all_gather(good, 17, 32, FAKE, None) == tp.TPMLP_ERR_ARG
    assert l.tpmlp_all_gather(good, 2, 31, FAKE, None) == tp.TPMLP_ERR_ARG
    assert l.tpmlp_all_gather(good, 2, 0, FAKE, None) == tp.TPMLP_OK  # nothing to copy
    assert l.tpmlp_all_gather(None, 2, 32, FAKE, None) == tp.TPMLP_ERR_ARG
    assert l.tpmlp_all_gather((P * 2)(FAKE, FAKE + 2), 2, 32, FAKE, None) == tp.TPMLP_ERR_ALIGN
    assert l.tpmlp_all_gather(good, 2, 32, FAKE + 8, None) == tp.TPMLP_ERR_ALIGN
    assert l.tpmlp_reduce_scatter(FAKE, 3, 16, (P * 3)(FAKE, FAKE, FAKE), None) == tp.TPMLP_ERR_DIVISIBILITY
    assert l.tpmlp_reduce_scatter(FAKE, 2, 16, (P * 2)(FAKE, None), None) == tp.TPMLP_ERR_ARG
    assert l.tpmlp_reduce_scatter(FAKE, 2, 0, good, None) == tp.TPMLP_OK
    assert l.tpmlp_sp_workspace_bytes(16, None, 0, 0) == 0
    assert l.tpmlp_forward_sp(good, 16, None, good, 0, FAKE, 1 << 20, None) == tp.TPMLP_ERR_ARG
    assert l.tpmlp_backward_sp(good, good, 16, None, good, None, None, 0, FAKE, 1 << 20, None) == tp.TPMLP_ERR_ARG


def test_attention_argument_errors_without_gpu(tp):
    import ctypes

    l = tp.lib()
    h = ctypes.c_void_p()
    assert l.tpmlp_attn_shard(FAKE, FAKE, FAKE, FAKE, 128, 2, 2, 1, None, None) == tp.TPMLP_ERR_ARG
    assert l.tpmlp_attn_shard(None, FAKE, FAKE, FAKE, 128, 2, 2, 1, None, ctypes.byref(h)) == tp.TPMLP_ERR_ARG
    assert l.tpmlp_attn_shard(FAKE, FAKE, FAKE, FAKE, 128, 3, 1, 1, None, ctypes.byref(h)) == tp.TPMLP_ERR_DIVISIBILITY
    assert l.tpmlp_attn_shard(FAKE, FAKE, FAKE, FAKE, 128, 2, 4, 1, None, ctypes.byref(h)) == tp.TPMLP_ERR_DIVISIBILITY
    assert l.tpmlp_attn_shard(FAKE, FAKE, FAKE, FAKE, 128, 4, 2, 1, None, ctypes.byref(h)) == tp.TPMLP_ERR_UNSUPPORTED
    assert l.tpmlp_attn_shard(FAKE, FAKE, FAKE, FAKE, 1024, 32, 32, 1, None,
                              ctypes.byref(h)) == tp.TPMLP_ERR_UNSUPPORTED
    assert l.tpmlp_attn_shard(FAKE + 2, FAKE, FAKE, FAKE, 128, 2, 2, 1, None, ctypes.byref(h)) == tp.TPMLP_ERR_ALIGN
    assert l.tpmlp_attn_workspace_bytes(2, 8, None, 0) == 0
    assert l.tpmlp_attn_heads(FAKE, 2, 8, None, FAKE, FAKE, 1 << 20, None) == tp.TPMLP_ERR_ARG
    assert l.tpmlp_attn_forward(FAKE, 2, 8, None, FAKE, 0, FAKE, 1 << 20, None) == tp.TPMLP_ERR_ARG
    assert l.tpmlp_attn_shard_get(None, 0, None, None) == tp.TPMLP_ERR_ARG
    l.tpmlp_attn_shards_free(None)


def test_trace_read_without_tracing(tp):
    """With TPMLP_TRACE unset nothing is recorded: the read returns an empty
    string and no records; a NULL buffer with a non-zero size is an argument
    error."""
    if os.environ.get("TPMLP_TRACE"):
        pytest.skip("TPMLP_TRACE is set in this process")
    assert tp.tpmlp_trace_enabled() is False
    assert tp.tpmlp_trace_read() == []
    buf = ctypes.create_string_buffer(b"x" * 15)
    count = ctypes.c_int(-1)
    assert tp.lib().tpmlp_trace_read(buf, 16, ctypes.byref(count)) == tp.TPMLP_OK
    assert buf.value == b"" and count.value == 0
    assert tp.lib().tpmlp_trace_read(None, 16, None) == tp.TPMLP_ERR_ARG
    assert tp.lib().tpmlp_trace_read(None, 0, None) == tp.TPMLP_OK


def test_normal_build_has_no_device_checks(tp):
    """The normal build reports no debug flag and refuses the debug self test
    before touching the device."""
    if tp.DEBUG:
        pytest.skip("TPMLP_DEBUG is set in this process")
    assert tp.tpmlp_build_flags() == 0
    assert tp.lib().tpmlp_selftest_bounds(40, None) == tp.TPMLP_ERR_UNSUPPORTED


def test_debug_build_loads_under_its_switch():
    """TPMLP_DEBUG=1 makes the binding load libtpmlp_debug.so, which exports
    every declared symbol and reports the debug flag."""
    import subprocess
    import sys

    from tensor_transformer_mlp_column_gb300 import build_lib

    build_lib.build(debug=True, quiet=True)
    code = (
        "import re, tensor_transformer_mlp_column_gb300 as tp\n"
        "assert tp.LIB_PATH.endswith('libtpmlp_debug.so'), tp.LIB_PATH\n"
        "assert tp.tpmlp_build_flags() == 1\n"
        "l = tp.lib()\n"
        "assert all(hasattr(l, n) for n in tp.SIGNATURES)\n"
        "print('ok')\n"
    )
    env = dict(os.environ, TPMLP_DEBUG="1")
    r = subprocess.run([sys.executable, "-c", code], env=env, cwd=ROOT, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0 and r.stdout.strip().endswith("ok"), r.stdout + r.stderr
