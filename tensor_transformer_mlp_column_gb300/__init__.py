"""tensor_transformer_mlp_column_gb300 — Python binding of libtpmlp (include/tpmlp.h).

The tensor-parallel MLP  Y = GeLU(X A) B  with A split by columns and B by
rows into n shards, each shard's partial computed on its own and the partials
summed (scratchllm.com "Tensor-Parallel MLP (Megatron)"), on one GB300.

This module only marshals arguments: torch tensors supply device memory and
the current CUDA stream, and every step runs in the library's CUDA kernels.
There is no CPU fallback; if libtpmlp.so is missing the first call raises.
Function names are those of the C ABI.
"""

from __future__ import annotations

import ctypes
import os
from typing import Optional, Sequence

import torch

# TPMLP_DEBUG=1 loads the debug build (device-side index checks; build it with
# build_lib.build(debug=True)) instead of the normal one.
DEBUG = os.environ.get("TPMLP_DEBUG", "") not in ("", "0")
LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libtpmlp_debug.so" if DEBUG else "libtpmlp.so")

TPMLP_F32, TPMLP_BF16 = 0, 1
TPMLP_FAITHFUL, TPMLP_FUSED = 0, 1
TPMLP_MAX_SHARDS = 16

STATUS_NAMES = {
    0: "TPMLP_OK",
    -1: "TPMLP_ERR_ARG",
    -2: "TPMLP_ERR_DIVISIBILITY",
    -3: "TPMLP_ERR_ALIGN",
    -4: "TPMLP_ERR_SHAPE",
    -5: "TPMLP_ERR_CUDA",
    -6: "TPMLP_ERR_TIMEOUT",
    -7: "TPMLP_ERR_WORKSPACE",
    -8: "TPMLP_ERR_UNSUPPORTED",
    -9: "TPMLP_ERR_DEVICE",
    -10: "TPMLP_ERR_BOUNDS",
}
globals().update({v: k for k, v in STATUS_NAMES.items()})

# Every entry point of include/tpmlp.h with its ctypes signature.
_P, _I, _I64, _SZ = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_size_t
SIGNATURES = {
    "tpmlp_version": (_I, []),
    "tpmlp_last_error": (ctypes.c_char_p, []),
    "tpmlp_check_status": (_I, [_P]),
    "tpmlp_gelu": (_I, [_P, _P, _I64, _I, _P]),
    "tpmlp_shard": (_I, [_P, _P, _I64, _I64, _I, _I, _P, ctypes.POINTER(_P)]),
    "tpmlp_shard_info": (_I, [_P, ctypes.POINTER(_I64), ctypes.POINTER(_I64), ctypes.POINTER(_I), ctypes.POINTER(_I)]),
    "tpmlp_shard_get": (_I, [_P, _I, ctypes.POINTER(_P), ctypes.POINTER(_P)]),
    "tpmlp_shard_get_transposed": (_I, [_P, _I, ctypes.POINTER(_P), ctypes.POINTER(_P)]),
    "tpmlp_shards_free": (None, [_P]),
    "tpmlp_workspace_bytes": (_SZ, [_I64, _P, _I, _I]),
    "tpmlp_forward": (_I, [_P, _I64, _P, _P, _I, _P, _SZ, _P]),
    "tpmlp_hidden": (_I, [_P, _I64, _P, _P, _P]),
    "tpmlp_partials": (_I, [_P, _I64, _P, _P, _P]),
    "tpmlp_allreduce": (_I, [_P, _I, _I64, _P, _P]),
    "tpmlp_fused_sum": (_I, [_P, _I64, _P, _P, _P]),
    "tpmlp_backward": (_I, [_P, _P, _I64, _P, _P, ctypes.POINTER(_P), ctypes.POINTER(_P), _I, _P, _SZ, _P]),
    "tpmlp_selftest_wait_timeout": (_I, [_I, _P]),
    "tpmlp_forward_noalloc": (_I, [_P, _I64, _P, _P, _I, _P]),
    "tpmlp_selftest_gemm_withheld_fill": (_I, [_P, _I64, _P, _P, _I, _I, _P]),
    "tpmlp_forward_save": (_I, [_P, _I64, _P, _P, _P, _I, _P, _SZ, _P]),
    "tpmlp_backward_saved": (_I, [_P, _P, _P, _I64, _P, _P, ctypes.POINTER(_P), ctypes.POINTER(_P), _I, _P, _SZ, _P]),
    "tpmlp_layer_norm": (_I, [_P, _I64, _I64, _I, ctypes.c_float, _P, _P]),
    "tpmlp_block_workspace_bytes": (_SZ, [_I64, _P, _I, _I]),
    "tpmlp_block_forward": (_I, [_P, _I64, _P, ctypes.c_float, _P, _P, _I, _P, _SZ, _P]),
    "tpmlp_block_backward": (_I, [_P, _P, _I64, _P, ctypes.c_float, _P, ctypes.POINTER(_P), ctypes.POINTER(_P), _I, _P,
                                  _SZ, _P]),
    "tpmlp_all_gather": (_I, [ctypes.POINTER(_P), _I, _I64, _P, _P]),
    "tpmlp_attn_shard": (_I, [_P, _P, _P, _P, _I64, _I, _I, _I, _P, ctypes.POINTER(_P)]),
    "tpmlp_attn_shard_get": (_I, [_P, _I, ctypes.POINTER(_P), ctypes.POINTER(_P)]),
    "tpmlp_attn_shards_free": (None, [_P]),
    "tpmlp_attn_workspace_bytes": (_SZ, [_I64, _I64, _P, _I]),
    "tpmlp_attn_heads": (_I, [_P, _I64, _I64, _P, _P, _P, _SZ, _P]),
    "tpmlp_attn_forward": (_I, [_P, _I64, _I64, _P, _P, _I, _P, _SZ, _P]),
    "tpmlp_reduce_scatter": (_I, [_P, _I, _I64, ctypes.POINTER(_P), _P]),
    "tpmlp_sp_workspace_bytes": (_SZ, [_I64, _P, _I, _I]),
    "tpmlp_forward_sp": (_I, [ctypes.POINTER(_P), _I64, _P, ctypes.POINTER(_P), _I, _P, _SZ, _P]),
    "tpmlp_backward_sp": (_I, [ctypes.POINTER(_P), ctypes.POINTER(_P), _I64, _P, ctypes.POINTER(_P),
                               ctypes.POINTER(_P), ctypes.POINTER(_P), _I, _P, _SZ, _P]),
    "tpmlp_trace_read": (_I, [ctypes.c_char_p, _SZ, ctypes.POINTER(_I)]),
    "tpmlp_trace_enabled": (_I, []),
    "tpmlp_build_flags": (_I, []),
    "tpmlp_selftest_forward_band_timeout": (_I, [_P, _I64, _P, _P, _I, _P, _SZ, _I, _P]),
    "tpmlp_selftest_backward_withheld_fill": (_I, [_P, _P, _I64, _P, _I, _I, _P, _SZ, _P]),
    "tpmlp_selftest_bounds": (_I, [_I, _P]),
}

_lib: Optional[ctypes.CDLL] = None


class TpmlpError(RuntimeError):
    def __init__(self, code: int, where: str, msg: str):
        super().__init__(f"{where} -> {STATUS_NAMES.get(code, code)}: {msg}")
        self.code = code


def lib() -> ctypes.CDLL:
    """The loaded C library; raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            how = ("`python -m tensor_transformer_mlp_column_gb300.build_lib --debug`" if DEBUG
                   else "`python -c 'import __graft_entry__ as g; g.build()'`")
            raise RuntimeError(f"{LIB_PATH} is missing: build it with {how}")
        l = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in SIGNATURES.items():
            f = getattr(l, name)
            f.restype = res
            f.argtypes = args
        _lib = l
    return _lib


def _check(code: int, where: str) -> None:
    if code != 0:
        raise TpmlpError(code, where, lib().tpmlp_last_error().decode())


def _stream(stream=None) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return int(stream.cuda_stream) if hasattr(stream, "cuda_stream") else int(stream)


def _dt(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return TPMLP_BF16
    if t.dtype == torch.float32:
        return TPMLP_F32
    raise TypeError(f"unsupported dtype {t.dtype}; use torch.float32 or torch.bfloat16")


def _dev(t: torch.Tensor, name: str) -> int:
    if not t.is_cuda or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous CUDA tensor")
    return t.data_ptr()


def _mode(mode) -> int:
    if mode in (TPMLP_FAITHFUL, "faithful"):
        return TPMLP_FAITHFUL
    if mode in (TPMLP_FUSED, "fused"):
        return TPMLP_FUSED
    raise ValueError(f"unknown mode {mode!r}")


class _DeviceArray:
    """Exposes library-owned device memory to torch without copying."""

    def __init__(self, ptr: int, shape, typestr: str):
        self.__cuda_array_interface__ = {"shape": tuple(shape), "typestr": typestr, "data": (ptr, False),
                                         "version": 3, "strides": None}


def _alias(ptr: int, shape, dtype: torch.dtype) -> torch.Tensor:
    if dtype == torch.bfloat16:
        return torch.as_tensor(_DeviceArray(ptr, shape, "<i2"), device="cuda").view(torch.bfloat16)
    return torch.as_tensor(_DeviceArray(ptr, shape, "<f4"), device="cuda")


# ----------------------------------------------------------------- API

def tpmlp_version() -> int:
    return lib().tpmlp_version()


def tpmlp_last_error() -> str:
    return lib().tpmlp_last_error().decode()


def tpmlp_check_status(stream=None) -> None:
    """Waits for the stream and raises TpmlpError if a kernel timed out on a wait."""
    _check(lib().tpmlp_check_status(_stream(stream)), "tpmlp_check_status")


def tpmlp_gelu(x: torch.Tensor, out: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """GeLU(x) elementwise (GPT-2 tanh form), same dtype as x."""
    y = torch.empty_like(x) if out is None else out
    _check(lib().tpmlp_gelu(_dev(x, "x"), _dev(y, "y"), x.numel(), _dt(x), _stream(stream)), "tpmlp_gelu")
    return y


class Shards:
    """The n shard pairs (A_i, B_i) owned by the library (tpmlp_shards handle)."""

    def __init__(self, handle: int, D: int, F: int, n: int, dtype: torch.dtype):
        self.handle, self.D, self.F, self.n, self.dtype = handle, D, F, n, dtype
        self.Fs = F // n

    def get(self, i: int):
        """(A_i [D, F/n], B_i [F/n, D]) as tensors aliasing the library's copies."""
        a, b = ctypes.c_void_p(), ctypes.c_void_p()
        _check(lib().tpmlp_shard_get(self.handle, i, ctypes.byref(a), ctypes.byref(b)), "tpmlp_shard_get")
        return _alias(a.value, (self.D, self.Fs), self.dtype), _alias(b.value, (self.Fs, self.D), self.dtype)

    def get_transposed(self, i: int):
        """(A_i^T [F/n, D], B_i^T [D, F/n]) for bf16 shards."""
        a, b = ctypes.c_void_p(), ctypes.c_void_p()
        _check(lib().tpmlp_shard_get_transposed(self.handle, i, ctypes.byref(a), ctypes.byref(b)),
               "tpmlp_shard_get_transposed")
        return _alias(a.value, (self.Fs, self.D), self.dtype), _alias(b.value, (self.D, self.Fs), self.dtype)

    def free(self) -> None:
        if self.handle:
            lib().tpmlp_shards_free(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.free()
        except Exception:
            pass


def tpmlp_shard(A: torch.Tensor, B: torch.Tensor, n: int, stream=None) -> Shards:
    """shard_mlp(A, B, n): the library's own copies of every (A_i, B_i)."""
    D, F = A.shape
    h = ctypes.c_void_p()
    _check(lib().tpmlp_shard(_dev(A, "A"), _dev(B, "B"), D, F, n, _dt(A), _stream(stream), ctypes.byref(h)),
           "tpmlp_shard")
    return Shards(h.value, D, F, n, A.dtype)


def tpmlp_workspace_bytes(T: int, shards: Shards, mode="faithful", backward: int = 0) -> int:
    """backward: 0 = forward, 1 = tpmlp_backward, 2 = tpmlp_backward_saved."""
    return int(lib().tpmlp_workspace_bytes(T, shards.handle, _mode(mode), int(backward)))


def _workspace(nbytes: int, workspace: Optional[torch.Tensor]) -> torch.Tensor:
    if workspace is not None:
        if workspace.numel() * workspace.element_size() < nbytes:
            raise ValueError(f"workspace too small: need {nbytes} bytes")
        return workspace
    return torch.empty(max(nbytes, 16), dtype=torch.uint8, device="cuda")


def tpmlp_forward(X: torch.Tensor, shards: Shards, mode="faithful", Y: Optional[torch.Tensor] = None,
                  workspace: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """tp_mlp(X, shards): Y = sum_i GeLU(X A_i) B_i, fp32 [T, D]."""
    T = X.shape[0]
    Y = torch.empty((T, shards.D), dtype=torch.float32, device=X.device) if Y is None else Y
    nb = tpmlp_workspace_bytes(T, shards, mode, False)
    ws = _workspace(nb, workspace)
    _check(lib().tpmlp_forward(_dev(X, "X"), T, shards.handle, _dev(Y, "Y"), _mode(mode), ws.data_ptr(),
                               ws.numel() * ws.element_size(), _stream(stream)), "tpmlp_forward")
    return Y


def tpmlp_hidden(X: torch.Tensor, shards: Shards, H: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """H_i = GeLU(X A_i) for all shards: [n, T, F/n] in the shards' dtype."""
    T = X.shape[0]
    H = torch.empty((shards.n, T, shards.Fs), dtype=shards.dtype, device=X.device) if H is None else H
    _check(lib().tpmlp_hidden(_dev(X, "X"), T, shards.handle, _dev(H, "H"), _stream(stream)), "tpmlp_hidden")
    return H


def tpmlp_partials(H: torch.Tensor, shards: Shards, Yp: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """Y_i = H_i B_i for all shards: [n, T, D] fp32."""
    T = H.shape[1]
    Yp = torch.empty((shards.n, T, shards.D), dtype=torch.float32, device=H.device) if Yp is None else Yp
    _check(lib().tpmlp_partials(_dev(H, "H"), T, shards.handle, _dev(Yp, "Yp"), _stream(stream)), "tpmlp_partials")
    return Yp


def tpmlp_allreduce(Yp: torch.Tensor, Y: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """Simulated all-reduce: Y = ((Yp[0] + Yp[1]) + ...) + Yp[n-1], fp32."""
    n = Yp.shape[0]
    Y = torch.empty(Yp.shape[1:], dtype=torch.float32, device=Yp.device) if Y is None else Y
    _check(lib().tpmlp_allreduce(_dev(Yp, "Yp"), n, Y.numel(), _dev(Y, "Y"), _stream(stream)), "tpmlp_allreduce")
    return Y


def tpmlp_fused_sum(H: torch.Tensor, shards: Shards, Y: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """Y = sum_i H_i B_i accumulated on chip in shard order: [T, D] fp32."""
    T = H.shape[1]
    Y = torch.empty((T, shards.D), dtype=torch.float32, device=H.device) if Y is None else Y
    _check(lib().tpmlp_fused_sum(_dev(H, "H"), T, shards.handle, _dev(Y, "Y"), _stream(stream)), "tpmlp_fused_sum")
    return Y


def tpmlp_backward(X: torch.Tensor, dY: torch.Tensor, shards: Shards, mode="faithful",
                   dX: Optional[torch.Tensor] = None, dA: Optional[Sequence[torch.Tensor]] = None,
                   dB: Optional[Sequence[torch.Tensor]] = None, workspace: Optional[torch.Tensor] = None,
                   stream=None, P: Optional[torch.Tensor] = None):
    """Gradients of sum(Y * dY): (dX [T, D], [dA_i [D, F/n]], [dB_i [F/n, D]]), all fp32.

    With P (from tpmlp_forward_save) this is tpmlp_backward_saved, which skips
    recomputing the pre-activations."""
    T, D, Fs, n = X.shape[0], shards.D, shards.Fs, shards.n
    dev = X.device
    dX = torch.empty((T, D), dtype=torch.float32, device=dev) if dX is None else dX
    dA = [torch.empty((D, Fs), dtype=torch.float32, device=dev) for _ in range(n)] if dA is None else list(dA)
    dB = [torch.empty((Fs, D), dtype=torch.float32, device=dev) for _ in range(n)] if dB is None else list(dB)
    pa = (ctypes.c_void_p * n)(*[_dev(t, "dA_i") for t in dA])
    pb = (ctypes.c_void_p * n)(*[_dev(t, "dB_i") for t in dB])
    nb = tpmlp_workspace_bytes(T, shards, mode, 2 if P is not None else 1)
    ws = _workspace(nb, workspace)
    if P is None:
        _check(lib().tpmlp_backward(_dev(X, "X"), _dev(dY, "dY"), T, shards.handle, _dev(dX, "dX"), pa, pb,
                                    _mode(mode), ws.data_ptr(), ws.numel() * ws.element_size(), _stream(stream)),
               "tpmlp_backward")
    else:
        _check(lib().tpmlp_backward_saved(_dev(X, "X"), _dev(dY, "dY"), _dev(P, "P"), T, shards.handle,
                                          _dev(dX, "dX"), pa, pb, _mode(mode), ws.data_ptr(),
                                          ws.numel() * ws.element_size(), _stream(stream)),
               "tpmlp_backward_saved")
    return dX, dA, dB


def tpmlp_backward_saved(X: torch.Tensor, dY: torch.Tensor, P: torch.Tensor, shards: Shards, mode="faithful", **kw):
    """tpmlp_backward with the pre-activations P saved by tpmlp_forward_save."""
    return tpmlp_backward(X, dY, shards, mode, P=P, **kw)


def tpmlp_forward_save(X: torch.Tensor, shards: Shards, mode="faithful", Y: Optional[torch.Tensor] = None,
                       P: Optional[torch.Tensor] = None, workspace: Optional[torch.Tensor] = None, stream=None):
    """Training-mode forward: (Y [T, D] fp32, P [n, T, F/n] fp32 pre-activations)."""
    T = X.shape[0]
    Y = torch.empty((T, shards.D), dtype=torch.float32, device=X.device) if Y is None else Y
    P = torch.empty((shards.n, T, shards.Fs), dtype=torch.float32, device=X.device) if P is None else P
    nb = tpmlp_workspace_bytes(T, shards, mode, 0)
    ws = _workspace(nb, workspace)
    _check(lib().tpmlp_forward_save(_dev(X, "X"), T, shards.handle, _dev(Y, "Y"), _dev(P, "P"), _mode(mode),
                                    ws.data_ptr(), ws.numel() * ws.element_size(), _stream(stream)),
           "tpmlp_forward_save")
    return Y, P


def tpmlp_forward_noalloc(X: torch.Tensor, shards: Shards, Y: torch.Tensor, mode="faithful", stream=None) -> torch.Tensor:
    """tp_mlp(X, shards) for callers that cannot allocate device memory: the
    library's fixed 64 MiB scratch replaces the workspace, and the caller
    passes the output Y [T, D] fp32 (nothing is allocated here either)."""
    _check(lib().tpmlp_forward_noalloc(_dev(X, "X"), X.shape[0], shards.handle, _dev(Y, "Y"), _mode(mode),
                                       _stream(stream)), "tpmlp_forward_noalloc")
    return Y


def tpmlp_layer_norm(x: torch.Tensor, eps: float = 1e-5, y: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """y = (x - mean) / sqrt(var + eps) per row of x [T, D] (no scale or shift), same dtype as x."""
    y = torch.empty_like(x) if y is None else y
    T, D = x.shape
    _check(lib().tpmlp_layer_norm(_dev(x, "x") if T else 0, T, D, _dt(x), float(eps), _dev(y, "y") if T else 0,
                                  _stream(stream)), "tpmlp_layer_norm")
    return y


def tpmlp_block_workspace_bytes(T: int, shards: Shards, mode="faithful", backward: int = 0) -> int:
    return int(lib().tpmlp_block_workspace_bytes(T, shards.handle, _mode(mode), int(backward)))


def tpmlp_block_forward(x: torch.Tensor, shards: Shards, mode="faithful", eps: float = 1e-5,
                        out: Optional[torch.Tensor] = None, xn: Optional[torch.Tensor] = None,
                        workspace: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """out = x + sum_i GeLU(LN(x) A_i) B_i, fp32 [T, D]. With xn, LN(x) is also written there."""
    T = x.shape[0]
    out = torch.empty((T, shards.D), dtype=torch.float32, device=x.device) if out is None else out
    ws = _workspace(tpmlp_block_workspace_bytes(T, shards, mode, 0), workspace)
    _check(lib().tpmlp_block_forward(_dev(x, "x"), T, shards.handle, float(eps), _dev(out, "out"),
                                     _dev(xn, "xn") if xn is not None else None, _mode(mode), ws.data_ptr(),
                                     ws.numel() * ws.element_size(), _stream(stream)), "tpmlp_block_forward")
    return out


def tpmlp_block_backward(x: torch.Tensor, dout: torch.Tensor, shards: Shards, mode="faithful", eps: float = 1e-5,
                         dx: Optional[torch.Tensor] = None, dA: Optional[Sequence[torch.Tensor]] = None,
                         dB: Optional[Sequence[torch.Tensor]] = None, workspace: Optional[torch.Tensor] = None,
                         stream=None):
    """Gradients of sum(out * dout) for tpmlp_block_forward: (dx [T, D], [dA_i], [dB_i]), all fp32."""
    T, D, Fs, n = x.shape[0], shards.D, shards.Fs, shards.n
    dev = x.device
    dx = torch.empty((T, D), dtype=torch.float32, device=dev) if dx is None else dx
    dA = [torch.empty((D, Fs), dtype=torch.float32, device=dev) for _ in range(n)] if dA is None else list(dA)
    dB = [torch.empty((Fs, D), dtype=torch.float32, device=dev) for _ in range(n)] if dB is None else list(dB)
    pa = (ctypes.c_void_p * n)(*[_dev(t, "dA_i") for t in dA])
    pb = (ctypes.c_void_p * n)(*[_dev(t, "dB_i") for t in dB])
    ws = _workspace(tpmlp_block_workspace_bytes(T, shards, mode, 1), workspace)
    _check(lib().tpmlp_block_backward(_dev(x, "x"), _dev(dout, "dout"), T, shards.handle, float(eps), _dev(dx, "dx"),
                                      pa, pb, _mode(mode), ws.data_ptr(), ws.numel() * ws.element_size(),
                                      _stream(stream)), "tpmlp_block_backward")
    return dx, dA, dB


def _ptrs(ts, name):
    return (ctypes.c_void_p * len(ts))(*[_dev(t, name) for t in ts])


def tpmlp_all_gather(slices: Sequence[torch.Tensor], out: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """The rank slices [T/n, ...] back to back: out [T, ...] (the simulated all-gather)."""
    n = len(slices)
    out = torch.empty((n * slices[0].shape[0],) + tuple(slices[0].shape[1:]), dtype=slices[0].dtype,
                      device=slices[0].device) if out is None else out
    nbytes = slices[0].numel() * slices[0].element_size()
    _check(lib().tpmlp_all_gather(_ptrs(slices, "slice"), n, nbytes, _dev(out, "out"), _stream(stream)),
           "tpmlp_all_gather")
    return out


def tpmlp_reduce_scatter(Yp: torch.Tensor, Y_slices: Optional[Sequence[torch.Tensor]] = None,
                         stream=None) -> list:
    """Rank j's rows of the shard-ordered sum of Yp [n, T, D] fp32: n tensors [T/n, D]."""
    n, T = Yp.shape[0], Yp.shape[1]
    rest = tuple(Yp.shape[2:])
    if Y_slices is None:
        Y_slices = [torch.empty((T // n,) + rest, dtype=torch.float32, device=Yp.device) for _ in range(n)]
    count = Yp[0].numel()
    _check(lib().tpmlp_reduce_scatter(_dev(Yp, "Yp"), n, count, _ptrs(Y_slices, "Y_slice"), _stream(stream)),
           "tpmlp_reduce_scatter")
    return list(Y_slices)


def tpmlp_sp_workspace_bytes(T: int, shards: Shards, mode="faithful", backward: int = 0) -> int:
    return int(lib().tpmlp_sp_workspace_bytes(T, shards.handle, _mode(mode), int(backward)))


def tpmlp_forward_sp(X_slices: Sequence[torch.Tensor], shards: Shards, mode="faithful",
                     Y_slices: Optional[Sequence[torch.Tensor]] = None, workspace: Optional[torch.Tensor] = None,
                     stream=None) -> list:
    """Sequence-parallel forward: rank j's rows of sum_i GeLU(X A_i) B_i, X the all-gather of X_slices."""
    n = shards.n
    Ts = X_slices[0].shape[0]
    dev = X_slices[0].device
    if Y_slices is None:
        Y_slices = [torch.empty((Ts, shards.D), dtype=torch.float32, device=dev) for _ in range(n)]
    T = Ts * len(X_slices)
    ws = _workspace(tpmlp_sp_workspace_bytes(T, shards, mode, 0), workspace)
    _check(lib().tpmlp_forward_sp(_ptrs(X_slices, "X_slice"), T, shards.handle, _ptrs(Y_slices, "Y_slice"),
                                  _mode(mode), ws.data_ptr(), ws.numel() * ws.element_size(), _stream(stream)),
           "tpmlp_forward_sp")
    return list(Y_slices)


def tpmlp_backward_sp(X_slices: Sequence[torch.Tensor], dY_slices: Sequence[torch.Tensor], shards: Shards,
                      mode="faithful", dX_slices: Optional[Sequence[torch.Tensor]] = None,
                      dA: Optional[Sequence[torch.Tensor]] = None, dB: Optional[Sequence[torch.Tensor]] = None,
                      workspace: Optional[torch.Tensor] = None, stream=None):
    """Sequence-parallel backward: ([dX_j [T/n, D]], [dA_i], [dB_i]), all fp32."""
    n, D, Fs = shards.n, shards.D, shards.Fs
    Ts = X_slices[0].shape[0]
    dev = X_slices[0].device
    T = Ts * len(X_slices)
    if dX_slices is None:
        dX_slices = [torch.empty((Ts, D), dtype=torch.float32, device=dev) for _ in range(n)]
    dA = [torch.empty((D, Fs), dtype=torch.float32, device=dev) for _ in range(n)] if dA is None else list(dA)
    dB = [torch.empty((Fs, D), dtype=torch.float32, device=dev) for _ in range(n)] if dB is None else list(dB)
    ws = _workspace(tpmlp_sp_workspace_bytes(T, shards, mode, 1), workspace)
    _check(lib().tpmlp_backward_sp(_ptrs(X_slices, "X_slice"), _ptrs(dY_slices, "dY_slice"), T, shards.handle,
                                   _ptrs(dX_slices, "dX_slice"), _ptrs(dA, "dA_i"), _ptrs(dB, "dB_i"), _mode(mode),
                                   ws.data_ptr(), ws.numel() * ws.element_size(), _stream(stream)),
           "tpmlp_backward_sp")
    return list(dX_slices), dA, dB


class AttnShards:
    """Handle of head-split attention weights (tpmlp_attn_shard)."""

    def __init__(self, handle, D: int, heads: int, n: int, dtype: torch.dtype, device):
        self.handle = handle
        self.D, self.heads, self.n, self.dtype, self.device = D, heads, n, dtype, device
        self.Dn = D // n
        self.dh = D // heads

    def get(self, i: int):
        """Rank i's (Wqkv_i, Wo_i) as tensors aliasing the handle's memory (layouts in tpmlp.h)."""
        a, b = ctypes.c_void_p(), ctypes.c_void_p()
        _check(lib().tpmlp_attn_shard_get(self.handle, i, ctypes.byref(a), ctypes.byref(b)), "tpmlp_attn_shard_get")
        if self.dtype == torch.bfloat16:
            return _alias(a.value, (3 * self.Dn, self.D), self.dtype), _alias(b.value, (self.D, self.Dn), self.dtype)
        return _alias(a.value, (self.D, 3 * self.Dn), self.dtype), _alias(b.value, (self.Dn, self.D), self.dtype)

    def free(self):
        if self.handle:
            lib().tpmlp_attn_shards_free(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.free()
        except Exception:
            pass


def tpmlp_attn_shard(Wq, Wk, Wv, Wo, heads: int, n: int, stream=None) -> AttnShards:
    """Split Wq, Wk, Wv by columns and Wo by rows into n ranks of heads/n heads each."""
    D = Wq.shape[0]
    h = ctypes.c_void_p()
    _check(lib().tpmlp_attn_shard(_dev(Wq, "Wq"), _dev(Wk, "Wk"), _dev(Wv, "Wv"), _dev(Wo, "Wo"), D, heads, n,
                                  _dt(Wq), _stream(stream), ctypes.byref(h)), "tpmlp_attn_shard")
    return AttnShards(h.value, D, heads, n, Wq.dtype, Wq.device)


def tpmlp_attn_workspace_bytes(batch: int, seq: int, shards: AttnShards, mode="faithful") -> int:
    m = -1 if mode is None else _mode(mode)
    return int(lib().tpmlp_attn_workspace_bytes(batch, seq, shards.handle, m))


def tpmlp_attn_heads(X: torch.Tensor, batch: int, shards: AttnShards, O: Optional[torch.Tensor] = None,
                     workspace: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """Every rank's local attention heads: O [n, T, D/n] of X's dtype."""
    T = X.shape[0]
    seq = T // batch
    O = torch.empty((shards.n, T, shards.Dn), dtype=X.dtype, device=X.device) if O is None else O
    ws = _workspace(tpmlp_attn_workspace_bytes(batch, seq, shards, None), workspace)
    _check(lib().tpmlp_attn_heads(_dev(X, "X"), batch, seq, shards.handle, _dev(O, "O"), ws.data_ptr(),
                                  ws.numel() * ws.element_size(), _stream(stream)), "tpmlp_attn_heads")
    return O


def tpmlp_attn_forward(X: torch.Tensor, batch: int, shards: AttnShards, mode="faithful",
                       Y: Optional[torch.Tensor] = None, workspace: Optional[torch.Tensor] = None,
                       stream=None) -> torch.Tensor:
    """Y = sum_i O_i Wo_i, fp32 [T, D]."""
    T = X.shape[0]
    seq = T // batch
    Y = torch.empty((T, shards.D), dtype=torch.float32, device=X.device) if Y is None else Y
    ws = _workspace(tpmlp_attn_workspace_bytes(batch, seq, shards, mode), workspace)
    _check(lib().tpmlp_attn_forward(_dev(X, "X"), batch, seq, shards.handle, _dev(Y, "Y"), _mode(mode),
                                    ws.data_ptr(), ws.numel() * ws.element_size(), _stream(stream)),
           "tpmlp_attn_forward")
    return Y


def tpmlp_selftest_gemm_withheld_fill(X: torch.Tensor, shards: Shards, H: torch.Tensor, fill: int, limit_ms: int,
                                      stream=None) -> None:
    """Runs the GeLU(X A_i) product with stage fill `fill` withheld (test hook)."""
    _check(lib().tpmlp_selftest_gemm_withheld_fill(_dev(X, "X"), X.shape[0], shards.handle, _dev(H, "H"), fill,
                                                   limit_ms, _stream(stream)), "tpmlp_selftest_gemm_withheld_fill")


def tpmlp_selftest_wait_timeout(limit_ms: int, stream=None) -> None:
    _check(lib().tpmlp_selftest_wait_timeout(limit_ms, _stream(stream)), "tpmlp_selftest_wait_timeout")


def tpmlp_trace_enabled() -> bool:
    """True when the library records per-step times (TPMLP_TRACE=1 when it was loaded)."""
    return bool(lib().tpmlp_trace_enabled())


def tpmlp_trace_read(max_bytes: int = 1 << 20):
    """Waits for the steps recorded since the last read and returns them as
    [(step name, device milliseconds)] in the order they were enqueued; [] when
    tracing is off."""
    buf = ctypes.create_string_buffer(max_bytes)
    count = ctypes.c_int(0)
    _check(lib().tpmlp_trace_read(buf, max_bytes, ctypes.byref(count)), "tpmlp_trace_read")
    out = []
    for line in buf.value.decode().splitlines():
        name, ms = line.rsplit(" ", 1)
        out.append((name, float(ms)))
    return out


def tpmlp_build_flags() -> int:
    """Bit 0: the loaded library is the debug build (device-side index checks)."""
    return lib().tpmlp_build_flags()


def tpmlp_selftest_bounds(index: int, stream=None) -> None:
    """Debug build: a device-side check of `index` against a 32-element array
    (test hook; a failed check shows in the next tpmlp_check_status)."""
    _check(lib().tpmlp_selftest_bounds(index, _stream(stream)), "tpmlp_selftest_bounds")


def tpmlp_selftest_forward_band_timeout(X: torch.Tensor, shards: Shards, Y: torch.Tensor, mode, limit_ms: int,
                                        workspace: Optional[torch.Tensor] = None, stream=None) -> None:
    """Runs the one-launch forward with bands of H that never complete (test hook)."""
    ws = _workspace(tpmlp_workspace_bytes(X.shape[0], shards, mode, 0), workspace)
    _check(lib().tpmlp_selftest_forward_band_timeout(_dev(X, "X"), X.shape[0], shards.handle, _dev(Y, "Y"),
                                                     _mode(mode), ws.data_ptr(), ws.numel() * ws.element_size(),
                                                     limit_ms, _stream(stream)), "tpmlp_selftest_forward_band_timeout")


def tpmlp_selftest_backward_withheld_fill(X: torch.Tensor, dY: torch.Tensor, shards: Shards, fill: int,
                                          limit_ms: int, workspace: Optional[torch.Tensor] = None,
                                          stream=None) -> None:
    """Runs the backward's dual-accumulator kernel with stage fill `fill` withheld (test hook)."""
    ws = _workspace(tpmlp_workspace_bytes(X.shape[0], shards, "fused", 1), workspace)
    _check(lib().tpmlp_selftest_backward_withheld_fill(_dev(X, "X"), _dev(dY, "dY"), X.shape[0], shards.handle,
                                                       fill, limit_ms, ws.data_ptr(), ws.numel() * ws.element_size(),
                                                       _stream(stream)), "tpmlp_selftest_backward_withheld_fill")
