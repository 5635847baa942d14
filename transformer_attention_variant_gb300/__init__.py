"""Python binding of libiha.so, the GB300 (sm_103a) Interleaved Head Attention forward.

Argument marshalling only: every function below has the name and arguments of
the C entry point it calls (include/iha.h) and returns its integer status.
Arrays may be passed as torch tensors (their data_ptr() is used) or as raw
integer addresses; streams as torch.cuda.Stream, raw handles, or None (the
legacy default stream).  Every step of the computation runs in the library's
CUDA kernels; importing this module fails loudly if the library is missing.
"""
from __future__ import annotations

import ctypes
import os

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libiha.so")

IHA_OK = 0
IHA_ERR_INVALID_ARG = 1
IHA_ERR_UNSUPPORTED = 2
IHA_ERR_WORKSPACE = 3
IHA_ERR_CUDA = 4
IHA_ERR_TIMEOUT = 5
IHA_ERR_BUILD = 6

IHA_DTYPE_F32 = 0
IHA_DTYPE_BF16 = 1

IHA_MASK_NONE = 0
IHA_MASK_CAUSAL = 1
IHA_MASK_WINDOW = 2

EXPORTED = ("iha_forward", "iha_forward_ex", "iha_workspace_bytes", "iha_error_string",
            "iha_check_device_status", "iha_forward_host", "iha_host_buffer_bytes",
            "iha_selftest_wait_timeout", "iha_fold_weights", "iha_project", "iha_attention",
            "iha_contract", "iha_forward_noalloc", "iha_projection_route", "iha_project_heads",
            "iha_mix_heads", "iha_stack_workspace_bytes", "iha_forward_stack", "iha_prefill",
            "iha_decode_workspace_bytes", "iha_decode_step", "iha_backward_workspace_bytes", "iha_backward",
            "iha_forward_train", "iha_backward_saved", "iha_project_mix", "iha_slice_weights",
            "iha_sliced_weights_bytes")

IHA_NOALLOC_SCRATCH_BYTES = 64 << 20


class IHAError(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        self.status = status
        super().__init__(f"{what}: {iha_error_string(status)} (status {status})" if what else iha_error_string(status))


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(
            f"{LIB_PATH} is missing: build the CUDA library first "
            "(python -c 'import __graft_entry__ as g; g.build()').")
    lib = ctypes.CDLL(LIB_PATH)
    vp, fp, i, sz = ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
    shape = [i] * 5
    lib.iha_forward.argtypes = [vp] * 4 + [fp] * 4 + shape + [i, i, vp]
    lib.iha_forward.restype = i
    lib.iha_forward_ex.argtypes = [vp] * 4 + [fp] * 4 + shape + [i, i, vp, i, vp, vp, sz]
    lib.iha_forward_ex.restype = i
    lib.iha_workspace_bytes.argtypes = shape + [i]
    lib.iha_workspace_bytes.restype = sz
    lib.iha_error_string.argtypes = [i]
    lib.iha_error_string.restype = ctypes.c_char_p
    lib.iha_check_device_status.argtypes = [vp, ctypes.POINTER(i)]
    lib.iha_check_device_status.restype = i
    lib.iha_forward_host.argtypes = [vp] * 4 + [fp] * 4 + shape + [i, i, vp, i, vp, vp, sz]
    lib.iha_forward_host.restype = i
    lib.iha_host_buffer_bytes.argtypes = shape + [i]
    lib.iha_host_buffer_bytes.restype = sz
    lib.iha_selftest_wait_timeout.argtypes = [vp, i]
    lib.iha_selftest_wait_timeout.restype = i
    lib.iha_fold_weights.argtypes = [vp] * 3 + [fp] * 3 + [i, i, i, i, vp, vp]
    lib.iha_fold_weights.restype = i
    lib.iha_project.argtypes = [vp, vp] + shape + [i, vp, vp]
    lib.iha_project.restype = i
    lib.iha_attention.argtypes = [vp] + shape + [i, i, i, vp, vp]
    lib.iha_attention.restype = i
    lib.iha_contract.argtypes = [vp, fp] + shape + [i, vp, vp]
    lib.iha_contract.restype = i
    lib.iha_projection_route.argtypes = [i, i, i, i]
    lib.iha_projection_route.restype = i
    lib.iha_project_heads.argtypes = [vp] * 4 + [i] * 5 + [vp, vp]
    lib.iha_project_heads.restype = i
    lib.iha_mix_heads.argtypes = [vp] + [fp] * 3 + [i] * 6 + [vp, vp]
    lib.iha_mix_heads.restype = i
    lib.iha_project_mix.argtypes = [vp, vp] + [fp] * 3 + [i] * 6 + [vp, vp]
    lib.iha_project_mix.restype = i
    lib.iha_slice_weights.argtypes = [vp] * 3 + [i] * 3 + [vp, vp]
    lib.iha_slice_weights.restype = i
    lib.iha_sliced_weights_bytes.argtypes = [i] * 3
    lib.iha_sliced_weights_bytes.restype = sz
    lib.iha_forward_noalloc.argtypes = [vp] * 4 + [fp] * 4 + shape + [i, i, vp, i, vp]
    lib.iha_forward_noalloc.restype = i
    ip = ctypes.POINTER(i)
    pp = ctypes.POINTER(vp)
    lib.iha_stack_workspace_bytes.argtypes = [i, ip, i, i, i, i, i]
    lib.iha_stack_workspace_bytes.restype = sz
    lib.iha_forward_stack.argtypes = [vp, i] + [pp] * 7 + [ip] * 3 + [i] * 5 + [vp, vp, vp, sz]
    lib.iha_forward_stack.restype = i
    lib.iha_prefill.argtypes = [vp] * 4 + [fp] * 4 + shape + [i, i, vp, vp, vp, i, i, vp, vp, sz]
    lib.iha_prefill.restype = i
    lib.iha_decode_workspace_bytes.argtypes = [i, i, i, i]
    lib.iha_decode_workspace_bytes.restype = sz
    lib.iha_decode_step.argtypes = [vp] * 4 + [fp] * 4 + [i] * 6 + [vp, vp, i, i, vp, i, vp, vp, sz]
    lib.iha_decode_step.restype = i
    lib.iha_backward_workspace_bytes.argtypes = shape + [i]
    lib.iha_backward_workspace_bytes.restype = sz
    lib.iha_backward.argtypes = [vp] * 4 + [fp] * 4 + shape + [i, i, vp] + [vp] * 4 + [fp] * 4 + [i, vp, vp, sz]
    lib.iha_backward.restype = i
    lib.iha_forward_train.argtypes = [vp] * 4 + [fp] * 4 + shape + [i, i, vp, i, vp, vp, sz]
    lib.iha_forward_train.restype = i
    lib.iha_backward_saved.argtypes = lib.iha_backward.argtypes
    lib.iha_backward_saved.restype = i
    return lib


_lib = _load()


def _p(x):
    """Address of a tensor (data_ptr), an int address, or None."""
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _s(stream):
    if stream is None:
        return None
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def iha_error_string(status: int) -> str:
    return _lib.iha_error_string(int(status)).decode()


def iha_workspace_bytes(B, N, H, d, P, dtype) -> int:
    return int(_lib.iha_workspace_bytes(B, N, H, d, P, dtype))


def iha_host_buffer_bytes(B, N, H, d, P, dtype) -> int:
    return int(_lib.iha_host_buffer_bytes(B, N, H, d, P, dtype))


def iha_forward(X, W_Q, W_K, W_V, alpha_Q, alpha_K, alpha_V, R, B, N, H, d, P, mask_mode, window, out) -> int:
    return _lib.iha_forward(_p(X), _p(W_Q), _p(W_K), _p(W_V), _p(alpha_Q), _p(alpha_K), _p(alpha_V), _p(R),
                            B, N, H, d, P, mask_mode, window, _p(out))


def iha_forward_ex(X, W_Q, W_K, W_V, alpha_Q, alpha_K, alpha_V, R, B, N, H, d, P, mask_mode, window, out,
                   dtype, stream=None, workspace=None, workspace_bytes=0) -> int:
    return _lib.iha_forward_ex(_p(X), _p(W_Q), _p(W_K), _p(W_V), _p(alpha_Q), _p(alpha_K), _p(alpha_V), _p(R),
                               B, N, H, d, P, mask_mode, window, _p(out), dtype, _s(stream), _p(workspace),
                               workspace_bytes)


def iha_forward_host(X, W_Q, W_K, W_V, alpha_Q, alpha_K, alpha_V, R, B, N, H, d, P, mask_mode, window, out,
                     dtype, stream=None, device_buffer=None, device_buffer_bytes=0) -> int:
    return _lib.iha_forward_host(_p(X), _p(W_Q), _p(W_K), _p(W_V), _p(alpha_Q), _p(alpha_K), _p(alpha_V),
                                 _p(R), B, N, H, d, P, mask_mode, window, _p(out), dtype, _s(stream),
                                 _p(device_buffer), device_buffer_bytes)


def iha_check_device_status(stream=None):
    """Returns (status, raw status word)."""
    code = ctypes.c_int(0)
    rc = _lib.iha_check_device_status(_s(stream), ctypes.byref(code))
    return int(rc), int(code.value)


def iha_selftest_wait_timeout(stream=None, limit_ms=20) -> int:
    return _lib.iha_selftest_wait_timeout(_s(stream), limit_ms)


def iha_fold_weights(W_Q, W_K, W_V, alpha_Q, alpha_K, alpha_V, H, d, P, dtype, Wt, stream=None) -> int:
    return _lib.iha_fold_weights(_p(W_Q), _p(W_K), _p(W_V), _p(alpha_Q), _p(alpha_K), _p(alpha_V),
                                 H, d, P, dtype, _p(Wt), _s(stream))


def iha_project(X, Wt, B, N, H, d, P, dtype, QKV, stream=None) -> int:
    return _lib.iha_project(_p(X), _p(Wt), B, N, H, d, P, dtype, _p(QKV), _s(stream))


def iha_projection_route(H, d, P, dtype) -> int:
    return int(_lib.iha_projection_route(H, d, P, dtype))


def iha_project_heads(X, W_Q, W_K, W_V, B, N, H, d, dtype, Y, stream=None) -> int:
    return _lib.iha_project_heads(_p(X), _p(W_Q), _p(W_K), _p(W_V), B, N, H, d, dtype, _p(Y), _s(stream))


def iha_sliced_weights_bytes(H, d, dtype) -> int:
    return int(_lib.iha_sliced_weights_bytes(H, d, dtype))


def iha_slice_weights(W_Q, W_K, W_V, H, d, dtype, Wp, stream=None) -> int:
    return _lib.iha_slice_weights(_p(W_Q), _p(W_K), _p(W_V), H, d, dtype, _p(Wp), _s(stream))


def iha_project_mix(X, Wp, alpha_Q, alpha_K, alpha_V, B, N, H, d, P, dtype, QKV, stream=None) -> int:
    return _lib.iha_project_mix(_p(X), _p(Wp), _p(alpha_Q), _p(alpha_K), _p(alpha_V), B, N, H, d, P, dtype,
                                _p(QKV), _s(stream))


def iha_mix_heads(Y, alpha_Q, alpha_K, alpha_V, B, N, H, d, P, dtype, QKV, stream=None) -> int:
    return _lib.iha_mix_heads(_p(Y), _p(alpha_Q), _p(alpha_K), _p(alpha_V), B, N, H, d, P, dtype, _p(QKV),
                              _s(stream))


def iha_attention(QKV, B, N, H, d, P, mask_mode, window, dtype, Pbar, stream=None) -> int:
    return _lib.iha_attention(_p(QKV), B, N, H, d, P, mask_mode, window, dtype, _p(Pbar), _s(stream))


def iha_contract(Pbar, R, B, N, H, d, P, dtype, out, stream=None) -> int:
    return _lib.iha_contract(_p(Pbar), _p(R), B, N, H, d, P, dtype, _p(out), _s(stream))


def iha_forward_noalloc(X, W_Q, W_K, W_V, alpha_Q, alpha_K, alpha_V, R, B, N, H, d, P, mask_mode, window, out,
                        dtype, stream=None) -> int:
    """The forward pass with its workspace in the library's fixed scratch array (no
    allocation).  For callers that cannot allocate device memory."""
    return _lib.iha_forward_noalloc(_p(X), _p(W_Q), _p(W_K), _p(W_V), _p(alpha_Q), _p(alpha_K), _p(alpha_V),
                                    _p(R), B, N, H, d, P, mask_mode, window, _p(out), dtype, _s(stream))


def _ptr_array(xs):
    arr = (ctypes.c_void_p * len(xs))()
    for k, x in enumerate(xs):
        arr[k] = _p(x)
    return arr


def _int_array(xs):
    arr = (ctypes.c_int * len(xs))()
    for k, x in enumerate(xs):
        arr[k] = int(x)
    return arr


def iha_stack_workspace_bytes(P, B, N, H, d, dtype) -> int:
    """Workspace of iha_forward_stack for the per-layer pseudo-head counts P (a list)."""
    return int(_lib.iha_stack_workspace_bytes(len(P), _int_array(P), B, N, H, d, dtype))


def iha_forward_stack(X, layers, B, N, H, d, dtype, out, stream=None, workspace=None, workspace_bytes=0) -> int:
    """layers: a list of dicts with W_Q, W_K, W_V, alpha_Q, alpha_K, alpha_V, R (device
    tensors or addresses) and P, mask_mode, window (ints), one per layer in order."""
    n = len(layers)
    arrs = [_ptr_array([L[k] for L in layers]) for k in ("W_Q", "W_K", "W_V", "alpha_Q", "alpha_K", "alpha_V", "R")]
    ints = [_int_array([L[k] for L in layers]) for k in ("P", "mask_mode", "window")]
    return _lib.iha_forward_stack(_p(X), n, *arrs, *ints, B, N, H, d, dtype, _p(out), _s(stream), _p(workspace),
                                  workspace_bytes)


def iha_prefill(X, W_Q, W_K, W_V, alpha_Q, alpha_K, alpha_V, R, B, N, H, d, P, mask_mode, window, out,
                K_cache, V_cache, cache_tokens, dtype, stream=None, workspace=None, workspace_bytes=0) -> int:
    return _lib.iha_prefill(_p(X), _p(W_Q), _p(W_K), _p(W_V), _p(alpha_Q), _p(alpha_K), _p(alpha_V), _p(R),
                            B, N, H, d, P, mask_mode, window, _p(out), _p(K_cache), _p(V_cache), cache_tokens,
                            dtype, _s(stream), _p(workspace), workspace_bytes)


def iha_decode_workspace_bytes(B, H, d, P) -> int:
    return int(_lib.iha_decode_workspace_bytes(B, H, d, P))


def iha_decode_step(x, W_Q, W_K, W_V, alpha_Q, alpha_K, alpha_V, R, B, H, d, P, mask_mode, window, K_cache,
                    V_cache, cache_tokens, t, out, dtype, stream=None, workspace=None, workspace_bytes=0) -> int:
    return _lib.iha_decode_step(_p(x), _p(W_Q), _p(W_K), _p(W_V), _p(alpha_Q), _p(alpha_K), _p(alpha_V), _p(R),
                                B, H, d, P, mask_mode, window, _p(K_cache), _p(V_cache), cache_tokens, t, _p(out),
                                dtype, _s(stream), _p(workspace), workspace_bytes)


def iha_backward_workspace_bytes(B, N, H, d, P, dtype) -> int:
    return int(_lib.iha_backward_workspace_bytes(B, N, H, d, P, dtype))


def iha_backward(X, W_Q, W_K, W_V, alpha_Q, alpha_K, alpha_V, R, B, N, H, d, P, mask_mode, window, dO, dX, dW_Q,
                 dW_K, dW_V, dalpha_Q, dalpha_K, dalpha_V, dR, dtype, stream=None, workspace=None,
                 workspace_bytes=0) -> int:
    return _lib.iha_backward(_p(X), _p(W_Q), _p(W_K), _p(W_V), _p(alpha_Q), _p(alpha_K), _p(alpha_V), _p(R), B, N, H,
                             d, P, mask_mode, window, _p(dO), _p(dX), _p(dW_Q), _p(dW_K), _p(dW_V), _p(dalpha_Q),
                             _p(dalpha_K), _p(dalpha_V), _p(dR), dtype, _s(stream), _p(workspace), workspace_bytes)


def iha_forward_train(X, W_Q, W_K, W_V, alpha_Q, alpha_K, alpha_V, R, B, N, H, d, P, mask_mode, window, out, dtype,
                      stream, workspace, workspace_bytes) -> int:
    return _lib.iha_forward_train(_p(X), _p(W_Q), _p(W_K), _p(W_V), _p(alpha_Q), _p(alpha_K), _p(alpha_V), _p(R), B,
                                  N, H, d, P, mask_mode, window, _p(out), dtype, _s(stream), _p(workspace),
                                  workspace_bytes)


def iha_backward_saved(X, W_Q, W_K, W_V, alpha_Q, alpha_K, alpha_V, R, B, N, H, d, P, mask_mode, window, dO, dX, dW_Q,
                       dW_K, dW_V, dalpha_Q, dalpha_K, dalpha_V, dR, dtype, stream, workspace, workspace_bytes) -> int:
    return _lib.iha_backward_saved(_p(X), _p(W_Q), _p(W_K), _p(W_V), _p(alpha_Q), _p(alpha_K), _p(alpha_V), _p(R), B,
                                   N, H, d, P, mask_mode, window, _p(dO), _p(dX), _p(dW_Q), _p(dW_K), _p(dW_V),
                                   _p(dalpha_Q), _p(dalpha_K), _p(dalpha_V), _p(dR), dtype, _s(stream),
                                   _p(workspace), workspace_bytes)


def check(status: int, what: str = "") -> None:
    """Raise IHAError unless status is IHA_OK."""
    if status != IHA_OK:
        raise IHAError(status, what)


def forward(inputs: dict, *, H, d, P, mask_mode, window=0, stream=None, workspace=None):
    """Allocate the output (torch, on the inputs' device) and run iha_forward_ex.

    inputs: CUDA tensors X [B, N, H*d], W_Q/W_K/W_V [H*d, H*d] (both bf16 or both
    float32), alpha_Q/K/V [H, H, P] and R [H, H*P] float32, all contiguous.
    """
    import torch
    X = inputs["X"]
    if X.dtype == torch.bfloat16:
        dtype = IHA_DTYPE_BF16
    elif X.dtype == torch.float32:
        dtype = IHA_DTYPE_F32
    else:
        raise TypeError("X must be bfloat16 or float32")
    B, N, D = X.shape
    for k, t in inputs.items():
        if not t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{k} must be a contiguous CUDA tensor")
        if k.startswith("W_") and t.dtype != X.dtype:
            raise TypeError(f"{k} must have X's dtype")
        if (k.startswith("alpha") or k == "R") and t.dtype != torch.float32:
            raise TypeError(f"{k} must be float32")
    out = torch.empty_like(X)
    nbytes = 0
    if workspace is not None:
        nbytes = workspace.numel() * workspace.element_size()
    rc = iha_forward_ex(X, inputs["W_Q"], inputs["W_K"], inputs["W_V"], inputs["alpha_Q"], inputs["alpha_K"],
                        inputs["alpha_V"], inputs["R"], B, N, H, d, P, mask_mode, window, out, dtype,
                        stream if stream is not None else torch.cuda.current_stream(X.device), workspace, nbytes)
    check(rc, "iha_forward_ex")
    return out
