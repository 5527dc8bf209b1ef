"""Python binding of libmuon: the Muon optimizer step on whole matrices, one GB300.

Argument marshalling only: every step runs in the CUDA kernels of
``_lib/libmuon.so`` (C ABI declared in ``include/muon.h``).  PyTorch supplies
device memory and the current stream.  There is no fallback: when the library
has not been built, every call raises ``MuonLibraryMissing``.

Method: "Training a 1T-Parameter MoE on EU public infrastructure with PyTorch
and TorchTitan", section "FlexShard: Muon without communication" -- one fp32
state per parameter, a few Newton-Schulz iterations on each whole matrix,
whole-expert ownership so that the step needs no communication.
"""

from __future__ import annotations

import ctypes
import os

_PKG = os.path.dirname(os.path.abspath(__file__))
# MUON_CHECKED=1 loads the checked build (device-side checks of the kernels'
# TMA coordinates, reported as MUON_ERR_DEVICE), for example to run the tests on it
CHECKED = os.environ.get("MUON_CHECKED") == "1"
LIB_PATH = os.path.join(_PKG, "_lib", "libmuon_checked.so" if CHECKED else "libmuon.so")

QUINTIC = (3.4445, -4.7750, 2.0315)

MUON_OK = 0
STATUS_NAMES = {
    0: "MUON_OK",
    -1: "MUON_ERR_INVALID_ARG",
    -2: "MUON_ERR_UNSUPPORTED",
    -3: "MUON_ERR_CUDA",
    -4: "MUON_ERR_NO_MEMORY",
    -5: "MUON_ERR_TIMEOUT",
    -6: "MUON_ERR_DEVICE",
}

# name -> (restype, argtypes) of every symbol declared in include/muon.h
_P = ctypes.c_void_p
_I64 = ctypes.c_int64
_F = ctypes.c_float
_INT = ctypes.c_int
_U64 = ctypes.c_uint64
_SIZE = ctypes.c_size_t


class TraceEntry(ctypes.Structure):
    _fields_ = [("kernel", ctypes.c_char_p), ("launches", ctypes.c_int64), ("total_ms", ctypes.c_double)]


class HostGroup(ctypes.Structure):
    """muon_host_group: one shape group of page-locked host arrays."""
    _fields_ = [("param_host", ctypes.c_void_p), ("grad_host", ctypes.c_void_p), ("momentum_host", ctypes.c_void_p),
                ("batch", ctypes.c_int64), ("rows", ctypes.c_int64), ("cols", ctypes.c_int64),
                ("scale", ctypes.c_float)]


SIGNATURES = {
    "muon_momentum_update": (_INT, [_P, _P, _P, _I64, _F, _INT, _P]),
    "muon_momentum_update_f32": (_INT, [_P, _P, _P, _I64, _F, _INT, _P]),
    "muon_ns_batched": (_INT, [_P, _I64, _I64, _I64, _INT, _P, _F, _P]),
    "muon_ns_workspace_bytes": (_SIZE, [_I64, _I64, _I64]),
    "muon_ns_batched_ws": (_INT, [_P, _I64, _I64, _I64, _INT, _P, _F, _P, _SIZE, _P]),
    "muon_ns_batched_static": (_INT, [_P, _I64, _I64, _I64, _INT, _P, _F, _P]),
    "muon_ns_batched_schedule": (_INT, [_P, _I64, _I64, _I64, _INT, _P, _F, _P]),
    "muon_ns_batched_schedule_f32": (_INT, [_P, _I64, _I64, _I64, _INT, _P, _F, _P]),
    "muon_ns_batched_f32": (_INT, [_P, _I64, _I64, _I64, _INT, _P, _F, _P]),
    "muon_ns_workspace_bytes_f32": (_SIZE, [_I64, _I64, _I64]),
    "muon_apply_update": (_INT, [_P, _P, _I64, _I64, _I64, _F, _F, _F, _P]),
    "muon_apply_update_f32": (_INT, [_P, _P, _I64, _I64, _I64, _F, _F, _F, _P]),
    "muon_default_scale": (_F, [_I64, _I64]),
    "muon_step_workspace_bytes": (_SIZE, [_I64, _I64, _I64]),
    "muon_step_batched": (_INT, [_P, _P, _P, _I64, _I64, _I64, _F, _INT, _INT, _P, _F, _F, _F, _F, _P, _SIZE, _P]),
    "muon_step_batched_schedule": (_INT, [_P, _P, _P, _I64, _I64, _I64, _F, _INT, _INT, _P, _F, _F, _F, _F, _P, _SIZE,
                                          _P]),
    "muon_step_batched_after": (_INT, [_P, _P, _P, _I64, _I64, _I64, _F, _INT, _INT, _P, _F, _F, _F, _F, _P, _SIZE,
                                       _P, _P]),
    "muon_step_host": (_INT, [_P, _P, _P, _I64, _I64, _I64, _F, _INT, _INT, _P, _F, _F, _F, _F, _I64, _P]),
    "muon_step_host_grouped": (_INT, [_P, _INT, _F, _INT, _INT, _P, _F, _F, _F, _I64, _P]),
    "muon_adamw_update": (_INT, [_P, _P, _P, _P, _I64, _F, _F, _F, _F, _F, _I64, _P]),
    "muon_adamw_update_f32": (_INT, [_P, _P, _P, _P, _I64, _F, _F, _F, _F, _F, _I64, _P]),
    "muon_get_device_status": (_INT, [_P]),
    "muon_status_string": (ctypes.c_char_p, [_INT]),
    "muon_set_wait_timeout_ns": (_U64, [_U64]),
    "muon_selftest_wait_timeout": (_INT, [_U64, _P]),
    "muon_launch_count": (_I64, []),
    "muon_inject_alloc_failures": (_INT, [_INT]),
    "muon_trace_begin": (_INT, []),
    "muon_trace_end": (_INT, [ctypes.POINTER(TraceEntry), _INT]),
}


class MuonLibraryMissing(RuntimeError):
    pass


class MuonError(RuntimeError):
    def __init__(self, call, status):
        super().__init__(f"{call} returned {STATUS_NAMES.get(status, status)}")
        self.status = status


_lib = None


def lib():
    """The loaded CUDA library (ctypes handle); raises if it was never built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise MuonLibraryMissing(
                f"{LIB_PATH} is missing: build it with muon_newton_schulz_expert_gb300.build.build()")
        handle = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(handle, name)
            fn.restype = res
            fn.argtypes = args
        _lib = handle
    return _lib


def _check(name, status):
    if status != MUON_OK:
        raise MuonError(name, status)


def _stream_handle(stream):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr())


def _need(t, dtype, name):
    import torch
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def _coeffs(coeffs):
    if len(coeffs) != 3:
        raise ValueError("coeffs must hold (a, b, c)")
    return (ctypes.c_float * 3)(*[float(c) for c in coeffs])


# ---------------------------------------------------------------------------- the C calls
def muon_momentum_update(grad, momentum, update_out, mu=0.95, nesterov=True, stream=None):
    """bf16 grad, fp32 momentum (in place), bf16 update_out; see muon.h."""
    import torch
    _need(grad, torch.bfloat16, "grad")
    _need(momentum, torch.float32, "momentum")
    _need(update_out, torch.bfloat16, "update_out")
    if not (grad.numel() == momentum.numel() == update_out.numel()):
        raise ValueError("grad, momentum and update_out must have the same number of elements")
    _check("muon_momentum_update", lib().muon_momentum_update(
        _ptr(grad), _ptr(momentum), _ptr(update_out), grad.numel(), float(mu), int(bool(nesterov)),
        _stream_handle(stream)))


def muon_momentum_update_f32(grad, momentum, update_out, mu=0.95, nesterov=True, stream=None):
    import torch
    for t, n in ((grad, "grad"), (momentum, "momentum"), (update_out, "update_out")):
        _need(t, torch.float32, n)
    if not (grad.numel() == momentum.numel() == update_out.numel()):
        raise ValueError("grad, momentum and update_out must have the same number of elements")
    _check("muon_momentum_update_f32", lib().muon_momentum_update_f32(
        _ptr(grad), _ptr(momentum), _ptr(update_out), grad.numel(), float(mu), int(bool(nesterov)),
        _stream_handle(stream)))


def _bmn(X):
    if X.dim() == 2:
        return 1, X.shape[0], X.shape[1]
    if X.dim() == 3:
        return X.shape[0], X.shape[1], X.shape[2]
    raise ValueError("X must be (m, n) or (batch, m, n)")


def muon_ns_workspace_bytes(batch, m, n):
    return int(lib().muon_ns_workspace_bytes(batch, m, n))


def muon_ns_batched(X, steps=5, coeffs=QUINTIC, eps=1e-7, stream=None, workspace=None):
    """In-place batched Newton-Schulz on a bf16 (batch, m, n) CUDA tensor.

    With ``workspace`` (a CUDA uint8 tensor of at least
    ``muon_ns_workspace_bytes`` bytes) the ``_ws`` entry point is used.
    """
    import torch
    _need(X, torch.bfloat16, "X")
    b, m, n = _bmn(X)
    if workspace is None:
        st = lib().muon_ns_batched(_ptr(X), b, m, n, int(steps), _coeffs(coeffs), float(eps), _stream_handle(stream))
        _check("muon_ns_batched", st)
    else:
        _need(workspace, torch.uint8, "workspace")
        st = lib().muon_ns_batched_ws(_ptr(X), b, m, n, int(steps), _coeffs(coeffs), float(eps), _ptr(workspace),
                                      workspace.numel(), _stream_handle(stream))
        _check("muon_ns_batched_ws", st)
    return X


NS_STATIC_SCRATCH_BYTES = 96 << 20


def muon_ns_batched_static(X, steps=5, coeffs=QUINTIC, eps=1e-7, stream=None):
    """muon_ns_batched on the library's static device scratch: allocates nothing.

    For callers that cannot allocate device memory.  At most
    NS_STATIC_SCRATCH_BYTES of workspace per call (one 1792 x 6144 expert
    matrix); calls that overlap on the GPU share the scratch and race.
    """
    import torch
    _need(X, torch.bfloat16, "X")
    b, m, n = _bmn(X)
    _check("muon_ns_batched_static", lib().muon_ns_batched_static(
        _ptr(X), b, m, n, int(steps), _coeffs(coeffs), float(eps), _stream_handle(stream)))
    return X


def _schedule(coeff_rows):
    rows = [tuple(float(v) for v in r) for r in coeff_rows]
    if any(len(r) != 3 for r in rows):
        raise ValueError("every schedule row must be (a, b, c)")
    flat = [v for r in rows for v in r]
    return len(rows), (ctypes.c_float * max(1, len(flat)))(*flat)


def muon_ns_batched_schedule(X, coeff_rows, eps=1e-7, stream=None):
    """Batched Newton-Schulz with one (a, b, c) row per step (bf16, in place)."""
    import torch
    _need(X, torch.bfloat16, "X")
    b, m, n = _bmn(X)
    steps, arr = _schedule(coeff_rows)
    _check("muon_ns_batched_schedule", lib().muon_ns_batched_schedule(
        _ptr(X), b, m, n, steps, arr, float(eps), _stream_handle(stream)))
    return X


def muon_ns_batched_schedule_f32(X, coeff_rows, eps=1e-7, stream=None):
    """fp32 verification mode of muon_ns_batched_schedule (in place)."""
    import torch
    _need(X, torch.float32, "X")
    b, m, n = _bmn(X)
    steps, arr = _schedule(coeff_rows)
    _check("muon_ns_batched_schedule_f32", lib().muon_ns_batched_schedule_f32(
        _ptr(X), b, m, n, steps, arr, float(eps), _stream_handle(stream)))
    return X


def muon_ns_batched_f32(X, steps=5, coeffs=QUINTIC, eps=1e-7, stream=None):
    """fp32 verification mode of muon_ns_batched (in place)."""
    import torch
    _need(X, torch.float32, "X")
    b, m, n = _bmn(X)
    _check("muon_ns_batched_f32", lib().muon_ns_batched_f32(
        _ptr(X), b, m, n, int(steps), _coeffs(coeffs), float(eps), _stream_handle(stream)))
    return X


def muon_apply_update(param, update, lr=0.02, weight_decay=0.1, scale=0.0, stream=None):
    """param <- (1 - lr*wd) param - lr*scale*update, bf16, in place; scale <= 0: sqrt(max(1, rows/cols))."""
    import torch
    _need(param, torch.bfloat16, "param")
    _need(update, torch.bfloat16, "update")
    if param.shape != update.shape:
        raise ValueError("param and update must have the same shape")
    b, r, c = _bmn(param)
    _check("muon_apply_update", lib().muon_apply_update(
        _ptr(param), _ptr(update), b, r, c, float(lr), float(weight_decay), float(scale), _stream_handle(stream)))


def muon_apply_update_f32(param, update, lr=0.02, weight_decay=0.1, scale=0.0, stream=None):
    import torch
    _need(param, torch.float32, "param")
    _need(update, torch.float32, "update")
    if param.shape != update.shape:
        raise ValueError("param and update must have the same shape")
    b, r, c = _bmn(param)
    _check("muon_apply_update_f32", lib().muon_apply_update_f32(
        _ptr(param), _ptr(update), b, r, c, float(lr), float(weight_decay), float(scale), _stream_handle(stream)))


def muon_adamw_update(param, grad, exp_avg, exp_avg_sq, step, lr=1e-3, beta1=0.9, beta2=0.95, eps=1e-8,
                      weight_decay=0.1, stream=None):
    """AdamW on bf16 params/grads with fp32 moments (in place); see muon.h."""
    import torch
    _need(param, torch.bfloat16, "param")
    _need(grad, torch.bfloat16, "grad")
    _need(exp_avg, torch.float32, "exp_avg")
    _need(exp_avg_sq, torch.float32, "exp_avg_sq")
    if not (param.numel() == grad.numel() == exp_avg.numel() == exp_avg_sq.numel()):
        raise ValueError("all AdamW tensors must have the same number of elements")
    _check("muon_adamw_update", lib().muon_adamw_update(
        _ptr(param), _ptr(grad), _ptr(exp_avg), _ptr(exp_avg_sq), param.numel(), float(lr), float(beta1),
        float(beta2), float(eps), float(weight_decay), int(step), _stream_handle(stream)))


def muon_adamw_update_f32(param, grad, exp_avg, exp_avg_sq, step, lr=1e-3, beta1=0.9, beta2=0.95, eps=1e-8,
                          weight_decay=0.1, stream=None):
    import torch
    for t, n in ((param, "param"), (grad, "grad"), (exp_avg, "exp_avg"), (exp_avg_sq, "exp_avg_sq")):
        _need(t, torch.float32, n)
    if not (param.numel() == grad.numel() == exp_avg.numel() == exp_avg_sq.numel()):
        raise ValueError("all AdamW tensors must have the same number of elements")
    _check("muon_adamw_update_f32", lib().muon_adamw_update_f32(
        _ptr(param), _ptr(grad), _ptr(exp_avg), _ptr(exp_avg_sq), param.numel(), float(lr), float(beta1),
        float(beta2), float(eps), float(weight_decay), int(step), _stream_handle(stream)))


def muon_step_workspace_bytes(batch, rows, cols):
    return int(lib().muon_step_workspace_bytes(batch, rows, cols))


def muon_step_batched(param, grad, momentum, *, mu=0.95, nesterov=True, steps=5, coeffs=QUINTIC, eps=1e-7, lr=0.02,
                      weight_decay=0.1, scale=0.0, workspace=None, stream=None, param_free=None):
    """The fused Muon step on one group of same-shape device matrices (in place).

    param and grad bf16 (batch, rows, cols), momentum fp32 of the same shape.
    Bit for bit the result of momentum -> Newton-Schulz -> update.  With
    ``workspace`` (CUDA uint8, at least ``muon_step_workspace_bytes``) no
    device memory is allocated; without it the library allocates it
    stream-ordered.  With ``param_free`` (a recorded torch.cuda.Event) only
    the launch that writes param waits for it (muon_step_batched_after).
    """
    import torch
    _need(param, torch.bfloat16, "param")
    _need(grad, torch.bfloat16, "grad")
    _need(momentum, torch.float32, "momentum")
    if not (param.shape == grad.shape == momentum.shape):
        raise ValueError("param, grad and momentum must have the same shape")
    b, r, c = _bmn(param)
    ws, ws_bytes = None, 0
    if workspace is not None:
        _need(workspace, torch.uint8, "workspace")
        ws, ws_bytes = _ptr(workspace), workspace.numel()
    args = (_ptr(param), _ptr(grad), _ptr(momentum), b, r, c, float(mu), int(bool(nesterov)), int(steps),
            _coeffs(coeffs), float(eps), float(lr), float(weight_decay), float(scale), ws, ws_bytes)
    if param_free is None:
        _check("muon_step_batched", lib().muon_step_batched(*args, _stream_handle(stream)))
    else:
        if not param_free.cuda_event:
            raise ValueError("param_free must be a recorded torch.cuda.Event")
        _check("muon_step_batched_after", lib().muon_step_batched_after(*args, ctypes.c_void_p(param_free.cuda_event),
                                                                        _stream_handle(stream)))


def muon_step_batched_schedule(param, grad, momentum, coeff_rows, *, mu=0.95, nesterov=True, eps=1e-7, lr=0.02,
                               weight_decay=0.1, scale=0.0, workspace=None, stream=None):
    """muon_step_batched with one (a, b, c) row per Newton-Schulz step (in place)."""
    import torch
    _need(param, torch.bfloat16, "param")
    _need(grad, torch.bfloat16, "grad")
    _need(momentum, torch.float32, "momentum")
    if not (param.shape == grad.shape == momentum.shape):
        raise ValueError("param, grad and momentum must have the same shape")
    b, r, c = _bmn(param)
    steps, arr = _schedule(coeff_rows)
    ws, ws_bytes = None, 0
    if workspace is not None:
        _need(workspace, torch.uint8, "workspace")
        ws, ws_bytes = _ptr(workspace), workspace.numel()
    _check("muon_step_batched_schedule", lib().muon_step_batched_schedule(
        _ptr(param), _ptr(grad), _ptr(momentum), b, r, c, float(mu), int(bool(nesterov)), steps, arr, float(eps),
        float(lr), float(weight_decay), float(scale), ws, ws_bytes, _stream_handle(stream)))


def _host_arrays(param_host, grad_host, momentum_host):
    import torch
    for t, n, dt in ((param_host, "param_host", torch.bfloat16), (grad_host, "grad_host", torch.bfloat16),
                     (momentum_host, "momentum_host", torch.float32)):
        if not isinstance(t, torch.Tensor) or t.is_cuda or t.dtype != dt or not t.is_contiguous():
            raise TypeError(f"{n} must be a contiguous host {dt} tensor")
        if t.numel() and not t.is_pinned():
            raise ValueError(f"{n} must be in page-locked (pinned) host memory")
    if not (param_host.shape == grad_host.shape == momentum_host.shape):
        raise ValueError("param, grad and momentum must have the same shape")
    return _bmn(param_host)


def muon_step_host(param_host, grad_host, momentum_host, *, mu=0.95, nesterov=True, steps=5, coeffs=QUINTIC,
                   eps=1e-7, lr=0.02, weight_decay=0.1, scale=0.0, chunk=0, stream=None):
    """One Muon step on pinned host tensors (batch, rows, cols), streamed through the GPU."""
    b, r, c = _host_arrays(param_host, grad_host, momentum_host)
    _check("muon_step_host", lib().muon_step_host(
        _ptr(param_host), _ptr(grad_host), _ptr(momentum_host), b, r, c, float(mu), int(bool(nesterov)), int(steps),
        _coeffs(coeffs), float(eps), float(lr), float(weight_decay), float(scale), int(chunk),
        _stream_handle(stream)))


def muon_step_host_grouped(groups, *, mu=0.95, nesterov=True, steps=5, coeffs=QUINTIC, eps=1e-7, lr=0.02,
                           weight_decay=0.1, chunk=0, stream=None):
    """muon_step_host over several shape groups in one pipeline.  groups: a list of
    (param_host, grad_host, momentum_host) or (param_host, grad_host, momentum_host, scale)."""
    arr = (HostGroup * max(1, len(groups)))()
    for i, grp in enumerate(groups):
        p, g, m = grp[:3]
        b, r, c = _host_arrays(p, g, m)
        arr[i] = HostGroup(p.data_ptr(), g.data_ptr(), m.data_ptr(), b, r, c, float(grp[3]) if len(grp) > 3 else 0.0)
    _check("muon_step_host_grouped", lib().muon_step_host_grouped(
        ctypes.cast(arr, ctypes.c_void_p), len(groups), float(mu), int(bool(nesterov)), int(steps), _coeffs(coeffs),
        float(eps), float(lr), float(weight_decay), int(chunk), _stream_handle(stream)))


def muon_default_scale(rows, cols):
    """The library's default shape scale for a stored rows x cols matrix (muon.h)."""
    return float(lib().muon_default_scale(int(rows), int(cols)))


def muon_get_device_status(stream=None):
    return int(lib().muon_get_device_status(_stream_handle(stream)))


def muon_status_string(status):
    return lib().muon_status_string(int(status)).decode()


def muon_set_wait_timeout_ns(timeout_ns):
    return int(lib().muon_set_wait_timeout_ns(int(timeout_ns)))


def muon_selftest_wait_timeout(timeout_ns, stream=None):
    _check("muon_selftest_wait_timeout", lib().muon_selftest_wait_timeout(int(timeout_ns), _stream_handle(stream)))


def muon_launch_count():
    return int(lib().muon_launch_count())


def muon_inject_alloc_failures(count):
    """Make the library's next `count` device allocations fail (host-side fault
    injection); returns how many were still pending."""
    r = int(lib().muon_inject_alloc_failures(int(count)))
    if r < 0:
        _check("muon_inject_alloc_failures", r)
    return r


def muon_trace_begin():
    _check("muon_trace_begin", lib().muon_trace_begin())


def muon_trace_end():
    """{kernel name: (launches, total_ms)} for the traced region."""
    entries = (TraceEntry * 32)()
    k = lib().muon_trace_end(entries, 32)
    if k < 0:
        raise MuonError("muon_trace_end", k)
    return {entries[i].kernel.decode(): (int(entries[i].launches), float(entries[i].total_ms)) for i in range(min(k, 32))}


# ---------------------------------------------------------------------------- one whole step
def muon_step(params, grads, momenta, update_bufs=None, *, mu=0.95, nesterov=True, steps=5, coeffs=QUINTIC,
              eps=1e-7, lr=0.02, weight_decay=0.1, scale=0.0, workspace=None, stream=None):
    """One Muon step over groups of same-shape matrices.

    Each argument is a list of tensors, one per shape group: params and grads
    bf16 (batch, rows, cols), momenta fp32 of the same shape.  Without
    update_bufs each group runs the fused muon_step_batched (on ``workspace``,
    one uint8 tensor large enough for the largest group, if given).  With
    update_bufs (bf16 scratch of each group's shape) each group runs
    momentum -> batched Newton-Schulz -> update as three calls, and the
    buffers keep the orthogonalised update; the parameters and momenta come
    out bit-identical either way.
    """
    if update_bufs is None:
        for p, g, m in zip(params, grads, momenta):
            muon_step_batched(p, g, m, mu=mu, nesterov=nesterov, steps=steps, coeffs=coeffs, eps=eps, lr=lr,
                              weight_decay=weight_decay, scale=scale, workspace=workspace, stream=stream)
        return
    for p, g, m, u in zip(params, grads, momenta, update_bufs):
        muon_momentum_update(g, m, u, mu, nesterov, stream)
        muon_ns_batched(u, steps, coeffs, eps, stream)
        muon_apply_update(p, u, lr, weight_decay, scale, stream)

