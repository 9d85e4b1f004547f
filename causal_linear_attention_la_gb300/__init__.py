"""GB300 causal linear attention (phi = elu + 1): Python binding of the C ABI.

The compute lives in ``lib/liblagb300.so`` (CUDA kernels for sm_103a); this
module only marshals arguments. Two layers:

* ``la_forward``, ``la_decode_step``, ``la_decode_steps``, ``la_backward`` (and the workspace-size
  queries) mirror the C entry points of ``include/la.h`` one to one and take
  raw device pointers (ints) and sizes.
* ``forward``, ``decode_step``, ``decode_steps``, ``backward`` take torch CUDA tensors, allocate
  outputs and workspace with torch, and call the C entry points on the current
  torch stream.

There is no fallback: if the library is missing or fails to load, every call
raises ``LibraryNotBuilt`` (build it with ``python -m
causal_linear_attention_la_gb300.build``).
"""

from __future__ import annotations

import ctypes
import os

from .build import LIBPATH

__all__ = [
    "LA_OK", "LA_F32", "LA_BF16", "LA_PATH_AUTO", "LA_PATH_SIMT",
    "LaError", "LibraryNotBuilt", "lib", "exported_symbols",
    "la_forward", "la_decode_step", "la_decode_steps", "la_backward",
    "la_decode_steps_decay", "la_decode_steps_delta", "la_state_copy", "la_forward_decay",
    "la_forward_workspace_size", "la_backward_workspace_size",
    "la_set_path", "la_forward_path", "la_backward_path", "la_decode_path",
    "la_profile_enable", "la_profile_read", "la_launch_count", "SPAN_NAMES",
    "la_device_status", "la_test_timeout_next_forward", "la_forward_noalloc", "LA_NOALLOC_SCRATCH_BYTES",
    "la_forward_host", "la_forward_host_workspace_size", "forward_host",
    "la_backward_saved", "backward_saved", "la_backward_decay", "backward_decay",
    "forward", "decode_step", "decode_steps", "backward",
    "decode_steps_decay", "decode_steps_delta", "state_copy", "forward_decay",
    "la_forward_delta", "forward_delta", "la_forward_plan", "forward_plan",
]

LA_OK, LA_ERR_INVALID_ARG, LA_ERR_UNSUPPORTED, LA_ERR_CUDA, LA_ERR_TIMEOUT = range(5)
LA_F32, LA_BF16 = 0, 1
LA_PATH_AUTO, LA_PATH_SIMT = 0, 1
LA_NOALLOC_SCRATCH_BYTES = 16 << 20   # include/la.h
SPAN_NAMES = ("fwd_state", "fwd_scan", "fwd_output", "decode", "bwd_state",
              "bwd_sweep1", "bwd_scan", "bwd_sweep2")

# every entry point of include/la.h
exported_symbols = (
    "la_status_string", "la_last_error", "la_version",
    "la_forward_workspace_size", "la_forward", "la_decode_step", "la_decode_steps",
    "la_decode_steps_decay", "la_decode_steps_delta", "la_state_copy", "la_forward_decay",
    "la_backward_workspace_size", "la_backward",
    "la_set_path", "la_forward_path", "la_backward_path", "la_decode_path",
    "la_profile_enable", "la_profile_read", "la_launch_count",
    "la_device_status", "la_test_timeout_next_forward", "la_forward_noalloc",
    "la_forward_host_workspace_size", "la_forward_host", "la_backward_saved",
    "la_backward_decay", "la_forward_delta", "la_forward_plan",
)


class LibraryNotBuilt(RuntimeError):
    pass


class LaError(RuntimeError):
    def __init__(self, status, message):
        super().__init__(f"{message} (status {status})")
        self.status = status


_lib = None

_c_int, _c_float, _c_size, _c_void = ctypes.c_int, ctypes.c_float, ctypes.c_size_t, ctypes.c_void_p


def lib():
    """Load (once) and return the ctypes handle of the CUDA library."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIBPATH):
        raise LibraryNotBuilt(f"{LIBPATH} not found; run the build first")
    try:
        h = ctypes.CDLL(LIBPATH)
    except OSError as e:  # pragma: no cover - environment specific
        raise LibraryNotBuilt(f"cannot load {LIBPATH}: {e}") from e
    h.la_status_string.restype = ctypes.c_char_p
    h.la_status_string.argtypes = [_c_int]
    h.la_last_error.restype = ctypes.c_char_p
    h.la_last_error.argtypes = []
    h.la_version.restype = _c_int
    h.la_forward_workspace_size.restype = _c_size
    h.la_forward_workspace_size.argtypes = [_c_int] * 6 + [_c_int]
    h.la_backward_workspace_size.restype = _c_size
    h.la_backward_workspace_size.argtypes = [_c_int] * 6 + [_c_int]
    h.la_forward.restype = _c_int
    h.la_forward.argtypes = ([_c_void] * 4 + [_c_int] * 6 + [_c_float, _c_int]
                             + [_c_void, _c_void, _c_void, _c_size, _c_void])
    h.la_backward_saved.restype = _c_int
    h.la_backward_saved.argtypes = ([_c_void] * 7 + [_c_int] * 6 + [_c_float, _c_int]
                                    + [_c_void, _c_size, _c_void, _c_size, _c_void])
    h.la_backward_decay.restype = _c_int
    h.la_backward_decay.argtypes = ([_c_void] * 7 + [_c_int] * 5 + [_c_void, _c_float, _c_int]
                                    + [_c_void, _c_size, _c_void])
    h.la_forward_host_workspace_size.restype = _c_size
    h.la_forward_host_workspace_size.argtypes = [_c_int] * 8
    h.la_forward_host.restype = _c_int
    h.la_forward_host.argtypes = ([_c_void] * 4 + [_c_int] * 6 + [_c_float, _c_int, _c_int]
                                  + [_c_void, _c_size, _c_void])
    h.la_decode_step.restype = _c_int
    h.la_decode_step.argtypes = [_c_void] * 6 + [_c_int] * 4 + [_c_float, _c_int, _c_void]
    h.la_decode_steps.restype = _c_int
    h.la_decode_steps.argtypes = [_c_void] * 6 + [_c_int] * 5 + [_c_float, _c_int, _c_void]
    h.la_decode_steps_decay.restype = _c_int
    h.la_decode_steps_decay.argtypes = [_c_void] * 6 + [_c_int] * 5 + [_c_void, _c_float, _c_int, _c_void]
    h.la_decode_steps_delta.restype = _c_int
    h.la_decode_steps_delta.argtypes = [_c_void] * 5 + [_c_int] * 6 + [_c_void]
    h.la_forward_delta.restype = _c_int
    h.la_forward_plan.restype = _c_int
    h.la_forward_plan.argtypes = [_c_int] * 8 + [_c_void]
    h.la_forward_delta.argtypes = [_c_void] * 5 + [_c_int] * 6 + [_c_void]
    h.la_forward_decay.restype = _c_int
    h.la_forward_decay.argtypes = [_c_void] * 4 + [_c_int] * 5 + [_c_void, _c_float, _c_int] + \
        [_c_void] * 3 + [ctypes.c_size_t, _c_void]
    h.la_state_copy.restype = _c_int
    h.la_state_copy.argtypes = [_c_void] * 4 + [_c_int] * 4 + [_c_void]
    h.la_backward.restype = _c_int
    h.la_backward.argtypes = ([_c_void] * 7 + [_c_int] * 6 + [_c_float, _c_int]
                              + [_c_void, _c_size, _c_void])
    h.la_set_path.restype = _c_int
    h.la_set_path.argtypes = [_c_int]
    h.la_forward_path.restype = _c_int
    h.la_forward_path.argtypes = [_c_int, _c_int, _c_int, _c_int]
    h.la_backward_path.restype = _c_int
    h.la_backward_path.argtypes = [_c_int, _c_int, _c_int, _c_int]
    h.la_decode_path.restype = _c_int
    h.la_decode_path.argtypes = [_c_int, _c_int, _c_int, _c_int]
    h.la_device_status.restype = _c_int
    h.la_device_status.argtypes = [_c_int]
    h.la_test_timeout_next_forward.restype = None
    h.la_test_timeout_next_forward.argtypes = []
    h.la_forward_noalloc.restype = _c_int
    h.la_forward_noalloc.argtypes = ([_c_void] * 4 + [_c_int] * 6 + [_c_float, _c_int]
                                     + [_c_void, _c_void, _c_void])
    h.la_profile_enable.restype = _c_int
    h.la_profile_enable.argtypes = [_c_int]
    h.la_profile_read.restype = _c_int
    h.la_profile_read.argtypes = [ctypes.POINTER(_c_int), ctypes.POINTER(_c_float), _c_int]
    h.la_launch_count.restype = ctypes.c_longlong
    h.la_launch_count.argtypes = []
    _lib = h
    return h


def _check(status):
    if status != LA_OK:
        h = lib()
        raise LaError(status, f"{h.la_status_string(status).decode()}: "
                              f"{h.la_last_error().decode()}")


# ---------------------------------------------------------------------------
# One-to-one wrappers of the C entry points (raw pointers and sizes)
# ---------------------------------------------------------------------------


def la_forward_workspace_size(B, H, N, dk, dv, causal, dtype):
    return lib().la_forward_workspace_size(B, H, N, dk, dv, int(causal), dtype)


def la_backward_workspace_size(B, H, N, dk, dv, causal, dtype):
    return lib().la_backward_workspace_size(B, H, N, dk, dv, int(causal), dtype)


def la_forward(q, k, v, out, B, H, N, dk, dv, causal, eps, dtype, S_final,
               z_final, workspace, workspace_bytes, stream):
    return lib().la_forward(q, k, v, out, B, H, N, dk, dv, int(causal), eps,
                            dtype, S_final, z_final, workspace,
                            workspace_bytes, stream)


def la_backward_decay(q, k, v, dout, dq, dk_, dv_, B, H, N, dk, dv, alpha, eps, dtype,
                      workspace, workspace_bytes, stream):
    return lib().la_backward_decay(q, k, v, dout, dq, dk_, dv_, B, H, N, dk, dv, alpha, eps, dtype,
                                   workspace, workspace_bytes, stream)


def la_backward_saved(q, k, v, dout, dq, dk_, dv_, B, H, N, dk, dv, causal, eps, dtype,
                      saved, saved_bytes, workspace, workspace_bytes, stream):
    return lib().la_backward_saved(q, k, v, dout, dq, dk_, dv_, B, H, N, dk, dv, int(causal), eps,
                                   dtype, saved, saved_bytes, workspace, workspace_bytes, stream)


def la_forward_host_workspace_size(B, H, N, dk, dv, causal, dtype, slices):
    return lib().la_forward_host_workspace_size(B, H, N, dk, dv, int(causal), dtype, slices)


def la_forward_host(q, k, v, out, B, H, N, dk, dv, causal, eps, dtype, slices,
                    workspace, workspace_bytes, stream):
    return lib().la_forward_host(q, k, v, out, B, H, N, dk, dv, int(causal), eps,
                                 dtype, slices, workspace, workspace_bytes, stream)


def la_forward_noalloc(q, k, v, out, B, H, N, dk, dv, causal, eps, dtype,
                       S_final, z_final, stream):
    """la_forward with its scratch in the library's static device array
    (no allocation; see include/la.h)."""
    return lib().la_forward_noalloc(q, k, v, out, B, H, N, dk, dv, int(causal),
                                    eps, dtype, S_final, z_final, stream)


def la_decode_step(S, z, q, k, v, out, B, H, dk, dv, eps, dtype, stream):
    return lib().la_decode_step(S, z, q, k, v, out, B, H, dk, dv, eps, dtype, stream)


def la_decode_steps(S, z, q, k, v, out, B, H, T, dk, dv, eps, dtype, stream):
    return lib().la_decode_steps(S, z, q, k, v, out, B, H, T, dk, dv, eps, dtype, stream)


def la_decode_steps_decay(S, z, q, k, v, out, B, H, T, dk, dv, alpha, eps, dtype, stream):
    return lib().la_decode_steps_decay(S, z, q, k, v, out, B, H, T, dk, dv, alpha, eps, dtype, stream)


def la_decode_steps_delta(S, q, k, v, out, B, H, T, dk, dv, dtype, stream):
    return lib().la_decode_steps_delta(S, q, k, v, out, B, H, T, dk, dv, dtype, stream)


def la_forward_plan(B, H, N, dk, dv, causal, dtype, final_state, out):
    return lib().la_forward_plan(B, H, N, dk, dv, causal, dtype, final_state, out)


def forward_plan(B, H, N, dk, dv, causal=True, dtype=LA_BF16, final_state=False):
    """The split la_forward uses for these sizes: dict with P, seg_len, F,
    pieces (0: by segments) and piece_len (chunks of 128 tokens)."""
    buf = (ctypes.c_int * 5)()
    _check(la_forward_plan(B, H, N, dk, dv, int(causal), dtype, int(final_state), ctypes.cast(buf, ctypes.c_void_p)))
    return dict(P=buf[0], seg_len=buf[1], F=buf[2], pieces=buf[3], piece_len=buf[4])


def la_forward_delta(S, q, k, v, out, B, H, N, dk, dv, dtype, stream):
    return lib().la_forward_delta(S, q, k, v, out, B, H, N, dk, dv, dtype, stream)


def la_forward_decay(q, k, v, out, B, H, N, dk, dv, alpha, eps, dtype, S_final, z_final,
                     workspace, workspace_bytes, stream):
    return lib().la_forward_decay(q, k, v, out, B, H, N, dk, dv, alpha, eps, dtype, S_final,
                                  z_final, workspace, workspace_bytes, stream)


def la_state_copy(dst_S, dst_z, src_S, src_z, B, H, dk, dv, stream):
    return lib().la_state_copy(dst_S, dst_z, src_S, src_z, B, H, dk, dv, stream)


def la_backward(q, k, v, dout, dq, dk_, dv_, B, H, N, dk, dv, causal, eps,
                dtype, workspace, workspace_bytes, stream):
    return lib().la_backward(q, k, v, dout, dq, dk_, dv_, B, H, N, dk, dv,
                             int(causal), eps, dtype, workspace,
                             workspace_bytes, stream)


def la_set_path(path):
    return lib().la_set_path(path)


def la_forward_path(dk, dv, dtype, causal=True):
    return lib().la_forward_path(dk, dv, dtype, int(causal))


def la_backward_path(dk, dv, dtype, causal=True):
    return lib().la_backward_path(dk, dv, dtype, int(causal))


def la_decode_path(dk, dv, dtype, T):
    return lib().la_decode_path(dk, dv, dtype, int(T))


def la_device_status(clear=False):
    return lib().la_device_status(int(clear))


def la_test_timeout_next_forward():
    lib().la_test_timeout_next_forward()


def la_profile_enable(on):
    return lib().la_profile_enable(int(on))


def la_profile_read():
    """[(span name, milliseconds), ...] for every span recorded since enable."""
    h = lib()
    n = h.la_profile_read(None, None, 0)
    labels = (_c_int * max(n, 1))()
    ms = (_c_float * max(n, 1))()
    n = h.la_profile_read(labels, ms, n)
    return [(SPAN_NAMES[labels[i]], float(ms[i])) for i in range(n)]


def la_launch_count():
    return int(lib().la_launch_count())


# ---------------------------------------------------------------------------
# torch-tensor convenience layer (allocation and pointers only)
# ---------------------------------------------------------------------------


def _dtype_code(t):
    import torch
    if t.dtype == torch.bfloat16:
        return LA_BF16
    if t.dtype == torch.float32:
        return LA_F32
    raise TypeError(f"unsupported dtype {t.dtype}")


def _need(t, name, dtype=None, cuda=True):
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if cuda and not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")


def _stream_ptr(t):
    import torch
    return torch.cuda.current_stream(t.device).cuda_stream


def forward(q, k, v, causal=True, eps=1e-6, return_state=False, out=None,
            workspace=None):
    """out = la_forward(q, k, v); q, k [B,H,N,dk], v [B,H,N,dv] (bf16 or f32).

    Returns out, or (out, S_N, z_N) with fp32 S_N [B,H,dk,dv], z_N [B,H,dk]
    when ``return_state``.
    """
    import torch
    B, H, N, dk = q.shape
    dv = v.shape[-1]
    code = _dtype_code(q)
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _need(t, n, q.dtype)
    if out is None:
        out = torch.empty((B, H, N, dv), dtype=q.dtype, device=q.device)
    S = z = None
    if return_state:
        S = torch.empty((B, H, dk, dv), dtype=torch.float32, device=q.device)
        z = torch.empty((B, H, dk), dtype=torch.float32, device=q.device)
    ws_bytes = la_forward_workspace_size(B, H, N, dk, dv, causal, code)
    if workspace is None or workspace.numel() < ws_bytes:
        workspace = torch.empty(max(ws_bytes, 1), dtype=torch.uint8, device=q.device)
    _check(la_forward(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                      B, H, N, dk, dv, causal, eps, code,
                      S.data_ptr() if S is not None else None,
                      z.data_ptr() if z is not None else None,
                      workspace.data_ptr(), workspace.numel(), _stream_ptr(q)))
    if return_state:
        return out, S, z
    return out


def forward_host(q, k, v, causal=True, eps=1e-6, out=None, slices=2, workspace=None,
                 device=None):
    """la_forward_host: q, k [B,H,N,dk], v [B,H,N,dv] CPU tensors (pinned for
    overlap), out a CPU tensor [B,H,N,dv] (allocated pinned when None). The
    copies and the forward are enqueued on the current stream of ``device``;
    synchronise it before reading ``out``."""
    import torch
    B, H, N, dk = q.shape
    dv = v.shape[-1]
    code = _dtype_code(q)
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _need(t, n, q.dtype, cuda=False)
        if t.is_cuda:
            raise ValueError(f"{n} must be a host tensor")
    if out is None:
        out = torch.empty((B, H, N, dv), dtype=q.dtype).pin_memory()
    _need(out, "out", q.dtype, cuda=False)
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    ws_bytes = la_forward_host_workspace_size(B, H, N, dk, dv, causal, code, slices)
    if workspace is None or workspace.numel() < ws_bytes:
        workspace = torch.empty(max(ws_bytes, 1), dtype=torch.uint8, device=dev)
    _check(la_forward_host(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                           B, H, N, dk, dv, causal, eps, code, slices,
                           workspace.data_ptr(), workspace.numel(),
                           torch.cuda.current_stream(dev).cuda_stream))
    return out


def decode_step(S, z, q, k, v, eps=1e-6, out=None):
    """In-place recurrent step on fp32 S [B,H,dk,dv], z [B,H,dk]; returns out [B,H,dv]."""
    import torch
    B, H, dk, dv = S.shape
    code = _dtype_code(q)
    _need(S, "S", torch.float32)
    _need(z, "z", torch.float32)
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _need(t, n, q.dtype)
    if out is None:
        out = torch.empty((B, H, dv), dtype=q.dtype, device=q.device)
    _check(la_decode_step(S.data_ptr(), z.data_ptr(), q.data_ptr(), k.data_ptr(),
                          v.data_ptr(), out.data_ptr(), B, H, dk, dv, eps, code,
                          _stream_ptr(q)))
    return out


def decode_steps(S, z, q, k, v, eps=1e-6, out=None):
    """T in-place recurrent steps on fp32 S [B,H,dk,dv], z [B,H,dk] with
    q, k [B,H,T,dk], v [B,H,T,dv]; returns out [B,H,T,dv]."""
    import torch
    B, H, dk, dv = S.shape
    T = q.shape[2]
    code = _dtype_code(q)
    _need(S, "S", torch.float32)
    _need(z, "z", torch.float32)
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _need(t, n, q.dtype)
    if out is None:
        out = torch.empty((B, H, T, dv), dtype=q.dtype, device=q.device)
    _check(la_decode_steps(S.data_ptr(), z.data_ptr(), q.data_ptr(), k.data_ptr(),
                           v.data_ptr(), out.data_ptr(), B, H, T, dk, dv, eps, code,
                           _stream_ptr(q)))
    return out


def decode_steps_decay(S, z, q, k, v, alpha, eps=1e-6, out=None):
    """decode_steps with the summary decayed by alpha [H] (fp32 CUDA) before each token."""
    import torch
    B, H, dk, dv = S.shape
    T = q.shape[2]
    code = _dtype_code(q)
    _need(S, "S", torch.float32)
    _need(z, "z", torch.float32)
    _need(alpha, "alpha", torch.float32)
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _need(t, n, q.dtype)
    if out is None:
        out = torch.empty((B, H, T, dv), dtype=q.dtype, device=q.device)
    _check(la_decode_steps_decay(S.data_ptr(), z.data_ptr(), q.data_ptr(), k.data_ptr(),
                                 v.data_ptr(), out.data_ptr(), B, H, T, dk, dv,
                                 alpha.data_ptr(), eps, code, _stream_ptr(q)))
    return out


def forward_decay(q, k, v, alpha, eps=1e-6, return_state=False, out=None, workspace=None):
    """Decay-gated causal forward (bf16, d = 64) with per-head factors alpha [H]."""
    import torch
    B, H, N, dk = q.shape
    dv = v.shape[-1]
    code = _dtype_code(q)
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _need(t, n, q.dtype)
    _need(alpha, "alpha", torch.float32)
    if out is None:
        out = torch.empty((B, H, N, dv), dtype=q.dtype, device=q.device)
    S = z = None
    if return_state:
        S = torch.empty((B, H, dk, dv), dtype=torch.float32, device=q.device)
        z = torch.empty((B, H, dk), dtype=torch.float32, device=q.device)
    ws_bytes = la_forward_workspace_size(B, H, N, dk, dv, True, code)
    if workspace is None or workspace.numel() < ws_bytes:
        workspace = torch.empty(max(ws_bytes, 1), dtype=torch.uint8, device=q.device)
    _check(la_forward_decay(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                            B, H, N, dk, dv, alpha.data_ptr(), eps, code,
                            S.data_ptr() if S is not None else None,
                            z.data_ptr() if z is not None else None,
                            workspace.data_ptr(), workspace.numel(), _stream_ptr(q)))
    if return_state:
        return out, S, z
    return out


def decode_steps_delta(S, q, k, v, out=None):
    """T delta-rule steps in place on fp32 S [B,H,dk,dv]; returns out [B,H,T,dv]."""
    import torch
    B, H, dk, dv = S.shape
    T = q.shape[2]
    code = _dtype_code(q)
    _need(S, "S", torch.float32)
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _need(t, n, q.dtype)
    if out is None:
        out = torch.empty((B, H, T, dv), dtype=q.dtype, device=q.device)
    _check(la_decode_steps_delta(S.data_ptr(), q.data_ptr(), k.data_ptr(), v.data_ptr(),
                                 out.data_ptr(), B, H, T, dk, dv, code, _stream_ptr(q)))
    return out


def forward_delta(S, q, k, v, out=None):
    """Delta rule over N tokens per (batch, head), chunk by chunk, from and
    into the fp32 state S [B,H,d,d] (in place); returns out [B,H,N,d]."""
    import torch
    B, H, dk, dv = S.shape
    N = q.shape[2]
    code = _dtype_code(q)
    _need(S, "S", torch.float32)
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _need(t, n, q.dtype)
    if out is None:
        out = torch.empty((B, H, N, dv), dtype=q.dtype, device=q.device)
    _check(la_forward_delta(S.data_ptr(), q.data_ptr(), k.data_ptr(), v.data_ptr(),
                            out.data_ptr(), B, H, N, dk, dv, code, _stream_ptr(q)))
    return out


def state_copy(dst_S, src_S, dst_z=None, src_z=None):
    """dst_S <- src_S and dst_z <- src_z (snapshot or restore of a state)."""
    import torch
    B, H, dk, dv = src_S.shape
    for t, n in ((dst_S, "dst_S"), (src_S, "src_S")):
        _need(t, n, torch.float32)
    _check(la_state_copy(dst_S.data_ptr(), dst_z.data_ptr() if dst_z is not None else None,
                         src_S.data_ptr(), src_z.data_ptr() if src_z is not None else None,
                         B, H, dk, dv, _stream_ptr(src_S)))
    return dst_S


def backward(q, k, v, dout, causal=True, eps=1e-6, workspace=None):
    """(dq, dk, dv) of sum(dout * la_forward(q, k, v))."""
    import torch
    B, H, N, dk = q.shape
    dv = v.shape[-1]
    code = _dtype_code(q)
    for t, n in ((q, "q"), (k, "k"), (v, "v"), (dout, "dout")):
        _need(t, n, q.dtype)
    dq = torch.empty_like(q)
    dkk = torch.empty_like(k)
    dvv = torch.empty_like(v)
    ws_bytes = la_backward_workspace_size(B, H, N, dk, dv, causal, code)
    if workspace is None or workspace.numel() < ws_bytes:
        workspace = torch.empty(max(ws_bytes, 1), dtype=torch.uint8, device=q.device)
    _check(la_backward(q.data_ptr(), k.data_ptr(), v.data_ptr(), dout.data_ptr(),
                       dq.data_ptr(), dkk.data_ptr(), dvv.data_ptr(), B, H, N,
                       dk, dv, causal, eps, code, workspace.data_ptr(),
                       workspace.numel(), _stream_ptr(q)))
    return dq, dkk, dvv


def backward_decay(q, k, v, dout, alpha, eps=1e-6, workspace=None):
    """Gradients (dq, dk, dv) of the decay-gated causal attention
    (la_backward_decay); alpha: fp32 CUDA tensor [H], one factor per head."""
    import torch
    B, H, N, dk = q.shape
    dv = v.shape[-1]
    code = _dtype_code(q)
    for t, n in ((q, "q"), (k, "k"), (v, "v"), (dout, "dout")):
        _need(t, n, q.dtype)
    if alpha.dtype != torch.float32 or not alpha.is_cuda or alpha.numel() != H:
        raise ValueError("alpha must be an fp32 CUDA tensor of H factors")
    dq = torch.empty_like(q)
    dkk = torch.empty_like(k)
    dvv = torch.empty_like(v)
    ws_bytes = la_backward_workspace_size(B, H, N, dk, dv, True, code)
    if workspace is None or workspace.numel() < ws_bytes:
        workspace = torch.empty(max(ws_bytes, 1), dtype=torch.uint8, device=q.device)
    _check(la_backward_decay(q.data_ptr(), k.data_ptr(), v.data_ptr(), dout.data_ptr(),
                             dq.data_ptr(), dkk.data_ptr(), dvv.data_ptr(), B, H, N,
                             dk, dv, alpha.contiguous().data_ptr(), eps, code, workspace.data_ptr(),
                             workspace.numel(), _stream_ptr(q)))
    return dq, dkk, dvv


def backward_saved(q, k, v, dout, saved, causal=True, eps=1e-6, workspace=None):
    """backward() reusing ``saved``, the workspace tensor of the matching
    forward(q, k, v, causal=causal, workspace=saved) call (left unchanged)."""
    import torch
    B, H, N, dk = q.shape
    dv = v.shape[-1]
    code = _dtype_code(q)
    for t, n in ((q, "q"), (k, "k"), (v, "v"), (dout, "dout")):
        _need(t, n, q.dtype)
    _need(saved, "saved")
    dq = torch.empty_like(q)
    dkk = torch.empty_like(k)
    dvv = torch.empty_like(v)
    ws_bytes = la_backward_workspace_size(B, H, N, dk, dv, causal, code)
    if workspace is None or workspace.numel() < ws_bytes:
        workspace = torch.empty(max(ws_bytes, 1), dtype=torch.uint8, device=q.device)
    _check(la_backward_saved(q.data_ptr(), k.data_ptr(), v.data_ptr(), dout.data_ptr(),
                             dq.data_ptr(), dkk.data_ptr(), dvv.data_ptr(), B, H, N,
                             dk, dv, causal, eps, code, saved.data_ptr(), saved.numel(),
                             workspace.data_ptr(), workspace.numel(), _stream_ptr(q)))
    return dq, dkk, dvv
