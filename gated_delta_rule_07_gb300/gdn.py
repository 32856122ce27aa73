"""ctypes binding of libgdn.so (the C ABI declared in include/gdn.h).

Argument marshalling only: every step of the computation runs in the library's CUDA
kernels.  Functions named after the C entry points take torch CUDA tensors, pass their
data pointers and the current torch stream, and raise ``GdnError`` on a non-OK status.
``forward()`` is the convenience call that allocates the outputs and the workspace.

Importing this module loads the library and raises ImportError when it has not been built
(``python -m gated_delta_rule_07_gb300.build``); there is no fallback implementation.
"""
from __future__ import annotations

import ctypes
import os

import torch

from . import build as _build

LIB_PATH = _build.LIB

if not os.path.exists(LIB_PATH):
    raise ImportError(f"libgdn.so is not built ({LIB_PATH}); run "
                      "`python -m gated_delta_rule_07_gb300.build` (needs nvcc)")

_lib = ctypes.CDLL(LIB_PATH)

GDN_OK = 0
STATUS_NAMES = {0: "GDN_OK", 1: "GDN_ERR_INVALID_ARGUMENT", 2: "GDN_ERR_UNSUPPORTED",
                3: "GDN_ERR_WORKSPACE", 4: "GDN_ERR_CUDA", 5: "GDN_ERR_DEVICE_TIMEOUT",
                6: "GDN_ERR_DEVICE_INPUT", 7: "GDN_ERR_DEVICE_RANGE"}
GDN_BF16, GDN_F32 = 0, 1
EXPORTED = ("gdn_status_string", "gdn_check_problem", "gdn_workspace_size", "gdn_forward",
            "gdn_chunk_prepare", "gdn_segment_summary", "gdn_state_prefix_scan",
            "gdn_chunk_emit", "gdn_device_status", "gdn_version",
            "gdn_segment_summary_fused", "gdn_chunk_emit_fused", "gdn_last_error_string",
            "gdn_forward_static_scratch", "gdn_forward_timed", "gdn_forward_with_limits",
            "gdn_check_decode_problem", "gdn_decode_step", "gdn_backward_workspace_size",
            "gdn_backward", "gdn_prologue")


class Problem(ctypes.Structure):
    _fields_ = [("total_tokens", ctypes.c_int64), ("num_seqs", ctypes.c_int32),
                ("hk", ctypes.c_int32), ("hv", ctypes.c_int32), ("k_dim", ctypes.c_int32),
                ("v_dim", ctypes.c_int32), ("chunk", ctypes.c_int32),
                ("segments_per_seq", ctypes.c_int32), ("io_dtype", ctypes.c_int32)]


class DecodeProblem(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int32), ("slots", ctypes.c_int32), ("hk", ctypes.c_int32),
                ("hv", ctypes.c_int32), ("k_dim", ctypes.c_int32), ("v_dim", ctypes.c_int32),
                ("io_dtype", ctypes.c_int32)]


class PrologueProblem(ctypes.Structure):
    _fields_ = [("total_tokens", ctypes.c_int64), ("num_seqs", ctypes.c_int32),
                ("hk", ctypes.c_int32), ("hv", ctypes.c_int32), ("k_dim", ctypes.c_int32),
                ("v_dim", ctypes.c_int32), ("conv_width", ctypes.c_int32),
                ("activation", ctypes.c_int32), ("io_dtype", ctypes.c_int32)]


class GdnError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        msg = f"{where}: {gdn_status_string(status)}"
        if status == 4:
            msg += f" ({_lib.gdn_last_error_string().decode()})"
        super().__init__(msg)


_vp, _fp, _ip = ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p
_pp = ctypes.POINTER(Problem)
_lib.gdn_status_string.restype = ctypes.c_char_p
_lib.gdn_status_string.argtypes = [ctypes.c_int]
_lib.gdn_last_error_string.restype = ctypes.c_char_p
_lib.gdn_last_error_string.argtypes = []
_lib.gdn_check_problem.argtypes = [_pp]
_lib.gdn_workspace_size.restype = ctypes.c_size_t
_lib.gdn_workspace_size.argtypes = [_pp]
_lib.gdn_forward.argtypes = [_pp, _vp, _vp, _vp, _fp, _fp, _fp, _ip, _vp, _fp, _vp,
                             ctypes.c_size_t, _vp]
_lib.gdn_forward_timed.argtypes = [_pp, _vp, _vp, _vp, _fp, _fp, _fp, _ip, _vp, _fp, _vp,
                             ctypes.c_size_t, _vp, ctypes.POINTER(ctypes.c_float)]
_lib.gdn_forward_with_limits.argtypes = [_pp, _vp, _vp, _vp, _fp, _fp, _fp, _ip, _vp, _fp, _vp,
                                         ctypes.c_size_t, _vp, ctypes.c_longlong, ctypes.c_int]
_lib.gdn_chunk_prepare.argtypes = [_pp, _vp, _vp, _fp, _fp, _ip, _vp, _vp, _fp, _ip, _vp]
_lib.gdn_segment_summary.argtypes = [_pp, _vp, _vp, _vp, _fp, _ip, _fp, _fp, _ip, _vp]
_lib.gdn_state_prefix_scan.argtypes = [_pp, _fp, _fp, _fp, _fp, _fp, _vp]
_lib.gdn_chunk_emit.argtypes = [_pp, _vp, _vp, _vp, _vp, _fp, _fp, _ip, _vp, _fp, _ip, _vp]
_lib.gdn_device_status.argtypes = [_vp, ctypes.c_int, _vp]
_lib.gdn_segment_summary_fused.argtypes = [_pp, _vp, _vp, _fp, _fp, _ip, _fp, _fp, ctypes.c_int,
                                           _ip, _vp]
_lib.gdn_chunk_emit_fused.argtypes = [_pp, _vp, _vp, _vp, _fp, _fp, _fp, _ip, _vp, _fp, _ip, _vp]
_lib.gdn_forward_static_scratch.argtypes = [_pp, _vp, _vp, _vp, _fp, _fp, _fp, _ip, _vp, _fp, _vp]
_lib.gdn_backward_workspace_size.restype = ctypes.c_size_t
_lib.gdn_backward_workspace_size.argtypes = [_pp]
_lib.gdn_backward.argtypes = [_pp, _vp, _vp, _vp, _fp, _fp, _fp, _ip, _vp, _fp, _vp, _vp, _vp,
                              _fp, _fp, _fp, _vp, ctypes.c_size_t, _vp]
_lib.gdn_prologue.argtypes = [ctypes.POINTER(PrologueProblem), _vp, _fp, _vp, _vp, _vp, _fp, _fp,
                              _ip, _vp, _vp, _vp, _fp, _fp, _vp, _ip, _vp]
_dpp = ctypes.POINTER(DecodeProblem)
_lib.gdn_check_decode_problem.argtypes = [_dpp]
_lib.gdn_decode_step.argtypes = [_dpp, _vp, _vp, _vp, _fp, _fp, _ip, _fp, _vp, _ip, _vp]
for _n in EXPORTED:
    if _n not in ("gdn_status_string", "gdn_workspace_size", "gdn_last_error_string",
                  "gdn_backward_workspace_size"):
        getattr(_lib, _n).restype = ctypes.c_int


def gdn_status_string(status: int) -> str:
    return _lib.gdn_status_string(int(status)).decode()


def gdn_version() -> int:
    return _lib.gdn_version()


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _check(status, where):
    if status != GDN_OK:
        raise GdnError(status, where)


def make_problem(T, N, hk, hv, K, V, P=1, dtype=torch.bfloat16, chunk=64):
    io = {torch.bfloat16: GDN_BF16, torch.float32: GDN_F32}.get(dtype)
    if io is None:
        raise GdnError(2, f"dtype {dtype}")
    return Problem(int(T), int(N), int(hk), int(hv), int(K), int(V), int(chunk), int(P), io)


def problem_for(q, v, cu_seqlens=None, P=1) -> Problem:
    T, hk, K = q.shape
    hv, V = v.shape[1], v.shape[2]
    N = 1 if cu_seqlens is None else cu_seqlens.numel() - 1
    return make_problem(T, N, hk, hv, K, V, P, q.dtype)


def gdn_check_problem(p: Problem) -> int:
    return _lib.gdn_check_problem(ctypes.byref(p))


def gdn_workspace_size(p: Problem) -> int:
    return int(_lib.gdn_workspace_size(ctypes.byref(p)))


def gdn_forward(p, q, k, v, g, beta, h0, cu_seqlens, out, h_final, workspace, ws_bytes=None,
                stream=None):
    ws_bytes = workspace.numel() * workspace.element_size() if ws_bytes is None else ws_bytes
    _check(_lib.gdn_forward(ctypes.byref(p), _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta),
                            _ptr(h0), _ptr(cu_seqlens), _ptr(out), _ptr(h_final),
                            _ptr(workspace), int(ws_bytes), _stream(stream)), "gdn_forward")


def gdn_forward_timed(p, q, k, v, g, beta, h0, cu_seqlens, out, h_final, workspace,
                      ws_bytes=None, stream=None):
    """gdn_forward that waits for its own end and returns the milliseconds of (summaries,
    prefix scan, phase 3, first summary kernel) measured with CUDA events on the stream."""
    ws_bytes = workspace.numel() * workspace.element_size() if ws_bytes is None else ws_bytes
    ms = (ctypes.c_float * 4)()
    _check(_lib.gdn_forward_timed(ctypes.byref(p), _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta),
                                  _ptr(h0), _ptr(cu_seqlens), _ptr(out), _ptr(h_final),
                                  _ptr(workspace), int(ws_bytes), _stream(stream), ms),
           "gdn_forward_timed")
    return float(ms[0]), float(ms[1]), float(ms[2]), float(ms[3])


def gdn_forward_with_limits(p, q, k, v, g, beta, h0, cu_seqlens, out, h_final, workspace,
                            wait_cycles=0, fault=0, ws_bytes=None, stream=None):
    """gdn_forward with a given limit on the device's bounded waits and an optional injected
    fault (tests of the failure detection; see include/gdn.h)."""
    ws_bytes = workspace.numel() * workspace.element_size() if ws_bytes is None else ws_bytes
    _check(_lib.gdn_forward_with_limits(ctypes.byref(p), _ptr(q), _ptr(k), _ptr(v), _ptr(g),
                                        _ptr(beta), _ptr(h0), _ptr(cu_seqlens), _ptr(out),
                                        _ptr(h_final), _ptr(workspace), int(ws_bytes),
                                        _stream(stream), int(wait_cycles), int(fault)),
           "gdn_forward_with_limits")


def gdn_forward_static_scratch(p, q, k, v, g, beta, h0, cu_seqlens, out, h_final, stream=None):
    """gdn_forward without a workspace: for callers that cannot allocate device memory.  Its
    scratch is the library's own 64 MiB device array (see include/gdn.h for the limits)."""
    _check(_lib.gdn_forward_static_scratch(ctypes.byref(p), _ptr(q), _ptr(k), _ptr(v), _ptr(g),
                                           _ptr(beta), _ptr(h0), _ptr(cu_seqlens), _ptr(out),
                                           _ptr(h_final), _stream(stream)),
           "gdn_forward_static_scratch")


def gdn_chunk_prepare(p, k, v, g, beta, cu_seqlens, w, u, gcum, dev_status=None, stream=None):
    _check(_lib.gdn_chunk_prepare(ctypes.byref(p), _ptr(k), _ptr(v), _ptr(g), _ptr(beta),
                                  _ptr(cu_seqlens), _ptr(w), _ptr(u), _ptr(gcum),
                                  _ptr(dev_status), _stream(stream)), "gdn_chunk_prepare")


def gdn_segment_summary(p, k, w, u, gcum, cu_seqlens, M, U, dev_status=None, stream=None):
    _check(_lib.gdn_segment_summary(ctypes.byref(p), _ptr(k), _ptr(w), _ptr(u), _ptr(gcum),
                                    _ptr(cu_seqlens), _ptr(M), _ptr(U), _ptr(dev_status),
                                    _stream(stream)), "gdn_segment_summary")


def gdn_state_prefix_scan(p, M, U, h0, h_in, h_final, stream=None):
    _check(_lib.gdn_state_prefix_scan(ctypes.byref(p), _ptr(M), _ptr(U), _ptr(h0), _ptr(h_in),
                                      _ptr(h_final), _stream(stream)), "gdn_state_prefix_scan")


def gdn_chunk_emit(p, q, k, w, u, gcum, h_in, cu_seqlens, out, h_final, dev_status=None,
                   stream=None):
    _check(_lib.gdn_chunk_emit(ctypes.byref(p), _ptr(q), _ptr(k), _ptr(w), _ptr(u), _ptr(gcum),
                               _ptr(h_in), _ptr(cu_seqlens), _ptr(out), _ptr(h_final),
                               _ptr(dev_status), _stream(stream)), "gdn_chunk_emit")


def gdn_segment_summary_fused(p, k, v, g, beta, cu_seqlens, M, U, skip_last=False,
                              dev_status=None, stream=None):
    _check(_lib.gdn_segment_summary_fused(ctypes.byref(p), _ptr(k), _ptr(v), _ptr(g),
                                          _ptr(beta), _ptr(cu_seqlens), _ptr(M), _ptr(U),
                                          int(bool(skip_last)), _ptr(dev_status),
                                          _stream(stream)), "gdn_segment_summary_fused")


def gdn_chunk_emit_fused(p, q, k, v, g, beta, h_in, cu_seqlens, out, h_final, dev_status=None,
                         stream=None):
    _check(_lib.gdn_chunk_emit_fused(ctypes.byref(p), _ptr(q), _ptr(k), _ptr(v), _ptr(g),
                                     _ptr(beta), _ptr(h_in), _ptr(cu_seqlens), _ptr(out),
                                     _ptr(h_final), _ptr(dev_status), _stream(stream)),
           "gdn_chunk_emit_fused")


def gdn_backward_workspace_size(p: Problem) -> int:
    return int(_lib.gdn_backward_workspace_size(ctypes.byref(p)))


def gdn_backward(p, q, k, v, g, beta, h0, cu_seqlens, dout, dh_final, dq, dk, dv, dg, dbeta,
                 dh0, workspace, ws_bytes=None, stream=None):
    ws_bytes = workspace.numel() * workspace.element_size() if ws_bytes is None else ws_bytes
    _check(_lib.gdn_backward(ctypes.byref(p), _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta),
                             _ptr(h0), _ptr(cu_seqlens), _ptr(dout), _ptr(dh_final), _ptr(dq),
                             _ptr(dk), _ptr(dv), _ptr(dg), _ptr(dbeta), _ptr(dh0),
                             _ptr(workspace), int(ws_bytes), _stream(stream)), "gdn_backward")


def backward(q, k, v, g, beta, dout, h0=None, dh_final=None, cu_seqlens=None, workspace=None,
             check_status=False, stream=None):
    """Gradients (dq, dk, dv, dg, dbeta, dh0) of <dout, out> + <dh_final, h_final> through the
    forward on the same inputs; allocates the outputs (and the workspace unless given)."""
    p = problem_for(q, v, cu_seqlens)
    N = p.num_seqs
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    dg, dbeta = torch.empty_like(g), torch.empty_like(beta)
    dh0 = torch.empty(N, p.hv, p.k_dim, p.v_dim, dtype=torch.float32, device=q.device)
    if workspace is None:
        workspace = torch.empty(max(gdn_backward_workspace_size(p), 256), dtype=torch.uint8,
                                device=q.device)
    gdn_backward(p, q, k, v, g, beta, h0, cu_seqlens, dout, dh_final, dq, dk, dv, dg, dbeta,
                 dh0, workspace, stream=stream)
    if check_status:
        _check(gdn_device_status(workspace, True, stream), "gdn_backward (device status)")
    return dq, dk, dv, dg, dbeta, dh0


def gdn_prologue(p, x, conv_w, conv_state_in, a, b, A_log, dt_bias, cu_seqlens, q, k, v, g,
                 beta, conv_state_out, dev_status=None, stream=None):
    _check(_lib.gdn_prologue(ctypes.byref(p), _ptr(x), _ptr(conv_w), _ptr(conv_state_in), _ptr(a),
                             _ptr(b), _ptr(A_log), _ptr(dt_bias), _ptr(cu_seqlens), _ptr(q),
                             _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(conv_state_out),
                             _ptr(dev_status), _stream(stream)), "gdn_prologue")


def prologue(x, conv_w, a, b, A_log, dt_bias, hk, hv, K, V, conv_state=None, cu_seqlens=None,
             activation="none", check_status=False, stream=None):
    """q, k, v, g, beta, new conv state from the projections (layouts of include/gdn.h)."""
    T = x.shape[0]
    N = 1 if cu_seqlens is None else cu_seqlens.numel() - 1
    W = conv_w.shape[1]
    io = {torch.bfloat16: GDN_BF16, torch.float32: GDN_F32}[x.dtype]
    p = PrologueProblem(T, N, hk, hv, K, V, W, {"none": 0, "silu": 1}[activation], io)
    dev = x.device
    q = torch.empty(T, hk, K, dtype=x.dtype, device=dev)
    k = torch.empty_like(q)
    v = torch.empty(T, hv, V, dtype=x.dtype, device=dev)
    g = torch.empty(T, hv, dtype=torch.float32, device=dev)
    beta = torch.empty_like(g)
    new_state = torch.empty(N, x.shape[1], max(W - 1, 0), dtype=x.dtype, device=dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev) if check_status else None
    gdn_prologue(p, x, conv_w, conv_state, a, b, A_log, dt_bias, cu_seqlens, q, k, v, g, beta,
                 new_state if W > 1 else None, st, stream)
    if check_status:
        _check(gdn_device_status(st, True, stream), "gdn_prologue (device status)")
    return q, k, v, g, beta, new_state


def make_decode_problem(B, slots, hk, hv, K, V, dtype=torch.bfloat16) -> DecodeProblem:
    io = {torch.bfloat16: GDN_BF16, torch.float32: GDN_F32}.get(dtype)
    if io is None:
        raise GdnError(2, f"dtype {dtype}")
    return DecodeProblem(int(B), int(slots), int(hk), int(hv), int(K), int(V), io)


def decode_problem_for(q, v, state) -> DecodeProblem:
    B, hk, K = q.shape
    return make_decode_problem(B, state.shape[0], hk, v.shape[1], K, v.shape[2], q.dtype)


def gdn_check_decode_problem(p: DecodeProblem) -> int:
    return _lib.gdn_check_decode_problem(ctypes.byref(p))


def gdn_decode_step(p, q, k, v, g, beta, slot, state, out, dev_status=None, stream=None):
    _check(_lib.gdn_decode_step(ctypes.byref(p), _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta),
                                _ptr(slot), _ptr(state), _ptr(out), _ptr(dev_status),
                                _stream(stream)), "gdn_decode_step")


def decode(q, k, v, g, beta, slot, state, out=None, check_status=False, stream=None):
    """One decode step: row b continues the request held in state[slot[b]] (updated in place).
    Returns out [B, hv, V]; with check_status, waits and raises on a device-side error."""
    p = decode_problem_for(q, v, state)
    if out is None:
        out = torch.empty_like(v)
    st = torch.zeros(1, dtype=torch.int32, device=q.device) if check_status else None
    gdn_decode_step(p, q, k, v, g, beta, slot, state, out, st, stream)
    if check_status:
        _check(gdn_device_status(st, reset=True, stream=stream), "gdn_decode_step (device status)")
    return out


def gdn_device_status(status_word, reset=True, stream=None) -> int:
    """Synchronous read of a device status word (a dev_status tensor or a workspace)."""
    return _lib.gdn_device_status(_ptr(status_word), int(bool(reset)), _stream(stream))


# ------------------------------------------------------------------ convenience API

def workspace_for(p: Problem, device="cuda") -> torch.Tensor:
    return torch.empty(max(gdn_workspace_size(p), 256), dtype=torch.uint8, device=device)


def forward(q, k, v, g, beta, h0=None, cu_seqlens=None, P=1, out=None,
            h_final=None, workspace=None, want_final=True, check_status=False, stream=None):
    """out, h_final = forward(...) on CUDA tensors (layouts of include/gdn.h).

    ``cu_seqlens`` is an int32 CUDA tensor [N+1] or None (one sequence).  With
    ``check_status`` the device status word is read back (a synchronisation)."""
    p = problem_for(q, v, cu_seqlens, P)
    N = p.num_seqs
    if out is None:
        out = torch.empty_like(v)
    if h_final is None and want_final:
        h_final = torch.empty(N, p.hv, p.k_dim, p.v_dim, dtype=torch.float32, device=q.device)
    if workspace is None:
        workspace = workspace_for(p, q.device)
    gdn_forward(p, q, k, v, g, beta, h0, cu_seqlens, out, h_final, workspace, stream=stream)
    if check_status:
        st = gdn_device_status(workspace, True, stream)
        _check(st, "gdn_forward (device status)")
    return out, h_final
