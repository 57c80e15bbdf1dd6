"""ctypes binding to libkda.so: argument marshalling only.

Every function takes torch CUDA tensors, checks their dtype / shape / layout,
allocates the outputs the caller did not pass (with torch, on the tensors'
device), and calls the C entry point of the same name on the current CUDA
stream.  All arithmetic runs in the library's kernels; there is no fallback.
"""
from __future__ import annotations

import ctypes
import threading

import torch

from . import build as _build

_lib = None
_lock = threading.Lock()


class KDAError(RuntimeError):
    """A libkda entry point returned a non-zero kda_status_t."""

    def __init__(self, fn, status, msg):
        super().__init__("%s failed: %s (status %d)" % (fn, msg, status))
        self.status = status


class PrefillDesc(ctypes.Structure):
    _fields_ = [("num_seqs", ctypes.c_int32), ("total_tokens", ctypes.c_int32),
                ("num_heads", ctypes.c_int32), ("dk", ctypes.c_int32), ("dv", ctypes.c_int32),
                ("act_dtype", ctypes.c_int32), ("chunk", ctypes.c_int32),
                ("num_segments", ctypes.c_int32)]


F32, BF16 = 0, 1
_ACT = {torch.float32: F32, torch.bfloat16: BF16}
_P = ctypes.c_void_p
_I = ctypes.c_int32


def lib():
    """Load (building first if needed) the in-tree libkda.so.  Raises if it cannot."""
    global _lib
    with _lock:
        if _lib is None:
            path = _build.build()
            L = ctypes.CDLL(path)
            L.kda_prefill_num_segments.restype = _I
            L.kda_prefill_num_segments.argtypes = [ctypes.POINTER(PrefillDesc)]
            L.kda_prefill_workspace_size.restype = ctypes.c_size_t
            L.kda_prefill_workspace_size.argtypes = [ctypes.POINTER(PrefillDesc)]
            L.kda_prefill_chunked.restype = ctypes.c_int
            L.kda_prefill_chunked.argtypes = [ctypes.POINTER(PrefillDesc)] + [_P] * 10 + \
                [ctypes.c_size_t, _P, _P]
            L.kda_prefill_chunked_timed.restype = ctypes.c_int
            L.kda_prefill_chunked_timed.argtypes = [ctypes.POINTER(PrefillDesc)] + [_P] * 10 + \
                [ctypes.c_size_t, _P, _P, _P]
            L.kda_prefill_chunked_gated.restype = ctypes.c_int
            L.kda_prefill_chunked_gated.argtypes = [ctypes.POINTER(PrefillDesc)] + [_P] * 10 + \
                [ctypes.c_size_t, _P, _P]
            L.kda_prefill_ckpt_workspace_size.restype = ctypes.c_size_t
            L.kda_prefill_ckpt_workspace_size.argtypes = [ctypes.POINTER(PrefillDesc), _I]
            L.kda_prefill_chunked_ckpt.restype = ctypes.c_int
            L.kda_prefill_chunked_ckpt.argtypes = [ctypes.POINTER(PrefillDesc)] + [_P] * 9 + \
                [_I, _P, _P, ctypes.c_size_t, _P, _P]
            L.kda_prefill_backward_workspace_size.restype = ctypes.c_size_t
            L.kda_prefill_backward_workspace_size.argtypes = [ctypes.POINTER(PrefillDesc)]
            L.kda_prefill_backward_num_segments.restype = _I
            L.kda_prefill_backward_num_segments.argtypes = [ctypes.POINTER(PrefillDesc)]
            L.kda_prefill_backward.restype = ctypes.c_int
            L.kda_prefill_backward.argtypes = [ctypes.POINTER(PrefillDesc)] + [_P] * 16 + \
                [ctypes.c_size_t, _P, _P]
            L.kda_prefill_segments.restype = ctypes.c_int
            L.kda_prefill_segments.argtypes = [ctypes.POINTER(PrefillDesc), _I, _I] + [_P] * 11
            L.kda_prefill_chunked_noalloc.restype = ctypes.c_int
            L.kda_prefill_chunked_noalloc.argtypes = [ctypes.POINTER(PrefillDesc)] + [_P] * 11
            L.kda_decode_step.restype = ctypes.c_int
            L.kda_decode_step.argtypes = [_I] * 5 + [_P] * 9
            L.kda_state_transfer.restype = ctypes.c_int
            L.kda_state_transfer.argtypes = [ctypes.POINTER(PrefillDesc), _I, _I] + [_P] * 12
            L.kda_prefill_combine.restype = ctypes.c_int
            L.kda_prefill_combine.argtypes = [ctypes.POINTER(PrefillDesc), _I] + [_P] * 7
            L.kda_state_compose.restype = ctypes.c_int
            L.kda_state_compose.argtypes = [_I] * 4 + [_P] * 8
            L.kda_selftest_wait_timeout.restype = ctypes.c_int
            L.kda_selftest_wait_timeout.argtypes = [_I, _P, _P]
            L.kda_status_string.restype = ctypes.c_char_p
            L.kda_status_string.argtypes = [ctypes.c_int]
            L.kda_build_info.restype = ctypes.c_char_p
            L.kda_build_info.argtypes = []
            _lib = L
    return _lib


def library_path() -> str:
    return _build.LIB


def _check(fn, rc):
    if rc != 0:
        raise KDAError(fn, rc, lib().kda_status_string(rc).decode())


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream, device):
    if stream is None:
        stream = torch.cuda.current_stream(device)
    return ctypes.c_void_p(stream.cuda_stream)


def _need(t, name, dtype=None, shape=None, device=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError("%s must be a torch.Tensor" % name)
    if not t.is_cuda:
        raise ValueError("%s must be a CUDA tensor" % name)
    if device is not None and t.device != device:
        raise ValueError("%s is on %s, expected %s" % (name, t.device, device))
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)
    if dtype is not None and t.dtype != dtype:
        raise ValueError("%s must be %s, got %s" % (name, dtype, t.dtype))
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError("%s must have shape %s, got %s" % (name, tuple(shape), tuple(t.shape)))
    return t


def _desc(N, T, H, dk, dv, act, num_segments):
    return PrefillDesc(N, T, H, dk, dv, act, 16, int(num_segments))


def prefill_desc(q_or_k, v, cu_seqlens, num_segments=0):
    T, H, dk = q_or_k.shape
    return _desc(cu_seqlens.numel() - 1, T, H, dk, v.shape[2], _ACT[q_or_k.dtype], num_segments)


def prefill_num_segments(desc) -> int:
    return int(lib().kda_prefill_num_segments(ctypes.byref(desc)))


def prefill_workspace_size(desc) -> int:
    return int(lib().kda_prefill_workspace_size(ctypes.byref(desc)))


def prefill_chunked(q, k, v, g, beta, S0=None, cu_seqlens=None, *, num_segments=0, out=None,
                    S_final=None, want_final_state=True, workspace=None, dev_status=None,
                    stream=None, stage_events=None):
    """Chunked KDA prefill over packed sequences (see kda_prefill_chunked in kda.h).

    q, k ``[T, H, dk]`` and v ``[T, H, dv]`` (fp32 or bf16, same dtype); g ``[T, H,
    dk]`` and beta ``[T, H]`` fp32; S0 ``[N, H, dk, dv]`` fp32 or None;
    cu_seqlens int32 ``[N+1]`` (None = one sequence).  Returns ``(out, S_final)``.
    ``stage_events`` (four ``torch.cuda.Event``) calls kda_prefill_chunked_timed
    instead, which records them around the call's launches (measurement only).
    """
    dev = q.device
    T, H, dk = q.shape
    dv = v.shape[2]
    act = _ACT.get(q.dtype)
    if act is None:
        raise ValueError("q must be float32 or bfloat16")
    _need(q, "q", q.dtype, (T, H, dk))
    _need(k, "k", q.dtype, (T, H, dk), dev)
    _need(v, "v", q.dtype, (T, H, dv), dev)
    _need(g, "g", torch.float32, (T, H, dk), dev)
    _need(beta, "beta", torch.float32, (T, H), dev)
    if cu_seqlens is None:
        cu_seqlens = torch.tensor([0, T], dtype=torch.int32, device=dev)
    _need(cu_seqlens, "cu_seqlens", torch.int32, None, dev)
    N = cu_seqlens.numel() - 1
    if S0 is not None:
        _need(S0, "S0", torch.float32, (N, H, dk, dv), dev)
    if out is None:
        out = torch.empty((T, H, dv), dtype=q.dtype, device=dev)
    _need(out, "out", q.dtype, (T, H, dv), dev)
    if S_final is None and want_final_state:
        S_final = torch.empty((N, H, dk, dv), dtype=torch.float32, device=dev)
    if S_final is not None:
        _need(S_final, "S_final", torch.float32, (N, H, dk, dv), dev)
    desc = _desc(N, T, H, dk, dv, act, num_segments)
    ws_bytes = prefill_workspace_size(desc)
    if ws_bytes > 0 and workspace is None:
        workspace = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    ws_len = 0 if workspace is None else workspace.numel() * workspace.element_size()
    if dev_status is not None:
        _need(dev_status, "dev_status", torch.int32, None, dev)
    if stage_events is None:
        rc = lib().kda_prefill_chunked(ctypes.byref(desc), _ptr(q), _ptr(k), _ptr(v), _ptr(g),
                                       _ptr(beta), _ptr(S0), _ptr(cu_seqlens), _ptr(out),
                                       _ptr(S_final), _ptr(workspace), ws_len, _ptr(dev_status),
                                       _stream(stream, dev))
        _check("kda_prefill_chunked", rc)
        return out, S_final
    if len(stage_events) != 4:
        raise ValueError("stage_events must be four torch.cuda.Event")
    st = torch.cuda.current_stream(dev) if stream is None else stream
    for e in stage_events:  # torch creates an event's handle at its first record
        if not e.cuda_event:
            e.record(st)
    evs = (ctypes.c_void_p * 4)(*[e.cuda_event for e in stage_events])
    rc = lib().kda_prefill_chunked_timed(ctypes.byref(desc), _ptr(q), _ptr(k), _ptr(v), _ptr(g),
                                         _ptr(beta), _ptr(S0), _ptr(cu_seqlens), _ptr(out),
                                         _ptr(S_final), _ptr(workspace), ws_len,
                                         _ptr(dev_status), ctypes.cast(evs, ctypes.c_void_p),
                                         _stream(st, dev))
    _check("kda_prefill_chunked_timed", rc)
    return out, S_final


def prefill_chunked_gated(q, k, v, x_g, x_beta, S0=None, cu_seqlens=None, *, num_segments=0,
                          out=None, S_final=None, want_final_state=True, workspace=None,
                          dev_status=None, stream=None):
    """Prefill from the pre-activations (see kda_prefill_chunked_gated in kda.h):
    q, k ``[T, H, 128]`` BF16 not normalised, v ``[T, H, 128]`` BF16, x_g ``[T, H,
    128]`` BF16, x_beta ``[T, H]`` fp32; the kernels form g = -5 sigmoid(x_g), beta =
    sigmoid(x_beta) and the normalised q, k.  Returns ``(out, S_final)``."""
    dev = q.device
    T, H, dk = q.shape
    dv = v.shape[2]
    act = _ACT.get(q.dtype)
    if act is None:
        raise ValueError("q must be float32 or bfloat16")
    _need(q, "q", q.dtype, (T, H, dk))
    _need(k, "k", q.dtype, (T, H, dk), dev)
    _need(v, "v", q.dtype, (T, H, dv), dev)
    _need(x_g, "x_g", q.dtype, (T, H, dk), dev)
    _need(x_beta, "x_beta", torch.float32, (T, H), dev)
    if cu_seqlens is None:
        cu_seqlens = torch.tensor([0, T], dtype=torch.int32, device=dev)
    _need(cu_seqlens, "cu_seqlens", torch.int32, None, dev)
    N = cu_seqlens.numel() - 1
    if S0 is not None:
        _need(S0, "S0", torch.float32, (N, H, dk, dv), dev)
    if out is None:
        out = torch.empty((T, H, dv), dtype=q.dtype, device=dev)
    _need(out, "out", q.dtype, (T, H, dv), dev)
    if S_final is None and want_final_state:
        S_final = torch.empty((N, H, dk, dv), dtype=torch.float32, device=dev)
    if S_final is not None:
        _need(S_final, "S_final", torch.float32, (N, H, dk, dv), dev)
    desc = _desc(N, T, H, dk, dv, act, num_segments)
    ws_bytes = prefill_workspace_size(desc)
    if ws_bytes > 0 and workspace is None:
        workspace = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    ws_len = 0 if workspace is None else workspace.numel() * workspace.element_size()
    if dev_status is not None:
        _need(dev_status, "dev_status", torch.int32, None, dev)
    rc = lib().kda_prefill_chunked_gated(ctypes.byref(desc), _ptr(q), _ptr(k), _ptr(v),
                                         _ptr(x_g), _ptr(x_beta), _ptr(S0), _ptr(cu_seqlens),
                                         _ptr(out), _ptr(S_final), _ptr(workspace), ws_len,
                                         _ptr(dev_status), _stream(stream, dev))
    _check("kda_prefill_chunked_gated", rc)
    return out, S_final


def prefill_ckpt_workspace_size(desc, ckpt_interval) -> int:
    return int(lib().kda_prefill_ckpt_workspace_size(ctypes.byref(desc), int(ckpt_interval)))


def num_checkpoints(cu_seqlens, ckpt_interval) -> int:
    """Number of state checkpoints kda_prefill_chunked_ckpt writes: sum over the
    sequences of floor(len / ckpt_interval) (reads cu_seqlens on the host)."""
    cu = cu_seqlens.detach().cpu().tolist()
    return sum((cu[i + 1] - cu[i]) // ckpt_interval for i in range(len(cu) - 1))


def prefill_chunked_ckpt(q, k, v, g, beta, S0=None, cu_seqlens=None, *, ckpt_interval,
                         ckpt_states=None, num_segments=0, out=None, S_final=None,
                         want_final_state=True, workspace=None, dev_status=None, stream=None):
    """prefill_chunked that also writes the state after every ckpt_interval tokens
    of each sequence (see kda_prefill_chunked_ckpt in kda.h).  ckpt_states
    ``[K, H, dk, dv]`` fp32 with K >= num_checkpoints(cu_seqlens, ckpt_interval)
    (allocated when None).  Returns ``(out, S_final, ckpt_states)``."""
    dev = q.device
    T, H, dk = q.shape
    dv = v.shape[2]
    act = _ACT.get(q.dtype)
    if act is None:
        raise ValueError("q must be float32 or bfloat16")
    if int(ckpt_interval) <= 0 or int(ckpt_interval) % 16:
        raise ValueError("ckpt_interval must be a positive multiple of 16")
    _need(q, "q", q.dtype, (T, H, dk))
    _need(k, "k", q.dtype, (T, H, dk), dev)
    _need(v, "v", q.dtype, (T, H, dv), dev)
    _need(g, "g", torch.float32, (T, H, dk), dev)
    _need(beta, "beta", torch.float32, (T, H), dev)
    if cu_seqlens is None:
        cu_seqlens = torch.tensor([0, T], dtype=torch.int32, device=dev)
    _need(cu_seqlens, "cu_seqlens", torch.int32, None, dev)
    N = cu_seqlens.numel() - 1
    if S0 is not None:
        _need(S0, "S0", torch.float32, (N, H, dk, dv), dev)
    if out is None:
        out = torch.empty((T, H, dv), dtype=q.dtype, device=dev)
    _need(out, "out", q.dtype, (T, H, dv), dev)
    if S_final is None and want_final_state:
        S_final = torch.empty((N, H, dk, dv), dtype=torch.float32, device=dev)
    if S_final is not None:
        _need(S_final, "S_final", torch.float32, (N, H, dk, dv), dev)
    ckpt_buf = ckpt_states
    if ckpt_states is None:  # at least one slot: the library takes a valid pointer
        K = num_checkpoints(cu_seqlens, int(ckpt_interval))
        ckpt_buf = torch.empty((max(K, 1), H, dk, dv), dtype=torch.float32, device=dev)
        ckpt_states = ckpt_buf[:K]
    _need(ckpt_buf, "ckpt_states", torch.float32, None, dev)
    if tuple(ckpt_buf.shape[1:]) != (H, dk, dv) or ckpt_buf.numel() == 0:
        raise ValueError("ckpt_states must have shape [K, %d, %d, %d], K >= 1" % (H, dk, dv))
    desc = _desc(N, T, H, dk, dv, act, num_segments)
    ws_bytes = prefill_ckpt_workspace_size(desc, ckpt_interval)
    if ws_bytes > 0 and workspace is None:
        workspace = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    ws_len = 0 if workspace is None else workspace.numel() * workspace.element_size()
    if dev_status is not None:
        _need(dev_status, "dev_status", torch.int32, None, dev)
    rc = lib().kda_prefill_chunked_ckpt(ctypes.byref(desc), _ptr(q), _ptr(k), _ptr(v), _ptr(g),
                                        _ptr(beta), _ptr(S0), _ptr(cu_seqlens), _ptr(out),
                                        _ptr(S_final), int(ckpt_interval), _ptr(ckpt_buf),
                                        _ptr(workspace), ws_len, _ptr(dev_status),
                                        _stream(stream, dev))
    _check("kda_prefill_chunked_ckpt", rc)
    return out, S_final, ckpt_states


def prefill_backward_workspace_size(desc) -> int:
    """Workspace bytes kda_prefill_backward needs for ``desc`` (0 on invalid input)."""
    return int(lib().kda_prefill_backward_workspace_size(ctypes.byref(desc)))


def prefill_backward_num_segments(desc) -> int:
    """Segments per sequence kda_prefill_backward uses for ``desc``."""
    return int(lib().kda_prefill_backward_num_segments(ctypes.byref(desc)))


def prefill_backward(q, k, v, g, beta, S0, cu_seqlens, d_out, d_S_final=None, *,
                     want_dS0=True, num_segments=0, workspace=None, dev_status=None,
                     stream=None):
    """Gradients of <d_out, o> + <d_S_final, S_final> for the prefill of the same
    inputs (see kda_prefill_backward in kda.h).  d_out ``[T, H, dv]`` in the
    activation dtype, d_S_final ``[N, H, dk, dv]`` fp32 or None; num_segments
    splits each sequence (0: the library's choice).  Returns fp32
    ``(dq, dk, dv, dg, dbeta, dS0)`` (dS0 None unless want_dS0)."""
    dev = q.device
    T, H, dk = q.shape
    dv = v.shape[2]
    act = _ACT.get(q.dtype)
    if act is None:
        raise ValueError("q must be float32 or bfloat16")
    _need(q, "q", q.dtype, (T, H, dk))
    _need(k, "k", q.dtype, (T, H, dk), dev)
    _need(v, "v", q.dtype, (T, H, dv), dev)
    _need(g, "g", torch.float32, (T, H, dk), dev)
    _need(beta, "beta", torch.float32, (T, H), dev)
    _need(d_out, "d_out", q.dtype, (T, H, dv), dev)
    if cu_seqlens is None:
        cu_seqlens = torch.tensor([0, T], dtype=torch.int32, device=dev)
    _need(cu_seqlens, "cu_seqlens", torch.int32, None, dev)
    N = cu_seqlens.numel() - 1
    if S0 is not None:
        _need(S0, "S0", torch.float32, (N, H, dk, dv), dev)
    if d_S_final is not None:
        _need(d_S_final, "d_S_final", torch.float32, (N, H, dk, dv), dev)
    f32 = dict(dtype=torch.float32, device=dev)
    dq = torch.empty((T, H, dk), **f32)
    dk_ = torch.empty((T, H, dk), **f32)
    dv_ = torch.empty((T, H, dv), **f32)
    dg = torch.empty((T, H, dk), **f32)
    dbeta = torch.empty((T, H), **f32)
    dS0 = torch.empty((N, H, dk, dv), **f32) if want_dS0 else None
    desc = _desc(N, T, H, dk, dv, act, num_segments)
    ws_bytes = prefill_backward_workspace_size(desc)
    if workspace is None:
        workspace = torch.empty(max(ws_bytes, 16), dtype=torch.uint8, device=dev)
    ws_len = workspace.numel() * workspace.element_size()
    if dev_status is not None:
        _need(dev_status, "dev_status", torch.int32, None, dev)
    rc = lib().kda_prefill_backward(ctypes.byref(desc), _ptr(q), _ptr(k), _ptr(v), _ptr(g),
                                    _ptr(beta), _ptr(S0), _ptr(cu_seqlens), _ptr(d_out),
                                    _ptr(d_S_final), _ptr(dq), _ptr(dk_), _ptr(dv_), _ptr(dg),
                                    _ptr(dbeta), _ptr(dS0), _ptr(workspace), ws_len,
                                    _ptr(dev_status), _stream(stream, dev))
    _check("kda_prefill_backward", rc)
    return dq, dk_, dv_, dg, dbeta, dS0


def prefill_segments(q, k, v, g, beta, seg_init_states, cu_seqlens, num_segments, *, seg_begin=0,
                     seg_end=None, out=None, S_final=None, want_final_state=True,
                     dev_status=None, stream=None):
    """Run segments [seg_begin, seg_end) from their given start states (see
    kda_prefill_segments in kda.h).  seg_init_states ``[N, H, S, dk, dv]`` fp32
    (None = zeros for every segment).  Returns ``(out, S_final)``."""
    dev = q.device
    T, H, dk = q.shape
    dv = v.shape[2]
    act = _ACT.get(q.dtype)
    if act is None:
        raise ValueError("q must be float32 or bfloat16")
    _need(q, "q", q.dtype, (T, H, dk))
    _need(k, "k", q.dtype, (T, H, dk), dev)
    _need(v, "v", q.dtype, (T, H, dv), dev)
    _need(g, "g", torch.float32, (T, H, dk), dev)
    _need(beta, "beta", torch.float32, (T, H), dev)
    _need(cu_seqlens, "cu_seqlens", torch.int32, None, dev)
    N = cu_seqlens.numel() - 1
    Sg = int(num_segments)
    if seg_init_states is not None:
        _need(seg_init_states, "seg_init_states", torch.float32, (N, H, Sg, dk, dv), dev)
    if out is None:
        out = torch.empty((T, H, dv), dtype=q.dtype, device=dev)
    _need(out, "out", q.dtype, (T, H, dv), dev)
    if S_final is None and want_final_state:
        S_final = torch.empty((N, H, dk, dv), dtype=torch.float32, device=dev)
    if S_final is not None:
        _need(S_final, "S_final", torch.float32, (N, H, dk, dv), dev)
    desc = _desc(N, T, H, dk, dv, act, Sg)
    seg_end = Sg if seg_end is None else int(seg_end)
    rc = lib().kda_prefill_segments(ctypes.byref(desc), int(seg_begin), seg_end, _ptr(q), _ptr(k),
                                    _ptr(v), _ptr(g),
                                    _ptr(beta), _ptr(seg_init_states), _ptr(cu_seqlens),
                                    _ptr(out), _ptr(S_final), _ptr(dev_status),
                                    _stream(stream, dev))
    _check("kda_prefill_segments", rc)
    return out, S_final


def decode_step(q, k, v, g, beta, S, *, out=None, dev_status=None, stream=None):
    """One decode token per sequence; updates S ``[B, H, dk, dv]`` in place and
    returns out ``[B, H, dv]`` (see kda_decode_step in kda.h)."""
    dev = S.device
    B, H, dk, dv = S.shape
    act = _ACT.get(q.dtype)
    if act is None:
        raise ValueError("q must be float32 or bfloat16")
    _need(q, "q", q.dtype, (B, H, dk), dev)
    _need(k, "k", q.dtype, (B, H, dk), dev)
    _need(v, "v", q.dtype, (B, H, dv), dev)
    _need(g, "g", torch.float32, (B, H, dk), dev)
    _need(beta, "beta", torch.float32, (B, H), dev)
    _need(S, "S", torch.float32, (B, H, dk, dv), dev)
    if out is None:
        out = torch.empty((B, H, dv), dtype=q.dtype, device=dev)
    _need(out, "out", q.dtype, (B, H, dv), dev)
    if dev_status is not None:
        _need(dev_status, "dev_status", torch.int32, None, dev)
    rc = lib().kda_decode_step(B, H, dk, dv, act, _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta),
                               _ptr(S), _ptr(out), _ptr(dev_status), _stream(stream, dev))
    _check("kda_decode_step", rc)
    return out


def state_transfer(k, v, g, beta, cu_seqlens, num_segments, *, seg_begin=0, seg_end=None,
                   transfer=None, zero_init_state=None, q=None, out_zero=None,
                   out_transfer=None, dev_status=None, stream=None):
    """Per (sequence, head, segment) transfer matrix and zero-initial state for
    segments [seg_begin, seg_end) (see kda_state_transfer in kda.h).  With q given
    it also writes the zero-start outputs and A_t^T q_t (allocated if not passed).
    Returns ``(A [N,H,S,dk,dk], B [N,H,S,dk,dv])``, plus ``(out_zero [T,H,dv],
    out_transfer [T,H,dk])`` when q is given."""
    dev = k.device
    T, H, dk = k.shape
    dv = v.shape[2]
    act = _ACT.get(k.dtype)
    if act is None:
        raise ValueError("k must be float32 or bfloat16")
    _need(k, "k", k.dtype, (T, H, dk))
    _need(v, "v", k.dtype, (T, H, dv), dev)
    _need(g, "g", torch.float32, (T, H, dk), dev)
    _need(beta, "beta", torch.float32, (T, H), dev)
    _need(cu_seqlens, "cu_seqlens", torch.int32, None, dev)
    N = cu_seqlens.numel() - 1
    Sg = int(num_segments)
    if transfer is None:
        transfer = torch.empty((N, H, Sg, dk, dk), dtype=torch.float32, device=dev)
    if zero_init_state is None:
        zero_init_state = torch.empty((N, H, Sg, dk, dv), dtype=torch.float32, device=dev)
    _need(transfer, "transfer", torch.float32, (N, H, Sg, dk, dk), dev)
    _need(zero_init_state, "zero_init_state", torch.float32, (N, H, Sg, dk, dv), dev)
    if q is not None:
        _need(q, "q", k.dtype, (T, H, dk), dev)
        if out_zero is None:
            out_zero = torch.empty((T, H, dv), dtype=k.dtype, device=dev)
        if out_transfer is None:
            out_transfer = torch.empty((T, H, dk), dtype=k.dtype, device=dev)
        _need(out_zero, "out_zero", k.dtype, (T, H, dv), dev)
        _need(out_transfer, "out_transfer", k.dtype, (T, H, dk), dev)
    desc = _desc(N, T, H, dk, dv, act, Sg)
    seg_end = Sg if seg_end is None else int(seg_end)
    rc = lib().kda_state_transfer(ctypes.byref(desc), int(seg_begin), seg_end, _ptr(q), _ptr(k),
                                  _ptr(v), _ptr(g), _ptr(beta), _ptr(cu_seqlens), _ptr(transfer),
                                  _ptr(zero_init_state), _ptr(out_zero), _ptr(out_transfer),
                                  _ptr(dev_status), _stream(stream, dev))
    _check("kda_state_transfer", rc)
    if q is not None:
        return transfer, zero_init_state, out_zero, out_transfer
    return transfer, zero_init_state


def prefill_combine(out, out_transfer, seg_init_states, cu_seqlens, *, first_segment=0,
                    start_images=None, num_segments=None, dev_status=None, stream=None):
    """Add start_s^T (A_t^T q_t) to the zero-start outputs in ``out`` (in place),
    see kda_prefill_combine in kda.h.  ``start_images`` (from state_compose) selects
    the tcgen05 path; ``seg_init_states`` may then be None, with ``num_segments``
    given.  Returns ``out``."""
    dev = out.device
    T, H, dv = out.shape
    dk = out_transfer.shape[2]
    act = _ACT.get(out.dtype)
    if act is None:
        raise ValueError("out must be float32 or bfloat16")
    _need(out, "out", out.dtype, (T, H, dv))
    _need(out_transfer, "out_transfer", out.dtype, (T, H, dk), dev)
    _need(cu_seqlens, "cu_seqlens", torch.int32, None, dev)
    N = cu_seqlens.numel() - 1
    if seg_init_states is not None:
        Sg = seg_init_states.shape[2]
        _need(seg_init_states, "seg_init_states", torch.float32, (N, H, Sg, dk, dv), dev)
    else:
        if start_images is None or num_segments is None:
            raise ValueError("seg_init_states, or start_images with num_segments, is required")
        Sg = int(num_segments)
    if start_images is not None:
        _need(start_images, "start_images", torch.bfloat16, (N * H, Sg, dk * dv), dev)
    desc = _desc(N, T, H, dk, dv, act, Sg)
    rc = lib().kda_prefill_combine(ctypes.byref(desc), int(first_segment), _ptr(seg_init_states),
                                   _ptr(start_images), _ptr(out_transfer), _ptr(cu_seqlens),
                                   _ptr(out), _ptr(dev_status), _stream(stream, dev))
    _check("kda_prefill_combine", rc)
    return out


def state_compose(transfer, zero_init_state, S0=None, *, seg_init_states=None, S_final=None,
                  want_starts=True, want_final_state=True, start_images=None, dev_status=None,
                  stream=None):
    """Prefix scan over segments (see kda_state_compose in kda.h): transfer ``[U, S,
    dk, dk]``, zero_init_state ``[U, S, dk, dv]``, S0 ``[U, dk, dv]`` or None.
    Returns ``(seg_init_states [U,S,dk,dv] or None, S_final [U,dk,dv] or None)``;
    without a final state the last pair is never read.  ``start_images`` (BF16
    ``[U, S, 128 * 128]``, dk = dv = 128) also receives each start state as the
    operand image prefill_combine's tcgen05 path reads."""
    dev = transfer.device
    U, Sg, dk, _ = transfer.shape
    dv = zero_init_state.shape[-1]
    _need(transfer, "transfer", torch.float32, (U, Sg, dk, dk))
    _need(zero_init_state, "zero_init_state", torch.float32, (U, Sg, dk, dv), dev)
    if S0 is not None:
        _need(S0, "S0", torch.float32, (U, dk, dv), dev)
    if seg_init_states is None and want_starts:
        seg_init_states = torch.empty((U, Sg, dk, dv), dtype=torch.float32, device=dev)
    if S_final is None and want_final_state:
        S_final = torch.empty((U, dk, dv), dtype=torch.float32, device=dev)
    if start_images is not None:
        _need(start_images, "start_images", torch.bfloat16, (U, Sg, dk * dv), dev)
    if dev_status is not None:
        _need(dev_status, "dev_status", torch.int32, None, dev)
    rc = lib().kda_state_compose(U, Sg, dk, dv, _ptr(transfer), _ptr(zero_init_state), _ptr(S0),
                                 _ptr(seg_init_states), _ptr(S_final), _ptr(start_images),
                                 _ptr(dev_status), _stream(stream, dev))
    _check("kda_state_compose", rc)
    return seg_init_states, S_final


def selftest_wait_timeout(limit_us, dev_status, stream=None):
    """Run the bounded-wait self-test (see kda_selftest_wait_timeout in kda.h): a
    wait that nothing completes gives up after ~limit_us and writes status 5
    (KDA_ERR_TIMEOUT) to dev_status (a device int32 tensor)."""
    _need(dev_status, "dev_status", torch.int32, None)
    rc = lib().kda_selftest_wait_timeout(int(limit_us), _ptr(dev_status),
                                         _stream(stream, dev_status.device))
    _check("kda_selftest_wait_timeout", rc)
