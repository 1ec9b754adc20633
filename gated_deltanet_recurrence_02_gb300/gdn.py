"""ctypes binding of libgdn (include/gdn.h): argument marshalling only.

Every entry point keeps its C name.  Tensors are torch CUDA tensors (the
library only sees their device pointers); shapes give the head counts and
head sizes; the stream defaults to torch's current stream.  Outputs the caller
does not pass are allocated here with torch (device memory is the only thing
torch provides on this path).  Every step of the computation runs in the
library's CUDA kernels; there is no other implementation to fall back to, so
a missing library raises.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

from . import build as _build

GDN_OK = 0
GDN_F32, GDN_F16, GDN_BF16 = 0, 1, 2
GDN_DEVERR_BAD_INDEX, GDN_DEVERR_TIMEOUT = 1, 2
# input conventions (include/gdn.h): OR'd into dtype_qkv / dtype_gate
GDN_QK_L2NORM, GDN_ALPHA_LOG, GDN_BETA_LOGIT = 0x100, 0x200, 0x400
_DT = {torch.float32: GDN_F32, torch.float16: GDN_F16, torch.bfloat16: GDN_BF16}

_lib = None


class GdnError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {status_string(status)} (status {status})")


def lib() -> ctypes.CDLL:
    """The loaded libgdn.so; raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    path = _build.LIB
    if not os.path.exists(path):
        raise RuntimeError(
            f"libgdn.so is not built ({path}); run "
            "`python -c 'import __graft_entry__ as g; g.build()'` first")
    L = ctypes.CDLL(path)
    vp, i, f, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
    L.gdn_prefill_workspace_size.argtypes = [i, i, i, i, i, i, i, i, i]
    L.gdn_prefill_workspace_size.restype = sz
    L.gdn_prefill_chunked.argtypes = [vp] * 8 + [i, vp, vp] + [i] * 8 + [f, i, i, vp, sz, vp]
    L.gdn_prefill_chunked.restype = i
    L.gdn_prefill_chunked_checkpoints.argtypes = ([vp] * 8 + [i, vp, vp] + [i] * 8 + [f, i, i]
                                                  + [vp, i, i, vp, sz, vp])
    L.gdn_prefill_chunked_checkpoints.restype = i
    L.gdn_prefill_chunked_capture.argtypes = ([vp] * 8 + [i, vp, vp] + [i] * 8 + [f, i, i]
                                              + [i, vp, vp, vp, vp, sz, vp])
    L.gdn_prefill_chunked_capture.restype = i
    L.gdn_recurrent_capture.argtypes = ([vp] * 8 + [i, vp, vp] + [i] * 7 + [f, i, i]
                                        + [i, vp, vp, vp, vp])
    L.gdn_recurrent_capture.restype = i
    L.gdn_replay_state_updates.argtypes = [vp, vp, vp, i, vp, i, i, i, i, i, vp]
    L.gdn_replay_state_updates.restype = i
    L.gdn_replay_verify.argtypes = ([vp] * 9 + [i] + [vp] * 3 + [i] * 7 + [f, i, i, i]
                                    + [vp] * 4)
    L.gdn_replay_verify.restype = i
    L.gdn_device_errors.argtypes = [vp, ctypes.POINTER(ctypes.c_uint32)]
    L.gdn_device_errors.restype = i
    L.gdn_status_string.argtypes = [i]
    L.gdn_status_string.restype = ctypes.c_char_p
    L.gdn_set_wait_limit_ns.argtypes = [ctypes.c_uint64]
    L.gdn_set_wait_limit_ns.restype = None
    _lib = L
    return L


def status_string(status: int) -> str:
    return lib().gdn_status_string(int(status)).decode()


def _p(t) -> Optional[int]:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    if not t.is_cuda:
        raise ValueError("libgdn takes device tensors")
    if not t.is_contiguous():
        raise ValueError("libgdn takes contiguous tensors")
    return t.data_ptr()


def _stream(stream) -> Optional[int]:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _codes(q, alpha, conventions: int):
    """dtype_qkv and dtype_gate arguments: storage types plus the input
    convention bits (GDN_QK_L2NORM goes with q/k, the gate bits with alpha/beta)."""
    return (_DT[q.dtype] | (conventions & GDN_QK_L2NORM),
            _DT[alpha.dtype] | (conventions & (GDN_ALPHA_LOG | GDN_BETA_LOGIT)))


def _check(status: int, where: str):
    if status != GDN_OK:
        raise GdnError(status, where)


def slot_width(Hk: int, Hv: int, dk: int, dv: int) -> int:
    """Floats per captured token: Hv decays, Hk*dk keys, Hv*dv deltas."""
    return Hv + Hk * dk + Hv * dv


def gdn_prefill_workspace_size(B, T, Hk, Hv, dk, dv, chunk, dtype_qkv, varlen=False) -> int:
    return int(lib().gdn_prefill_workspace_size(B, T, Hk, Hv, dk, dv, chunk,
                                                _DT.get(dtype_qkv, dtype_qkv), int(bool(varlen))))


def _dims(q, v, B, T, cu_seqlens):
    total_T, Hk, dk = q.shape
    _, Hv, dv = v.shape
    if cu_seqlens is None and T is None:
        T = total_T // B if B else 0
    if cu_seqlens is not None:
        T = total_T
    return int(T), int(Hk), int(dk), int(Hv), int(dv)


def gdn_prefill_chunked(q, k, v, alpha, beta, *, B: int, T: Optional[int] = None,
                        cu_seqlens=None, initial_state=None,
                        initial_state_indices=None, final_state=None, out=None,
                        chunk: int = 64, scale: float = 1.0, workspace=None,
                        want_final_state: bool = True, conventions: int = 0, stream=None):
    """Chunked prefill.  Returns (out, final_state)."""
    T, Hk, dk, Hv, dv = _dims(q, v, B, T, cu_seqlens)
    if out is None:
        out = torch.empty_like(v)
    if final_state is None and want_final_state:
        final_state = torch.empty((B, Hv, dv, dk), dtype=torch.float32, device=v.device)
    n0 = initial_state.shape[0] if initial_state is not None else 0
    need = gdn_prefill_workspace_size(B, T, Hk, Hv, dk, dv, chunk, q.dtype,
                                      varlen=cu_seqlens is not None)
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=v.device)
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    st = lib().gdn_prefill_chunked(
        _p(q), _p(k), _p(v), _p(alpha), _p(beta), _p(cu_seqlens), _p(initial_state),
        _p(initial_state_indices), n0, _p(final_state), _p(out), B, T, Hk, Hk, Hv,
        dk, dv, chunk, scale, *_codes(q, alpha, conventions), _p(workspace),
        ws_bytes, _stream(stream))
    _check(st, "gdn_prefill_chunked")
    return out, final_state


def gdn_prefill_chunked_checkpoints(q, k, v, alpha, beta, *, B: int, checkpoint_capacity: int,
                                    checkpoint_interval: int = 1, T: Optional[int] = None,
                                    cu_seqlens=None, initial_state=None,
                                    initial_state_indices=None, final_state=None, out=None,
                                    checkpoints=None, chunk: int = 64, scale: float = 1.0,
                                    workspace=None, want_final_state: bool = True,
                                    conventions: int = 0, stream=None):
    """Chunked prefill that also writes the state every checkpoint_interval
    chunks.  Returns (out, final_state, checkpoints [B, capacity, Hv, dv, dk])."""
    T, Hk, dk, Hv, dv = _dims(q, v, B, T, cu_seqlens)
    if out is None:
        out = torch.empty_like(v)
    if final_state is None and want_final_state:
        final_state = torch.empty((B, Hv, dv, dk), dtype=torch.float32, device=v.device)
    cap = int(checkpoint_capacity)
    if checkpoints is None and cap > 0:
        checkpoints = torch.empty((B, cap, Hv, dv, dk), dtype=torch.float32, device=v.device)
    n0 = initial_state.shape[0] if initial_state is not None else 0
    need = gdn_prefill_workspace_size(B, T, Hk, Hv, dk, dv, chunk, q.dtype,
                                      varlen=cu_seqlens is not None)
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=v.device)
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    st = lib().gdn_prefill_chunked_checkpoints(
        _p(q), _p(k), _p(v), _p(alpha), _p(beta), _p(cu_seqlens), _p(initial_state),
        _p(initial_state_indices), n0, _p(final_state), _p(out), B, T, Hk, Hk, Hv,
        dk, dv, chunk, scale, *_codes(q, alpha, conventions), _p(checkpoints), cap,
        int(checkpoint_interval), _p(workspace), ws_bytes, _stream(stream))
    _check(st, "gdn_prefill_chunked_checkpoints")
    return out, final_state, checkpoints


def gdn_prefill_chunked_capture(q, k, v, alpha, beta, *, B: int, state_update_capacity: int,
                                capture_count, T: Optional[int] = None, cu_seqlens=None,
                                initial_state=None, initial_state_indices=None,
                                final_state=None, out=None, state_update_active=None,
                                state_update=None, chunk: int = 64, scale: float = 1.0,
                                workspace=None, want_final_state: bool = True,
                                conventions: int = 0, stream=None):
    """Chunked prefill with the compact capture of gdn_recurrent_capture.
    Returns (out, final_state, state_update)."""
    T, Hk, dk, Hv, dv = _dims(q, v, B, T, cu_seqlens)
    if out is None:
        out = torch.empty_like(v)
    if final_state is None and want_final_state:
        final_state = torch.empty((B, Hv, dv, dk), dtype=torch.float32, device=v.device)
    cap = int(state_update_capacity)
    if cap > 0 and state_update is None:
        state_update = torch.empty((B, cap, slot_width(Hk, Hv, dk, dv)),
                                   dtype=torch.float32, device=v.device)
    n0 = initial_state.shape[0] if initial_state is not None else 0
    need = gdn_prefill_workspace_size(B, T, Hk, Hv, dk, dv, chunk, q.dtype,
                                      varlen=cu_seqlens is not None)
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=v.device)
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    st = lib().gdn_prefill_chunked_capture(
        _p(q), _p(k), _p(v), _p(alpha), _p(beta), _p(cu_seqlens), _p(initial_state),
        _p(initial_state_indices), n0, _p(final_state), _p(out), B, T, Hk, Hk, Hv,
        dk, dv, chunk, scale, *_codes(q, alpha, conventions), cap, _p(capture_count),
        _p(state_update_active), _p(state_update), _p(workspace), ws_bytes, _stream(stream))
    _check(st, "gdn_prefill_chunked_capture")
    return out, final_state, state_update


def gdn_recurrent_capture(q, k, v, alpha, beta, *, B: int, T: Optional[int] = None,
                          cu_seqlens=None, initial_state=None,
                          initial_state_indices=None, final_state=None, out=None,
                          scale: float = 1.0, state_update_capacity: int = 0,
                          capture_count=None, state_update_active=None,
                          state_update=None, want_final_state: bool = True,
                          conventions: int = 0, stream=None):
    """Recurrent path with compact capture.  Returns (out, final_state,
    state_update).  final_state may be initial_state itself (in place)."""
    T, Hk, dk, Hv, dv = _dims(q, v, B, T, cu_seqlens)
    if out is None:
        out = torch.empty_like(v)
    if final_state is None and want_final_state:
        final_state = torch.empty((B, Hv, dv, dk), dtype=torch.float32, device=v.device)
    cap = int(state_update_capacity)
    if cap > 0 and state_update is None:
        state_update = torch.empty((B, cap, slot_width(Hk, Hv, dk, dv)),
                                   dtype=torch.float32, device=v.device)
    n0 = initial_state.shape[0] if initial_state is not None else 0
    st = lib().gdn_recurrent_capture(
        _p(q), _p(k), _p(v), _p(alpha), _p(beta), _p(cu_seqlens), _p(initial_state),
        _p(initial_state_indices), n0, _p(final_state), _p(out), B, T, Hk, Hk, Hv,
        dk, dv, scale, *_codes(q, alpha, conventions), cap, _p(capture_count),
        _p(state_update_active), _p(state_update), _stream(stream))
    _check(st, "gdn_recurrent_capture")
    return out, final_state, state_update


def gdn_replay_state_updates(state_in, state_update, accepted_count, *,
                             state_update_capacity: int, Hk: int,
                             state_out=None, stream=None):
    """Replay the first accepted_count[b] captured slots onto state_in.
    Returns state_out (state_in itself is allowed, in place)."""
    B, Hv, dv, dk = state_in.shape
    if state_out is None:
        state_out = torch.empty_like(state_in)
    st = lib().gdn_replay_state_updates(
        _p(state_in), _p(state_out), _p(state_update), int(state_update_capacity),
        _p(accepted_count), B, int(Hk), Hv, dk, dv, _stream(stream))
    _check(st, "gdn_replay_state_updates")
    return state_out


def gdn_replay_verify(q, k, v, alpha, beta, *, B: int, T: Optional[int] = None,
                      cu_seqlens=None, state_in=None, state_out=None,
                      prev_state_update=None, prev_capacity: int = 0,
                      accepted_count=None, draft_final_state=None, out=None,
                      scale: float = 1.0, state_update_capacity: int = 0,
                      capture_count=None, state_update_active=None,
                      state_update=None, want_draft_final_state: bool = False,
                      conventions: int = 0, stream=None):
    """One speculative step: replay the accepted prefix of prev_state_update
    onto state_in, write it to state_out (state_in itself allowed), then run
    the draft tokens with capture.  Returns (out, state_out, state_update,
    draft_final_state)."""
    T, Hk, dk, Hv, dv = _dims(q, v, B, T, cu_seqlens)
    if out is None:
        out = torch.empty_like(v)
    if state_out is None:
        state_out = torch.empty((B, Hv, dv, dk), dtype=torch.float32, device=v.device)
    if draft_final_state is None and want_draft_final_state:
        draft_final_state = torch.empty((B, Hv, dv, dk), dtype=torch.float32, device=v.device)
    cap = int(state_update_capacity)
    if cap > 0 and state_update is None:
        state_update = torch.empty((B, cap, slot_width(Hk, Hv, dk, dv)),
                                   dtype=torch.float32, device=v.device)
    st = lib().gdn_replay_verify(
        _p(q), _p(k), _p(v), _p(alpha), _p(beta), _p(cu_seqlens), _p(state_in),
        _p(state_out), _p(prev_state_update), int(prev_capacity), _p(accepted_count),
        _p(draft_final_state), _p(out), B, T, Hk, Hk, Hv, dk, dv, scale,
        *_codes(q, alpha, conventions), cap, _p(capture_count),
        _p(state_update_active), _p(state_update), _stream(stream))
    _check(st, "gdn_replay_verify")
    return out, state_out, state_update, draft_final_state


def gdn_set_wait_limit_ns(ns: int) -> None:
    """Testing hook: limit of the kernels' waits on another warp's work, in
    nanoseconds (0 restores the 1 s default; below 1000 gives up at the first
    incomplete check)."""
    lib().gdn_set_wait_limit_ns(int(ns))


def gdn_device_errors(stream=None) -> int:
    """Synchronise the stream and return (and clear) the GDN_DEVERR_* bits."""
    flags = ctypes.c_uint32(0)
    st = lib().gdn_device_errors(_stream(stream), ctypes.byref(flags))
    if st not in (GDN_OK,):
        raise GdnError(st, "gdn_device_errors")
    return int(flags.value)


NOALLOC_SCRATCH_BYTES = 32 * 1024 * 1024


def gdn_prefill_chunked_noalloc(q, k, v, alpha, beta, *, B: int, T: Optional[int] = None,
                                cu_seqlens=None, initial_state=None,
                                initial_state_indices=None, final_state, out,
                                chunk: int = 64, scale: float = 1.0, conventions: int = 0,
                                stream=None):
    """Chunked prefill that allocates nothing: the library's fixed device
    scratch replaces the workspace, and the caller passes `out` and
    `final_state` (None allowed for final_state only if not wanted).  For
    callers that cannot allocate device memory; see include/gdn.h for the size
    limit and the rule that calls must not overlap on the GPU."""
    L = lib()
    fn = L.gdn_prefill_chunked_noalloc
    if fn.restype is not ctypes.c_int or fn.argtypes is None:
        vp, i, f = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
        fn.argtypes = [vp] * 8 + [i, vp, vp] + [i] * 8 + [f, i, i, vp]
        fn.restype = ctypes.c_int
    T, Hk, dk, Hv, dv = _dims(q, v, B, T, cu_seqlens)
    n0 = initial_state.shape[0] if initial_state is not None else 0
    st = fn(_p(q), _p(k), _p(v), _p(alpha), _p(beta), _p(cu_seqlens), _p(initial_state),
            _p(initial_state_indices), n0, _p(final_state), _p(out), B, T, Hk, Hk, Hv, dk, dv,
            chunk, scale, *_codes(q, alpha, conventions), _stream(stream))
    _check(st, "gdn_prefill_chunked_noalloc")
    return out, final_state
