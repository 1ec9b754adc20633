"""fp64 CPU oracle for the gated delta-rule recurrence.

TEST INFRASTRUCTURE ONLY.  Only the tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline / reference arm may import this package.  It shares
no code with the CUDA library and never imports it.

The arithmetic lives in ``gdn_oracle.c`` (plain sequential C, fp64), one
(row, value head) unit per call; this module only builds that file with gcc,
widens inputs to fp64 and walks the units, optionally on a thread pool
(ctypes releases the GIL during each call).  The unrolled-product brute force
for T <= 4 is written here in numpy as a second, independent formulation.

Sources (page title, section):
  * the per-token gated delta rule of Gated DeltaNet (decay, delta, rank-1
    update, readout);
  * "[WebGPU EP] adds state update capacity support for GatedDeltaNet"
    (onnxruntime PR 32767), "Changes": state_update_capacity, the [batch]
    capture_count, the clamped per-row prefix of decay / shared-key / delta
    factors, the replay S = decay * S + outer(key, delta), and
    state_update_active = 0 clearing the whole output;
  * "Enable the native Kev example on NVIDIA GPUs through ExecuTorch's AOTI
    CUDA backend" (executorch issue 23097), work list: chunked prefill with
    explicit initial / final state.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from concurrent.futures import ThreadPoolExecutor

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gdn_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "liboracle.so")
_lib = None
_lock = threading.Lock()

_dp = ctypes.POINTER(ctypes.c_double)


def build(force: bool = False) -> str:
    """Compile gdn_oracle.c into oracle/_build/liboracle.so with gcc."""
    os.makedirs(_BUILD, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    subprocess.check_call(["gcc", "-O2", "-fPIC", "-shared", "-std=c11",
                           "-fno-fast-math", "-ffp-contract=off",
                           _SRC, "-o", tmp, "-lm"])
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            i, l, d = ctypes.c_int, ctypes.c_long, ctypes.c_double
            lib.gdn_oracle_recurrent_unit.argtypes = [
                _dp, _dp, _dp, _dp, _dp, l, i, i, i, i, i, i, d, _dp, _dp, i, _dp]
            lib.gdn_oracle_recurrent_unit.restype = None
            lib.gdn_oracle_replay_unit.argtypes = [_dp, _dp, i, i, i, i, i, i]
            lib.gdn_oracle_replay_unit.restype = None
            lib.gdn_oracle_chunked_unit.argtypes = [
                _dp, _dp, _dp, _dp, _dp, l, i, i, i, i, i, i, d, i, _dp, _dp]
            lib.gdn_oracle_chunked_unit.restype = None
            _lib = lib
    return _lib


def f64(x) -> np.ndarray:
    """Exact widening of a torch tensor or numpy array to C-contiguous fp64."""
    if hasattr(x, "detach"):
        x = x.detach().cpu().double().numpy()
    return np.ascontiguousarray(x, dtype=np.float64)


def _ptr(a: np.ndarray, offset: int = 0):
    assert a.dtype == np.float64 and a.flags.c_contiguous
    return ctypes.cast(a.ctypes.data + 8 * offset, _dp)


def _row_bounds(cu_seqlens, B, T):
    if cu_seqlens is None:
        return [(b * T, T) for b in range(B)]
    cu = [int(x) for x in np.asarray(cu_seqlens).reshape(-1)]
    return [(cu[b], cu[b + 1] - cu[b]) for b in range(B)]


def _run_units(fn, units, threads):
    if threads is None or threads <= 1 or len(units) <= 1:
        for u in units:
            fn(u)
        return
    with ThreadPoolExecutor(max_workers=threads) as ex:
        list(ex.map(fn, units))


def capture_counts_clamped(capture_count, capacity, row_lengths):
    """n_b = clamp(capture_count[b], 0, min(capacity, T_b)): the clamped
    per-row prefix of captured tokens ("Changes" of the onnxruntime PR)."""
    return [max(0, min(int(c), capacity, int(tb)))
            for c, tb in zip(capture_count, row_lengths)]


def recurrent(q, k, v, alpha, beta, *, B, Hk, Hv, dk, dv, T=None,
              cu_seqlens=None, initial_state=None, initial_state_indices=None,
              scale=1.0, capacity=0, capture_count=None, active=True,
              state_update=None, units=None, threads=None):
    """Per-token recurrence for every (row, value head) unit.

    Inputs are widened to fp64.  Returns (o [total_T, Hv, dv],
    final_state [B, Hv, dv, dk], state_update [B, capacity, slot] or None).
    ``units``: optional list of (b, h) to compute (others left as NaN).
    ``state_update``: optional fp64 array pre-filled by the caller (e.g. with
    a sentinel); uncaptured slots are left as given while capture is active.
    When inactive the whole capture output is zero.
    """
    lib = _load()
    q, k, v, alpha, beta = (f64(x) for x in (q, k, v, alpha, beta))
    rows = _row_bounds(cu_seqlens, B, T)
    total_T = rows[-1][0] + rows[-1][1] if rows else 0
    S = _gather_states(initial_state, initial_state_indices, B, Hv, dv, dk)
    o = np.full((total_T, Hv, dv), np.nan)
    slot = Hv + Hk * dk + Hv * dv
    su = None
    n_cap = [0] * B
    if capacity > 0:
        if state_update is None:
            su = np.full((B, capacity, slot), np.nan)
        else:
            su = np.ascontiguousarray(state_update, dtype=np.float64)
        if not active:
            su[...] = 0.0
        else:
            n_cap = capture_counts_clamped(capture_count, capacity,
                                           [tb for _, tb in rows])
    if units is None:
        units = [(b, h) for b in range(B) for h in range(Hv)]

    def one(u):
        b, h = u
        tok0, tb = rows[b]
        Sbh = np.ascontiguousarray(S[b, h])
        cap_ptr = None
        if su is not None and active:
            cap_ptr = _ptr(su, b * capacity * slot)
        lib.gdn_oracle_recurrent_unit(
            _ptr(q), _ptr(k), _ptr(v), _ptr(alpha), _ptr(beta), tok0, tb,
            Hk, Hv, dk, dv, h, float(scale), _ptr(Sbh), _ptr(o), n_cap[b],
            cap_ptr)
        S[b, h] = Sbh

    _run_units(one, units, threads)
    return o, S, su


def chunked(q, k, v, alpha, beta, *, B, Hk, Hv, dk, dv, chunk, T=None,
            cu_seqlens=None, initial_state=None, initial_state_indices=None,
            scale=1.0, units=None, threads=None):
    """Chunked (UT/WY) form of the same recurrence; returns (o, final_state)."""
    lib = _load()
    q, k, v, alpha, beta = (f64(x) for x in (q, k, v, alpha, beta))
    rows = _row_bounds(cu_seqlens, B, T)
    total_T = rows[-1][0] + rows[-1][1] if rows else 0
    S = _gather_states(initial_state, initial_state_indices, B, Hv, dv, dk)
    o = np.full((total_T, Hv, dv), np.nan)
    if units is None:
        units = [(b, h) for b in range(B) for h in range(Hv)]

    def one(u):
        b, h = u
        tok0, tb = rows[b]
        Sbh = np.ascontiguousarray(S[b, h])
        lib.gdn_oracle_chunked_unit(
            _ptr(q), _ptr(k), _ptr(v), _ptr(alpha), _ptr(beta), tok0, tb,
            Hk, Hv, dk, dv, h, float(scale), int(chunk), _ptr(Sbh), _ptr(o))
        S[b, h] = Sbh

    _run_units(one, units, threads)
    return o, S


def replay(state_in, state_update, accepted_count, *, B, Hk, Hv, dk, dv,
           capacity, units=None, threads=None):
    """S <- decay * S + outer(delta, key) for the first m_b slots of row b,
    m_b = clamp(accepted_count[b], 0, capacity).  Returns a new array."""
    lib = _load()
    S = f64(state_in).copy()
    su = f64(state_update)
    slot = Hv + Hk * dk + Hv * dv
    m = [max(0, min(int(a), capacity)) for a in accepted_count]
    if units is None:
        units = [(b, h) for b in range(B) for h in range(Hv)]

    def one(u):
        b, h = u
        Sbh = np.ascontiguousarray(S[b, h])
        lib.gdn_oracle_replay_unit(_ptr(Sbh), _ptr(su, b * capacity * slot),
                                   m[b], Hk, Hv, dk, dv, h)
        S[b, h] = Sbh

    _run_units(one, units, threads)
    return S


def prefix_checkpoints(q, k, v, alpha, beta, *, B, Hk, Hv, dk, dv, every, capacity,
                       T=None, cu_seqlens=None, initial_state=None,
                       initial_state_indices=None, scale=1.0, heads=None, threads=None):
    """State of row b after (j + 1) * every tokens, for
    j < min(capacity, floor(T_b / every)): snapshots of growing prefixes of
    each row ("Enable the native Kev example on the WebGPU backend",
    executorch issue 23099: an immutable prefix snapshot reused later), kept
    at every boundary.  Each is the recurrence (``recurrent``) run over that
    prefix, continued segment by segment from the previous snapshot.
    ``heads``: optional value heads to compute (others NaN).  Returns
    [B, capacity, Hv, dv, dk] with NaN in slots that are not defined."""
    rows = _row_bounds(cu_seqlens, B, T)
    S = _gather_states(initial_state, initial_state_indices, B, Hv, dv, dk)
    out = np.full((B, capacity, Hv, dv, dk), np.nan)
    hs = range(Hv) if heads is None else heads
    for b, (tok0, tb) in enumerate(rows):
        Sb = S[b:b + 1]
        for j in range(min(capacity, tb // every)):
            seg = slice(tok0 + j * every, tok0 + (j + 1) * every)
            _, Sb, _ = recurrent(q[seg], k[seg], v[seg], alpha[seg], beta[seg], B=1,
                                 Hk=Hk, Hv=Hv, dk=dk, dv=dv, T=every, initial_state=Sb,
                                 scale=scale, units=[(0, h) for h in hs],
                                 threads=threads)
            out[b, j, list(hs)] = Sb[0, list(hs)]
    return out


def replay_verify(q, k, v, alpha, beta, *, B, Hk, Hv, dk, dv, T=None,
                  cu_seqlens=None, state_in=None, prev_state_update=None,
                  prev_capacity=0, accepted_count=None, scale=1.0, capacity=0,
                  capture_count=None, active=True, state_update=None,
                  units=None, threads=None):
    """One speculative-decoding step: replay the accepted prefix of the
    previous capture, then run the draft tokens with capture ("[WebGPU EP]
    adds state update capacity support for GatedDeltaNet", onnxruntime PR
    32767, "DFlash2 Prerequisite": replay after partial acceptance, state and
    output matching the non-speculative run).  Written as what it is, the
    replay of ``replay`` followed by the recurrence of ``recurrent``.

    Returns (o, committed_state, draft_final_state, state_update)."""
    if state_in is None:
        S = np.zeros((B, Hv, dv, dk))
    else:
        S = f64(state_in).copy()
    if prev_capacity > 0:
        S = replay(S, prev_state_update, accepted_count, B=B, Hk=Hk, Hv=Hv,
                   dk=dk, dv=dv, capacity=prev_capacity, units=units,
                   threads=threads)
    o, S_final, su = recurrent(q, k, v, alpha, beta, B=B, Hk=Hk, Hv=Hv, dk=dk,
                               dv=dv, T=T, cu_seqlens=cu_seqlens,
                               initial_state=S, scale=scale, capacity=capacity,
                               capture_count=capture_count, active=active,
                               state_update=state_update, units=units,
                               threads=threads)
    return o, S, S_final, su


def front_end(q, k, alpha, beta, *, qk_l2norm=False, alpha_log=False,
              beta_logit=False, eps=1e-6):
    """The layer's input conventions ("adapting layouts, gate/scaling
    conventions", executorch issue 23097, work list), applied in fp64 to
    give the recurrence's own inputs: with ``qk_l2norm`` q and k are
    L2-normalised per head, x / sqrt(sum x^2 + eps); with ``alpha_log``
    alpha holds the log-decay g and the decay is e^g; with ``beta_logit``
    beta holds logits and the write strength is 1 / (1 + e^-x).  Returns
    (q, k, alpha, beta) in fp64."""
    q, k, alpha, beta = (f64(x) for x in (q, k, alpha, beta))
    if qk_l2norm:
        q = q / np.sqrt(np.sum(q * q, axis=-1, keepdims=True) + eps)
        k = k / np.sqrt(np.sum(k * k, axis=-1, keepdims=True) + eps)
    if alpha_log:
        alpha = np.exp(alpha)
    if beta_logit:
        beta = 1.0 / (1.0 + np.exp(-beta))
    return q, k, alpha, beta


def _gather_states(initial_state, indices, B, Hv, dv, dk):
    if initial_state is None:
        return np.zeros((B, Hv, dv, dk))
    s0 = f64(initial_state)
    if indices is None:
        return s0[:B].copy()
    idx = [int(i) for i in np.asarray(indices).reshape(-1)]
    return np.stack([s0[i] for i in idx]).copy()


def bruteforce_unrolled(q, k, v, alpha, beta, S0, *, scale=1.0):
    """Unrolled-product form for one unit and a handful of tokens (T <= 4).

    q, k: [T, dk]; v: [T, dv]; alpha, beta: [T]; S0: [dv, dk].  Each token is
    the affine map S -> S M_t + beta_t v_t k_t^T with the dk x dk matrix
    M_t = alpha_t (I - beta_t k_t k_t^T), so
      S_T = S0 M_1...M_T + sum_t beta_t v_t k_t^T M_{t+1}...M_T,
    built here from explicit matrix products; o_t = S_t (scale q_t).
    """
    q, k, v, alpha, beta, S0 = (f64(x) for x in (q, k, v, alpha, beta, S0))
    T, dk = k.shape
    assert T <= 4, "brute force is for tiny cases only"
    I = np.eye(dk)
    M = [alpha[t] * (I - beta[t] * np.outer(k[t], k[t])) for t in range(T)]
    outs, S_t = [], None
    for t_end in range(1, T + 1):
        P = I.copy()
        for t in range(t_end):
            P = P @ M[t]
        S_t = S0 @ P
        for t in range(t_end):
            tail = I.copy()
            for s in range(t + 1, t_end):
                tail = tail @ M[s]
            S_t = S_t + beta[t] * np.outer(v[t], k[t]) @ tail
        outs.append(S_t @ (scale * q[t_end - 1]))
    return np.stack(outs), S_t
