"""GPU parity of the in-kernel input conventions (GDN_QK_L2NORM,
GDN_ALPHA_LOG, GDN_BETA_LOGIT) on every path, against the fp64 oracle
applied to the same raw inputs through its front end.

Source: "Enable the native Kev example on NVIDIA GPUs through ExecuTorch's
AOTI CUDA backend" (executorch issue 23097), work list: reuse the GDN prefill
kernel, adapting layouts and gate/scaling conventions.  The capture stores the
factors the recurrence used (the decay e^g and the normalised key); those are
computed in fp32 here, so they compare to 1e-6 rather than bit for bit.
"""
import os

import numpy as np
import pytest
import torch

from helpers import TOL, TOL_CAPTURE, rel

pytestmark = pytest.mark.gpu
THREADS = min(32, os.cpu_count() or 4)
F32 = torch.float32


@pytest.fixture(scope="module")
def gdn():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from gated_deltanet_recurrence_02_gb300 import build, gdn as g
    build.build()
    g.lib()
    return g


def _acc(vals):
    return torch.tensor(vals, dtype=torch.int32, device="cuda")


CASES = {
    # path: (lengths, Hk, Hv, d, dtype, chunk, capacity, counts)
    "decode": ([1] * 48, 2, 4, 128, "bf16", None, 1, [1, 0] * 24),
    "recurrent": ([5, 9, 1], 2, 6, 128, "f16", None, 4, [4, 2, 3]),
    "cuda_core_prefill": ([40, 7, 64], 1, 2, 32, "f32", 16, 0, None),
    "tensor_core_prefill": ([150, 64, 30], 2, 4, 128, "bf16", 64, 70, [70, 64, 30]),
}


@pytest.mark.parametrize("path,conv", [
    ("decode", 0x700), ("recurrent", 0x700), ("cuda_core_prefill", 0x700),
    ("tensor_core_prefill", 0x100), ("tensor_core_prefill", 0x200),
    ("tensor_core_prefill", 0x400), ("tensor_core_prefill", 0x700),
])
def test_conventions(gdn, oracle_mod, path, conv):
    from gated_deltanet_recurrence_02_gb300.inputs import make_raw_inputs
    lengths, Hk, Hv, d, dt, chunk, cap, counts = CASES[path]
    x = make_raw_inputs(1500 + conv, lengths=lengths, Hk=Hk, Hv=Hv, dk=d, dv=d, dtype_qkv=dt,
                        dtype_gate=dt)
    # q/k already normalised when GDN_QK_L2NORM is off; alpha a decay, beta in (0, 1)
    # when their flags are off: convert the raw draw on the host, exactly as
    # the oracle's front end would, and store it in the same dtype
    qk, alog, blog = bool(conv & 0x100), bool(conv & 0x200), bool(conv & 0x400)
    pre = [not qk, not alog, not blog]
    q, k, a, b = x.q, x.k, x.alpha, x.beta
    if any(pre):
        fq, fk, fa, fb = oracle_mod.front_end(q, k, a, b, qk_l2norm=pre[0], alpha_log=pre[1],
                                              beta_logit=pre[2])
        to = lambda arr, like: torch.from_numpy(np.asarray(arr, np.float32)).to(like.dtype)  # noqa: E731
        q, k, a, b = to(fq, q), to(fk, k), to(fa, a), to(fb, b)
    g = {n: t.cuda() for n, t in zip(("q", "k", "alpha", "beta"), (q, k, a, b))}
    g["v"] = x.v.cuda()
    B, sc = len(lengths), x.scale
    S0 = x.initial_state.cuda()
    cc = _acc(counts) if cap else None
    if path == "decode":
        out, fs, su = gdn.gdn_recurrent_capture(g["q"], g["k"], g["v"], g["alpha"], g["beta"], B=B,
                                                T=1, initial_state=S0, scale=sc,
                                                state_update_capacity=cap, capture_count=cc,
                                                conventions=conv)
    elif path == "recurrent":
        out, fs, su = gdn.gdn_recurrent_capture(g["q"], g["k"], g["v"], g["alpha"], g["beta"], B=B,
                                                cu_seqlens=x.cu_seqlens.cuda(), initial_state=S0,
                                                scale=sc, state_update_capacity=cap,
                                                capture_count=cc, conventions=conv)
    elif cap:
        out, fs, su = gdn.gdn_prefill_chunked_capture(
            g["q"], g["k"], g["v"], g["alpha"], g["beta"], B=B, cu_seqlens=x.cu_seqlens.cuda(),
            initial_state=S0, scale=sc, chunk=chunk, state_update_capacity=cap,
            capture_count=cc, conventions=conv)
    else:
        out, fs = gdn.gdn_prefill_chunked(g["q"], g["k"], g["v"], g["alpha"], g["beta"], B=B,
                                          cu_seqlens=x.cu_seqlens.cuda(), initial_state=S0,
                                          scale=sc, chunk=chunk, conventions=conv)
        su = None
    torch.cuda.synchronize()
    rq, rk, ra, rb = oracle_mod.front_end(q, k, a, b, qk_l2norm=qk, alpha_log=alog,
                                          beta_logit=blog)
    ro, rS, rsu = oracle_mod.recurrent(rq, rk, x.v, ra, rb, B=B, Hk=Hk, Hv=Hv, dk=d, dv=d,
                                       cu_seqlens=x.cu_seqlens, initial_state=x.initial_state,
                                       scale=sc, capacity=cap, capture_count=counts,
                                       threads=THREADS)
    tol = TOL[x.q.dtype]
    assert rel(out, ro) < tol
    assert rel(fs, rS) < tol
    if su is not None:
        off = Hv + Hk * d
        dtol = TOL_CAPTURE if path in ("decode", "recurrent") else tol
        for r, nb in enumerate(min(c, cap, L) for c, L in zip(counts, lengths)):
            if nb == 0:
                continue
            assert rel(su[r, :nb, :Hv], rsu[r, :nb, :Hv]) < 1e-6, r
            assert rel(su[r, :nb, Hv:off], rsu[r, :nb, Hv:off]) < 1e-6, r
            assert rel(su[r, :nb, off:], rsu[r, :nb, off:]) < dtol, r


def test_conventions_fused_replay_verify(gdn, oracle_mod):
    """The fused speculative step with every convention on: the replayed
    factors are the stored (converted) ones; the drafts go through the front
    end in the kernel."""
    from gated_deltanet_recurrence_02_gb300.inputs import make_raw_inputs
    Hk, Hv, d, cap, B, T = 2, 4, 128, 4, 3, 4
    x1 = make_raw_inputs(1600, lengths=[T] * B, Hk=Hk, Hv=Hv, dk=d, dv=d, dtype_qkv="bf16",
                         dtype_gate="bf16")
    x2 = make_raw_inputs(1601, lengths=[T] * B, Hk=Hk, Hv=Hv, dk=d, dv=d, dtype_qkv="bf16",
                         dtype_gate="bf16", zero_state=True)
    flags = dict(qk_l2norm=True, alpha_log=True, beta_logit=True)
    # previous verify pass: the oracle's capture of x1's drafts (converted factors), as fp32
    q1, k1, a1, b1 = oracle_mod.front_end(x1.q, x1.k, x1.alpha, x1.beta, **flags)
    _, _, su1 = oracle_mod.recurrent(q1, k1, x1.v, a1, b1, B=B, Hk=Hk, Hv=Hv, dk=d, dv=d, T=T,
                                     initial_state=x1.initial_state, scale=x1.scale,
                                     capacity=cap, capture_count=[cap] * B)
    su1 = torch.from_numpy(su1.astype(np.float32))
    accepted = [0, 2, 4]
    g = {n: getattr(x2, n).cuda() for n in ("q", "k", "v", "alpha", "beta")}
    out, Sc, su2, _ = gdn.gdn_replay_verify(g["q"], g["k"], g["v"], g["alpha"], g["beta"], B=B,
                                            T=T, state_in=x1.initial_state.cuda(),
                                            prev_state_update=su1.cuda(), prev_capacity=cap,
                                            accepted_count=_acc(accepted), scale=x2.scale,
                                            state_update_capacity=cap,
                                            capture_count=_acc([cap] * B), conventions=0x700)
    torch.cuda.synchronize()
    q2, k2, a2, b2 = oracle_mod.front_end(x2.q, x2.k, x2.alpha, x2.beta, **flags)
    ro, rSc, _, rsu = oracle_mod.replay_verify(
        q2, k2, x2.v, a2, b2, B=B, Hk=Hk, Hv=Hv, dk=d, dv=d, T=T, state_in=x1.initial_state,
        prev_state_update=su1, prev_capacity=cap, accepted_count=accepted, scale=x2.scale,
        capacity=cap, capture_count=[cap] * B)
    tol = TOL[torch.bfloat16]
    assert rel(Sc, rSc) < tol
    assert rel(out, ro) < tol
    off = Hv + Hk * d
    assert rel(su2[:, :, :off], rsu[:, :, :off]) < 1e-6
    assert rel(su2[:, :, off:], rsu[:, :, off:]) < TOL_CAPTURE
