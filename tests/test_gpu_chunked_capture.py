"""GPU parity of gdn_prefill_chunked_capture -- the chunked prefill emitting
the compact state-update capture of the recurrent path -- against the fp64
oracle's recurrent capture, on both prefill kernels.

Source: "[WebGPU EP] adds state update capacity support for GatedDeltaNet"
(onnxruntime PR 32767), "Changes" (clamped per-row prefix of decay /
shared-key / delta factors; state_update_active = 0 clears the output) and
"Test Coverage" (compare only captured ranges; ragged capacity-7 cases with
zero, partial and full counts; the fp16 Hq=2 / Hv=6 / 128 case).

Decay and key are exact widenings of the inputs and compare bit for bit.
The deltas are an intermediate of the chunked form with that path's
accuracy, so they are held to the path's tolerance (2e-4 relative for fp32
inputs, 2e-2 for 16-bit inputs on the tensor-core path).
"""
import os

import numpy as np
import pytest
import torch

from helpers import TOL, Guarded, rel

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


def _dev(x):
    return {n: getattr(x, n).cuda() for n in ("q", "k", "v", "alpha", "beta")}


def _acc(vals):
    return torch.tensor(vals, dtype=torch.int32, device="cuda")


def _check(su: Guarded, ref, counts, x, cap, tol):
    n = [max(0, min(int(c), cap, L)) for c, L in zip(counts, x.lengths)]
    off = x.Hv + x.Hk * x.dk
    for b, nb in enumerate(n):
        if nb > 0:
            g = su.t[b, :nb].cpu().double().numpy()
            assert np.array_equal(g[:, :off], ref[b, :nb, :off]), b
            assert rel(su.t[b, :nb, off:], ref[b, :nb, off:]) < tol, b
        if nb < cap:
            assert bool(torch.all(su.untouched((b, slice(nb, cap)))).item()), b
    assert su.guards_intact()
    return n


def _run(gdn, oracle_mod, x, counts, cap, chunk, active=1, uniform=False):
    g = _dev(x)
    B = x.B
    slot = gdn.slot_width(x.Hk, x.Hv, x.dk, x.dv)
    su = Guarded((B, cap, slot), F32)
    S0 = x.initial_state.cuda() if x.initial_state is not None else None
    rows = dict(T=x.uniform_T) if uniform else dict(cu_seqlens=x.cu_seqlens.cuda())
    out, fs, _ = gdn.gdn_prefill_chunked_capture(
        g["q"], g["k"], g["v"], g["alpha"], g["beta"], B=B, initial_state=S0, chunk=chunk,
        state_update_capacity=cap, capture_count=_acc(counts),
        state_update_active=_acc([active]), state_update=su.t, **rows)
    out0, fs0 = gdn.gdn_prefill_chunked(g["q"], g["k"], g["v"], g["alpha"], g["beta"], B=B,
                                        initial_state=S0, chunk=chunk, **rows)
    torch.cuda.synchronize()
    # the capture is extra writes only
    assert torch.equal(out, out0) and torch.equal(fs, fs0)
    _, _, ref = oracle_mod.recurrent(x.q, x.k, x.v, x.alpha, x.beta, B=B, Hk=x.Hk, Hv=x.Hv,
                                     dk=x.dk, dv=x.dv, cu_seqlens=x.cu_seqlens,
                                     initial_state=x.initial_state, capacity=cap,
                                     capture_count=counts, active=bool(active),
                                     threads=THREADS)
    return su, ref


def test_tiny_f32_cuda_core_path(gdn, oracle_mod):
    from gated_deltanet_recurrence_02_gb300.inputs import WORKLOADS, make_inputs
    w = WORKLOADS["tiny_f32"]
    x = make_inputs(w["seed"], lengths=w["lengths"], Hk=w["Hk"], Hv=w["Hv"], dk=w["dk"],
                    dv=w["dv"], dtype_qkv="f32", dtype_gate="f32")
    su, ref = _run(gdn, oracle_mod, x, w["capture_count"], w["capacity"], w["chunk"],
                   uniform=True)
    assert _check(su, ref, w["capture_count"], x, w["capacity"], TOL[F32]) == [3, 7]


@pytest.mark.parametrize("chunk", [64, 16])
@pytest.mark.parametrize("active", [1, 0])
def test_qwenlike_f16_both_paths(gdn, oracle_mod, chunk, active):
    """chunk 64: tensor-core path (d=128, fp16); chunk 16: CUDA-core path."""
    from gated_deltanet_recurrence_02_gb300.inputs import WORKLOADS, make_inputs
    w = WORKLOADS["ragged_capture_qwenlike_f16"]
    x = make_inputs(w["seed"], lengths=w["lengths"], Hk=w["Hk"], Hv=w["Hv"], dk=w["dk"],
                    dv=w["dv"], dtype_qkv=w["dtype_qkv"], dtype_gate=w["dtype_gate"])
    su, ref = _run(gdn, oracle_mod, x, w["capture_count"], w["capacity"], chunk, active=active,
                   uniform=True)
    if active:
        tol = TOL[torch.float16] if chunk == 64 else TOL[F32]
        assert _check(su, ref, w["capture_count"], x, w["capacity"], tol) == [0, 4, 7]
    else:
        assert bool(torch.all(su.t == 0).item()) and su.guards_intact()


def test_bf16_tensor_core_capture_across_chunks_then_replay(gdn, oracle_mod):
    """Ragged rows with captures reaching past the first 64-token chunk; the
    replay of each row's captured prefix rebuilds the oracle's state after
    that many tokens (the verify-then-replay use of the capture)."""
    from gated_deltanet_recurrence_02_gb300.inputs import make_inputs
    lengths, counts, cap = [150, 64, 90, 30], [100, 64, 80, 5], 100
    x = make_inputs(1300, lengths=lengths, Hk=2, Hv=4, dk=128, dv=128, dtype_qkv="bf16",
                    dtype_gate="bf16")
    su, ref = _run(gdn, oracle_mod, x, counts, cap, 64)
    n = _check(su, ref, counts, x, cap, TOL[torch.bfloat16])
    assert n == [100, 64, 80, 5]
    acc = [97, 64, 33, 5]
    S = gdn.gdn_replay_state_updates(x.initial_state.cuda(), su.t, _acc(acc),
                                     state_update_capacity=cap, Hk=x.Hk)
    torch.cuda.synchronize()
    for b, m in enumerate(acc):
        t0 = int(x.cu_seqlens[b])
        sl = slice(t0, t0 + m)
        _, Sm, _ = oracle_mod.recurrent(x.q[sl], x.k[sl], x.v[sl], x.alpha[sl], x.beta[sl], B=1,
                                        Hk=x.Hk, Hv=x.Hv, dk=x.dk, dv=x.dv, T=m,
                                        initial_state=x.initial_state[b:b + 1])
        assert rel(S[b], Sm[0]) < TOL[torch.bfloat16], b
