"""GPU parity of the tensor-core prefill's wide carry tiles.

The carry phase runs on 32-row state tiles while one wave of them fits the
GPU and on 128-row tiles (64-row ones when dv = 64) for more (row, value
head) pairs.  These cases have 4 Hv B > the SM count, so every call below
takes a wide instance (128 rows at d = 128): plain, with capture, with
checkpoints and with the in-kernel input conventions, against the fp64
oracle.

Sources: the chunked form of the gated delta rule (the prefill path of
"Enable the native Kev example on NVIDIA GPUs through ExecuTorch's AOTI CUDA
backend", executorch issue 23097, "Work to cover"); "[WebGPU EP] adds state
update capacity support for GatedDeltaNet" (onnxruntime PR 32767),
"Changes" (the capture contract); "Enable the native Kev example on the
WebGPU backend" (executorch issue 23099): prefix snapshots, here kept at
chunk boundaries.
"""
import os

import numpy as np
import pytest
import torch

from helpers import TOL, Guarded, rel

pytestmark = pytest.mark.gpu
THREADS = min(32, os.cpu_count() or 4)
F32 = torch.float32
LENGTHS = [150, 64, 37, 200, 90, 129]
HK, HV, D, C = 2, 8, 128, 64


@pytest.fixture(scope="module")
def gdn():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from gated_deltanet_recurrence_02_gb300 import build, gdn as g
    build.build()
    g.lib()
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    if 4 * HV * len(LENGTHS) <= sms:
        pytest.skip("the 64-row carry instance needs more (row, head) tiles than SMs")
    return g


@pytest.fixture(scope="module")
def case():
    from gated_deltanet_recurrence_02_gb300.inputs import make_inputs
    return make_inputs(2500, lengths=LENGTHS, Hk=HK, Hv=HV, dk=D, dv=D, dtype_qkv="bf16",
                       dtype_gate="bf16")


def _dev(x):
    return {n: getattr(x, n).cuda() for n in ("q", "k", "v", "alpha", "beta")}


def test_plain_and_capture(gdn, oracle_mod, case):
    x = case
    B, cap = len(LENGTHS), 70
    counts = [70, 10, 37, 0, 64, 129]
    g = _dev(x)
    cu, S0 = x.cu_seqlens.cuda(), x.initial_state.cuda()
    out, fs = gdn.gdn_prefill_chunked(g["q"], g["k"], g["v"], g["alpha"], g["beta"], B=B,
                                      cu_seqlens=cu, initial_state=S0, chunk=C)
    su = Guarded((B, cap, gdn.slot_width(HK, HV, D, D)), F32)
    out2, fs2, _ = gdn.gdn_prefill_chunked_capture(
        g["q"], g["k"], g["v"], g["alpha"], g["beta"], B=B, cu_seqlens=cu, initial_state=S0,
        chunk=C, state_update_capacity=cap,
        capture_count=torch.tensor(counts, dtype=torch.int32, device="cuda"), state_update=su.t)
    torch.cuda.synchronize()
    ro, rS, rsu = oracle_mod.recurrent(x.q, x.k, x.v, x.alpha, x.beta, B=B, Hk=HK, Hv=HV, dk=D,
                                       dv=D, cu_seqlens=x.cu_seqlens,
                                       initial_state=x.initial_state, capacity=cap,
                                       capture_count=counts, threads=THREADS)
    tol = TOL[torch.bfloat16]
    cuh = x.cu_seqlens.tolist()
    for b in range(B):
        sl = slice(cuh[b], cuh[b + 1])
        assert rel(out[sl], ro[sl]) < tol, b
        assert rel(fs[b], rS[b]) < tol, b
    # the capture variant computes the same outputs; the deltas it stores
    # are the chunked form's, to the path's tolerance
    assert torch.equal(out, out2) and torch.equal(fs, fs2)
    off = HV + HK * D
    for b, nb in enumerate(min(c, cap, L) for c, L in zip(counts, LENGTHS)):
        if nb > 0:
            gsu = su.t[b, :nb].cpu().double().numpy()
            assert np.array_equal(gsu[:, :off], rsu[b, :nb, :off]), b
            assert rel(su.t[b, :nb, off:], rsu[b, :nb, off:]) < tol, b
        if nb < cap:
            assert bool(torch.all(su.untouched((b, slice(nb, cap)))).item()), b
    assert su.guards_intact()


def test_checkpoints(gdn, oracle_mod, case):
    x = case
    B, cap = len(LENGTHS), 3
    g = _dev(x)
    cu, S0 = x.cu_seqlens.cuda(), x.initial_state.cuda()
    ck = Guarded((B, cap, HV, D, D), F32)
    out, fs, _ = gdn.gdn_prefill_chunked_checkpoints(
        g["q"], g["k"], g["v"], g["alpha"], g["beta"], B=B, cu_seqlens=cu, initial_state=S0,
        checkpoints=ck.t, checkpoint_capacity=cap, checkpoint_interval=1, chunk=C)
    torch.cuda.synchronize()
    ref = oracle_mod.prefix_checkpoints(x.q, x.k, x.v, x.alpha, x.beta, B=B, Hk=HK, Hv=HV,
                                        dk=D, dv=D, every=C, capacity=cap,
                                        cu_seqlens=x.cu_seqlens, initial_state=x.initial_state,
                                        threads=THREADS)
    for b, tb in enumerate(LENGTHS):
        n = min(cap, tb // C)
        for j in range(n):
            assert rel(ck.t[b, j], ref[b, j]) < TOL[torch.bfloat16], (b, j)
        if n < cap:
            assert bool(torch.all(ck.untouched((b, slice(n, cap)))).item()), b
    assert ck.guards_intact()


def test_conventions(gdn, oracle_mod):
    from gated_deltanet_recurrence_02_gb300.inputs import make_raw_inputs
    x = make_raw_inputs(2501, lengths=LENGTHS, Hk=HK, Hv=HV, dk=D, dv=D, dtype_qkv="bf16",
                        dtype_gate="bf16")
    B = len(LENGTHS)
    g = _dev(x)
    out, fs = gdn.gdn_prefill_chunked(g["q"], g["k"], g["v"], g["alpha"], g["beta"], B=B,
                                      cu_seqlens=x.cu_seqlens.cuda(),
                                      initial_state=x.initial_state.cuda(), scale=x.scale,
                                      chunk=C, conventions=0x700)
    torch.cuda.synchronize()
    rq, rk, ra, rb = oracle_mod.front_end(x.q, x.k, x.alpha, x.beta, qk_l2norm=True,
                                          alpha_log=True, beta_logit=True)
    ro, rS, _ = oracle_mod.recurrent(rq, rk, x.v, ra, rb, B=B, Hk=HK, Hv=HV, dk=D, dv=D,
                                     cu_seqlens=x.cu_seqlens, initial_state=x.initial_state,
                                     scale=x.scale, threads=THREADS)
    assert rel(out, ro) < TOL[torch.bfloat16]
    assert rel(fs, rS) < TOL[torch.bfloat16]


def test_prefill_batch_B64_sampled_units(gdn, oracle_mod):
    """The benchmark's packed batch (64 rows of 500..1500 tokens, 64.7k in
    all, the 64-row carry instance) at full size: sampled (row, head) units
    against the oracle run on those rows alone (rows are independent)."""
    from gated_deltanet_recurrence_02_gb300.inputs import WORKLOADS, make_inputs, ragged_lengths
    w = WORKLOADS["prefill_batch_B64"]
    lengths = ragged_lengths(w["seed"], w["B"], w["lo"], w["hi"])
    dims = dict(Hk=w["Hk"], Hv=w["Hv"], dk=w["dk"], dv=w["dv"])
    x = make_inputs(w["seed"] + 1, lengths=lengths, dtype_qkv=w["dtype_qkv"],
                    dtype_gate=w["dtype_gate"], **dims)
    B = w["B"]
    g = {n: getattr(x, n).cuda() for n in ("q", "k", "v", "alpha", "beta", "initial_state")}
    out, fs = gdn.gdn_prefill_chunked(g["q"], g["k"], g["v"], g["alpha"], g["beta"], B=B,
                                      cu_seqlens=x.cu_seqlens.cuda(),
                                      initial_state=g["initial_state"], chunk=w["chunk"])
    torch.cuda.synchronize()
    out, fs = out.cpu(), fs.cpu()
    del g
    rows = sorted({0, 17, B - 1, int(np.argmin(lengths)), int(np.argmax(lengths))})
    heads = [0, 13, w["Hv"] - 1]
    cu = x.cu_seqlens.tolist()
    tol = TOL[torch.bfloat16]
    for b in rows:
        sl = slice(cu[b], cu[b + 1])
        ro, rS, _ = oracle_mod.recurrent(x.q[sl], x.k[sl], x.v[sl], x.alpha[sl], x.beta[sl], B=1,
                                         T=lengths[b], initial_state=x.initial_state[b:b + 1],
                                         units=[(0, hh) for hh in heads], threads=THREADS, **dims)
        for hh in heads:
            assert rel(out[sl, hh], ro[:, hh]) < tol, (b, hh)
            assert rel(fs[b, hh], rS[0, hh]) < tol, (b, hh)


@pytest.mark.parametrize("Hv", [4, 32])
def test_empty_rows_tensor_core_path(gdn, oracle_mod, Hv):
    """Rows of length 0 next to ragged ones on the tensor-core prefill (both
    carry instances: Hv = 4 takes the 32-row tiles, Hv = 32 the 64-row ones),
    and a call whose rows are all empty: every empty row keeps its initial
    state bit for bit, the others match the oracle."""
    from gated_deltanet_recurrence_02_gb300.inputs import make_inputs
    for lengths in ([0, 70, 0, 1, 129, 0], [0, 0]):
        x = make_inputs(2600 + Hv + len(lengths), lengths=lengths, Hk=2, Hv=Hv, dk=D, dv=D,
                        dtype_qkv="bf16", dtype_gate="bf16")
        B = len(lengths)
        g = _dev(x)
        S0 = x.initial_state.cuda()
        out, fs = gdn.gdn_prefill_chunked(g["q"], g["k"], g["v"], g["alpha"], g["beta"], B=B,
                                          cu_seqlens=x.cu_seqlens.cuda(), initial_state=S0,
                                          chunk=C)
        torch.cuda.synchronize()
        assert gdn.gdn_device_errors() == 0
        for b, L in enumerate(lengths):
            if L == 0:
                assert torch.equal(fs[b], S0[b]), b
        if sum(lengths) == 0:
            continue
        ro, rS, _ = oracle_mod.recurrent(x.q, x.k, x.v, x.alpha, x.beta, B=B, Hk=2, Hv=Hv,
                                         dk=D, dv=D, cu_seqlens=x.cu_seqlens,
                                         initial_state=x.initial_state, threads=THREADS)
        assert rel(out, ro) < TOL[torch.bfloat16]
        assert rel(fs, rS) < TOL[torch.bfloat16]
