"""GPU parity of gdn_prefill_chunked_checkpoints -- the chunked prefill that
also writes the state at chunk boundaries -- against the fp64 oracle, on
both prefill kernels (CUDA-core: fp32, d=32, chunk 16; tensor-core: bf16,
d=128, chunk 64; smaller heads on the tensor-core path are covered in
test_gpu_tc_head_sizes.py).

Source: "Enable the native Kev example on the WebGPU backend" (executorch
issue 23099): an immutable prefix snapshot reused later; here a snapshot is
kept every L tokens so that a prefix can be resumed at any such offset.
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


def _check_slots(ck: Guarded, ref, lengths, L, cap, tol, heads=None):
    """Slots j < min(cap, T_b // L) against the oracle; later slots untouched."""
    for b, tb in enumerate(lengths):
        n = min(cap, tb // L)
        for j in range(n):
            hs = list(range(ref.shape[2])) if heads is None else heads
            assert rel(ck.t[b, j, hs], ref[b, j, hs]) < tol, (b, j)
        if n < cap:
            assert bool(torch.all(ck.untouched((b, slice(n, cap)))).item()), b
    assert ck.guards_intact()


@pytest.mark.parametrize("interval", [1, 2])
def test_ragged_f32_cuda_core_path(gdn, oracle_mod, interval):
    from gated_deltanet_recurrence_02_gb300.inputs import make_inputs
    lengths, Hk, Hv, d, C, cap = [40, 7, 64], 1, 2, 32, 16, 3
    x = make_inputs(1200, lengths=lengths, Hk=Hk, Hv=Hv, dk=d, dv=d, dtype_qkv="f32",
                    dtype_gate="f32")
    g = _dev(x)
    B, L = len(lengths), interval * C
    cu = x.cu_seqlens.cuda()
    S0 = x.initial_state.cuda()
    ck = Guarded((B, cap, Hv, d, d), F32)
    out, fs, _ = gdn.gdn_prefill_chunked_checkpoints(
        g["q"], g["k"], g["v"], g["alpha"], g["beta"], B=B, cu_seqlens=cu, initial_state=S0,
        checkpoints=ck.t, checkpoint_capacity=cap, checkpoint_interval=interval, chunk=C)
    out0, fs0 = gdn.gdn_prefill_chunked(g["q"], g["k"], g["v"], g["alpha"], g["beta"], B=B,
                                        cu_seqlens=cu, initial_state=S0, chunk=C)
    torch.cuda.synchronize()
    ref = oracle_mod.prefix_checkpoints(x.q, x.k, x.v, x.alpha, x.beta, B=B, Hk=Hk, Hv=Hv,
                                        dk=d, dv=d, every=L, capacity=cap,
                                        cu_seqlens=x.cu_seqlens, initial_state=x.initial_state)
    _check_slots(ck, ref, lengths, L, cap, TOL[F32])
    # the checkpoints are extra writes only
    assert torch.equal(out, out0) and torch.equal(fs, fs0)


@pytest.mark.parametrize("interval", [1, 3])
def test_ragged_bf16_tensor_core_path(gdn, oracle_mod, interval):
    from gated_deltanet_recurrence_02_gb300.inputs import make_inputs
    lengths, Hk, Hv, d, C, cap = [200, 64, 130, 50], 2, 4, 128, 64, 3
    x = make_inputs(1201, lengths=lengths, Hk=Hk, Hv=Hv, dk=d, dv=d, dtype_qkv="bf16",
                    dtype_gate="bf16")
    g = _dev(x)
    B = len(lengths)
    cu = x.cu_seqlens.cuda()
    S0 = x.initial_state.cuda()
    ck = Guarded((B, cap, Hv, d, d), F32)
    out, fs, _ = gdn.gdn_prefill_chunked_checkpoints(
        g["q"], g["k"], g["v"], g["alpha"], g["beta"], B=B, cu_seqlens=cu, initial_state=S0,
        checkpoints=ck.t, checkpoint_capacity=cap, checkpoint_interval=interval, chunk=C)
    out0, fs0 = gdn.gdn_prefill_chunked(g["q"], g["k"], g["v"], g["alpha"], g["beta"], B=B,
                                        cu_seqlens=cu, initial_state=S0, chunk=C)
    torch.cuda.synchronize()
    L = interval * C
    ref = oracle_mod.prefix_checkpoints(x.q, x.k, x.v, x.alpha, x.beta, B=B, Hk=Hk, Hv=Hv,
                                        dk=d, dv=d, every=L, capacity=cap,
                                        cu_seqlens=x.cu_seqlens, initial_state=x.initial_state,
                                        threads=THREADS)
    _check_slots(ck, ref, lengths, L, cap, TOL[torch.bfloat16])
    assert torch.equal(out, out0) and torch.equal(fs, fs0)


def test_prefill_T4100_checkpoints_and_resume(gdn, oracle_mod):
    """The benchmark's prefill (T=4100, 64 full chunks + a 4-token tail) with a
    checkpoint after every chunk: sampled heads of sampled slots against the
    oracle; resuming the prefill from checkpoint 40 over the last 1540 tokens
    reproduces the final state."""
    from gated_deltanet_recurrence_02_gb300.inputs import WORKLOADS, make_inputs
    w = WORKLOADS["prefill_T4100"]
    T, C = w["lengths"][0], w["chunk"]
    x = make_inputs(w["seed"], lengths=w["lengths"], Hk=w["Hk"], Hv=w["Hv"], dk=w["dk"],
                    dv=w["dv"], dtype_qkv=w["dtype_qkv"], dtype_gate=w["dtype_gate"])
    g = _dev(x)
    Hk, Hv, d = x.Hk, x.Hv, x.dk
    cap = T // C
    S0 = x.initial_state.cuda()
    ck = Guarded((1, cap, Hv, d, d), F32)
    out, fs, _ = gdn.gdn_prefill_chunked_checkpoints(
        g["q"], g["k"], g["v"], g["alpha"], g["beta"], B=1, T=T, initial_state=S0,
        checkpoints=ck.t, checkpoint_capacity=cap, checkpoint_interval=1, chunk=C)
    out0, fs0 = gdn.gdn_prefill_chunked(g["q"], g["k"], g["v"], g["alpha"], g["beta"], B=1, T=T,
                                        initial_state=S0, chunk=C)
    j = 40
    t1 = (j + 1) * C
    rest = {n: getattr(x, n)[t1:].cuda() for n in ("q", "k", "v", "alpha", "beta")}
    _, fs_res = gdn.gdn_prefill_chunked(rest["q"], rest["k"], rest["v"], rest["alpha"],
                                        rest["beta"], B=1, T=T - t1,
                                        initial_state=ck.t[:, j].contiguous(), chunk=C)
    torch.cuda.synchronize()
    assert torch.equal(out, out0) and torch.equal(fs, fs0)
    assert ck.guards_intact()
    heads = [0, 13, 31]
    ref = oracle_mod.prefix_checkpoints(x.q, x.k, x.v, x.alpha, x.beta, B=1, Hk=Hk, Hv=Hv,
                                        dk=d, dv=d, every=C, capacity=cap, T=T,
                                        initial_state=x.initial_state, heads=heads)
    tol = TOL[torch.bfloat16]
    for jj in (0, 20, j, cap - 1):
        assert rel(ck.t[0, jj, heads], ref[0, jj, heads]) < tol, jj
    _, rS, _ = oracle_mod.recurrent(x.q, x.k, x.v, x.alpha, x.beta, B=1, Hk=Hk, Hv=Hv, dk=d,
                                    dv=d, T=T, initial_state=x.initial_state,
                                    units=[(0, h) for h in heads], threads=THREADS)
    assert rel(fs_res[0, heads], rS[0, heads]) < tol
    assert rel(fs[0, heads], rS[0, heads]) < tol
