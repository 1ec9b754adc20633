"""GPU parity at the edges: every single-token decode instance (head sizes
32 / 64 / 128, each storage type), gate extremes on every path, and wide
key-head sharing, against the fp64 oracle.

Sources: the per-token gated delta rule of Gated DeltaNet (decay in (0, 1],
write strength in [0, 1]); "[WebGPU EP] adds state update capacity support
for GatedDeltaNet" (onnxruntime PR 32767), "Changes" (inverse-GQA key
sharing, the capture contract).
"""
import os

import numpy as np
import pytest
import torch

from helpers import TOL, Guarded, check_capture, rel, to_dev

pytestmark = pytest.mark.gpu
THREADS = min(32, os.cpu_count() or 4)
F32 = torch.float32
DT = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}


@pytest.fixture(scope="module")
def gdn():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from gated_deltanet_recurrence_02_gb300 import build, gdn as g
    build.build()
    g.lib()
    return g


@pytest.mark.parametrize("dk,dv", [(32, 32), (64, 128), (128, 64), (32, 128), (64, 64)])
@pytest.mark.parametrize("dt", ["f32", "f16", "bf16"])
def test_single_token_decode_instances(gdn, oracle_mod, dk, dv, dt):
    """T = 1 with uniform rows takes the single-token decode instance of the
    recurrent kernel; in place, with capture (capacity 2)."""
    from gated_deltanet_recurrence_02_gb300.inputs import capture_counts, make_inputs
    B, cap = 37, 2
    x = make_inputs(1700 + dk + dv, lengths=[1] * B, Hk=2, Hv=4, dk=dk, dv=dv, dtype_qkv=dt,
                    dtype_gate=dt)
    counts = capture_counts(1701, B, cap).tolist()
    g = to_dev(x)
    S = g["initial_state"].clone()
    su = Guarded((B, cap, gdn.slot_width(2, 4, dk, dv)), F32)
    out, _, _ = gdn.gdn_recurrent_capture(g["q"], g["k"], g["v"], g["alpha"], g["beta"], B=B,
                                          T=1, initial_state=S, final_state=S,
                                          state_update_capacity=cap,
                                          capture_count=torch.tensor(counts, dtype=torch.int32,
                                                                     device="cuda"),
                                          state_update=su.t)
    torch.cuda.synchronize()
    ro, rS, rsu = oracle_mod.recurrent(x.q, x.k, x.v, x.alpha, x.beta, B=B, Hk=2, Hv=4, dk=dk,
                                       dv=dv, T=1, initial_state=x.initial_state, capacity=cap,
                                       capture_count=counts)
    tol = TOL[DT[dt]]
    assert rel(out, ro) < tol
    assert rel(S, rS) < tol
    check_capture(su, rsu, counts, x, cap)


def _gates(x, kind, rng):
    """Replace the drawn gates with an extreme regime (same storage dtype)."""
    a, b = x.alpha.float().numpy(), x.beta.float().numpy()
    if kind == "strong_decay":      # decay 1e-3 .. 1e-2: the chunk's gamma underflows fp32
        a = rng.uniform(1e-3, 1e-2, size=a.shape)
    elif kind == "no_decay_full_write":  # alpha = 1 and beta = 1 exactly
        a, b = np.ones_like(a), np.ones_like(b)
    elif kind == "no_write":        # beta = 0: only the decay acts
        b = np.zeros_like(b)
    x.alpha = torch.from_numpy(a.astype(np.float32)).to(x.alpha.dtype)
    x.beta = torch.from_numpy(b.astype(np.float32)).to(x.beta.dtype)
    return x


@pytest.mark.parametrize("kind", ["strong_decay", "no_decay_full_write", "no_write"])
@pytest.mark.parametrize("path", ["tensor_core_prefill", "cuda_core_prefill", "recurrent"])
def test_gate_extremes(gdn, oracle_mod, kind, path):
    from gated_deltanet_recurrence_02_gb300.inputs import make_inputs
    d, dt, chunk = (128, "bf16", 64) if path == "tensor_core_prefill" else (64, "f32", 32)
    lengths = [130, 64, 7]
    x = make_inputs(1800, lengths=lengths, Hk=2, Hv=4, dk=d, dv=d, dtype_qkv=dt, dtype_gate=dt)
    x = _gates(x, kind, np.random.default_rng(1801))
    g = to_dev(x)
    B = len(lengths)
    if path == "recurrent":
        out, fs, _ = gdn.gdn_recurrent_capture(g["q"], g["k"], g["v"], g["alpha"], g["beta"], B=B,
                                               cu_seqlens=g["cu_seqlens"],
                                               initial_state=g["initial_state"])
    else:
        out, fs = gdn.gdn_prefill_chunked(g["q"], g["k"], g["v"], g["alpha"], g["beta"], B=B,
                                          cu_seqlens=g["cu_seqlens"],
                                          initial_state=g["initial_state"], chunk=chunk)
    torch.cuda.synchronize()
    ro, rS, _ = oracle_mod.recurrent(x.q, x.k, x.v, x.alpha, x.beta, B=B, Hk=2, Hv=4, dk=d, dv=d,
                                     cu_seqlens=x.cu_seqlens, initial_state=x.initial_state,
                                     threads=THREADS)
    tol = TOL[DT[dt]]
    assert rel(out, ro) < tol
    assert rel(fs, rS) < tol


def test_eight_value_heads_per_key_head(gdn, oracle_mod):
    """Hk = 2, Hv = 16 (G = 8): the tensor-core prefill, the recurrent path
    with capture (keys stored once per key head) and a replay."""
    from gated_deltanet_recurrence_02_gb300.inputs import make_inputs
    Hk, Hv, d, cap = 2, 16, 128, 5
    lengths = [100, 9]
    x = make_inputs(1900, lengths=lengths, Hk=Hk, Hv=Hv, dk=d, dv=d, dtype_qkv="bf16",
                    dtype_gate="bf16")
    g = to_dev(x)
    B = len(lengths)
    counts = [5, 3]
    o1, fs1 = gdn.gdn_prefill_chunked(g["q"], g["k"], g["v"], g["alpha"], g["beta"], B=B,
                                      cu_seqlens=g["cu_seqlens"],
                                      initial_state=g["initial_state"], chunk=64)
    su = Guarded((B, cap, gdn.slot_width(Hk, Hv, d, d)), F32)
    o2, fs2, _ = gdn.gdn_recurrent_capture(g["q"], g["k"], g["v"], g["alpha"], g["beta"], B=B,
                                           cu_seqlens=g["cu_seqlens"],
                                           initial_state=g["initial_state"],
                                           state_update_capacity=cap,
                                           capture_count=torch.tensor(counts, dtype=torch.int32,
                                                                      device="cuda"),
                                           state_update=su.t)
    acc = [4, 3]
    Sr = gdn.gdn_replay_state_updates(g["initial_state"], su.t,
                                      torch.tensor(acc, dtype=torch.int32, device="cuda"),
                                      state_update_capacity=cap, Hk=Hk)
    torch.cuda.synchronize()
    ro, rS, rsu = oracle_mod.recurrent(x.q, x.k, x.v, x.alpha, x.beta, B=B, Hk=Hk, Hv=Hv, dk=d,
                                       dv=d, cu_seqlens=x.cu_seqlens,
                                       initial_state=x.initial_state, capacity=cap,
                                       capture_count=counts, threads=THREADS)
    tol = TOL[torch.bfloat16]
    for o, fs in ((o1, fs1), (o2, fs2)):
        assert rel(o, ro) < tol and rel(fs, rS) < tol
    check_capture(su, rsu, counts, x, cap)
    for b, m in enumerate(acc):
        t0 = int(x.cu_seqlens[b])
        sl = slice(t0, t0 + m)
        _, Sm, _ = oracle_mod.recurrent(x.q[sl], x.k[sl], x.v[sl], x.alpha[sl], x.beta[sl], B=1,
                                        Hk=Hk, Hv=Hv, dk=d, dv=d, T=m,
                                        initial_state=x.initial_state[b:b + 1])
        assert rel(Sr[b], Sm[0]) < TOL[torch.bfloat16], b


@pytest.mark.parametrize("path", ["tensor_core_prefill", "cuda_core_prefill", "recurrent"])
def test_one_value_head_per_key_head(gdn, oracle_mod, path):
    """Hk = Hv = 4 (G = 1, no key sharing) on each path; the recurrent path
    with capture (a key stored per value head) and a replay of the capture."""
    from gated_deltanet_recurrence_02_gb300.inputs import make_inputs
    Hk = Hv = 4
    d, dt, chunk = (128, "bf16", 64) if path != "cuda_core_prefill" else (64, "f32", 32)
    lengths, cap, counts = [100, 9, 64], 5, [5, 3, 0]
    x = make_inputs(1950, lengths=lengths, Hk=Hk, Hv=Hv, dk=d, dv=d, dtype_qkv=dt, dtype_gate=dt)
    g = to_dev(x)
    B = len(lengths)
    su = None
    if path == "recurrent":
        su = Guarded((B, cap, gdn.slot_width(Hk, Hv, d, d)), F32)
        out, fs, _ = gdn.gdn_recurrent_capture(g["q"], g["k"], g["v"], g["alpha"], g["beta"], B=B,
                                               cu_seqlens=g["cu_seqlens"],
                                               initial_state=g["initial_state"],
                                               state_update_capacity=cap,
                                               capture_count=torch.tensor(counts, dtype=torch.int32,
                                                                          device="cuda"),
                                               state_update=su.t)
    else:
        out, fs = gdn.gdn_prefill_chunked(g["q"], g["k"], g["v"], g["alpha"], g["beta"], B=B,
                                          cu_seqlens=g["cu_seqlens"],
                                          initial_state=g["initial_state"], chunk=chunk)
    torch.cuda.synchronize()
    ro, rS, rsu = oracle_mod.recurrent(x.q, x.k, x.v, x.alpha, x.beta, B=B, Hk=Hk, Hv=Hv, dk=d,
                                       dv=d, cu_seqlens=x.cu_seqlens,
                                       initial_state=x.initial_state, capacity=cap if su else 0,
                                       capture_count=counts if su else None, threads=THREADS)
    tol = TOL[DT[dt]]
    assert rel(out, ro) < tol
    assert rel(fs, rS) < tol
    if su is not None:
        check_capture(su, rsu, counts, x, cap)
        acc = [4, 3, 0]
        Sr = gdn.gdn_replay_state_updates(g["initial_state"], su.t,
                                          torch.tensor(acc, dtype=torch.int32, device="cuda"),
                                          state_update_capacity=cap, Hk=Hk)
        torch.cuda.synchronize()
        for b, m in enumerate(acc):
            t0 = int(x.cu_seqlens[b])
            sl = slice(t0, t0 + m)
            _, Sm, _ = oracle_mod.recurrent(x.q[sl], x.k[sl], x.v[sl], x.alpha[sl], x.beta[sl], B=1,
                                            Hk=Hk, Hv=Hv, dk=d, dv=d, T=m,
                                            initial_state=x.initial_state[b:b + 1])
            assert rel(Sr[b], Sm[0]) < tol, b
