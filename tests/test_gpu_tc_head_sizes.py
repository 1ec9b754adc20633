"""GPU parity of the tensor-core prefill at head sizes below 128.

The tensor-core kernels work on 128-wide tiles; a head of 32 or 64 features
(dk, dv in {32, 64, 128}, chunk 64, 16-bit q/k/v) is read as zero-padded to
128 (the tensor maps' out-of-bounds fill), which leaves every product with
the real features unchanged, and only the real rows and columns of the state,
the outputs, the checkpoints and the capture are written.  Each case is
checked against the fp64 oracle per (row, value head), on packed rows with a
ragged tail, an empty row and rows of one and of several chunks.  The
tensor-core path is the one taken: it is the only one that asks for a
workspace.

Sources: the chunked form of the gated delta rule ("Enable the native Kev
example on NVIDIA GPUs through ExecuTorch's AOTI CUDA backend", executorch
issue 23097, "Work to cover": varying batch and sequence shapes); the
capture contract ("[WebGPU EP] adds state update capacity support for
GatedDeltaNet", onnxruntime PR 32767, "Changes"); prefix snapshots kept at
chunk boundaries ("Enable the native Kev example on the WebGPU backend",
executorch issue 23099).
"""
import os

import numpy as np
import pytest
import torch

from helpers import TOL, TOL_CAPTURE, Guarded, rel

pytestmark = pytest.mark.gpu
THREADS = min(32, os.cpu_count() or 4)
F32 = torch.float32
LENGTHS = [130, 1, 0, 64, 257, 63]


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


def _per_row_head(out, fs, ro, rS, cu, Hv, tol):
    ro, rS = np.asarray(ro), np.asarray(rS)
    for r in range(len(cu) - 1):
        for h in range(Hv):
            if cu[r + 1] > cu[r]:
                assert rel(out[cu[r]:cu[r + 1], h], ro[cu[r]:cu[r + 1], h]) < tol, (r, h)
            assert rel(fs[r, h], rS[r, h]) < tol, (r, h)


@pytest.mark.parametrize("dk,dv,dtype", [(64, 64, "bf16"), (32, 32, "bf16"), (64, 128, "f16"),
                                         (128, 64, "bf16"), (32, 64, "f16"), (128, 32, "bf16")])
def test_plain(gdn, oracle_mod, dk, dv, dtype):
    from gated_deltanet_recurrence_02_gb300.inputs import make_inputs
    Hk, Hv, B = 2, 4, len(LENGTHS)
    x = make_inputs(3100 + dk + 3 * dv, lengths=LENGTHS, Hk=Hk, Hv=Hv, dk=dk, dv=dv, dtype_qkv=dtype,
                    dtype_gate="f32")
    T = int(x.cu_seqlens[-1])
    assert gdn.gdn_prefill_workspace_size(B, T, Hk, Hv, dk, dv, 64, x.q.dtype, varlen=True) > 0
    g = _dev(x)
    cu_d = x.cu_seqlens.cuda()
    out, fs = gdn.gdn_prefill_chunked(g["q"], g["k"], g["v"], g["alpha"], g["beta"], B=B,
                                      cu_seqlens=cu_d, initial_state=x.initial_state.cuda(), chunk=64)
    torch.cuda.synchronize()
    ro, rS, _ = oracle_mod.recurrent(x.q, x.k, x.v, x.alpha, x.beta, B=B, Hk=Hk, Hv=Hv, dk=dk, dv=dv,
                                     cu_seqlens=x.cu_seqlens, initial_state=x.initial_state,
                                     threads=THREADS)
    _per_row_head(out, fs, ro, rS, x.cu_seqlens.tolist(), Hv, TOL[x.q.dtype])
    # the empty row keeps its initial state exactly
    assert torch.equal(fs[2].cpu(), x.initial_state[2])


def test_uniform_rows_many_heads(gdn, oracle_mod):
    """Uniform rows (no cu_seqlens) at d = 64 with 16 value heads per key
    head's pair, enough (row, head) tiles for several CTAs per head."""
    from gated_deltanet_recurrence_02_gb300.inputs import make_inputs
    Hk, Hv, B, T, d = 4, 16, 2, 300, 64
    x = make_inputs(3150, lengths=[T] * B, Hk=Hk, Hv=Hv, dk=d, dv=d, dtype_qkv="bf16",
                    dtype_gate="bf16")
    g = _dev(x)
    out, fs = gdn.gdn_prefill_chunked(g["q"], g["k"], g["v"], g["alpha"], g["beta"], B=B, T=T,
                                      initial_state=x.initial_state.cuda(), chunk=64)
    torch.cuda.synchronize()
    ro, rS, _ = oracle_mod.recurrent(x.q, x.k, x.v, x.alpha, x.beta, B=B, Hk=Hk, Hv=Hv, dk=d, dv=d,
                                     T=T, initial_state=x.initial_state, threads=THREADS)
    tol = TOL[torch.bfloat16]
    for b in range(B):
        for h in range(Hv):
            assert rel(out[b * T:(b + 1) * T, h], np.asarray(ro)[b * T:(b + 1) * T, h]) < tol, (b, h)
            assert rel(fs[b, h], np.asarray(rS)[b, h]) < tol, (b, h)


def test_capture_checkpoints_and_conventions(gdn, oracle_mod):
    """d = 64 through the capture, the checkpoints and the in-kernel input
    conventions (the XO and NORM instances of both kernels)."""
    from gated_deltanet_recurrence_02_gb300.inputs import make_raw_inputs
    Hk, Hv, d, B = 2, 4, 64, len(LENGTHS)
    x = make_raw_inputs(3170, lengths=LENGTHS, Hk=Hk, Hv=Hv, dk=d, dv=d, dtype_qkv="bf16",
                        dtype_gate="bf16")
    q, k, a, b_ = oracle_mod.front_end(x.q, x.k, x.alpha, x.beta, qk_l2norm=True, alpha_log=True,
                                       beta_logit=True)
    g = _dev(x)
    cu_d, S0 = x.cu_seqlens.cuda(), x.initial_state.cuda()
    conv = 0x700
    cap, counts = 70, [70, 1, 5, 64, 3, 0]
    su = Guarded((B, cap, gdn.slot_width(Hk, Hv, d, d)), F32)
    out, fs, _ = gdn.gdn_prefill_chunked_capture(
        g["q"], g["k"], g["v"], g["alpha"], g["beta"], B=B, cu_seqlens=cu_d, initial_state=S0,
        chunk=64, state_update_capacity=cap, conventions=conv,
        capture_count=torch.tensor(counts, dtype=torch.int32, device="cuda"), state_update=su.t)
    ck_cap = 4
    out2, fs2, ck = gdn.gdn_prefill_chunked_checkpoints(
        g["q"], g["k"], g["v"], g["alpha"], g["beta"], B=B, checkpoint_capacity=ck_cap,
        checkpoint_interval=1, cu_seqlens=cu_d, initial_state=S0, chunk=64, conventions=conv)
    torch.cuda.synchronize()
    assert su.guards_intact()
    ro, rS, rsu = oracle_mod.recurrent(q, k, x.v, a, b_, B=B, Hk=Hk, Hv=Hv, dk=d, dv=d,
                                       cu_seqlens=x.cu_seqlens, initial_state=x.initial_state,
                                       capacity=cap, capture_count=counts, threads=THREADS)
    tol = TOL[torch.bfloat16]
    cu = x.cu_seqlens.tolist()
    _per_row_head(out, fs, ro, rS, cu, Hv, tol)
    _per_row_head(out2, fs2, ro, rS, cu, Hv, tol)
    off = Hv + Hk * d
    for r, nb in enumerate(min(c, cap, L) for c, L in zip(counts, LENGTHS)):
        if nb == 0:
            continue
        assert rel(su.t[r, :nb, :Hv], rsu[r, :nb, :Hv]) < TOL_CAPTURE, r
        assert rel(su.t[r, :nb, Hv:off], rsu[r, :nb, Hv:off]) < TOL_CAPTURE, r
        assert rel(su.t[r, :nb, off:], rsu[r, :nb, off:]) < tol, r
    # checkpoint j of row r: the state after 64 (j + 1) tokens, where the row has them
    cks = oracle_mod.prefix_checkpoints(q, k, x.v, a, b_, B=B, Hk=Hk, Hv=Hv, dk=d, dv=d, every=64,
                                        capacity=ck_cap, cu_seqlens=x.cu_seqlens,
                                        initial_state=x.initial_state, threads=THREADS)
    for r, L in enumerate(LENGTHS):
        for j in range(min(ck_cap, L // 64)):
            assert rel(ck[r, j], cks[r, j]) < tol, (r, j)


@pytest.mark.parametrize("dk,dv", [(64, 64), (32, 128)])
def test_wide_carry_instance(gdn, oracle_mod, dk, dv):
    """Enough (row, head) tiles that the launcher takes the 64-row carry
    instance (dv / 32 x Hv x B above the SM count): one 64-row tile per head
    at dv = 64, two at dv = 128 with a 32-feature key."""
    from gated_deltanet_recurrence_02_gb300.inputs import make_inputs
    Hk, Hv = 4, 16
    lengths = [70, 130, 1, 64, 200, 90, 65, 33]
    B = len(lengths)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    if (dv // 32) * Hv * B <= sms:
        pytest.skip("the 64-row carry instance needs more (row, head) tiles than SMs")
    x = make_inputs(3190 + dk + dv, lengths=lengths, Hk=Hk, Hv=Hv, dk=dk, dv=dv, dtype_qkv="bf16",
                    dtype_gate="f32")
    g = _dev(x)
    out, fs = gdn.gdn_prefill_chunked(g["q"], g["k"], g["v"], g["alpha"], g["beta"], B=B,
                                      cu_seqlens=x.cu_seqlens.cuda(), initial_state=x.initial_state.cuda(),
                                      chunk=64)
    torch.cuda.synchronize()
    ro, rS, _ = oracle_mod.recurrent(x.q, x.k, x.v, x.alpha, x.beta, B=B, Hk=Hk, Hv=Hv, dk=dk, dv=dv,
                                     cu_seqlens=x.cu_seqlens, initial_state=x.initial_state,
                                     threads=THREADS)
    _per_row_head(out, fs, ro, rS, x.cu_seqlens.tolist(), Hv, TOL[torch.bfloat16])
