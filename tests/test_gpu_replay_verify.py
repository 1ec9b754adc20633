"""GPU parity of gdn_replay_verify -- one speculative-decoding step in one
launch: replay of the accepted prefix of the previous capture, then the draft
tokens with capture -- against the fp64 oracle on the same seeded inputs.

Source: "[WebGPU EP] adds state update capacity support for GatedDeltaNet"
(onnxruntime PR 32767), "DFlash2 Prerequisite": full, partial and zero draft
acceptance must reproduce the non-speculative output and state.
"""
import os

import numpy as np
import pytest
import torch

from helpers import TOL, TOL_CAPTURE, Guarded, check_capture, rel

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


def _inputs(seed, lengths, Hk, Hv, d, dt, dtg, zero_state=False):
    from gated_deltanet_recurrence_02_gb300.inputs import make_inputs
    return make_inputs(seed, lengths=lengths, Hk=Hk, Hv=Hv, dk=d, dv=d, dtype_qkv=dt,
                       dtype_gate=dtg, zero_state=zero_state)


def _prev_capture(oracle_mod, x, cap, units=None):
    """The previous verify pass's capture (every draft captured), computed by
    the oracle and stored as fp32 like the library's buffer.  Rows outside
    `units` are zeros (valid factors that are never checked)."""
    _, _, su = oracle_mod.recurrent(x.q, x.k, x.v, x.alpha, x.beta, B=x.B, Hk=x.Hk, Hv=x.Hv,
                                    dk=x.dk, dv=x.dv, cu_seqlens=x.cu_seqlens,
                                    initial_state=x.initial_state, capacity=cap,
                                    capture_count=[cap] * x.B, units=units, threads=THREADS)
    return torch.from_numpy(np.nan_to_num(su, nan=0.0).astype(np.float32))


def _dev(x):
    return {n: getattr(x, n).cuda() for n in ("q", "k", "v", "alpha", "beta")}


def _acc(vals):
    return torch.tensor(vals, dtype=torch.int32, device="cuda")


# ------------------------------------------------------------- tiny fp32

@pytest.mark.parametrize("accepted", [[0, 4], [2, 1], [4, 0], [-3, 9]])
def test_tiny_f32_replay_then_ragged_drafts(gdn, oracle_mod, accepted):
    """Zero, partial, full and out-of-range acceptance; the second row has no
    new drafts (it only replays)."""
    Hk, Hv, d, cap, B = 1, 2, 32, 4, 2
    x1 = _inputs(1100, [4, 4], Hk, Hv, d, "f32", "f32")
    x2 = _inputs(1101, [3, 0], Hk, Hv, d, "f32", "f32", zero_state=True)
    su1 = _prev_capture(oracle_mod, x1, cap)
    slot = gdn.slot_width(Hk, Hv, d, d)
    so = Guarded((B, Hv, d, d), F32)
    sf = Guarded((B, Hv, d, d), F32)
    out = Guarded(tuple(x2.v.shape), F32)
    su2 = Guarded((B, cap, slot), F32)
    g = _dev(x2)
    gdn.gdn_replay_verify(g["q"], g["k"], g["v"], g["alpha"], g["beta"], B=B,
                          cu_seqlens=x2.cu_seqlens.cuda(), state_in=x1.initial_state.cuda(),
                          state_out=so.t, prev_state_update=su1.cuda(), prev_capacity=cap,
                          accepted_count=_acc(accepted), draft_final_state=sf.t, out=out.t,
                          state_update_capacity=cap, capture_count=_acc([4, 4]),
                          state_update=su2.t)
    torch.cuda.synchronize()
    ro, rSc, rSf, rsu = oracle_mod.replay_verify(
        x2.q, x2.k, x2.v, x2.alpha, x2.beta, B=B, Hk=Hk, Hv=Hv, dk=d, dv=d,
        cu_seqlens=x2.cu_seqlens, state_in=x1.initial_state, prev_state_update=su1,
        prev_capacity=cap, accepted_count=accepted, capacity=cap, capture_count=[4, 4])
    assert rel(so.t, rSc) < TOL[F32]
    assert rel(sf.t, rSf) < TOL[F32]
    assert rel(out.t, ro) < TOL[F32]
    assert so.guards_intact() and sf.guards_intact() and out.guards_intact()
    assert check_capture(su2, rsu, [4, 4], x2, cap) == [3, 0]


# ------------------------------------------------- fp16, Hk=2 / Hv=6 / 128

@pytest.mark.parametrize("active", [1, 0])
def test_qwenlike_f16_long_acceptance_and_drafts(gdn, oracle_mod, active):
    """Capacity 7: acceptance beyond the four slots the kernel stages and
    eight drafts (beyond the four staged tokens) take the direct-load paths;
    the slot width (1030 floats) leaves the factors unaligned.  Inactive
    capture zeroes the whole new buffer."""
    Hk, Hv, d, cap, B, T = 2, 6, 128, 7, 3, 8
    x1 = _inputs(1102, [7, 7, 7], Hk, Hv, d, "f16", "f16")
    x2 = _inputs(1103, [T] * B, Hk, Hv, d, "f16", "f16", zero_state=True)
    su1 = _prev_capture(oracle_mod, x1, cap)
    accepted, counts = [0, 5, 7], [0, 4, 7]
    slot = gdn.slot_width(Hk, Hv, d, d)
    so = Guarded((B, Hv, d, d), F32)
    sf = Guarded((B, Hv, d, d), F32)
    out = Guarded(tuple(x2.v.shape), torch.float16)
    su2 = Guarded((B, cap, slot), F32)
    g = _dev(x2)
    gdn.gdn_replay_verify(g["q"], g["k"], g["v"], g["alpha"], g["beta"], B=B, T=T,
                          state_in=x1.initial_state.cuda(), state_out=so.t,
                          prev_state_update=su1.cuda(), prev_capacity=cap,
                          accepted_count=_acc(accepted), draft_final_state=sf.t, out=out.t,
                          state_update_capacity=cap, capture_count=_acc(counts),
                          state_update_active=_acc([active]), state_update=su2.t)
    torch.cuda.synchronize()
    ro, rSc, rSf, rsu = oracle_mod.replay_verify(
        x2.q, x2.k, x2.v, x2.alpha, x2.beta, B=B, Hk=Hk, Hv=Hv, dk=d, dv=d, T=T,
        state_in=x1.initial_state, prev_state_update=su1, prev_capacity=cap,
        accepted_count=accepted, capacity=cap, capture_count=counts, active=bool(active),
        threads=THREADS)
    assert rel(so.t, rSc) < TOL[torch.float16]
    assert rel(sf.t, rSf) < TOL[torch.float16]
    assert rel(out.t, ro) < TOL[torch.float16]
    assert so.guards_intact() and sf.guards_intact() and out.guards_intact()
    if active:
        check_capture(su2, rsu, counts, x2, cap)
    else:
        assert bool(torch.all(su2.t == 0).item()) and su2.guards_intact()


# ------------------------------------------- in place, bit-exact invariants

def test_in_place_replay_is_bitwise_the_verify_state(gdn):
    """The kernel's replay performs the same fp32 operations as its token
    update on the captured decay / key / delta, so the committed state equals,
    bit for bit, the state the same kernel reaches after running the accepted
    tokens; the new drafts' outputs then equal a plain recurrent call from that
    state.  In place, a row that accepted nothing is not rewritten."""
    Hk, Hv, d, cap, B = 2, 4, 128, 4, 4
    x1 = _inputs(1110, [cap] * B, Hk, Hv, d, "bf16", "bf16")
    x2 = _inputs(1111, [2, 0, 3, 1], Hk, Hv, d, "bf16", "bf16", zero_state=True)
    S0 = x1.initial_state.cuda()
    g1 = _dev(x1)
    _, _, su1 = gdn.gdn_recurrent_capture(g1["q"], g1["k"], g1["v"], g1["alpha"], g1["beta"],
                                          B=B, T=cap, initial_state=S0, want_final_state=False,
                                          state_update_capacity=cap,
                                          capture_count=_acc([cap] * B))
    accepted = [0, 1, 3, 4]
    # the same kernel over each row's accepted tokens
    idx = torch.tensor([b * cap + t for b in range(B) for t in range(accepted[b])])
    cu = torch.tensor(np.concatenate([[0], np.cumsum(accepted)]), dtype=torch.int32).cuda()
    sel = {n: getattr(x1, n)[idx].cuda() for n in ("q", "k", "v", "alpha", "beta")}
    _, S_m, _ = gdn.gdn_recurrent_capture(sel["q"], sel["k"], sel["v"], sel["alpha"],
                                          sel["beta"], B=B, cu_seqlens=cu, initial_state=S0)
    g2 = _dev(x2)
    cu2 = x2.cu_seqlens.cuda()
    o_ref, _, _ = gdn.gdn_recurrent_capture(g2["q"], g2["k"], g2["v"], g2["alpha"], g2["beta"],
                                            B=B, cu_seqlens=cu2, initial_state=S_m)
    state = S0.clone()
    out, _, _, _ = gdn.gdn_replay_verify(g2["q"], g2["k"], g2["v"], g2["alpha"], g2["beta"], B=B,
                                         cu_seqlens=cu2, state_in=state, state_out=state,
                                         prev_state_update=su1, prev_capacity=cap,
                                         accepted_count=_acc(accepted))
    torch.cuda.synchronize()
    assert torch.equal(state, S_m)
    assert torch.equal(state[0], S0[0])
    assert torch.equal(out, o_ref)


# ------------------------------------------------------- speculative loop

def test_speculative_loop_matches_non_speculative_run(gdn, oracle_mod):
    """Five speculative steps (4 drafts per row, seeded acceptance
    U{0..4}, state in place, two alternating capture buffers), then a
    replay-only call: the committed state equals the oracle's run over the
    accepted tokens, and each step's draft outputs equal the oracle's outputs
    for (accepted history + drafts)."""
    from gated_deltanet_recurrence_02_gb300.inputs import accepted_counts
    Hk, Hv, d, T, B, steps = 2, 6, 128, 4, 3, 5
    dt = "bf16"
    xs = [_inputs(1120 + s, [T] * B, Hk, Hv, d, dt, dt, zero_state=(s > 0)) for s in range(steps)]
    S0 = xs[0].initial_state
    acc = [accepted_counts(1130 + s, B, T).tolist() for s in range(steps)]
    slot = gdn.slot_width(Hk, Hv, d, d)
    su = [torch.empty((B, T, slot), dtype=F32, device="cuda") for _ in range(2)]
    state = S0.cuda()
    outs = []
    for s in range(steps):
        g = _dev(xs[s])
        kw = {}
        if s > 0:
            kw = dict(prev_state_update=su[(s - 1) % 2], prev_capacity=T,
                      accepted_count=_acc(acc[s - 1]))
        o, _, _, _ = gdn.gdn_replay_verify(g["q"], g["k"], g["v"], g["alpha"], g["beta"], B=B,
                                           T=T, state_in=state, state_out=state,
                                           state_update_capacity=T,
                                           capture_count=_acc([T] * B),
                                           state_update=su[s % 2], **kw)
        outs.append(o.cpu())
    empty = {n: getattr(xs[0], n)[:0].cuda() for n in ("q", "k", "v", "alpha", "beta")}
    gdn.gdn_replay_verify(empty["q"], empty["k"], empty["v"], empty["alpha"], empty["beta"], B=B,
                          cu_seqlens=torch.zeros(B + 1, dtype=torch.int32, device="cuda"),
                          state_in=state, state_out=state, prev_state_update=su[(steps - 1) % 2],
                          prev_capacity=T, accepted_count=_acc(acc[steps - 1]))
    torch.cuda.synchronize()
    one = dict(B=1, Hk=Hk, Hv=Hv, dk=d, dv=d)

    def cat(parts, name):
        return torch.cat([getattr(x, name)[sl] for x, sl in parts]) if parts else \
            getattr(xs[0], name)[:0]

    for b in range(B):
        hist = []  # (inputs, token slice) of row b's accepted tokens so far
        for s in range(steps):
            draft = (xs[s], slice(b * T, b * T + T))
            parts = hist + [draft]
            n = sum(sl.stop - sl.start for _, sl in parts)
            o_ns, _, _ = oracle_mod.recurrent(*(cat(parts, nm) for nm in ("q", "k", "v", "alpha", "beta")),
                                              T=n, initial_state=S0[b:b + 1], **one)
            assert rel(outs[s][b * T:(b + 1) * T], o_ns[n - T:]) < TOL[torch.bfloat16], (b, s)
            hist.append((xs[s], slice(b * T, b * T + acc[s][b])))
        n = sum(sl.stop - sl.start for _, sl in hist)
        _, S_ns, _ = oracle_mod.recurrent(*(cat(hist, nm) for nm in ("q", "k", "v", "alpha", "beta")),
                                          T=n, initial_state=S0[b:b + 1], **one)
        assert rel(state[b], S_ns[0]) < TOL[torch.bfloat16], b


# ------------------------------------------- the timed configuration, sampled

def test_verify_B256_T4_sampled_rows(gdn, oracle_mod):
    """The benchmark's speculative step (B=256, Hk=16, Hv=32, d=128, bf16,
    4 drafts, capacity 4, acceptance U{0..4}, in place), checked on sampled
    rows (all heads) against the oracle."""
    from gated_deltanet_recurrence_02_gb300.inputs import WORKLOADS, accepted_counts, make_inputs
    w = WORKLOADS["verify_B256_T4"]
    B, T, cap, Hk, Hv, d = w["B"], w["T"], w["capacity"], w["Hk"], w["Hv"], w["dk"]
    common = dict(Hk=Hk, Hv=Hv, dk=d, dv=d, dtype_qkv=w["dtype_qkv"], dtype_gate=w["dtype_gate"])
    x1 = make_inputs(w["seed"], lengths=[T] * B, **common)
    x2 = make_inputs(w["seed"] + 1, lengths=[T] * B, zero_state=True, **common)
    accepted = accepted_counts(w["seed"] + 2, B, cap)
    rows = [0, 1, 77, 128, 200, 255]
    units = [(b, h) for b in rows for h in range(Hv)]
    su1 = _prev_capture(oracle_mod, x1, cap, units=units)
    slot = gdn.slot_width(Hk, Hv, d, d)
    state = x1.initial_state.cuda()
    su2 = Guarded((B, cap, slot), F32)
    g = _dev(x2)
    out, _, _, _ = gdn.gdn_replay_verify(g["q"], g["k"], g["v"], g["alpha"], g["beta"], B=B, T=T,
                                         state_in=state, state_out=state,
                                         prev_state_update=su1.cuda(), prev_capacity=cap,
                                         accepted_count=accepted.cuda(),
                                         state_update_capacity=cap,
                                         capture_count=_acc([cap] * B), state_update=su2.t)
    torch.cuda.synchronize()
    ro, rSc, _, rsu = oracle_mod.replay_verify(
        x2.q, x2.k, x2.v, x2.alpha, x2.beta, B=B, Hk=Hk, Hv=Hv, dk=d, dv=d, T=T,
        state_in=x1.initial_state, prev_state_update=su1, prev_capacity=cap,
        accepted_count=accepted.tolist(), capacity=cap, capture_count=[cap] * B,
        units=units, threads=THREADS)
    tol = TOL[torch.bfloat16]
    off = Hv + Hk * d
    for b in rows:
        assert rel(state[b], rSc[b]) < tol, b
        assert rel(out[b * T:(b + 1) * T], ro[b * T:(b + 1) * T]) < tol, b
        gsu = su2.t[b].cpu().double().numpy()
        assert np.array_equal(gsu[:, :off], rsu[b][:, :off]), b
        assert rel(su2.t[b, :, off:], rsu[b][:, off:]) < TOL_CAPTURE, b
    assert su2.guards_intact()
