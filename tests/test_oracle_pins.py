"""Pins for the fp64 oracle: facts the definition fixes, checked on the CPU.

Each pin is chosen so that a plausible slip in the oracle (a dropped decay,
delta formed from the undecayed state, readout before the update, a
transposed state, a wrong key-head index, a wrong capture clamp) fails at
least one of them.  Sources: the per-token gated delta rule of Gated DeltaNet;
"[WebGPU EP] adds state update capacity support for GatedDeltaNet"
(onnxruntime PR 32767), "Changes" and "Test Coverage".
"""
import json
import os

import numpy as np
import pytest

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rand_case(rng, T, Hk, Hv, dk, dv, unit_k=True, alpha_lo=0.6):
    q = rng.standard_normal((T, Hk, dk))
    k = rng.standard_normal((T, Hk, dk))
    if unit_k:
        k /= np.linalg.norm(k, axis=-1, keepdims=True)
        q /= np.linalg.norm(q, axis=-1, keepdims=True)
    v = rng.standard_normal((T, Hv, dv))
    alpha = rng.uniform(alpha_lo, 1.0, size=(T, Hv))
    beta = rng.uniform(0.0, 1.0, size=(T, Hv))
    S0 = 0.3 * rng.standard_normal((1, Hv, dv, dk))
    return q, k, v, alpha, beta, S0


def _rel(a, b):
    return np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300)


# --- worked example -------------------------------------------------------

def test_hand_worked_example(oracle_mod):
    g = json.load(open(os.path.join(GOLDEN, "hand_worked_T2_d2.json")))
    q = np.array(g["q"])[:, None, :]
    k = np.array(g["k"])[:, None, :]
    v = np.array(g["v"])[:, None, :]
    a = np.array(g["alpha"])[:, None]
    b = np.array(g["beta"])[:, None]
    S0 = np.array(g["S0"])[None, None]
    dims = dict(B=1, Hk=1, Hv=1, dk=2, dv=2, T=2)
    o, S, su = oracle_mod.recurrent(q, k, v, a, b, initial_state=S0, capacity=2,
                                    capture_count=[2], **dims)
    assert np.array_equal(o[:, 0, :], np.array(g["o"]))
    assert np.array_equal(S[0, 0], np.array(g["S_final"]))
    assert np.array_equal(su[0], np.array(g["state_update"]))
    for C in (1, 2, 3):
        oc, Sc = oracle_mod.chunked(q, k, v, a, b, initial_state=S0, chunk=C, **dims)
        assert np.allclose(oc[:, 0, :], g["o"], rtol=0, atol=1e-14)
        assert np.allclose(Sc[0, 0], g["S_final"], rtol=0, atol=1e-14)
    Sr = oracle_mod.replay(S0, su, [2], B=1, Hk=1, Hv=1, dk=2, dv=2, capacity=2)
    assert np.array_equal(Sr[0, 0], np.array(g["S_final"]))


# --- closed forms -----------------------------------------------------------

def test_identity_alpha1_beta0(oracle_mod):
    """alpha = 1, beta = 0: the state never changes and o_t = S0 q_t."""
    rng = np.random.default_rng(1)
    T, Hk, Hv, dk, dv = 9, 1, 2, 6, 4
    q, k, v, _, _, S0 = _rand_case(rng, T, Hk, Hv, dk, dv)
    a = np.ones((T, Hv))
    b = np.zeros((T, Hv))
    dims = dict(B=1, Hk=Hk, Hv=Hv, dk=dk, dv=dv, T=T)
    o, S, _ = oracle_mod.recurrent(q, k, v, a, b, initial_state=S0, scale=0.5, **dims)
    assert np.array_equal(S, S0)
    for h in range(Hv):
        ref = 0.5 * np.einsum("ij,tj->ti", S0[0, h], q[:, 0, :])
        assert _rel(o[:, h, :], ref) < 1e-15
    oc, Sc = oracle_mod.chunked(q, k, v, a, b, initial_state=S0, scale=0.5,
                                chunk=4, **dims)
    assert _rel(Sc, S0) < 1e-15 and _rel(oc, o) < 1e-15


def test_beta0_pure_decay(oracle_mod):
    """beta = 0: S_t = (prod_{s<=t} alpha_s) S0 and o_t = S_t q_t."""
    rng = np.random.default_rng(2)
    T, Hk, Hv, dk, dv = 7, 1, 1, 5, 3
    q, k, v, a, _, S0 = _rand_case(rng, T, Hk, Hv, dk, dv)
    b = np.zeros((T, Hv))
    o, S, _ = oracle_mod.recurrent(q, k, v, a, b, initial_state=S0, B=1, Hk=Hk,
                                   Hv=Hv, dk=dk, dv=dv, T=T)
    cum = np.cumprod(a[:, 0])
    assert _rel(S[0, 0], cum[-1] * S0[0, 0]) < 1e-14
    ref = cum[:, None] * np.einsum("ij,tj->ti", S0[0, 0], q[:, 0, :])
    assert _rel(o[:, 0, :], ref) < 1e-14


def test_delta_rule_writes_exactly(oracle_mod):
    """beta = 1 and a unit key: after the update, S k_t = v_t.  Reading out
    with q_t = k_t (scale 1) makes o_t that product, for every token."""
    rng = np.random.default_rng(3)
    T, Hk, Hv, dk, dv = 12, 1, 2, 8, 5
    _, k, v, a, _, S0 = _rand_case(rng, T, Hk, Hv, dk, dv)
    b = np.ones((T, Hv))
    o, _, _ = oracle_mod.recurrent(k, k, v, a, b, initial_state=S0, B=1, Hk=Hk,
                                   Hv=Hv, dk=dk, dv=dv, T=T)
    assert np.max(np.abs(o - v)) < 1e-13


def test_single_token_from_zero_state(oracle_mod):
    """T = 1, S0 = 0: S = beta v k^T and o = beta (k . q) v."""
    rng = np.random.default_rng(4)
    Hk, Hv, dk, dv = 1, 1, 7, 3
    q, k, v, a, b, _ = _rand_case(rng, 1, Hk, Hv, dk, dv)
    o, S, _ = oracle_mod.recurrent(q, k, v, a, b, B=1, Hk=Hk, Hv=Hv, dk=dk,
                                   dv=dv, T=1, scale=2.0)
    assert _rel(S[0, 0], b[0, 0] * np.outer(v[0, 0], k[0, 0])) < 1e-15
    ref = b[0, 0] * 2.0 * np.dot(k[0, 0], q[0, 0]) * v[0, 0]
    assert _rel(o[0, 0], ref) < 1e-14


# --- independent formulations ---------------------------------------------

@pytest.mark.parametrize("T", [1, 2, 3, 4])
def test_bruteforce_unrolled_products(oracle_mod, T):
    """Unrolled products of explicit dk x dk matrices; dk != dv and a
    non-symmetric S0 so that a transposed state cannot pass."""
    rng = np.random.default_rng(10 + T)
    Hk, Hv, dk, dv = 1, 1, 5, 3
    q, k, v, a, b, S0 = _rand_case(rng, T, Hk, Hv, dk, dv, unit_k=False)
    o, S, _ = oracle_mod.recurrent(q, k, v, a, b, initial_state=S0, B=1, Hk=Hk,
                                   Hv=Hv, dk=dk, dv=dv, T=T, scale=0.7)
    ob, Sb = oracle_mod.bruteforce_unrolled(q[:, 0], k[:, 0], v[:, 0], a[:, 0],
                                            b[:, 0], S0[0, 0], scale=0.7)
    assert _rel(S[0, 0], Sb) < 1e-13
    assert _rel(o[:, 0, :], ob) < 1e-13


@pytest.mark.parametrize("chunk,lengths", [(16, [37, 64]), (64, [130]),
                                           (5, [23, 1, 10]), (1, [6])])
def test_chunked_equals_recurrent(oracle_mod, chunk, lengths):
    """The chunked UT/WY form and the per-token form agree in fp64, with a
    ragged last chunk, ragged rows and three value heads per key head."""
    rng = np.random.default_rng(20 + chunk)
    Hk, Hv, dk, dv = 2, 6, 12, 10
    T = sum(lengths)
    q, k, v, a, b, _ = _rand_case(rng, T, Hk, Hv, dk, dv, alpha_lo=0.5)
    S0 = 0.3 * rng.standard_normal((len(lengths), Hv, dv, dk))
    cu = np.concatenate([[0], np.cumsum(lengths)])
    dims = dict(B=len(lengths), Hk=Hk, Hv=Hv, dk=dk, dv=dv, cu_seqlens=cu)
    o, S, _ = oracle_mod.recurrent(q, k, v, a, b, initial_state=S0, scale=0.9, **dims)
    oc, Sc = oracle_mod.chunked(q, k, v, a, b, initial_state=S0, scale=0.9,
                                chunk=chunk, **dims)
    assert _rel(oc, o) < 1e-12
    assert _rel(Sc, S) < 1e-12


def test_replay_reproduces_every_accepted_prefix(oracle_mod):
    """Replaying the first n captured factors from S0 gives the state the
    recurrence reaches after n tokens, for every n, and the final state at n=T."""
    rng = np.random.default_rng(30)
    T, Hk, Hv, dk, dv = 7, 2, 4, 6, 5
    q, k, v, a, b, S0 = _rand_case(rng, T, Hk, Hv, dk, dv)
    dims = dict(B=1, Hk=Hk, Hv=Hv, dk=dk, dv=dv)
    _, S_full, su = oracle_mod.recurrent(q, k, v, a, b, initial_state=S0, T=T,
                                         capacity=T, capture_count=[T], **dims)
    for n in range(T + 1):
        _, S_n, _ = oracle_mod.recurrent(q[:n], k[:n], v[:n], a[:n], b[:n],
                                         initial_state=S0, T=n, **dims)
        S_r = oracle_mod.replay(S0, su, [n], capacity=T, **dims)
        assert _rel(S_r, S_n) < 1e-13, n
    assert _rel(oracle_mod.replay(S0, su, [T], capacity=T, **dims), S_full) < 1e-13


def test_key_head_sharing(oracle_mod):
    """Inverse GQA: with Hk = 2 and Hv = 6, value head h gives exactly what a
    single-head run with key/query head h // 3 gives."""
    rng = np.random.default_rng(40)
    T, Hk, Hv, dk, dv = 9, 2, 6, 4, 3
    q, k, v, a, b, S0 = _rand_case(rng, T, Hk, Hv, dk, dv)
    o, S, su = oracle_mod.recurrent(q, k, v, a, b, initial_state=S0, B=1, Hk=Hk,
                                    Hv=Hv, dk=dk, dv=dv, T=T, capacity=T,
                                    capture_count=[T])
    for h in range(Hv):
        hk = h // 3
        o1, S1, su1 = oracle_mod.recurrent(
            q[:, hk:hk + 1], k[:, hk:hk + 1], v[:, h:h + 1], a[:, h:h + 1],
            b[:, h:h + 1], initial_state=S0[:, h:h + 1], B=1, Hk=1, Hv=1,
            dk=dk, dv=dv, T=T, capacity=T, capture_count=[T])
        assert np.array_equal(o[:, h], o1[:, 0])
        assert np.array_equal(S[0, h], S1[0, 0])
        # decay of head h, key of head hk, delta of head h
        assert np.array_equal(su[0, :, h], su1[0, :, 0])
        assert np.array_equal(su[0, :, Hv + hk * dk:Hv + (hk + 1) * dk],
                              su1[0, :, 1:1 + dk])
        off = Hv + Hk * dk + h * dv
        assert np.array_equal(su[0, :, off:off + dv], su1[0, :, 1 + dk:])


# --- capture contract -------------------------------------------------------

def test_capture_clamp_prefix_and_inactive(oracle_mod):
    """Captured tokens are the first n_b = clamp(count, 0, min(capacity, T_b));
    decay and key are the inputs themselves; slots >= n_b are untouched while
    active; the inactive run zeroes the whole output."""
    rng = np.random.default_rng(50)
    lengths = [5, 5, 2, 6]
    counts = [-1, 3, 100, 4]
    cap = 4
    Hk, Hv, dk, dv = 1, 2, 3, 2
    T = sum(lengths)
    q, k, v, a, b, _ = _rand_case(rng, T, Hk, Hv, dk, dv)
    cu = np.concatenate([[0], np.cumsum(lengths)])
    slot = Hv + Hk * dk + Hv * dv
    sentinel = np.full((4, cap, slot), 12345.0)
    dims = dict(B=4, Hk=Hk, Hv=Hv, dk=dk, dv=dv, cu_seqlens=cu)
    o, S, su = oracle_mod.recurrent(q, k, v, a, b, capacity=cap,
                                    capture_count=counts,
                                    state_update=sentinel.copy(), **dims)
    n = oracle_mod.capture_counts_clamped(counts, cap, lengths)
    assert n == [0, 3, 2, 4]
    for r in range(4):
        for t in range(cap):
            if t < n[r]:
                tok = cu[r] + t
                assert np.array_equal(su[r, t, :Hv], a[tok])
                assert np.array_equal(su[r, t, Hv:Hv + dk], k[tok, 0])
            else:
                assert np.all(su[r, t] == 12345.0)
    o2, S2, su0 = oracle_mod.recurrent(q, k, v, a, b, capacity=cap,
                                       capture_count=counts, active=False,
                                       state_update=sentinel.copy(), **dims)
    assert np.all(su0 == 0.0)
    assert np.array_equal(o2, o) and np.array_equal(S2, S)


# --- speculative loop (replay + verify) -----------------------------------

@pytest.mark.parametrize("accepted", [[0, 0], [2, 4], [4, 4], [4, 1]])
def test_speculative_loop_matches_non_speculative_run(oracle_mod, accepted):
    """"DFlash2 Prerequisite" (onnxruntime PR 32767): with full, partial and
    zero acceptance, verify-with-capture then replay-and-verify must give the
    output and state of running the accepted tokens and the next drafts
    straight through the recurrence.  Two rows with different acceptance;
    ragged second drafts (one row has none)."""
    rng = np.random.default_rng(60)
    B, Hk, Hv, dk, dv, T1 = 2, 1, 2, 5, 4, 4
    lens2 = [3, 0]
    q, k, v, a, b, _ = _rand_case(rng, B * T1 + sum(lens2), Hk, Hv, dk, dv)
    S0 = 0.3 * rng.standard_normal((B, Hv, dv, dk))
    dims = dict(B=B, Hk=Hk, Hv=Hv, dk=dk, dv=dv)
    X = slice(0, B * T1)
    Y = slice(B * T1, None)
    # verify pass 1: T1 drafts per row, all captured
    _, _, su1 = oracle_mod.recurrent(q[X], k[X], v[X], a[X], b[X], T=T1,
                                     initial_state=S0, capacity=T1,
                                     capture_count=[T1] * B, **dims)
    cu2 = np.concatenate([[0], np.cumsum(lens2)])
    o2, S_commit, S_draft, su2 = oracle_mod.replay_verify(
        q[Y], k[Y], v[Y], a[Y], b[Y], cu_seqlens=cu2, state_in=S0,
        prev_state_update=su1, prev_capacity=T1, accepted_count=accepted,
        capacity=4, capture_count=[4, 4], **dims)
    for r in range(B):
        m = accepted[r]
        # non-speculative: accepted tokens then the new drafts, one row
        toks = list(range(r * T1, r * T1 + m)) + [B * T1 + cu2[r] + i for i in range(lens2[r])]
        one = dict(B=1, Hk=Hk, Hv=Hv, dk=dk, dv=dv)
        _, S_m, _ = oracle_mod.recurrent(q[toks[:m]], k[toks[:m]], v[toks[:m]],
                                         a[toks[:m]], b[toks[:m]], T=m,
                                         initial_state=S0[r:r + 1], **one)
        o_ns, S_ns, _ = oracle_mod.recurrent(q[toks], k[toks], v[toks], a[toks],
                                             b[toks], T=len(toks),
                                             initial_state=S0[r:r + 1], **one)
        assert _rel(S_commit[r], S_m[0]) < 1e-13
        assert _rel(S_draft[r], S_ns[0]) < 1e-13
        if lens2[r]:
            got = o2[cu2[r]:cu2[r + 1]]
            assert _rel(got, o_ns[m:]) < 1e-13


# --- chunk-boundary checkpoints -------------------------------------------

def test_prefix_checkpoints_match_the_chunked_form_and_resume(oracle_mod):
    """Checkpoint j is the state after (j + 1) * L tokens: it equals the
    independent chunked (UT/WY) formulation run over that prefix, resuming
    the recurrence from any checkpoint over the rest of the row gives the
    row's final state, and slots past floor(T_b / L) (or the capacity) stay
    undefined."""
    rng = np.random.default_rng(70)
    lengths = [37, 12, 50]
    Hk, Hv, dk, dv, L, cap = 1, 2, 4, 3, 8, 5
    T = sum(lengths)
    q, k, v, a, b, _ = _rand_case(rng, T, Hk, Hv, dk, dv)
    S0 = 0.3 * rng.standard_normal((3, Hv, dv, dk))
    cu = np.concatenate([[0], np.cumsum(lengths)])
    dims = dict(B=3, Hk=Hk, Hv=Hv, dk=dk, dv=dv)
    ck = oracle_mod.prefix_checkpoints(q, k, v, a, b, every=L, capacity=cap,
                                       cu_seqlens=cu, initial_state=S0, **dims)
    _, S_fin, _ = oracle_mod.recurrent(q, k, v, a, b, cu_seqlens=cu, initial_state=S0, **dims)
    one = dict(B=1, Hk=Hk, Hv=Hv, dk=dk, dv=dv)
    for r, tb in enumerate(lengths):
        n = min(cap, tb // L)
        assert np.all(np.isnan(ck[r, n:]))
        for j in range(n):
            t1 = cu[r] + (j + 1) * L
            _, Sc = oracle_mod.chunked(q[cu[r]:t1], k[cu[r]:t1], v[cu[r]:t1], a[cu[r]:t1],
                                       b[cu[r]:t1], T=t1 - cu[r], chunk=5,
                                       initial_state=S0[r:r + 1], **one)
            assert _rel(ck[r, j], Sc[0]) < 1e-12, (r, j)
            rest = slice(t1, cu[r + 1])
            _, S_res, _ = oracle_mod.recurrent(q[rest], k[rest], v[rest], a[rest], b[rest],
                                               T=cu[r + 1] - t1, initial_state=ck[r, j][None],
                                               **one)
            assert _rel(S_res[0], S_fin[r]) < 1e-12, (r, j)


# --- input conventions (front end) -----------------------------------------

def test_front_end_closed_forms(oracle_mod):
    """Normalised vectors have norm sqrt(s / (s + eps)), s = |x|^2; the log-
    decay round-trips; sigmoid(0) = 1/2 and sigmoid(x) + sigmoid(-x) = 1."""
    rng = np.random.default_rng(80)
    q = rng.standard_normal((5, 2, 7)) * 3.0
    k = rng.standard_normal((5, 2, 7)) * 0.4
    a = rng.uniform(0.6, 1.0, size=(5, 3))
    x = rng.standard_normal((5, 3))
    qn, kn, an, bn = oracle_mod.front_end(q, k, np.log(a), x, qk_l2norm=True, alpha_log=True,
                                          beta_logit=True)
    for raw, got in ((q, qn), (k, kn)):
        s = np.sum(raw * raw, axis=-1)
        assert np.allclose(np.linalg.norm(got, axis=-1), np.sqrt(s / (s + 1e-6)), rtol=1e-14)
        assert np.allclose(got / np.linalg.norm(got, axis=-1, keepdims=True),
                           raw / np.linalg.norm(raw, axis=-1, keepdims=True), rtol=1e-14)
    assert np.allclose(an, a, rtol=1e-15)
    _, _, _, b0 = oracle_mod.front_end(q, k, a, np.zeros((5, 3)), beta_logit=True)
    assert np.all(b0 == 0.5)
    _, _, _, bneg = oracle_mod.front_end(q, k, a, -x, beta_logit=True)
    assert np.allclose(bn + bneg, 1.0, rtol=1e-15)
    # without flags the inputs pass through unchanged
    q2, k2, a2, b2 = oracle_mod.front_end(q, k, a, x)
    assert np.array_equal(q2, q) and np.array_equal(a2, a) and np.array_equal(b2, x)


def test_front_end_composes_with_the_recurrence(oracle_mod):
    """Raw inputs in the layer's conventions -- q and k scaled by arbitrary
    per-token magnitudes, alpha as log-decay, beta as logits -- give, through
    the front end, the recurrence of the normalised inputs (to the eps effect)."""
    rng = np.random.default_rng(81)
    T, Hk, Hv, dk, dv = 9, 1, 2, 6, 4
    q, k, v, a, b, S0 = _rand_case(rng, T, Hk, Hv, dk, dv)
    mq = rng.uniform(0.5, 2.0, size=(T, Hk, 1))
    mk = rng.uniform(0.5, 2.0, size=(T, Hk, 1))
    dims = dict(B=1, Hk=Hk, Hv=Hv, dk=dk, dv=dv, T=T, initial_state=S0)
    o_ref, S_ref, _ = oracle_mod.recurrent(q, k, v, a, b, **dims)
    qf, kf, af, bf = oracle_mod.front_end(q * mq, k * mk, np.log(a), np.log(b / (1 - b)),
                                          qk_l2norm=True, alpha_log=True, beta_logit=True)
    o, S, _ = oracle_mod.recurrent(qf, kf, v, af, bf, **dims)
    assert _rel(o, o_ref) < 1e-5 and _rel(S, S_ref) < 1e-5
