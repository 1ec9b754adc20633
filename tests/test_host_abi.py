"""Host-side checks of the C ABI: the library loads, exports every entry
point that include/gdn.h declares, and rejects bad arguments before any
launch.  No GPU is touched: every call here fails validation first, and the
fake device addresses are never dereferenced."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    from gated_deltanet_recurrence_02_gb300 import build, gdn
    build.build()
    return gdn.lib()


def _declared():
    src = open(os.path.join(ROOT, "include", "gdn.h")).read()
    return sorted(set(re.findall(r"GDN_API\s+[\w\s\*]*?\b(gdn_\w+)\s*\(", src)))


def test_exports_every_declared_symbol(L):
    names = _declared()
    assert len(names) >= 6
    for n in names:
        assert hasattr(L, n), n


def test_status_strings(L):
    from gated_deltanet_recurrence_02_gb300 import gdn
    assert gdn.status_string(0) == "ok"
    for s in range(1, 8):
        assert gdn.status_string(s) not in ("ok", "unknown status")


A = 1 << 32  # fake, 16-byte aligned "device" addresses, far apart
GiB = 1 << 30


def rec(L, **kw):
    a = dict(q=A, k=A + GiB, v=A + 2 * GiB, alpha=A + 3 * GiB, beta=A + 4 * GiB, cu=None,
             s0=A + 5 * GiB, idx=None, n0=2, sf=A + 6 * GiB, out=A + 7 * GiB, B=2, T=8,
             Hq=2, Hk=2, Hv=6, dk=128, dv=128, scale=1.0, dtq=2, dtg=2, cap=4,
             cc=A + 8 * GiB, act=None, su=A + 9 * GiB)
    a.update(kw)
    return L.gdn_recurrent_capture(a["q"], a["k"], a["v"], a["alpha"], a["beta"], a["cu"],
                                   a["s0"], a["idx"], a["n0"], a["sf"], a["out"], a["B"],
                                   a["T"], a["Hq"], a["Hk"], a["Hv"], a["dk"], a["dv"],
                                   a["scale"], a["dtq"], a["dtg"], a["cap"], a["cc"],
                                   a["act"], a["su"], None)


def pre(L, **kw):
    a = dict(q=A, k=A + GiB, v=A + 2 * GiB, alpha=A + 3 * GiB, beta=A + 4 * GiB, cu=None,
             s0=A + 5 * GiB, idx=None, n0=1, sf=A + 6 * GiB, out=A + 7 * GiB, B=1, T=100,
             Hq=16, Hk=16, Hv=32, dk=128, dv=128, chunk=64, scale=1.0, dtq=2, dtg=0,
             ws=A + 8 * GiB, wsb=1 << 30)
    a.update(kw)
    return L.gdn_prefill_chunked(a["q"], a["k"], a["v"], a["alpha"], a["beta"], a["cu"],
                                 a["s0"], a["idx"], a["n0"], a["sf"], a["out"], a["B"],
                                 a["T"], a["Hq"], a["Hk"], a["Hv"], a["dk"], a["dv"],
                                 a["chunk"], a["scale"], a["dtq"], a["dtg"], a["ws"],
                                 a["wsb"], None)


def rep(L, **kw):
    a = dict(si=A, so=A + GiB, su=A + 2 * GiB, cap=4, acc=A + 3 * GiB, B=2, Hk=2, Hv=6,
             dk=128, dv=128)
    a.update(kw)
    return L.gdn_replay_state_updates(a["si"], a["so"], a["su"], a["cap"], a["acc"], a["B"],
                                      a["Hk"], a["Hv"], a["dk"], a["dv"], None)


def prc(L, **kw):
    a = dict(q=A, k=A + GiB, v=A + 2 * GiB, alpha=A + 3 * GiB, beta=A + 4 * GiB, cu=None,
             s0=A + 5 * GiB, idx=None, n0=1, sf=A + 6 * GiB, out=A + 7 * GiB, B=1, T=100,
             Hq=16, Hk=16, Hv=32, dk=128, dv=128, chunk=64, scale=1.0, dtq=2, dtg=0,
             ck=A + 9 * GiB, cap=2, every=1, ws=A + 8 * GiB, wsb=1 << 30)
    a.update(kw)
    return L.gdn_prefill_chunked_checkpoints(
        a["q"], a["k"], a["v"], a["alpha"], a["beta"], a["cu"], a["s0"], a["idx"], a["n0"],
        a["sf"], a["out"], a["B"], a["T"], a["Hq"], a["Hk"], a["Hv"], a["dk"], a["dv"],
        a["chunk"], a["scale"], a["dtq"], a["dtg"], a["ck"], a["cap"], a["every"], a["ws"],
        a["wsb"], None)


def pcap(L, **kw):
    a = dict(q=A, k=A + GiB, v=A + 2 * GiB, alpha=A + 3 * GiB, beta=A + 4 * GiB, cu=None,
             s0=A + 5 * GiB, idx=None, n0=1, sf=A + 6 * GiB, out=A + 7 * GiB, B=1, T=100,
             Hq=16, Hk=16, Hv=32, dk=128, dv=128, chunk=64, scale=1.0, dtq=2, dtg=0,
             cap=4, cc=A + 9 * GiB, act=None, su=A + 10 * GiB, ws=A + 8 * GiB, wsb=1 << 30)
    a.update(kw)
    return L.gdn_prefill_chunked_capture(
        a["q"], a["k"], a["v"], a["alpha"], a["beta"], a["cu"], a["s0"], a["idx"], a["n0"],
        a["sf"], a["out"], a["B"], a["T"], a["Hq"], a["Hk"], a["Hv"], a["dk"], a["dv"],
        a["chunk"], a["scale"], a["dtq"], a["dtg"], a["cap"], a["cc"], a["act"], a["su"],
        a["ws"], a["wsb"], None)


def rv(L, **kw):
    a = dict(q=A, k=A + GiB, v=A + 2 * GiB, alpha=A + 3 * GiB, beta=A + 4 * GiB, cu=None,
             si=A + 5 * GiB, so=A + 5 * GiB, psu=A + 6 * GiB, pcap=4, acc=A + 7 * GiB,
             sf=None, out=A + 8 * GiB, B=2, T=4, Hq=2, Hk=2, Hv=6, dk=128, dv=128,
             scale=1.0, dtq=2, dtg=2, cap=4, cc=A + 9 * GiB, act=None, su=A + 10 * GiB)
    a.update(kw)
    return L.gdn_replay_verify(a["q"], a["k"], a["v"], a["alpha"], a["beta"], a["cu"],
                               a["si"], a["so"], a["psu"], a["pcap"], a["acc"], a["sf"],
                               a["out"], a["B"], a["T"], a["Hq"], a["Hk"], a["Hv"], a["dk"],
                               a["dv"], a["scale"], a["dtq"], a["dtg"], a["cap"], a["cc"],
                               a["act"], a["su"], None)


INVALID, UNSUP, ALIAS, ALIGN, WS = 1, 2, 3, 4, 7


@pytest.mark.parametrize("kw,code", [
    (dict(Hq=1), INVALID),                   # Hq != Hk
    (dict(Hv=5), INVALID),                   # Hv % Hk != 0
    (dict(B=-1), INVALID),
    (dict(T=-3), INVALID),
    (dict(cap=-1), INVALID),
    (dict(cc=None), INVALID),                # capacity > 0 needs capture_count
    (dict(su=None), INVALID),                # ... and the output buffer
    (dict(q=None), INVALID),
    (dict(dtq=7), INVALID),
    (dict(dk=96), UNSUP),
    (dict(dv=256), UNSUP),
    (dict(q=A + 8), ALIGN),
    (dict(su=A + 9 * GiB + 4), ALIGN),
    (dict(cc=A + 8 * GiB + 2), ALIGN),
    (dict(out=A + 16), ALIAS),               # out overlaps q
    (dict(su=A + 7 * GiB + 64), ALIAS),      # capture overlaps out
    (dict(sf=A + 5 * GiB + 4096), ALIAS),    # partial overlap with the initial state
    (dict(sf=A + 5 * GiB, idx=A + 10 * GiB), ALIAS),  # in place with shared snapshots
    (dict(s0=None, idx=A + 10 * GiB), INVALID),
    (dict(n0=1), INVALID),                   # fewer initial states than rows
])
def test_recurrent_rejects(L, kw, code):
    assert rec(L, **kw) == code


@pytest.mark.parametrize("kw,code", [
    (dict(chunk=48), UNSUP),
    (dict(chunk=128), UNSUP),
    (dict(Hq=8), INVALID),
    (dict(dk=16), UNSUP),
    (dict(alpha=A + 3 * GiB + 8), ALIGN),
    (dict(out=A + 2 * GiB), ALIAS),          # out is v
    (dict(sf=A + 7 * GiB + 128), ALIAS),     # final state overlaps out
    (dict(dtg=3), INVALID),
    (dict(ws=None, wsb=0), WS),              # tensor-core path needs its workspace
    (dict(wsb=1024), WS),
    (dict(ws=A + 7 * GiB + 1024), ALIAS),    # workspace overlaps out
])
def test_prefill_rejects(L, kw, code):
    assert pre(L, **kw) == code


@pytest.mark.parametrize("kw,code", [
    (dict(cap=-2), INVALID),
    (dict(Hv=7), INVALID),
    (dict(dk=48), UNSUP),
    (dict(so=A + 16), ALIAS),                # partial in-place overlap
    (dict(so=A + 2 * GiB), ALIAS),           # output over the factors
    (dict(si=A + 4), ALIGN),
    (dict(acc=None), INVALID),
])
def test_replay_rejects(L, kw, code):
    assert rep(L, **kw) == code


@pytest.mark.parametrize("kw,code", [
    (dict(pcap=-1), INVALID),
    (dict(acc=None), INVALID),               # replay needs the acceptance counts
    (dict(psu=None), INVALID),               # ... and the previous capture
    (dict(so=None), INVALID),                # the committed state is required
    (dict(cc=None), INVALID),
    (dict(Hv=5), INVALID),
    (dict(dk=80), UNSUP),
    (dict(psu=A + 6 * GiB + 4), ALIGN),
    (dict(acc=A + 7 * GiB + 2), ALIGN),
    (dict(so=A + 5 * GiB + 512), ALIAS),     # partial overlap with state_in
    (dict(su=A + 6 * GiB + 1024), ALIAS),    # new capture over the previous one
    (dict(sf=A + 5 * GiB), ALIAS),           # draft final state over the committed state
    (dict(so=A + 8 * GiB), ALIAS),           # committed state over out
    (dict(out=A + 2 * GiB), ALIAS),          # out is v
])
def test_replay_verify_rejects(L, kw, code):
    assert rv(L, **kw) == code


@pytest.mark.parametrize("kw,code", [
    (dict(cap=-1), INVALID),
    (dict(every=0), INVALID),
    (dict(ck=None), INVALID),                # capacity > 0 needs the buffer
    (dict(ck=A + 9 * GiB + 8), ALIGN),
    (dict(ck=A + 7 * GiB + 4096), ALIAS),    # checkpoints over out
    (dict(ck=A + 8 * GiB), ALIAS),           # checkpoints over the workspace
    (dict(chunk=40), UNSUP),
])
def test_prefill_checkpoints_rejects(L, kw, code):
    assert prc(L, **kw) == code


def test_prefill_checkpoints_empty_and_without_slots(L):
    assert prc(L, B=0, T=0) == 0
    assert prc(L, B=0, T=0, ck=None, cap=0) == 0


@pytest.mark.parametrize("kw,code", [
    (dict(cap=-1), INVALID),
    (dict(cc=None), INVALID),
    (dict(su=None), INVALID),
    (dict(su=A + 10 * GiB + 4), ALIGN),
    (dict(cc=A + 9 * GiB + 2), ALIGN),
    (dict(su=A + 7 * GiB + 256), ALIAS),     # capture over out
    (dict(su=A + 8 * GiB), ALIAS),           # capture over the workspace
    (dict(chunk=48), UNSUP),
])
def test_prefill_capture_rejects(L, kw, code):
    assert pcap(L, **kw) == code


def test_prefill_capture_empty(L):
    assert pcap(L, B=0, T=0) == 0
    assert pcap(L, B=0, T=0, cap=0, cc=None, su=None) == 0


def test_replay_verify_accepts_plain_verify_and_no_replay_buffers(L):
    # prev_capacity == 0: nothing to replay, the factor pointers may be NULL;
    # B = 0 returns before any CUDA call.
    assert rv(L, pcap=0, psu=None, acc=None, B=0, T=0) == 0


def test_empty_batch_is_a_no_op(L):
    # B = 0 passes validation and returns before any CUDA call.
    assert rec(L, B=0, T=0) == 0
    assert pre(L, B=0, T=0) == 0
    assert rep(L, B=0) == 0
    assert rv(L, B=0, T=0) == 0


def test_workspace_size_query(L):
    big = L.gdn_prefill_workspace_size(1, 4100, 16, 32, 128, 128, 64, 2, 0)
    assert big == 65 * 32 * 41984  # tensor-core path: one record per (chunk, value head)
    assert L.gdn_prefill_workspace_size(2, 100, 1, 2, 32, 32, 16, 0, 0) == 0  # CUDA-core path
    # packed rows: a per-row chunk table and the carry's row order (4 (2 B + 1)
    # bytes, in 1 KB units) ahead of the records, which cover up to T / 64 + B chunks
    assert L.gdn_prefill_workspace_size(300, 6000, 2, 4, 128, 128, 64, 2, 1) == \
        3072 + (6000 // 64 + 300) * 4 * 41984
    assert L.gdn_prefill_workspace_size(-1, 4100, 16, 32, 128, 128, 64, 2, 0) == ctypes.c_size_t(-1).value


def test_workspace_size_accepts_the_prefill_dtype_code(L):
    """The dtype code a caller passes to the prefill (storage type plus the
    GDN_QK_L2NORM bit) gives the same workspace size as the bare type; a gate
    bit or an unknown bit in dtype_qkv is rejected."""
    QK, ALOG = 0x100, 0x200
    for B, T, varlen in ((1, 4100, 0), (300, 6000, 1), (2, 100, 0)):
        bare = L.gdn_prefill_workspace_size(B, T, 16, 32, 128, 128, 64, 2, varlen)
        assert L.gdn_prefill_workspace_size(B, T, 16, 32, 128, 128, 64, 2 | QK, varlen) == bare
    assert L.gdn_prefill_workspace_size(2, 100, 1, 2, 32, 32, 16, 0 | QK, 0) == 0
    bad = ctypes.c_size_t(-1).value
    assert L.gdn_prefill_workspace_size(1, 4100, 16, 32, 128, 128, 64, 2 | ALOG, 0) == bad
    assert L.gdn_prefill_workspace_size(1, 4100, 16, 32, 128, 128, 64, 2 | 0x800, 0) == bad


def test_binding_fails_loudly_without_library(monkeypatch, tmp_path):
    from gated_deltanet_recurrence_02_gb300 import build, gdn
    monkeypatch.setattr(build, "LIB", str(tmp_path / "missing.so"))
    monkeypatch.setattr(gdn, "_lib", None)
    with pytest.raises(RuntimeError, match="not built"):
        gdn.lib()


def test_convention_bits_are_validated(L):
    """GDN_QK_L2NORM belongs to dtype_qkv, the gate bits to dtype_gate; any
    other bit is an invalid argument (checked before anything is launched)."""
    QK, ALOG, BLOG = 0x100, 0x200, 0x400
    assert rec(L, dtq=2 | ALOG) == INVALID
    assert rec(L, dtg=2 | QK) == INVALID
    assert rec(L, dtq=2 | 0x800) == INVALID
    assert pre(L, dtg=0 | QK) == INVALID
    assert rv(L, dtq=2 | BLOG) == INVALID
    assert rec(L, B=0, T=0, dtq=2 | QK, dtg=2 | ALOG | BLOG) == 0
    assert pre(L, B=0, T=0, dtq=2 | QK, dtg=0 | ALOG | BLOG) == 0
