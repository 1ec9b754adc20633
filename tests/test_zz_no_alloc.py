"""The allocation-free entry point against the regular one and the oracle.

gdn_prefill_chunked_noalloc serves callers that cannot allocate device
memory -- runtimes with their own memory planner that forbid hidden
allocations, and latency paths that must never enter the allocator.  It runs the same prefill
on the library's fixed device scratch buffer instead of a caller workspace.
Checked here: two calls in a row on the shared buffer (each against
gdn_prefill_chunked and against the fp64 oracle), the input-convention bits,
a problem that fills the buffer almost to its limit, a shape that needs no
scratch at all, and the rejection of a problem beyond the limit.  This file
is named to be collected last, so a run that stops at the first failure has
already run every other test.
"""
import ctypes
import os

import numpy as np
import pytest
import torch

from helpers import TOL, rel, to_dev

pytestmark = pytest.mark.gpu
THREADS = min(32, os.cpu_count() or 4)
DT = {"bf16": torch.bfloat16, "f16": torch.float16, "f32": torch.float32}
QK, ALOG, BLOG = 0x100, 0x200, 0x400


@pytest.fixture(scope="module")
def gdn():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from gated_deltanet_recurrence_02_gb300 import build, gdn as g
    build.build()
    g.lib()
    return g


def _noalloc_fn(L):
    fn = L.gdn_prefill_chunked_noalloc
    vp, i, f = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
    fn.argtypes = [vp] * 8 + [i, vp, vp] + [i] * 8 + [f, i, i, vp]
    fn.restype = ctypes.c_int
    return fn


def _call(fn, g, dims, B, T, cu, out, fs, dtq, dtg, chunk=64, scale=1.0):
    Hk, Hv, d = dims
    s0 = g["initial_state"]
    return fn(g["q"].data_ptr(), g["k"].data_ptr(), g["v"].data_ptr(), g["alpha"].data_ptr(),
              g["beta"].data_ptr(), cu.data_ptr() if cu is not None else None,
              s0.data_ptr() if s0 is not None else None, None,
              s0.shape[0] if s0 is not None else 0, fs.data_ptr(), out.data_ptr(), B, T, Hk, Hk,
              Hv, d, d, chunk, scale, dtq, dtg, torch.cuda.current_stream().cuda_stream)


def _run_both(gdn, oracle_mod, x, dt, chunk=64, conv=0, raw=False):
    """One noalloc call and one regular call on the same inputs; both against
    the oracle (through its front end for raw inputs)."""
    fn = _noalloc_fn(gdn.lib())
    g = to_dev(x)
    B = len(x.lengths)
    cu = g["cu_seqlens"] if len(set(x.lengths)) > 1 else None
    T = x.total_T if cu is not None else x.lengths[0]
    dims = (x.Hk, x.Hv, x.dk)
    sc = x.scale if raw else 1.0
    o_ref, s_ref = gdn.gdn_prefill_chunked(g["q"], g["k"], g["v"], g["alpha"], g["beta"], B=B,
                                           T=T, cu_seqlens=cu, initial_state=g["initial_state"],
                                           chunk=chunk, scale=sc, conventions=conv)
    out = torch.empty_like(g["v"])
    fs = torch.empty((B, x.Hv, x.dv, x.dk), dtype=torch.float32, device="cuda")
    st = _call(fn, g, dims, B, T, cu, out, fs, gdn._DT[DT[dt]] | (conv & QK),
               gdn._DT[x.alpha.dtype] | (conv & (ALOG | BLOG)), chunk=chunk, scale=sc)
    assert st == gdn.GDN_OK, gdn.status_string(st)
    torch.cuda.synchronize()
    assert gdn.gdn_device_errors() == 0
    q, k, a, b = x.q, x.k, x.alpha, x.beta
    if raw:
        q, k, a, b = oracle_mod.front_end(q, k, a, b, qk_l2norm=bool(conv & QK),
                                          alpha_log=bool(conv & ALOG),
                                          beta_logit=bool(conv & BLOG))
    ro, rS, _ = oracle_mod.recurrent(q, k, x.v, a, b, B=B, Hk=x.Hk, Hv=x.Hv, dk=x.dk, dv=x.dv,
                                     cu_seqlens=x.cu_seqlens, initial_state=x.initial_state,
                                     scale=sc, threads=THREADS)
    tol = TOL[DT[dt]]
    for got in ((out, fs), (o_ref, s_ref)):
        assert rel(got[0], ro) < tol and rel(got[1], rS) < tol
    # the two entry points run the same kernels on the same inputs
    assert rel(out, o_ref.cpu().double().numpy()) < tol
    assert rel(fs, s_ref.cpu().double().numpy()) < tol
    return out, fs


def test_noalloc_prefill_two_calls_in_a_row(gdn, oracle_mod):
    from gated_deltanet_recurrence_02_gb300.inputs import make_inputs
    # ragged bf16 rows, then one fp16 row, on the shared scratch
    for seed, lengths, dt in ((11, [300, 333], "bf16"), (12, [512], "f16")):
        x = make_inputs(seed, lengths=lengths, Hk=16, Hv=32, dk=128, dv=128, dtype_qkv=dt,
                        dtype_gate="f32")
        _run_both(gdn, oracle_mod, x, dt)


def test_noalloc_prefill_input_conventions(gdn, oracle_mod):
    """The dtype codes carry GDN_QK_L2NORM and the gate bits, exactly as for
    gdn_prefill_chunked; raw inputs go through the oracle's front end."""
    from gated_deltanet_recurrence_02_gb300.inputs import make_raw_inputs
    x = make_raw_inputs(14, lengths=[200, 77], Hk=2, Hv=4, dk=128, dv=128, dtype_qkv="bf16",
                        dtype_gate="bf16")
    _run_both(gdn, oracle_mod, x, "bf16", conv=QK | ALOG | BLOG, raw=True)


def test_noalloc_prefill_near_the_limit(gdn, oracle_mod):
    """The longest single row (a multiple of the chunk) at Hk=16, Hv=32 whose
    workspace still fits the fixed buffer: it fills the buffer almost
    completely, and the next chunk would not fit."""
    from gated_deltanet_recurrence_02_gb300.inputs import make_inputs
    size = lambda T: gdn.gdn_prefill_workspace_size(1, T, 16, 32, 128, 128, 64,  # noqa: E731
                                                    torch.bfloat16)
    T = 64
    while size(T + 64) <= gdn.NOALLOC_SCRATCH_BYTES:
        T += 64
    assert size(T) <= gdn.NOALLOC_SCRATCH_BYTES < size(T + 64)
    assert size(T) > 0.9 * gdn.NOALLOC_SCRATCH_BYTES
    x = make_inputs(15, lengths=[T], Hk=16, Hv=32, dk=128, dv=128, dtype_qkv="bf16",
                    dtype_gate="f32")
    _run_both(gdn, oracle_mod, x, "bf16")


def test_noalloc_prefill_shape_without_scratch(gdn, oracle_mod):
    """fp32 inputs at d=32, chunk 16 take the CUDA-core path, which needs no
    scratch: the call passes none."""
    from gated_deltanet_recurrence_02_gb300.inputs import make_inputs
    assert gdn.gdn_prefill_workspace_size(2, 50, 1, 2, 32, 32, 16, torch.float32, True) == 0
    x = make_inputs(16, lengths=[50, 17], Hk=1, Hv=2, dk=32, dv=32, dtype_qkv="f32",
                    dtype_gate="f32")
    _run_both(gdn, oracle_mod, x, "f32", chunk=16)


def test_noalloc_rejects_problems_beyond_its_scratch(gdn):
    from gated_deltanet_recurrence_02_gb300.inputs import make_inputs
    fn = _noalloc_fn(gdn.lib())
    T = 64
    while gdn.gdn_prefill_workspace_size(1, T, 16, 32, 128, 128, 64, torch.bfloat16) <= \
            gdn.NOALLOC_SCRATCH_BYTES:
        T += 64
    x = make_inputs(13, lengths=[T], Hk=16, Hv=32, dk=128, dv=128, dtype_qkv="bf16",
                    dtype_gate="f32")
    g = to_dev(x)
    out = torch.zeros_like(g["v"])
    fs = torch.zeros((1, 32, 128, 128), dtype=torch.float32, device="cuda")
    st = _call(fn, g, (16, 32, 128), 1, T, None, out, fs, gdn.GDN_BF16, gdn.GDN_F32)
    assert st == 7  # GDN_ERR_WORKSPACE, returned before anything is launched
    torch.cuda.synchronize()
    assert bool((out == 0).all().item()) and bool((fs == 0).all().item())
