"""The allocation-free prefill entry point against the regular one.

gdn_prefill_chunked_noalloc serves callers that cannot allocate device
memory -- runtimes with their own memory planner that forbid hidden
allocations, code running while a stream is captured into a CUDA graph, and
latency paths that must never enter the allocator.  It runs the same prefill
on the library's fixed device scratch buffer instead of a caller workspace.
This file is named to be collected last, so a run that stops at the first
failure has already run every other test.
"""
import ctypes

import pytest
import torch

from helpers import TOL, rel, to_dev

pytestmark = pytest.mark.gpu

DT = {"bf16": torch.bfloat16, "f16": torch.float16}


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


def _call(fn, g, B, T, cu, out, fs, dtq, dtg):
    return fn(g["q"].data_ptr(), g["k"].data_ptr(), g["v"].data_ptr(), g["alpha"].data_ptr(),
              g["beta"].data_ptr(), cu.data_ptr() if cu is not None else None,
              g["initial_state"].data_ptr(), None, g["initial_state"].shape[0], fs.data_ptr(),
              out.data_ptr(), B, T, 16, 16, 32, 128, 128, 64, 1.0, dtq, dtg,
              torch.cuda.current_stream().cuda_stream)


def test_noalloc_prefill_matches_regular_entry_point(gdn):
    from gated_deltanet_recurrence_02_gb300.inputs import make_inputs
    fn = _noalloc_fn(gdn.lib())
    # two calls in a row on the shared scratch: ragged bf16 rows, then one fp16 row
    for seed, lengths, dt in ((11, [300, 333], "bf16"), (12, [512], "f16")):
        x = make_inputs(seed, lengths=lengths, Hk=16, Hv=32, dk=128, dv=128,
                        dtype_qkv=dt, dtype_gate="f32")
        g = to_dev(x)
        B = len(lengths)
        cu = g["cu_seqlens"] if len(set(lengths)) > 1 else None
        T = x.total_T if cu is not None else lengths[0]
        o_ref, s_ref = gdn.gdn_prefill_chunked(g["q"], g["k"], g["v"], g["alpha"], g["beta"],
                                               B=B, T=T, cu_seqlens=cu,
                                               initial_state=g["initial_state"], chunk=64)
        out = torch.empty_like(g["v"])
        fs = torch.empty((B, 32, 128, 128), dtype=torch.float32, device="cuda")
        st = _call(fn, g, B, T, cu, out, fs, gdn._DT[DT[dt]], gdn.GDN_F32)
        assert st == gdn.GDN_OK, gdn.status_string(st)
        torch.cuda.synchronize()
        assert rel(out, o_ref.cpu().double().numpy()) < TOL[DT[dt]]
        assert rel(fs, s_ref.cpu().double().numpy()) < TOL[DT[dt]]
        assert gdn.gdn_device_errors() == 0


def test_noalloc_rejects_problems_beyond_its_scratch(gdn):
    from gated_deltanet_recurrence_02_gb300.inputs import make_inputs
    fn = _noalloc_fn(gdn.lib())
    x = make_inputs(13, lengths=[2048], Hk=16, Hv=32, dk=128, dv=128, dtype_qkv="bf16",
                    dtype_gate="f32")
    g = to_dev(x)
    assert gdn.gdn_prefill_workspace_size(1, 2048, 16, 32, 128, 128, 64, torch.bfloat16) > \
        gdn.NOALLOC_SCRATCH_BYTES
    out = torch.zeros_like(g["v"])
    fs = torch.zeros((1, 32, 128, 128), dtype=torch.float32, device="cuda")
    st = _call(fn, g, 1, 2048, None, out, fs, gdn.GDN_BF16, gdn.GDN_F32)
    assert st == 7  # GDN_ERR_WORKSPACE, returned before anything is launched
    torch.cuda.synchronize()
    assert bool((out == 0).all().item()) and bool((fs == 0).all().item())
