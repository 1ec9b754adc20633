"""The bounded-wait failure path, driven on the GPU without a fault.

Every kernel bounds its waits on another warp's work; a wait that runs out
raises GDN_DEVERR_TIMEOUT, the CTA still waits (with the full limit) for its
own copies in flight, frees its tensor memory and exits.  A test lowers the
limit below a microsecond, so the first hand-off a consumer finds incomplete
(its first pipeline stage, whose copies were issued a moment earlier) gives
up.  Nothing hangs and nothing faults: the context must stay usable, and the
same call with the default limit must then match the oracle.
"""
import ctypes

import pytest
import torch

from helpers import TOL, rel, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def gdn():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from gated_deltanet_recurrence_02_gb300 import build, gdn as g
    build.build()
    g.lib()
    yield g
    g.gdn_set_wait_limit_ns(0)


def _device_errors(gdn):
    """(status, flags) of the C call gdn_device_errors."""
    flags = ctypes.c_uint32(0)
    st = gdn.lib().gdn_device_errors(torch.cuda.current_stream().cuda_stream, ctypes.byref(flags))
    return st, flags.value


def _timed_out_then_recovers(gdn, run, check):
    assert _device_errors(gdn) == (0, 0)
    gdn.gdn_set_wait_limit_ns(1)
    try:
        run()
        st, flags = _device_errors(gdn)
    finally:
        gdn.gdn_set_wait_limit_ns(0)
    assert flags & gdn.GDN_DEVERR_TIMEOUT, "the shortened wait did not run out"
    assert st == 6  # GDN_ERR_TIMEOUT
    # the context still works: the same call with the default limit is correct
    res = run()
    assert _device_errors(gdn) == (0, 0)
    check(res)


def test_decode_wait_runs_out_and_recovers(gdn, oracle_mod):
    from gated_deltanet_recurrence_02_gb300.inputs import make_inputs
    x = make_inputs(4401, lengths=[1, 1, 1], Hk=2, Hv=4, dk=128, dv=128, dtype_qkv="bf16",
                    dtype_gate="bf16")
    g = to_dev(x)

    def run():
        o, S, _ = gdn.gdn_recurrent_capture(g["q"], g["k"], g["v"], g["alpha"], g["beta"], B=3,
                                            T=1, initial_state=g["initial_state"])
        return o, S

    def check(res):
        ro, rS, _ = oracle_mod.recurrent(x.q, x.k, x.v, x.alpha, x.beta, B=3, Hk=2, Hv=4,
                                         dk=128, dv=128, T=1, initial_state=x.initial_state)
        assert rel(res[0], ro) < TOL[torch.bfloat16] and rel(res[1], rS) < TOL[torch.bfloat16]

    _timed_out_then_recovers(gdn, run, check)


def test_tensor_core_prefill_wait_runs_out_and_recovers(gdn, oracle_mod):
    from gated_deltanet_recurrence_02_gb300.inputs import make_inputs
    x = make_inputs(4402, lengths=[130], Hk=1, Hv=2, dk=128, dv=128, dtype_qkv="bf16",
                    dtype_gate="f32")
    g = to_dev(x)

    def run():
        return gdn.gdn_prefill_chunked(g["q"], g["k"], g["v"], g["alpha"], g["beta"], B=1, T=130,
                                       initial_state=g["initial_state"], chunk=64)

    def check(res):
        ro, rS, _ = oracle_mod.recurrent(x.q, x.k, x.v, x.alpha, x.beta, B=1, Hk=1, Hv=2,
                                         dk=128, dv=128, T=130, initial_state=x.initial_state)
        assert rel(res[0], ro) < TOL[torch.bfloat16] and rel(res[1], rS) < TOL[torch.bfloat16]

    _timed_out_then_recovers(gdn, run, check)
