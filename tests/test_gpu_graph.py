"""The decode step and the fused speculative step captured into CUDA graphs
and replayed with new inputs, against the same calls run eagerly (bit for
bit: the same kernels on the same data).

Source: "[WebGPU EP] adds state update capacity support for GatedDeltaNet"
(onnxruntime PR 32767), "Changes": state_update_active = 0 clears the whole
output -- here a device scalar, so that one captured graph serves both
settings; "[WebGPU] Graph capture support for KV-shared decoder models"
(onnxruntime PR 29000), item 2: buffers referenced by captured work must
outlive it (the caller owns every buffer; the library allocates nothing).
"""
import pytest
import torch

pytestmark = pytest.mark.gpu
I32 = torch.int32


@pytest.fixture(scope="module")
def gdn():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from gated_deltanet_recurrence_02_gb300 import build, gdn as g
    build.build()
    g.lib()
    return g


def _tokens(x, B, steps):
    """Per step, every row's token as a [B, ...] device tensor (step-major)."""
    out = []
    for t in range(steps):
        out.append({n: getattr(x, n).view(B, steps, *getattr(x, n).shape[1:])[:, t].contiguous().cuda()
                    for n in ("q", "k", "v", "alpha", "beta")})
    return out


def _capture(fn):
    """fn() once outside capture (first-call set-up), then captured."""
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        fn()
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    return g


def test_decode_step_graph_and_device_active_flag(gdn):
    from gated_deltanet_recurrence_02_gb300.inputs import make_inputs
    B, Hk, Hv, d, cap, steps = 64, 2, 4, 128, 2, 3
    x = make_inputs(2100, lengths=[steps] * B, Hk=Hk, Hv=Hv, dk=d, dv=d, dtype_qkv="bf16",
                    dtype_gate="bf16")
    toks = _tokens(x, B, steps)
    S0 = x.initial_state.cuda()
    counts = torch.tensor([1, 0] * (B // 2), dtype=I32, device="cuda")
    active = torch.ones(1, dtype=I32, device="cuda")
    slot = gdn.slot_width(Hk, Hv, d, d)
    # eager
    S_e, outs, caps = S0.clone(), [], []
    for t in range(steps):
        o, _, su = gdn.gdn_recurrent_capture(*(toks[t][n] for n in ("q", "k", "v", "alpha", "beta")),
                                             B=B, T=1, initial_state=S_e, final_state=S_e,
                                             state_update_capacity=cap, capture_count=counts,
                                             state_update_active=active)
        outs.append(o.clone())
        caps.append(su.clone())
    # graph over static buffers
    inp = {n: torch.empty_like(v) for n, v in toks[0].items()}
    S_g = S0.clone()
    out_g = torch.empty_like(inp["v"])
    su_g = torch.full((B, cap, slot), 7.0, dtype=torch.float32, device="cuda")

    def call():
        gdn.gdn_recurrent_capture(inp["q"], inp["k"], inp["v"], inp["alpha"], inp["beta"], B=B, T=1,
                                  initial_state=S_g, final_state=S_g, out=out_g,
                                  state_update_capacity=cap, capture_count=counts,
                                  state_update_active=active, state_update=su_g)

    for n in inp:
        inp[n].copy_(toks[0][n])
    g = _capture(call)
    S_g.copy_(S0)
    rows = counts.bool()
    for t in range(steps):
        for n in inp:
            inp[n].copy_(toks[t][n])
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(out_g, outs[t]), t
        assert torch.equal(su_g[rows, 0], caps[t][rows, 0]), t
    assert torch.equal(S_g, S_e)
    # the same graph, capture switched off on the device: the whole buffer is cleared
    active.fill_(0)
    g.replay()
    torch.cuda.synchronize()
    assert bool(torch.all(su_g == 0).item())


def test_speculative_loop_as_two_alternating_graphs(gdn):
    """verify (eager), then replay + verify steps from two captured graphs that
    alternate the capture buffers; acceptance counts and drafts change between
    replays through device buffers."""
    from gated_deltanet_recurrence_02_gb300.inputs import accepted_counts, make_inputs
    B, Hk, Hv, d, T, n_steps = 32, 2, 4, 128, 4, 4
    xs = [make_inputs(2200 + s, lengths=[T] * B, Hk=Hk, Hv=Hv, dk=d, dv=d, dtype_qkv="bf16",
                      dtype_gate="bf16", zero_state=(s > 0)) for s in range(n_steps)]
    drafts = [{n: getattr(x, n).cuda() for n in ("q", "k", "v", "alpha", "beta")} for x in xs]
    acc = [accepted_counts(2300 + s, B, T).cuda() for s in range(n_steps)]
    full = torch.full((B,), T, dtype=I32, device="cuda")
    S0 = xs[0].initial_state.cuda()
    slot = gdn.slot_width(Hk, Hv, d, d)

    def run_eager():
        S = S0.clone()
        bufs = [torch.empty((B, T, slot), dtype=torch.float32, device="cuda") for _ in range(2)]
        outs = []
        o, _, _ = gdn.gdn_recurrent_capture(*(drafts[0][n] for n in ("q", "k", "v", "alpha", "beta")),
                                            B=B, T=T, initial_state=S, want_final_state=False,
                                            state_update_capacity=T, capture_count=full,
                                            state_update=bufs[0])
        outs.append(o.clone())
        for s in range(1, n_steps):
            o, _, _, _ = gdn.gdn_replay_verify(*(drafts[s][n] for n in ("q", "k", "v", "alpha", "beta")),
                                               B=B, T=T, state_in=S, state_out=S,
                                               prev_state_update=bufs[(s - 1) % 2], prev_capacity=T,
                                               accepted_count=acc[s - 1], state_update_capacity=T,
                                               capture_count=full, state_update=bufs[s % 2])
            outs.append(o.clone())
        return S, outs

    S_e, outs_e = run_eager()
    # graphs: static drafts, acceptance and output buffers
    inp = {n: torch.empty_like(v) for n, v in drafts[0].items()}
    acc_in = torch.empty(B, dtype=I32, device="cuda")
    S_g = S0.clone()
    out_g = torch.empty_like(inp["v"])
    bufs = [torch.empty((B, T, slot), dtype=torch.float32, device="cuda") for _ in range(2)]

    def step(prev, new):
        gdn.gdn_replay_verify(inp["q"], inp["k"], inp["v"], inp["alpha"], inp["beta"], B=B, T=T,
                              state_in=S_g, state_out=S_g, prev_state_update=bufs[prev],
                              prev_capacity=T, accepted_count=acc_in, out=out_g,
                              state_update_capacity=T, capture_count=full, state_update=bufs[new])

    acc_in.zero_()  # the warm-up before capture replays nothing...
    for n in inp:   # ...and runs real drafts (its results are discarded below)
        inp[n].copy_(drafts[1][n])
    graphs = [_capture(lambda: step(0, 1)), _capture(lambda: step(1, 0))]
    S_g.copy_(S0)
    gdn.gdn_recurrent_capture(*(drafts[0][n] for n in ("q", "k", "v", "alpha", "beta")), B=B, T=T,
                              initial_state=S_g, want_final_state=False, state_update_capacity=T,
                              capture_count=full, state_update=bufs[0])
    for s in range(1, n_steps):
        for n in inp:
            inp[n].copy_(drafts[s][n])
        acc_in.copy_(acc[s - 1])
        graphs[(s - 1) % 2].replay()
        torch.cuda.synchronize()
        assert torch.equal(out_g, outs_e[s]), s
    assert torch.equal(S_g, S_e)


@pytest.mark.parametrize("path", ["tensor_core", "cuda_core"])
def test_prefill_graph_replay(gdn, path):
    """The chunked prefill (packed rows; on the tensor-core path the carry
    kernel is a programmatic dependent of the chunk-parallel one) captured
    into a CUDA graph over static buffers and replayed with new inputs: bit
    for bit the eager calls."""
    from gated_deltanet_recurrence_02_gb300.inputs import make_inputs
    d, dt, chunk = (128, "bf16", 64) if path == "tensor_core" else (64, "f32", 32)
    lengths = [150, 64, 0, 37]
    B = len(lengths)
    xs = [make_inputs(2400 + i, lengths=lengths, Hk=2, Hv=4, dk=d, dv=d, dtype_qkv=dt,
                      dtype_gate=dt) for i in range(3)]
    names = ("q", "k", "v", "alpha", "beta", "initial_state")
    cu = xs[0].cu_seqlens.cuda()
    T = int(xs[0].cu_seqlens[-1])
    ws_bytes = gdn.gdn_prefill_workspace_size(B, T, 2, 4, d, d, chunk, xs[0].q.dtype, varlen=True)
    ws = torch.empty(max(ws_bytes, 16), dtype=torch.uint8, device="cuda")
    # eager
    ref = []
    for x in xs:
        g = {n: getattr(x, n).cuda() for n in names}
        o, fs = gdn.gdn_prefill_chunked(g["q"], g["k"], g["v"], g["alpha"], g["beta"], B=B,
                                        cu_seqlens=cu, initial_state=g["initial_state"],
                                        chunk=chunk, workspace=ws)
        torch.cuda.synchronize()
        ref.append((o.clone(), fs.clone()))
    # graph over static buffers
    inp = {n: getattr(xs[0], n).cuda() for n in names}
    out = torch.empty_like(inp["v"])
    fs = torch.empty_like(inp["initial_state"])

    def call():
        gdn.gdn_prefill_chunked(inp["q"], inp["k"], inp["v"], inp["alpha"], inp["beta"], B=B,
                                cu_seqlens=cu, initial_state=inp["initial_state"], final_state=fs,
                                out=out, chunk=chunk, workspace=ws)

    gr = _capture(call)
    for x, (ro, rfs) in zip(xs, ref):
        for n in names:
            inp[n].copy_(getattr(x, n))
        gr.replay()
        torch.cuda.synchronize()
        assert torch.equal(out, ro) and torch.equal(fs, rfs)
    assert gdn.gdn_device_errors() == 0
