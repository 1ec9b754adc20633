#!/usr/bin/env python
"""Benchmark of the gated delta-rule hot path on one GB300.

One step is one pass of the whole path over one batch of synthetic input:
  1. chunked prefill     B=1, T=4100, Hk=16, Hv=32, dk=dv=128, chunk 64, bf16
                         q/k/v, fp32 alpha/beta, random fp32 initial state;
  2. decode with capture B=256 rows, 64 sequential single-token calls, same
                         heads, bf16 q/k/v/alpha/beta, the fp32 state updated
                         in place in HBM, capacity 4, capture_count ~ U{0..4};
  3. replay              the decode state, capacity 4, accepted ~ U{0..4},
                         written to a separate output state;
  4. speculative step    B=256: one fused replay + verify launch -- replay of
                         the accepted prefix (U{0..4}) of a 4-slot capture,
                         then 4 draft tokens per row with capture, the
                         committed state in place.
The headline `value` is the decode phase's state throughput (algorithmic
bytes moved per second: state read + write, token vectors, outputs and
captured factors).  Prefill tokens/s, replay GB/s and the speculative
step's GB/s ride along in "prefill" / "replay" / "replay_verify"; the last
also reports the same step done unfused (replay, then verify) for
comparison, timed outside the step.  Inputs are resident in HBM before the timed region;
the decode state (512 MiB) is larger than L2, and the L2 is flushed (a
256 MiB write) before every prefill, outside the phase timers.

`--impl reference` times the fp64 CPU oracle on a bounded sample of the same
decode workload instead (rank 0 only).  Multi-GPU (torchrun): every rank runs
the same per-GPU workload on its own rows (weak scaling, no data-path
collective); only the barrier and the max/sum of timings cross ranks.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "GDN prefill tokens/s & decode state GB/s on 1 GB300, % of roofline"

# workload shapes
DEC = dict(B=256, steps=64, Hk=16, Hv=32, dk=128, dv=128, cap=4, seed=1004)
PRE = dict(T=4100, Hk=16, Hv=32, dk=128, dv=128, chunk=64, seed=1002)
REP_SEED = 2004
VER = dict(B=256, T=4, cap=4, seed=1005)  # speculative step: 4 drafts, capacity 4
CPU_SAMPLE_ROWS = 128  # oracle sample: 128 rows x 32 heads x 64 tokens


# ----------------------------------------------------------- distributed --

def dist_init():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    if ws <= 1:
        return 0, 1, 0
    import torch
    import torch.distributed as dist
    backend = "nccl" if torch.cuda.is_available() else "gloo"
    dist.init_process_group(backend=backend)
    return dist.get_rank(), dist.get_world_size(), int(os.environ.get("LOCAL_RANK", "0"))


def reduce_scalar(x: float, op: str, device=None) -> float:
    """max / sum of a per-rank scalar over all ranks (identity when alone)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64,
                     device=device if dist.get_backend() == "nccl" else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX if op == "max" else dist.ReduceOp.SUM)
    return float(t.item())


def barrier():
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized():
        dist.barrier()


# ---------------------------------------------------------------- clocks --

class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons while running."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    NAMES = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "100", "-f", self.path],
                stdout=subprocess.DEVNULL, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.3)

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        time.sleep(0.15)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        pw = [float(r[3]) for r in rows if r[3].replace(".", "").isdigit()]
        reasons = sorted({self.NAMES[i] for r in rows for i in range(4)
                          if r[5 + i].lower().startswith("active")})
        top = sorted(sm)[len(sm) // 2:] if sm else []  # samples under load
        return {"sm_mhz": statistics.median(top) if top else None,
                "sm_max_mhz": max(mx) if mx else None,
                "power_w_max": max(pw) if pw else None,
                "samples": len(rows), "reasons": reasons}


# ------------------------------------------------------------- workloads --

def decode_bytes(counts, d=DEC) -> int:
    """Algorithmic bytes of ONE decode call over all rows: fp32 state read and
    written, bf16 q, k, v, alpha, beta read, bf16 o written, int32 counts read,
    and the captured slot (decay, keys, deltas in fp32) of every row whose
    clamped count is >= 1 (T = 1 per call)."""
    B, Hk, Hv, dk, dv = d["B"], d["Hk"], d["Hv"], d["dk"], d["dv"]
    state = 2 * B * Hv * dv * dk * 4
    vecs = B * (2 * Hk * dk + 2 * Hv * dv + 2 * Hv) * 2 + B * 4
    slot = (Hv + Hk * dk + Hv * dv) * 4
    cap_rows = sum(1 for c in counts if min(max(int(c), 0), d["cap"], 1) >= 1)
    return state + vecs + cap_rows * slot


def replay_bytes(accepted, d=DEC) -> int:
    """State read + write for every row, plus the slots each row replays."""
    B, Hk, Hv, dk, dv = d["B"], d["Hk"], d["Hv"], d["dk"], d["dv"]
    slot = (Hv + Hk * dk + Hv * dv) * 4
    return 2 * B * Hv * dv * dk * 4 + sum(min(max(int(a), 0), d["cap"]) for a in accepted) * slot + B * 4


def verify_bytes(accepted, B, d=DEC, v=VER) -> int:
    """Algorithmic bytes of ONE fused replay + verify call, state in place:
    the state read for every row and written for rows that replay (m_b >= 1;
    rows with m_b = 0 are left in place), the replayed slots read, the draft
    tokens' bf16 q, k, v, alpha, beta read and o written, every draft
    captured (fp32 slots written), int32 counts read."""
    Hk, Hv, dk, dv, T, cap = d["Hk"], d["Hv"], d["dk"], d["dv"], v["T"], v["cap"]
    st = Hv * dv * dk * 4
    slot = (Hv + Hk * dk + Hv * dv) * 4
    m = [min(max(int(a), 0), cap) for a in accepted]
    state = B * st + sum(1 for x in m if x > 0) * st
    tokens = B * T * ((2 * Hk * dk + 2 * Hv * dv + 2 * Hv) * 2)
    return state + sum(m) * slot + B * min(cap, T) * slot + 2 * B * 4 + tokens


def prefill_bytes_flops(p=PRE):
    """Minimum HBM bytes and the chunked form's flops of one prefill call."""
    T, Hk, Hv, dk, dv, C = p["T"], p["Hk"], p["Hv"], p["dk"], p["dv"], p["chunk"]
    byts = (2 * T * Hk * dk * 2 + 2 * T * Hv * dv * 2 + 2 * T * Hv * 4
            + 2 * Hv * dv * dk * 4)
    flops = T * Hv * (6 * dk * dv + 10 * C * dk)
    return byts, flops


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            j = json.load(f)
        return float(j["hbm_gbs"]), float(j["bf16_tflops"]), "measured"
    except (OSError, KeyError, ValueError):
        return 6800.0, 1900.0, "fallback"


# ------------------------------------------------------------ our arm ----

def run_ours(args, rank, world, local_rank):
    import torch
    from gated_deltanet_recurrence_02_gb300 import gdn
    from gated_deltanet_recurrence_02_gb300.inputs import accepted_counts, capture_counts, make_inputs

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    gdn.lib()
    stream = torch.cuda.current_stream()
    if args.only in ("batch", "snapshot"):
        # profiling mode: one of the many-row prefill legs alone
        hbm_peak, tf_peak, _ = load_peaks()
        if args.only == "batch":
            return run_prefill_batch(gdn, dev, stream, rank, hbm_peak, tf_peak)
        return run_prefix_snapshot(gdn, dev, stream, rank, hbm_peak)
    d = dict(DEC, B=args.decode_rows)
    do_pre, do_dec, do_rep, do_ver = (args.only in ("all", ph)
                                      for ph in ("prefill", "decode", "replay", "verify"))
    B, S_, Hk, Hv, dk, dv, cap = d["B"], d["steps"], d["Hk"], d["Hv"], d["dk"], d["dv"], d["cap"]

    # ---- decode inputs (step-major on the device) ----
    x = make_inputs(d["seed"] + 100 * rank, lengths=[S_] * B, Hk=Hk, Hv=Hv, dk=dk, dv=dv,
                    dtype_qkv="bf16", dtype_gate="bf16")
    counts = capture_counts(d["seed"] + 1 + 100 * rank, B, cap)

    def step_major_host(t):
        return t.view(B, S_, *t.shape[1:]).transpose(0, 1).contiguous()
    hq, hk_, hv, ha, hb = (step_major_host(getattr(x, n)) for n in ("q", "k", "v", "alpha", "beta"))
    S0_host = x.initial_state
    q, k, v, a, bt = (t.to(dev) for t in (hq, hk_, hv, ha, hb))
    S = S0_host.to(dev)
    cc = counts.to(dev)
    out = torch.empty_like(v)
    slot = gdn.slot_width(Hk, Hv, dk, dv)
    su = torch.empty((B, cap, slot), dtype=torch.float32, device=dev)

    # ---- replay inputs: a capacity-4 capture of 4 tokens, accepted ~ U{0..4}
    xr = make_inputs(REP_SEED + 100 * rank, lengths=[cap] * B, Hk=Hk, Hv=Hv, dk=dk, dv=dv,
                     dtype_qkv="bf16", dtype_gate="bf16", zero_state=True)
    gr = {n: getattr(xr, n).to(dev) for n in ("q", "k", "v", "alpha", "beta")}
    su_r = torch.empty((B, cap, slot), dtype=torch.float32, device=dev)
    gdn.gdn_recurrent_capture(gr["q"], gr["k"], gr["v"], gr["alpha"], gr["beta"], B=B, T=cap,
                              state_update_capacity=cap,
                              capture_count=torch.full((B,), cap, dtype=torch.int32, device=dev),
                              state_update=su_r, want_final_state=False)
    accepted = capture_counts(REP_SEED + 1 + 100 * rank, B, cap)
    acc_d = accepted.to(dev)
    S_rep = torch.empty_like(S)

    # ---- speculative step inputs: a 4-draft capture to replay (made here,
    # outside the timed region), accepted ~ U{0..4}, 4 new drafts per row
    vt, vcap = VER["T"], VER["cap"]
    xv1 = make_inputs(VER["seed"] + 100 * rank, lengths=[vt] * B, Hk=Hk, Hv=Hv, dk=dk, dv=dv,
                      dtype_qkv="bf16", dtype_gate="bf16")
    xv2 = make_inputs(VER["seed"] + 1 + 100 * rank, lengths=[vt] * B, Hk=Hk, Hv=Hv, dk=dk,
                      dv=dv, dtype_qkv="bf16", dtype_gate="bf16", zero_state=True)
    gv1 = {n: getattr(xv1, n).to(dev) for n in ("q", "k", "v", "alpha", "beta")}
    gv = {n: getattr(xv2, n).to(dev) for n in ("q", "k", "v", "alpha", "beta")}
    S_ver = xv1.initial_state.to(dev)
    v_full = torch.full((B,), vcap, dtype=torch.int32, device=dev)
    su_prev = torch.empty((B, vcap, slot), dtype=torch.float32, device=dev)
    gdn.gdn_recurrent_capture(gv1["q"], gv1["k"], gv1["v"], gv1["alpha"], gv1["beta"], B=B, T=vt,
                              initial_state=S_ver, state_update_capacity=vcap,
                              capture_count=v_full, state_update=su_prev, want_final_state=False)
    v_acc = accepted_counts(VER["seed"] + 2 + 100 * rank, B, vcap)
    v_acc_d = v_acc.to(dev)
    v_out = torch.empty_like(gv["v"])
    su_new = torch.empty_like(su_prev)
    del xv1, gv1

    def verify():
        gdn.gdn_replay_verify(gv["q"], gv["k"], gv["v"], gv["alpha"], gv["beta"], B=B, T=vt,
                              state_in=S_ver, state_out=S_ver, prev_state_update=su_prev,
                              prev_capacity=vcap, accepted_count=v_acc_d, out=v_out,
                              state_update_capacity=vcap, capture_count=v_full,
                              state_update=su_new)

    # ---- prefill inputs ----
    p = PRE
    xp = make_inputs(p["seed"] + 100 * rank, lengths=[p["T"]], Hk=p["Hk"], Hv=p["Hv"],
                     dk=p["dk"], dv=p["dv"], dtype_qkv="bf16", dtype_gate="f32")
    gp = {n: getattr(xp, n).to(dev) for n in ("q", "k", "v", "alpha", "beta", "initial_state")}
    p_out = torch.empty_like(gp["v"])
    p_fs = torch.empty((1, p["Hv"], p["dv"], p["dk"]), dtype=torch.float32, device=dev)
    ws_n = gdn.gdn_prefill_workspace_size(1, p["T"], p["Hk"], p["Hv"], p["dk"], p["dv"],
                                          p["chunk"], torch.bfloat16)
    ws = torch.empty(max(ws_n, 16), dtype=torch.uint8, device=dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    # --flush read: a read-only pass over 512 MiB instead, so that L2 holds only
    # clean lines when the step starts (for DRAM-traffic captures of one step)
    flush_r = torch.ones(512 << 20, dtype=torch.uint8, device=dev) if args.flush == "read" else None

    def flush_l2():
        if flush_r is None:
            flush.fill_(1)
        else:
            flush_r.sum(dtype=torch.int64)

    def prefill():
        gdn.gdn_prefill_chunked(gp["q"], gp["k"], gp["v"], gp["alpha"], gp["beta"], B=1,
                                T=p["T"], initial_state=gp["initial_state"], final_state=p_fs,
                                out=p_out, chunk=p["chunk"], workspace=ws)

    def decode_call(t):
        gdn.gdn_recurrent_capture(q[t], k[t], v[t], a[t], bt[t], B=B, T=1, initial_state=S,
                                  final_state=S, out=out[t], state_update_capacity=cap,
                                  capture_count=cc, state_update=su)

    def replay():
        gdn.gdn_replay_state_updates(S, su_r, acc_d, state_update_capacity=cap, Hk=Hk,
                                     state_out=S_rep)

    E = lambda: torch.cuda.Event(enable_timing=True)  # noqa: E731
    n_ev = S_ + 5
    ev = [[E() for _ in range(n_ev)] for _ in range(args.steps)]

    def step(evs=None):
        flush_l2()
        if evs: evs[0].record(stream)
        if do_pre:
            prefill()
        if evs: evs[1].record(stream)
        for t in range(S_):
            if do_dec:
                decode_call(t)
            if evs: evs[2 + t].record(stream)
        if do_rep:
            replay()
        if evs: evs[2 + S_].record(stream)
        if do_ver:
            verify()
        if evs: evs[3 + S_].record(stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    sampler = ClockSampler(torch.cuda.current_device()) if rank == 0 else None
    if sampler:
        sampler.start()
    barrier()
    torch.cuda.synchronize()
    t_wall = time.perf_counter()
    for s in range(args.steps):
        step(ev[s])
    torch.cuda.synchronize()
    barrier()
    t_wall = time.perf_counter() - t_wall
    clocks = sampler.stop() if sampler else None

    pre_ms = [ev[s][0].elapsed_time(ev[s][1]) for s in range(args.steps)]
    dec_launch_ms = [ev[s][1 + t].elapsed_time(ev[s][2 + t])
                     for s in range(args.steps) for t in range(S_)]
    dec_ms = [ev[s][1].elapsed_time(ev[s][1 + S_]) for s in range(args.steps)]
    rep_ms = [ev[s][1 + S_].elapsed_time(ev[s][2 + S_]) for s in range(args.steps)]
    ver_ms = [ev[s][2 + S_].elapsed_time(ev[s][3 + S_]) for s in range(args.steps)]
    assert torch.isfinite(out).all() and torch.isfinite(S).all() and torch.isfinite(p_out.float()).all()
    assert torch.isfinite(S_ver).all() and torch.isfinite(v_out.float()).all()
    p_ref = p_out.clone()  # the step's prefill output (one call), before the extra legs

    if args.only != "all":
        # profiling mode: one phase only, no JSON contract line
        return {"only": args.only, "decode_rows": B, "prefill_ms": statistics.mean(pre_ms),
                "decode_ms": statistics.mean(dec_ms), "replay_ms": statistics.mean(rep_ms),
                "verify_ms": statistics.mean(ver_ms)}
    dec_bytes_call = decode_bytes(counts.tolist(), d)
    dec_total_bytes = dec_bytes_call * S_ * args.steps
    dec_time = reduce_scalar(sum(dec_ms) / 1e3, "max", dev)
    all_bytes = reduce_scalar(dec_total_bytes, "sum", dev)
    value = all_bytes / dec_time / 1e9

    hbm_peak, tf_peak, peak_kind = load_peaks()
    launch_avg_s = statistics.mean(dec_launch_ms) / 1e3
    achieved = dec_bytes_call / launch_avg_s / 1e9
    pb, pf = prefill_bytes_flops()
    pre_avg_s = statistics.mean(pre_ms) / 1e3
    pre_time = reduce_scalar(sum(pre_ms) / 1e3, "max", dev)
    pre_tokens = reduce_scalar(p["T"] * args.steps, "sum", dev)
    rep_bytes_call = replay_bytes(accepted.tolist())
    rep_avg_s = statistics.mean(rep_ms) / 1e3
    ver_bytes_call = verify_bytes(v_acc.tolist(), B, d)
    ver_avg_s = statistics.mean(ver_ms) / 1e3
    unfused = run_verify_unfused(gdn, stream, gv, su_prev, v_acc_d, v_full, S_ver, d)
    ckpt = run_prefill_variant(gdn, stream, gp, p_out, p_fs, ws, flush, "checkpoints")
    pcap = run_prefill_variant(gdn, stream, gp, p_out, p_fs, ws, flush, "capture")
    pbatch = run_prefill_batch(gdn, dev, stream, rank, hbm_peak, tf_peak)
    psnap = run_prefix_snapshot(gdn, dev, stream, rank, hbm_peak)
    fe = run_front_end(gdn, stream, q, k, v, a, bt, S, out, cc, su, gp, p_out, p_fs, ws, flush, d)
    ms_per_step = (sum(pre_ms) + sum(dec_ms) + sum(rep_ms) + sum(ver_ms)) / args.steps
    ms_per_step = reduce_scalar(ms_per_step, "max", dev)

    # ---- end to end through the public API with host buffers (decode) ----
    e2e = run_e2e(args, gdn, dev, stream, hq, hk_, hv, ha, hb, S0_host, counts, d)
    # the step's prefill output (same inputs, one call) checks the segmented e2e run
    e2e_pre = run_e2e_prefill(args, gdn, dev, stream, xp, ref_out=p_ref if do_pre else None)

    line = None
    if rank == 0:
        line = {
            "metric": METRIC,
            "value": round(value, 2),
            "unit": "GB/s",
            "n_gpus": world,
            "steps": args.steps,
            "warmup": args.warmup,
            "ms_per_step": round(ms_per_step, 4),
            "higher_is_better": True,
            "scaling": "weak",
            "vs_baseline": None,
            "dtype": "f32",
            "storage_dtype": "bf16",
            "data": "synthetic (seeded; q,k L2-normalised N(0,1), v N(0,1), "
                    "beta=sigmoid(N(0,1)), alpha=exp(-U(0.01,0.5)), S0=0.1*N(0,1))",
            "config": {
                "workload": "decode_B256: B=256 rows x 64 single-token steps, Hq=Hk=16, Hv=32, "
                            "dk=dv=128, bf16 q/k/v/alpha/beta, fp32 state in place, capture "
                            "capacity 4, capture_count~U{0..4}; plus prefill_T4100 and replay",
                "B": B, "steps_per_call_chain": S_, "Hk": Hk, "Hv": Hv, "dk": dk, "dv": dv,
                "capacity": cap,
                "l2": "decode state 512 MiB > L2 (inputs larger than L2); "
                      "L2 flushed by a 256 MiB write before each prefill",
                "parallelism": f"replicas x{world} (rows independent)",
            },
            "roofline": {
                "kernel": "recurrent_kernel<128, bf16, 1, 0, 4> (decode, T=1)",
                "bound": "hbm", "achieved": round(achieved, 1), "peak": hbm_peak,
                "peak_kind": f"{peak_kind} hbm_gbs (burst copy)",
                "unit": "GB/s", "frac": round(achieved / hbm_peak, 4), "traffic": DECODE_TRAFFIC_BYTES,
                "algorithmic_bytes_per_launch": dec_bytes_call,
                "avg_launch_us": round(launch_avg_s * 1e6, 2),
            },
            "prefill": {
                "workload": "prefill_T4100: B=1, T=4100, Hk=16, Hv=32, d=128, chunk 64, bf16 "
                            "q/k/v, fp32 alpha/beta and state",
                "value": round(pre_tokens / pre_time, 1), "unit": "tokens/s",
                "avg_launch_us": round(pre_avg_s * 1e6, 2),
                "roofline": {
                    "bound": "hbm", "achieved": round(pb / pre_avg_s / 1e9, 1),
                    "peak": hbm_peak, "unit": "GB/s",
                    "frac": round(pb / pre_avg_s / 1e9 / hbm_peak, 4),
                    "algorithmic_bytes_per_launch": pb,
                    "tensor_frac": round(pf / pre_avg_s / 1e12 / tf_peak, 4),
                    "algorithmic_flops_per_launch": pf, "traffic": PREFILL_TRAFFIC_BYTES,
                },
                "e2e": e2e_pre,
                "checkpoints": {
                    "workload": "prefill_T4100 with the fp32 state written after every "
                                "64-token chunk (64 checkpoints, gdn_prefill_chunked_checkpoints)",
                    "avg_launch_us": ckpt["us"],
                    "value": round(p["T"] / (ckpt["us"] * 1e-6), 1), "unit": "tokens/s",
                    "checkpoint_bytes_per_launch": ckpt["bytes"],
                    "frac": round((pb + ckpt["bytes"]) / (ckpt["us"] * 1e-6) / 1e9 / hbm_peak, 4),
                    "overhead_vs_plain": round(ckpt["us"] / (pre_avg_s * 1e6) - 1.0, 4),
                },
                "batch": pbatch,
                "snapshot": psnap,
                "capture": {
                    "workload": "prefill_T4100 with the compact capture of its first 64 tokens "
                                "(capacity 64, gdn_prefill_chunked_capture)",
                    "avg_launch_us": pcap["us"],
                    "value": round(p["T"] / (pcap["us"] * 1e-6), 1), "unit": "tokens/s",
                    "capture_bytes_per_launch": pcap["bytes"],
                    "overhead_vs_plain": round(pcap["us"] / (pre_avg_s * 1e6) - 1.0, 4),
                },
            },
            "replay": {
                "value": round(rep_bytes_call / rep_avg_s / 1e9, 1), "unit": "GB/s",
                "avg_launch_us": round(rep_avg_s * 1e6, 2),
                "frac": round(rep_bytes_call / rep_avg_s / 1e9 / hbm_peak, 4),
                "algorithmic_bytes_per_launch": rep_bytes_call,
            },
            "replay_verify": {
                "workload": "verify_B256_T4: B=256, replay of accepted~U{0..4} of 4 captured "
                            "slots, then 4 bf16 draft tokens per row with capture (capacity 4), "
                            "state in place; one fused launch",
                "value": round(ver_bytes_call / ver_avg_s / 1e9, 1), "unit": "GB/s",
                "frac": round(ver_bytes_call / ver_avg_s / 1e9 / hbm_peak, 4),
                "avg_launch_us": round(ver_avg_s * 1e6, 2),
                "draft_tokens_per_s": round(B * VER["T"] / ver_avg_s, 1),
                "algorithmic_bytes_per_launch": ver_bytes_call,
                "traffic": VERIFY_TRAFFIC_BYTES,
                "unfused_us": unfused,
                "speedup_vs_unfused": round(unfused["total"] / (ver_avg_s * 1e6), 3),
            },
            "front_end": {
                "workload": "in-kernel input conventions (q/k L2 normalisation, alpha as "
                            "log-decay, beta as logits): decode_B256 (one T=1 call) and "
                            "prefill_T4100, against the same calls without them",
                "decode_us": fe["decode_us"], "decode_plain_us": round(launch_avg_s * 1e6, 2),
                "decode_overhead": round(fe["decode_us"] / (launch_avg_s * 1e6) - 1.0, 4),
                "prefill_us": fe["prefill_us"], "prefill_plain_us": round(pre_avg_s * 1e6, 2),
                "prefill_overhead": round(fe["prefill_us"] / (pre_avg_s * 1e6) - 1.0, 4),
            },
            "e2e": e2e,
            "gpu_launches": args.steps * (PREFILL_LAUNCHES + S_ + 2),
            "clocks": clocks,
            "wall_s_timed_region": round(t_wall, 4),
        }
    return line


def run_verify_unfused(gdn, stream, gv, su_prev, acc_d, full, S_src, d, n=20, warm=3):
    """The speculative step done as two calls -- replay in place, then the
    drafts through gdn_recurrent_capture (no final state) -- on a copy of the
    state, outside the step's timed region: per-call means in microseconds."""
    import torch
    B, vt, vcap, Hk = d["B"], VER["T"], VER["cap"], d["Hk"]
    S = S_src.clone()
    out = torch.empty_like(gv["v"])
    su = torch.empty_like(su_prev)
    E = lambda: torch.cuda.Event(enable_timing=True)  # noqa: E731
    ev = [[E(), E(), E()] for _ in range(n)]
    for i in range(warm + n):
        e = ev[i - warm] if i >= warm else None
        if e: e[0].record(stream)
        gdn.gdn_replay_state_updates(S, su_prev, acc_d, state_update_capacity=vcap, Hk=Hk,
                                     state_out=S)
        if e: e[1].record(stream)
        gdn.gdn_recurrent_capture(gv["q"], gv["k"], gv["v"], gv["alpha"], gv["beta"], B=B, T=vt,
                                  initial_state=S, want_final_state=False, out=out,
                                  state_update_capacity=vcap, capture_count=full,
                                  state_update=su)
        if e: e[2].record(stream)
    torch.cuda.synchronize()
    rep = statistics.mean(e[0].elapsed_time(e[1]) for e in ev) * 1e3
    ver = statistics.mean(e[1].elapsed_time(e[2]) for e in ev) * 1e3
    del S
    return {"replay": round(rep, 2), "verify": round(ver, 2), "total": round(rep + ver, 2)}


def run_prefill_batch(gdn, dev, stream, rank, hbm_peak, tf_peak, n=5, warm=3):
    """prefill_batch_B64: 64 packed rows of 500 .. 1500 tokens in one call, timed
    outside the step (the inputs, ~2 GB, exceed L2).  Tokens/s and the bytes
    and flops rooflines of the call."""
    import torch
    from gated_deltanet_recurrence_02_gb300.inputs import WORKLOADS, make_inputs, ragged_lengths
    w = WORKLOADS["prefill_batch_B64"]
    lengths = ragged_lengths(w["seed"] + 100 * rank, w["B"], w["lo"], w["hi"])
    x = make_inputs(w["seed"] + 1 + 100 * rank, lengths=lengths, Hk=w["Hk"], Hv=w["Hv"],
                    dk=w["dk"], dv=w["dv"], dtype_qkv=w["dtype_qkv"], dtype_gate=w["dtype_gate"])
    g = {n: getattr(x, n).to(dev) for n in ("q", "k", "v", "alpha", "beta", "initial_state")}
    cu = x.cu_seqlens.to(dev)
    B, T, Hk, Hv, d, C = w["B"], int(x.cu_seqlens[-1]), w["Hk"], w["Hv"], w["dk"], w["chunk"]
    out = torch.empty_like(g["v"])
    fs = torch.empty_like(g["initial_state"])
    ws = torch.empty(gdn.gdn_prefill_workspace_size(B, T, Hk, Hv, d, d, C, torch.bfloat16,
                                                    varlen=True), dtype=torch.uint8, device=dev)
    E = lambda: torch.cuda.Event(enable_timing=True)  # noqa: E731
    ev = [[E(), E()] for _ in range(n)]
    for i in range(warm + n):
        e = ev[i - warm] if i >= warm else None
        if e: e[0].record(stream)
        gdn.gdn_prefill_chunked(g["q"], g["k"], g["v"], g["alpha"], g["beta"], B=B, cu_seqlens=cu,
                                initial_state=g["initial_state"], final_state=fs, out=out,
                                chunk=C, workspace=ws)
        if e: e[1].record(stream)
    torch.cuda.synchronize()
    assert torch.isfinite(out.float()).all() and torch.isfinite(fs).all()
    sec = statistics.mean(e[0].elapsed_time(e[1]) for e in ev) / 1e3
    byts = (T * (2 * Hk * d * 2 + 2 * Hv * d * 2 + 2 * Hv * 4) + 2 * B * Hv * d * d * 4)
    flops = T * Hv * (6 * d * d + 10 * C * d)
    del g, out, fs, ws
    return {"workload": f"prefill_batch_B64: {B} packed rows of {w['lo']}..{w['hi']} tokens "
                        f"({T} in all), Hk=16, Hv=32, d=128, bf16 q/k/v, fp32 alpha/beta",
            "avg_launch_us": round(sec * 1e6, 2), "value": round(T / sec, 1), "unit": "tokens/s",
            "frac": round(byts / sec / 1e9 / hbm_peak, 4),
            "tensor_frac": round(flops / sec / 1e12 / tf_peak, 4),
            "algorithmic_bytes_per_launch": byts, "algorithmic_flops_per_launch": flops}


def run_prefix_snapshot(gdn, dev, stream, rank, hbm_peak, n=10, warm=3):
    """prefix_snapshot_B12: a 2048-token prefill from a zero state gives one
    snapshot; 12 packed rows of 200 .. 1000 tokens then all start from it
    (initial_state_indices = 0, read-only).  Tokens/s of the 12-row call, its
    bytes roofline, and a check that the snapshot bytes never change."""
    import torch
    from gated_deltanet_recurrence_02_gb300.inputs import WORKLOADS, make_inputs, ragged_lengths
    w = WORKLOADS["prefix_snapshot_B12"]
    dims = dict(Hk=w["Hk"], Hv=w["Hv"], dk=w["dk"], dv=w["dv"])
    pre = make_inputs(w["seed"] + 100 * rank, lengths=[w["prefix_len"]], dtype_qkv=w["dtype_qkv"],
                      dtype_gate=w["dtype_gate"], zero_state=True, **dims)
    lens = ragged_lengths(w["seed"] + 1 + 100 * rank, w["B"], w["lo"], w["hi"])
    x = make_inputs(w["seed"] + 2 + 100 * rank, lengths=lens, dtype_qkv=w["dtype_qkv"],
                    dtype_gate=w["dtype_gate"], zero_state=True, **dims)
    gp = {n: getattr(pre, n).to(dev) for n in ("q", "k", "v", "alpha", "beta")}
    g = {n: getattr(x, n).to(dev) for n in ("q", "k", "v", "alpha", "beta")}
    cu = x.cu_seqlens.to(dev)
    B, T, Hk, Hv, d, C = w["B"], int(x.cu_seqlens[-1]), w["Hk"], w["Hv"], w["dk"], w["chunk"]
    snap = torch.empty((1, Hv, d, d), dtype=torch.float32, device=dev)
    E = lambda: torch.cuda.Event(enable_timing=True)  # noqa: E731
    e_snap = [E(), E()]
    with torch.cuda.stream(stream):
        for i in range(2):  # the first call of a process sets kernel attributes up
            e_snap[0].record(stream)
            gdn.gdn_prefill_chunked(gp["q"], gp["k"], gp["v"], gp["alpha"], gp["beta"], B=1,
                                    T=w["prefix_len"], final_state=snap, chunk=C)
            e_snap[1].record(stream)
    stream.synchronize()
    before = snap.clone()
    idx = torch.zeros(B, dtype=torch.int32, device=dev)
    out = torch.empty_like(g["v"])
    fs = torch.empty((B, Hv, d, d), dtype=torch.float32, device=dev)
    ws = torch.empty(gdn.gdn_prefill_workspace_size(B, T, Hk, Hv, d, d, C, torch.bfloat16,
                                                    varlen=True), dtype=torch.uint8, device=dev)
    ev = [[E(), E()] for _ in range(n)]
    for i in range(warm + n):
        e = ev[i - warm] if i >= warm else None
        if e: e[0].record(stream)
        gdn.gdn_prefill_chunked(g["q"], g["k"], g["v"], g["alpha"], g["beta"], B=B, cu_seqlens=cu,
                                initial_state=snap, initial_state_indices=idx, final_state=fs,
                                out=out, chunk=C, workspace=ws)
        if e: e[1].record(stream)
    torch.cuda.synchronize()
    assert torch.equal(snap.view(torch.int32), before.view(torch.int32)), "snapshot modified"
    assert torch.isfinite(out.float()).all() and torch.isfinite(fs).all()
    sec = statistics.mean(e[0].elapsed_time(e[1]) for e in ev) / 1e3
    # q, k, v, o (bf16), alpha, beta (bf16), the snapshot read once per row, B final states
    byts = T * (2 * Hk * d * 2 + 2 * Hv * d * 2 + 2 * Hv * 2) + 2 * B * Hv * d * d * 4
    res = {"workload": f"prefix_snapshot_B12: snapshot of a {w['prefix_len']}-token prefill, then "
                       f"{B} packed rows of {w['lo']}..{w['hi']} tokens ({T} in all) from it, "
                       f"Hk=16, Hv=32, d=128, bf16",
           "snapshot_us": round(e_snap[0].elapsed_time(e_snap[1]) * 1e3, 2),
           "avg_launch_us": round(sec * 1e6, 2), "value": round(T / sec, 1), "unit": "tokens/s",
           "frac": round(byts / sec / 1e9 / hbm_peak, 4), "algorithmic_bytes_per_launch": byts,
           "snapshot_bit_identical": True}
    del gp, g, out, fs, ws, snap
    return res


def run_prefill_variant(gdn, stream, gp, out, fs, ws, flush, kind, n=10, warm=3):
    """The prefill with an extra output, timed outside the step (L2 flushed
    before each launch): kind "checkpoints" writes the state after every chunk,
    kind "capture" captures the first 64 tokens (capacity 64).  Returns the
    mean microseconds and the extra bytes written per launch."""
    import torch
    p = PRE
    dev = gp["q"].device
    if kind == "checkpoints":
        cap = p["T"] // p["chunk"]
        buf = torch.empty((1, cap, p["Hv"], p["dv"], p["dk"]), dtype=torch.float32, device=dev)
        extra = buf.numel() * 4
    else:
        cap = 64
        slot = p["Hv"] + p["Hk"] * p["dk"] + p["Hv"] * p["dv"]
        buf = torch.empty((1, cap, slot), dtype=torch.float32, device=dev)
        count = torch.full((1,), cap, dtype=torch.int32, device=dev)
        extra = buf.numel() * 4
    E = lambda: torch.cuda.Event(enable_timing=True)  # noqa: E731
    ev = [[E(), E()] for _ in range(n)]
    common = dict(B=1, T=p["T"], initial_state=gp["initial_state"], final_state=fs, out=out,
                  chunk=p["chunk"], workspace=ws)
    for i in range(warm + n):
        flush.fill_(2)
        e = ev[i - warm] if i >= warm else None
        if e: e[0].record(stream)
        if kind == "checkpoints":
            gdn.gdn_prefill_chunked_checkpoints(gp["q"], gp["k"], gp["v"], gp["alpha"], gp["beta"],
                                                checkpoints=buf, checkpoint_capacity=cap,
                                                checkpoint_interval=1, **common)
        else:
            gdn.gdn_prefill_chunked_capture(gp["q"], gp["k"], gp["v"], gp["alpha"], gp["beta"],
                                            state_update_capacity=cap, capture_count=count,
                                            state_update=buf, **common)
        if e: e[1].record(stream)
    torch.cuda.synchronize()
    assert torch.isfinite(buf).all()
    us = statistics.mean(e[0].elapsed_time(e[1]) for e in ev) * 1e3
    return {"us": round(us, 2), "bytes": extra}


def run_front_end(gdn, stream, q, k, v, a, bt, S, out, cc, su, gp, p_out, p_fs, ws, flush, d,
                  n=10, warm=3):
    """Decode (one T=1 call on the decode state, kept finite) and prefill with
    every input convention on (GDN_QK_L2NORM | GDN_ALPHA_LOG | GDN_BETA_LOGIT),
    timed outside the step: mean microseconds per call.  The gates are the
    workload's, re-expressed as log-decay and logits on the host beforehand."""
    import torch
    conv = gdn.GDN_QK_L2NORM | gdn.GDN_ALPHA_LOG | gdn.GDN_BETA_LOGIT
    a_log = torch.log(a[0].float()).to(a.dtype)
    b_logit = torch.logit(bt[0].float().clamp(1e-4, 1 - 1e-4)).to(bt.dtype)
    S_fe = S.clone()
    pa = torch.log(gp["alpha"].float()).to(gp["alpha"].dtype)
    pb = torch.logit(gp["beta"].float().clamp(1e-4, 1 - 1e-4)).to(gp["beta"].dtype)
    E = lambda: torch.cuda.Event(enable_timing=True)  # noqa: E731
    res = {}
    for kind in ("decode", "prefill"):
        ev = [[E(), E()] for _ in range(n)]
        for i in range(warm + n):
            if kind == "prefill":
                flush.fill_(3)
            e = ev[i - warm] if i >= warm else None
            if e: e[0].record(stream)
            if kind == "decode":
                gdn.gdn_recurrent_capture(q[0], k[0], v[0], a_log, b_logit, B=d["B"], T=1,
                                          initial_state=S_fe, final_state=S_fe, out=out[0],
                                          state_update_capacity=d["cap"], capture_count=cc,
                                          state_update=su, conventions=conv)
            else:
                gdn.gdn_prefill_chunked(gp["q"], gp["k"], gp["v"], pa, pb, B=1, T=PRE["T"],
                                        initial_state=gp["initial_state"], final_state=p_fs,
                                        out=p_out, chunk=PRE["chunk"], workspace=ws,
                                        conventions=conv)
            if e: e[1].record(stream)
        torch.cuda.synchronize()
        res[kind + "_us"] = round(statistics.mean(e[0].elapsed_time(e[1]) for e in ev) * 1e3, 2)
    assert torch.isfinite(S_fe).all() and torch.isfinite(p_out.float()).all()
    del S_fe
    return res


PREFILL_LAUNCHES = 2  # kernels one gdn_prefill_chunked call launches on this workload (tensor-core path)
# DRAM bytes (read + write) of one launch of the current kernels, each from one
# ncu capture of that kernel on this workload: decode at B=256, the fused
# replay + verify step, and one prefill call (its two kernels, chunk-parallel
# then carry, captured back to back without ncu's cache flushing, after a
# read-only pass over a buffer larger than L2, so that the carry meets the
# chunk-parallel kernel's records where they are).  Reset to None whenever the
# kernel changes.
DECODE_TRAFFIC_BYTES = 541_206_272 + 483_718_912
VERIFY_TRAFFIC_BYTES = 567_203_072 + 391_274_240
PREFILL_TRAFFIC_BYTES = (68_530_176 + 20_282_880) + (87_194_880 + 46_133_504)


E2E_GROUPS = 8       # decode e2e: row groups pipelined on their own streams
E2E_SEGMENT = 1024   # prefill e2e: tokens per call (a multiple of the 64-token chunk)


def run_e2e(args, gdn, dev, stream, hq, hk_, hv, ha, hb, S0_host, counts, d):
    """Decode through the public API with host-resident data.  Every step
    copies the initial state and the 64 tokens' inputs from pinned host memory,
    runs the 64 calls and copies the final state, outputs and capture back.
    Rows are independent, so the batch runs as E2E_GROUPS row groups, each on
    its own stream (copy in, 64 calls, copy out): one group's copies overlap
    the others' kernels."""
    import torch
    B, S_, cap = d["B"], d["steps"], d["cap"]
    G = E2E_GROUPS if B % E2E_GROUPS == 0 else 1
    Bg = B // G
    slot = gdn.slot_width(d["Hk"], d["Hv"], d["dk"], d["dv"])
    pin = lambda t: t.contiguous().pin_memory()  # noqa: E731
    grp = []
    for g in range(G):
        r = slice(g * Bg, (g + 1) * Bg)
        h_in = [pin(t[:, r]) for t in (hq, hk_, hv, ha, hb)]  # step-major [S_, rows, ...]
        e = dict(h_in=h_in, h_S0=pin(S0_host[r]), h_cc=pin(counts[r]),
                 d_in=[torch.empty_like(t, device=dev) for t in h_in],
                 d_S=torch.empty(S0_host[r].shape, dtype=torch.float32, device=dev),
                 d_cc=torch.empty(Bg, dtype=torch.int32, device=dev),
                 d_su=torch.empty((Bg, cap, slot), dtype=torch.float32, device=dev),
                 stream=torch.cuda.Stream(dev))
        e["d_out"] = torch.empty_like(e["d_in"][2])
        e["h_S"] = torch.empty_like(e["h_S0"]).pin_memory()
        e["h_out"] = torch.empty_like(e["d_out"], device="cpu").pin_memory()
        e["h_su"] = torch.empty_like(e["d_su"], device="cpu").pin_memory()
        grp.append(e)
    h2d = sum(sum(t.numel() * t.element_size() for t in e["h_in"]) + e["h_S0"].numel() * 4
              + e["h_cc"].numel() * 4 for e in grp)
    d2h = sum(e["h_S"].numel() * 4 + e["h_out"].numel() * e["h_out"].element_size()
              + e["h_su"].numel() * 4 for e in grp)

    def one(start):
        done = []
        for e in grp:
            s = e["stream"]
            s.wait_event(start)
            with torch.cuda.stream(s):
                for dt, ht in zip(e["d_in"], e["h_in"]):
                    dt.copy_(ht, non_blocking=True)
                e["d_S"].copy_(e["h_S0"], non_blocking=True)
                e["d_cc"].copy_(e["h_cc"], non_blocking=True)
                q, k, v, a, bt = e["d_in"]
                for t in range(S_):
                    gdn.gdn_recurrent_capture(q[t], k[t], v[t], a[t], bt[t], B=Bg, T=1,
                                              initial_state=e["d_S"], final_state=e["d_S"],
                                              out=e["d_out"][t], state_update_capacity=cap,
                                              capture_count=e["d_cc"], state_update=e["d_su"],
                                              stream=s)
                e["h_S"].copy_(e["d_S"], non_blocking=True)
                e["h_out"].copy_(e["d_out"], non_blocking=True)
                e["h_su"].copy_(e["d_su"], non_blocking=True)
            ev = torch.cuda.Event()
            ev.record(s)
            done.append(ev)
        for ev in done:
            stream.wait_event(ev)

    def mark():
        ev = torch.cuda.Event(enable_timing=True)
        ev.record(stream)
        return ev

    for _ in range(max(1, args.warmup)):
        one(mark())
    torch.cuda.synchronize()
    n = max(1, args.steps // 2)
    e0 = mark()
    for _ in range(n):
        one(mark())
    e1 = mark()
    torch.cuda.synchronize()
    sec = e0.elapsed_time(e1) / 1e3
    byts = decode_bytes(counts.tolist(), d) * S_ * n
    val = reduce_scalar(byts, "sum", dev) / reduce_scalar(sec, "max", dev) / 1e9
    return {"value": round(val, 2), "unit": "GB/s", "h2d_bytes_per_step": int(h2d),
            "d2h_bytes_per_step": int(d2h), "steps": n, "row_groups": G}


def run_e2e_prefill(args, gdn, dev, stream, xp, ref_out=None):
    """Prefill through the public API with host-resident inputs and results.
    The row runs as calls of E2E_SEGMENT tokens (chunk-aligned, so the result
    is the single call's), the state carried between them; a copy-in stream,
    the compute stream and a copy-out stream overlap segment j + 1's inputs and
    segment j - 1's outputs with segment j's prefill."""
    import torch
    T, C = PRE["T"], PRE["chunk"]
    names = ("q", "k", "v", "alpha", "beta")
    h = {n: getattr(xp, n).pin_memory() for n in names}
    h_S0 = xp.initial_state.pin_memory()
    dd = {n: torch.empty_like(h[n], device=dev) for n in names}
    d_S = [torch.empty_like(h_S0, device=dev) for _ in range(3)]  # S0, then ping-pong
    d_out = torch.empty_like(dd["v"])
    h_out = torch.empty_like(d_out, device="cpu").pin_memory()
    h_fs = torch.empty_like(h_S0).pin_memory()
    bounds = list(range(0, T, E2E_SEGMENT)) + [T]
    if len(bounds) > 2 and bounds[-1] - bounds[-2] < C:
        bounds.pop(-2)  # a short tail joins the previous segment
    seg_max = max(b1 - b0 for b0, b1 in zip(bounds, bounds[1:]))
    ws_n = gdn.gdn_prefill_workspace_size(1, seg_max, PRE["Hk"], PRE["Hv"], PRE["dk"], PRE["dv"],
                                          C, torch.bfloat16)
    ws = torch.empty(max(ws_n, 16), dtype=torch.uint8, device=dev)
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)

    def one(start):
        s_in.wait_event(start)
        with torch.cuda.stream(s_in):
            d_S[0].copy_(h_S0, non_blocking=True)
        loaded = []
        for b0, b1 in zip(bounds, bounds[1:]):
            with torch.cuda.stream(s_in):
                for n in names:
                    dd[n][b0:b1].copy_(h[n][b0:b1], non_blocking=True)
                ev = torch.cuda.Event()
                ev.record(s_in)
                loaded.append(ev)
        for j, (b0, b1) in enumerate(zip(bounds, bounds[1:])):
            stream.wait_event(loaded[j])
            s_prev = d_S[0] if j == 0 else d_S[1 + (j - 1) % 2]
            s_next = d_S[1 + j % 2]
            gdn.gdn_prefill_chunked(dd["q"][b0:b1], dd["k"][b0:b1], dd["v"][b0:b1],
                                    dd["alpha"][b0:b1], dd["beta"][b0:b1], B=1, T=b1 - b0,
                                    initial_state=s_prev, final_state=s_next,
                                    out=d_out[b0:b1], chunk=C, workspace=ws, stream=stream)
            ev = torch.cuda.Event()
            ev.record(stream)
            s_out.wait_event(ev)
            with torch.cuda.stream(s_out):
                h_out[b0:b1].copy_(d_out[b0:b1], non_blocking=True)
                if b1 == T:
                    h_fs.copy_(s_next, non_blocking=True)
        fin = torch.cuda.Event()
        fin.record(s_out)
        stream.wait_event(fin)

    def mark():
        ev = torch.cuda.Event(enable_timing=True)
        ev.record(stream)
        return ev

    for _ in range(max(1, args.warmup)):
        one(mark())
    torch.cuda.synchronize()
    n = max(1, args.steps)
    e0 = mark()
    for _ in range(n):
        one(mark())
    e1 = mark()
    torch.cuda.synchronize()
    sec = e0.elapsed_time(e1) / 1e3
    if ref_out is not None:
        # chunk-aligned segments reproduce the single call bit for bit
        assert torch.equal(h_out.to(dev), ref_out)
    val = reduce_scalar(T * n, "sum", dev) / reduce_scalar(sec, "max", dev)
    h2d = sum(t.numel() * t.element_size() for t in h.values()) + h_S0.numel() * 4
    return {"value": round(val, 1), "unit": "tokens/s", "h2d_bytes_per_step": int(h2d),
            "d2h_bytes_per_step": int(h_out.numel() * 2 + h_fs.numel() * 4),
            "segments": len(bounds) - 1}


# ------------------------------------------------------ oracle (CPU) arm --

def oracle_decode_sample(rows: int, seed: int):
    """Inputs of a bounded slice of the decode workload: `rows` rows, all 32
    heads, 64 tokens each (the same per-row recipe as the GPU run)."""
    from gated_deltanet_recurrence_02_gb300.inputs import make_inputs
    d = DEC
    return make_inputs(seed, lengths=[d["steps"]] * rows, Hk=d["Hk"], Hv=d["Hv"], dk=d["dk"],
                       dv=d["dv"], dtype_qkv="bf16", dtype_gate="bf16")


def time_oracle_decode(x, rows: int, threads: int):
    import oracle
    from gated_deltanet_recurrence_02_gb300.inputs import capture_counts
    d = DEC
    counts = capture_counts(d["seed"] + 1, rows, d["cap"]).tolist()
    t0 = time.perf_counter()
    oracle.recurrent(x.q, x.k, x.v, x.alpha, x.beta, B=rows, T=d["steps"], Hk=d["Hk"],
                     Hv=d["Hv"], dk=d["dk"], dv=d["dv"], initial_state=x.initial_state,
                     capacity=d["cap"], capture_count=counts, threads=threads)
    sec = time.perf_counter() - t0
    # the same algorithmic bytes per (row, step) as the GPU figure
    byts = decode_bytes(counts, dict(d, B=rows)) * d["steps"]
    return byts / sec / 1e9, sec


def cpu_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def cpu_model() -> str:
    """The host CPU's model name (x86 /proc/cpuinfo, else lscpu, else the
    machine type)."""
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith("model name"):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    try:
        import subprocess
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.strip().lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    import platform
    return platform.machine()


def time_oracle_prefill(x, B, units, threads):
    """The oracle (the per-token recurrence, fp64) over `units` (row, head)
    pairs of a prefill workload; returns (tokens/s scaled by the share of
    units done, seconds)."""
    import oracle
    t0 = time.perf_counter()
    oracle.recurrent(x.q, x.k, x.v, x.alpha, x.beta, B=B, Hk=x.Hk, Hv=x.Hv, dk=x.dk, dv=x.dv,
                     cu_seqlens=x.cu_seqlens, initial_state=x.initial_state, units=units,
                     threads=threads)
    sec = time.perf_counter() - t0
    total_units = B * x.Hv
    return x.total_T * (len(units) / total_units) / sec, sec


def cpu_baseline_prefill(cores):
    """Oracle tokens/s on the two prefill workloads: every (row, head) unit on
    all host cores, and a sixteenth of the units on one thread (scaled by the
    share of units done)."""
    from gated_deltanet_recurrence_02_gb300.inputs import WORKLOADS, make_inputs, ragged_lengths
    res = {}
    w = WORKLOADS["prefill_T4100"]
    xp = make_inputs(w["seed"], lengths=w["lengths"], Hk=w["Hk"], Hv=w["Hv"], dk=w["dk"],
                     dv=w["dv"], dtype_qkv=w["dtype_qkv"], dtype_gate=w["dtype_gate"])
    ws = WORKLOADS["prefix_snapshot_B12"]
    lens = ragged_lengths(ws["seed"] + 1, ws["B"], ws["lo"], ws["hi"])
    xs = make_inputs(ws["seed"] + 2, lengths=lens, Hk=ws["Hk"], Hv=ws["Hv"], dk=ws["dk"],
                     dv=ws["dv"], dtype_qkv=ws["dtype_qkv"], dtype_gate=ws["dtype_gate"],
                     zero_state=True)  # (the snapshot's values do not change the work)
    for name, x, B in (("prefill_T4100", xp, 1), ("prefix_snapshot_B12", xs, ws["B"])):
        units = [(b, h) for b in range(B) for h in range(x.Hv)]
        val, sec = time_oracle_prefill(x, B, units, cores)
        one = units[::16]
        val1, sec1 = time_oracle_prefill(x, B, one, 1)
        res[name] = {"value": round(val, 1), "unit": "tokens/s", "cores": cores,
                     "sample": f"all {len(units)} (row, head) units, {x.total_T} tokens "
                               f"(fp64 C oracle, per-token recurrence, {cores} threads, "
                               f"{sec:.2f} s wall)",
                     "single_thread": {"value": round(val1, 1), "unit": "tokens/s",
                                       "sample": f"{len(one)} of {len(units)} units on one "
                                                 f"thread, scaled by the share of units, "
                                                 f"{sec1:.2f} s wall"}}
    return res


def cpu_baseline():
    import oracle
    oracle.build()
    cores = cpu_cores()
    rows = CPU_SAMPLE_ROWS
    x = oracle_decode_sample(rows, DEC["seed"])
    val, sec = time_oracle_decode(x, rows, cores)
    # the same oracle on one thread, over a sixteenth of the rows
    rows1 = max(1, rows // 16)
    x1 = oracle_decode_sample(rows1, DEC["seed"])
    val1, sec1 = time_oracle_decode(x1, rows1, 1)
    return {"value": round(val, 4), "unit": "GB/s", "cores": cores, "kind": "oracle",
            "sample": f"decode: {rows} of 256 rows x 32 heads x 64 single-token steps "
                      f"(fp64 C oracle, {cores} threads over (row, head) units, "
                      f"{sec:.2f} s wall)",
            "single_thread": {"value": round(val1, 4), "unit": "GB/s",
                              "sample": f"decode: {rows1} rows x 32 heads x 64 single-token steps "
                                        f"on one thread, {sec1:.2f} s wall"},
            "prefill": cpu_baseline_prefill(cores),
            "cpu_model": cpu_model()}


def run_reference(args, rank, world):
    if rank != 0:
        return None
    import oracle
    oracle.build()
    cores = cpu_cores()
    rows = 16
    x = oracle_decode_sample(rows, DEC["seed"])
    for _ in range(args.warmup):
        time_oracle_decode(x, rows, cores)
    vals, secs = [], []
    for _ in range(args.steps):
        v, s = time_oracle_decode(x, rows, cores)
        vals.append(v)
        secs.append(s)
    value = statistics.median(vals)
    sample = (f"decode: {rows} of 256 rows x 32 heads x 64 single-token steps per step "
              f"(fp64 C oracle, {cores} threads)")
    return {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(statistics.median(secs) * 1e3, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded)",
        "config": {"workload": "decode_B256 (bounded sample on host cores)", "B": rows,
                   "steps_per_call_chain": DEC["steps"], "Hk": DEC["Hk"], "Hv": DEC["Hv"],
                   "dk": DEC["dk"], "dv": DEC["dv"], "capacity": DEC["cap"]},
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": cores,
                         "kind": "oracle", "sample": sample, "cpu_model": cpu_model()},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=30)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--only", choices=["all", "prefill", "decode", "replay", "verify", "batch", "snapshot"],
                    default="all",
                    help="profiling aid: run one phase only (prints timings, not the contract line)")
    ap.add_argument("--flush", choices=["write", "read"], default="write",
                    help="profiling aid: L2 flush before each step (read: a read-only pass, "
                         "no dirty lines for a traffic capture)")
    ap.add_argument("--decode-rows", type=int, default=DEC["B"],
                    help="profiling aid: rows of the decode / replay phases (default 256)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    rank, world, local_rank = dist_init()
    if args.impl == "reference":
        line = run_reference(args, rank, world)
        if line is not None:
            print(json.dumps(line), flush=True)
        return
    line = run_ours(args, rank, world, local_rank)
    if args.only != "all" or args.decode_rows != DEC["B"]:
        if rank == 0:
            print(json.dumps(line), flush=True)
        return
    if rank == 0:
        if world == 1 and not args.no_cpu_baseline:
            line["cpu_baseline"] = cpu_baseline()
        else:
            line["cpu_baseline"] = None
        print(json.dumps(line), flush=True)
    barrier()


if __name__ == "__main__":
    main()
