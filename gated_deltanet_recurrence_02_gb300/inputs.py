"""Seeded synthetic inputs for the gated delta-rule workloads.

This module holds none of the recurrence's arithmetic.  It draws random
tensors with the distributions of the workloads and rounds them to their
storage dtype; the CUDA path and the CPU oracle are both fed from here, so
both see bit-identical inputs.

Recipe (every workload): q, k ~ N(0, 1), L2-normalised per head over dk,
then q *= 1/sqrt(dk); v ~ N(0, 1); beta = sigmoid(N(0, 1));
alpha = exp(-U(0.01, 0.5)); initial state ~ 0.1 * N(0, 1).  Draws come from
numpy's PCG64 in a fixed order (q, k, v, beta, alpha, state), in fp32, and
are rounded to fp16 / bf16 by round-to-nearest-even where the workload stores
16-bit values.
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import Optional, Sequence

import numpy as np
import torch

DTYPES = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}


@dataclass
class GdnInputs:
    q: torch.Tensor                 # [total_T, Hk, dk]  (CPU, storage dtype)
    k: torch.Tensor                 # [total_T, Hk, dk]
    v: torch.Tensor                 # [total_T, Hv, dv]
    alpha: torch.Tensor             # [total_T, Hv]      decay in (0, 1]
    beta: torch.Tensor              # [total_T, Hv]
    cu_seqlens: torch.Tensor        # [B + 1] int32
    initial_state: Optional[torch.Tensor]   # [N0, Hv, dv, dk] fp32 or None
    B: int
    Hk: int
    Hv: int
    dk: int
    dv: int
    scale: float = 1.0
    lengths: list = field(default_factory=list)

    @property
    def total_T(self) -> int:
        return int(self.cu_seqlens[-1])

    @property
    def uniform_T(self) -> Optional[int]:
        """Tokens per row when every row has the same length, else None."""
        return self.lengths[0] if len(set(self.lengths)) == 1 else None


def _round(x: np.ndarray, dtype: str) -> torch.Tensor:
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32))
    return t.to(DTYPES[dtype]).contiguous()


def _l2norm(x: np.ndarray) -> np.ndarray:
    n = np.sqrt(np.sum(x.astype(np.float64) ** 2, axis=-1, keepdims=True))
    return (x / np.maximum(n, 1e-12)).astype(np.float32)


def make_inputs(seed: int, *, lengths: Sequence[int], Hk: int, Hv: int,
                dk: int, dv: int, dtype_qkv: str = "bf16",
                dtype_gate: str = "f32", n_states: Optional[int] = None,
                zero_state: bool = False) -> GdnInputs:
    """Draw one workload.  ``lengths``: tokens per row (ragged allowed).
    ``n_states``: number of initial states to draw (default: one per row);
    ``zero_state``: no initial state (the path starts from zeros)."""
    rng = np.random.Generator(np.random.PCG64(seed))
    B = len(lengths)
    total = int(sum(lengths))
    q = rng.standard_normal((total, Hk, dk), dtype=np.float32)
    k = rng.standard_normal((total, Hk, dk), dtype=np.float32)
    q = _l2norm(q) * np.float32(1.0 / np.sqrt(dk))
    k = _l2norm(k)
    v = rng.standard_normal((total, Hv, dv), dtype=np.float32)
    beta = 1.0 / (1.0 + np.exp(-rng.standard_normal((total, Hv), dtype=np.float32)))
    alpha = np.exp(-rng.uniform(0.01, 0.5, size=(total, Hv)).astype(np.float32))
    S0 = None
    if not zero_state:
        n0 = B if n_states is None else n_states
        S0 = torch.from_numpy(
            np.float32(0.1) * rng.standard_normal((n0, Hv, dv, dk), dtype=np.float32))
    cu = np.zeros(B + 1, dtype=np.int32)
    cu[1:] = np.cumsum(np.asarray(lengths, dtype=np.int64))
    return GdnInputs(
        q=_round(q, dtype_qkv), k=_round(k, dtype_qkv), v=_round(v, dtype_qkv),
        alpha=_round(alpha, dtype_gate), beta=_round(beta, dtype_gate),
        cu_seqlens=torch.from_numpy(cu), initial_state=S0, B=B, Hk=Hk, Hv=Hv,
        dk=dk, dv=dv, scale=1.0, lengths=[int(x) for x in lengths])


def make_raw_inputs(seed: int, *, lengths: Sequence[int], Hk: int, Hv: int, dk: int,
                    dv: int, dtype_qkv: str = "bf16", dtype_gate: str = "f32",
                    zero_state: bool = False) -> GdnInputs:
    """Inputs in a layer's raw conventions, for the in-kernel front end: q, k
    ~ N(0, 1) times a per-token, per-head magnitude ~ U(0.5, 2) (neither
    normalised nor scaled), v ~ N(0, 1), beta as logits ~ N(0, 1), alpha as the
    log-decay g = -U(0.01, 0.5), initial state 0.1 * N(0, 1).  Drawn in that
    order from PCG64(seed), rounded to the storage dtypes."""
    rng = np.random.Generator(np.random.PCG64(seed))
    B = len(lengths)
    total = int(sum(lengths))
    q = rng.standard_normal((total, Hk, dk), dtype=np.float32)
    k = rng.standard_normal((total, Hk, dk), dtype=np.float32)
    q *= rng.uniform(0.5, 2.0, size=(total, Hk, 1)).astype(np.float32)
    k *= rng.uniform(0.5, 2.0, size=(total, Hk, 1)).astype(np.float32)
    v = rng.standard_normal((total, Hv, dv), dtype=np.float32)
    beta = rng.standard_normal((total, Hv), dtype=np.float32)
    alpha = -rng.uniform(0.01, 0.5, size=(total, Hv)).astype(np.float32)
    S0 = None
    if not zero_state:
        S0 = torch.from_numpy(
            np.float32(0.1) * rng.standard_normal((B, Hv, dv, dk), dtype=np.float32))
    cu = np.zeros(B + 1, dtype=np.int32)
    cu[1:] = np.cumsum(np.asarray(lengths, dtype=np.int64))
    return GdnInputs(
        q=_round(q, dtype_qkv), k=_round(k, dtype_qkv), v=_round(v, dtype_qkv),
        alpha=_round(alpha, dtype_gate), beta=_round(beta, dtype_gate),
        cu_seqlens=torch.from_numpy(cu), initial_state=S0, B=B, Hk=Hk, Hv=Hv,
        dk=dk, dv=dv, scale=float(1.0 / np.sqrt(dk)), lengths=[int(x) for x in lengths])


def capture_counts(seed: int, B: int, capacity: int) -> torch.Tensor:
    """capture_count[b] ~ U{0..capacity}, int32."""
    rng = np.random.Generator(np.random.PCG64(seed))
    return torch.from_numpy(rng.integers(0, capacity + 1, size=B).astype(np.int32))


def ragged_lengths(seed: int, B: int, lo: int, hi: int) -> list:
    """B row lengths ~ U{lo..hi}."""
    rng = np.random.Generator(np.random.PCG64(seed))
    return [int(x) for x in rng.integers(lo, hi + 1, size=B)]


def accepted_counts(seed: int, B: int, capacity: int) -> torch.Tensor:
    """Draft tokens accepted per row ~ U{0..capacity}, int32."""
    rng = np.random.Generator(np.random.PCG64(seed))
    return torch.from_numpy(rng.integers(0, capacity + 1, size=B).astype(np.int32))


# The workloads, by what they are.  Seeds are fixed per workload.
WORKLOADS = {
    "tiny_f32": dict(seed=1000, lengths=[64, 64], Hk=1, Hv=2, dk=32, dv=32,
                     dtype_qkv="f32", dtype_gate="f32", chunk=16,
                     capacity=7, capture_count=[3, 7]),
    "ragged_capture_qwenlike_f16": dict(
        seed=1001, lengths=[8, 8, 8], Hk=2, Hv=6, dk=128, dv=128,
        dtype_qkv="f16", dtype_gate="f16", capacity=7,
        capture_count=[0, 4, 7]),
    "prefill_T4100": dict(seed=1002, lengths=[4100], Hk=16, Hv=32, dk=128,
                          dv=128, dtype_qkv="bf16", dtype_gate="f32",
                          chunk=64),
    "prefix_snapshot_B12": dict(seed=1003, prefix_len=2048, B=12, lo=200,
                                hi=1000, Hk=16, Hv=32, dk=128, dv=128,
                                dtype_qkv="bf16", dtype_gate="bf16", chunk=64),
    "decode_B256": dict(seed=1004, B=256, steps=64, Hk=16, Hv=32, dk=128,
                        dv=128, dtype_qkv="bf16", dtype_gate="bf16",
                        capacity=4),
    # batched prefill of packed rows: 64 rows of 500 .. 1500 tokens
    "prefill_batch_B64": dict(seed=1006, B=64, lo=500, hi=1500, Hk=16, Hv=32, dk=128,
                              dv=128, dtype_qkv="bf16", dtype_gate="f32", chunk=64),
    # speculative decoding: each step replays the accepted prefix of the
    # previous step's 4 captured drafts (accepted ~ U{0..4}) and verifies 4
    # new draft tokens per row, all captured
    "verify_B256_T4": dict(seed=1005, B=256, steps=16, T=4, Hk=16, Hv=32,
                           dk=128, dv=128, dtype_qkv="bf16", dtype_gate="bf16",
                           capacity=4),
}
