"""Shared helpers for the GPU parity tests (comparison, guard bands, moving
seeded inputs to the device).  Tolerances are the ones the recurrence's
accuracy contract fixes: relative Frobenius error 2e-4 for fp32 inputs and
2e-2 for fp16 / bf16 inputs (fp32 state either way), 1e-5 for captured
factors; decay and key captures are exact widenings and compare bit for bit.
"""
import numpy as np
import torch

TOL = {torch.float32: 2e-4, torch.float16: 2e-2, torch.bfloat16: 2e-2}
TOL_CAPTURE = 1e-5
GUARD = 256  # elements of guard band on each side (keeps 16-byte alignment)
SENTINEL_F32 = 0x7FC0DEAD  # a NaN bit pattern no kernel produces


def rel(gpu, ref) -> float:
    g = gpu.detach().cpu().double().numpy() if hasattr(gpu, "detach") else np.asarray(gpu)
    r = np.asarray(ref, dtype=np.float64)
    assert g.shape == r.shape, (g.shape, r.shape)
    assert np.all(np.isfinite(g)), "non-finite values in the GPU result"
    den = np.linalg.norm(r)
    return float(np.linalg.norm(g - r) / (den if den > 0 else 1.0))


def rel_per_unit(gpu, ref, bounds, keep_axis=1):
    """Worst relative Frobenius error over units: each unit is the slice
    [bounds[u], bounds[u+1]) of the leading (token or row) axis and one index
    of `keep_axis` (the value head), the norm taken over everything else.
    Returns (worst error, (u, head)).  Units whose reference is all zero are
    compared absolutely."""
    g = gpu.detach().cpu().double().numpy() if hasattr(gpu, "detach") else np.asarray(gpu)
    r = np.asarray(ref, dtype=np.float64)
    assert g.shape == r.shape, (g.shape, r.shape)
    assert np.all(np.isfinite(g)), "non-finite values in the GPU result"
    worst, where = 0.0, None
    for u in range(len(bounds) - 1):
        a, b = int(bounds[u]), int(bounds[u + 1])
        if b <= a:
            continue
        d = np.moveaxis(g[a:b] - r[a:b], keep_axis, 0).reshape(g.shape[keep_axis], -1)
        n = np.moveaxis(r[a:b], keep_axis, 0).reshape(r.shape[keep_axis], -1)
        num, den = np.linalg.norm(d, axis=1), np.linalg.norm(n, axis=1)
        e = num / np.where(den > 0, den, 1.0)
        h = int(np.argmax(e))
        if e[h] > worst:
            worst, where = float(e[h]), (u, h)
    return worst, where


class Guarded:
    """A device tensor with sentinel-filled guard bands on both sides."""

    def __init__(self, shape, dtype, device="cuda"):
        n = int(np.prod(shape))
        self.n = n
        self.buf = torch.empty(n + 2 * GUARD, dtype=dtype, device=device)
        self._ibuf = self.buf.view(torch.int32 if dtype == torch.float32 else torch.int16)
        pat = SENTINEL_F32 if dtype == torch.float32 else 0x7E5A
        self._ibuf.fill_(pat)
        self.pattern = self._ibuf[:1].clone()
        self.t = self.buf[GUARD:GUARD + n].view(shape)

    def guards_intact(self) -> bool:
        lo = self._ibuf[:GUARD]
        hi = self._ibuf[GUARD + self.n:]
        return bool(torch.all(lo == self.pattern).item() and torch.all(hi == self.pattern).item())

    def untouched(self, sel) -> torch.Tensor:
        """Bool mask over self.t[sel] of elements still holding the sentinel."""
        iv = self._ibuf[GUARD:GUARD + self.n].view(self.t.shape)
        return iv[sel] == self.pattern


def to_dev(x, dev="cuda"):
    g = {n: getattr(x, n).to(dev) for n in ("q", "k", "v", "alpha", "beta")}
    g["cu_seqlens"] = x.cu_seqlens.to(dev)
    g["initial_state"] = x.initial_state.to(dev) if x.initial_state is not None else None
    return g


def check_capture(su_gpu: Guarded, su_ref, counts, x, cap):
    """Captured slots [0, n_b) against the oracle (decay and key bit for bit,
    delta to TOL_CAPTURE); slots past n_b still hold the sentinel; guard
    bands intact.  Returns the n_b."""
    n = [max(0, min(int(c), cap, L)) for c, L in zip(counts, x.lengths)]
    Hv, Hk, dk = x.Hv, x.Hk, x.dk
    su = su_gpu.t
    for b, nb in enumerate(n):
        if nb > 0:
            g = su[b, :nb].cpu().double().numpy()
            r = su_ref[b, :nb]
            # decay and key: exact widenings of the inputs
            assert np.array_equal(g[:, :Hv + Hk * dk], r[:, :Hv + Hk * dk]), b
            assert rel(su[b, :nb, Hv + Hk * dk:], r[:, Hv + Hk * dk:]) < TOL_CAPTURE, b
        if nb < cap:
            assert bool(torch.all(su_gpu.untouched((b, slice(nb, cap)))).item()), \
                f"row {b}: uncaptured slots were written"
    assert su_gpu.guards_intact()
    return n
