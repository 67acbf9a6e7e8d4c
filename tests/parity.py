"""Comparison of CUDA outputs with the oracle, shared by the GPU tests and
the benchmark's parity line.

Bar: reduced and residual_out bit for bit; norm_out within 1 bf16 ulp
(ordered-integer distance, +0 == -0); NaN where the oracle has NaN and
nowhere else (payloads are not compared).
"""
from __future__ import annotations

import numpy as np

NORM_ULP_TOL = 1


def u16(t) -> np.ndarray:
    """torch bf16 tensor (any device) -> numpy uint16 bit patterns."""
    import torch
    return t.detach().view(torch.int16).cpu().numpy().view(np.uint16)


def _nan(b):
    return ((b & 0x7F80) == 0x7F80) & ((b & 0x7F) != 0)


def _ordered(b):
    b = b.astype(np.int32)
    return np.where(b & 0x8000, -(b & 0x7FFF), b & 0x7FFF)


def compare(got, want) -> dict:
    """got/want: (reduced, residual_out, norm_out) uint16 arrays."""
    out = {}
    for name, g, w in zip(("reduced", "residual_out", "norm_out"), got, want):
        g, w = np.asarray(g), np.asarray(w)
        assert g.shape == w.shape, (name, g.shape, w.shape)
        gn, wn = _nan(g), _nan(w)
        nan_mismatch = int((gn != wn).sum())
        both = ~gn & ~wn
        if name == "norm_out":
            d = np.abs(_ordered(g) - _ordered(w))
            d = np.where(both, d, 0)
            out[name] = dict(max_ulp=int(d.max()) if d.size else 0,
                             n_off=int((d > 0).sum()),
                             n_bad=int((d > NORM_ULP_TOL).sum()) + nan_mismatch)
        else:
            neq = both & (g != w)
            out[name] = dict(n_bad=int(neq.sum()) + nan_mismatch)
    return out


def assert_parity(got, want, what: str = "") -> dict:
    r = compare(got, want)
    assert r["reduced"]["n_bad"] == 0, f"{what}: reduced differs in {r['reduced']['n_bad']} elements"
    assert r["residual_out"]["n_bad"] == 0, \
        f"{what}: residual_out differs in {r['residual_out']['n_bad']} elements"
    assert r["norm_out"]["n_bad"] == 0, \
        f"{what}: norm_out beyond {NORM_ULP_TOL} ulp in {r['norm_out']['n_bad']} elements " \
        f"(max {r['norm_out']['max_ulp']})"
    return r


def sample_rows(T: int, n: int, seed: int = 0) -> np.ndarray:
    """First, last and a seeded spread of rows (sorted, unique)."""
    rng = np.random.default_rng(seed)
    rows = {0, T - 1, T // 2}
    rows.update(int(v) for v in rng.integers(0, T, size=max(0, n - 3)))
    return np.array(sorted(r for r in rows if 0 <= r < T), dtype=np.int64)
