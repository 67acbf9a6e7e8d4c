"""Helpers shared by the GPU test files (no tests here)."""
import os

import torch

import rank_sum_residual_gb300 as farn
from parity import u16


def make_ctx(**env):
    """A context created under the given FARN_* environment (read at create)."""
    old = {k: os.environ.get(k) for k in env}
    try:
        for k, v in env.items():
            os.environ[k] = str(v)
        return farn.Context(0)
    finally:
        for k, v in old.items():
            if v is None:
                os.environ.pop(k, None)
            else:
                os.environ[k] = v


def host(t):
    """Partials for the oracle: bf16 patterns, or fp32 values as they are."""
    if t.dtype == torch.float32:
        return t.detach().cpu().numpy()
    return u16(t)


def oracle_rows(O, xs, res, w, eps, rows=None):
    """The oracle's (reduced, residual_out, norm_out) for all rows or the
    given ones, from the device tensors' bytes."""
    if rows is None:
        return O.forward([host(x) for x in xs], u16(res), u16(w), eps)
    idx = torch.as_tensor(rows, device=res.device)
    return O.forward([host(x.index_select(0, idx)) for x in xs],
                     u16(res.index_select(0, idx)), u16(w), eps)
