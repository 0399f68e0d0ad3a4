"""Helpers shared by the GPU parity tests: host copies for the oracle and the error metric.

Tolerances (normwise, per head): outputs and states of fp32 inputs within 1e-4 relative;
with bf16 q/k/v, outputs within 2e-2 and fp32 states within 5e-3. The metric is
max_i |x_i - y_i| / max_i |y_i| over one head's tensor, the largest over heads: an
element-wise relative error is meaningless where strongly decayed states are ~0.
"""
import numpy as np
import torch

TOL_F32 = 1e-4
TOL_BF16_O = 2e-2
TOL_BF16_S = 5e-3


def f64(t):
    """Host float64 copy of a tensor (bf16 values widen exactly)."""
    return t.detach().float().cpu().numpy().astype(np.float64)


def rel_per_head(x, y, head_axis):
    x = np.asarray(x, dtype=np.float64)
    y = np.asarray(y, dtype=np.float64)
    worst = 0.0
    for h in range(x.shape[head_axis]):
        xs = np.take(x, h, axis=head_axis)
        ys = np.take(y, h, axis=head_axis)
        den = np.abs(ys).max()
        err = np.abs(xs - ys).max()
        worst = max(worst, float(err / den) if den > 0 else float(err))
    return worst


def rel_o(x, y):
    """o / v layout [T, H, d]."""
    return rel_per_head(x, y, 1)


def rel_s(x, y):
    """state layout [N, H, dk, dv]."""
    return rel_per_head(x, y, 1)


def oracle_inputs(x, heads=None):
    """float64 host copies of a PrefillInputs, optionally restricted to some heads."""
    sel = (lambda t: t) if heads is None else (lambda t: t[:, heads])
    d = dict(q=f64(sel(x.q)), k=f64(sel(x.k)), v=f64(sel(x.v)), g=f64(sel(x.g)),
             beta=f64(sel(x.beta)), cu_seqlens=x.cu_seqlens.cpu().numpy().astype(np.int64))
    d["init_state"] = None if x.init_state is None else f64(sel(x.init_state))
    return d


def tols(dtype):
    if dtype == torch.float32:
        return TOL_F32, TOL_F32
    return TOL_BF16_O, TOL_BF16_S


def rel_gpu(x, y, head_axis=1):
    """Same metric as rel_per_head, evaluated on the device (for GPU-vs-GPU comparisons of
    large tensors)."""
    x = x.float().movedim(head_axis, 0).reshape(x.shape[head_axis], -1)
    y = y.float().movedim(head_axis, 0).reshape(y.shape[head_axis], -1)
    err = (x - y).abs().amax(dim=1)
    den = y.abs().amax(dim=1)
    r = torch.where(den > 0, err / den.clamp_min(1e-30), err)
    return float(r.max().item())
