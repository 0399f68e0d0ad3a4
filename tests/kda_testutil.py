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


def row_errors(x, y, head_axis, row_axes):
    """Two finer views of the error, per head (the largest over heads is returned):
      rows: for every row (the elements sharing the indices in `row_axes`, e.g. one token of
            an output or one key channel of a state), max |x - y| over the row divided by the
            row's own max |y|, that max floored at 1e-6 of the head's max |y|;
      elems: max over elements of |x - y| / max(|y|, 1e-6 max |y| of the head).
    A mistake confined to a few small-magnitude rows (the tail rows of a partial chunk, say)
    stands out in `rows` while it may hide under the normwise metric of the whole head."""
    x = np.asarray(x, dtype=np.float64)
    y = np.asarray(y, dtype=np.float64)
    xm = np.moveaxis(x, head_axis, 0)
    ym = np.moveaxis(y, head_axis, 0)
    ra = tuple(a - (1 if a > head_axis else 0) + 1 for a in row_axes)
    red = tuple(a for a in range(1, xm.ndim) if a not in ra)
    worst_rows = worst_elems = 0.0
    for h in range(xm.shape[0]):
        xs, ys = xm[h], ym[h]
        floor = 1e-6 * np.abs(ys).max()
        if floor == 0:
            continue
        err = np.abs(xs - ys)
        r_red = tuple(a - 1 for a in red)
        row_err = err.max(axis=r_red) if r_red else err
        row_den = np.maximum(np.abs(ys).max(axis=r_red) if r_red else np.abs(ys), floor)
        worst_rows = max(worst_rows, float((row_err / row_den).max()))
        worst_elems = max(worst_elems, float((err / np.maximum(np.abs(ys), floor)).max()))
    return worst_rows, worst_elems


def rows_o(x, y):
    """row_errors of an output [T, H, dv]: one row per (token, head)."""
    return row_errors(x, y, 1, (0,))


def rows_s(x, y):
    """row_errors of states [N, H, dk, dv]: one row per (state, head, key channel)."""
    return row_errors(x, y, 1, (0, 2))


def tc_path(n_ranges, T, H, dk=128, dv=128):
    """True when a bf16 chunked call of this shape runs on the tensor-core kernels: their
    workspace query is positive exactly then, and such a call never falls back to the CUDA-core
    kernel (it fails with an error instead)."""
    from linear_attention_state_kda_gb300 import kda
    return kda.chunk_workspace(torch.bfloat16, n_ranges, T, H, dk, dv) > 0
