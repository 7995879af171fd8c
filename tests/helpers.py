"""Shared test helpers: tolerance checks against the fp64 oracle.

Tolerances: bf16 outputs max-abs <= 2e-2 and mean-abs <= 2e-3, fp32 lse
abs <= 1e-3; rows whose oracle lse is +inf (no visible key) must be exactly
zero with lse +inf.
"""
import numpy as np
import torch

OUT_MAX_ABS = 2e-2
OUT_MEAN_ABS = 2e-3
LSE_ABS = 1e-3


def as_np(t):
    if isinstance(t, torch.Tensor):
        return t.detach().float().cpu().numpy().astype(np.float64)
    return np.asarray(t, dtype=np.float64)


def lse_rows_heads(lse_ref, rows, heads):
    """The oracle's lse as [rows, heads]: FIA BSND gives [B, QN, S_q], FIA TND
    and sparse give [rows, heads] already."""
    lse_ref = np.asarray(lse_ref)
    if lse_ref.ndim == 3:
        return lse_ref.transpose(0, 2, 1).reshape(rows, heads)
    return lse_ref.reshape(rows, heads)


def check_close(out_gpu, lse_gpu, out_ref, lse_ref, what=""):
    o = as_np(out_gpu).reshape(out_ref.shape)
    assert np.all(np.isfinite(o)), f"{what}: non-finite output"
    err = np.abs(o - out_ref)
    assert err.max() <= OUT_MAX_ABS, f"{what}: out max-abs {err.max():.3e}"
    assert err.mean() <= OUT_MEAN_ABS, f"{what}: out mean-abs {err.mean():.3e}"
    # rows that see no key: exactly zero, not merely within the tolerance
    rows, heads = out_ref.shape[0], out_ref.shape[1]
    empty = np.isinf(lse_rows_heads(lse_ref, rows, heads))
    if empty.any():
        assert np.all(o[empty] == 0.0), f"{what}: a row without visible keys is not exactly 0"
    if lse_gpu is not None:
        l = as_np(lse_gpu).reshape(lse_ref.shape)
        inf_ref = np.isinf(lse_ref)
        assert np.array_equal(np.isinf(l) & (l > 0), inf_ref), f"{what}: +inf pattern of lse"
        if (~inf_ref).any():
            le = np.abs(l[~inf_ref] - lse_ref[~inf_ref])
            assert le.max() <= LSE_ABS, f"{what}: lse abs {le.max():.3e}"
    return err.max(), err.mean()
