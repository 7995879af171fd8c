"""Second, independent fp64 statement of the attention the oracle computes.

TEST INFRASTRUCTURE (see oracle/__init__.py).  Written as matrices rather than
rows: gather each sequence's K and V into dense [kv_len, KVN, D] arrays through
the block table, form the whole score matrix S = scale * Q K^T per head, build
the boolean visibility matrix of the mask mode (query rows aligned to the
bottom-right corner, or to the top-left for the left-up causal mode; an
explicit mask's ones removed), and apply a textbook softmax with the sink as one
extra column that carries no value ("aclnnFusedInferAttentionScoreV5" formula
section; "...V2" softmax_lse restriction; "...V4" empty-tensor rule).  Only for
tiny shapes: it materialises every score.
"""
from __future__ import annotations

import numpy as np


def _bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def _e4m3_to_f64(codes: np.ndarray) -> np.ndarray:
    c = codes.astype(np.int64)
    s = np.where(c >> 7, -1.0, 1.0)
    e = (c >> 3) & 15
    m = c & 7
    v = np.where(e == 0, m / 8.0 * 2.0 ** -6, (1.0 + m / 8.0) * np.exp2(e - 7.0))
    v = np.where((e == 15) & (m == 7), np.nan, v)
    return s * v


def _as_np(t):
    import torch
    t = t.detach().cpu().contiguous()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()


def _dense_kv(p, b, which):
    pool = _as_np(p.k_cache if which == "k" else p.v_cache)
    if getattr(p, "kv_layout", 0) == 1:
        # head-major pages [nb, KVN, bs, D] -> token-major [nb, bs, KVN, D]
        pool = pool.transpose(0, 2, 1, 3)
    kvl = p.kv_lens[b]
    if p.kv_dtype == 0:
        vals = _bf16_bits_to_f64(pool)
    else:
        # stored [pages, KVN, rows, D/64]; back to [pages, rows, KVN, D/64]
        sc = _as_np(p.k_scale if which == "k" else p.v_scale).astype(np.float64)
        sc = sc.transpose(0, 2, 1, 3)
        vals = _e4m3_to_f64(pool) * np.repeat(sc, 64, axis=-1)
    if p.block_table is not None:
        bt = _as_np(p.block_table)
        bs = p.block_size
        j = np.arange(kvl)
        phys = bt[b, j // bs].astype(np.int64) * bs + j % bs
        flat = vals.reshape(-1, p.KVN, p.D)
        return flat[phys]
    return vals[b, :kvl]


def fia(p):
    """Returns (out [rows, QN, D], lse like the oracle's)."""
    q_all = _bf16_bits_to_f64(_as_np(p.q)).reshape(-1, p.QN, p.D)
    G = p.QN // p.KVN
    out = np.zeros((p.rows, p.QN, p.D))
    lse_rows = np.full((p.rows, p.QN), np.inf)
    sinks = None if p.sinks is None else _as_np(p.sinks).astype(np.float64)
    start = 0
    for b in range(p.B):
        ql, kl = p.q_lens[b], p.kv_lens[b]
        qs = start if p.layout == 1 else b * p.S_q
        start += ql
        if ql == 0:
            continue
        if kl == 0:
            continue
        K = _dense_kv(p, b, "k")
        V = _dense_kv(p, b, "v")
        i = np.arange(ql)[:, None]
        j = np.arange(kl)[None, :]
        pos = (0 if p.mask_mode == 2 else kl - ql) + i
        if p.mask_mode in (2, 3):
            vis = j <= pos
        elif p.mask_mode == 4:
            vis = (j >= pos - p.pre_tokens) & (j <= pos + p.next_tokens)
        else:
            vis = np.ones((ql, kl), dtype=bool)
        mask = getattr(p, "atten_mask", None)
        if mask is not None:  # 1 = masked out
            mk = _as_np(mask)
            vis = vis & (mk[0 if mk.shape[0] == 1 else b, :ql, :kl] == 0)
        for h in range(p.QN):
            g = h // G
            S = p.scale * (q_all[qs:qs + ql, h, :] @ K[:, g, :].T)
            S = np.where(vis, S, -np.inf)
            cols = [S]
            if sinks is not None:
                cols.append(np.full((ql, 1), sinks[h]))
            Z = np.concatenate(cols, axis=1)
            m = Z.max(axis=1, keepdims=True)
            any_vis = vis.any(axis=1)
            m = np.where(np.isfinite(m), m, 0.0)
            E = np.exp(Z - m)
            den = E.sum(axis=1, keepdims=True)
            P = E[:, :kl] / den
            O = P @ V[:, g, :]
            O[~any_vis] = 0.0
            out[qs:qs + ql, h, :] = O
            lse = (m + np.log(den))[:, 0]
            lse[~any_vis] = np.inf
            lse_rows[qs:qs + ql, h] = lse
    if p.layout == 1:
        return out, lse_rows
    return out, lse_rows.reshape(p.B, p.S_q, p.QN).transpose(0, 2, 1).copy()
