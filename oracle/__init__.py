"""CPU oracle for fused inference attention over a paged KV cache.

TEST INFRASTRUCTURE.  Only the tests, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package.  The product path
(the CUDA library and its Python binding) never imports or calls it.

Two independent formulations live here:
  * ``oracle.c`` (built into ``_build/liboracle.so``): fp64, one output row at
    a time, OpenMP over rows.  It follows the formula of the FIA pages
    ("aclnnFusedInferAttentionScoreV5", formula section:
    Attention = Softmax(Q K^T / sqrt(d)) V; "...V2", softmax_lse restriction:
    lse = log(sum(exp(s - max))) + max; "...V4", empty-tensor rule: out 0,
    lse +inf) and of the shared-KV sparse page ("kv_quant_sparse_attn_sharedkv",
    formula O = softmax(Q K~^T * softmax_scale) V~, K~ = V~).
  * ``naive.py``: a second fp64 statement in numpy that builds the whole masked
    score matrix and applies a textbook softmax, used to cross-check the C
    code on tiny shapes.

Pins (tests/test_oracle_pins.py, all CPU): probabilities of every row sum to
one; constant V returns V; Q = 0 returns the mean of the visible V rows; a
single visible key returns its V row exactly; band pre=next=0 returns v_p;
lse recomputed from the exposed probabilities; a sink only enlarges the
denominator (O_sink = O * exp(lse - lse_sink), lse_sink = logaddexp(lse, sink));
any block-table permutation equals the contiguous layout; decode equals the
last row of causal prefill; replicated KV heads equal GQA; empty KV gives 0 /
+inf; E4M3 decoding matches the OCP definition on all 256 codes and the
library's own float8 cast; the sparse path with only a window equals the band
mask of FIA, and CSA with every compressed row listed equals HCA; the
schedules cover every work item exactly once, in order, within one item of
balance; and the C code agrees with naive.py on tiny brute-force shapes.
"""
from __future__ import annotations

import ctypes
import math
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile oracle.c with gcc (-O2, OpenMP) into oracle/_build/liboracle.so."""
    os.makedirs(_BUILD, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c99", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


class _FiaArgs(ctypes.Structure):
    _fields_ = [
        ("B", ctypes.c_int32), ("QN", ctypes.c_int32), ("KVN", ctypes.c_int32),
        ("D", ctypes.c_int32), ("layout", ctypes.c_int32), ("S_q", ctypes.c_int32),
        ("T", ctypes.c_int32), ("q", ctypes.c_void_p), ("cu_seqlens_q", ctypes.c_void_p),
        ("kv_dtype", ctypes.c_int32), ("k", ctypes.c_void_p), ("v", ctypes.c_void_p),
        ("k_scale", ctypes.c_void_p), ("v_scale", ctypes.c_void_p),
        ("quant_tile", ctypes.c_int32), ("block_table", ctypes.c_void_p),
        ("max_blocks", ctypes.c_int32), ("block_size", ctypes.c_int32),
        ("S_kv", ctypes.c_int32), ("seqused_kv", ctypes.c_void_p), ("scale", ctypes.c_double),
        ("mask_mode", ctypes.c_int32), ("pre_tokens", ctypes.c_int32),
        ("next_tokens", ctypes.c_int32), ("sinks", ctypes.c_void_p),
        ("kv_layout", ctypes.c_int32), ("max_seqlen_q", ctypes.c_int32),
        ("atten_mask", ctypes.c_void_p), ("mask_batch_stride", ctypes.c_int64),
        ("mask_row_stride", ctypes.c_int64),
    ]


class _SparseArgs(ctypes.Structure):
    _fields_ = [
        ("B", ctypes.c_int32), ("N1", ctypes.c_int32), ("D", ctypes.c_int32),
        ("layout", ctypes.c_int32), ("S1", ctypes.c_int32), ("T1", ctypes.c_int32),
        ("q", ctypes.c_void_p), ("cu_seqlens_q", ctypes.c_void_p),
        ("ori_kv", ctypes.c_void_p), ("ori_block_table", ctypes.c_void_p),
        ("ori_max_blocks", ctypes.c_int32), ("ori_block_size", ctypes.c_int32),
        ("cmp_kv", ctypes.c_void_p), ("cmp_block_table", ctypes.c_void_p),
        ("cmp_max_blocks", ctypes.c_int32), ("cmp_block_size", ctypes.c_int32),
        ("cmp_sparse_indices", ctypes.c_void_p), ("K2", ctypes.c_int32),
        ("seqused_kv", ctypes.c_void_p), ("sinks", ctypes.c_void_p), ("scale", ctypes.c_double),
        ("cmp_ratio", ctypes.c_int32), ("win_left", ctypes.c_int32),
        ("win_right", ctypes.c_int32), ("kv_dtype", ctypes.c_int32),
    ]


def lib():
    global _lib
    with _lock:
        if _lib is None:
            L = ctypes.CDLL(build())
            L.oracle_fia.argtypes = [ctypes.POINTER(_FiaArgs), ctypes.c_void_p, ctypes.c_void_p,
                                     ctypes.c_int]
            L.oracle_fia.restype = ctypes.c_int
            L.oracle_sparse.argtypes = [ctypes.POINTER(_SparseArgs), ctypes.c_void_p,
                                        ctypes.c_void_p, ctypes.c_int]
            L.oracle_sparse.restype = ctypes.c_int
            L.oracle_e4m3_to_double.argtypes = [ctypes.c_uint8]
            L.oracle_e4m3_to_double.restype = ctypes.c_double
            L.oracle_bf16_to_double.argtypes = [ctypes.c_uint16]
            L.oracle_bf16_to_double.restype = ctypes.c_double
            L.oracle_e8m0_to_double.argtypes = [ctypes.c_uint8]
            L.oracle_e8m0_to_double.restype = ctypes.c_double
            L.oracle_fia_row_probs.argtypes = [ctypes.POINTER(_FiaArgs), ctypes.c_int,
                                               ctypes.c_int, ctypes.c_int64, ctypes.c_void_p,
                                               ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p]
            L.oracle_fia_row_probs.restype = ctypes.c_int64
            L.oracle_decode_schedule.argtypes = [ctypes.POINTER(_FiaArgs), ctypes.c_int32,
                                                 ctypes.c_int32, ctypes.c_void_p,
                                                 ctypes.c_void_p, ctypes.c_int64]
            L.oracle_decode_schedule.restype = ctypes.c_int64
            L.oracle_prefill_units.argtypes = [ctypes.POINTER(_FiaArgs), ctypes.c_void_p,
                                               ctypes.c_void_p, ctypes.c_int64]
            L.oracle_prefill_units.restype = ctypes.c_int64
            L.oracle_sparse_metadata.argtypes = [ctypes.POINTER(_SparseArgs), ctypes.c_int32,
                                                 ctypes.c_int32, ctypes.c_int32, ctypes.c_void_p]
            L.oracle_sparse_metadata.restype = ctypes.c_int
            L.oracle_sparse_rows.argtypes = [ctypes.POINTER(_SparseArgs), ctypes.c_int,
                                             ctypes.c_int64, ctypes.c_void_p, ctypes.c_int64]
            L.oracle_sparse_rows.restype = ctypes.c_int64
            L.oracle_fia_sample.argtypes = [ctypes.POINTER(_FiaArgs), ctypes.c_void_p,
                                            ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p,
                                            ctypes.c_void_p, ctypes.c_int]
            L.oracle_fia_sample.restype = ctypes.c_int
            _lib = L
    return _lib


# ----------------------------------------------------------------------------
# marshalling (CPU tensors / numpy arrays -> C structs)
# ----------------------------------------------------------------------------

def _np(t, dtype=None):
    """Contiguous host numpy view of a CPU torch tensor (bf16 -> uint16 bits,
    uint8 codes stay uint8)."""
    if t is None:
        return None
    import torch
    if isinstance(t, torch.Tensor):
        t = t.detach().cpu().contiguous()
        if t.dtype == torch.bfloat16:
            t = t.view(torch.int16)
        a = t.numpy()
        if a.dtype == np.int16:
            a = a.view(np.uint16)
    else:
        a = np.ascontiguousarray(t)
    if dtype is not None:
        a = a.astype(dtype, copy=False)
    return np.ascontiguousarray(a)


def _ptr(a):
    return None if a is None else a.ctypes.data


def _fia_struct(p):
    keep = {
        "q": _np(p.q), "cu": _np(p.cu_seqlens_q, np.int32), "k": _np(p.k_cache),
        "v": _np(p.v_cache), "ks": _np(p.k_scale, np.float32), "vs": _np(p.v_scale, np.float32),
        "bt": _np(p.block_table, np.int32), "sk": _np(p.seqused_kv, np.int32),
        "sinks": _np(p.sinks, np.float32),
        "mask": _np(getattr(p, "atten_mask", None)),
    }
    mask = getattr(p, "atten_mask", None)
    if mask is not None:
        mrs, mbs = int(mask.shape[2]), (0 if mask.shape[0] == 1 else int(mask.shape[1] * mask.shape[2]))
    else:
        mrs = mbs = 0
    s = _FiaArgs(B=p.B, QN=p.QN, KVN=p.KVN, D=p.D, layout=p.layout, S_q=p.S_q, T=p.T,
                 q=_ptr(keep["q"]), cu_seqlens_q=_ptr(keep["cu"]), kv_dtype=p.kv_dtype,
                 k=_ptr(keep["k"]), v=_ptr(keep["v"]), k_scale=_ptr(keep["ks"]),
                 v_scale=_ptr(keep["vs"]), quant_tile=64, block_table=_ptr(keep["bt"]),
                 max_blocks=p.max_blocks, block_size=p.block_size or 1, S_kv=p.S_kv,
                 seqused_kv=_ptr(keep["sk"]), scale=p.scale, mask_mode=p.mask_mode,
                 pre_tokens=p.pre_tokens, next_tokens=p.next_tokens, sinks=_ptr(keep["sinks"]),
                 kv_layout=getattr(p, "kv_layout", 0), max_seqlen_q=max(p.S_q, 1),
                 atten_mask=_ptr(keep["mask"]), mask_batch_stride=mbs, mask_row_stride=mrs)
    return s, keep


def _sparse_struct(p):
    keep = {
        "q": _np(p.q), "cu": _np(p.cu_seqlens_q, np.int32), "ori": _np(p.ori_kv),
        "obt": _np(p.ori_block_table, np.int32), "cmp": _np(p.cmp_kv),
        "cbt": _np(p.cmp_block_table, np.int32), "idx": _np(p.cmp_sparse_indices, np.int32),
        "sk": _np(p.seqused_kv, np.int32), "sinks": _np(p.sinks, np.float32),
    }
    s = _SparseArgs(B=p.B, N1=p.N1, D=p.D, layout=p.layout, S1=p.S1, T1=p.T1,
                    q=_ptr(keep["q"]), cu_seqlens_q=_ptr(keep["cu"]), ori_kv=_ptr(keep["ori"]),
                    ori_block_table=_ptr(keep["obt"]),
                    ori_max_blocks=int(p.ori_block_table.shape[1]),
                    ori_block_size=p.ori_block_size, cmp_kv=_ptr(keep["cmp"]),
                    cmp_block_table=_ptr(keep["cbt"]),
                    cmp_max_blocks=0 if p.cmp_block_table is None else int(
                        p.cmp_block_table.shape[1]),
                    cmp_block_size=p.cmp_block_size or 1,
                    cmp_sparse_indices=_ptr(keep["idx"]), K2=p.K2, seqused_kv=_ptr(keep["sk"]),
                    sinks=_ptr(keep["sinks"]), scale=p.scale, cmp_ratio=p.cmp_ratio or 1,
                    win_left=p.win_left, win_right=p.win_right,
                    kv_dtype=getattr(p, "kv_dtype", 0))
    return s, keep


# ----------------------------------------------------------------------------
# public oracle calls
# ----------------------------------------------------------------------------

def fia(p, nthreads: int = 0):
    """Fused inference attention in fp64.  Returns (out [rows, QN, D] float64,
    lse float64: BSND [B, QN, S_q], TND [T, QN])."""
    s, keep = _fia_struct(p)
    rows = p.rows
    out = np.zeros((rows, p.QN, p.D), dtype=np.float64)
    if p.layout == 1:
        lse = np.zeros((rows, p.QN), dtype=np.float64)
    else:
        lse = np.zeros((p.B, p.QN, p.S_q), dtype=np.float64)
    rc = lib().oracle_fia(ctypes.byref(s), out.ctypes.data, lse.ctypes.data, nthreads)
    assert rc == 0
    del keep
    return out, lse


def fia_sample(p, rows, heads, nthreads: int = 0):
    """Oracle values for a sample of (query row, head) pairs only (full-size
    parity where the whole oracle would take too long).  Returns
    (out [n, D], lse [n])."""
    s, keep = _fia_struct(p)
    rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
    heads = np.ascontiguousarray(np.asarray(heads, dtype=np.int32))
    n = rows.shape[0]
    out = np.zeros((n, p.D), dtype=np.float64)
    lse = np.zeros(n, dtype=np.float64)
    rc = lib().oracle_fia_sample(ctypes.byref(s), rows.ctypes.data, heads.ctypes.data, n,
                                 out.ctypes.data, lse.ctypes.data, nthreads)
    assert rc == 0
    del keep
    return out, lse


def sparse(p, nthreads: int = 0):
    """Shared-KV sparse attention in fp64.  Returns (out [rows, N1, D],
    lse [rows, N1])."""
    s, keep = _sparse_struct(p)
    out = np.zeros((p.rows, p.N1, p.D), dtype=np.float64)
    lse = np.zeros((p.rows, p.N1), dtype=np.float64)
    rc = lib().oracle_sparse(ctypes.byref(s), out.ctypes.data, lse.ctypes.data, nthreads)
    assert rc == 0
    del keep
    return out, lse


def sparse_rows(p, b: int, i: int):
    """Logical K~ rows of query i of batch b: list of ('ori'|'cmp', row)."""
    s, keep = _sparse_struct(p)
    cap = 1 << 20
    buf = np.zeros(cap, dtype=np.int64)
    n = lib().oracle_sparse_rows(ctypes.byref(s), b, i, buf.ctypes.data, cap)
    assert n >= 0
    return [("cmp" if (e & 1) else "ori", int(e >> 1)) for e in buf[:n]]


def fia_row_probs(p, b: int, h: int, i: int):
    """(lo, probabilities of the visible positions lo.., sink probability)."""
    s, keep = _fia_struct(p)
    cap = max(p.S_kv, 1) + 1
    buf = np.zeros(cap, dtype=np.float64)
    lo = ctypes.c_int64(0)
    ps = ctypes.c_double(0.0)
    n = lib().oracle_fia_row_probs(ctypes.byref(s), b, h, i, buf.ctypes.data, cap,
                                   ctypes.addressof(lo), ctypes.addressof(ps))
    assert n >= 0
    return lo.value, buf[:n].copy(), ps.value


def e4m3_to_double(code: int) -> float:
    return lib().oracle_e4m3_to_double(code)


def bf16_to_double(bits: int) -> float:
    return lib().oracle_bf16_to_double(bits)


def e8m0_to_double(code: int) -> float:
    return lib().oracle_e8m0_to_double(code)


def lse_combine(outs, lses, sinks=None, head_axis=None):
    """Attention over the union of disjoint key sets from the results over
    each set ("aclnnFusedInferAttentionScoreV2", softmax_lse restriction: the
    lse exists for ring attention, which joins partial results this way):
        lse = log(sum_k exp(lse_k) + exp(sink)),   O = sum_k exp(lse_k - lse) * O_k,
    leaving out parts with lse_k = +inf (they saw no key); when every part is
    left out, O = 0 and lse = +inf.  The parts are computed without sinks;
    `sinks[h]` (optional) is the sink of head h, the index along `head_axis`
    of the lse arrays, added once.  `outs[k]` is [..., D], `lses[k]` the
    matching [...]; fp64 throughout, parts in the order given."""
    outs = [np.asarray(o, dtype=np.float64) for o in outs]
    lses = [np.asarray(l, dtype=np.float64) for l in lses]
    shape = lses[0].shape
    out = np.zeros(outs[0].shape, dtype=np.float64)
    lse = np.full(shape, np.inf)
    for idx in np.ndindex(*shape):
        vals = [l[idx] for l in lses if not np.isinf(l[idx])]
        if not vals:
            continue
        if sinks is not None:
            vals.append(float(sinks[idx[head_axis]]))
        m = max(vals)
        tot = m + math.log(sum(math.exp(v - m) for v in vals))
        lse[idx] = tot
        for o, l in zip(outs, lses):
            if not np.isinf(l[idx]):
                out[idx] += math.exp(l[idx] - tot) * o[idx]
    return out, lse


def decode_schedule(p, num_ctas: int, per_cta: int):
    """(sched int64 [8 + 3(B+1) + B], queue int32 [N, 4]) of the decode chunk
    schedule for n CTAs and W = per_cta chunks per CTA."""
    s, keep = _fia_struct(p)
    G = p.QN // p.KVN
    HG = -(-(max(1, p.S_q) * G) // 8)  # units per KV head, at most (8-column groups)
    U = p.B * p.KVN * HG
    k = 2 if (p.kv_dtype == 0 and max(p.S_q, 1) == 1) else 1  # small chunks: ceil(C/k) tiles
    cap = num_ctas * per_cta + 2 * k * U
    sched = np.zeros(8 + 3 * (p.B + 1) + p.B, dtype=np.int64)
    queue = np.zeros((max(cap, 1), 4), dtype=np.int32)
    n = lib().oracle_decode_schedule(ctypes.byref(s), num_ctas, per_cta, sched.ctypes.data,
                                     queue.ctypes.data, cap)
    assert n >= 0, "more chunks than the bound"
    return sched, queue[:n].copy()


def prefill_units(p):
    """(units int32 [n,4] as (b, q_tile, hk, pair), cost int64 [n]) in canonical
    order."""
    s, keep = _fia_struct(p)
    cap = 1
    for b in range(p.B):
        cap += -(-p.q_lens[b] // 128)
    cap *= p.QN
    units = np.zeros((cap, 4), dtype=np.int32)
    cost = np.zeros(cap, dtype=np.int64)
    n = lib().oracle_prefill_units(ctypes.byref(s), units.ctypes.data, cost.ctypes.data, cap)
    assert n >= 0
    return units[:n].copy(), cost[:n].copy()


def sparse_metadata(p, num_ctas: int, chunk: int = 64, heads: int = 8):
    s, keep = _sparse_struct(p)
    md = np.zeros(1024, dtype=np.int32)
    rc = lib().oracle_sparse_metadata(ctypes.byref(s), num_ctas, chunk, heads, md.ctypes.data)
    assert rc == 0
    return md
