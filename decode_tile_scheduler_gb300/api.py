"""PyTorch-facing helpers: build the C-ABI parameter structs from tensors,
allocate outputs and workspaces with torch, and launch on torch's current
CUDA stream.  Memory and streams only -- the computation is libfia's.
"""
from __future__ import annotations

import math
from typing import Optional

import torch

from . import _abi
from ._abi import FiaParams, SparseParams


def _ptr(t: Optional[torch.Tensor]) -> Optional[int]:
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("libfia takes CUDA tensors")
    return t.data_ptr()


def _stream(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _contig(t: Optional[torch.Tensor], name: str):
    if t is not None and not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t


def make_fia_params(*, q: torch.Tensor, out: torch.Tensor, k_cache: torch.Tensor,
                    v_cache: torch.Tensor, num_q_heads: int, num_kv_heads: int, head_dim: int,
                    batch: int, layout: int, max_seqlen_q: int, total_q: int = 0,
                    lse: Optional[torch.Tensor] = None, kv_dtype: int = _abi.KV_BF16,
                    k_scale: Optional[torch.Tensor] = None,
                    v_scale: Optional[torch.Tensor] = None,
                    block_table: Optional[torch.Tensor] = None, block_size: int = 0,
                    num_blocks: int = 0, max_seqlen_kv: int = 0,
                    cu_seqlens_q: Optional[torch.Tensor] = None,
                    seqused_kv: Optional[torch.Tensor] = None, scale: Optional[float] = None,
                    mask_mode: int = _abi.MASK_NONE, pre_tokens: int = 0, next_tokens: int = 0,
                    sinks: Optional[torch.Tensor] = None, num_sms: int = 0,
                    kv_layout: int = _abi.KV_LAYOUT_BNBSH,
                    atten_mask: Optional[torch.Tensor] = None) -> FiaParams:
    """`atten_mask`: int8/uint8/bool [B or 1, rows, cols] (nonzero = masked
    out), rows >= the query length, cols a multiple of 16 >= the KV capacity;
    a first dimension of 1 is shared by every batch."""
    for name, t in (("q", q), ("out", out), ("k_cache", k_cache), ("v_cache", v_cache)):
        _contig(t, name)
    p = FiaParams()
    p.batch, p.num_q_heads, p.num_kv_heads, p.head_dim = batch, num_q_heads, num_kv_heads, head_dim
    p.layout, p.max_seqlen_q, p.total_q = layout, max_seqlen_q, total_q
    p.q, p.out, p.lse = _ptr(q), _ptr(out), _ptr(lse)
    p.k_cache, p.v_cache = _ptr(k_cache), _ptr(v_cache)
    p.k_scale, p.v_scale = _ptr(k_scale), _ptr(v_scale)
    p.kv_dtype = kv_dtype
    p.quant_tile = 64 if kv_dtype == _abi.KV_FP8_E4M3 else 0
    p.block_table = _ptr(block_table)
    p.max_blocks_per_seq = 0 if block_table is None else int(block_table.shape[1])
    p.block_size, p.num_blocks, p.max_seqlen_kv = block_size, num_blocks, max_seqlen_kv
    p.cu_seqlens_q, p.seqused_kv = _ptr(cu_seqlens_q), _ptr(seqused_kv)
    p.scale = 1.0 / math.sqrt(head_dim) if scale is None else scale
    p.mask_mode, p.pre_tokens, p.next_tokens = mask_mode, pre_tokens, next_tokens
    p.sinks = _ptr(sinks)
    p.num_sms = num_sms
    p.kv_layout = kv_layout
    if atten_mask is not None:
        _contig(atten_mask, "atten_mask")
        if atten_mask.dim() != 3 or atten_mask.element_size() != 1:
            raise ValueError("atten_mask must be a 3-d tensor of 1-byte elements")
        p.atten_mask = _ptr(atten_mask)
        p.mask_row_stride = int(atten_mask.stride(1))
        p.mask_batch_stride = 0 if atten_mask.shape[0] == 1 else int(atten_mask.stride(0))
    return p


def params_from_problem(prob, out: torch.Tensor, lse: Optional[torch.Tensor],
                        num_sms: int = 0) -> FiaParams:
    """Parameters for a problem object with the generator's field names
    (B, QN, KVN, D, layout, S_q, T, q, k_cache, ...)."""
    return make_fia_params(
        q=prob.q, out=out, k_cache=prob.k_cache, v_cache=prob.v_cache, num_q_heads=prob.QN,
        num_kv_heads=prob.KVN, head_dim=prob.D, batch=prob.B, layout=prob.layout,
        max_seqlen_q=prob.S_q, total_q=prob.T, lse=lse, kv_dtype=prob.kv_dtype,
        k_scale=prob.k_scale, v_scale=prob.v_scale, block_table=prob.block_table,
        block_size=prob.block_size, num_blocks=prob.num_blocks,
        max_seqlen_kv=0 if prob.block_table is not None else prob.S_kv,
        cu_seqlens_q=prob.cu_seqlens_q, seqused_kv=prob.seqused_kv, scale=prob.scale,
        mask_mode=prob.mask_mode, pre_tokens=prob.pre_tokens, next_tokens=prob.next_tokens,
        sinks=prob.sinks, num_sms=num_sms, kv_layout=getattr(prob, "kv_layout", 0),
        atten_mask=getattr(prob, "atten_mask", None))


def lse_shape(prob):
    return (prob.T, prob.QN, 1) if prob.layout == _abi.LAYOUT_TND else (prob.B, prob.QN, prob.S_q, 1)


class FiaCall:
    """One configured FIA call: owns its outputs and workspace (torch
    allocations) and launches plan/execute/run on a stream."""

    def __init__(self, prob, with_lse: bool = True, num_sms: int = 0, out=None, lse=None):
        dev = prob.q.device
        self.prob = prob
        self.out = torch.empty_like(prob.q) if out is None else out
        self.lse = (torch.empty(lse_shape(prob), dtype=torch.float32, device=dev)
                    if (with_lse and lse is None) else lse)
        self.params = params_from_problem(prob, self.out, self.lse, num_sms)
        self.ws_bytes = _abi.fia_get_workspace_size(self.params)
        self.ws = torch.empty(max(self.ws_bytes, 256), dtype=torch.uint8, device=dev)

    def plan(self, stream=None):
        _abi.fia_plan(self.params, self.ws.data_ptr(), self.ws_bytes, _stream(stream))

    def execute(self, stream=None):
        _abi.fia_execute(self.params, self.ws.data_ptr(), self.ws_bytes, _stream(stream))

    def run(self, stream=None):
        _abi.fia_run(self.params, self.ws.data_ptr(), self.ws_bytes, _stream(stream))
        return self.out, self.lse

    def plan_layout(self):
        return _abi.fia_get_plan_layout(self.params)

    def error_word(self) -> int:
        return int(self.ws[:4].view(torch.int32).item())


def fused_infer_attention(prob, with_lse: bool = True, num_sms: int = 0, stream=None):
    """Run FIA on a problem object; returns (out, lse)."""
    c = FiaCall(prob, with_lse=with_lse, num_sms=num_sms)
    return c.run(stream)


# ----------------------------------------------------------------------------
# sparse shared-KV attention
# ----------------------------------------------------------------------------

def sparse_params_from_problem(sp, out: torch.Tensor, lse: Optional[torch.Tensor],
                               num_sms: int = 0) -> SparseParams:
    p = SparseParams()
    p.batch, p.num_q_heads, p.head_dim, p.layout = sp.B, sp.N1, sp.D, sp.layout
    p.max_seqlen_q, p.total_q = sp.S1, sp.T1
    p.q, p.out, p.lse = _ptr(sp.q), _ptr(out), _ptr(lse)
    p.ori_kv, p.ori_block_table = _ptr(sp.ori_kv), _ptr(sp.ori_block_table)
    p.ori_max_blocks = int(sp.ori_block_table.shape[1])
    p.ori_block_size, p.ori_num_blocks = sp.ori_block_size, int(sp.ori_kv.shape[0])
    p.cmp_kv, p.cmp_block_table = _ptr(sp.cmp_kv), _ptr(sp.cmp_block_table)
    p.cmp_max_blocks = 0 if sp.cmp_block_table is None else int(sp.cmp_block_table.shape[1])
    p.cmp_block_size = sp.cmp_block_size if sp.cmp_kv is not None else 0
    p.cmp_num_blocks = 0 if sp.cmp_kv is None else int(sp.cmp_kv.shape[0])
    p.topk = sp.K2
    p.cmp_sparse_indices = _ptr(sp.cmp_sparse_indices)
    p.cu_seqlens_q, p.seqused_kv, p.sinks = _ptr(sp.cu_seqlens_q), _ptr(sp.seqused_kv), _ptr(
        sp.sinks)
    p.softmax_scale = sp.scale
    p.cmp_ratio = sp.cmp_ratio if sp.cmp_kv is not None else 1
    p.ori_win_left, p.ori_win_right = sp.win_left, sp.win_right
    p.num_sms = num_sms
    p.kv_dtype = getattr(sp, "kv_dtype", _abi.SPARSE_KV_BF16)
    if p.kv_dtype == _abi.SPARSE_KV_FP8_PACKED:
        p.tile_size, p.rope_head_dim = 64, 64
    return p


class SparseCall:
    """Metadata + main call of the shared-KV sparse attention."""

    def __init__(self, sp, with_lse: bool = True, num_sms: int = 0):
        dev = sp.q.device
        self.sp = sp
        self.out = torch.empty_like(sp.q)
        self.lse = (torch.empty((sp.rows, sp.N1), dtype=torch.float32, device=dev)
                    if with_lse else None)
        self.params = sparse_params_from_problem(sp, self.out, self.lse, num_sms)
        self.metadata = torch.zeros(1024, dtype=torch.int32, device=dev)
        self.ws = None
        self.ws_bytes = 0

    def plan(self, stream=None):
        n = _abi.sparse_attn_metadata(self.params, self.metadata.data_ptr(), _stream(stream))
        if self.ws is None or self.ws.numel() < n:
            self.ws = torch.empty(max(n, 256), dtype=torch.uint8, device=self.out.device)
        self.ws_bytes = n

    def run(self, stream=None):
        if self.ws is None:
            self.plan(stream)
        _abi.sparse_attn_run(self.params, self.metadata.data_ptr(), self.ws.data_ptr(),
                             self.ws_bytes, _stream(stream))
        return self.out, self.lse


# ----------------------------------------------------------------------------
# log-sum-exp combine of partial results (context parallelism over the keys)
# ----------------------------------------------------------------------------

def lse_combine(outs, lses, *, layout: int, num_heads: int, batch: int = 0, seqlen_q: int = 0,
                total_q: int = 0, out: Optional[torch.Tensor] = None,
                lse: Optional[torch.Tensor] = None, sinks: Optional[torch.Tensor] = None,
                stream=None):
    """Combine results of the same query rows against disjoint key sets with
    fia_lse_combine.  `outs` are bf16 tensors in the FIA out layout, `lses`
    the matching fp32 lse tensors, computed without sinks; `sinks` (fp32
    [num_heads]) enter here, once.  Returns (out, lse)."""
    import ctypes
    n = len(outs)
    if n != len(lses) or not 1 <= n <= _abi.COMBINE_MAX_PARTS:
        raise ValueError("one lse per part, 1..16 parts")
    for t in list(outs) + list(lses):
        _contig(t, "part")
    out = torch.empty_like(outs[0]) if out is None else out
    lse = torch.empty_like(lses[0]) if lse is None else lse
    c = _abi.CombineParams()
    c.n_parts, c.layout, c.batch, c.seqlen_q, c.total_q = n, layout, batch, seqlen_q, total_q
    c.num_heads, c.head_dim = num_heads, int(outs[0].shape[-1])
    o_arr = (ctypes.c_void_p * n)(*[_ptr(t) for t in outs])
    l_arr = (ctypes.c_void_p * n)(*[_ptr(t) for t in lses])
    c.o_parts = ctypes.cast(o_arr, ctypes.POINTER(ctypes.c_void_p))
    c.lse_parts = ctypes.cast(l_arr, ctypes.POINTER(ctypes.c_void_p))
    c.out, c.lse, c.sinks = _ptr(out), _ptr(lse), _ptr(sinks)
    _abi.fia_lse_combine(c, _stream(stream))
    return out, lse
