"""GPU parity of fia_lse_combine and of context parallelism emulated in one
process, through the C ABI, against the fp64 oracle:

* KV split of the long FP8 decode workload at a rank boundary: each part
  through fia_run with its lse, joined by fia_lse_combine, equals the oracle
  on the whole sequence (every row);
* combine of 3 parts with BSND multi-row lse layout and TND, a sink on one
  part, parts and sequences without keys;
* query split ("sparse_flash_mla", CP example): two ranks' calls over their
  query ranges with prefix KV lengths; the rows equal the whole call -- bit
  for bit for the sparse kernel (batch invariant), within the tolerance of
  the oracle for the prefill kernel.
"""
import dataclasses

import numpy as np
import pytest
import torch

import fia_inputs as fi
import oracle
from helpers import check_close

pytestmark = pytest.mark.gpu
dev = "cuda"


def _kv_part(p, world, rank):
    from decode_tile_scheduler_gb300 import cp
    ks = cp.kv_split(p.block_table, p.kv_lens, p.block_size, world, rank)
    return dataclasses.replace(p, block_table=ks.block_table.to(dev), kv_lens=ks.kv_lens,
                               seqused_kv=torch.tensor(ks.kv_lens, dtype=torch.int32,
                                                       device=dev),
                               sinks=None)  # the combine adds the sinks


def _combine(p, parts):
    import decode_tile_scheduler_gb300 as fia
    outs, lses = [], []
    for part in parts:
        o, l = fia.FiaCall(part, with_lse=True).run()
        outs.append(o)
        lses.append(l)
    out, lse = fia.lse_combine(outs, lses, layout=p.layout, num_heads=p.QN, batch=p.B,
                               seqlen_q=p.S_q, total_q=p.T, sinks=p.sinks)
    torch.cuda.synchronize()
    return out, lse


def test_kv_split_of_the_long_fp8_decode_every_row():
    p = fi.workload_fp8_long_decode(device=dev)
    out, lse = _combine(p, [_kv_part(p, 2, r) for r in range(2)])
    ro, rl = oracle.fia(p.to("cpu"))
    check_close(out, lse, ro, rl, "two-rank FP8 decode")


@pytest.mark.parametrize("layout", [fi.LAYOUT_BSND, fi.LAYOUT_TND])
def test_three_part_combine_with_sinks_and_empty_parts(layout):
    # mode 0: every row sees every key, so the key parts are independent;
    # sequence 1 has keys in the last part only, sequence 3 none at all (the
    # sink then enters through the combine, not through an empty part)
    ql = [4, 4, 4, 4] if layout == fi.LAYOUT_BSND else [4, 1, 0, 3]
    p = fi.make_fia(B=4, QN=16, KVN=2, D=128, q_lens=ql, kv_lens=[2000, 60, 900, 0],
                    layout=layout, block_size=64, with_sinks=True, seed=61, device=dev)
    out, lse = _combine(p, [_kv_part(p, 3, r) for r in range(3)])
    ro, rl = oracle.fia(p.to("cpu"))
    check_close(out, lse, ro, rl, "three parts")


def test_combine_rejects_bad_arguments():
    import ctypes
    import decode_tile_scheduler_gb300 as fia
    from decode_tile_scheduler_gb300 import _abi
    o = torch.zeros((2, 4, 128), dtype=torch.bfloat16, device=dev)
    l = torch.zeros((2, 4), dtype=torch.float32, device=dev)
    c = _abi.CombineParams()
    c.n_parts, c.layout, c.total_q, c.num_heads, c.head_dim = 1, fi.LAYOUT_TND, 2, 4, 128
    arr_o = (ctypes.c_void_p * 1)(o.data_ptr())
    arr_l = (ctypes.c_void_p * 1)(l.data_ptr())
    c.o_parts = ctypes.cast(arr_o, ctypes.POINTER(ctypes.c_void_p))
    c.lse_parts = ctypes.cast(arr_l, ctypes.POINTER(ctypes.c_void_p))
    c.out = o.data_ptr()  # the output may not be one of the parts
    assert fia.lib().fia_lse_combine(ctypes.byref(c), None) == fia.FIA_ERR_BAD_SHAPE
    c.out = torch.empty_like(o).data_ptr()
    c.n_parts = 17
    assert fia.lib().fia_lse_combine(ctypes.byref(c), None) == fia.FIA_ERR_BAD_SHAPE
    c.n_parts, c.head_dim = 1, 100
    assert fia.lib().fia_lse_combine(ctypes.byref(c), None) == fia.FIA_ERR_BAD_SHAPE


def _query_part_fia(p, sl):
    idx = torch.tensor(sl.batches, dtype=torch.long, device=dev)
    return dataclasses.replace(
        p, B=len(sl.batches), T=sl.token_end - sl.token_begin, S_q=max(sl.q_lens),
        q=p.q[sl.token_begin:sl.token_end].contiguous(),
        cu_seqlens_q=torch.tensor(sl.cu_seqlens_q, dtype=torch.int32, device=dev),
        block_table=p.block_table[idx].contiguous(),
        seqused_kv=torch.tensor(sl.kv_lens, dtype=torch.int32, device=dev), q_lens=sl.q_lens,
        kv_lens=sl.kv_lens)


def test_query_split_prefill_matches_the_whole_call():
    import decode_tile_scheduler_gb300 as fia
    from decode_tile_scheduler_gb300 import cp
    p = fi.make_fia(B=2, QN=8, KVN=2, D=128, q_lens=[700, 300], kv_lens=[900, 300],
                    layout=fi.LAYOUT_TND, block_size=64, mask_mode=3, with_sinks=True, seed=63,
                    device=dev)
    rows_o, rows_l = [], []
    for r in range(2):
        sl = cp.query_split(p.cu_seqlens_q.tolist(), p.kv_lens, 2, r)
        o, l = fia.FiaCall(_query_part_fia(p, sl), with_lse=True).run()
        rows_o.append(o)
        rows_l.append(l)
    torch.cuda.synchronize()
    out, lse = torch.cat(rows_o), torch.cat(rows_l)
    ro, rl = oracle.fia(p.to("cpu"))
    check_close(out, lse, ro, rl, "query split prefill")


def test_query_split_sparse_is_bit_exact():
    """The pages' CP example: two ranks run one after the other, rank 1 only a
    part of the second sequence's rows with the KV prefix up to its end."""
    import decode_tile_scheduler_gb300 as fia
    from decode_tile_scheduler_gb300 import cp
    sp = fi.make_sparse(B=2, N1=64, D=512, q_lens=[5, 9], kv_lens=[3000, 4100],
                        layout=fi.LAYOUT_TND, mode="csa", K2=512, seed=65, device=dev)
    whole = fia.SparseCall(sp, with_lse=True)
    wo, wl = whole.run()
    rows_o, rows_l = [], []
    for r in range(2):
        sl = cp.query_split(sp.cu_seqlens_q.tolist(), sp.kv_lens, 2, r)
        idx = torch.tensor(sl.batches, dtype=torch.long, device=dev)
        part = dataclasses.replace(
            sp, B=len(sl.batches), T1=sl.token_end - sl.token_begin, S1=max(sl.q_lens),
            q=sp.q[sl.token_begin:sl.token_end].contiguous(),
            cu_seqlens_q=torch.tensor(sl.cu_seqlens_q, dtype=torch.int32, device=dev),
            ori_block_table=sp.ori_block_table[idx].contiguous(),
            cmp_block_table=sp.cmp_block_table[idx].contiguous(),
            cmp_sparse_indices=sp.cmp_sparse_indices[sl.token_begin:sl.token_end].contiguous(),
            seqused_kv=torch.tensor(sl.kv_lens, dtype=torch.int32, device=dev),
            q_lens=sl.q_lens, kv_lens=sl.kv_lens)
        o, l = fia.SparseCall(part, with_lse=True).run()
        rows_o.append(o.clone())
        rows_l.append(l.clone())
    torch.cuda.synchronize()
    assert torch.equal(torch.cat(rows_o), wo)
    assert torch.equal(torch.cat(rows_l), wl)
    ro, rl = oracle.sparse(sp.to("cpu"))
    check_close(wo, wl, ro, rl, "sparse CP")
