"""Context parallelism across ranks, world size 2 over gloo on the CPU: the
rank bookkeeping of decode_tile_scheduler_gb300.cp and the exchange of
partial results, with the fp64 oracle standing in for each rank's kernels.

* Query split ("sparse_flash_mla", CP example): each rank passes its
  contiguous range of the global TND query tokens with the KV prefix up to
  its last row, so the query start the kernels derive (kv_len - q_len) is
  the cut; the rows gathered from both ranks equal the whole call.
* KV split (the ring-attention use of softmax_lse): each rank computes every
  query row against its blocks of each sequence, the (out, lse) pairs are
  all-gathered and joined by the log-sum-exp combine; the result equals the
  whole call.
"""
import dataclasses
import os
import socket
import sys

import numpy as np
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _global_prefill():
    import fia_inputs as fi
    return fi.make_fia(B=3, QN=4, KVN=2, D=32, q_lens=[37, 5, 60], kv_lens=[50, 5, 200],
                       layout=fi.LAYOUT_TND, block_size=16, mask_mode=3, with_sinks=True,
                       seed=91)


def _global_decode():
    import fia_inputs as fi
    return fi.make_fia(B=3, QN=8, KVN=2, D=32, q_lens=[1, 1, 1], kv_lens=[300, 17, 70],
                       block_size=16, with_sinks=True, seed=92)


def _local_query_problem(p, sl):
    """The rank's call of a query split: its rows of q, its batches' block
    table rows and KV prefixes."""
    import fia_inputs as fi
    q = p.q[sl.token_begin:sl.token_end].contiguous()
    idx = torch.tensor(sl.batches, dtype=torch.long)
    return dataclasses.replace(
        p, B=len(sl.batches), T=sl.token_end - sl.token_begin, S_q=max(sl.q_lens), q=q,
        cu_seqlens_q=torch.tensor(sl.cu_seqlens_q, dtype=torch.int32),
        block_table=p.block_table[idx].contiguous(),
        seqused_kv=torch.tensor(sl.kv_lens, dtype=torch.int32), q_lens=sl.q_lens,
        kv_lens=sl.kv_lens, layout=fi.LAYOUT_TND)


def _worker(rank, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE="2", LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    dist.init_process_group("gloo", rank=rank, world_size=2)
    import oracle
    from decode_tile_scheduler_gb300 import cp
    res = {}
    # ---- query split ----
    p = _global_prefill()
    sl = cp.query_split(p.cu_seqlens_q.tolist(), p.kv_lens, 2, rank)
    # the first row each local batch computes sits where it sits in the whole call
    for b, ql, kl, r0 in zip(sl.batches, sl.q_lens, sl.kv_lens, sl.row_begin):
        assert kl - ql == p.kv_lens[b] - p.q_lens[b] + r0
    o, l = oracle.fia(_local_query_problem(p, sl))
    rows = torch.from_numpy(o)
    sizes = [torch.zeros(1, dtype=torch.int64) for _ in range(2)]
    dist.all_gather(sizes, torch.tensor([rows.shape[0]]))
    n = int(max(s.item() for s in sizes))
    pad = torch.zeros((n,) + tuple(rows.shape[1:]), dtype=torch.float64)
    pad[:rows.shape[0]] = rows
    got = [torch.empty_like(pad) for _ in range(2)]
    dist.all_gather(got, pad)
    gathered = torch.cat([g[:int(s.item())] for g, s in zip(got, sizes)])
    if rank == 0:
        whole, _ = oracle.fia(p)
        res["query_split"] = float(np.abs(gathered.numpy() - whole).max())
    # ---- KV split ----
    d = _global_decode()
    ks = cp.kv_split(d.block_table, d.kv_lens, d.block_size, 2, rank)
    part = dataclasses.replace(d, block_table=ks.block_table, kv_lens=ks.kv_lens,
                               seqused_kv=torch.tensor(ks.kv_lens, dtype=torch.int32),
                               sinks=None)
    o, l = oracle.fia(part)
    outs, lses = cp.gather_parts(torch.from_numpy(o), torch.from_numpy(l.reshape(d.B, d.QN)))
    if rank == 0:
        co, cl = oracle.lse_combine([x.numpy() for x in outs], [x.numpy() for x in lses],
                                    sinks=d.sinks.numpy(), head_axis=1)
        wo, wl = oracle.fia(d)
        res["kv_split"] = (float(np.abs(co - wo).max()),
                           float(np.abs(cl - wl.reshape(d.B, d.QN)).max()))
        res["kv_lens"] = [ks.kv_lens]
    q.put((rank, res))
    dist.destroy_process_group()


def test_two_rank_query_and_kv_splits_equal_the_whole_call():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = dict(q.get(timeout=300) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    res = out[0]
    assert res["query_split"] < 1e-12
    assert res["kv_split"][0] < 1e-12 and res["kv_split"][1] < 1e-12


def test_split_bookkeeping():
    sys.path.insert(0, ROOT)
    from decode_tile_scheduler_gb300 import cp
    # two sequences of 6 and 10 query rows, keys 8 and 30: 16 tokens, cut at 8
    s0 = cp.query_split([0, 6, 16], [8, 30], 2, 0)
    s1 = cp.query_split([0, 6, 16], [8, 30], 2, 1)
    assert (s0.token_begin, s0.token_end, s1.token_begin, s1.token_end) == (0, 8, 8, 16)
    assert s0.batches == [0, 1] and s0.q_lens == [6, 2] and s0.kv_lens == [8, 22]
    assert s1.batches == [1] and s1.q_lens == [8] and s1.kv_lens == [30] and s1.row_begin == [2]
    # rank 1's first row (row 2 of sequence 1) keeps its position 30 - 10 + 2
    assert s1.kv_lens[0] - s1.q_lens[0] == 22
    bt = torch.arange(20, dtype=torch.int32).reshape(2, 10)
    k0 = cp.kv_split(bt, [100, 16], 16, 2, 0)
    k1 = cp.kv_split(bt, [100, 16], 16, 2, 1)
    # 7 and 1 blocks: rank 0 takes 3 and 0, rank 1 takes 4 and 1
    assert k0.kv_lens == [48, 0] and k1.kv_lens == [52, 16]
    assert k0.block_table[0, :3].tolist() == [0, 1, 2]
    assert k1.block_table[0, :4].tolist() == [3, 4, 5, 6] and k1.block_table[1, 0] == 10
