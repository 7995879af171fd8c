"""GPU parity of the prefill branch (query length > 1, tcgen05/TMEM kernel)
against the fp64 oracle through the C ABI: right-down causal, band and no
mask; TND and BSND; paged (block sizes 16..128) and contiguous KV; GQA ratios
1..8; sinks; ragged query tiles; query longer than KV (fully masked rows);
the tiny prefill and the varlen causal prefill workloads; the schedule's unit
order; determinism."""
import zlib

import numpy as np
import pytest
import torch

import fia_inputs as fi
import oracle
from helpers import check_close

pytestmark = pytest.mark.gpu
dev = "cuda"


def _run(p, num_sms=0):
    import decode_tile_scheduler_gb300 as fia
    c = fia.FiaCall(p, with_lse=True, num_sms=num_sms)
    out, lse = c.run()
    torch.cuda.synchronize()
    assert c.error_word() == 0
    return c, out, lse


def test_tiny_prefill_workload():
    p = fi.workload_tiny_prefill(device=dev)
    _, out, lse = _run(p)
    ro, rl = oracle.fia(p.to("cpu"))
    check_close(out, lse, ro, rl, "tiny prefill")


CASES = {
    "tnd_causal_gqa4": dict(B=3, QN=8, KVN=2, D=128, q_lens=[300, 1, 129], kv_lens=None,
                            layout=fi.LAYOUT_TND, block_size=128, mask_mode=3),
    "tnd_causal_sinks_bs16": dict(B=2, QN=4, KVN=2, D=128, q_lens=[200, 77], kv_lens=None,
                                  layout=fi.LAYOUT_TND, block_size=16, mask_mode=3,
                                  with_sinks=True),
    "bsnd_no_mask_kv_longer": dict(B=2, QN=4, KVN=1, D=128, q_lens=[100, 100],
                                   kv_lens=[700, 230], block_size=64, mask_mode=0),
    "band": dict(B=2, QN=8, KVN=4, D=128, q_lens=[257, 257], kv_lens=[400, 257],
                 block_size=32, mask_mode=4, pre_tokens=100, next_tokens=5),
    "band_neg_pre": dict(B=1, QN=4, KVN=4, D=64, q_lens=[150], kv_lens=[150], block_size=16,
                         mask_mode=4, pre_tokens=-3, next_tokens=40),
    "q_longer_than_kv": dict(B=2, QN=4, KVN=2, D=128, q_lens=[200, 130], kv_lens=[70, 0],
                             layout=fi.LAYOUT_TND, block_size=32, mask_mode=3, with_sinks=True),
    "gqa1_d64": dict(B=2, QN=3, KVN=3, D=64, q_lens=[129, 129], kv_lens=[129, 300],
                     block_size=128, mask_mode=3),
    "gqa8_bs48": dict(B=1, QN=16, KVN=2, D=128, q_lens=[333], kv_lens=[500], block_size=48,
                      mask_mode=3),
    "contiguous_bsnd": dict(B=2, QN=8, KVN=2, D=128, q_lens=[64, 64], kv_lens=[64, 200],
                            paged=False, mask_mode=3),
    "bsnd_sq2": dict(B=4, QN=8, KVN=2, D=128, q_lens=[2] * 4, kv_lens=[2, 513, 40, 1],
                     block_size=16, mask_mode=3),
}


@pytest.mark.parametrize("name", sorted(CASES))
def test_prefill_matches_oracle(name):
    kw = dict(seed=zlib.crc32(name.encode()) % 1000, device=dev)
    kw.update(CASES[name])
    if kw["kv_lens"] is None:
        kw["kv_lens"] = kw["q_lens"]
    p = fi.make_fia(**kw)
    _, out, lse = _run(p)
    ro, rl = oracle.fia(p.to("cpu"))
    check_close(out, lse, ro, rl, name)


@pytest.mark.parametrize("num_sms", [1, 7, 152])
def test_prefill_any_cta_count(num_sms):
    p = fi.make_fia(B=3, QN=8, KVN=2, D=128, q_lens=[400, 50, 260], kv_lens=[400, 50, 260],
                    layout=fi.LAYOUT_TND, block_size=64, mask_mode=3, with_sinks=True, seed=17,
                    device=dev)
    _, out, lse = _run(p, num_sms)
    ro, rl = oracle.fia(p.to("cpu"))
    check_close(out, lse, ro, rl, f"ctas={num_sms}")


def test_prefill_unit_order_is_a_cost_sorted_permutation():
    import decode_tile_scheduler_gb300 as fia
    p = fi.make_fia(B=4, QN=8, KVN=2, D=128, q_lens=[700, 1, 129, 300], kv_lens=[700, 1, 129, 300],
                    layout=fi.LAYOUT_TND, block_size=16, mask_mode=3, seed=23, device=dev)
    c, _, _ = _run(p)
    lay = c.plan_layout()
    ws = c.ws.cpu()
    n = int(ws[8:16].view(torch.int64).item())
    lst = ws[lay.unit_list_off: lay.unit_list_off + 8 * n].view(torch.int32).numpy().reshape(n, 2)
    units, cost = oracle.prefill_units(p.to("cpu"))
    assert n == units.shape[0]
    got = [(int(b), int(y) & 0x3FFFF, (int(y) >> 18) & 0xFF, (int(y) >> 26) & 0x3F)
           for b, y in lst]
    ref = {tuple(u): int(cst) for u, cst in zip(units.tolist(), cost.tolist())}
    assert sorted(got) == sorted(ref)
    costs = [ref[g] for g in got]
    assert all(x >= y for x, y in zip(costs, costs[1:]))


def test_prefill_deterministic_bitwise():
    p = fi.make_fia(B=2, QN=8, KVN=2, D=128, q_lens=[500, 260], kv_lens=[500, 260],
                    layout=fi.LAYOUT_TND, block_size=128, mask_mode=3, seed=29, device=dev)
    _, o1, l1 = _run(p)
    o1, l1 = o1.clone(), l1.clone()
    _, o2, l2 = _run(p, num_sms=77)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_varlen_causal_prefill_workload_sampled():
    # every 8th query row with all 32 heads, plus the first and the last row
    # of every sequence (its shortest and longest rows), element by element
    p = fi.workload_varlen_prefill(device=dev)
    _, out, lse = _run(p)
    pc = p.to("cpu")
    cu = pc.cu_seqlens_q.tolist()
    sel = sorted(set(range(0, p.T, 8)) | set(cu[:-1]) | set(c - 1 for c in cu[1:]))
    rows = np.repeat(np.array(sel, dtype=np.int64), p.QN)
    heads = np.tile(np.arange(p.QN, dtype=np.int32), len(sel))
    ro, rl = oracle.fia_sample(pc, rows, heads)
    o = out.float().cpu().numpy().reshape(p.T, p.QN, p.D)
    l = lse.cpu().numpy().reshape(p.T, p.QN)
    err = np.abs(o[rows, heads] - ro)
    assert err.max() <= 2e-2 and err.mean() <= 2e-3, (err.max(), err.mean())
    assert np.abs(l[rows, heads] - rl).max() <= 1e-3


@pytest.mark.parametrize("q_mult,scale", [(2.0 ** 17, 2.0 ** -17 / 11.3),
                                          (2.0 ** -20, 2.0 ** 20 / 11.3)])
def test_prefill_query_range(q_mult, scale):
    p = fi.make_fia(B=2, QN=8, KVN=2, D=128, q_lens=[200, 77], kv_lens=[200, 77],
                    layout=fi.LAYOUT_TND, block_size=64, mask_mode=3, with_sinks=True,
                    seed=83, device=dev, q_mult=q_mult, scale=scale)
    _, out, lse = _run(p)
    ro, rl = oracle.fia(p.to("cpu"))
    check_close(out, lse, ro, rl, f"q x {q_mult}")


def test_execute_reuses_one_plan():
    # fia_plan once, fia_execute twice: the claim counter re-arms itself
    import decode_tile_scheduler_gb300 as fia
    p = fi.make_fia(B=2, QN=8, KVN=2, D=128, q_lens=[300, 129], kv_lens=[300, 129],
                    layout=fi.LAYOUT_TND, block_size=64, mask_mode=3, with_sinks=True, seed=31,
                    device=dev)
    c = fia.FiaCall(p, with_lse=True)
    c.plan()
    outs = []
    for _ in range(2):
        c.out.fill_(float("nan"))
        c.execute()
        torch.cuda.synchronize()
        assert c.error_word() == 0
        outs.append((c.out.clone(), c.lse.clone()))
    assert torch.equal(outs[0][0], outs[1][0]) and torch.equal(outs[0][1], outs[1][1])
    ro, rl = oracle.fia(p.to("cpu"))
    check_close(outs[1][0], outs[1][1], ro, rl, "plan reuse")


def test_execute_without_a_plan_runs_nothing():
    """The prefill kernel, too, runs nothing without its plan's mark."""
    import decode_tile_scheduler_gb300 as fia
    p = fi.make_fia(B=2, QN=8, KVN=2, D=128, q_lens=[300, 77], kv_lens=[300, 77],
                    layout=fi.LAYOUT_TND, block_size=64, mask_mode=3, seed=33, device=dev)
    c = fia.FiaCall(p)
    for fill in (0x00, 0x5A):
        c.ws.fill_(fill)
        c.out.fill_(7.0)
        c.execute()
        torch.cuda.synchronize()
        assert c.error_word() == 2
        assert bool(torch.all(c.out == 7.0))
    c.run()
    torch.cuda.synchronize()
    assert c.error_word() == 0


def test_unit_list_entries_outside_the_arguments_run_nothing():
    """A plan whose mark matches but whose unit entries name no unit of these
    arguments (batch, KV head or head pair out of range) runs every such
    entry as an empty unit: nothing is loaded or written, and the error word
    says 2.  A fresh plan makes the workspace usable again."""
    import decode_tile_scheduler_gb300 as fia
    p = fi.make_fia(B=2, QN=8, KVN=2, D=128, q_lens=[300, 77], kv_lens=[300, 77],
                    layout=fi.LAYOUT_TND, block_size=64, mask_mode=3, seed=35, device=dev)
    c = fia.FiaCall(p)
    c.plan()
    lay = c.plan_layout()
    n = int(c.ws[8:16].view(torch.int64).item())  # units of the plan
    assert n > 0
    c.ws[lay.unit_list_off: lay.unit_list_off + 8 * n].fill_(0x7F)  # batch 0x7F7F7F7F
    c.out.fill_(7.0)
    c.execute()
    torch.cuda.synchronize()
    assert c.error_word() == 2
    assert bool(torch.all(c.out == 7.0))
    c.run()
    torch.cuda.synchronize()
    assert c.error_word() == 0
    ro, rl = oracle.fia(p.to("cpu"))
    check_close(c.out, c.lse, ro, rl, "after a fresh plan")


def test_execute_waits_for_its_plan_when_queued_behind_busy_work():
    """The prefill kernel is launched behind its scheduler with programmatic
    serialization and may start while the unit list is being written.
    Queued behind a busy stream over a poisoned workspace, it still reads
    only the finished plan: error word 0 and the oracle's outputs."""
    import decode_tile_scheduler_gb300 as fia
    p = fi.make_fia(B=3, QN=8, KVN=2, D=128, q_lens=[400, 50, 260], kv_lens=[400, 50, 260],
                    layout=fi.LAYOUT_TND, block_size=64, mask_mode=3, with_sinks=True, seed=49,
                    device=dev)
    ro, rl = oracle.fia(p.to("cpu"))
    c = fia.FiaCall(p, with_lse=True)
    for _ in range(3):
        c.ws.fill_(0x5A)
        c.out.fill_(float("nan"))
        torch.cuda._sleep(2_000_000)
        c.plan()
        c.execute()
        torch.cuda.synchronize()
        assert c.error_word() == 0
        check_close(c.out, c.lse, ro, rl, "queued behind busy work")
