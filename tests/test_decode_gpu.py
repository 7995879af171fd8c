"""GPU parity of the decode branch (query length 1) against the fp64 oracle,
through the C ABI: bf16 and FP8 KV, GQA groups, block sizes, mask modes,
sinks, empty and ragged KV, forced split-KV (few CTAs / many CTAs), the paged
GQA decode workload at full size, bit-exact schedule metadata, determinism."""
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


def _ref(p):
    return oracle.fia(p.to("cpu"))


CASES = {
    "gqa4_bs128": dict(B=3, QN=8, KVN=2, D=128, kv_lens=[700, 1, 300], block_size=128),
    "gqa1_d64_bs16": dict(B=2, QN=4, KVN=4, D=64, kv_lens=[33, 200], block_size=16),
    "gqa8_bs48": dict(B=2, QN=16, KVN=2, D=128, kv_lens=[257, 129], block_size=48),
    "gqa32_two_groups": dict(B=2, QN=32, KVN=1, D=128, kv_lens=[300, 77], block_size=64),
    "gqa20_ragged_group": dict(B=1, QN=20, KVN=1, D=64, kv_lens=[150], block_size=32),
    "empty_kv": dict(B=3, QN=4, KVN=2, D=128, kv_lens=[0, 5, 0], block_size=16),
    "sinks": dict(B=2, QN=8, KVN=2, D=128, kv_lens=[513, 64], block_size=128, with_sinks=True),
    "band": dict(B=2, QN=8, KVN=2, D=128, kv_lens=[1000, 90], block_size=32, mask_mode=4,
                 pre_tokens=300, next_tokens=0),
    "band_neg_pre": dict(B=2, QN=4, KVN=2, D=64, kv_lens=[500, 3], block_size=16, mask_mode=4,
                         pre_tokens=-1, next_tokens=5),
    "causal": dict(B=2, QN=4, KVN=1, D=128, kv_lens=[129, 128], block_size=128, mask_mode=3),
    "contiguous": dict(B=2, QN=8, KVN=2, D=128, kv_lens=[200, 17], paged=False),
    "fp8": dict(B=3, QN=16, KVN=2, D=128, kv_lens=[1000, 31, 257], block_size=64,
                kv_dtype=fi.KV_FP8_E4M3),
    "fp8_sinks_band": dict(B=2, QN=8, KVN=1, D=128, kv_lens=[3000, 200], block_size=32,
                           kv_dtype=fi.KV_FP8_E4M3, with_sinks=True, mask_mode=4,
                           pre_tokens=1000, next_tokens=0),
    "fp8_contiguous": dict(B=2, QN=8, KVN=2, D=128, kv_lens=[100, 300], paged=False,
                           kv_dtype=fi.KV_FP8_E4M3),
    # FP8 with 16 query heads per KV head (two head groups per unit) and with 2
    "fp8_gqa16": dict(B=2, QN=32, KVN=2, D=128, kv_lens=[900, 130], block_size=128,
                      kv_dtype=fi.KV_FP8_E4M3, with_sinks=True),
    "fp8_gqa2": dict(B=3, QN=4, KVN=2, D=128, kv_lens=[700, 1, 64], block_size=32,
                     kv_dtype=fi.KV_FP8_E4M3),
    # pages of 96 and 272 rows: tiles straddle pages, and the page index of a
    # row is not a shift
    "fp8_bs96": dict(B=3, QN=16, KVN=2, D=128, kv_lens=[1500, 95, 97], block_size=96,
                     kv_dtype=fi.KV_FP8_E4M3),
    "gqa4_bs272": dict(B=2, QN=8, KVN=2, D=64, kv_lens=[2000, 273], block_size=272),
}


@pytest.mark.parametrize("name", sorted(CASES))
@pytest.mark.parametrize("num_sms", [0, 3])
def test_decode_matches_oracle(name, num_sms):
    kw = dict(q_lens=None, seed=zlib.crc32(name.encode()) % 1000, device=dev)
    kw.update(CASES[name])
    kw["q_lens"] = [1] * kw["B"]
    p = fi.make_fia(**kw)
    _, out, lse = _run(p, num_sms)
    ro, rl = _ref(p)
    check_close(out, lse, ro, rl, name)


def test_decode_tnd_layout_with_empty_query_rows():
    p = fi.make_fia(B=3, QN=8, KVN=2, D=128, q_lens=[1, 0, 1], kv_lens=[300, 50, 7],
                    layout=fi.LAYOUT_TND, block_size=32, seed=5, device=dev)
    _, out, lse = _run(p)
    ro, rl = _ref(p)
    check_close(out, lse, ro, rl, "tnd")


@pytest.mark.parametrize("num_sms", [1, 2, 7, 64, 152, 500])
def test_split_kv_combine_any_cta_count(num_sms):
    p = fi.make_fia(B=4, QN=16, KVN=4, D=128, q_lens=[1] * 4, kv_lens=[2000, 130, 1, 900],
                    block_size=64, with_sinks=True, seed=11, device=dev)
    _, out, lse = _run(p, num_sms)
    ro, rl = _ref(p)
    check_close(out, lse, ro, rl, f"ctas={num_sms}")


def test_schedule_metadata_bit_exact():
    import decode_tile_scheduler_gb300 as fia
    p = fi.make_fia(B=6, QN=32, KVN=2, D=128, q_lens=[1] * 6, kv_lens=[0, 5000, 1, 128, 129, 3001],
                    block_size=16, seed=3, device=dev)
    for n in (1, 5, 152, 333):
        c, _, _ = _run(p, n)
        lay = c.plan_layout()
        ws = c.ws.cpu()
        U = lay.num_units
        per_cta = (lay.max_chunks - 4 * U) // n  # bf16, one row: the bound n*W + 4*U
        nsched = 8 + 3 * (p.B + 1) + p.B
        sched = ws[lay.sched_off: lay.sched_off + 8 * nsched].view(torch.int64).numpy()
        rs, rq = oracle.decode_schedule(p.to("cpu"), n, per_cta)
        assert np.array_equal(sched, rs)
        N = int(sched[2])
        queue = ws[lay.queue_off: lay.queue_off + 16 * N].view(torch.int32).numpy().reshape(N, 4)
        assert np.array_equal(queue, rq)


def test_schedule_fp8_bit_exact():
    # an FP8 cache: the rest of a unit in chunks of C tiles, the bound n*W + 2*U
    import decode_tile_scheduler_gb300 as fia
    p = fi.make_fia(B=4, QN=32, KVN=4, D=128, q_lens=[1] * 4, kv_lens=[40000, 3, 9000, 129],
                    block_size=128, kv_dtype=fi.KV_FP8_E4M3, seed=31, device=dev)
    for n in (1, 7, 152):
        c, out, lse = _run(p, n)
        lay = c.plan_layout()
        ws = c.ws.cpu()
        per_cta = (lay.max_chunks - 2 * lay.num_units) // n
        nsched = 8 + 3 * (p.B + 1) + p.B
        sched = ws[lay.sched_off: lay.sched_off + 8 * nsched].view(torch.int64).numpy()
        rs, rq = oracle.decode_schedule(p.to("cpu"), n, per_cta)
        assert np.array_equal(sched, rs)
        N = int(sched[2])
        queue = ws[lay.queue_off: lay.queue_off + 16 * N].view(torch.int32).numpy().reshape(N, 4)
        assert np.array_equal(queue, rq)
    ro, rl = _ref(p)
    check_close(out, lse, ro, rl, "FP8 schedule")


def test_schedule_many_batches_bit_exact_and_parity():
    # more batches than the scheduler keeps in shared memory: the global path
    import decode_tile_scheduler_gb300 as fia
    g = np.random.default_rng(41)
    B = 2100
    kv = [int(x) for x in g.integers(0, 600, B)]
    p = fi.make_fia(B=B, QN=8, KVN=2, D=128, q_lens=[1] * B, kv_lens=kv, block_size=64,
                    seed=43, device=dev)
    c, out, lse = _run(p, 152)
    lay = c.plan_layout()
    ws = c.ws.cpu()
    per_cta = (lay.max_chunks - 4 * lay.num_units) // 152
    nsched = 8 + 3 * (B + 1) + B
    sched = ws[lay.sched_off: lay.sched_off + 8 * nsched].view(torch.int64).numpy()
    rs, rq = oracle.decode_schedule(p.to("cpu"), 152, per_cta)
    assert np.array_equal(sched, rs)
    N = int(sched[2])
    queue = ws[lay.queue_off: lay.queue_off + 16 * N].view(torch.int32).numpy().reshape(N, 4)
    assert np.array_equal(queue, rq)
    ro, rl = _ref(p)
    check_close(out, lse, ro, rl, "2100 batches")


@pytest.mark.parametrize("B", [33, 64, 65, 300])
def test_schedule_batch_counts_bit_exact(B):
    # batch counts across warp boundaries of the scheduler's block-wide scans
    # and well inside its shared-memory path: the plan is the oracle's
    g = np.random.default_rng(100 + B)
    kv = [int(x) for x in g.integers(0, 3000, B)]
    p = fi.make_fia(B=B, QN=16, KVN=2, D=128, q_lens=[1] * B, kv_lens=kv, block_size=64,
                    seed=7 + B, device=dev)
    c, out, lse = _run(p, 152)
    lay = c.plan_layout()
    ws = c.ws.cpu()
    per_cta = (lay.max_chunks - 4 * lay.num_units) // 152
    nsched = 8 + 3 * (B + 1) + B
    sched = ws[lay.sched_off: lay.sched_off + 8 * nsched].view(torch.int64).numpy()
    rs, rq = oracle.decode_schedule(p.to("cpu"), 152, per_cta)
    assert np.array_equal(sched, rs)
    N = int(sched[2])
    queue = ws[lay.queue_off: lay.queue_off + 16 * N].view(torch.int32).numpy().reshape(N, 4)
    assert np.array_equal(queue, rq)
    if B == 65:
        ro, rl = _ref(p)
        check_close(out, lse, ro, rl, "65 batches")


def test_execute_reuses_one_plan():
    # fia_plan once, fia_execute three times: the claim queue and the split
    # counters re-arm themselves, so every execute gives the same result
    import decode_tile_scheduler_gb300 as fia
    p = fi.make_fia(B=5, QN=32, KVN=8, D=128, q_lens=[1] * 5, kv_lens=[4000, 700, 1, 129, 2500],
                    block_size=128, with_sinks=True, seed=19, device=dev)
    c = fia.FiaCall(p, with_lse=True)
    c.plan()
    outs = []
    for _ in range(3):
        c.out.fill_(float("nan"))
        c.execute()
        torch.cuda.synchronize()
        assert c.error_word() == 0
        outs.append((c.out.clone(), c.lse.clone()))
    for o, l in outs[1:]:
        assert torch.equal(o, outs[0][0]) and torch.equal(l, outs[0][1])
    ro, rl = _ref(p)
    check_close(outs[0][0], outs[0][1], ro, rl, "plan reuse")


def test_decode_and_prefill_share_a_workspace():
    """One workspace for a decode and a prefill problem: each branch's plan
    leaves the other's execute without a plan (the prefill mark in the
    workspace header, which a decode plan clears), so fia_execute of the
    branch whose plan was replaced runs nothing (error word 2), and fia_run
    of either is right."""
    import decode_tile_scheduler_gb300 as fia
    pd = fi.make_fia(B=3, QN=16, KVN=2, D=128, q_lens=[1] * 3, kv_lens=[900, 2, 3000],
                     block_size=64, seed=29, device=dev)
    pp = fi.make_fia(B=2, QN=8, KVN=2, D=128, q_lens=[300, 64], kv_lens=[300, 64],
                     layout=fi.LAYOUT_TND, block_size=64, mask_mode=3, seed=37, device=dev)
    cd = fia.FiaCall(pd, with_lse=True)
    cp = fia.FiaCall(pp, with_lse=True)
    ws = torch.empty(max(cd.ws_bytes, cp.ws_bytes), dtype=torch.uint8, device=dev)
    cd.ws = ws
    cp.ws = ws
    rdo, rdl = _ref(pd)
    rpo, rpl = _ref(pp)
    for _ in range(2):
        cp.run()
        torch.cuda.synchronize()
        assert cp.error_word() == 0
        check_close(cp.out, cp.lse, rpo, rpl, "prefill")
        cd.out.fill_(7.0)
        cd.execute()  # the decode plan was replaced by the prefill plan
        torch.cuda.synchronize()
        assert cd.error_word() == 2
        assert bool(torch.all(cd.out == 7.0))
        cd.run()
        torch.cuda.synchronize()
        assert cd.error_word() == 0
        check_close(cd.out, cd.lse, rdo, rdl, "decode")
        cp.out.fill_(7.0)
        cp.execute()  # the prefill plan was replaced by the decode plan
        torch.cuda.synchronize()
        assert cp.error_word() == 2
        assert bool(torch.all(cp.out == 7.0))


def test_plan_with_slot_prefixes_outside_the_partials():
    """A plan whose mark matches but whose partial-slot prefix Q points past
    the partial slots: the split chunks' writes stay inside the slots, the
    combine rejects every such batch, and the error word says 2.  A fresh
    plan makes the workspace usable again."""
    import decode_tile_scheduler_gb300 as fia
    p = fi.make_fia(B=3, QN=16, KVN=2, D=128, q_lens=[1] * 3, kv_lens=[3000, 5, 2000],
                    block_size=64, seed=41, device=dev)
    c = fia.FiaCall(p, with_lse=True, num_sms=4)  # few CTAs: every long unit is split
    c.plan()
    lay = c.plan_layout()
    q = c.ws[lay.sched_off + 64: lay.sched_off + 64 + 8 * (p.B + 1)].view(torch.int64)
    q.copy_(torch.arange(p.B + 1, device=dev, dtype=torch.int64) + (1 << 40))
    c.execute()
    torch.cuda.synchronize()
    assert c.error_word() == 2
    c.run()
    torch.cuda.synchronize()
    assert c.error_word() == 0
    ro, rl = _ref(p)
    check_close(c.out, c.lse, ro, rl, "after a fresh plan")


def test_execute_waits_for_its_plan_when_queued_behind_busy_work():
    """The decode kernel is launched behind the scheduler with programmatic
    serialization and may start while the plan is being written.  Queued
    behind a busy stream over a poisoned workspace, it still reads only the
    finished plan: error word 0 and the oracle's outputs, every time."""
    import decode_tile_scheduler_gb300 as fia
    p = fi.make_fia(B=5, QN=32, KVN=8, D=128, q_lens=[1] * 5, kv_lens=[4000, 700, 1, 129, 2500],
                    block_size=128, with_sinks=True, seed=47, device=dev)
    ro, rl = _ref(p)
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


def test_deterministic_bitwise():
    p = fi.make_fia(B=5, QN=32, KVN=8, D=128, q_lens=[1] * 5, kv_lens=[4000, 700, 1, 129, 2500],
                    block_size=128, seed=9, device=dev)
    _, o1, l1 = _run(p)
    o1, l1 = o1.clone(), l1.clone()
    _, o2, l2 = _run(p)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_poisoned_unused_pages_never_reach_the_output():
    # every row past kv_len in the pool is NaN (generator poison); also the
    # table slots past each sequence's last block point at a NaN block
    p = fi.make_fia(B=4, QN=8, KVN=2, D=128, q_lens=[1] * 4, kv_lens=[17, 129, 255, 1],
                    block_size=16, seed=13, device=dev)
    _, out, lse = _run(p)
    assert torch.isfinite(out.float()).all() and torch.isfinite(lse).all()


def test_paged_gqa_decode_workload_full_size():
    p = fi.workload_paged_decode(device=dev)
    _, out, lse = _run(p)
    ro, rl = _ref(p)
    check_close(out, lse, ro, rl, "paged GQA decode")


def test_fp8_long_decode_workload_every_row():
    # all B x Q_N = 256 (batch, head) rows of the long FP8 decode workload
    p = fi.workload_fp8_long_decode(device=dev)
    _, out, lse = _run(p)
    ro, rl = oracle.fia(p.to("cpu"))
    check_close(out, lse, ro, rl, "long FP8 decode, every row")


# The other decode workloads the bench times, at their bench sizes, every
# (query row, head) against the oracle: the same sequences with 4 query rows
# each (multi-token decode), with head-major pages, and the long FP8 decode
# with 16 query heads per KV head.
BENCH_FORMS = {
    "mtp_decode_s4": lambda: fi.workload_paged_decode(device=dev, S_q=4),
    "paged_decode_bnnbsd": lambda: fi.workload_paged_decode(device=dev,
                                                            kv_layout=fi.KV_LAYOUT_BNNBSD),
    "fp8_gqa16_decode": lambda: fi.workload_fp8_long_decode(device=dev, KVN=4),
}


@pytest.mark.parametrize("name", sorted(BENCH_FORMS))
def test_bench_decode_forms_every_row(name):
    p = BENCH_FORMS[name]()
    _, out, lse = _run(p)
    ro, rl = _ref(p)
    check_close(out, lse, ro, rl, name)


# Query magnitudes across the whole bf16 range.  The FP8 products run in fp16,
# so the kernel moves each head's query by a power of two before narrowing it;
# the bf16 products see the query unchanged.  Powers of two keep the inputs
# exact, and the scale brings the scores back to a moderate size.
Q_RANGE = {
    # |q| up to ~2^19, beyond fp16's largest finite value (65504)
    "large": dict(q_mult=2.0 ** 17, scale=2.0 ** -17 / 11.3),
    # |q| around 2^-20: fp16 subnormals would keep only a few bits
    "tiny": dict(q_mult=2.0 ** -20, scale=2.0 ** 20 / 11.3),
    # heads of one unit 2^6 apart: each head takes its own shift, so a head
    # scaled with its neighbour's shift would be off by 64
    "mixed_heads": dict(q_mult=[2.0 ** 3 if h % 2 else 2.0 ** -3 for h in range(16)],
                        scale=1.0 / 11.3),
}


@pytest.mark.parametrize("kv_dtype", [fi.KV_BF16, fi.KV_FP8_E4M3])
@pytest.mark.parametrize("name", sorted(Q_RANGE))
def test_decode_query_range(name, kv_dtype):
    p = fi.make_fia(B=3, QN=16, KVN=2, D=128, q_lens=[1] * 3, kv_lens=[900, 40, 257],
                    block_size=64, kv_dtype=kv_dtype, with_sinks=True,
                    seed=zlib.crc32(name.encode()) % 1000, device=dev, **Q_RANGE[name])
    _, out, lse = _run(p)
    ro, rl = _ref(p)
    check_close(out, lse, ro, rl, f"{name} {kv_dtype}")


def test_fp8_decode_query_range_gqa16():
    # 16 query heads per KV head: two head groups per unit on the FP8 path
    p = fi.make_fia(B=2, QN=32, KVN=2, D=128, q_lens=[1, 1], kv_lens=[700, 129],
                    block_size=128, kv_dtype=fi.KV_FP8_E4M3, seed=77, device=dev,
                    q_mult=[2.0 ** 17 if h % 3 else 2.0 ** 15 for h in range(32)],
                    scale=2.0 ** -17 / 11.3)
    _, out, lse = _run(p)
    ro, rl = _ref(p)
    check_close(out, lse, ro, rl, "fp8 gqa16 large q")


@pytest.mark.parametrize("fp8", [False, True])
def test_execute_without_a_plan_runs_nothing(fp8):
    """fia_execute on a workspace that holds no plan of these arguments (never
    planned, or overwritten) finds no plan mark: nothing is loaded or written,
    and the error word reports 2."""
    import decode_tile_scheduler_gb300 as fia
    kw = dict(kv_dtype=fi.KV_FP8_E4M3) if fp8 else {}
    p = fi.make_fia(B=3, QN=16, KVN=2, D=128, q_lens=[1] * 3, kv_lens=[700, 5, 2000],
                    block_size=64, seed=31, device=dev, **kw)
    c = fia.FiaCall(p)
    for fill in (0x00, 0x5A):
        c.ws.fill_(fill)
        c.out.fill_(7.0)
        c.execute()
        torch.cuda.synchronize()
        assert c.error_word() == 2
        assert bool(torch.all(c.out == 7.0))
    # a plan makes the same workspace usable again
    c.run()
    torch.cuda.synchronize()
    assert c.error_word() == 0
    ro, rl = oracle.fia(p.to("cpu"))
    check_close(c.out, c.lse, ro, rl, "after a fresh plan")


def test_bounded_wait_times_out_and_the_context_stays_usable():
    """Failure detection without a GPU fault: the bounded wait that every
    pipeline barrier uses gives up on a barrier that nothing completes, sets
    the error word to 1 and returns; the next launches run normally."""
    import decode_tile_scheduler_gb300 as fia
    from decode_tile_scheduler_gb300 import _abi
    status = torch.full((3,), -1, dtype=torch.int32, device=dev)
    _abi.selftest_bounded_wait(status.data_ptr(), 20_000_000, torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    err, waited_us, completed = status.tolist()
    assert err == 1 and completed == 0
    assert 20_000 <= waited_us < 1_000_000          # the 20 ms limit, not longer than a second
    p = fi.make_fia(B=2, QN=8, KVN=2, D=128, q_lens=[1, 1], kv_lens=[300, 77], block_size=64,
                    seed=41, device=dev)
    c = fia.FiaCall(p)
    c.run()
    torch.cuda.synchronize()
    assert c.error_word() == 0
    ro, rl = oracle.fia(p.to("cpu"))
    check_close(c.out, c.lse, ro, rl, "after a timed-out wait")
