"""GPU parity of the decode kernel beyond one query row and one mask shape,
through the C ABI, against the fp64 oracle:

* multi-token decode: 2..16 query rows per sequence (the (row, head) pairs of
  a KV head packed as mma columns), bf16 and FP8, GQA 1..8, BSND and ragged
  TND, causal and band masks, forced split-KV;
* mask mode 2 (causal from the top-left corner) and the explicit attention
  mask of modes 0/1 (per batch or shared, fully hidden rows);
* head-major (BnNBsD) pages, bf16 and FP8;
* the decode schedule of multi-row units bit-exact against its twin.
"""
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
    assert c.plan_layout().branch == 1  # the decode kernel
    out, lse = c.run()
    torch.cuda.synchronize()
    assert c.error_word() == 0
    return c, out, lse


def _seed(name):
    return zlib.crc32(name.encode()) % 1000


MTP = {
    # (S_q, G, dtype)
    "s2_g4_bf16": dict(S=2, QN=16, KVN=4, kv_dtype=fi.KV_BF16),
    "s4_g4_bf16": dict(S=4, QN=16, KVN=4, kv_dtype=fi.KV_BF16),
    "s16_g4_bf16": dict(S=16, QN=8, KVN=2, kv_dtype=fi.KV_BF16),
    "s4_g8_bf16": dict(S=4, QN=16, KVN=2, kv_dtype=fi.KV_BF16),
    "s16_g8_bf16": dict(S=16, QN=16, KVN=2, kv_dtype=fi.KV_BF16),
    "s3_g1_bf16": dict(S=3, QN=4, KVN=4, kv_dtype=fi.KV_BF16),
    "s2_g4_fp8": dict(S=2, QN=16, KVN=4, kv_dtype=fi.KV_FP8_E4M3),
    "s4_g4_fp8": dict(S=4, QN=16, KVN=4, kv_dtype=fi.KV_FP8_E4M3),
    "s16_g4_fp8": dict(S=16, QN=8, KVN=2, kv_dtype=fi.KV_FP8_E4M3),
    "s4_g8_fp8": dict(S=4, QN=16, KVN=2, kv_dtype=fi.KV_FP8_E4M3),
    "s16_g8_fp8": dict(S=16, QN=16, KVN=2, kv_dtype=fi.KV_FP8_E4M3),
}


@pytest.mark.parametrize("num_sms", [0, 5])
@pytest.mark.parametrize("name", sorted(MTP))
def test_multi_token_decode(name, num_sms):
    c = MTP[name]
    S = c["S"]
    kv = [S + 700, S, 2 * S + 129, 3000]  # every sequence holds its query rows
    p = fi.make_fia(B=4, QN=c["QN"], KVN=c["KVN"], D=128, q_lens=[S] * 4, kv_lens=kv,
                    block_size=64, kv_dtype=c["kv_dtype"], mask_mode=3, with_sinks=True,
                    seed=_seed(name), device=dev)
    _, out, lse = _run(p, num_sms)
    ro, rl = oracle.fia(p.to("cpu"))
    check_close(out, lse, ro, rl, name)


@pytest.mark.parametrize("kv_dtype", [fi.KV_BF16, fi.KV_FP8_E4M3])
def test_multi_token_decode_ragged_tnd(kv_dtype):
    # TND rows per sequence from 0 to 16 (max_seqlen_q 16), one sequence with
    # fewer keys than query rows (rows past the keys see nothing)
    ql = [3, 0, 16, 1, 7, 2]
    kv = [900, 40, 2000, 1, 130, 1]
    p = fi.make_fia(B=6, QN=16, KVN=2, D=128, q_lens=ql, kv_lens=kv, layout=fi.LAYOUT_TND,
                    block_size=32, kv_dtype=kv_dtype, mask_mode=3, with_sinks=True, seed=31,
                    device=dev)
    _, out, lse = _run(p)
    ro, rl = oracle.fia(p.to("cpu"))
    check_close(out, lse, ro, rl, "ragged tnd")


@pytest.mark.parametrize("mask", [dict(mask_mode=4, pre_tokens=300, next_tokens=0),
                                  dict(mask_mode=4, pre_tokens=-2, next_tokens=6),
                                  dict(mask_mode=0)])
def test_multi_token_decode_masks(mask):
    p = fi.make_fia(B=3, QN=8, KVN=2, D=64, q_lens=[5] * 3, kv_lens=[1000, 8, 260],
                    block_size=16, seed=41, device=dev, **mask)
    _, out, lse = _run(p, num_sms=7)
    ro, rl = oracle.fia(p.to("cpu"))
    check_close(out, lse, ro, rl, str(mask))


@pytest.mark.parametrize("S", [1, 4])
@pytest.mark.parametrize("kv_dtype", [fi.KV_BF16, fi.KV_FP8_E4M3])
def test_left_up_causal(S, kv_dtype):
    p = fi.make_fia(B=3, QN=16, KVN=2, D=128, q_lens=[S] * 3, kv_lens=[700, 3, 129],
                    block_size=64, kv_dtype=kv_dtype, mask_mode=2, with_sinks=True, seed=43,
                    device=dev)
    _, out, lse = _run(p)
    ro, rl = oracle.fia(p.to("cpu"))
    check_close(out, lse, ro, rl, "mode 2")


MASKS = {
    "mode0_per_batch": dict(mask_mode=0, mask_density=0.3),
    "mode1_shared": dict(mask_mode=1, mask_density=0.5, mask_shared=True),
    "mode1_full_rows": dict(mask_mode=1, mask_density=0.2, mask_full_rows=3, with_sinks=True),
    "mode0_dense": dict(mask_mode=0, mask_density=0.97),
}


@pytest.mark.parametrize("S", [1, 4])
@pytest.mark.parametrize("kv_dtype", [fi.KV_BF16, fi.KV_FP8_E4M3])
@pytest.mark.parametrize("name", sorted(MASKS))
def test_explicit_mask(name, kv_dtype, S):
    p = fi.make_fia(B=3, QN=8, KVN=2, D=128, q_lens=[S] * 3, kv_lens=[1500, 17, 300],
                    block_size=32, kv_dtype=kv_dtype, seed=_seed(name), device=dev,
                    **MASKS[name])
    _, out, lse = _run(p, num_sms=11)
    ro, rl = oracle.fia(p.to("cpu"))
    check_close(out, lse, ro, rl, name)


@pytest.mark.parametrize("bs", [16, 64, 128])
@pytest.mark.parametrize("kv_dtype", [fi.KV_BF16, fi.KV_FP8_E4M3])
def test_head_major_pages(kv_dtype, bs):
    if kv_dtype == fi.KV_FP8_E4M3 and bs == 16:
        bs = 32  # FP8 pages are multiples of 32 rows
    p = fi.make_fia(B=4, QN=32, KVN=4, D=128, q_lens=[2] * 4, kv_lens=[1000, 1, 257, 4000],
                    block_size=bs, kv_dtype=kv_dtype, kv_layout=fi.KV_LAYOUT_BNNBSD,
                    mask_mode=3, with_sinks=True, seed=bs, device=dev)
    _, out, lse = _run(p)
    ro, rl = oracle.fia(p.to("cpu"))
    check_close(out, lse, ro, rl, "BnNBsD")


def test_multi_row_schedule_bit_exact():
    p = fi.make_fia(B=5, QN=16, KVN=2, D=128, q_lens=[4, 0, 9, 1, 16],
                    kv_lens=[700, 30, 129, 0, 5000], layout=fi.LAYOUT_TND, block_size=16,
                    mask_mode=3, seed=47, device=dev)
    for n in (1, 7, 152):
        c, _, _ = _run(p, n)
        lay = c.plan_layout()
        ws = c.ws.cpu()
        U = lay.num_units
        per_cta = (lay.max_chunks - 2 * U) // n  # several rows: the bound n*W + 2*U
        nsched = 8 + 3 * (p.B + 1) + p.B
        sched = ws[lay.sched_off: lay.sched_off + 8 * nsched].view(torch.int64).numpy()
        rs, rq = oracle.decode_schedule(p.to("cpu"), n, per_cta)
        assert np.array_equal(sched, rs)
        N = int(sched[2])
        queue = ws[lay.queue_off: lay.queue_off + 16 * N].view(torch.int32).numpy().reshape(N, 4)
        assert np.array_equal(queue, rq)


def test_multi_token_decode_deterministic():
    p = fi.make_fia(B=2, QN=16, KVN=2, D=128, q_lens=[4, 4], kv_lens=[5000, 300],
                    block_size=128, mask_mode=3, seed=53, device=dev)
    _, o1, l1 = _run(p)
    o1, l1 = o1.clone(), l1.clone()
    _, o2, l2 = _run(p, num_sms=33)
    _, o3, l3 = _run(p)
    assert torch.equal(o1, o3) and torch.equal(l1, l3)
