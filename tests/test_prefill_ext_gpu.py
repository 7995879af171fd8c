"""GPU parity of the prefill branch (tcgen05 kernel) for the mask and cache
forms beyond the right-down causal / band / none masks on token-major bf16
pages, through the C ABI, against the fp64 oracle:

* mask mode 2 (causal from the top-left corner), queries shorter, equal and
  longer than the keys;
* the explicit attention mask of modes 0 and 1: per batch and shared,
  fully hidden rows, BSND and TND, D 64 and 128;
* head-major (BnNBsD) pages;
* FP8 E4M3 K/V with fp32 per-64 scales (dequantised once to bf16 in the
  workspace), paged token- and head-major and contiguous, and the varlen
  causal prefill workload with an FP8 cache, sampled.
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
    assert c.plan_layout().branch == 2  # the tcgen05 prefill kernel
    out, lse = c.run()
    torch.cuda.synchronize()
    assert c.error_word() == 0
    return c, out, lse


CASES = {
    "mode2_tnd": dict(B=3, QN=8, KVN=2, D=128, q_lens=[300, 40, 129], kv_lens=[700, 40, 50],
                      layout=fi.LAYOUT_TND, block_size=64, mask_mode=2, with_sinks=True),
    "mode2_bsnd_d64": dict(B=2, QN=4, KVN=4, D=64, q_lens=[200, 200], kv_lens=[130, 400],
                           block_size=16, mask_mode=2),
    "mask0_per_batch": dict(B=2, QN=8, KVN=2, D=128, q_lens=[150, 150], kv_lens=[300, 90],
                            block_size=32, mask_mode=0, mask_density=0.3),
    "mask1_shared_tnd": dict(B=3, QN=8, KVN=2, D=128, q_lens=[40, 200, 17],
                             kv_lens=[40, 333, 500], layout=fi.LAYOUT_TND, block_size=64,
                             mask_mode=1, mask_density=0.6, mask_shared=True, with_sinks=True),
    "mask1_full_rows_d64": dict(B=2, QN=4, KVN=2, D=64, q_lens=[130, 130], kv_lens=[260, 20],
                                block_size=16, mask_mode=1, mask_density=0.1,
                                mask_full_rows=5),
    "head_major_bs16": dict(B=2, QN=8, KVN=2, D=128, q_lens=[300, 77], kv_lens=[300, 77],
                            layout=fi.LAYOUT_TND, block_size=16, mask_mode=3,
                            kv_layout=fi.KV_LAYOUT_BNNBSD, with_sinks=True),
    "head_major_bs128_band": dict(B=2, QN=16, KVN=4, D=128, q_lens=[257, 257],
                                  kv_lens=[400, 257], block_size=128, mask_mode=4,
                                  pre_tokens=100, next_tokens=5,
                                  kv_layout=fi.KV_LAYOUT_BNNBSD),
    "fp8_causal_tnd": dict(B=3, QN=8, KVN=2, D=128, q_lens=[300, 20, 129], kv_lens=[300, 20, 129],
                           layout=fi.LAYOUT_TND, block_size=64, mask_mode=3, with_sinks=True,
                           kv_dtype=fi.KV_FP8_E4M3),
    "fp8_head_major": dict(B=2, QN=16, KVN=2, D=128, q_lens=[200, 200], kv_lens=[500, 210],
                           block_size=32, mask_mode=3, kv_dtype=fi.KV_FP8_E4M3,
                           kv_layout=fi.KV_LAYOUT_BNNBSD),
    "fp8_contiguous_band": dict(B=2, QN=8, KVN=2, D=128, q_lens=[64, 64], kv_lens=[200, 64],
                                paged=False, mask_mode=4, pre_tokens=50, next_tokens=0,
                                kv_dtype=fi.KV_FP8_E4M3),
    "fp8_mask": dict(B=2, QN=8, KVN=2, D=128, q_lens=[100, 100], kv_lens=[180, 100],
                     block_size=32, mask_mode=1, mask_density=0.4, kv_dtype=fi.KV_FP8_E4M3),
}


@pytest.mark.parametrize("name", sorted(CASES))
def test_prefill_ext_matches_oracle(name):
    kw = dict(seed=zlib.crc32(name.encode()) % 1000, device=dev)
    kw.update(CASES[name])
    p = fi.make_fia(**kw)
    _, out, lse = _run(p, num_sms=0 if "fp8" in name else 37)
    ro, rl = oracle.fia(p.to("cpu"))
    check_close(out, lse, ro, rl, name)


def test_fp8_varlen_causal_prefill_workload_sampled():
    # the varlen causal prefill workload with an FP8 E4M3 cache: every 16th
    # query row with all heads, plus each sequence's first and last row
    g = torch.Generator().manual_seed(1003)
    L = torch.randint(256, 4097, (8,), generator=g).tolist()
    p = fi.make_fia(B=8, QN=32, KVN=8, D=128, q_lens=L, kv_lens=L, layout=fi.LAYOUT_TND,
                    block_size=128, mask_mode=3, with_sinks=True, kv_dtype=fi.KV_FP8_E4M3,
                    seed=1003, device=dev)
    _, out, lse = _run(p)
    pc = p.to("cpu")
    cu = pc.cu_seqlens_q.tolist()
    sel = sorted(set(range(0, p.T, 16)) | set(cu[:-1]) | set(c - 1 for c in cu[1:]))
    rows = np.repeat(np.array(sel, dtype=np.int64), p.QN)
    heads = np.tile(np.arange(p.QN, dtype=np.int32), len(sel))
    ro, rl = oracle.fia_sample(pc, rows, heads)
    o = out.float().cpu().numpy().reshape(p.T, p.QN, p.D)
    l = lse.cpu().numpy().reshape(p.T, p.QN)
    err = np.abs(o[rows, heads] - ro)
    assert err.max() <= 2e-2 and err.mean() <= 2e-3, (err.max(), err.mean())
    assert np.abs(l[rows, heads] - rl).max() <= 1e-3
