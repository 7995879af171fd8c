"""FIA_DEBUG: with the switch set, the kernels report a block_table entry that
names a page outside the pool, for a key position they read, as 3 in the
error word; without it the same call reports nothing.  Either way such rows
are read as zeros (TMA boxes past the tensor map's rows fill with zeros) or
left out (sparse rows, the FP8 conversion pass), so the calls stay inside
every buffer."""
import pytest
import torch

import fia_inputs as fi

pytestmark = pytest.mark.gpu

dev = "cuda"


def _fia_problem(kind):
    fp8 = fi.KV_FP8_E4M3 if kind.endswith("fp8") else fi.KV_BF16
    if kind.startswith("decode"):
        return fi.make_fia(B=3, QN=8, KVN=2, D=128, q_lens=[1] * 3, kv_lens=[300, 40, 129],
                           block_size=64, kv_dtype=fp8, seed=5, device=dev)
    return fi.make_fia(B=2, QN=8, KVN=2, D=128, q_lens=[200, 77], kv_lens=[200, 77],
                       layout=fi.LAYOUT_TND, block_size=64, mask_mode=fi.MASK_RIGHT_DOWN_CAUSAL,
                       kv_dtype=fp8, seed=6, device=dev)


@pytest.mark.parametrize("kind", ["decode", "decode_fp8", "prefill", "prefill_fp8"])
def test_debug_reports_a_page_outside_the_pool(kind, monkeypatch):
    import decode_tile_scheduler_gb300 as fia
    p = _fia_problem(kind)
    # the first page of batch 1 (every batch sees its first keys)
    p.block_table[1, 0] = p.num_blocks + 5
    for switch, want in (("0", 0), ("1", 3)):
        monkeypatch.setenv("FIA_DEBUG", switch)
        c = fia.FiaCall(p, with_lse=True)
        c.run()
        torch.cuda.synchronize()
        assert c.error_word() == want, (kind, switch)


def test_debug_clean_call_reports_nothing(monkeypatch):
    import decode_tile_scheduler_gb300 as fia
    monkeypatch.setenv("FIA_DEBUG", "1")
    for kind in ("decode", "prefill"):
        c = fia.FiaCall(_fia_problem(kind), with_lse=True)
        c.run()
        torch.cuda.synchronize()
        assert c.error_word() == 0, kind


def test_debug_sparse_reports_a_window_page_outside_the_pool(monkeypatch):
    import decode_tile_scheduler_gb300 as fia
    sp = fi.make_sparse(B=2, N1=16, D=128, q_lens=[1, 1], kv_lens=[700, 300], mode="csa",
                        K2=64, seed=9, device=dev)
    for switch, want in (("1", 0), ("0", 0)):  # an intact table reports nothing
        monkeypatch.setenv("FIA_DEBUG", switch)
        c = fia.SparseCall(sp, with_lse=True)
        c.plan()
        c.run()
        torch.cuda.synchronize()
        assert int(c.ws[:4].view(torch.int32).item()) == want
    sp.ori_block_table[0, :] = int(sp.ori_kv.shape[0]) + 5
    for switch, want in (("0", 0), ("1", 3)):
        monkeypatch.setenv("FIA_DEBUG", switch)
        c = fia.SparseCall(sp, with_lse=True)
        c.plan()
        c.run()
        torch.cuda.synchronize()
        assert int(c.ws[:4].view(torch.int32).item()) == want, switch
