"""GPU parity of the shared-KV sparse attention (SWA / CSA / HCA) against the
fp64 oracle through the C ABI: the sparse CSA decode workload at full size,
TND and BSND, short sequences whose window starts before row 0, fewer
visible compressed rows than top-k, trailing -1 indices, sinks, head counts
4..128, D 128..512; the [1024] metadata bit-exact against the oracle's twin;
batch invariance; a metadata/shape mismatch reported in the status word."""
import numpy as np
import pytest
import torch

import fia_inputs as fi
import oracle
from helpers import check_close

pytestmark = pytest.mark.gpu
dev = "cuda"


def _run(sp, num_sms=0):
    import decode_tile_scheduler_gb300 as fia
    c = fia.SparseCall(sp, with_lse=True, num_sms=num_sms)
    c.plan()
    out, lse = c.run()
    torch.cuda.synchronize()
    assert int(c.ws[:4].view(torch.int32).item()) == 0
    return c, out, lse


def test_sparse_csa_workload_full_size():
    sp = fi.workload_sparse_csa(device=dev)
    c, out, lse = _run(sp)
    ro, rl = oracle.sparse(sp.to("cpu"))
    check_close(out, lse, ro, rl, "sparse CSA workload")


CASES = {
    "swa_tnd": dict(B=3, N1=8, D=128, q_lens=[5, 1, 3], kv_lens=[300, 20, 1000], mode="swa",
                    layout=fi.LAYOUT_TND, ori_block_size=16),
    "csa_short_seqs": dict(B=3, N1=16, D=256, q_lens=[2, 2, 2], kv_lens=[40, 3, 900], mode="csa",
                           K2=128, cmp_ratio=4, ori_block_size=32, cmp_block_size=16),
    "hca": dict(B=2, N1=4, D=128, q_lens=[3, 3], kv_lens=[5000, 700], mode="hca", cmp_ratio=128,
                ori_block_size=128, cmp_block_size=16),
    "csa_128_heads": dict(B=2, N1=128, D=512, q_lens=[1, 1], kv_lens=[3000, 517], mode="csa",
                          K2=512, cmp_ratio=4),
    "csa_no_sinks_window_right": dict(B=2, N1=8, D=128, q_lens=[4, 4], kv_lens=[200, 90],
                                      mode="csa", K2=64, win_left=30, win_right=2,
                                      with_sinks=False, ori_block_size=16, cmp_block_size=16),
    # pages of 48 and 80 rows (the page index is not a shift), one head group
    # of 2 heads, a long HCA list (several compressed chunks)
    "hca_odd_pages_two_heads": dict(B=2, N1=2, D=256, q_lens=[2, 1], kv_lens=[9000, 333],
                                    layout=fi.LAYOUT_TND, mode="hca", cmp_ratio=16,
                                    ori_block_size=48, cmp_block_size=80),
    "csa_odd_pages": dict(B=3, N1=32, D=128, q_lens=[1, 1, 1], kv_lens=[2500, 64, 700],
                          mode="csa", K2=300, cmp_ratio=4, ori_block_size=80,
                          cmp_block_size=48),
}


@pytest.mark.parametrize("name", sorted(CASES))
@pytest.mark.parametrize("num_sms", [0, 5])
def test_sparse_matches_oracle(name, num_sms):
    kw = dict(seed=len(name) * 7 + num_sms, device=dev)
    kw.update(CASES[name])
    sp = fi.make_sparse(**kw)
    _, out, lse = _run(sp, num_sms)
    ro, rl = oracle.sparse(sp.to("cpu"))
    check_close(out, lse, ro, rl, name)


def test_sparse_trailing_invalid_indices_and_duplicates():
    sp = fi.make_sparse(B=2, N1=4, D=128, q_lens=[1, 1], kv_lens=[2000, 1500], mode="csa", K2=256,
                        cmp_ratio=4, seed=91, device=dev)
    idx = sp.cmp_sparse_indices.clone()
    idx[0, 0, 100:] = -1            # a shorter valid prefix
    idx[1, 0, 10] = -1              # values after the first -1 are ignored
    idx[1, 0, 11:20] = 3
    sp.cmp_sparse_indices = idx
    _, out, lse = _run(sp)
    ro, rl = oracle.sparse(sp.to("cpu"))
    check_close(out, lse, ro, rl, "trailing -1")


def test_sparse_cta_count_invariance_and_one_cta_takes_every_item():
    """A row's chunks all run in one CTA, in order, whatever the CTA count:
    one CTA walking every item in turn (its stages and query buffer reused
    item after item), a few CTAs, and the default give the same bits, and
    match the oracle.  Rows of one, two and many chunks are mixed."""
    sp = fi.make_sparse(B=5, N1=32, D=128, q_lens=[1, 2, 1, 3, 1],
                        kv_lens=[4000, 30, 700, 129, 64], layout=fi.LAYOUT_TND, mode="csa",
                        K2=300, win_left=63, seed=23, device=dev)
    outs = []
    for n in (1, 6, 0):
        _, out, lse = _run(sp, n)
        outs.append((out.clone(), lse.clone()))
    for o, l in outs[1:]:
        assert torch.equal(o, outs[0][0]) and torch.equal(l, outs[0][1])
    ro, rl = oracle.sparse(sp.to("cpu"))
    check_close(outs[0][0], outs[0][1], ro, rl, "one CTA")


@pytest.mark.parametrize("num_sms", [1, 7, 152, 503, 1007])
def test_sparse_metadata_bit_exact(num_sms):
    import decode_tile_scheduler_gb300 as fia
    sp = fi.make_sparse(B=4, N1=8, D=128, q_lens=[3, 1, 2, 5], kv_lens=[600, 10, 3000, 128],
                        layout=fi.LAYOUT_TND, mode="csa", K2=200, seed=5, device=dev)
    c = fia.SparseCall(sp, num_sms=num_sms)
    c.plan()
    torch.cuda.synchronize()
    ref = oracle.sparse_metadata(sp.to("cpu"), num_sms, 64)
    assert np.array_equal(c.metadata.cpu().numpy(), ref)


@pytest.mark.parametrize("mode", ["swa", "hca"])
def test_sparse_metadata_bit_exact_other_modes(mode):
    import decode_tile_scheduler_gb300 as fia
    sp = fi.make_sparse(B=3, N1=32, D=128, q_lens=[1, 4, 2], kv_lens=[4000, 7, 900],
                        layout=fi.LAYOUT_TND, mode=mode, cmp_ratio=16, cmp_block_size=64,
                        seed=15, device=dev)
    for n in (3, 152):
        c = fia.SparseCall(sp, num_sms=n)
        c.plan()
        torch.cuda.synchronize()
        ref = oracle.sparse_metadata(sp.to("cpu"), n, 64)
        assert np.array_equal(c.metadata.cpu().numpy(), ref)


# packed FP8 K~ rows ("kv_quant_sparse_attn_sharedkv": bf16 rope 64, E4M3
# nope 448, E8M0 scales; D = 512)
PACKED = {
    "csa": dict(B=3, N1=64, q_lens=[1, 1, 1], kv_lens=[5000, 70, 1200], mode="csa", K2=512),
    "swa_tnd": dict(B=2, N1=8, q_lens=[3, 2], kv_lens=[400, 90], mode="swa",
                    layout=fi.LAYOUT_TND, ori_block_size=32),
    "hca_128_heads": dict(B=2, N1=128, q_lens=[1, 1], kv_lens=[9000, 300], mode="hca",
                          cmp_ratio=128, cmp_block_size=16),
    "csa_odd_pages": dict(B=2, N1=16, q_lens=[2, 2], kv_lens=[3000, 64], mode="csa", K2=300,
                          ori_block_size=80, cmp_block_size=48),
}


@pytest.mark.parametrize("num_sms", [0, 7])
@pytest.mark.parametrize("name", sorted(PACKED))
def test_sparse_packed_fp8_rows(name, num_sms):
    sp = fi.make_sparse(D=512, kv_dtype=fi.SPARSE_KV_FP8_PACKED, seed=70 + len(name), device=dev,
                        **PACKED[name])
    _, out, lse = _run(sp, num_sms)
    ro, rl = oracle.sparse(sp.to("cpu"))
    check_close(out, lse, ro, rl, name)


def test_sparse_packed_csa_workload_full_size():
    sp = fi.workload_sparse_csa(device=dev, kv_dtype=fi.SPARSE_KV_FP8_PACKED)
    _, out, lse = _run(sp)
    ro, rl = oracle.sparse(sp.to("cpu"))
    check_close(out, lse, ro, rl, "packed CSA workload")


def test_sparse_batch_invariance():
    full = fi.make_sparse(B=4, N1=8, D=128, q_lens=[2] * 4, kv_lens=[900, 300, 2500, 64],
                          mode="csa", K2=128, seed=7, device=dev)
    _, o_full, l_full = _run(full)
    o_full, l_full = o_full.clone(), l_full.clone()
    # the same third sequence alone, with the same caches and tables
    one = fi.SparseProblem(**{**full.__dict__})
    one.B = 1
    one.q = full.q[2:3].contiguous()
    one.ori_block_table = full.ori_block_table[2:3].contiguous()
    one.cmp_block_table = full.cmp_block_table[2:3].contiguous()
    one.cmp_sparse_indices = full.cmp_sparse_indices[4:6].contiguous()
    one.seqused_kv = full.seqused_kv[2:3].contiguous()
    one.q_lens, one.kv_lens = [2], [2500]
    one.T1 = 2
    _, o_one, l_one = _run(one, num_sms=3)
    assert torch.equal(o_full[2:3], o_one)
    assert torch.equal(l_full[4:6], l_one)


def test_sparse_metadata_mismatch_is_reported():
    import decode_tile_scheduler_gb300 as fia
    a = fi.make_sparse(B=2, N1=8, D=128, q_lens=[1, 1], kv_lens=[300, 200], mode="csa", K2=64,
                       seed=8, device=dev)
    b = fi.make_sparse(B=3, N1=8, D=128, q_lens=[1, 1, 1], kv_lens=[300, 200, 100], mode="csa",
                       K2=64, seed=9, device=dev)
    ca = fia.SparseCall(a)
    ca.plan()
    cb = fia.SparseCall(b)
    cb.plan()
    torch.cuda.synchronize()
    cb.out.fill_(0)
    # run b with a's metadata: detected on the device, nothing written
    fia.sparse_attn_run(cb.params, ca.metadata.data_ptr(), cb.ws.data_ptr(), cb.ws_bytes,
                        torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    assert int(cb.ws[:4].view(torch.int32).item()) == fia.FIA_ERR_BAD_SHAPE
    assert torch.count_nonzero(cb.out) == 0


def test_attention_waits_for_its_metadata_when_queued_behind_busy_work():
    """The attention kernel is launched behind the metadata kernel with
    programmatic serialization, so it may start while the metadata is still
    being written.  Queued behind a busy stream (the early start then really
    happens) over poisoned metadata, it still reads only the finished
    metadata: status 0 and the oracle's outputs, every time."""
    import decode_tile_scheduler_gb300 as fia
    sp = fi.make_sparse(device=dev, seed=61, **CASES["csa_odd_pages"])
    ro, rl = oracle.sparse(sp.to("cpu"))
    c = fia.SparseCall(sp, with_lse=True)
    c.plan()
    for _ in range(3):
        c.metadata.fill_(0x5A5A5A5A)
        c.out.fill_(float("nan"))
        torch.cuda._sleep(2_000_000)
        c.plan()
        c.run()
        torch.cuda.synchronize()
        assert int(c.ws[:4].view(torch.int32).item()) == 0
        check_close(c.out, c.lse, ro, rl, "queued behind busy work")
