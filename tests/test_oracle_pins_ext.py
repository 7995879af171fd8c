"""Pins of the oracle's mask modes 1 and 2, the explicit attention mask, the
head-major (BnNBsD) page layout, the packed FP8 rows of the shared-KV sparse
variant (E8M0 tile scales) and the log-sum-exp combine of partial results.

Each test checks a property fixed by the pages or by the mathematics, chosen
so that a plausible slip in the oracle (a wrong mask anchor, a transposed page,
a scale taken from the wrong tile, an exponent bias off by one, a missing
renormalisation) fails it.  None re-types the oracle's row formula.
"""
import copy
import dataclasses
import math

import numpy as np
import pytest
import torch

import fia_inputs as fi
import oracle
from oracle import naive


def _small(**kw):
    base = dict(B=2, QN=4, KVN=2, D=16, q_lens=[5, 5], kv_lens=[21, 9], layout=fi.LAYOUT_BSND,
                paged=True, block_size=8, seed=7)
    base.update(kw)
    return fi.make_fia(**base)


# --------------------------------------------------------------------------
# E8M0 and the packed FP8 rows ("kv_quant_sparse_attn_sharedkv" constraints)
# --------------------------------------------------------------------------

def test_e8m0_decode_on_all_codes():
    vals = np.array([oracle.e8m0_to_double(c) for c in range(256)])
    assert np.isnan(vals[255])
    # printed anchors of the format: bias 127, no mantissa, no sign
    assert vals[127] == 1.0 and vals[128] == 2.0 and vals[126] == 0.5
    assert vals[0] == 2.0 ** -127 and vals[254] == 2.0 ** 127
    # the library's own cast, where this torch has the type
    if hasattr(torch, "float8_e8m0fnu"):
        lib = torch.arange(256, dtype=torch.int32).to(torch.uint8).view(torch.float8_e8m0fnu)
        lib = lib.to(torch.float64).numpy()
        assert np.array_equal(np.isnan(lib), np.isnan(vals))
        assert np.array_equal(lib[:255], vals[:255])


def _grid_values(shape, seed):
    """bf16 K~ rows whose nope tiles sit on an E4M3 grid times a power of two
    (2^-3 .. 2^3 per tile), so the packed format holds them exactly."""
    g = torch.Generator().manual_seed(seed)
    x = torch.randn(shape, generator=g)
    rows = x.reshape(-1, 512)
    k = torch.randint(-3, 4, (rows.shape[0], 7), generator=g).double()
    nope = rows[:, 64:].reshape(-1, 7, 64).double()
    s = torch.exp2(k).unsqueeze(-1)
    on_grid = (nope / s).float().to(torch.float8_e4m3fn).double() * s
    rows = torch.cat([rows[:, :64].double(), on_grid.reshape(-1, 448)], dim=1)
    return rows.reshape(shape).to(torch.bfloat16)


def test_packed_rows_on_the_grid_equal_their_bf16_values():
    """The packed rows of values the format holds exactly give the attention of
    those values: this fixes the byte order (rope, nope codes, then the 7
    scales), the E8M0 bias and the tile of each nope element."""
    sp = fi.make_sparse(B=2, N1=8, D=512, q_lens=[2, 2], kv_lens=[300, 700], mode="csa",
                        K2=64, seed=13, poison=False)
    ori = _grid_values(sp.ori_kv.shape, 1)
    cmp = _grid_values(sp.cmp_kv.shape, 2)
    bf = dataclasses.replace(sp, ori_kv=ori, cmp_kv=cmp)
    pk = dataclasses.replace(sp, ori_kv=fi.pack_fp8_sparse_rows(ori),
                             cmp_kv=fi.pack_fp8_sparse_rows(cmp), kv_dtype=fi.SPARSE_KV_FP8_PACKED)
    ob, lb = oracle.sparse(bf)
    op, lp = oracle.sparse(pk)
    np.testing.assert_allclose(op, ob, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lp, lb, rtol=0, atol=1e-12)


def test_packed_quantiser_error_bound():
    """The cache-write side: every nope element is within half an E4M3 step of
    its source (relative 2^-4, or 2^-10 of the tile scale among subnormals),
    the scale is the smallest power of two keeping the tile within 448, and the
    rope part is stored unchanged."""
    g = torch.Generator().manual_seed(5)
    x = (torch.randn((40, 512), generator=g) * torch.exp2(torch.randint(-6, 7, (40, 1),
                                                                          generator=g))).to(
        torch.bfloat16)
    pk = fi.pack_fp8_sparse_rows(x).numpy()
    src = x.double().numpy()
    for r in range(40):
        rope = pk[r, :128].view(np.uint16)
        assert np.array_equal(rope, x[r, :64].view(torch.int16).numpy().view(np.uint16))
        for t in range(7):
            e = int(pk[r, 576 + t])
            sc = oracle.e8m0_to_double(e)
            tile = src[r, 64 + 64 * t: 128 + 64 * t]
            amax = np.abs(tile).max()
            assert amax / sc <= 448 and (amax == 0 or amax / (sc / 2) > 448)
            dec = np.array([oracle.e4m3_to_double(int(c)) for c in pk[r, 128 + 64 * t:192 + 64 * t]])
            err = np.abs(dec * sc - tile)
            bound = np.maximum(np.abs(tile) * 2.0 ** -4, sc * 2.0 ** -10)
            assert np.all(err <= bound * (1 + 1e-12))
        assert np.all(pk[r, 583:] == 0)


# --------------------------------------------------------------------------
# head-major pages ("aclnnFusedInferAttentionScoreV5", Paged Attention group)
# --------------------------------------------------------------------------

@pytest.mark.parametrize("kvd", [fi.KV_BF16, fi.KV_FP8_E4M3])
def test_head_major_pages_equal_token_major(kvd):
    kw = dict(kv_dtype=kvd, D=128 if kvd else 16, block_size=32 if kvd else 8)
    a = _small(**kw)
    b = _small(kv_layout=fi.KV_LAYOUT_BNNBSD, **kw)
    # same draws (bit for bit, NaN poison included): only the storage order differs
    bits = torch.int16 if kvd == fi.KV_BF16 else torch.uint8
    assert torch.equal(a.k_cache.permute(0, 2, 1, 3).contiguous().view(bits), b.k_cache.view(bits))
    oa, la = oracle.fia(a)
    ob, lb = oracle.fia(b)
    assert np.array_equal(oa, ob) and np.array_equal(la, lb)
    on, ln = naive.fia(b)
    np.testing.assert_allclose(ob, on, rtol=0, atol=1e-12)


# --------------------------------------------------------------------------
# mask modes 1 and 2 and the explicit mask ("...V5", Attention Mask group)
# --------------------------------------------------------------------------

def test_left_up_causal_equals_right_down_when_square():
    a = _small(q_lens=[9, 9], kv_lens=[9, 9], mask_mode=2)
    b = _small(q_lens=[9, 9], kv_lens=[9, 9], mask_mode=3)
    oa, la = oracle.fia(a)
    ob, lb = oracle.fia(b)
    assert np.array_equal(oa, ob) and np.array_equal(la, lb)


def test_left_up_causal_anchors_at_the_first_key():
    """Left-up causal: query row i sees keys 0..i whatever the KV length, so a
    single query row sees key 0 alone (its value, exactly), and a row past the
    keys sees them all."""
    p = _small(q_lens=[1, 1], kv_lens=[21, 9], mask_mode=2)
    o, l = oracle.fia(p)
    for b in range(2):
        j = 0
        blk = int(p.block_table[b, j // p.block_size])
        for h in range(p.QN):
            v = p.v_cache[blk, j % p.block_size, h // 2].double().numpy()
            np.testing.assert_array_equal(o[b, h], v)
    q = _small(q_lens=[12, 12], kv_lens=[5, 9], mask_mode=2, layout=fi.LAYOUT_BSND)
    o2, l2 = oracle.fia(q)
    n2, m2 = naive.fia(q)
    np.testing.assert_allclose(o2, n2, rtol=0, atol=1e-12)
    # rows 8..11 of batch 1 see all 9 keys: the same as mode 0 there
    r = _small(q_lens=[12, 12], kv_lens=[5, 9], mask_mode=0, layout=fi.LAYOUT_BSND)
    o3, _ = oracle.fia(r)
    np.testing.assert_array_equal(o2[12 + 8:24], o3[12 + 8:24])


def test_zero_mask_equals_no_mask():
    a = _small(q_lens=[5, 5], kv_lens=[21, 9], mask_density=0.0)
    b = _small(q_lens=[5, 5], kv_lens=[21, 9])
    assert a.atten_mask is not None and int(a.atten_mask.sum()) == 0
    oa, la = oracle.fia(a)
    ob, lb = oracle.fia(b)
    assert np.array_equal(oa, ob) and np.array_equal(la, lb)


def test_causal_pattern_mask_equals_right_down_causal():
    """A mask holding exactly the keys past each row's diagonal reproduces
    mode 3; under mode 1 (mask required) it means the same."""
    a = _small(q_lens=[5, 5], kv_lens=[21, 9], mask_density=0.0)
    m = a.atten_mask.clone()
    for b in range(2):
        for i in range(5):
            p = a.kv_lens[b] - 5 + i
            m[b, i, p + 1:] = 1
    a = dataclasses.replace(a, atten_mask=m)
    ref = dataclasses.replace(a, atten_mask=None, mask_mode=3)
    oa, la = oracle.fia(a)
    orf, lrf = oracle.fia(ref)
    assert np.array_equal(oa, orf) and np.array_equal(la, lrf)
    o1, l1 = oracle.fia(dataclasses.replace(a, mask_mode=1))
    assert np.array_equal(o1, orf) and np.array_equal(l1, lrf)


def test_fully_masked_row_gives_zero_and_inf_even_with_a_sink():
    p = _small(q_lens=[5, 5], kv_lens=[21, 9], mask_density=0.3, mask_full_rows=2,
               with_sinks=True)
    o, l = oracle.fia(p)
    # rows 0 and 1 of batch 0 hide every key
    assert np.all(o[0:2] == 0.0) and np.all(np.isinf(l[0, :, 0:2]))
    assert np.all(np.isfinite(l[0, :, 2:]))


@pytest.mark.parametrize("case", [
    dict(mask_density=0.4),
    dict(mask_density=0.4, mask_shared=True),
    dict(mask_density=0.7, mask_mode=1, layout=fi.LAYOUT_TND, q_lens=[7, 2], kv_lens=[30, 2]),
    dict(mask_density=0.2, kv_dtype=fi.KV_FP8_E4M3, D=128, block_size=32),
    dict(mask_mode=2, q_lens=[3, 3], kv_lens=[7, 1]),
    dict(mask_mode=2, layout=fi.LAYOUT_TND, q_lens=[11, 4], kv_lens=[6, 20], with_sinks=True),
])
def test_oracle_matches_naive_with_masks(case):
    p = _small(**case)
    o, l = oracle.fia(p)
    on, ln = naive.fia(p)
    np.testing.assert_allclose(o, on, rtol=0, atol=1e-12)
    fin = np.isfinite(ln)
    assert np.array_equal(np.isfinite(l), fin)
    np.testing.assert_allclose(l[fin], ln[fin], rtol=0, atol=1e-12)


# --------------------------------------------------------------------------
# log-sum-exp combine ("...V2" softmax_lse: the ring-attention use)
# --------------------------------------------------------------------------

def _kv_part(p, first_block, n_blocks):
    """The same decode problem restricted to keys [first_block*bs,
    (first_block+n_blocks)*bs) of each sequence (clipped to its length),
    built by slicing the block table and the lengths; without sinks."""
    bs = p.block_size
    lens = [max(0, min(k, (first_block + n_blocks) * bs) - first_block * bs) for k in p.kv_lens]
    bt = p.block_table[:, first_block:first_block + n_blocks].contiguous()
    return dataclasses.replace(p, block_table=bt, kv_lens=lens,
                               seqused_kv=torch.tensor(lens, dtype=torch.int32), sinks=None)


@pytest.mark.parametrize("cuts", [[2], [1, 3], [1, 2, 3], [5, 8]])
def test_combine_of_disjoint_key_parts_equals_the_whole(cuts):
    # the cut at block 5 leaves the second and third sequences without keys
    # in the later parts; the sink enters through the combine
    p = fi.make_fia(B=3, QN=8, KVN=2, D=32, q_lens=[1] * 3, kv_lens=[70, 17, 33],
                    block_size=8, with_sinks=True, seed=21)
    bounds = [0] + cuts + [p.max_blocks]
    parts = []
    for k in range(len(bounds) - 1):
        parts.append(oracle.fia(_kv_part(p, bounds[k], bounds[k + 1] - bounds[k])))
    # one query row per sequence: out [B, QN, D] goes with lse [B, QN]
    out, lse = oracle.lse_combine([o for o, _ in parts],
                                  [l.reshape(p.B, p.QN) for _, l in parts],
                                  sinks=p.sinks.numpy(), head_axis=1)
    ow, lw = oracle.fia(p)
    np.testing.assert_allclose(out, ow, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, lw.reshape(p.B, p.QN), rtol=0, atol=1e-12)


def test_combine_sink_alone_does_not_make_a_row_visible():
    # every part empty: 0 / +inf even with a sink (the empty-row rule)
    o = np.ones((2, 3, 4))
    l = np.full((2, 3), np.inf)
    out, lse = oracle.lse_combine([o, o], [l, l], sinks=np.array([0.5, 1.0, 2.0]), head_axis=1)
    assert np.all(out == 0.0) and np.all(np.isinf(lse))


def test_combine_skips_empty_parts_and_keeps_the_empty_rule():
    o1 = np.random.default_rng(0).standard_normal((3, 4))
    l1 = np.array([0.5, np.inf, -2.0])
    o2 = np.random.default_rng(1).standard_normal((3, 4))
    l2 = np.array([np.inf, np.inf, 1.0])
    out, lse = oracle.lse_combine([o1, o2], [l1, l2])
    np.testing.assert_array_equal(out[0], o1[0])            # one part saw keys
    assert lse[0] == 0.5
    assert np.all(out[1] == 0.0) and np.isinf(lse[1])       # no part saw a key
    w1 = math.exp(-2.0) / (math.exp(-2.0) + math.exp(1.0))
    np.testing.assert_allclose(out[2], w1 * o1[2] + (1 - w1) * o2[2], rtol=0, atol=1e-15)
    assert abs(lse[2] - math.log(math.exp(-2.0) + math.exp(1.0))) < 1e-15
