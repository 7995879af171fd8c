"""Pins of the CPU oracle against what the pages and the mathematics fix.

Each test checks one property that a plausible mistake in the oracle (a dropped
term, a wrong sign or index, a transposed operand, a wrong mask bound) breaks.
None of them re-types the oracle's own row formula.
"""
import copy
import json
import math
import os

import numpy as np
import pytest
import torch

import fia_inputs as fi
import oracle
from oracle import naive

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _bf16(x):
    return torch.as_tensor(x, dtype=torch.float32).to(torch.bfloat16)


def _small(**kw):
    base = dict(B=2, QN=4, KVN=2, D=16, q_lens=[5, 5], kv_lens=[21, 9], layout=fi.LAYOUT_BSND,
                paged=True, block_size=8, seed=7)
    base.update(kw)
    return fi.make_fia(**base)


# --------------------------------------------------------------------------
# number formats
# --------------------------------------------------------------------------

def test_e4m3_decode_matches_library_cast_on_all_codes():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    lib_vals = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    mine = np.array([oracle.e4m3_to_double(c) for c in range(256)])
    nan = np.isnan(lib_vals)
    assert np.array_equal(nan, np.isnan(mine))
    assert nan.sum() == 2  # 0x7F and 0xFF only
    assert np.array_equal(lib_vals[~nan], mine[~nan])


def test_e4m3_known_values():
    # OCP FP8 E4M3: max normal 448, min normal 2^-6, min subnormal 2^-9, 1.0
    assert oracle.e4m3_to_double(0x7E) == 448.0
    assert oracle.e4m3_to_double(0x08) == 2.0 ** -6
    assert oracle.e4m3_to_double(0x01) == 2.0 ** -9
    assert oracle.e4m3_to_double(0x38) == 1.0
    assert oracle.e4m3_to_double(0xB8) == -1.0
    assert oracle.e4m3_to_double(0x80) == 0.0


def test_bf16_decode_matches_library():
    bits = np.arange(0, 65536, 257, dtype=np.int64)
    t = torch.tensor(bits.astype(np.uint16).view(np.int16)).view(torch.bfloat16)
    lib_vals = t.to(torch.float64).numpy()
    mine = np.array([oracle.bf16_to_double(int(b)) for b in bits])
    nan = np.isnan(lib_vals)
    assert np.array_equal(nan, np.isnan(mine))
    assert np.array_equal(lib_vals[~nan], mine[~nan])


# --------------------------------------------------------------------------
# closed forms and exact special cases
# --------------------------------------------------------------------------

def test_two_key_closed_form_golden():
    with open(os.path.join(GOLDEN, "two_key_closed_form.json")) as f:
        g = json.load(f)
    D = g["D"]
    p = fi.make_fia(B=1, QN=1, KVN=1, D=D, q_lens=[1], kv_lens=[2], paged=False, seed=1,
                    scale=g["scale"], poison=False)
    p.q = _bf16(np.array(g["q"]).reshape(1, 1, 1, D))
    p.k_cache = _bf16(np.array(g["k"]).reshape(1, 2, 1, D))
    p.v_cache = _bf16(np.array(g["v"]).reshape(1, 2, 1, D))
    out, lse = oracle.fia(p)
    np.testing.assert_allclose(out[0, 0], np.array(g["expected_out"]), rtol=0, atol=1e-15)
    assert abs(lse[0, 0, 0] - g["expected_lse"]) < 1e-15


def test_rows_sum_to_one_with_and_without_sink():
    for sinks in (False, True):
        for mode, pre, nxt in ((0, 0, 0), (3, 0, 0), (4, 3, 1)):
            p = _small(with_sinks=sinks, mask_mode=mode, pre_tokens=pre, next_tokens=nxt)
            for b in range(p.B):
                for h in range(p.QN):
                    for i in range(p.S_q):
                        lo, pr, ps = oracle.fia_row_probs(p, b, h, i)
                        if pr.size == 0:
                            continue
                        assert np.all(pr >= 0)
                        assert abs(pr.sum() + ps - 1.0) < 1e-12
                        if not sinks:
                            assert ps == 0.0


def test_lse_equals_logsumexp_of_scores():
    from scipy.special import logsumexp
    p = _small(mask_mode=3)
    out, lse = oracle.fia(p)
    q = p.q.double().numpy()
    for b in range(p.B):
        K = naive._dense_kv(p, b, "k")
        kl, ql = p.kv_lens[b], p.q_lens[b]
        for h in range(p.QN):
            g = h // (p.QN // p.KVN)
            for i in range(ql):
                pos = kl - ql + i
                s = p.scale * (K[: pos + 1, g, :] @ q[b, i, h])
                assert abs(lse[b, h, i] - logsumexp(s)) < 1e-12


def test_constant_v_returns_v():
    p = _small(mask_mode=3, with_sinks=False)
    c = torch.linspace(-2, 3, p.KVN * p.D).reshape(p.KVN, p.D)
    p.v_cache = _bf16(c).expand_as(p.v_cache).contiguous()
    out, _ = oracle.fia(p)
    G = p.QN // p.KVN
    expect = _bf16(c).double().numpy()
    for h in range(p.QN):
        np.testing.assert_allclose(out[:, h, :], np.broadcast_to(expect[h // G], (p.rows, p.D)),
                                   rtol=0, atol=1e-13)


def test_zero_query_gives_mean_of_visible_values():
    p = _small(mask_mode=0)
    p.q = torch.zeros_like(p.q)
    out, lse = oracle.fia(p)
    G = p.QN // p.KVN
    for b in range(p.B):
        V = naive._dense_kv(p, b, "v")
        for h in range(p.QN):
            np.testing.assert_allclose(out[b * p.S_q, h], V[:, h // G].mean(axis=0), rtol=0,
                                       atol=1e-13)
            assert abs(lse[b, h, 0] - math.log(p.kv_lens[b])) < 1e-13


def test_single_visible_key_returns_its_value_exactly():
    p = _small(kv_lens=[1, 1], q_lens=[1, 1])
    out, lse = oracle.fia(p)
    G = p.QN // p.KVN
    for b in range(p.B):
        V = naive._dense_kv(p, b, "v")
        for h in range(p.QN):
            assert np.array_equal(out[b, h], V[0, h // G])


def test_band_zero_width_returns_v_at_position():
    p = _small(mask_mode=4, pre_tokens=0, next_tokens=0)
    out, _ = oracle.fia(p)
    G = p.QN // p.KVN
    for b in range(p.B):
        V = naive._dense_kv(p, b, "v")
        kl, ql = p.kv_lens[b], p.q_lens[b]
        for i in range(ql):
            for h in range(p.QN):
                assert np.array_equal(out[b * ql + i, h], V[kl - ql + i, h // G])


def test_sink_only_enlarges_denominator():
    p0 = _small(mask_mode=3, with_sinks=False, seed=11)
    p1 = copy.copy(p0)
    p1.sinks = torch.tensor([0.3, -1.2, 2.5, 0.0], dtype=torch.float32)
    o0, l0 = oracle.fia(p0)
    o1, l1 = oracle.fia(p1)
    sinks = p1.sinks.double().numpy()
    for h in range(p0.QN):
        expect_l = np.logaddexp(l0[:, h, :], sinks[h])
        np.testing.assert_allclose(l1[:, h, :], expect_l, rtol=0, atol=1e-12)
        fac = np.exp(l0[:, h, :] - l1[:, h, :]).reshape(-1)
        np.testing.assert_allclose(o1[:, h, :], o0[:, h, :] * fac[:, None], rtol=0, atol=1e-12)


# --------------------------------------------------------------------------
# layout invariances
# --------------------------------------------------------------------------

def _to_contiguous(p):
    """The same problem with K/V gathered into a contiguous [B, S_kv, KVN, D]."""
    q = copy.copy(p)
    S = max(p.kv_lens)
    k = torch.zeros((p.B, S, p.KVN, p.D), dtype=p.k_cache.dtype)
    v = torch.zeros_like(k)
    bs = p.block_size
    for b in range(p.B):
        for j in range(p.kv_lens[b]):
            blk = int(p.block_table[b, j // bs])
            k[b, j] = p.k_cache[blk, j % bs]
            v[b, j] = p.v_cache[blk, j % bs]
    q.k_cache, q.v_cache = k, v
    if p.k_scale is not None:
        # head-major inside a page: [pages, KVN, rows, D/64]
        ks = torch.zeros((p.B, p.KVN, S, p.D // 64), dtype=torch.float32)
        vs = torch.zeros_like(ks)
        for b in range(p.B):
            for j in range(p.kv_lens[b]):
                blk = int(p.block_table[b, j // bs])
                ks[b, :, j] = p.k_scale[blk, :, j % bs]
                vs[b, :, j] = p.v_scale[blk, :, j % bs]
        q.k_scale, q.v_scale = ks, vs
    q.block_table = None
    q.S_kv = S
    return q


@pytest.mark.parametrize("kvd", [fi.KV_BF16, fi.KV_FP8_E4M3])
def test_paged_equals_contiguous_under_permutation(kvd):
    D = 64 if kvd == fi.KV_FP8_E4M3 else 16
    p = _small(D=D, kv_dtype=kvd, mask_mode=3, with_sinks=True)
    c = _to_contiguous(p)
    o1, l1 = oracle.fia(p)
    o2, l2 = oracle.fia(c)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)
    # and a second, different permutation of the same logical cache
    p2 = copy.copy(p)
    nb = p.num_blocks
    perm = torch.randperm(nb, generator=torch.Generator().manual_seed(5))
    inv = torch.argsort(perm)
    p2.k_cache = p.k_cache[perm]
    p2.v_cache = p.v_cache[perm]
    if p.k_scale is not None:
        p2.k_scale, p2.v_scale = p.k_scale[perm], p.v_scale[perm]
    p2.block_table = inv[p.block_table.long()].to(torch.int32)
    o3, l3 = oracle.fia(p2)
    assert np.array_equal(o1, o3) and np.array_equal(l1, l3)


def test_decode_equals_last_row_of_causal_prefill():
    L = 37
    pre = fi.make_fia(B=1, QN=4, KVN=2, D=16, q_lens=[L], kv_lens=[L], paged=True, block_size=8,
                      mask_mode=3, seed=3, with_sinks=True)
    dec = copy.copy(pre)
    dec.q = pre.q[:, L - 1:L].contiguous()
    dec.S_q, dec.T, dec.q_lens = 1, 1, [1]
    dec.mask_mode = 0
    o_p, l_p = oracle.fia(pre)
    o_d, l_d = oracle.fia(dec)
    assert np.array_equal(o_p[L - 1], o_d[0])
    assert np.array_equal(l_p[0, :, L - 1], l_d[0, :, 0])


def test_gqa_equals_replicated_kv_heads():
    p = _small(QN=8, KVN=2, mask_mode=3)
    r = copy.copy(p)
    G = 4
    r.KVN = 8
    r.k_cache = p.k_cache.repeat_interleave(G, dim=2).contiguous()
    r.v_cache = p.v_cache.repeat_interleave(G, dim=2).contiguous()
    o1, l1 = oracle.fia(p)
    o2, l2 = oracle.fia(r)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


def test_fp8_on_grid_equals_bf16():
    # codes times power-of-two scales are exact in bf16, so the FP8 cache and
    # the bf16 cache holding the decoded values are the same operand
    p = _small(D=64, kv_dtype=fi.KV_FP8_E4M3, mask_mode=0, poison=False)
    g = torch.Generator().manual_seed(9)
    ks = torch.exp2(torch.randint(-4, 4, p.k_scale.shape, generator=g).float())
    vs = torch.exp2(torch.randint(-4, 4, p.v_scale.shape, generator=g).float())
    codes_k = torch.randint(0, 256, p.k_cache.shape, generator=g, dtype=torch.int32)
    codes_v = torch.randint(0, 256, p.v_cache.shape, generator=g, dtype=torch.int32)
    codes_k[(codes_k & 0x7F) == 0x7F] = 0  # avoid the NaN codes
    codes_v[(codes_v & 0x7F) == 0x7F] = 0
    p.k_cache, p.v_cache = codes_k.to(torch.uint8), codes_v.to(torch.uint8)
    p.k_scale, p.v_scale = ks, vs
    b = copy.copy(p)
    b.kv_dtype = fi.KV_BF16
    # scales are stored [pages, KVN, rows, D/64]; the pool is [pages, rows, KVN, D]
    dk = p.k_cache.view(torch.float8_e4m3fn).float() * ks.transpose(1, 2).repeat_interleave(64, -1)
    dv = p.v_cache.view(torch.float8_e4m3fn).float() * vs.transpose(1, 2).repeat_interleave(64, -1)
    b.k_cache, b.v_cache = dk.to(torch.bfloat16), dv.to(torch.bfloat16)
    assert torch.equal(b.k_cache.float(), dk) and torch.equal(b.v_cache.float(), dv)
    b.k_scale = b.v_scale = None
    o1, l1 = oracle.fia(p)
    o2, l2 = oracle.fia(b)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


def test_quantiser_round_trip_bound():
    x = torch.randn(64, 128, generator=torch.Generator().manual_seed(4)).to(torch.bfloat16)
    codes, scales = fi.quantize_e4m3_per_tile(x)
    deq = np.array([oracle.e4m3_to_double(int(c)) for c in codes.reshape(-1)]).reshape(64, 128)
    deq *= np.repeat(scales.double().numpy(), 64, axis=-1)
    err = np.abs(deq - x.double().numpy())
    # half an E4M3 ulp of |x|/scale, times the scale (2^-4 relative for
    # normals, 2^-10 absolute in code units for subnormals), plus the rounding
    # of the fp32 division x/scale that precedes the cast (2^-24 relative)
    xs = np.abs(x.double().numpy()) / np.repeat(scales.double().numpy(), 64, axis=-1)
    ulp = np.where(xs >= 2.0 ** -6, 2.0 ** (np.floor(np.log2(np.maximum(xs, 1e-30))) - 3),
                   2.0 ** -9)
    bound = (0.5 * ulp + 2.0 ** -23 * xs) * np.repeat(scales.double().numpy(), 64, axis=-1)
    assert np.all(err <= bound)


# --------------------------------------------------------------------------
# empty and degenerate cases
# --------------------------------------------------------------------------

@pytest.mark.parametrize("sinks", [False, True])
def test_empty_kv_gives_zero_and_inf(sinks):
    p = _small(kv_lens=[0, 9], with_sinks=sinks)
    out, lse = oracle.fia(p)
    assert np.all(out[: p.S_q] == 0.0)
    assert np.all(np.isinf(lse[0])) and np.all(lse[0] > 0)
    assert np.all(np.isfinite(lse[1]))


def test_fully_masked_rows_when_q_longer_than_kv():
    p = _small(q_lens=[6, 6], kv_lens=[4, 9], mask_mode=3, with_sinks=True)
    out, lse = oracle.fia(p)
    # batch 0: p = 4 - 6 + i < 0 for i < 2
    assert np.all(out[0:2] == 0.0) and np.all(np.isinf(lse[0, :, 0:2]))
    assert np.all(np.isfinite(lse[0, :, 2:]))


# --------------------------------------------------------------------------
# brute force against the independent numpy statement
# --------------------------------------------------------------------------

CASES = [
    dict(B=2, QN=4, KVN=4, D=16, q_lens=[7, 7], kv_lens=[13, 33], mask_mode=3),
    dict(B=2, QN=4, KVN=2, D=32, q_lens=[1, 1], kv_lens=[17, 1], mask_mode=0),
    dict(B=1, QN=8, KVN=2, D=16, q_lens=[33], kv_lens=[33], mask_mode=4, pre_tokens=5,
         next_tokens=2),
    dict(B=2, QN=2, KVN=1, D=16, q_lens=[3, 9], kv_lens=[11, 9], layout=fi.LAYOUT_TND,
         mask_mode=3, with_sinks=True),
    dict(B=2, QN=4, KVN=2, D=64, q_lens=[5, 5], kv_lens=[31, 12], kv_dtype=fi.KV_FP8_E4M3,
         mask_mode=3),
    dict(B=2, QN=4, KVN=2, D=16, q_lens=[4, 4], kv_lens=[9, 3], mask_mode=4, pre_tokens=-1,
         next_tokens=3, with_sinks=True),
    dict(B=1, QN=2, KVN=2, D=16, q_lens=[5], kv_lens=[20], paged=False, mask_mode=3),
]


@pytest.mark.parametrize("case", range(len(CASES)))
def test_oracle_matches_naive(case):
    kw = dict(paged=True, block_size=16, seed=100 + case)
    kw.update(CASES[case])
    p = fi.make_fia(**kw)
    o1, l1 = oracle.fia(p)
    o2, l2 = naive.fia(p)
    np.testing.assert_allclose(o1, o2, rtol=0, atol=1e-12)
    fin = np.isfinite(l2)
    assert np.array_equal(fin, np.isfinite(l1))
    np.testing.assert_allclose(l1[fin], l2[fin], rtol=0, atol=1e-12)


def test_sample_equals_full():
    p = fi.make_fia(B=2, QN=4, KVN=2, D=16, q_lens=[6, 3], kv_lens=[19, 7], layout=fi.LAYOUT_TND,
                    mask_mode=3, with_sinks=True, block_size=8, seed=21)
    o, l = oracle.fia(p)
    rows = [0, 5, 6, 8, 2]
    heads = [0, 3, 1, 2, 2]
    so, sl = oracle.fia_sample(p, rows, heads)
    for k, (r, h) in enumerate(zip(rows, heads)):
        assert np.array_equal(so[k], o[r, h]) and sl[k] == l[r, h]


# --------------------------------------------------------------------------
# sparse shared-KV attention
# --------------------------------------------------------------------------

def _swa_as_fia(sp):
    """FIA problem with the ori pool as a one-head paged cache, band 127/0."""
    return fi.FiaProblem(B=sp.B, QN=sp.N1, KVN=1, D=sp.D, layout=sp.layout, S_q=sp.S1, T=sp.T1,
                         q=sp.q, cu_seqlens_q=sp.cu_seqlens_q, kv_dtype=0, k_cache=sp.ori_kv,
                         v_cache=sp.ori_kv, k_scale=None, v_scale=None,
                         block_table=sp.ori_block_table, block_size=sp.ori_block_size,
                         num_blocks=sp.ori_kv.shape[0],
                         S_kv=sp.ori_block_table.shape[1] * sp.ori_block_size,
                         seqused_kv=sp.seqused_kv, scale=sp.scale, mask_mode=4,
                         pre_tokens=sp.win_left, next_tokens=sp.win_right, sinks=sp.sinks,
                         q_lens=sp.q_lens, kv_lens=sp.kv_lens)


def test_sparse_swa_equals_fia_band():
    sp = fi.make_sparse(B=2, N1=4, D=32, q_lens=[3, 3], kv_lens=[200, 90], mode="swa",
                        ori_block_size=16, seed=31, win_left=20, win_right=0)
    o1, l1 = oracle.sparse(sp)
    o2, l2 = oracle.fia(_swa_as_fia(sp))
    np.testing.assert_allclose(o1, o2, rtol=0, atol=1e-13)
    np.testing.assert_allclose(l1, l2.transpose(0, 2, 1).reshape(-1, sp.N1), rtol=0, atol=1e-13)


def test_sparse_csa_listing_all_equals_hca():
    hca = fi.make_sparse(B=2, N1=4, D=32, q_lens=[2, 2], kv_lens=[90, 57], mode="hca",
                         ori_block_size=16, cmp_block_size=8, seed=41, win_left=9)
    csa = copy.copy(hca)
    rows = hca.rows
    K2 = 40
    idx = torch.full((rows, 1, K2), -1, dtype=torch.int32)
    r = 0
    for b in range(hca.B):
        for i in range(hca.q_lens[b]):
            p = hca.kv_lens[b] - hca.q_lens[b] + i
            n = (p + 1) // hca.cmp_ratio
            idx[r, 0, :n] = torch.arange(n, dtype=torch.int32)
            r += 1
    csa.cmp_sparse_indices, csa.K2 = idx, K2
    o1, l1 = oracle.sparse(hca)
    o2, l2 = oracle.sparse(csa)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


def test_sparse_csa_equals_dense_over_gathered_rows():
    sp = fi.make_sparse(B=2, N1=4, D=32, q_lens=[1, 1], kv_lens=[300, 160], mode="csa", K2=16,
                        ori_block_size=16, cmp_block_size=16, seed=51, win_left=7)
    o, l = oracle.sparse(sp)
    for b in range(sp.B):
        rows = oracle.sparse_rows(sp, b, 0)
        kk = []
        for kind, r in rows:
            if kind == "ori":
                blk = int(sp.ori_block_table[b, r // sp.ori_block_size])
                kk.append(sp.ori_kv[blk, r % sp.ori_block_size, 0])
            else:
                blk = int(sp.cmp_block_table[b, r // sp.cmp_block_size])
                kk.append(sp.cmp_kv[blk, r % sp.cmp_block_size, 0])
        K = torch.stack(kk).double().numpy()
        # window part is the band, compressed part the valid listed indices
        p = sp.kv_lens[b] - 1
        nwin = sum(1 for k, _ in rows if k == "ori")
        assert nwin == min(sp.win_left + 1, p + 1)
        listed = sp.cmp_sparse_indices[b, 0].tolist()
        valid = [c for c in listed if c >= 0 and c < (p + 1) // sp.cmp_ratio]
        assert [r for k, r in rows if k == "cmp"] == valid
        q = sp.q[b, 0].double().numpy()
        for h in range(sp.N1):
            s = sp.scale * (K @ q[h])
            z = np.concatenate([s, [float(sp.sinks[h])]])
            m = z.max()
            e = np.exp(z - m)
            pr = e[:-1] / e.sum()
            np.testing.assert_allclose(o[b, h], pr @ K, rtol=0, atol=1e-12)
            assert abs(l[b, h] - (m + math.log(e.sum()))) < 1e-12


# --------------------------------------------------------------------------
# schedules
# --------------------------------------------------------------------------

def _unit_chunks(sched, queue, B, UPB):
    """{unit: [(queue position, chunk index)]} from the queue entries."""
    out = {}
    for pos, (x, y, _, _) in enumerate(queue.tolist()):
        b = x & 0xFFFF
        w, i = y & 0xFFFF, y >> 16
        assert 0 <= b < B and w < UPB
        out.setdefault(b * UPB + w, []).append((pos, i))
    return out


@pytest.mark.parametrize("ctas,per_cta", [(1, 8), (7, 8), (152, 8), (500, 8), (152, 1), (3, 50)])
def test_decode_schedule_chunks_cover_each_unit_once(ctas, per_cta):
    kv = [0, 1, 300, 129, 1000, 5000, 128]
    p = fi.make_fia(B=len(kv), QN=8, KVN=2, D=16, q_lens=[1] * len(kv), kv_lens=kv,
                    block_size=16, seed=2)
    sched, queue = oracle.decode_schedule(p, ctas, per_cta)
    B, UPB = p.B, 2
    costs = [max(1, -(-k // 128)) for k in kv]          # no mask: every tile, at least 1
    T = UPB * sum(costs)
    C = max(1, -(-T // (ctas * per_cta)))
    c2 = -(-C // 2)                                      # bf16, one query row: k = 2
    assert list(sched[:2]) == [C, c2] and list(sched[5:8]) == [0x4649414445434F44, p.B, ctas]
    N, F = int(sched[2]), int(sched[3])
    assert N == queue.shape[0] and 0 <= F <= N
    assert N <= ctas * per_cta + 4 * B * UPB             # the workspace bound, 2k U
    Q = sched[8:8 + B + 1]
    # batches whose units need a split-KV combine, in order, then -1
    split = [b for b in range(B) if (Q[b + 1] - Q[b]) // UPB > 1]
    SB = sched[8 + 3 * (B + 1):]
    assert sched[4] == len(split) and list(SB) == split + [-1] * (B - len(split))
    chunks = _unit_chunks(sched, queue, B, UPB)
    for b in range(B):
        for w in range(UPB):
            lst = chunks[b * UPB + w]
            idx = sorted(i for _, i in lst)
            assert idx == list(range(len(idx)))          # chunks 0..k-1, once each
            assert Q[b + 1] - Q[b] == len(idx) * UPB
            n1 = sum(pos < F for pos, _ in lst)
            # big chunks come first in the unit; the small ones cover the rest
            assert all(i < n1 for pos, i in lst if pos < F)
            rest = costs[b] - n1 * C
            n2 = len(idx) - n1
            assert n2 >= 1 and (n2 - 1) * c2 < rest <= n2 * c2
            if n1 > 0:
                assert C <= rest < 2 * C                 # one big chunk left for the small ones
    # claim order: big chunks, then small, each batch-major, chunk, then unit
    keys = [(x & 0xFFFF, y >> 16, y & 0xFFFF) for x, y, _, _ in queue.tolist()]
    assert keys[:F] == sorted(keys[:F]) and keys[F:] == sorted(keys[F:])
    # every entry carries its batch, query length (one row here), KV length
    # and first query row (BSND: b * S_q)
    assert all(x >> 16 == 1 for x, _, _, _ in queue.tolist())
    assert [(kl, qr) for x, _, kl, qr in queue.tolist()] == \
        [(kv[x & 0xFFFF], x & 0xFFFF) for x, _, _, _ in queue.tolist()]


def test_decode_schedule_fp8_rest_in_at_most_two_chunks():
    """With an FP8 cache (k = 1) the rest of a unit (between C and 2C tiles)
    goes in chunks of C tiles, at most 2 of them."""
    kv = [30000, 70000, 128, 129 * 128]
    p = fi.make_fia(B=len(kv), QN=16, KVN=2, D=128, q_lens=[1] * len(kv), kv_lens=kv,
                    block_size=128, kv_dtype=fi.KV_FP8_E4M3, seed=4)
    for ctas, per in ((2, 5), (9, 5), (152, 5)):
        sched, queue = oracle.decode_schedule(p, ctas, per)
        costs = [max(1, -(-k // 128)) for k in kv]
        T = 2 * sum(costs)
        C = max(1, -(-T // (ctas * per)))
        c2 = C
        assert list(sched[:2]) == [C, c2]
        assert sched[2] <= ctas * per + 2 * 2 * len(kv)
        chunks = _unit_chunks(sched, queue, p.B, 2)
        F = int(sched[3])
        for b, c in enumerate(costs):
            for w in range(2):
                lst = chunks[b * 2 + w]
                n1 = sum(pos < F for pos, _ in lst)
                n2 = len(lst) - n1
                rest = c - n1 * C
                assert n2 <= 2 and (n2 - 1) * c2 < rest <= n2 * c2


def test_decode_schedule_band_counts_window_tiles_only():
    p = fi.make_fia(B=2, QN=2, KVN=1, D=16, q_lens=[1, 1], kv_lens=[1000, 100], block_size=16,
                    mask_mode=4, pre_tokens=200, next_tokens=0, seed=2)
    sched, queue = oracle.decode_schedule(p, 3, 8)
    # row position 999 sees [799, 999] -> tiles 6..7; position 99 sees [0, 99] -> tile 0
    # T = 3 tiles over 24 chunk slots: C = 1, so each tile is one chunk
    assert sched[0] == 1
    Q = sched[8:11]
    assert list(np.diff(Q)) == [2, 1]


@pytest.mark.parametrize("S,G,layout", [(4, 4, fi.LAYOUT_BSND), (2, 8, fi.LAYOUT_BSND),
                                         (16, 2, fi.LAYOUT_TND), (3, 1, fi.LAYOUT_TND)])
def test_decode_schedule_multi_row_units(S, G, layout):
    """Several query rows per sequence: a KV head's columns are its (row,
    head) pairs, S*G of them in groups of GH = 8 (16 only for one row with
    more than 8 heads per KV head); only the groups that
    hold columns of the sequence's own rows are scheduled, every active unit
    of a sequence costs the tiles its rows see together, and each of its
    chunks owns the slot Q[b] + i * A(b) + a."""
    kv = [700, 3, 129, 0, 1500]
    ql = [S] * 5 if layout == fi.LAYOUT_BSND else [S, 1, 0, 2, S]
    KVN = 2
    p = fi.make_fia(B=5, QN=G * KVN, KVN=KVN, D=16, q_lens=ql, kv_lens=kv, layout=layout,
                    block_size=16, mask_mode=3, seed=9)
    p.S_q = S  # the rows every decode unit covers (max_seqlen_q)
    GH = 16 if (S == 1 and G > 8) else 8
    HG = -(-S * G // GH)
    UPB = KVN * HG
    for ctas, per in ((1, 5), (9, 5), (152, 5)):
        sched, queue = oracle.decode_schedule(p, ctas, per)
        B = p.B
        Q = sched[8:8 + B + 1]
        HA = [-(-q * G // GH) if q > 0 else 0 for q in ql]
        A = [KVN * h for h in HA]
        # cost: tiles from row 0's bound to the last row's bound (causal:
        # keys 0 .. kv-1 for the last row), at least 1; none without rows
        cost = [0 if q == 0 else max(1, -(-k // 128)) for q, k in zip(ql, kv)]
        T = sum(c * a for c, a in zip(cost, A))
        C = max(1, -(-T // (ctas * per)))
        assert sched[0] == C
        chunks = {}
        for pos, (x, y, klen, qrow) in enumerate(queue.tolist()):
            b, qlen = x & 0xFFFF, x >> 16
            assert qlen == min(ql[b], S)
            w, i = y & 0xFFFF, y >> 16
            hk, hg = divmod(w, HG)
            assert hg < HA[b] and hk < KVN          # only units with columns
            assert klen == kv[b]
            assert qrow == (b * S if layout == fi.LAYOUT_BSND else sum(ql[:b]))
            chunks.setdefault((b, w), []).append(i)
        for b in range(B):
            for hk in range(KVN):
                for hg in range(HA[b]):
                    idx = sorted(chunks[(b, hk * HG + hg)])
                    assert idx == list(range(len(idx)))
                    assert Q[b + 1] - Q[b] == len(idx) * A[b]
            assert Q[b + 1] - Q[b] == 0 or A[b] > 0
        assert len(chunks) == sum(A)
        assert queue.shape[0] <= ctas * per + 2 * B * UPB  # several rows: k = 1


def test_prefill_units_enumerate_every_tile_and_head_pair():
    p = fi.make_fia(B=3, QN=8, KVN=2, D=16, q_lens=[300, 1, 129], kv_lens=[300, 1, 129],
                    layout=fi.LAYOUT_TND, block_size=16, mask_mode=3, seed=2)
    units, cost = oracle.prefill_units(p)
    assert units.shape[0] == (3 + 1 + 2) * 2 * 2
    # causal, kv == q: tile t sees KV tiles 0..t
    for (b, t, hk, pr), c in zip(units.tolist(), cost.tolist()):
        assert c == 1 + t + 1


def test_sparse_metadata_worked_example():
    """SWA with a 128-row band: every row weighs 2 chunks; N1 = 16 gives two
    8-head items per row.  Three rows -> item weights 2 x 6, T = 12; over 4
    CTAs the thresholds are 0, 3, 6, 9, 12 and the item offsets 0, 2, ..., 10,
    so the CTAs begin at items 0, 2, 3, 5 and the list ends at 6."""
    sp = fi.make_sparse(B=3, N1=16, D=32, q_lens=[1, 1, 1], kv_lens=[500, 7, 130], mode="swa",
                        ori_block_size=16, seed=62)
    md = oracle.sparse_metadata(sp, 4, 64, 8)
    assert list(md[:14]) == [0x46534D32, 4, 3, 64, 12, 3, 16, 0, 1, 127, 0, 0, 8, 6]
    assert list(md[16:21]) == [0, 2, 3, 5, 6]
    assert np.all(md[21:] == 0) and md[14] == 0 and md[15] == 0
    # the packed FP8 row format is recorded in [14]; nothing else changes
    spp = fi.make_sparse(B=3, N1=16, D=512, q_lens=[1, 1, 1], kv_lens=[500, 7, 130], mode="swa",
                         ori_block_size=16, seed=62, kv_dtype=fi.SPARSE_KV_FP8_PACKED)
    mdp = oracle.sparse_metadata(spp, 4, 64, 8)
    assert mdp[14] == 1 and list(mdp[:14]) == list(md[:14]) and list(mdp[16:21]) == [0, 2, 3, 5, 6]


def test_sparse_metadata_covers_every_item_in_order():
    sp = fi.make_sparse(B=3, N1=16, D=32, q_lens=[2, 2, 2], kv_lens=[600, 40, 3000], mode="csa",
                        K2=64, ori_block_size=16, cmp_block_size=16, seed=61)
    G = 2
    # per-row chunk counts from the definition: 2 window chunks (band 128)
    # plus the capped visible compressed rows in chunks of 64
    counts = []
    for b in range(sp.B):
        for i in range(2):
            p = sp.kv_lens[b] - 2 + i
            kc = min(64, (p + 1) // 4)
            counts.append(2 + -(-kc // 64))
    weights = np.repeat(counts, G)
    for n in (1, 5, 13, 152, 1007):
        md = oracle.sparse_metadata(sp, n, 64, 8)
        assert md[0] == 0x46534D32 and md[1] == n and md[2] == sp.rows and md[3] == 64
        assert md[4] == weights.sum() and md[13] == len(weights)
        begins = md[16:17 + n]
        # contiguous, ordered, every item exactly once
        assert begins[0] == 0 and begins[-1] == len(weights)
        assert np.all(np.diff(begins) >= 0)
        # balance: a CTA's weight exceeds its share by less than one item
        pre = np.concatenate([[0], np.cumsum(weights)])
        load = pre[begins[1:]] - pre[begins[:-1]]
        share = weights.sum() / n
        assert load.max() < share + weights.max()
        assert np.all(md[17 + n:] == 0)
    with pytest.raises(AssertionError):
        oracle.sparse_metadata(sp, 1008, 64, 8)
