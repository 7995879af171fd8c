"""Seeded synthetic inputs for fused inference attention over a paged KV cache.

This module is the only code shared by the CUDA path's tests/benchmark and the
CPU oracle.  It draws random numbers, lays them out in the tensors the operators
take (paged pools, block tables, length arrays, sparse index lists) and packs a
KV cache into FP8 E4M3 with one fp32 scale per 64-element tile (the cache-write
side of the FP8 KV format).  It holds none of the attention arithmetic.

Recipe (per workload, seed s):
  1. lengths from a CPU ``torch.Generator`` seeded with s (``randint``),
  2. the physical block permutation (``randperm``),
  3. Q, K, V ~ N(0, 1) in fp32, rounded to bf16 (round-to-nearest-even), drawn
     from a generator on the target device seeded with s + 1,
  4. sinks ~ N(0, 1) fp32,
  5. sparse indices: per query, ``randperm`` of the causally visible compressed
     rows, first K2 kept (unsorted), padded with -1.
Pool rows that hold no token of any sequence (spare blocks, and the unused tail
of each sequence's last block) are poisoned with NaN so that an over-read shows.
Unused block-table slots point at a poisoned spare block.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional, Sequence

import torch

LAYOUT_BSND = 0
LAYOUT_TND = 1
KV_BF16 = 0
KV_FP8_E4M3 = 1
MASK_NONE = 0
MASK_ALL = 1
MASK_LEFT_UP_CAUSAL = 2
MASK_RIGHT_DOWN_CAUSAL = 3
MASK_BAND = 4
KV_LAYOUT_BNBSH = 0
KV_LAYOUT_BNNBSD = 1
SPARSE_KV_BF16 = 0
SPARSE_KV_FP8_PACKED = 1

N_SPARE_BLOCKS = 8
FP8_TILE = 64
FP8_MAX = 448.0


@dataclasses.dataclass
class FiaProblem:
    """One fused-inference-attention call: tensors plus scalar attributes."""
    B: int
    QN: int
    KVN: int
    D: int
    layout: int
    S_q: int                      # BSND query length (TND: max query length)
    T: int                        # TND total query rows (BSND: B*S_q)
    q: torch.Tensor               # bf16 [B,S_q,QN,D] or [T,QN,D]
    cu_seqlens_q: Optional[torch.Tensor]   # int32 [B+1] (TND)
    kv_dtype: int
    k_cache: torch.Tensor         # bf16 or uint8 (E4M3 codes)
    v_cache: torch.Tensor
    k_scale: Optional[torch.Tensor]        # fp32 [nb,KVN,bs,D/64] / [B,KVN,S_kv,D/64] (FP8)
    v_scale: Optional[torch.Tensor]
    block_table: Optional[torch.Tensor]    # int32 [B,max_blocks] or None
    block_size: int
    num_blocks: int
    S_kv: int                     # contiguous KV length (paged: max_blocks*bs)
    seqused_kv: Optional[torch.Tensor]     # int32 [B]
    scale: float
    mask_mode: int = MASK_NONE
    pre_tokens: int = 0
    next_tokens: int = 0
    sinks: Optional[torch.Tensor] = None   # fp32 [QN]
    q_lens: Optional[list] = None          # host copy of query lengths
    kv_lens: Optional[list] = None         # host copy of KV lengths
    kv_layout: int = KV_LAYOUT_BNBSH       # paged pools: [nb,bs,KVN,D] or [nb,KVN,bs,D]
    atten_mask: Optional[torch.Tensor] = None  # uint8 [B or 1, rows, cols], 1 = hidden

    @property
    def max_blocks(self) -> int:
        return 0 if self.block_table is None else int(self.block_table.shape[1])

    @property
    def rows(self) -> int:
        return self.T if self.layout == LAYOUT_TND else self.B * self.S_q

    def to(self, device) -> "FiaProblem":
        kw = {}
        for f in dataclasses.fields(self):
            v = getattr(self, f.name)
            kw[f.name] = v.to(device) if isinstance(v, torch.Tensor) else v
        return FiaProblem(**kw)

    def kv_bytes_visible(self) -> int:
        """Bytes of K and V (and FP8 scales) the method must read: every
        visible (token, kv-head) row once for K and once for V."""
        per_row = self.D * (2 if self.kv_dtype == KV_BF16 else 1)
        if self.kv_dtype == KV_FP8_E4M3:
            per_row += 4 * (self.D // FP8_TILE)
        return 2 * per_row * self.KVN * sum(self.visible_kv_per_seq())

    def visible_kv_per_seq(self):
        """Union over query rows of the visible KV positions, per sequence."""
        out = []
        for b in range(self.B):
            ql, kl = self.q_lens[b], self.kv_lens[b]
            if ql == 0 or kl == 0:
                out.append(0)
                continue
            off = 0 if self.mask_mode == MASK_LEFT_UP_CAUSAL else kl - ql
            p0, p1 = off, off + ql - 1
            lo = p0 - self.pre_tokens if self.mask_mode == MASK_BAND else 0
            hi = (p1 if self.mask_mode in (MASK_RIGHT_DOWN_CAUSAL, MASK_LEFT_UP_CAUSAL) else
                  p1 + self.next_tokens if self.mask_mode == MASK_BAND else kl - 1)
            lo, hi = max(lo, 0), min(hi, kl - 1)
            out.append(max(0, hi - lo + 1))
        return out


@dataclasses.dataclass
class SparseProblem:
    """One shared-KV sparse attention call (SWA / CSA / HCA)."""
    B: int
    N1: int
    D: int
    layout: int
    S1: int
    T1: int
    q: torch.Tensor                 # bf16 [B,S1,N1,D] or [T1,N1,D]
    cu_seqlens_q: Optional[torch.Tensor]
    ori_kv: torch.Tensor            # bf16 [nb1,bs1,1,D]
    ori_block_table: torch.Tensor   # int32 [B, >=ceil(S2max/bs1)]
    ori_block_size: int
    cmp_kv: Optional[torch.Tensor]  # bf16 [nb2,bs2,1,D]
    cmp_block_table: Optional[torch.Tensor]
    cmp_block_size: int
    cmp_sparse_indices: Optional[torch.Tensor]   # int32 [rows,1,K2]
    K2: int
    seqused_kv: torch.Tensor        # int32 [B]
    sinks: Optional[torch.Tensor]   # fp32 [N1]
    scale: float
    cmp_ratio: int = 4
    win_left: int = 127
    win_right: int = 0
    q_lens: Optional[list] = None
    kv_lens: Optional[list] = None
    kv_dtype: int = SPARSE_KV_BF16   # packed FP8: uint8 pools [nb, bs, 1, 640]

    @property
    def rows(self) -> int:
        return self.T1 if self.layout == LAYOUT_TND else self.B * self.S1

    def to(self, device) -> "SparseProblem":
        kw = {}
        for f in dataclasses.fields(self):
            v = getattr(self, f.name)
            kw[f.name] = v.to(device) if isinstance(v, torch.Tensor) else v
        return SparseProblem(**kw)


# ----------------------------------------------------------------------------
# helpers
# ----------------------------------------------------------------------------

def _normal_bf16(shape, gen, device) -> torch.Tensor:
    return torch.randn(shape, generator=gen, device=device, dtype=torch.float32).to(torch.bfloat16)


def _dev_gen(device, seed):
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def quantize_e4m3_per_tile(x: torch.Tensor, tile: int = FP8_TILE):
    """Pack a bf16 KV tensor [..., D] as FP8 E4M3 codes plus one fp32 scale per
    `tile` consecutive elements of D: scale = amax(|x_tile|) / 448 (1 when the
    tile is all zero), code = RNE(x / scale) saturated to +-448, computed in
    fp32 from the bf16 source.  Returns (codes uint8 [..., D], scales fp32
    [..., D/tile])."""
    shp = x.shape
    D = shp[-1]
    xt = x.float().reshape(*shp[:-1], D // tile, tile)
    amax = xt.abs().amax(dim=-1)
    scale = torch.where(amax > 0, amax / FP8_MAX, torch.ones_like(amax))
    y = (xt / scale.unsqueeze(-1)).clamp_(-FP8_MAX, FP8_MAX)
    codes = y.to(torch.float8_e4m3fn).view(torch.uint8).reshape(shp)
    return codes.contiguous(), scale.contiguous()


def pack_fp8_sparse_rows(x: torch.Tensor) -> torch.Tensor:
    """Pack bf16 K~ rows [..., 512] into the 640-byte shared-KV rows of the
    kv_quant_sparse_attn_sharedkv format: the first 64 values (rope) kept as
    bf16 (128 bytes), the other 448 (nope) as E4M3 codes (448 bytes) with one
    E8M0 scale per 64 of them (7 bytes: 2^(e - 127)), zero padding after.
    The scale of a tile is the smallest power of two s with amax / s <= 448
    (1 for an all-zero tile); codes are RNE(x / s) in fp32 from the bf16
    source.  This is the cache-write side of the format."""
    shp = x.shape
    assert shp[-1] == 512
    xf = x.float().reshape(-1, 512)
    rows = xf.shape[0]
    out = torch.zeros((rows, 640), dtype=torch.uint8, device=x.device)
    out[:, :128] = x.reshape(-1, 512)[:, :64].contiguous().view(torch.uint8).reshape(rows, 128)
    nope = xf[:, 64:].reshape(rows, 7, 64)
    amax = nope.abs().amax(dim=-1)
    e = torch.where(amax > 0, torch.ceil(torch.log2(amax / FP8_MAX)), torch.zeros_like(amax))
    # log2 may round: make sure amax / 2^e <= 448 and amax / 2^(e-1) > 448
    e = torch.where((amax > 0) & (amax / torch.exp2(e) > FP8_MAX), e + 1, e)
    e = torch.where((amax > 0) & (amax / torch.exp2(e - 1) <= FP8_MAX), e - 1, e)
    e = e.clamp(-127, 127)
    y = (nope / torch.exp2(e).unsqueeze(-1)).clamp(-FP8_MAX, FP8_MAX)
    out[:, 128:576] = y.to(torch.float8_e4m3fn).view(torch.uint8).reshape(rows, 448)
    out[:, 576:583] = (e + 127).to(torch.uint8)
    return out.reshape(*shp[:-1], 640)


def scales_head_major(scales: torch.Tensor) -> torch.Tensor:
    """Reorder per-row scales [pages, rows, KVN, D/64] (the shape the quantiser
    returns for a pool [pages, rows, KVN, D]) to the stored layout
    [pages, KVN, rows, D/64]: inside a page the scales of one KV head are
    contiguous, as the page-managed per-token, per-head scale shape
    (blockNum, N, blockSize) of the FIA dequantisation parameter group."""
    return scales.permute(0, 2, 1, 3).contiguous()


def _paged_layout(kv_lens, block_size, gen_cpu, max_blocks=None):
    """Block table for the given KV lengths over a randomly permuted pool
    with N_SPARE_BLOCKS poisoned spare blocks.  Returns (table int32
    [B,max_blocks], num_blocks, list of (b, j0, phys_block) for used
    blocks)."""
    B = len(kv_lens)
    nblk = [math.ceil(l / block_size) for l in kv_lens]
    used = sum(nblk)
    num_blocks = used + N_SPARE_BLOCKS
    perm = torch.randperm(num_blocks, generator=gen_cpu).tolist()
    mb = max(max(nblk) if nblk else 0, 1) if max_blocks is None else max_blocks
    spare = perm[used:]
    table = torch.empty((B, mb), dtype=torch.int32)
    table[:] = spare[0]
    k = 0
    placed = []
    for b in range(B):
        for j in range(nblk[b]):
            table[b, j] = perm[k]
            placed.append((b, j, perm[k]))
            k += 1
    return table, num_blocks, placed


def _valid_row_mask(kv_lens, block_size, placed, num_blocks):
    valid = torch.zeros(num_blocks * block_size, dtype=torch.bool)
    for (b, j, pb) in placed:
        n = min(block_size, kv_lens[b] - j * block_size)
        valid[pb * block_size: pb * block_size + n] = True
    return valid


# ----------------------------------------------------------------------------
# general generators
# ----------------------------------------------------------------------------

def make_fia(*, B, QN, KVN, D, q_lens, kv_lens, layout=LAYOUT_BSND, paged=True,
             block_size=128, kv_dtype=KV_BF16, mask_mode=MASK_NONE, pre_tokens=0,
             next_tokens=0, with_sinks=False, scale=None, seed=0, device="cpu",
             poison=True, max_blocks=None, S_kv=None, q_mult=None, kv_layout=KV_LAYOUT_BNBSH,
             mask_density=None, mask_shared=False, mask_full_rows=0) -> FiaProblem:
    """Build one FIA problem.  `q_lens`/`kv_lens` are host lists of length B
    (for BSND all q_lens must be equal).  `paged=False` gives a contiguous
    BSND KV cache [B, S_kv, KVN, D].  `q_mult` (a power of two, or one per
    query head) multiplies Q after it is drawn and rounded: powers of two
    scale bf16 exactly, so the draws and every other tensor stay the same.
    `kv_layout=KV_LAYOUT_BNNBSD` stores paged pools as [nb, KVN, bs, D].
    `mask_density` (modes 0/1) adds an explicit uint8 mask [B (or 1 with
    `mask_shared`), max query length, KV capacity rounded up to 16] with that
    fraction of ones (hidden keys), drawn after everything else from the CPU
    generator; `mask_full_rows` of its rows (row i of batch 0, i = 0, 1, ...)
    are then hidden entirely."""
    gen_cpu = torch.Generator().manual_seed(seed)
    gdev = _dev_gen(device, seed + 1)
    q_lens = [int(x) for x in q_lens]
    kv_lens = [int(x) for x in kv_lens]
    if layout == LAYOUT_BSND:
        assert len(set(q_lens)) <= 1
        S_q = q_lens[0] if q_lens else 0
        T = B * S_q
        q = _normal_bf16((B, S_q, QN, D), gdev, device)
        cu = None
    else:
        T = sum(q_lens)
        S_q = max(q_lens) if q_lens else 0
        q = _normal_bf16((T, QN, D), gdev, device)
        cu = torch.tensor([0] + list(torch.tensor(q_lens).cumsum(0).tolist()), dtype=torch.int32)
    if q_mult is not None:
        m = torch.tensor(q_mult if isinstance(q_mult, (list, tuple)) else [q_mult] * QN,
                         dtype=torch.float32, device=device)
        for x in m.tolist():
            assert x > 0 and math.frexp(x)[0] == 0.5, "q_mult must be a power of two"
        q = (q.float() * m.view(QN, 1)).to(torch.bfloat16)
    if paged:
        table, nb, placed = _paged_layout(kv_lens, block_size, gen_cpu, max_blocks)
        rows = nb * block_size
        k_src = _normal_bf16((nb, block_size, KVN, D), gdev, device)
        v_src = _normal_bf16((nb, block_size, KVN, D), gdev, device)
        valid = _valid_row_mask(kv_lens, block_size, placed, nb).to(device)
        skv = table.shape[1] * block_size
        seqused = torch.tensor(kv_lens, dtype=torch.int32)
    else:
        skv = S_kv if S_kv is not None else max(kv_lens)
        table, nb = None, 0
        rows = B * skv
        k_src = _normal_bf16((B, skv, KVN, D), gdev, device)
        v_src = _normal_bf16((B, skv, KVN, D), gdev, device)
        valid = torch.zeros((B, skv), dtype=torch.bool)
        for b in range(B):
            valid[b, :kv_lens[b]] = True
        valid = valid.reshape(-1).to(device)
        seqused = torch.tensor(kv_lens, dtype=torch.int32)
    sinks = torch.randn((QN,), generator=gen_cpu, dtype=torch.float32) if with_sinks else None
    if kv_dtype == KV_FP8_E4M3:
        kc, ks = quantize_e4m3_per_tile(k_src)
        vc, vs = quantize_e4m3_per_tile(v_src)
        del k_src, v_src
        if poison:
            inv = ~valid
            kc.view(rows, -1)[inv] = 0x7F
            vc.view(rows, -1)[inv] = 0x7F
            ks.view(rows, -1)[inv] = float("nan")
            vs.view(rows, -1)[inv] = float("nan")
        k_cache, v_cache = kc, vc
        k_scale, v_scale = scales_head_major(ks), scales_head_major(vs)
    else:
        if poison:
            inv = ~valid
            k_src.view(rows, -1)[inv] = float("nan")
            v_src.view(rows, -1)[inv] = float("nan")
        k_cache, v_cache, k_scale, v_scale = k_src, v_src, None, None
    if kv_layout == KV_LAYOUT_BNNBSD:
        assert paged, "head-major pages need a paged cache"
        k_cache = k_cache.permute(0, 2, 1, 3).contiguous()
        v_cache = v_cache.permute(0, 2, 1, 3).contiguous()
    atten_mask = None
    if mask_density is not None:
        cap = skv
        cols = (cap + 15) // 16 * 16
        mrows = max(max(q_lens) if q_lens else 0, 1)
        mb = 1 if mask_shared else B
        atten_mask = (torch.rand((mb, mrows, cols), generator=gen_cpu) < mask_density).to(
            torch.uint8)
        for i in range(min(mask_full_rows, mrows)):
            atten_mask[0, i, :] = 1
        atten_mask = atten_mask.to(device)
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    return FiaProblem(B=B, QN=QN, KVN=KVN, D=D, layout=layout, S_q=S_q, T=T, q=q,
                      cu_seqlens_q=None if cu is None else cu.to(device), kv_dtype=kv_dtype,
                      k_cache=k_cache, v_cache=v_cache, k_scale=k_scale, v_scale=v_scale,
                      block_table=None if table is None else table.to(device),
                      block_size=block_size if paged else 0, num_blocks=nb, S_kv=skv,
                      seqused_kv=seqused.to(device), scale=float(scale), mask_mode=mask_mode,
                      pre_tokens=pre_tokens, next_tokens=next_tokens,
                      sinks=None if sinks is None else sinks.to(device),
                      q_lens=q_lens, kv_lens=kv_lens, kv_layout=kv_layout,
                      atten_mask=atten_mask)


def make_sparse(*, B, N1, D, q_lens, kv_lens, layout=LAYOUT_BSND, mode="csa", K2=512,
                cmp_ratio=4, ori_block_size=128, cmp_block_size=128, win_left=127, win_right=0,
                with_sinks=True, scale=None, seed=0, device="cpu", poison=True,
                distinct=True, kv_dtype=SPARSE_KV_BF16) -> SparseProblem:
    """Build one shared-KV sparse attention problem.  mode: 'swa' (ori only),
    'csa' (ori window + top-K indexed compressed rows) or 'hca' (ori window +
    every causally visible compressed row)."""
    gen_cpu = torch.Generator().manual_seed(seed)
    gdev = _dev_gen(device, seed + 1)
    q_lens = [int(x) for x in q_lens]
    kv_lens = [int(x) for x in kv_lens]
    if layout == LAYOUT_BSND:
        assert len(set(q_lens)) <= 1
        S1 = q_lens[0]
        T1 = B * S1
        q = _normal_bf16((B, S1, N1, D), gdev, device)
        cu = None
    else:
        T1 = sum(q_lens)
        S1 = max(q_lens)
        q = _normal_bf16((T1, N1, D), gdev, device)
        cu = torch.tensor([0] + list(torch.tensor(q_lens).cumsum(0).tolist()), dtype=torch.int32)
    def _store(src, valid):
        # bf16 rows poisoned with NaN, or packed FP8 rows poisoned with NaN
        # rope values, NaN codes (0x7F) and NaN scales (0xFF)
        if kv_dtype == SPARSE_KV_BF16:
            if valid is not None:
                src.view(-1, D)[~valid] = float("nan")
            return src
        packed = pack_fp8_sparse_rows(src)
        if valid is not None:
            flat = packed.view(-1, 640)
            bad = ~valid
            flat[bad, 0:128] = torch.tensor([0xC0, 0x7F], dtype=torch.uint8,
                                            device=packed.device).repeat(64)
            flat[bad, 128:576] = 0x7F
            flat[bad, 576:583] = 0xFF
        return packed

    o_table, o_nb, o_placed = _paged_layout(kv_lens, ori_block_size, gen_cpu)
    ori = _normal_bf16((o_nb, ori_block_size, 1, D), gdev, device)
    ov = _valid_row_mask(kv_lens, ori_block_size, o_placed, o_nb).to(device) if poison else None
    ori = _store(ori, ov)
    cmp_kv = c_table = idx = None
    if mode in ("csa", "hca"):
        cmp_lens = [l // cmp_ratio for l in kv_lens]
        c_table, c_nb, c_placed = _paged_layout([max(c, 0) for c in cmp_lens], cmp_block_size,
                                                gen_cpu)
        cmp_kv = _normal_bf16((c_nb, cmp_block_size, 1, D), gdev, device)
        cv = (_valid_row_mask(cmp_lens, cmp_block_size, c_placed, c_nb).to(device)
              if poison else None)
        cmp_kv = _store(cmp_kv, cv)
    sinks = torch.randn((N1,), generator=gen_cpu, dtype=torch.float32) if with_sinks else None
    if mode == "csa":
        rows = T1
        idx = torch.full((rows, 1, K2), -1, dtype=torch.int32)
        r = 0
        for b in range(B):
            for i in range(q_lens[b]):
                p = kv_lens[b] - q_lens[b] + i
                nvis = max(0, (p + 1) // cmp_ratio)
                if distinct:
                    sel = torch.randperm(nvis, generator=gen_cpu)[:K2] if nvis > 0 else \
                        torch.empty(0, dtype=torch.int64)
                else:
                    sel = torch.randint(0, max(nvis, 1), (min(K2, nvis),), generator=gen_cpu)
                idx[r, 0, :sel.numel()] = sel.to(torch.int32)
                r += 1
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    return SparseProblem(B=B, N1=N1, D=D, layout=layout, S1=S1, T1=T1, q=q,
                         cu_seqlens_q=None if cu is None else cu.to(device),
                         ori_kv=ori, ori_block_table=o_table.to(device),
                         ori_block_size=ori_block_size,
                         cmp_kv=cmp_kv,
                         cmp_block_table=None if c_table is None else c_table.to(device),
                         cmp_block_size=cmp_block_size,
                         cmp_sparse_indices=None if idx is None else idx.to(device),
                         K2=K2 if mode == "csa" else 0,
                         seqused_kv=torch.tensor(kv_lens, dtype=torch.int32).to(device),
                         sinks=None if sinks is None else sinks.to(device), scale=float(scale),
                         cmp_ratio=cmp_ratio, win_left=win_left, win_right=win_right,
                         q_lens=q_lens, kv_lens=kv_lens, kv_dtype=kv_dtype)


# ----------------------------------------------------------------------------
# the five workloads (seed 1000 + k)
# ----------------------------------------------------------------------------

def _lens(gen, n, lo, hi):
    return torch.randint(lo, hi + 1, (n,), generator=gen).tolist()


def workload_tiny_prefill(device="cpu") -> FiaProblem:
    """B=1, Q_N=KV_N=4, D=64, S_q=S_kv=128, BSND contiguous, scale 1/8,
    right-down causal, bf16 out + fp32 lse."""
    return make_fia(B=1, QN=4, KVN=4, D=64, q_lens=[128], kv_lens=[128], layout=LAYOUT_BSND,
                    paged=False, mask_mode=MASK_RIGHT_DOWN_CAUSAL, scale=1.0 / 8.0, seed=1001,
                    device=device)


def workload_paged_decode(device="cpu", B=32, S_q=1, kv_layout=KV_LAYOUT_BNBSH) -> FiaProblem:
    """B=32, S_q=1, Q_N=32, KV_N=8, D=128, kv len ~ U[512,4096], block 128,
    permuted pages, scale 1/sqrt(128).  S_q > 1 gives the same sequences with
    S_q query rows each (multi-token decode, right-down causal);
    kv_layout=KV_LAYOUT_BNNBSD stores the pages head-major."""
    g = torch.Generator().manual_seed(1002)
    kv = _lens(g, B, 512, 4096)
    return make_fia(B=B, QN=32, KVN=8, D=128, q_lens=[S_q] * B, kv_lens=kv, layout=LAYOUT_BSND,
                    paged=True, block_size=128, seed=1002, device=device,
                    mask_mode=MASK_RIGHT_DOWN_CAUSAL if S_q > 1 else MASK_NONE,
                    kv_layout=kv_layout)


def workload_varlen_prefill(device="cpu", B=8, kv_dtype=KV_BF16) -> FiaProblem:
    """TND, B=8, lengths ~ U[256,4096], Q_N=32, KV_N=8, D=128, paged block 128,
    kv_len = q_len, right-down causal, per-head fp32 sinks (kv_dtype
    KV_FP8_E4M3: the same sequences with an FP8 cache)."""
    g = torch.Generator().manual_seed(1003)
    L = _lens(g, B, 256, 4096)
    return make_fia(B=B, QN=32, KVN=8, D=128, q_lens=L, kv_lens=L, layout=LAYOUT_TND, paged=True,
                    block_size=128, mask_mode=MASK_RIGHT_DOWN_CAUSAL, with_sinks=True, seed=1003,
                    device=device, kv_dtype=kv_dtype)


def workload_fp8_long_decode(device="cpu", B=4, lo=32768, hi=131072, QN=64, KVN=8) -> FiaProblem:
    """B=4, S_q=1, Q_N=64, KV_N=8, D=128, kv len ~ U[32768,131072], E4M3 KV
    with fp32 per-64 scales, block 128 (KVN=4: the same sequences with 16
    query heads per KV head)."""
    g = torch.Generator().manual_seed(1004)
    kv = _lens(g, B, lo, hi)
    return make_fia(B=B, QN=QN, KVN=KVN, D=128, q_lens=[1] * B, kv_lens=kv, layout=LAYOUT_BSND,
                    paged=True, block_size=128, kv_dtype=KV_FP8_E4M3, seed=1004, device=device)


def workload_sparse_csa(device="cpu", B=16, kv_dtype=SPARSE_KV_BF16) -> SparseProblem:
    """B=16, S_q=1, N1=64, KV_N=1, D=512; ori len 8192, band 127/0; cmp 2048
    rows (ratio 4); top-512 distinct visible indices; fp32 sinks; block 128
    (kv_dtype SPARSE_KV_FP8_PACKED: the same rows in the packed FP8 format)."""
    return make_sparse(B=B, N1=64, D=512, q_lens=[1] * B, kv_lens=[8192] * B,
                       layout=LAYOUT_BSND, mode="csa", K2=512, cmp_ratio=4, seed=1005,
                       device=device, kv_dtype=kv_dtype)
