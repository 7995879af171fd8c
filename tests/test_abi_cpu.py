"""CPU checks of the C ABI: the library loads, exports every function that
include/fia.h declares, agrees with the binding on struct layouts, and its
first phase rejects invalid parameters with the documented status codes
(no device pointer is dereferenced and no GPU is needed)."""
import ctypes
import os
import re

import pytest

import decode_tile_scheduler_gb300 as fia
from decode_tile_scheduler_gb300 import _abi

HDR = os.path.join(os.path.dirname(os.path.dirname(__file__)), "include", "fia.h")


def _declared_functions():
    src = open(HDR).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[a-z_0-9]+\s*\*?\s*([a-z_0-9]+)\s*\(", src, flags=re.M)
    return sorted(set(n for n in names if n not in ("if", "while")))


def test_header_declares_the_binding_exports():
    assert set(_declared_functions()) == set(_abi.EXPORTS)


def test_library_exports_every_declared_symbol():
    L = fia.lib()
    for name in _declared_functions():
        assert hasattr(L, name), name


def test_struct_layouts_agree():
    L = fia.lib()
    assert L.fia_sizeof_params() == ctypes.sizeof(_abi.FiaParams)
    assert L.fia_sizeof_sparse_params() == ctypes.sizeof(_abi.SparseParams)
    assert L.fia_sizeof_combine_params() == ctypes.sizeof(_abi.CombineParams)
    assert L.fia_abi_version() == 3


def test_status_strings():
    assert fia.status_string(0) == "FIA_OK"
    assert fia.status_string(5) == "FIA_ERR_WORKSPACE_TOO_SMALL"
    assert fia.status_string(99) == "FIA_ERR_UNKNOWN"


FAKE = 0x10000  # aligned, never dereferenced by the first phase


def _decode_params(**kw):
    p = _abi.FiaParams()
    p.batch, p.num_q_heads, p.num_kv_heads, p.head_dim = 4, 8, 2, 128
    p.layout, p.max_seqlen_q = fia.LAYOUT_BSND, 1
    p.q = p.out = p.k_cache = p.v_cache = FAKE
    p.block_table = p.seqused_kv = FAKE
    p.max_blocks_per_seq, p.block_size, p.num_blocks = 8, 128, 40
    p.scale = 0.088
    p.num_sms = 152
    for k, v in kw.items():
        setattr(p, k, v)
    return p


def _status(p):
    n = ctypes.c_size_t(0)
    return fia.lib().fia_get_workspace_size(ctypes.byref(p), ctypes.byref(n)), n.value


def test_valid_decode_params_size_the_workspace():
    st, n = _status(_decode_params())
    assert st == fia.FIA_OK and n > 0
    # depends on scalar fields only: more CTAs -> more partial slots
    st2, n2 = _status(_decode_params(num_sms=300))
    assert st2 == fia.FIA_OK and n2 > n


@pytest.mark.parametrize("field,value,status", [
    ("q", 0, fia.FIA_ERR_NULL_ARG),
    ("k_cache", 0, fia.FIA_ERR_NULL_ARG),
    ("seqused_kv", 0, fia.FIA_ERR_NULL_ARG),        # required with paging
    ("batch", 0, fia.FIA_ERR_BAD_SHAPE),
    ("batch", 65537, fia.FIA_ERR_BAD_SHAPE),         # B <= 65536
    ("num_q_heads", 257, fia.FIA_ERR_BAD_SHAPE),     # N <= 256
    ("num_q_heads", 7, fia.FIA_ERR_BAD_SHAPE),       # Q_N % KV_N
    ("head_dim", 513, fia.FIA_ERR_BAD_SHAPE),        # D <= 512
    ("head_dim", 96, fia.FIA_ERR_UNSUPPORTED),       # valid, not built
    ("block_size", 24, fia.FIA_ERR_BAD_SHAPE),       # multiple of 16
    ("block_size", 2048, fia.FIA_ERR_BAD_SHAPE),     # <= 1024
    ("kv_dtype", 7, fia.FIA_ERR_BAD_DTYPE),
    ("mask_mode", 5, fia.FIA_ERR_BAD_SHAPE),
    ("mask_mode", -1, fia.FIA_ERR_BAD_SHAPE),
    ("mask_mode", 1, fia.FIA_ERR_NULL_ARG),          # mode 1 needs an explicit mask
    ("kv_layout", 2, fia.FIA_ERR_BAD_SHAPE),
    ("layout", 5, fia.FIA_ERR_BAD_SHAPE),
    ("q", FAKE + 8, fia.FIA_ERR_BAD_SHAPE),          # TMA needs 16-byte alignment
    ("q_token_stride", 1028, fia.FIA_ERR_BAD_SHAPE),  # multiple of 8 elements
])
def test_invalid_params_are_rejected(field, value, status):
    assert _status(_decode_params(**{field: value}))[0] == status


def test_gqa_ratio_limit():
    assert _status(_decode_params(num_q_heads=130, num_kv_heads=2))[0] == fia.FIA_ERR_BAD_SHAPE
    assert _status(_decode_params(num_q_heads=128, num_kv_heads=2))[0] == fia.FIA_OK


def test_band_needs_non_negative_width():
    assert _status(_decode_params(mask_mode=4, pre_tokens=-3, next_tokens=2))[0] == \
        fia.FIA_ERR_BAD_SHAPE
    assert _status(_decode_params(mask_mode=4, pre_tokens=-2, next_tokens=2))[0] == fia.FIA_OK


def test_fp8_needs_scales_and_tile_64():
    assert _status(_decode_params(kv_dtype=1, quant_tile=64))[0] == fia.FIA_ERR_NULL_ARG
    assert _status(_decode_params(kv_dtype=1, quant_tile=32, k_scale=FAKE, v_scale=FAKE))[0] == \
        fia.FIA_ERR_BAD_SHAPE
    assert _status(_decode_params(kv_dtype=1, quant_tile=64, k_scale=FAKE, v_scale=FAKE))[0] == \
        fia.FIA_OK
    # FP8 block size: multiple of 32, <= 512
    assert _status(_decode_params(kv_dtype=1, quant_tile=64, k_scale=FAKE, v_scale=FAKE,
                                  block_size=48))[0] == fia.FIA_ERR_BAD_SHAPE


def test_fp8_scale_alignment_and_contiguous_length():
    fp8 = dict(kv_dtype=1, quant_tile=64, k_scale=FAKE, v_scale=FAKE)
    # scale arrays are copied in 16-byte pieces
    assert _status(_decode_params(**{**fp8, "k_scale": FAKE + 8}))[0] == fia.FIA_ERR_BAD_SHAPE
    assert _status(_decode_params(**{**fp8, "v_scale": FAKE + 8}))[0] == fia.FIA_ERR_BAD_SHAPE
    # a contiguous FP8 cache needs an even max_seqlen_kv
    contig = dict(block_table=None, seqused_kv=None, max_blocks_per_seq=0, num_blocks=0,
                  block_size=0)
    assert _status(_decode_params(**fp8, **contig, max_seqlen_kv=301))[0] == \
        fia.FIA_ERR_BAD_SHAPE
    assert _status(_decode_params(**fp8, **contig, max_seqlen_kv=300))[0] == fia.FIA_OK


def test_tnd_needs_cu_seqlens():
    assert _status(_decode_params(layout=fia.LAYOUT_TND, total_q=4))[0] == fia.FIA_ERR_NULL_ARG
    assert _status(_decode_params(layout=fia.LAYOUT_TND, total_q=4, cu_seqlens_q=FAKE))[0] == \
        fia.FIA_OK


def test_reserved_must_be_zero():
    p = _decode_params()
    p.reserved[3] = 1
    assert _status(p)[0] == fia.FIA_ERR_BAD_SHAPE


def test_workspace_too_small_is_reported_before_launch():
    p = _decode_params()
    st = fia.lib().fia_run(ctypes.byref(p), FAKE, 16, None)
    assert st == fia.FIA_ERR_WORKSPACE_TOO_SMALL
    st = fia.lib().fia_run(ctypes.byref(p), None, 1 << 30, None)
    assert st == fia.FIA_ERR_WORKSPACE_TOO_SMALL


def test_plan_layout_describes_decode_schedule():
    lay = fia.fia_get_plan_layout(_decode_params())
    assert lay.branch == 1 and lay.num_ctas == 152 and lay.num_units == 4 * 2 * 1
    # bf16 with one query row: small chunks of ceil(C/2) tiles, at most 4 per unit
    per_cta = (lay.max_chunks - 4 * lay.num_units) // lay.num_ctas
    assert per_cta >= 1 and lay.max_chunks == 152 * per_cta + 4 * lay.num_units
    assert lay.sched_off >= 256 and lay.queue_off >= lay.sched_off + 8 * (8 + 3 * 5 + 4)
    # partial slots: max_chunks x 8 heads x (D + 2) floats fit in the workspace
    assert lay.total_bytes >= lay.queue_off + 16 * lay.max_chunks + 4 * lay.max_chunks * 8 * 130
    # an FP8 cache takes its units' rest in chunks of C tiles: at most 2 per unit
    lay8 = fia.fia_get_plan_layout(_decode_params(kv_dtype=fia.KV_FP8_E4M3, k_scale=FAKE,
                                                  v_scale=FAKE, quant_tile=64))
    assert lay8.max_chunks == 152 * per_cta + 2 * lay8.num_units


# --------------------------------------------------------------------------
# shared-KV sparse attention: first-phase validation (no GPU: a metadata
# pointer is needed only after validation passes, so invalid calls return
# before anything is launched)
# --------------------------------------------------------------------------

def _sparse_params(**kw):
    p = _abi.SparseParams()
    p.batch, p.num_q_heads, p.head_dim, p.layout = 4, 64, 512, fia.LAYOUT_BSND
    p.max_seqlen_q = 1
    p.q = p.out = p.ori_kv = p.ori_block_table = p.seqused_kv = FAKE
    p.ori_max_blocks, p.ori_block_size, p.ori_num_blocks = 64, 128, 300
    p.cmp_kv = p.cmp_block_table = p.cmp_sparse_indices = FAKE
    p.cmp_max_blocks, p.cmp_block_size, p.cmp_num_blocks, p.topk = 16, 128, 80, 512
    p.softmax_scale = 0.044
    p.cmp_ratio, p.ori_win_left, p.ori_win_right = 4, 127, 0
    p.num_sms = 152
    for k, v in kw.items():
        setattr(p, k, v)
    return p


def _sparse_status(p):
    n = ctypes.c_size_t(0)
    # a fake metadata pointer: validation fails before anything is launched
    return fia.lib().sparse_attn_metadata(ctypes.byref(p), ctypes.c_void_p(FAKE),
                                          ctypes.byref(n), None)


@pytest.mark.parametrize("field,value,status", [
    ("q", 0, fia.FIA_ERR_NULL_ARG),
    ("ori_block_table", 0, fia.FIA_ERR_NULL_ARG),
    ("seqused_kv", 0, fia.FIA_ERR_NULL_ARG),
    ("num_q_heads", 48, fia.FIA_ERR_BAD_SHAPE),      # a power of two
    ("num_q_heads", 256, fia.FIA_ERR_BAD_SHAPE),     # <= 128
    ("head_dim", 640, fia.FIA_ERR_BAD_SHAPE),        # <= 512
    ("head_dim", 192, fia.FIA_ERR_UNSUPPORTED),      # valid, not built
    ("ori_block_size", 40, fia.FIA_ERR_BAD_SHAPE),   # multiple of 16
    ("cmp_block_size", 2048, fia.FIA_ERR_BAD_SHAPE),  # <= 1024
    ("topk", 4096, fia.FIA_ERR_BAD_SHAPE),
    ("cmp_ratio", 0, fia.FIA_ERR_BAD_SHAPE),
    ("ori_win_left", -1, fia.FIA_ERR_BAD_SHAPE),
    ("layout", 1, fia.FIA_ERR_NULL_ARG),             # TND needs cu_seqlens_q
])
def test_sparse_invalid_params_are_rejected(field, value, status):
    assert _sparse_status(_sparse_params(**{field: value})) == status


def test_sparse_indices_need_a_compressed_cache():
    assert _sparse_status(_sparse_params(cmp_kv=0, cmp_block_table=0)) == fia.FIA_ERR_BAD_SHAPE


def test_sparse_metadata_pointer_required():
    p = _sparse_params()
    n = ctypes.c_size_t(0)
    assert fia.lib().sparse_attn_metadata(ctypes.byref(p), None, ctypes.byref(n), None) == \
        fia.FIA_ERR_NULL_ARG


def test_explicit_mask_rules():
    # an explicit mask goes with modes 0 and 1 only
    for mode in (2, 3, 4):
        assert _status(_decode_params(mask_mode=mode, atten_mask=FAKE, mask_row_stride=1024))[0] \
            == fia.FIA_ERR_BAD_SHAPE
    # 16-byte aligned, row stride a multiple of 16 covering the KV capacity
    # (max_blocks_per_seq * block_size = 1024 here)
    assert _status(_decode_params(atten_mask=FAKE + 8, mask_row_stride=1024))[0] == \
        fia.FIA_ERR_BAD_SHAPE
    assert _status(_decode_params(atten_mask=FAKE, mask_row_stride=1000))[0] == \
        fia.FIA_ERR_BAD_SHAPE
    assert _status(_decode_params(atten_mask=FAKE, mask_row_stride=1008))[0] == \
        fia.FIA_ERR_BAD_SHAPE
    assert _status(_decode_params(atten_mask=FAKE, mask_row_stride=1024,
                                  mask_batch_stride=-16))[0] == fia.FIA_ERR_BAD_SHAPE


def test_head_major_pages_need_a_block_table():
    contig = dict(block_table=None, seqused_kv=None, max_blocks_per_seq=0, num_blocks=0,
                  block_size=0, max_seqlen_kv=300)
    assert _status(_decode_params(**contig, kv_layout=1))[0] == fia.FIA_ERR_BAD_SHAPE
