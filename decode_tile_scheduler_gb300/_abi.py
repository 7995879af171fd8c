"""ctypes mirror of include/fia.h and thin wrappers around its entry points.

Argument marshalling only: every step of the attention runs in libfia's CUDA
kernels.  If the library is missing or cannot be loaded the first call raises
RuntimeError -- there is no fallback path.
"""
from __future__ import annotations

import ctypes
import os
import threading

from . import _build

FIA_OK = 0
FIA_ERR_NULL_ARG = 1
FIA_ERR_BAD_SHAPE = 2
FIA_ERR_BAD_DTYPE = 3
FIA_ERR_UNSUPPORTED = 4
FIA_ERR_WORKSPACE_TOO_SMALL = 5
FIA_ERR_CUDA = 6

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
SPARSE_PACKED_ROW_BYTES = 640
COMBINE_MAX_PARTS = 16
ABI_VERSION = 3

_P = ctypes.c_void_p
_I = ctypes.c_int32
_L = ctypes.c_int64


class FiaParams(ctypes.Structure):
    _fields_ = [
        ("batch", _I), ("num_q_heads", _I), ("num_kv_heads", _I), ("head_dim", _I),
        ("layout", _I), ("max_seqlen_q", _I), ("total_q", _I), ("pad0_", _I),
        ("q", _P), ("out", _P), ("lse", _P),
        ("q_token_stride", _L), ("out_token_stride", _L),
        ("k_cache", _P), ("v_cache", _P), ("k_scale", _P), ("v_scale", _P),
        ("kv_dtype", _I), ("quant_tile", _I),
        ("block_table", _P),
        ("max_blocks_per_seq", _I), ("block_size", _I), ("num_blocks", _I),
        ("max_seqlen_kv", _I),
        ("cu_seqlens_q", _P), ("seqused_kv", _P),
        ("scale", ctypes.c_float), ("mask_mode", _I), ("pre_tokens", _I), ("next_tokens", _I),
        ("sinks", _P),
        ("num_sms", _I), ("kv_layout", _I),
        ("atten_mask", _P), ("mask_batch_stride", _L), ("mask_row_stride", _L),
        ("reserved", _I * 8),
    ]


class SparseParams(ctypes.Structure):
    _fields_ = [
        ("batch", _I), ("num_q_heads", _I), ("head_dim", _I), ("layout", _I),
        ("max_seqlen_q", _I), ("total_q", _I),
        ("q", _P), ("out", _P), ("lse", _P),
        ("ori_kv", _P), ("ori_block_table", _P),
        ("ori_max_blocks", _I), ("ori_block_size", _I), ("ori_num_blocks", _I), ("pad0_", _I),
        ("cmp_kv", _P), ("cmp_block_table", _P),
        ("cmp_max_blocks", _I), ("cmp_block_size", _I), ("cmp_num_blocks", _I), ("topk", _I),
        ("cmp_sparse_indices", _P), ("cu_seqlens_q", _P), ("seqused_kv", _P), ("sinks", _P),
        ("softmax_scale", ctypes.c_float), ("cmp_ratio", _I), ("ori_win_left", _I),
        ("ori_win_right", _I), ("num_sms", _I), ("kv_dtype", _I), ("tile_size", _I),
        ("rope_head_dim", _I), ("reserved", _I * 8),
    ]


class CombineParams(ctypes.Structure):
    _fields_ = [
        ("n_parts", _I), ("layout", _I), ("batch", _I), ("seqlen_q", _I), ("total_q", _I),
        ("num_heads", _I), ("head_dim", _I), ("pad0_", _I),
        ("o_parts", ctypes.POINTER(_P)), ("lse_parts", ctypes.POINTER(_P)),
        ("out", _P), ("lse", _P), ("sinks", _P), ("reserved", _I * 8),
    ]


class FiaPlanLayout(ctypes.Structure):
    _fields_ = [
        ("branch", _I), ("num_ctas", _I), ("num_units", _L), ("max_chunks", _L),
        ("sched_off", _L), ("queue_off", _L), ("unit_list_off", _L), ("total_bytes", _L),
    ]


# every symbol include/fia.h declares
EXPORTS = (
    "fia_status_string", "fia_abi_version", "fia_sizeof_params", "fia_sizeof_sparse_params",
    "fia_sizeof_combine_params",
    "fia_get_workspace_size", "fia_plan", "fia_execute", "fia_run", "fia_get_plan_layout",
    "sparse_attn_metadata", "sparse_attn_run", "fia_decode_run_noalloc",
    "fia_selftest_bounded_wait", "fia_lse_combine",
)
NOALLOC_SCRATCH_BYTES = 8 << 20


class FiaError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {status_string(status)} ({status})")


_lock = threading.Lock()
_lib = None


def lib_path() -> str:
    return _build.LIB


def lib(build_if_missing: bool = True) -> ctypes.CDLL:
    """Load libfia.so (building it first when absent and nvcc is available)."""
    global _lib
    with _lock:
        if _lib is None:
            path = _build.LIB
            if not os.path.exists(path):
                if not build_if_missing:
                    raise RuntimeError(f"libfia.so not built at {path}")
                _build.build()
            try:
                L = ctypes.CDLL(path)
            except OSError as e:
                raise RuntimeError(f"cannot load {path}: {e}") from e
            L.fia_status_string.restype = ctypes.c_char_p
            L.fia_status_string.argtypes = [ctypes.c_int]
            L.fia_abi_version.restype = _I
            L.fia_sizeof_params.restype = ctypes.c_size_t
            L.fia_sizeof_sparse_params.restype = ctypes.c_size_t
            L.fia_sizeof_combine_params.restype = ctypes.c_size_t
            L.fia_get_workspace_size.argtypes = [ctypes.POINTER(FiaParams),
                                                 ctypes.POINTER(ctypes.c_size_t)]
            L.fia_get_plan_layout.argtypes = [ctypes.POINTER(FiaParams),
                                              ctypes.POINTER(FiaPlanLayout)]
            for f in ("fia_plan", "fia_execute", "fia_run"):
                getattr(L, f).argtypes = [ctypes.POINTER(FiaParams), _P, ctypes.c_size_t, _P]
            L.sparse_attn_metadata.argtypes = [ctypes.POINTER(SparseParams), _P,
                                               ctypes.POINTER(ctypes.c_size_t), _P]
            L.sparse_attn_run.argtypes = [ctypes.POINTER(SparseParams), _P, _P, ctypes.c_size_t,
                                          _P]
            L.fia_decode_run_noalloc.argtypes = [ctypes.POINTER(FiaParams), _P, _P]
            L.fia_lse_combine.argtypes = [ctypes.POINTER(CombineParams), _P]
            L.fia_selftest_bounded_wait.argtypes = [_P, ctypes.c_uint64, _P]
            for f in EXPORTS:
                if f not in ("fia_status_string", "fia_abi_version", "fia_sizeof_params",
                             "fia_sizeof_sparse_params", "fia_sizeof_combine_params"):
                    getattr(L, f).restype = ctypes.c_int
            if L.fia_abi_version() != ABI_VERSION:
                raise RuntimeError("libfia ABI version differs from the binding's")
            if L.fia_sizeof_params() != ctypes.sizeof(FiaParams):
                raise RuntimeError("fia_params layout mismatch between fia.h and the binding")
            if L.fia_sizeof_sparse_params() != ctypes.sizeof(SparseParams):
                raise RuntimeError("sparse_attn_params layout mismatch")
            if L.fia_sizeof_combine_params() != ctypes.sizeof(CombineParams):
                raise RuntimeError("fia_combine_params layout mismatch")
            _lib = L
    return _lib


def status_string(s: int) -> str:
    return lib().fia_status_string(s).decode()


def _check(status: int, where: str):
    if status != FIA_OK:
        raise FiaError(status, where)


def fia_get_workspace_size(p: FiaParams) -> int:
    n = ctypes.c_size_t(0)
    _check(lib().fia_get_workspace_size(ctypes.byref(p), ctypes.byref(n)),
           "fia_get_workspace_size")
    return n.value


def fia_get_plan_layout(p: FiaParams) -> FiaPlanLayout:
    out = FiaPlanLayout()
    _check(lib().fia_get_plan_layout(ctypes.byref(p), ctypes.byref(out)), "fia_get_plan_layout")
    return out


def fia_plan(p: FiaParams, ws: int, nbytes: int, stream: int = 0):
    _check(lib().fia_plan(ctypes.byref(p), ws, nbytes, stream), "fia_plan")


def fia_execute(p: FiaParams, ws: int, nbytes: int, stream: int = 0):
    _check(lib().fia_execute(ctypes.byref(p), ws, nbytes, stream), "fia_execute")


def fia_run(p: FiaParams, ws: int, nbytes: int, stream: int = 0):
    _check(lib().fia_run(ctypes.byref(p), ws, nbytes, stream), "fia_run")


def fia_decode_run_noalloc(p: FiaParams, status: int = 0, stream: int = 0):
    """`status`: device address of an int32 that receives the run's error word
    (0 = clean), or 0 for none."""
    _check(lib().fia_decode_run_noalloc(ctypes.byref(p), status or None, stream),
           "fia_decode_run_noalloc")


def fia_lse_combine(p: CombineParams, stream: int = 0):
    _check(lib().fia_lse_combine(ctypes.byref(p), stream), "fia_lse_combine")


def sparse_attn_metadata(p: SparseParams, metadata: int, stream: int = 0) -> int:
    n = ctypes.c_size_t(0)
    _check(lib().sparse_attn_metadata(ctypes.byref(p), metadata, ctypes.byref(n), stream),
           "sparse_attn_metadata")
    return n.value


def selftest_bounded_wait(status: int, limit_ns: int, stream: int = 0):
    _check(lib().fia_selftest_bounded_wait(status, limit_ns, stream), "fia_selftest_bounded_wait")


def sparse_attn_run(p: SparseParams, metadata: int, ws: int, nbytes: int, stream: int = 0):
    _check(lib().sparse_attn_run(ctypes.byref(p), metadata, ws, nbytes, stream),
           "sparse_attn_run")
