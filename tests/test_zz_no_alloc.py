"""fia_decode_run_noalloc: the decode call that needs no workspace.

For callers that cannot allocate device memory when they run attention (the
device belongs to another component's pool, or allocation is forbidden after
start-up), the library keeps the decode scratch in a fixed device array of
FIA_NOALLOC_SCRATCH_BYTES.  This file is collected last on purpose.  The test
calls the entry point through the C ABI twice in a row, on two different
batches, and checks each result against fia_run with a caller-provided
workspace, within the tolerances of the other parity tests; it also checks
that an oversized plan is refused before anything is launched.
"""
import ctypes

import numpy as np
import pytest
import torch

import fia_inputs as fi
from helpers import as_np

pytestmark = pytest.mark.gpu


def _noalloc(p):
    import decode_tile_scheduler_gb300 as fia
    out = torch.full_like(p.q, float("nan"))
    lse = torch.full(fia.lse_shape(p), float("nan"), dtype=torch.float32, device=p.q.device)
    params = fia.params_from_problem(p, out, lse)
    st = fia.lib().fia_decode_run_noalloc(ctypes.byref(params),
                                          torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    return st, out, lse


def _with_workspace(p):
    import decode_tile_scheduler_gb300 as fia
    out, lse = fia.FiaCall(p, with_lse=True).run()
    torch.cuda.synchronize()
    return out, lse


def test_noalloc_matches_fia_run_on_two_calls_in_a_row():
    import decode_tile_scheduler_gb300 as fia
    first = fi.make_fia(B=8, QN=32, KVN=8, D=128, q_lens=[1] * 8,
                        kv_lens=[4096, 512, 1, 2000, 777, 3000, 129, 64], block_size=128,
                        with_sinks=True, seed=71, device="cuda")
    second = fi.make_fia(B=3, QN=16, KVN=2, D=128, q_lens=[1] * 3, kv_lens=[5000, 0, 300],
                         block_size=64, seed=72, device="cuda")
    for p in (first, second):
        st, out, lse = _noalloc(p)
        assert st == fia.FIA_OK, fia.status_string(st)
        ref_out, ref_lse = _with_workspace(p)
        o, r = as_np(out), as_np(ref_out)
        err = abs(o - r)
        assert err.max() <= 2e-2 and err.mean() <= 2e-3
        l, rl = as_np(lse), as_np(ref_lse)
        fin = np.isfinite(rl)
        assert np.array_equal(fin, np.isfinite(l))
        assert np.array_equal(l[~fin], rl[~fin])
        assert (np.abs(l[fin] - rl[fin]) <= 1e-3).all()


def test_noalloc_refuses_a_plan_larger_than_the_scratch():
    import decode_tile_scheduler_gb300 as fia
    from decode_tile_scheduler_gb300._abi import NOALLOC_SCRATCH_BYTES
    p = fi.make_fia(B=2, QN=8, KVN=2, D=128, q_lens=[1, 1], kv_lens=[10, 20], block_size=16,
                    seed=73, device="cuda")
    out = torch.zeros_like(p.q)
    params = fia.params_from_problem(p, out, None)
    # 65536 batches x 64 KV heads: a plan far beyond the fixed scratch.  The
    # call must refuse it on the host, before any launch (the tensors are only
    # sized for the small problem, so nothing may run).
    params.batch, params.num_q_heads, params.num_kv_heads = 65536, 256, 64
    need = ctypes.c_size_t(0)
    assert fia.lib().fia_get_workspace_size(ctypes.byref(params), ctypes.byref(need)) == 0
    assert need.value > NOALLOC_SCRATCH_BYTES
    st = fia.lib().fia_decode_run_noalloc(ctypes.byref(params), None)
    assert st == fia.FIA_ERR_WORKSPACE_TOO_SMALL
    torch.cuda.synchronize()
    assert torch.count_nonzero(out) == 0
