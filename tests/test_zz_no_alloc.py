"""fia_decode_run_noalloc: the decode call that needs no workspace.

For callers that cannot allocate device memory when they run attention (the
device belongs to another component's pool, or allocation is forbidden after
start-up), the library keeps the decode scratch in a fixed device array of
FIA_NOALLOC_SCRATCH_BYTES.  This file is collected last on purpose.  The test
calls the entry point through the C ABI twice in a row, on two different
batches, and checks each result against fia_run with a caller-provided
workspace: the same plan and the same kernels run on both, so the outputs
must agree bit for bit.  It also checks the error word the call hands back,
that an oversized plan is refused before anything is launched, and that the
prefill branch is refused while an empty query is accepted.
"""
import ctypes

import pytest
import torch

import fia_inputs as fi

pytestmark = pytest.mark.gpu


def _noalloc(p):
    import decode_tile_scheduler_gb300 as fia
    out = torch.full_like(p.q, float("nan"))
    lse = torch.full(fia.lse_shape(p), float("nan"), dtype=torch.float32, device=p.q.device)
    status = torch.full((1,), -7, dtype=torch.int32, device=p.q.device)
    params = fia.params_from_problem(p, out, lse)
    st = fia.lib().fia_decode_run_noalloc(ctypes.byref(params), ctypes.c_void_p(status.data_ptr()),
                                          ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    torch.cuda.synchronize()
    return st, out, lse, int(status.item())


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
        st, out, lse, word = _noalloc(p)
        assert st == fia.FIA_OK, fia.status_string(st)
        assert word == 0
        ref_out, ref_lse = _with_workspace(p)
        assert torch.equal(out, ref_out)
        assert torch.equal(lse, ref_lse)


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
    st = fia.lib().fia_decode_run_noalloc(ctypes.byref(params), None, None)
    assert st == fia.FIA_ERR_WORKSPACE_TOO_SMALL
    torch.cuda.synchronize()
    assert torch.count_nonzero(out) == 0


def test_noalloc_refuses_prefill_and_accepts_an_empty_query():
    import decode_tile_scheduler_gb300 as fia
    p = fi.make_fia(B=2, QN=8, KVN=2, D=128, q_lens=[40, 40], kv_lens=[40, 60], block_size=16,
                    mask_mode=3, seed=74, device="cuda")
    out = torch.zeros_like(p.q)
    params = fia.params_from_problem(p, out, None)
    st = fia.lib().fia_decode_run_noalloc(ctypes.byref(params), None, None)
    assert st == fia.FIA_ERR_UNSUPPORTED
    torch.cuda.synchronize()
    assert torch.count_nonzero(out) == 0
    # no query row at all: nothing runs, the call succeeds and reports 0
    e = fi.make_fia(B=2, QN=8, KVN=2, D=128, q_lens=[0, 0], kv_lens=[40, 60], block_size=16,
                    layout=fi.LAYOUT_TND, seed=75, device="cuda")
    out = torch.zeros(16, dtype=torch.bfloat16, device="cuda")
    status = torch.full((1,), -7, dtype=torch.int32, device="cuda")
    params = fia.params_from_problem(e, out, None)
    # an empty tensor may have no address; any valid one will do, as no
    # query row is read or written
    params.q, params.out = out.data_ptr(), out.data_ptr()
    params.max_seqlen_q = 1
    st = fia.lib().fia_decode_run_noalloc(ctypes.byref(params), ctypes.c_void_p(status.data_ptr()),
                                          None)
    torch.cuda.synchronize()
    assert st == fia.FIA_OK and int(status.item()) == 0
