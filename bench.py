"""Benchmark: paged GQA decode (B=32, Q_N=32, KV_N=8, D=128, kv len ~
U[512,4096], block 128, permuted pages) through libfia on one GB300 per rank.

A step is one fia_run (tile scheduler + split-KV decode with its in-kernel
combine) over the whole batch, inputs resident in HBM.  `value` is KV GB/s:
the algorithmic bytes (every visible K and V row once) over the step time.
Between timed steps L2 is flushed: a buffer of twice its size is written, then
another of the same size is read, so no dirty line is written back in a step.

Extra lines of evidence in the same JSON object: the decode kernel's own
roofline (CUDA events around fia_execute on the launching stream), the
end-to-end number through the C ABI with host buffers, the CPU oracle baseline,
SM clocks sampled during the timed region, and the other workloads
(varlen causal prefill, long FP8 decode, sparse shared-KV decode) when built.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl fia|reference]
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

METRIC = "paged-decode KV GB/s and prefill TFLOP/s on 1 GB300, % of roofline"
WORKLOAD = ("paged GQA decode: B=32, S_q=1, Q_N=32, KV_N=8, D=128, bf16, kv len ~ U[512,4096], "
            "block 128, permuted block table")


def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained", d["bf16_tflops"]),
                "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
            "source": "fallback"}


def _src_hash(*names):
    h = hashlib.sha256()
    for n in names:
        with open(os.path.join(ROOT, "decode_tile_scheduler_gb300", "csrc", n), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def _ncu_traffic(kernel_key, src_files, units_now):
    """DRAM bytes per launch from the committed ncu summary, scaled by the
    units processed; None when absent or when the kernel source changed."""
    path = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        d = json.load(f).get(kernel_key)
    if not d or d.get("src_hash") != _src_hash(*src_files):
        return None
    return d["dram_bytes_per_launch"] * units_now / d["units"]


class ClockSampler:
    """nvidia-smi sampling of SM clock and throttle reasons (every 200 ms)."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.tmp = None

    def start(self):
        try:
            self.tmp = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=self.tmp, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
            return
        # Wait (at most 5 s) for the first sample: nvidia-smi's start-up then
        # lies before the timed region, which its samples cover from the
        # first step on, and does not compete with the host's launches
        # inside it.
        t_end = time.time() + 5.0
        while time.time() < t_end and self.proc.poll() is None:
            if os.path.getsize(self.tmp.name) > 0:
                break
            time.sleep(0.01)

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.tmp.flush()
        self.tmp.seek(0)
        rows = [r.strip().split(", ") for r in self.tmp.read().splitlines() if r.strip()]
        os.unlink(self.tmp.name)
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            try:
                sm.append(float(r[1]))
                mx = float(r[2])
                for nm, v in zip(names, r[5:9]):
                    if v.strip().lower() == "active":
                        reasons.add(nm)
            except Exception:
                continue
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


def _dist():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def _barrier(ws):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


def _max_over_ranks(x, ws):
    """The largest x over the ranks (a step is as slow as its slowest rank)."""
    if ws == 1:
        return x
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def _job_rate(units_per_rank, step_ms_max, ws):
    """Whole-job throughput: every rank processes its own replica of the
    workload (weak scaling), so the job moves ws * units in the slowest
    rank's step time."""
    return ws * units_per_rank / (step_ms_max / 1e3)


class L2Flush:
    """Evicts L2 between timed steps: writes a buffer of twice the L2 size, then
    reads a second one of the same size, so that L2 ends up holding only clean
    lines and no write-back of the flush itself lands inside a timed step."""

    def __init__(self):
        l2 = torch.cuda.get_device_properties(0).L2_cache_size
        n = max(2 * l2, 256 << 20) // 4
        self.w = torch.empty(n, dtype=torch.float32, device="cuda")
        self.r = torch.ones(n, dtype=torch.float32, device="cuda")
        self.sink = torch.empty(1, dtype=torch.float32, device="cuda")

    def zero_(self):
        self.w.zero_()
        torch.sum(self.r, dim=0, out=self.sink[0])
        # Hold the stream for ~100 us (200k cycles at 2.07 GHz) after the
        # flush so that the host has queued the whole step (two or three C-ABI
        # calls, 3-12 us each on a 16-core Arm host, the Python wrapper
        # included) before its first event runs: the events then time device
        # work only, never the host's launch latency (which the e2e figure
        # includes).
        torch.cuda._sleep(200_000)


def _flush_buf():
    return L2Flush()


def _time_steps(fn_plan, fn_exec, steps, flush):
    """CUDA events on the current stream: (step ms list, exec ms list).

    A step is plan + execute with nothing between them, as fia_run issues
    them (an event in between would break the programmatic launch chaining);
    the execute-only times, for the kernel roofline, come from a second pass
    of the same number of steps with an event after the plan."""
    s = torch.cuda.current_stream()
    step_ms, exec_ms = [], []
    for _ in range(steps):
        flush.zero_()
        e0 = torch.cuda.Event(enable_timing=True)
        e2 = torch.cuda.Event(enable_timing=True)
        e0.record(s)
        fn_plan()
        fn_exec()
        e2.record(s)
        e2.synchronize()
        step_ms.append(e0.elapsed_time(e2))
    for _ in range(steps):
        flush.zero_()
        fn_plan()
        e1 = torch.cuda.Event(enable_timing=True)
        e2 = torch.cuda.Event(enable_timing=True)
        e1.record(s)
        fn_exec()
        e2.record(s)
        e2.synchronize()
        exec_ms.append(e1.elapsed_time(e2))
    return step_ms, exec_ms


# ---------------------------------------------------------------------------
# CPU oracle baselines (bounded samples of each workload)
# ---------------------------------------------------------------------------

def _cores():
    return len(os.sched_getaffinity(0))


def _timed_repeats(fn, min_seconds):
    """Run fn until min_seconds have passed (at least once): (runs, seconds)."""
    t0 = time.perf_counter()
    n = 0
    while True:
        fn()
        n += 1
        if time.perf_counter() - t0 >= min_seconds:
            break
    return n, time.perf_counter() - t0


def cpu_baseline(prob_cpu, bytes_per_run, min_seconds=10.0):
    import oracle
    cores = _cores()
    oracle.fia(prob_cpu, cores)  # build + warm
    n, dt = _timed_repeats(lambda: oracle.fia(prob_cpu, cores), min_seconds)
    return {"value": bytes_per_run * n / dt / 1e9, "unit": "GB/s", "cores": cores,
            "kind": "oracle",
            "sample": f"the whole paged GQA decode batch, repeated {n}x ({dt:.1f} s, fp64, "
                      f"OpenMP over output rows)"}


def cpu_single_thread(prob_cpu, bytes_per_run):
    """The same oracle on one thread, one whole pass."""
    import oracle
    t0 = time.perf_counter()
    oracle.fia(prob_cpu, 1)
    dt = time.perf_counter() - t0
    return {"value": bytes_per_run / dt / 1e9, "unit": "GB/s", "cores": 1, "kind": "oracle",
            "sample": f"the whole batch once ({dt:.1f} s)"}


def _sample_rows_heads(p, n_pairs, seed):
    g = np.random.default_rng(seed)
    rows = g.integers(0, p.rows, n_pairs)
    heads = g.integers(0, p.QN, n_pairs)
    return rows, heads


def _row_kv(p, rows):
    """Visible keys of each sampled query row (for the work it stands for)."""
    out = []
    cu = None if p.cu_seqlens_q is None else p.cu_seqlens_q.tolist()
    for r in rows.tolist():
        if cu is None:
            b, i = divmod(r, p.S_q)
        else:
            b = max(k for k in range(p.B) if cu[k] <= r)
            i = r - cu[b]
        ql, kl = p.q_lens[b], p.kv_lens[b]
        hi = kl - ql + i if p.mask_mode == 3 else kl - 1
        out.append(max(0, min(hi, kl - 1) + 1))
    return out


def cpu_sampled(p_cpu, units_total, unit, nthreads, min_seconds, n_pairs, seed):
    """The oracle on a sample of (query row, head) pairs of a workload.  The
    sample does a fraction f of the whole workload's oracle work (its pairs'
    visible keys over those of every pair), so the rate credited is
    f * units_total per elapsed second: the whole workload's metric at the
    oracle's speed on this sample."""
    import oracle
    rows, heads = _sample_rows_heads(p_cpu, n_pairs, seed)
    all_rows = np.arange(p_cpu.rows)
    work_all = p_cpu.QN * sum(_row_kv(p_cpu, all_rows))
    f = sum(_row_kv(p_cpu, rows)) / max(1, work_all)
    oracle.fia_sample(p_cpu, rows, heads, nthreads)  # build + warm
    n, dt = _timed_repeats(lambda: oracle.fia_sample(p_cpu, rows, heads, nthreads), min_seconds)
    scale = 1e9 if unit == "GB/s" else 1e12
    return {"value": f * units_total * n / dt / scale, "unit": unit, "cores": nthreads,
            "kind": "oracle",
            "sample": f"{n_pairs} (query row, head) pairs ({100 * f:.3g} % of the workload's "
                      f"oracle work), repeated {n}x ({dt:.1f} s)"}


def cpu_both(p_cpu, units_total, unit, min_seconds, n_pairs, seed):
    """All host cores, and one thread, on the same sample."""
    allc = cpu_sampled(p_cpu, units_total, unit, _cores(), min_seconds, n_pairs, seed)
    one = cpu_sampled(p_cpu, units_total, unit, 1, min(1.0, min_seconds), max(1, n_pairs // 8),
                      seed)
    return allc, one


def cpu_sparse(sp_cpu, by, nthreads, min_seconds):
    import oracle
    n, dt = _timed_repeats(lambda: oracle.sparse(sp_cpu, nthreads), min_seconds)
    return {"value": by * n / dt / 1e9, "unit": "GB/s", "cores": nthreads, "kind": "oracle",
            "sample": f"the whole sparse CSA batch, {n}x ({dt:.1f} s)"}


# ---------------------------------------------------------------------------
# extra workloads (evidence only)
# ---------------------------------------------------------------------------

class _Skip(Exception):
    """A workload left out by --only."""


def _warm_up(fn_plan, fn_exec, warmup, flush):
    """Warm-up steps: the timed sequence (L2 flush, device sleep, plan,
    execute), untimed.  The first launches of the flush and sleep kernels
    carry one-off costs (a first timed step of 160 us against 65 us when the
    warm-up ran fia_run alone)."""
    for _ in range(warmup):
        flush.zero_()
        fn_plan()
        fn_exec()
    torch.cuda.synchronize()


def _bench_call(call, steps, warmup, flush):
    _warm_up(call.plan, call.execute, warmup, flush)
    return _time_steps(call.plan, call.execute, steps, flush)


def _stats(xs):
    return statistics.mean(xs), statistics.median(xs)


def extra_workloads(steps, warmup, flush, peaks, with_cpu, cpu_seconds, only=None):
    import decode_tile_scheduler_gb300 as fia
    import fia_inputs as fi
    res = {}

    def want(key):
        return only is None or key in only.split(",")

    # long-context FP8 decode
    try:
        if not want("fp8_long_decode"):
            raise _Skip
        p = fi.workload_fp8_long_decode(device="cuda")
        call = fia.FiaCall(p, with_lse=True)
        st, ex = _bench_call(call, steps, warmup, flush)
        (ms, ms_med), (kms, kms_med) = _stats(st), _stats(ex)
        by = p.kv_bytes_visible()
        res["fp8_long_decode"] = {
            "workload": "B=4, Q_N=64, KV_N=8, D=128, E4M3 KV + fp32/64 scales, kv len ~ "
                        "U[32768,131072], block 128",
            "ms_per_step": ms, "ms_median": ms_med, "kernel_ms": kms, "kernel_ms_median": kms_med,
            "GB/s": by / ms / 1e6, "kernel_GB/s": by / kms / 1e6,
            "frac_of_hbm": by / kms / 1e6 / peaks["hbm_gbs"], "algorithmic_bytes": by}
        if with_cpu:
            r = res["fp8_long_decode"]
            r["cpu_baseline"], r["cpu_single_thread"] = cpu_both(p.to("cpu"), by, "GB/s",
                                                                 cpu_seconds, 32, 5)
        del call, p
    except _Skip:
        pass
    except Exception as e:  # not built yet
        res["fp8_long_decode"] = {"unavailable": str(e)[:200]}
    torch.cuda.empty_cache()
    try:
        if not want("varlen_causal_prefill"):
            raise _Skip
        p = fi.workload_varlen_prefill(device="cuda")
        call = fia.FiaCall(p, with_lse=True)
        st, ex = _bench_call(call, steps, warmup, flush)
        (ms, ms_med), (kms, kms_med) = _stats(st), _stats(ex)
        fl = 4 * p.D * p.QN * sum(L * (L + 1) // 2 for L in p.q_lens)
        res["varlen_causal_prefill"] = {
            "workload": "TND B=8, L ~ U[256,4096], Q_N=32, KV_N=8, D=128, paged block 128, "
                        "right-down causal, sinks",
            "ms_per_step": ms, "ms_median": ms_med, "kernel_ms": kms, "kernel_ms_median": kms_med,
            "TFLOP/s": fl / ms / 1e9, "kernel_TFLOP/s": fl / kms / 1e9,
            "frac_of_bf16": fl / kms / 1e9 / peaks["bf16_tflops"], "flops": fl}
        if with_cpu:
            r = res["varlen_causal_prefill"]
            r["cpu_baseline"], r["cpu_single_thread"] = cpu_both(p.to("cpu"), fl, "TFLOP/s",
                                                                 cpu_seconds, 256, 7)
        del call, p
    except _Skip:
        pass
    except Exception as e:
        res["varlen_causal_prefill"] = {"unavailable": str(e)[:200]}
    torch.cuda.empty_cache()
    # forms beyond the headline workloads: multi-token decode (4 query rows
    # per sequence), head-major pages, FP8 decode with 16 query heads per KV
    # head, FP8 prefill
    for key, mk, what in (
            ("fp8_gqa16_decode",
             lambda: fi.workload_fp8_long_decode(device="cuda", KVN=4),
             "the long FP8 decode with KV_N=4 (16 query heads per KV head)"),
            ("mtp_decode_s4", lambda: fi.workload_paged_decode(device="cuda", S_q=4),
             "paged GQA decode sequences with 4 query rows each (right-down causal)"),
            ("paged_decode_bnnbsd",
             lambda: fi.workload_paged_decode(device="cuda", kv_layout=fi.KV_LAYOUT_BNNBSD),
             "paged GQA decode with head-major pages [nb, KV_N, bs, D]")):
        try:
            if not want(key):
                raise _Skip
            p = mk()
            call = fia.FiaCall(p, with_lse=True)
            st, ex = _bench_call(call, steps, warmup, flush)
            (ms, ms_med), (kms, kms_med) = _stats(st), _stats(ex)
            by = p.kv_bytes_visible()
            res[key] = {"workload": what, "ms_per_step": ms, "ms_median": ms_med,
                        "kernel_ms": kms, "kernel_ms_median": kms_med, "GB/s": by / ms / 1e6,
                        "kernel_GB/s": by / kms / 1e6,
                        "frac_of_hbm": by / kms / 1e6 / peaks["hbm_gbs"], "algorithmic_bytes": by}
            if with_cpu:
                res[key]["cpu_baseline"], res[key]["cpu_single_thread"] = cpu_both(
                    p.to("cpu"), by, "GB/s", cpu_seconds, 64, 11)
            del call, p
        except _Skip:
            pass
        except Exception as e:
            res[key] = {"unavailable": str(e)[:200]}
        torch.cuda.empty_cache()
    try:
        if not want("fp8_varlen_causal_prefill"):
            raise _Skip
        p = fi.workload_varlen_prefill(device="cuda", kv_dtype=fi.KV_FP8_E4M3)
        call = fia.FiaCall(p, with_lse=True)
        st, ex = _bench_call(call, steps, warmup, flush)
        (ms, ms_med), (kms, kms_med) = _stats(st), _stats(ex)
        fl = 4 * p.D * p.QN * sum(L * (L + 1) // 2 for L in p.q_lens)
        res["fp8_varlen_causal_prefill"] = {
            "workload": "the varlen causal prefill with an FP8 E4M3 cache (converted to fp16 "
                        "once per call, then the tcgen05 kernel on fp16 operands)",
            "ms_per_step": ms, "ms_median": ms_med, "kernel_ms": kms, "kernel_ms_median": kms_med,
            "TFLOP/s": fl / ms / 1e9, "kernel_TFLOP/s": fl / kms / 1e9,
            "frac_of_bf16": fl / kms / 1e9 / peaks["bf16_tflops"], "flops": fl}
        if with_cpu:
            r = res["fp8_varlen_causal_prefill"]
            r["cpu_baseline"], r["cpu_single_thread"] = cpu_both(p.to("cpu"), fl, "TFLOP/s",
                                                                 cpu_seconds, 256, 7)
        del call, p
    except _Skip:
        pass
    except Exception as e:
        res["fp8_varlen_causal_prefill"] = {"unavailable": str(e)[:200]}
    torch.cuda.empty_cache()
    try:
        if not want("sparse_csa_decode"):
            raise _Skip
        sp = fi.workload_sparse_csa(device="cuda")
        call = fia.SparseCall(sp, with_lse=True)
        call.plan()
        _warm_up(call.plan, call.run, warmup, flush)
        st, ex = _time_steps(call.plan, call.run, steps, flush)
        (ms, ms_med), (kms, kms_med) = _stats(st), _stats(ex)
        by = sp.B * (sp.win_left + 1 + sp.K2) * sp.D * 2
        res["sparse_csa_decode"] = {
            "workload": "B=16, N1=64, D=512, ori 8192 band 127/0, cmp 2048 (ratio 4), top-512",
            "ms_per_step": ms, "ms_median": ms_med, "kernel_ms": kms, "kernel_ms_median": kms_med,
            "GB/s": by / ms / 1e6, "kernel_GB/s": by / kms / 1e6,
            "frac_of_hbm": by / kms / 1e6 / peaks["hbm_gbs"], "algorithmic_bytes": by}
        if with_cpu:
            spc = sp.to("cpu")
            res["sparse_csa_decode"]["cpu_baseline"] = cpu_sparse(spc, by, _cores(), cpu_seconds)
            res["sparse_csa_decode"]["cpu_single_thread"] = cpu_sparse(spc, by, 1, 0.0)
        del call, sp
    except _Skip:
        pass
    except Exception as e:
        res["sparse_csa_decode"] = {"unavailable": str(e)[:200]}
    try:
        if not want("sparse_csa_decode_fp8_packed"):
            raise _Skip
        sp = fi.workload_sparse_csa(device="cuda", kv_dtype=fi.SPARSE_KV_FP8_PACKED)
        call = fia.SparseCall(sp, with_lse=True)
        call.plan()
        _warm_up(call.plan, call.run, warmup, flush)
        st, ex = _time_steps(call.plan, call.run, steps, flush)
        (ms, ms_med), (kms, kms_med) = _stats(st), _stats(ex)
        by = sp.B * (sp.win_left + 1 + sp.K2) * 640  # packed rows, once each
        res["sparse_csa_decode_fp8_packed"] = {
            "workload": "the sparse CSA decode with packed FP8 K~ rows (640 bytes: bf16 rope "
                        "64, E4M3 nope 448, E8M0 scales)",
            "ms_per_step": ms, "ms_median": ms_med, "kernel_ms": kms, "kernel_ms_median": kms_med,
            "GB/s": by / ms / 1e6, "kernel_GB/s": by / kms / 1e6,
            "frac_of_hbm": by / kms / 1e6 / peaks["hbm_gbs"], "algorithmic_bytes": by}
        if with_cpu:
            spc = sp.to("cpu")
            r = res["sparse_csa_decode_fp8_packed"]
            r["cpu_baseline"] = cpu_sparse(spc, by, _cores(), cpu_seconds)
            r["cpu_single_thread"] = cpu_sparse(spc, by, 1, 0.0)
        del call, sp
    except _Skip:
        pass
    except Exception as e:
        res["sparse_csa_decode_fp8_packed"] = {"unavailable": str(e)[:200]}
    if with_cpu and only is None:
        try:
            import oracle
            t = fi.workload_tiny_prefill(device="cpu")
            fl = 4 * t.D * t.QN * sum(L * (L + 1) // 2 for L in t.q_lens)
            oracle.fia(t, 1)
            n, dt = _timed_repeats(lambda: oracle.fia(t, 1), 1.0)
            res["tiny_prefill_cpu_single_thread"] = {
                "value": fl * n / dt / 1e9, "unit": "GFLOP/s", "cores": 1, "kind": "oracle",
                "sample": f"the whole tiny prefill, {n}x ({dt:.1f} s)"}
        except Exception as e:
            res["tiny_prefill_cpu_single_thread"] = {"unavailable": str(e)[:200]}
    return res


# ---------------------------------------------------------------------------
# arms
# ---------------------------------------------------------------------------

def run_reference(args):
    ws, rank, _ = _dist()
    if rank != 0:
        return
    import fia_inputs as fi
    import oracle
    p = fi.workload_paged_decode(device="cpu")
    by = p.kv_bytes_visible()
    cores = len(os.sched_getaffinity(0))
    for _ in range(args.warmup):
        oracle.fia(p, cores)
    times = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        oracle.fia(p, cores)
        times.append(time.perf_counter() - t0)
    ms = 1e3 * statistics.mean(times)
    val = by / (ms / 1e3) / 1e9
    sample = "the whole paged GQA decode batch per step (fp64 oracle, OpenMP)"
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": val, "unit": "GB/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": WORKLOAD, "l2": "oracle on host cores"},
        "cpu_baseline": {"value": val, "unit": "GB/s", "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": val, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }))


def run_fia(args):
    ws, rank, local = _dist()
    torch.cuda.set_device(local)
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    import decode_tile_scheduler_gb300 as fia
    import fia_inputs as fi
    fia.lib()
    peaks = _peaks()

    # ---- device-resident workload (each rank: one replica of the batch) ----
    p = fi.workload_paged_decode(device="cuda")
    by = p.kv_bytes_visible()
    call = fia.FiaCall(p, with_lse=True)
    flush = _flush_buf()
    _warm_up(call.plan, call.execute, max(args.warmup, 3), flush)
    _barrier(ws)
    clocks = ClockSampler(local)
    clocks.start()
    torch.cuda.synchronize()
    step_ms, exec_ms = _time_steps(call.plan, call.execute, args.steps, flush)
    torch.cuda.synchronize()
    clk = clocks.stop()
    _barrier(ws)
    ms = _max_over_ranks(statistics.mean(step_ms), ws)
    kern_ms = _max_over_ranks(statistics.mean(exec_ms), ws)
    ms_med = _max_over_ranks(statistics.median(step_ms), ws)
    kern_ms_med = _max_over_ranks(statistics.median(exec_ms), ws)
    value = _job_rate(by, ms, ws) / 1e9
    achieved = by / (kern_ms / 1e3) / 1e9

    # ---- end to end through the C ABI with host buffers ----
    # The step's inputs (q, KV lengths, block table) share one device buffer
    # and its results (out, lse) another, as a serving loop would lay them
    # out, so each step moves them with one host-to-device and one
    # device-to-host copy (pinned host memory) around fia_run.
    def _packed(tensors, dev):
        offs, total = [], 0
        for t in tensors:
            offs.append(total)
            total += (t.numel() * t.element_size() + 255) // 256 * 256
        buf = torch.zeros(total, dtype=torch.uint8, device=dev)
        views = [buf[o:o + t.numel() * t.element_size()].view(t.dtype).view(t.shape)
                 for t, o in zip(tensors, offs)]
        return buf, views

    dev_in, (v_q, v_len, v_bt) = _packed([p.q, p.seqused_kv, p.block_table], "cuda")
    v_q.copy_(p.q)
    v_len.copy_(p.seqused_kv)
    v_bt.copy_(p.block_table)
    p.q, p.seqused_kv, p.block_table = v_q, v_len, v_bt
    dev_out, (v_out, v_lse) = _packed([call.out, call.lse], "cuda")
    call_e2e = fia.FiaCall(p, with_lse=True, out=v_out, lse=v_lse)
    host_in = dev_in.cpu().pin_memory()
    host_res = torch.empty(dev_out.numel(), dtype=torch.uint8).pin_memory()
    # Host wall clock around each step: the copy in, fia_run (host-side
    # validation, tensor-map encoding and launches through the C ABI) and the
    # copy out, ending with a stream synchronise.  L2 is flushed and the
    # stream drained before the clock starts, so nothing queued earlier runs
    # inside the timed region and no device sleep hides the host's cost.
    s = torch.cuda.current_stream()
    e2e_ms = []
    for i in range(args.warmup + args.steps):
        flush.zero_()
        s.synchronize()
        t0 = time.perf_counter()
        dev_in.copy_(host_in, non_blocking=True)
        call_e2e.run()
        host_res.copy_(dev_out, non_blocking=True)
        s.synchronize()
        t1 = time.perf_counter()
        if i >= args.warmup:
            e2e_ms.append(1e3 * (t1 - t0))
    h2d = host_in.numel()
    d2h = host_res.numel()
    e2e = _job_rate(by, _max_over_ranks(statistics.mean(e2e_ms), ws), ws) / 1e9

    extras = {}
    if rank == 0 and not args.no_extras:
        extras = extra_workloads(max(3, min(args.steps, 50)), 3, flush, peaks,
                                 not args.no_cpu, min(3.0, args.cpu_seconds))

    cpu = None
    if rank == 0 and not args.no_cpu:
        pc = p.to("cpu")
        cpu = cpu_baseline(pc, by, min_seconds=args.cpu_seconds)
        cpu["single_thread"] = cpu_single_thread(pc, by)

    traffic = _ncu_traffic("decode_kernel_bf16_d128", ["decode.cu", "common.cuh", "internal.h"], by)
    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": ws, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": WORKLOAD, "l2": "flushed between timed steps (write 2x L2, then read another 2x L2 buffer)",
                       "parallelism": f"replicas x{ws}" if ws > 1 else "single GPU",
                       "algorithmic_bytes_per_step": by},
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"],
                         "unit": "GB/s", "frac": achieved / peaks["hbm_gbs"],
                         "traffic": traffic, "kernel": "decode_kernel<128,bf16> + decode_combine_flat (fia_execute)",
                         "peak_source": peaks["source"] + " (burst copy)"},
            "e2e": {"value": e2e, "unit": "GB/s", "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h, "clock": "host wall clock (perf_counter) around "
                    "H2D copy + fia_run + D2H copy + stream synchronise",
                    "ms_per_step": statistics.mean(e2e_ms),
                    "ms_median": statistics.median(e2e_ms)},
            "timing": {"step_ms_median": ms_med, "kernel_ms_mean": kern_ms,
                       "kernel_ms_median": kern_ms_med,
                       "note": "value and ms_per_step: mean of the K timed steps; medians beside"},
            "gpu_launches": 3 * args.steps,
            "clocks": clk,
            "cpu_baseline": cpu,
            "extra": extras,
        }
        print(json.dumps(line))
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def run_only(args):
    """One extra workload alone: its JSON object on one line (not the
    contract's line).  Launches: W warm-up steps, then K timed steps."""
    peaks = _peaks()
    flush = _flush_buf()
    res = extra_workloads(max(1, args.steps), args.warmup, flush, peaks, not args.no_cpu,
                          min(3.0, args.cpu_seconds), only=args.only)
    if not res:
        raise SystemExit(f"no extra workload named {args.only!r}")
    print(json.dumps(res))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="fia", choices=["fia", "reference"])
    ap.add_argument("--no-extras", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--only", default=None,
                    help="time one extra workload alone (e.g. mtp_decode_s4) and print "
                         "its figures; for profiling")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    elif args.only:
        run_only(args)
    else:
        run_fia(args)


if __name__ == "__main__":
    main()
