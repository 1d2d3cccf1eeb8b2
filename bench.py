"""Benchmark: paged GQA attention on GB300 through the library's C ABI.

Default workload (N=1): the MTP verify batch -- 64 sequences, q_len 4, 16 q heads /
1 kv head, head_dim 256, context lengths uniform in [1024, 32768], 16-token pages,
FP8 e4m3 K/V with per-tensor descales, bf16 Q and output. One step = one
paged_gqa_attn call (plan + attention kernels) over that batch.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--config 1..5] [--impl reference]
  python bench.py --op cache_write [--config 1..5] ...   # the paged KV-cache write alone

Prints ONE JSON line (rank 0). The value is KV-read GB/s (algorithmic bytes: each
valid token's K and V once per kv head) for verify-bound workloads and TFLOP/s
(causal-exact) for prefill-bound ones; us/call is reported beside it. Under
torchrun each rank runs an independent replica (the path shards by sequence and
kv head with no exchange), so the value is the sum over ranks divided by the
slowest rank's time.

--impl reference times the fp64 CPU oracle (the only reference this path has) on a
bounded sample of the same workload on the host cores.

--op attn_quant_q times paged_gqa_attn_quant_q: the same workload with its Q given in bf16
(configs whose Q is e4m3 take the bf16 values it was made from) and quantised inside the
call to e4m3 under one per-tensor scale (amax / 448).

--op sparse times paged_gqa_sparse_attn on the sparse prefill workload (8192 new tokens on
a 32768-token context, 2051 selected positions per (token, kv head), heads of --sparse-tp):
TFLOP/s of the used (row, key) pairs at 4 * 256 FLOPs each.

--op cache_write times paged_gqa_cache_write instead: the config's new tokens (every
sequence's last q_len positions, bf16 K and V for each kv head) quantised to e4m3 and
scattered into their pages. Its value is GB/s of algorithmic bytes (per (token, kv head)
row: 2 x 512 bytes of bf16 read, 2 x 256 bytes of e4m3 written) against the HBM roofline.
"""
from __future__ import annotations

import argparse
import dataclasses
import json
import hashlib
import os
import statistics
import subprocess
import sys
import threading
import time

import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads as wl  # noqa: E402

METRIC = "us/call and KV-read GB/s (verify) / TFLOP/s (prefill) as % of GB300 roofline"
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0
L2_FLUSH_BYTES = 512 << 20
L2_NOTE = "flushed: 512 MiB memset, then a 512 MiB read, between timed calls (no input line and no dirty line left in L2)"


class L2Flush:
    """Between timed calls: write a buffer four times the L2 (evicts every input line), then
    read another as large, so the memset's dirty lines are written back here and not inside
    the next timed call (a memset alone left ~130 MB of dirty lines whose write-back cost the
    MTP verify call ~4.5 us and workload 3 ~12 us)."""

    def __init__(self, dev):
        self.w = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
        self.r = torch.ones(L2_FLUSH_BYTES // 4, dtype=torch.int32, device=dev)
        self.acc = torch.zeros((), dtype=torch.int32, device=dev)

    def zero_(self):
        self.w.zero_()
        torch.amax(self.r, 0, out=self.acc)  # reads every byte once, no dtype conversion


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--config", type=int, default=2)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--op", default="attn", choices=["attn", "attn_quant_q", "cache_write", "sparse"])
    ap.add_argument("--sparse-tp", type=int, default=1, choices=[1, 2, 4, 8],
                    help="sparse: head layout of the sparse page's TP1/2/4/8 shapes")
    ap.add_argument("--write-case", default="config", choices=["config", "chunks"],
                    help="cache_write: the config's new tokens, or 32 fresh 4096-token chunks (profiling size)")
    ap.add_argument("--cpu-seconds", type=float, default=15.0, help="target CPU time of the oracle sample")
    ap.add_argument("--extra-cpu-seconds", type=float, default=3.0,
                    help="target CPU time of the oracle sample of each extra workload")
    ap.add_argument("--no-extra-configs", action="store_true",
                    help="time only --config (by default the MTP verify line also times workloads 1, 3, 4, 5)")
    ap.add_argument("--path", type=int, default=0, choices=[0, 1, 2, 3],
                    help="kernel path (paged_gqa_set_path): 0 auto, 1 warp-level MMA, 2 auto + tcgen05 sparse "
                         "kernel, 3 auto with the verify class planned by the plan kernel")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    return ap.parse_args()


class PinnedInputs:
    """A step's host inputs packed into one pinned buffer and copied to the device in one
    transfer, into views of one device buffer (as a serving loop stages its per-step data:
    one copy instead of one per tensor, each of which costs a few microseconds of its own)."""

    def __init__(self, tensors, dev):
        offs, at = [], 0
        for t in tensors:
            offs.append(at)
            at += (t.numel() * t.element_size() + 255) // 256 * 256
        self.nbytes = at  # bytes copied per step (each tensor padded to 256 bytes)
        self.host = torch.empty(at, dtype=torch.uint8, pin_memory=True)
        self.dev = torch.empty(at, dtype=torch.uint8, device=dev)
        self.views = []
        for t, o in zip(tensors, offs):
            n = t.numel() * t.element_size()
            self.host[o:o + n].copy_(t.detach().contiguous().cpu().reshape(-1).view(torch.uint8))
            self.views.append(self.dev[o:o + n].view(t.dtype).view(t.shape))

    def copy(self):
        self.dev.copy_(self.host, non_blocking=True)


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def max_over_ranks(values, world: int, device) -> list:
    """Each rank's timings -> the maximum over ranks (the slowest replica sets the job time)."""
    t = torch.tensor(values, dtype=torch.float64, device=device)
    if world > 1:
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return t.tolist()


def whole_job_value(units_per_step: float, world: int, step_ms: float) -> float:
    """Replicas (weak scaling): every rank processes units_per_step per step, so the job's
    throughput is world x units_per_step over the slowest rank's step time."""
    return units_per_step * world / (step_ms / 1e3)


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), float(d.get("bf16_tflops_sustained", d["bf16_tflops"])), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS, FALLBACK_BF16_TFLOPS * 0.9, "fallback"


def workload_kind(spec: wl.CaseSpec) -> str:
    """'hbm' when KV bytes dominate the roofline time, else 'tensor'."""
    hbm, bf16, _, _ = load_peaks()
    fp8 = 2 * bf16
    t_mem = spec.kv_bytes / (hbm * 1e9)
    t_mma = spec.flops / (fp8 * 1e12)
    return "hbm" if t_mem >= t_mma else "tensor"


def config_dict(spec: wl.CaseSpec, idx: int, n: int, l2_note: str, quant_q: bool = False):
    return {"workload": spec.name + (":quant_q" if quant_q else ""), "config_index": idx, "num_seqs": spec.num_seqs, "total_q": spec.total_q,
            "num_q_heads": spec.num_q_heads, "num_kv_heads": spec.num_kv_heads, "head_dim": wl.HEAD_DIM,
            "page_size": spec.page_size, "q_dtype": spec.q_dtype, "kv_dtype": spec.kv_dtype, "out_dtype": "bf16",
            "kv_bytes": spec.kv_bytes, "flops": spec.flops, "parallelism": f"replicas{n}", "l2": l2_note,
            "seed": 0}


class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled during the timed region."""

    FIELDS = ("index,pci.bus_id,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.proc = None
        self.lines = []
        self.bus = None
        try:
            props = torch.cuda.get_device_properties(device_index)
            self.bus = "%08X:%02X:%02X.0" % (getattr(props, "pci_domain_id", 0), props.pci_bus_id,
                                               props.pci_device_id)
        except Exception:
            pass

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                                          "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        rows = [l.split(", ") for l in self.lines if l]
        if self.bus:
            mine = [r for r in rows if len(r) > 1 and r[1].upper().endswith(self.bus[-7:].upper())]
            rows = mine or rows
        sm = [float(r[2]) for r in rows if len(r) >= 10 and r[2].replace(".", "").isdigit()]
        smax = [float(r[3]) for r in rows if len(r) >= 10 and r[3].replace(".", "").isdigit()]
        reasons = set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            if len(r) < 10:
                continue
            for name, val in zip(names, r[6:10]):
                if val.strip().lower() == "active":
                    reasons.add(name)
        busy = [s for s in sm]
        return {"sm_mhz": statistics.median(busy) if busy else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(rows)}


def kernel_source_hash(cls_kind: str) -> str:
    names = {"verify": ["verify_tc.cu"], "prefill": ["prefill_tc.cu"], "portable": ["portable.cu"],
             "cache_write": ["cache_write.cu"], "bf16": ["bf16_tc.cu"], "sparse": ["sparse.cu"],
             "sparse_tc": ["sparse_tc.cu"]}[cls_kind]
    h = hashlib.sha256()
    for n in names + ["common.cuh", "device_util.cuh", "tc_util.cuh"]:
        p = os.path.join(ROOT, "paged_gqa_gb300", "csrc", n)
        if os.path.exists(p):
            h.update(open(p, "rb").read())
    return h.hexdigest()[:16]


def traffic_for(kernel_kind: str, workload: str):
    """DRAM bytes per launch from the committed ncu summary, if the kernel is unchanged."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)
        e = d.get(f"{kernel_kind}:{workload}")
        if e and e.get("source_sha") == kernel_source_hash(kernel_kind):
            return float(e["dram_bytes_per_launch"])
    except Exception:
        pass
    return None


# ------------------------------------------------------------------------ ours --

def attn_spec(args) -> wl.CaseSpec:
    """The config's workload; for the quantising call its q is given in bf16 (the call
    makes the e4m3 q itself)."""
    spec = wl.config_spec(args.config)
    if args.op == "attn_quant_q" and spec.q_dtype != "bf16":
        spec = dataclasses.replace(spec, q_dtype="bf16")
    return spec


def _time_graph(pg, case, out, flush, K, warmup):
    """The caller-workspace call (paged_gqa_attn_ex) captured once in a CUDA graph, then
    replayed K times with the same L2 flush before each replay (outside the events): the
    call's cost without its host-side launch work. Returns the median us per replay."""
    spec = case.spec
    ws = torch.empty(pg.paged_gqa_workspace_size(spec.num_seqs, spec.total_q, spec.num_q_heads, spec.num_kv_heads,
                                                 spec.page_size, case.block_table.shape[1],
                                                 torch.cuda.current_device()),
                     dtype=torch.uint8, device=out.device)

    def call_ex():
        pg.paged_gqa_attn_ex(case.q, case.k_cache, case.v_cache, case.block_table, case.seq_lens,
                             case.query_start_loc, 1.0, case.k_descale, case.v_descale, case.softmax_scale, out, ws)

    call_ex()  # per-device set-up happens outside the capture
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        call_ex()
    for _ in range(max(3, warmup)):
        graph.replay()
    torch.cuda.synchronize()
    assert pg.paged_gqa_check_device_errors() == 0, pg.paged_gqa_last_error()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    for i in range(K):
        flush.zero_()
        ev[i][0].record()
        graph.replay()
        ev[i][1].record()
    torch.cuda.synchronize()
    us = statistics.median(a.elapsed_time(b) for a, b in ev) * 1e3
    del graph, ws
    return us


def _time_attn(pg, call, flush, K, warmup, dominant_cls, local, world):
    """Per-call CUDA events over K calls (an L2 flush before each, outside the events),
    then a second pass with the library's events around the dominant kernel. Returns
    (call_ms list, kernel_ms list, clocks, wall_s)."""
    for _ in range(max(3, warmup)):
        call()
    torch.cuda.synchronize()
    assert pg.paged_gqa_check_device_errors() == 0, pg.paged_gqa_last_error()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    kev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    sampler = ClockSampler(local)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    sampler.start()
    time.sleep(0.3)
    wall0 = time.perf_counter()
    for i in range(K):
        flush.zero_()  # L2 flush between timed iterations (outside the events)
        ev[i][0].record()
        call()
        ev[i][1].record()
    torch.cuda.synchronize()
    wall = time.perf_counter() - wall0
    # The dominant kernel alone, from events the library records around it on its
    # launch stream (a second pass: events between kernels stop their launch overlap).
    for i in range(K):
        flush.zero_()
        pg.paged_gqa_set_kernel_events(dominant_cls, kev[i][0], kev[i][1])
        call()
    pg.paged_gqa_set_kernel_events(dominant_cls, None, None)
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    clocks = sampler.stop()
    assert pg.paged_gqa_check_device_errors() == 0, pg.paged_gqa_last_error()
    return [a.elapsed_time(b) for a, b in ev], [a.elapsed_time(b) for a, b in kev], clocks, wall


def _roofline(spec, kind, kern_ms_mean, kernel_kind, clocks=None, q_split=False):
    """The dominant kernel against its peak. Tensor-bound kernels take the FP8 peak as 2 x the
    measured bf16 GEMM rate (the nominal ratio): the burst rate, or the sustained one when the
    clocks sampled in the timed region show the power cap (a kernel timed inside a long step),
    with the burst fraction kept beside it. frac_of_attainable divides by the bound of this
    path's arithmetic: P.V runs as two e4m3 products (P hi + lo), and so does S when q is bf16
    (q hi + lo), so half the FLOPs (e4m3 q) or all of them (bf16 q) cost twice."""
    hbm, bf16, bf16_sus, peak_src = load_peaks()
    extra = {}
    if kind == "hbm":
        units, peak, peak_unit = spec.kv_bytes / 1e9, hbm, "GB/s"
        src = f"{peak_src} (hbm_gbs)"
    else:
        units, peak_unit = spec.flops / 1e12, "TFLOP/s"
        capped = bool(clocks) and "sw_power_cap" in (clocks.get("reasons") or [])
        peak = 2 * (bf16_sus if capped else bf16)
        src = f"{peak_src} (2 x bf16_tflops{'_sustained: sw_power_cap in the timed region' if capped else ' burst'})"
        if capped:
            extra["frac_of_burst_peak"] = round(units / (kern_ms_mean / 1e3) / (2 * bf16), 4)
    achieved = units / (kern_ms_mean / 1e3)
    r = {"bound": kind, "achieved": round(achieved, 2), "peak": peak, "unit": peak_unit,
         "frac": round(achieved / peak, 4), "peak_source": src, "kernel": kernel_kind,
         "kernel_us": round(kern_ms_mean * 1e3, 2), "traffic": traffic_for(kernel_kind, spec.name), **extra}
    if kind == "tensor":
        r["frac_of_attainable"] = round(r["frac"] * (2.0 if q_split else 1.5), 4)
        r["attainable"] = "1/2 of the FP8 peak (bf16 q: S and P.V as hi + lo)" if q_split else \
            "2/3 of the FP8 peak (e4m3 q: P.V as hi + lo)"
    return r


def _dominant(spec, config_index):
    kind = workload_kind(spec)
    cls = 0 if kind == "hbm" else 1
    if config_index == 5:
        cls = 1  # the mixed batch: prefill blocks hold nearly all of the work
    return kind, cls


def _kernel_kind(plan, cls, kind, spec=None):
    """Name of the class-`cls` kernel the last call ran (its traffic.json key prefix)."""
    if not plan["path_bits"] & (2 << cls):
        return "portable"
    if spec is not None and spec.kv_dtype == "bf16":
        return "bf16"
    return "verify" if cls == 0 else "prefill"


def extra_config(pg, args, idx, dev, flush, local, world, quant_q):
    """One more workload timed in the same run: median/mean us per call, the dominant
    kernel's roofline, clocks and a short oracle sample."""
    spec = dataclasses.replace(wl.config_spec(idx), q_dtype="bf16") if quant_q else wl.config_spec(idx)
    if quant_q and spec.kv_dtype != "e4m3":
        return None
    case = wl.make_case(spec, device=dev, seed=0)
    T, Hq = case.q.shape[0], case.q.shape[1]
    out = torch.empty(T, Hq, wl.HEAD_DIM, dtype=torch.bfloat16, device=dev)
    attn = pg.paged_gqa_attn_quant_q if quant_q else pg.paged_gqa_attn

    def call():
        attn(case.q, case.k_cache, case.v_cache, case.block_table, case.seq_lens,
             case.query_start_loc, case.k_descale, case.v_descale, case.softmax_scale, out)

    kind, cls = _dominant(spec, idx)
    K = max(5, min(args.steps, 20))
    call_ms, kern_ms, clocks, _ = _time_attn(pg, call, flush, K, args.warmup, cls, local, world)
    plan = pg.paged_gqa_last_plan()
    med, mean = statistics.median(call_ms), sum(call_ms) / K
    per = spec.kv_bytes / 1e9 if kind == "hbm" else spec.flops / 1e12
    r = {"workload": spec.name + (":quant_q" if quant_q else ""), "steps": K,
         "value": round(per / (med / 1e3), 3), "unit": "GB/s" if kind == "hbm" else "TFLOP/s",
         "us_per_call": round(med * 1e3, 2), "us_per_call_mean": round(mean * 1e3, 2),
         "kernel_us_median": round(statistics.median(kern_ms) * 1e3, 2),
         "roofline": _roofline(spec, kind, sum(kern_ms) / K, _kernel_kind(plan, cls, kind, spec), clocks,
                               q_split=spec.q_dtype == "bf16" and not quant_q),
         "path_bits": int(plan["path_bits"]), "clocks": clocks, "kv_bytes": spec.kv_bytes, "flops": spec.flops}
    if idx == 1 and not quant_q:
        # the launch-bound tiny call: also as one CUDA-graph replay
        r["graph_us_per_call"] = round(_time_graph(pg, case, out, flush, K, args.warmup), 2)
    if not args.no_cpu_baseline:
        r["cpu_baseline"] = cpu_baseline(spec, case, args.extra_cpu_seconds, kind, quant_q)
    del case, out
    torch.cuda.empty_cache()
    return r


def run_ours(args, rank, world, local):
    import paged_gqa_gb300 as pg
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    pg.load()
    pg.paged_gqa_set_path(args.path)
    spec = attn_spec(args)
    case = wl.make_case(spec, device=dev, seed=rank)  # each rank: an independent replica
    T, Hq = case.q.shape[0], case.q.shape[1]
    out = torch.empty(T, Hq, wl.HEAD_DIM, dtype=torch.bfloat16, device=dev)
    flush = L2Flush(dev)
    kind, dominant_cls = _dominant(spec, args.config)

    quant_q = args.op == "attn_quant_q"
    attn = pg.paged_gqa_attn_quant_q if quant_q else pg.paged_gqa_attn

    def call():
        attn(case.q, case.k_cache, case.v_cache, case.block_table, case.seq_lens,
             case.query_start_loc, case.k_descale, case.v_descale, case.softmax_scale, out)

    K = args.steps
    call_ms, kern_ms, clocks, wall = _time_attn(pg, call, flush, K, args.warmup, dominant_cls, local, world)
    plan = pg.paged_gqa_last_plan()
    step_ms = statistics.median(call_ms)
    step_mean_ms = sum(call_ms) / K
    kern_avg_ms = sum(kern_ms) / K

    # e2e: pinned host inputs -> device, call, device -> host result, every step
    e2e = None
    if not args.no_e2e:
        staged = PinnedInputs((case.q, case.block_table, case.seq_lens, case.query_start_loc), dev)
        dev_in = staged.views
        host_out = torch.empty(out.shape, dtype=out.dtype, pin_memory=True)
        h2d = staged.nbytes
        d2h = host_out.numel() * host_out.element_size()

        def e2e_step():
            staged.copy()
            attn(dev_in[0], case.k_cache, case.v_cache, dev_in[1], dev_in[2], dev_in[3],
                 case.k_descale, case.v_descale, case.softmax_scale, out)
            host_out.copy_(out, non_blocking=True)

        for _ in range(3):
            e2e_step()
        torch.cuda.synchronize()
        e_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
        for i in range(K):
            flush.zero_()
            e_ev[i][0].record()
            e2e_step()
            e_ev[i][1].record()
        torch.cuda.synchronize()
        e2e_ms = statistics.median(a.elapsed_time(b) for a, b in e_ev)
        e2e = (e2e_ms, h2d, d2h)
    # the same call as one CUDA-graph replay (no host launch work)
    graph_us = _time_graph(pg, case, out, flush, K, args.warmup) if args.op == "attn" else 0.0

    # reduce over ranks: max time
    step_ms, step_mean_ms, kern_avg_ms, e2e_ms, graph_us = max_over_ranks(
        [step_ms, step_mean_ms, kern_avg_ms, e2e[0] if e2e else 0.0, graph_us], world, dev)
    if rank != 0:
        return None
    cpu = None
    if world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(spec, case, args.cpu_seconds, kind, quant_q)
    extras = {}
    if world == 1 and not args.no_extra_configs and args.config == 2 and args.op in ("attn", "attn_quant_q"):
        for idx in (1, 3, 4, 5):
            r = extra_config(pg, args, idx, dev, flush, local, world, quant_q)
            if r is not None:
                extras[str(idx)] = r

    per_step = spec.kv_bytes / 1e9 if kind == "hbm" else spec.flops / 1e12
    unit = "GB/s" if kind == "hbm" else "TFLOP/s"
    value = whole_job_value(per_step, world, step_ms)
    kernel_kind = _kernel_kind(plan, dominant_cls, kind, spec)
    res = {
        "metric": METRIC, "value": round(value, 3), "unit": unit, "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": round(step_ms, 5), "ms_per_step_mean": round(step_mean_ms, 5),
        "us_per_call": round(step_ms * 1e3, 2),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "e4m3" if kernel_kind != "portable" else "tf32",
        "data": "synthetic (seeded N(0,1), FP8 per-tensor amax/448)",
        "config": config_dict(spec, args.config, world, L2_NOTE, quant_q),
        "roofline": _roofline(spec, kind, kern_avg_ms, kernel_kind, clocks,
                              q_split=spec.q_dtype == "bf16" and not quant_q),
        "gpu_launches": int(plan["kernels_launched"]) * K,
        "clocks": clocks,
        "wall_s": round(wall, 3),
        "stat": "value and ms_per_step from the median call; roofline.achieved from the mean kernel time",
    }
    if graph_us > 0:
        res["graph_us_per_call"] = round(graph_us, 2)
    if e2e:
        res["e2e"] = {"value": round(per_step * world / (e2e_ms / 1e3), 3), "unit": unit,
                      "h2d_bytes_per_step": e2e[1], "d2h_bytes_per_step": e2e[2],
                      "note": "per step: q, block_table, seq_lens, query_start_loc H2D as one transfer from one pinned buffer; out D2H; KV cache resident"}
    if cpu is not None:
        res["cpu_baseline"] = cpu
    if extras:
        res["configs"] = extras
    return res


# ----------------------------------------------------------- cache write --

CW_ROW_BYTES = 2 * wl.HEAD_DIM * 2 + 2 * wl.HEAD_DIM  # bf16 K and V read, e4m3 K and V written
CW_METRIC = "GB/s of the paged KV-cache write (bf16 new K/V read + e4m3 pages written) as % of HBM roofline"


def cw_config(spec: wl.CaseSpec, idx: int, n: int, l2_note: str):
    rows = spec.total_q * spec.num_kv_heads
    return {"workload": "cache_write:" + spec.name, "config_index": idx, "num_seqs": spec.num_seqs,
            "new_tokens": spec.total_q, "num_kv_heads": spec.num_kv_heads, "head_dim": wl.HEAD_DIM,
            "page_size": spec.page_size, "in_dtype": "bf16", "cache_dtype": "e4m3", "rows": rows,
            "bytes": rows * CW_ROW_BYTES, "parallelism": f"replicas{n}", "l2": l2_note, "seed": 0}


def _cw_spec(args) -> wl.CaseSpec:
    if args.write_case == "chunks":
        return wl.write_chunks_spec()
    return dataclasses.replace(wl.config_spec(args.config), kv_dtype="e4m3")


def _new_tokens(spec, device, seed):
    g = torch.Generator(device=device).manual_seed(seed + 101)
    shape = (spec.total_q, spec.num_kv_heads, wl.HEAD_DIM)
    kn = torch.randn(shape, generator=g, device=device).to(torch.bfloat16)
    vn = torch.randn(shape, generator=g, device=device).to(torch.bfloat16)
    return kn, vn


def run_cache_write(args, rank, world, local):
    import paged_gqa_gb300 as pg
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    pg.load()
    pg.paged_gqa_set_path(args.path)
    spec = _cw_spec(args)
    case = wl.make_case(spec, device=dev, seed=rank)
    kn, vn = _new_tokens(spec, dev, rank)
    flush = L2Flush(dev)
    bytes_per_step = spec.total_q * spec.num_kv_heads * CW_ROW_BYTES

    def call(k_new=kn, v_new=vn, bt=case.block_table, sl=case.seq_lens, qsl=case.query_start_loc):
        pg.paged_gqa_cache_write(k_new, v_new, case.k_cache, case.v_cache, bt, sl, qsl,
                                 case.k_descale, case.v_descale)

    for _ in range(max(3, args.warmup)):
        call()
    assert pg.paged_gqa_check_device_errors() == 0, pg.paged_gqa_last_error()
    K = args.steps
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    sampler = ClockSampler(local)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    sampler.start()
    time.sleep(0.3)
    wall0 = time.perf_counter()
    for i in range(K):
        flush.zero_()  # L2 flush between timed iterations (outside the events)
        ev[i][0].record()
        call()  # one kernel per call: the events bracket that kernel alone
        ev[i][1].record()
    torch.cuda.synchronize()
    wall = time.perf_counter() - wall0
    if world > 1:
        torch.distributed.barrier()
    clocks = sampler.stop()
    step_ms = sum(a.elapsed_time(b) for a, b in ev) / K

    e2e = None
    if not args.no_e2e:
        staged = PinnedInputs((kn, vn, case.block_table, case.seq_lens, case.query_start_loc), dev)
        dev_in = staged.views
        h2d = staged.nbytes

        def e2e_step():
            staged.copy()
            call(*dev_in)
            # the step's result on the host: the device status word (synchronises the stream)
            assert pg.paged_gqa_check_device_errors() == 0

        for _ in range(3):
            e2e_step()
        e_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
        for i in range(K):
            flush.zero_()
            e_ev[i][0].record()
            e2e_step()
            e_ev[i][1].record()
        torch.cuda.synchronize()
        e2e = (sum(a.elapsed_time(b) for a, b in e_ev) / K, h2d, 4)

    step_ms, e2e_ms = max_over_ranks([step_ms, e2e[0] if e2e else 0.0], world, dev)
    if rank != 0:
        return None
    hbm, _, _, peak_src = load_peaks()
    value = whole_job_value(bytes_per_step / 1e9, world, step_ms)
    achieved = bytes_per_step / 1e9 / (step_ms / 1e3)
    res = {
        "metric": CW_METRIC, "value": round(value, 3), "unit": "GB/s", "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": round(step_ms, 5), "us_per_call": round(step_ms * 1e3, 2),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16->e4m3",
        "data": "synthetic (seeded N(0,1) new K/V; the config's paged cache and block table)",
        "config": cw_config(spec, args.config, world, L2_NOTE),
        "roofline": {"bound": "hbm", "achieved": round(achieved, 2), "peak": hbm, "unit": "GB/s",
                     "frac": round(achieved / hbm, 4), "peak_source": f"{peak_src} (hbm_gbs)",
                     "kernel": "cache_write", "kernel_us": round(step_ms * 1e3, 2),
                     "traffic": cw_traffic(spec)},
        "gpu_launches": K, "clocks": clocks, "wall_s": round(wall, 3),
    }
    if e2e:
        res["e2e"] = {"value": round(bytes_per_step * world / 1e9 / (e2e_ms / 1e3), 3), "unit": "GB/s",
                      "h2d_bytes_per_step": e2e[1], "d2h_bytes_per_step": e2e[2],
                      "note": "per step: new K/V, block_table, seq_lens, query_start_loc H2D as one transfer from one pinned buffer; "
                              "the device status word D2H; the cache stays resident"}
    if world == 1 and not args.no_cpu_baseline:
        res["cpu_baseline"] = cw_cpu_sample(spec, case, kn, vn, args.cpu_seconds)
    return res


def cw_traffic(spec):
    """DRAM bytes per launch: the committed capture's bytes per (token, kv head) row times
    this workload's rows (the write's traffic grows with its rows), if the kernel is unchanged."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            e = json.load(f).get("cache_write:per_row")
        if e and e.get("source_sha") == kernel_source_hash("cache_write"):
            return round(float(e["dram_bytes_per_row"]) * spec.total_q * spec.num_kv_heads)
    except Exception:
        pass
    return None


def cw_cpu_sample(spec, case, kn, vn, target_s):
    """The write oracle on random whole sequences until ~target_s; scaled to the workload's rows."""
    from oracle import cache_write as cw
    gen = torch.Generator().manual_seed(4321)
    qsl = case.query_start_loc.cpu().tolist()
    order = torch.randperm(spec.num_seqs, generator=gen).tolist()
    elapsed, rows, nseq = 0.0, 0, 0
    for s in order:
        sub = wl.subcase(case, [s])
        k_new = kn[qsl[s]:qsl[s + 1]].float().cpu().numpy()
        v_new = vn[qsl[s]:qsl[s + 1]].float().cpu().numpy()
        args = (sub.k_cache.numpy(), sub.v_cache.numpy(), sub.block_table.numpy(), sub.seq_lens.numpy(),
                sub.query_start_loc.numpy(), case.k_descale, case.v_descale)
        t0 = time.perf_counter()
        cw.cache_write(k_new, v_new, *args)
        elapsed += time.perf_counter() - t0
        rows += k_new.shape[0] * k_new.shape[1]
        nseq += 1
        if elapsed >= target_s:
            break
    total_rows = spec.total_q * spec.num_kv_heads
    est_s = elapsed * total_rows / max(rows, 1)
    value = total_rows * CW_ROW_BYTES / 1e9 / est_s
    return {"value": round(value, 6), "unit": "GB/s", "cores": 1, "kind": "oracle",
            "sample": f"{nseq} random whole sequences ({rows} (token, kv head) rows) in {elapsed:.1f} s; "
                      f"scaled by the workload's {total_rows} rows",
            "est_full_s": round(est_s, 6), "sample_s": round(elapsed, 6)}


def run_cache_write_reference(args, rank, world):
    if rank != 0:
        return None
    spec = _cw_spec(args)
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    case = wl.make_case(spec, device=dev, seed=0)
    kn, vn = _new_tokens(spec, dev, 0)
    per = max(1.0, min(args.cpu_seconds, 60.0 / max(1, args.steps + args.warmup)))
    for _ in range(args.warmup):
        cw_cpu_sample(spec, case, kn, vn, per / 4)
    runs = [cw_cpu_sample(spec, case, kn, vn, per) for _ in range(args.steps)]
    value = statistics.median(r["value"] for r in runs)
    est_s = statistics.median(r["est_full_s"] for r in runs)
    return {"impl": "reference", "metric": CW_METRIC, "value": round(value, 6), "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(est_s * 1e3, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32->e4m3",
            "data": "synthetic (seeded N(0,1) new K/V; the config's paged cache and block table)",
            "config": cw_config(spec, args.config, world, "n/a (CPU)"),
            "cpu_baseline": {"value": round(value, 6), "unit": "GB/s", "cores": 1, "kind": "oracle",
                             "sample": runs[-1]["sample"]},
            "e2e": {"value": round(value, 6), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


# ---------------------------------------------------------------- sparse --

SP_METRIC = "us/call and TFLOP/s of sparse paged GQA (used (row, key) pairs x 4 x 256)"


def sp_used_pairs(spec, idx):
    """(row, key) pairs the call uses: per (token, kv head) the entries in [0, causal
    limit], times the kv head's G query heads."""
    lim = torch.cat([torch.arange(L - q, L) for q, L in spec.seqs]).to(idx.device)
    used = ((idx >= 0) & (idx <= lim.view(-1, 1, 1))).sum().item()
    return int(used) * spec.group


def sp_config(spec, tp, n, l2_note, used_pairs):
    return {"workload": spec.name, "tp_shape": tp, "num_seqs": spec.num_seqs, "total_q": spec.total_q,
            "num_q_heads": spec.num_q_heads, "num_kv_heads": spec.num_kv_heads, "head_dim": wl.HEAD_DIM,
            "page_size": spec.page_size, "topk": wl.SPARSE_TOPK, "q_dtype": "bf16", "kv_dtype": "e4m3",
            "used_pairs": used_pairs, "flops": used_pairs * 4 * wl.HEAD_DIM,
            "gathered_kv_bytes": used_pairs // spec.group * 2 * wl.HEAD_DIM,
            "parallelism": f"replicas{n}", "l2": l2_note, "seed": 0}


def run_sparse(args, rank, world, local):
    import paged_gqa_gb300 as pg
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    pg.load()
    pg.paged_gqa_set_path(args.path)
    spec = wl.sparse_spec(args.sparse_tp)
    case = wl.make_case(spec, device=dev, seed=rank)
    idx = wl.sparse_indices(spec, wl.SPARSE_TOPK, device=dev, seed=rank)
    used = sp_used_pairs(spec, idx)
    flops = used * 4 * wl.HEAD_DIM
    out = torch.empty(case.q.shape[0], case.q.shape[1], wl.HEAD_DIM, dtype=torch.bfloat16, device=dev)
    flush = L2Flush(dev)

    def call(q=case.q, ix=idx, bt=case.block_table, sl=case.seq_lens, qsl=case.query_start_loc):
        pg.paged_gqa_sparse_attn(q, case.k_cache, case.v_cache, bt, sl, qsl, ix, case.k_descale,
                                 case.v_descale, case.softmax_scale, out)

    for _ in range(max(3, args.warmup)):
        call()
    assert pg.paged_gqa_check_device_errors() == 0, pg.paged_gqa_last_error()
    K = args.steps
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    sampler = ClockSampler(local)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    sampler.start()
    time.sleep(0.3)
    wall0 = time.perf_counter()
    for i in range(K):
        flush.zero_()
        ev[i][0].record()
        call()  # one kernel per call: the events bracket that kernel alone
        ev[i][1].record()
    torch.cuda.synchronize()
    wall = time.perf_counter() - wall0
    if world > 1:
        torch.distributed.barrier()
    clocks = sampler.stop()
    step_ms = sum(a.elapsed_time(b) for a, b in ev) / K
    e2e = None
    if not args.no_e2e:
        staged = PinnedInputs((case.q, idx, case.block_table, case.seq_lens, case.query_start_loc), dev)
        dev_in = staged.views
        host_out = torch.empty(out.shape, dtype=out.dtype, pin_memory=True)
        h2d = staged.nbytes

        def e2e_step():
            staged.copy()
            call(dev_in[0], dev_in[1], dev_in[2], dev_in[3], dev_in[4])
            host_out.copy_(out, non_blocking=True)

        for _ in range(3):
            e2e_step()
        torch.cuda.synchronize()
        e_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
        for i in range(K):
            flush.zero_()
            e_ev[i][0].record()
            e2e_step()
            e_ev[i][1].record()
        torch.cuda.synchronize()
        e2e = (sum(a.elapsed_time(b) for a, b in e_ev) / K, h2d, host_out.numel() * host_out.element_size())
    step_ms, e2e_ms = max_over_ranks([step_ms, e2e[0] if e2e else 0.0], world, dev)
    if rank != 0:
        return None
    _, bf16, _, peak_src = load_peaks()
    value = whole_job_value(flops / 1e12, world, step_ms)
    achieved = flops / 1e12 / (step_ms / 1e3)
    res = {
        "metric": SP_METRIC, "value": round(value, 3), "unit": "TFLOP/s", "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": round(step_ms, 5), "us_per_call": round(step_ms * 1e3, 2),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f16 (e4m3 K/V, bf16 q)",
        "data": "synthetic (seeded N(0,1) Q/K/V, FP8 per-tensor amax/448; stratified random top-k lists)",
        "config": dict(sp_config(spec, args.sparse_tp, world, L2_NOTE, used),
                       kernel_path=args.path),
        "roofline": {"bound": "tensor", "achieved": round(achieved, 2), "peak": bf16, "unit": "TFLOP/s",
                     "frac": round(achieved / bf16, 4), "peak_source": f"{peak_src} (bf16_tflops burst; f16 dense = bf16)",
                     "kernel": "sparse_tc" if pg.paged_gqa_last_plan()["path_bits"] & 32 else "sparse",
                     "kernel_us": round(step_ms * 1e3, 2),
                     "gathered_GBps": round(used // spec.group * 512 / 1e9 / (step_ms / 1e3), 1),
                     "traffic": traffic_for("sparse_tc" if pg.paged_gqa_last_plan()["path_bits"] & 32 else "sparse",
                                            spec.name)},
        "gpu_launches": K, "clocks": clocks, "wall_s": round(wall, 3),
    }
    if e2e:
        res["e2e"] = {"value": round(flops * world / 1e12 / (e2e_ms / 1e3), 3), "unit": "TFLOP/s",
                      "h2d_bytes_per_step": e2e[1], "d2h_bytes_per_step": e2e[2],
                      "note": "per step: q, indices, block_table, seq_lens, query_start_loc H2D as one transfer from one pinned buffer; out D2H; KV cache resident"}
    if world == 1 and not args.no_cpu_baseline:
        res["cpu_baseline"] = sp_cpu_sample(spec, case, idx, used, args.cpu_seconds)
    return res


def sp_cpu_sample(spec, case, idx, used, target_s):
    """The sparse oracle on growing random row samples until ~target_s; scaled by pairs."""
    import numpy as np
    import oracle
    threads = oracle.max_threads()
    c = wl.to_device(case, "cpu")
    ix = idx.cpu()
    lim = torch.cat([torch.arange(L - q, L) for q, L in spec.seqs])
    per_row = ((ix >= 0) & (ix <= lim.view(-1, 1, 1))).sum(-1)  # [T, Hkv]
    Hq, G = spec.num_q_heads, spec.group
    gen = torch.Generator().manual_seed(4321)
    n, elapsed, pairs, nrows = 16, 0.0, 0, 0
    while elapsed < target_s:
        rows = torch.randperm(spec.total_q * Hq, generator=gen)[:n].sort().values.numpy().astype(np.int64)
        t0 = time.perf_counter()
        oracle.sparse_attention(c.q, c.k_cache, c.v_cache, c.block_table, c.seq_lens, c.query_start_loc, ix,
                                q_dtype="bf16", kv_dtype="e4m3", q_descale=1.0, k_descale=case.k_descale,
                                v_descale=case.v_descale, softmax_scale=spec.softmax_scale, rows=rows,
                                threads=threads)
        elapsed += time.perf_counter() - t0
        r = torch.from_numpy(rows)
        pairs += int(per_row[r // Hq, (r % Hq) // G].sum())
        nrows += len(rows)
        n = min(spec.total_q * Hq, n * 4)
    est_s = elapsed * used / max(pairs, 1)
    value = used * 4 * wl.HEAD_DIM / 1e12 / est_s
    return {"value": round(value, 6), "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
            "sample": f"{nrows} random (token, head) rows, {pairs} used (row, key) pairs in {elapsed:.1f} s; "
                      f"scaled by the workload's {used} pairs",
            "est_full_s": round(est_s, 6), "sample_s": round(elapsed, 6)}


def run_sparse_reference(args, rank, world):
    if rank != 0:
        return None
    spec = wl.sparse_spec(args.sparse_tp)
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    case = wl.make_case(spec, device=dev, seed=0)
    idx = wl.sparse_indices(spec, wl.SPARSE_TOPK, device=dev, seed=0)
    used = sp_used_pairs(spec, idx)
    per = max(1.0, min(args.cpu_seconds, 60.0 / max(1, args.steps + args.warmup)))
    for _ in range(args.warmup):
        sp_cpu_sample(spec, case, idx, used, per / 4)
    runs = [sp_cpu_sample(spec, case, idx, used, per) for _ in range(args.steps)]
    value = statistics.median(r["value"] for r in runs)
    est_s = statistics.median(r["est_full_s"] for r in runs)
    return {"impl": "reference", "metric": SP_METRIC, "value": round(value, 6), "unit": "TFLOP/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(est_s * 1e3, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded N(0,1) Q/K/V, FP8 per-tensor amax/448; stratified random top-k lists)",
            "config": sp_config(spec, args.sparse_tp, world, "n/a (CPU)", used),
            "cpu_baseline": {"value": round(value, 6), "unit": "TFLOP/s", "cores": runs[-1]["cores"], "kind": "oracle",
                             "sample": runs[-1]["sample"]},
            "e2e": {"value": round(value, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


# ------------------------------------------------------------------- oracle --

def _oracle_sample(spec, case, target_s, kind, quant_q=False):
    """Time the oracle on growing row samples until ~target_s; scale to the workload.

    quant_q: the oracle of the quantising call (the whole Q's scale, timed once, then the
    sampled rows' attention on their e4m3 codes)."""
    import numpy as np
    import oracle
    from oracle import quant_q as qq
    threads = oracle.max_threads()
    gen = torch.Generator().manual_seed(1234)
    total_pairs = spec.flops // (4 * wl.HEAD_DIM)  # (row, visible key) pairs of the whole workload
    # sample whole sequences' rows at random, a few rows per sequence
    seq_ids = torch.randperm(spec.num_seqs, generator=gen)[: min(spec.num_seqs, 16)].tolist()
    sub = wl.subcase(case, seq_ids)
    sub = wl.to_device(sub, "cpu")
    Hq = spec.num_q_heads
    nrows_all = sub.q.shape[0] * Hq
    qsl = sub.query_start_loc.tolist()
    sl = sub.seq_lens.tolist()

    def pairs_of(rows):
        n = 0
        for r in rows:
            tok = r // Hq
            s = max(i for i in range(len(qsl) - 1) if qsl[i] <= tok)
            qn, L = qsl[s + 1] - qsl[s], sl[s]
            n += L - qn + (tok - qsl[s]) + 1
        return n

    n = 8
    elapsed, done_pairs = 0.0, 0
    rows_used = 0
    scales = None
    if quant_q:
        t0 = time.perf_counter()
        scales = qq.q_scales(case.q.float().cpu().numpy())
        elapsed += time.perf_counter() - t0
    while True:
        rows = torch.randperm(nrows_all, generator=gen)[: min(n, nrows_all)].sort().values.numpy().astype(np.int64)
        t0 = time.perf_counter()
        if quant_q:
            qq.attention_quant_q(sub.q, sub.k_cache, sub.v_cache, sub.block_table, sub.seq_lens,
                                 sub.query_start_loc, kv_dtype=spec.kv_dtype, k_descale=case.k_descale,
                                 v_descale=case.v_descale, softmax_scale=spec.softmax_scale, rows=rows,
                                 threads=threads, scales=scales)
        else:
            oracle.attention_case(sub, rows=rows, threads=threads)
        dt = time.perf_counter() - t0
        elapsed += dt
        done_pairs += pairs_of(rows.tolist())
        rows_used += len(rows)
        if elapsed >= target_s:
            break
        # grow the sample; once it covers the pool, keep timing fresh draws from it until the
        # target time is reached (a small workload can take well under target_s in full)
        n = min(nrows_all, int(n * max(2.0, min(8.0, target_s / max(dt, 1e-3)))))
    est_total_s = elapsed * total_pairs / max(done_pairs, 1)
    if kind == "hbm":
        value, unit = spec.kv_bytes / 1e9 / est_total_s, "GB/s"
    else:
        value, unit = spec.flops / 1e12 / est_total_s, "TFLOP/s"
    sample = (f"{rows_used} (token, head) row draws from {len(seq_ids)} random sequences of the workload; "
              f"{done_pairs} (row, key) pairs in {elapsed:.1f} s; scaled by the workload's {total_pairs} pairs")
    return {"value": value, "unit": unit, "cores": threads, "kind": "oracle", "sample": sample,
            "est_full_s": est_total_s, "sample_s": elapsed}


def cpu_baseline(spec, case, target_s, kind, quant_q=False):
    r = _oracle_sample(spec, case, target_s, kind, quant_q)
    return {k: (round(v, 6) if isinstance(v, float) else v) for k, v in r.items()}


def run_reference(args, rank, world):
    if rank != 0:
        return None
    spec = attn_spec(args)
    kind = workload_kind(spec)
    # structure on the host, values on the GPU if there is one (fast generation), then host copies
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    case = wl.make_case(spec, device=dev, seed=0)
    per = max(1.0, min(args.cpu_seconds, 60.0 / max(1, args.steps + args.warmup)))
    quant_q = args.op == "attn_quant_q"
    for _ in range(args.warmup):
        _oracle_sample(spec, case, per / 4, kind, quant_q)
    times, vals, last = [], [], None
    for _ in range(args.steps):
        last = _oracle_sample(spec, case, per, kind, quant_q)
        times.append(last["est_full_s"])
        vals.append(last["value"])
    est_s = statistics.median(times)
    value = statistics.median(vals)
    res = {"impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": last["unit"], "n_gpus": world,
           "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(est_s * 1e3, 3),
           "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
           "dtype": "f64", "data": "synthetic (seeded N(0,1), FP8 per-tensor amax/448)",
           "config": config_dict(spec, args.config, world, "n/a (CPU)", quant_q),
           "cpu_baseline": {"value": round(value, 6), "unit": last["unit"], "cores": last["cores"], "kind": "oracle",
                            "sample": last["sample"]},
           "e2e": {"value": round(value, 6), "unit": last["unit"], "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    return res


def main():
    args = parse()
    rank, world, local = dist_env()
    if world > 1 and args.impl == "ours":
        torch.distributed.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    if args.impl == "reference":
        res = {"cache_write": run_cache_write_reference, "sparse": run_sparse_reference}.get(
            args.op, run_reference)(args, rank, world)
    else:
        res = {"cache_write": run_cache_write, "sparse": run_sparse}.get(args.op, run_ours)(args, rank, world, local)
    if rank == 0 and res is not None:
        print(json.dumps(res), flush=True)
    if world > 1 and args.impl == "ours":
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
