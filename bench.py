"""Benchmark: paged GQA attention on GB300 through the library's C ABI.

Default workload (N=1): the MTP verify batch -- 64 sequences, q_len 4, 16 q heads /
1 kv head, head_dim 256, context lengths uniform in [1024, 32768], 16-token pages,
FP8 e4m3 K/V with per-tensor descales, bf16 Q and output. One step = one
paged_gqa_attn call (plan + attention kernels) over that batch.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--config 1..5] [--impl reference]

Prints ONE JSON line (rank 0). The value is KV-read GB/s (algorithmic bytes: each
valid token's K and V once per kv head) for verify-bound workloads and TFLOP/s
(causal-exact) for prefill-bound ones; us/call is reported beside it. Under
torchrun each rank runs an independent replica (the path shards by sequence and
kv head with no exchange), so the value is the sum over ranks divided by the
slowest rank's time.

--impl reference times the fp64 CPU oracle (the only reference this path has) on a
bounded sample of the same workload on the host cores.
"""
from __future__ import annotations

import argparse
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


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--config", type=int, default=2)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--cpu-seconds", type=float, default=15.0, help="target CPU time of the oracle sample")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    return ap.parse_args()


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


def config_dict(spec: wl.CaseSpec, idx: int, n: int, l2_note: str):
    return {"workload": spec.name, "config_index": idx, "num_seqs": spec.num_seqs, "total_q": spec.total_q,
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
    names = {"verify": ["verify_tc.cu"], "prefill": ["prefill_tc.cu"], "portable": ["portable.cu"]}[cls_kind]
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

def run_ours(args, rank, world, local):
    import paged_gqa_gb300 as pg
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    pg.load()
    spec = wl.config_spec(args.config)
    case = wl.make_case(spec, device=dev, seed=rank)  # each rank: an independent replica
    T, Hq = case.q.shape[0], case.q.shape[1]
    out = torch.empty(T, Hq, wl.HEAD_DIM, dtype=torch.bfloat16, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    kind = workload_kind(spec)
    dominant_cls = 0 if kind == "hbm" else 1
    if args.config == 5:
        dominant_cls = 1

    def call():
        pg.paged_gqa_attn(case.q, case.k_cache, case.v_cache, case.block_table, case.seq_lens,
                          case.query_start_loc, case.k_descale, case.v_descale, case.softmax_scale, out)

    for _ in range(max(3, args.warmup)):
        call()
    torch.cuda.synchronize()
    assert pg.paged_gqa_check_device_errors() == 0, pg.paged_gqa_last_error()
    plan = pg.paged_gqa_last_plan()

    K = args.steps
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
    call_ms = [a.elapsed_time(b) for a, b in ev]
    kern_ms = [a.elapsed_time(b) for a, b in kev]
    step_ms = sum(call_ms) / K
    kern_avg_ms = sum(kern_ms) / K

    # e2e: pinned host inputs -> device, call, device -> host result, every step
    e2e = None
    if not args.no_e2e:
        host_in = [t.cpu().pin_memory() for t in (case.q, case.block_table, case.seq_lens, case.query_start_loc)]
        dev_in = [torch.empty_like(t) for t in (case.q, case.block_table, case.seq_lens, case.query_start_loc)]
        host_out = torch.empty(out.shape, dtype=out.dtype, pin_memory=True)
        h2d = sum(t.numel() * t.element_size() for t in host_in)
        d2h = host_out.numel() * host_out.element_size()

        def e2e_step():
            for h, d in zip(host_in, dev_in):
                d.copy_(h, non_blocking=True)
            pg.paged_gqa_attn(dev_in[0], case.k_cache, case.v_cache, dev_in[1], dev_in[2], dev_in[3],
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
        e2e_ms = sum(a.elapsed_time(b) for a, b in e_ev) / K
        e2e = (e2e_ms, h2d, d2h)

    # reduce over ranks: max time
    step_ms, kern_avg_ms, e2e_ms = max_over_ranks([step_ms, kern_avg_ms, e2e[0] if e2e else 0.0], world, dev)
    if rank != 0:
        return None

    hbm, bf16, bf16_sus, peak_src = load_peaks()
    if kind == "hbm":
        unit, per_step = "GB/s", spec.kv_bytes / 1e9
        kern_units = spec.kv_bytes / 1e9
        peak, peak_unit = hbm, "GB/s"
        traffic_kind = "verify"
    else:
        unit, per_step = "TFLOP/s", spec.flops / 1e12
        kern_units = spec.flops / 1e12
        peak, peak_unit = 2 * bf16, "TFLOP/s"  # FP8 dense = 2 x measured bf16 (nominal ratio)
        traffic_kind = "prefill"
    value = whole_job_value(per_step, world, step_ms)
    achieved = kern_units / (kern_avg_ms / 1e3)
    used = plan["path_bits"]
    kernel_kind = traffic_kind if used & (2 << dominant_cls) else "portable"
    res = {
        "metric": METRIC, "value": round(value, 3), "unit": unit, "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": round(step_ms, 5), "us_per_call": round(step_ms * 1e3, 2),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "e4m3" if kernel_kind != "portable" else "tf32",
        "data": "synthetic (seeded N(0,1), FP8 per-tensor amax/448)",
        "config": config_dict(spec, args.config, world, "flushed: 512 MiB memset between timed calls"),
        "roofline": {"bound": kind, "achieved": round(achieved, 2), "peak": peak, "unit": peak_unit,
                     "frac": round(achieved / peak, 4), "peak_source": f"{peak_src} ({'hbm_gbs' if kind == 'hbm' else '2 x bf16_tflops burst'})",
                     "kernel": kernel_kind, "kernel_us": round(kern_avg_ms * 1e3, 2),
                     "traffic": traffic_for(kernel_kind, spec.name)},
        "gpu_launches": int(plan["kernels_launched"]) * K,
        "clocks": clocks,
        "wall_s": round(wall, 3),
    }
    if e2e:
        res["e2e"] = {"value": round(per_step * world / (e2e_ms / 1e3), 3), "unit": unit,
                      "h2d_bytes_per_step": e2e[1], "d2h_bytes_per_step": e2e[2],
                      "note": "per step: q, block_table, seq_lens, query_start_loc H2D from pinned memory; out D2H; KV cache resident"}
    if world == 1 and not args.no_cpu_baseline:
        res["cpu_baseline"] = cpu_baseline(spec, case, args.cpu_seconds, kind)
    return res


# ------------------------------------------------------------------- oracle --

def _oracle_sample(spec, case, target_s, kind):
    """Time the oracle on growing row samples until ~target_s; scale to the workload."""
    import numpy as np
    import oracle
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
    while True:
        rows = torch.randperm(nrows_all, generator=gen)[: min(n, nrows_all)].sort().values.numpy().astype(np.int64)
        t0 = time.perf_counter()
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


def cpu_baseline(spec, case, target_s, kind):
    r = _oracle_sample(spec, case, target_s, kind)
    return {k: (round(v, 6) if isinstance(v, float) else v) for k, v in r.items()}


def run_reference(args, rank, world):
    if rank != 0:
        return None
    spec = wl.config_spec(args.config)
    kind = workload_kind(spec)
    # structure on the host, values on the GPU if there is one (fast generation), then host copies
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    case = wl.make_case(spec, device=dev, seed=0)
    per = max(1.0, min(args.cpu_seconds, 60.0 / max(1, args.steps + args.warmup)))
    for _ in range(args.warmup):
        _oracle_sample(spec, case, per / 4, kind)
    times, vals, last = [], [], None
    for _ in range(args.steps):
        last = _oracle_sample(spec, case, per, kind)
        times.append(last["est_full_s"])
        vals.append(last["value"])
    est_s = statistics.median(times)
    value = statistics.median(vals)
    res = {"impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": last["unit"], "n_gpus": world,
           "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(est_s * 1e3, 3),
           "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
           "dtype": "f64", "data": "synthetic (seeded N(0,1), FP8 per-tensor amax/448)",
           "config": config_dict(spec, args.config, world, "n/a (CPU)"),
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
        res = run_reference(args, rank, world)
    else:
        res = run_ours(args, rank, world, local)
    if rank == 0 and res is not None:
        print(json.dumps(res), flush=True)
    if world > 1 and args.impl == "ours":
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
