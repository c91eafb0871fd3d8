#!/usr/bin/env python
"""Selection-latency benchmark of the GB300 PISA block selector.

One step = one full selection pass on the workload of the pages' latency
benchmark ("Block Sparse Attention with Log-Linear Complexity", §7.3: random
bf16 Q/K with a fixed seed, B=1, Hq=32, Hkv=2, d=64, C=64, K=8, g=2; timing
covers summary construction and all selection levels, not attention):
pisa_build_pyramid + pisa_select_prefill at N = 262144, causal.

Prints one JSON line (rank 0).  `value` is query-rows/s (B*N per pass) over all
ranks; `ms_per_step` the mean device time of one pass (CUDA events, L2 flushed
between passes).  `--impl reference` times the fp64 CPU oracle instead, on a
bounded sample of query rows of the same workload.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "selection ms/pass and query-rows/s at 32K–256K; % of roofline (1×GB300)"
UNIT = "query-rows/s"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
MUFU_EX2_PER_CLK_SM = 29.0  # measured ex2.approx throughput per SM and clock on GB300 (probe, 1 GPU)
kC_TOKENS = 64  # tokens per leaf (C)
L2_GATHER_TBS = 11.6  # measured rate of random 256-byte gathers served by L2 on GB300 (probe, 1 GPU), TB/s

# DRAM traffic per launch (dram__bytes_read.sum + dram__bytes_write.sum) of the
# kernels that can dominate a pass, from one ncu capture of the workload named
# (summaries under profiles/).  A figure is reported only while the kernel's
# sources, comments and blank lines aside, are identical to the ones captured.
KERNEL_SOURCES = {"leaf": ["leaf_tc.cu", "tc.cuh", "common.cuh", "api.cuh"],
                  "walk": ["walk_mma.cu", "tc.cuh", "common.cuh", "api.cuh"]}
NCU_TRAFFIC = {
    ("leaf", "latency-256k"): {"bytes": 1769379000 + 35506176, "src_sha1": "90efb4cdf3682fe708e3b2efbf32f181fad4bf1c",
                               "profile": "profiles/leaf_tc_kernel_latency-256k.md"},
    ("walk", "latency-256k"): {"bytes": 1076080000 + 34955520, "src_sha1": "78fe5a3dcf827d0c84980291f7df775ee342fd81",
                               "profile": "profiles/walk_k8s_kernel_latency-256k.md"},
}


def code_only(text):
    """CUDA source text without its comments, blank lines and runs of white space (such an
    edit leaves the compiled kernel, and so a capture of it, unchanged)."""
    import re
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    text = re.sub(r"//[^\n]*", "", text)
    return "\n".join(" ".join(line.split()) for line in text.splitlines() if line.strip())


def source_sha1(kernel, read=None):
    import hashlib
    h = hashlib.sha1()
    for f in KERNEL_SOURCES[kernel]:
        if read is None:
            with open(os.path.join(ROOT, "pyramid_top_block_gb300", "csrc", f), encoding="utf-8") as fh:
                text = fh.read()
        else:
            text = read(f)
        h.update(code_only(text).encode())
    return h.hexdigest()


def ncu_traffic(kernel, workload):
    t = NCU_TRAFFIC.get((kernel, workload))
    if t and t["src_sha1"] == source_sha1(kernel):
        return t["bytes"]
    return None


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def level_sizes(n, C=64):
    m = -(-n // C)
    out = [m]
    while m > 1:
        m = -(-m // 2)
        out.append(m)
    return out


def algorithmic(w):
    """Work model of one selection pass, as the metric defines it (non-causal upper bound).

    FLOPs = Hq*B*N*[g*K*C*2d (leaf) + (#scored intermediate levels)*g*K*g*2d]
    bytes = Q + K read once + pyramid written and read once + idx written.
    A level is scored when it has more than K candidates: with g = 2 the walk
    reaches level l with min(M_l, 2K) candidates.
    """
    B, N, Hq, Hkv, K, d, C, g = w["B"], w["N"], w["Hq"], w["Hkv"], w["K"], 64, 64, 2
    sizes = level_sizes(N, C)
    L = len(sizes)
    scored_inter = sum(1 for lvl in range(2, L) if min(sizes[lvl - 1], g * K) > K)
    leaf_scored = min(sizes[0], g * K) > K
    leaf_flops = Hq * B * N * g * K * C * 2 * d if leaf_scored else 0
    inter_flops = Hq * B * N * scored_inter * g * K * g * 2 * d
    exps = Hq * B * N * ((g * K * C if leaf_scored else 0) + scored_inter * g * K * g)
    pyr_bytes = B * Hkv * sum(sizes) * d * 4
    byts = B * N * Hq * d * 2 + B * N * Hkv * d * 2 + 2 * pyr_bytes + B * Hkv * N * K * 4
    return dict(flops=leaf_flops + inter_flops, leaf_flops=leaf_flops, inter_flops=inter_flops,
                bytes=byts, scored_intermediate_levels=scored_inter, levels=L, exps=exps,
                leaf_row_gather_bytes=B * Hkv * N * K * (Hq // Hkv) * d * 2)


class Clocks:
    """nvidia-smi sampler for the timed region."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=self.fh, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.15)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.fh.close()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    rows.append(dict(sm=float(parts[1]), smax=float(parts[2]),
                                     power=float(parts[3]) if parts[3] not in ("[N/A]", "") else 0.0,
                                     hw=parts[5], hwt=parts[6], swt=parts[7], swp=parts[8]))
                except ValueError:
                    continue
        os.unlink(self.path)
        if not rows:
            return None
        reasons = set()
        for r in rows:
            for key, name in (("hw", "hw_slowdown"), ("hwt", "hw_thermal_slowdown"),
                              ("swt", "sw_thermal_slowdown"), ("swp", "sw_power_cap")):
                if r[key].lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(r["sm"] for r in rows), "sm_max_mhz": max(r["smax"] for r in rows),
                "reasons": sorted(reasons), "samples": len(rows),
                "power_w_max": max(r["power"] for r in rows)}


def max_over_ranks(x, dist, device):
    """The slowest rank's value (every rank gets it)."""
    if dist is None:
        return x
    import torch
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_rows_per_s(world, rows_per_rank, ms):
    """Whole-job throughput: every rank processes rows_per_rank rows; the job takes
    the slowest rank's ms."""
    return world * rows_per_rank / (ms / 1000.0)


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def oracle_rows_per_s(q, k, w, target_s: float, n_rows: int | None = None, threads: int = 0):
    """Time the fp64 oracle (as it stands, all host threads) on a bounded sample:
    its pyramid build over all N tokens, plus the walks of n query rows (all KV
    heads) spread evenly over the sequence.  A full pass is then
    t_build + (B*N) * t_row, and the value is B*N over that time."""
    import oracle
    oracle.build()
    N = w["N"]
    kf = k.float().numpy()
    t0 = time.perf_counter()
    oracle.build_pyramid(kf)
    t_build = time.perf_counter() - t0

    def run(n):
        t = np.unique(np.linspace(0, N - 1, n).round().astype(np.int64))
        qr = q[:, t].float().numpy()
        t0 = time.perf_counter()
        oracle.select(qr, kf, K=w["K"], t_list=t, threads=threads)
        return len(t), max(time.perf_counter() - t0 - t_build, 1e-9)

    # grow the sample until it takes about target_s (per-row cost from a small
    # sample is inflated by fixed start-up costs)
    budget = max(target_s - t_build, 0.2)
    if n_rows:
        n, secs = run(n_rows)
    else:
        n, secs = run(64)
        while secs < 0.7 * budget and n < N:
            n, secs = run(int(min(N, n * min(8.0, max(1.5, budget / secs)))))
    t_row = secs / (n * w["B"])
    t_full = t_build + w["B"] * N * t_row
    return dict(value=w["B"] * N / t_full, unit=UNIT, cores=threads or oracle.max_threads(), kind="oracle",
                extrapolated=n < N, rows_timed=n * w["B"], seconds_timed=round(secs + t_build, 3),
                full_pass_s_extrapolated=round(t_full, 2), rows=n * w["B"],
                sample=f"fp64 pyramid build over all N={N} tokens ({t_build:.2f} s) + walks of {n} query "
                       f"rows x {w['Hkv']} KV heads evenly spaced over the sequence ({secs:.2f} s); "
                       f"value = B*N / (build + B*N x measured seconds per row)"
                       + (f": an extrapolation to a full pass ({t_full:.1f} s), not a timed full pass"
                          if n < N else " (every row walked)"))


def run_reference(args):
    world, rank, _ = dist_setup()
    if rank != 0:
        return 0
    from pyramid_top_block_gb300 import synth
    q, k, w = synth.make(args.workload)
    vals = []
    secs = []
    info = None
    per_step = max(0.5, min(args.ref_step_s, 150.0 / (args.warmup + args.steps)))
    n_rows = None
    for i in range(args.warmup + args.steps):
        r = oracle_rows_per_s(q, k, w, target_s=per_step, n_rows=n_rows)
        n_rows = r["rows"] // w["B"]  # the first step sizes the sample, the others reuse it
        if i >= args.warmup:
            vals.append(r["value"])
            secs.append(r["seconds_timed"])
            info = r
    value = statistics.mean(vals)
    # a step is one bounded sample (pyramid build + a fixed set of query rows); ms_per_step is
    # its measured wall time, and value extrapolates the sample's per-row cost to a full pass
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1000.0 * statistics.mean(secs),
            "extrapolated": True, "rows_timed_per_step": info["rows_timed"],
            "full_pass_ms_extrapolated": 1000.0 * w["B"] * w["N"] / value,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": cfg(w, args),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": info["cores"], "kind": "oracle",
                             "extrapolated": True, "rows_timed": info["rows_timed"],
                             "seconds_timed": info["seconds_timed"], "sample": info["sample"]},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def cfg(w, args):
    return {"workload": args.workload, "B": w["B"], "N": w["N"], "Hq": w["Hq"], "Hkv": w["Hkv"], "d": 64,
            "C": 64, "g": 2, "K": w["K"], "causal": True, "seed": w["seed"],
            "inputs": "bf16 i.i.d. N(0,1) Q/K" if w["kind"] == "iid" else "bf16 structured",
            "l2": "flushed between timed passes (256 MiB write)", "accumulate": "fp32"}


def run_ours(args):
    import torch
    import pyramid_top_block_gb300 as pisa
    from pyramid_top_block_gb300 import synth

    world, rank, local = dist_setup()
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    pk, pk_kind = peaks()
    q, k, w = synth.make(args.workload)
    alg = algorithmic(w)
    K = w["K"]
    lib = pisa.load()
    qd, kd = q.to(dev), k.to(dev)
    pyr = pisa.Pyramid.allocate(kd)
    B, N, Hq, Hkv = w["B"], w["N"], w["Hq"], w["Hkv"]
    ws = torch.empty(pisa.select_workspace_bytes(B, N, Hq, Hkv, K), dtype=torch.uint8, device=dev)
    idx = torch.empty(B, Hkv, N, K, dtype=torch.int32, device=dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()
    phases = pisa.prefill_phases()

    def step(ev_build=None):
        pisa.build_pyramid(pyr)
        if ev_build is not None:
            ev_build.record(stream)
        pisa.select_prefill(qd, pyr, K, workspace=ws, out=(idx, None), with_scores=False)

    for _ in range(args.warmup):
        flush.zero_()
        step()
    torch.cuda.synchronize()

    n = args.steps
    mk = lambda: torch.cuda.Event(enable_timing=True)
    ev_s = [mk() for _ in range(n)]
    ev_e = [mk() for _ in range(n)]
    ev_b = [mk() for _ in range(n)]
    ev_p = [[mk() for _ in range(len(phases) + 1)] for _ in range(n)]
    for evs in ev_p:  # torch creates the CUDA event at its first record
        for e in evs:
            e.record(stream)
    torch.cuda.synchronize()
    clocks = Clocks(local) if rank == 0 else None
    if clocks:
        clocks.start()
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    launches0 = pisa.kernel_launches()
    for i in range(n):
        flush.zero_()
        pisa.set_phase_events(ev_p[i])
        ev_s[i].record(stream)
        step(ev_b[i])
        ev_e[i].record(stream)
    torch.cuda.synchronize()
    launches = pisa.kernel_launches() - launches0
    device_status = pisa.check_device_status(ws)
    pisa.set_phase_events(None)
    if dist:
        dist.barrier()
    clk = clocks.stop() if clocks else None
    ms = [ev_s[i].elapsed_time(ev_e[i]) for i in range(n)]
    total = max_over_ranks(sum(ms), dist, dev)
    ms_step = total / n
    value = job_rows_per_s(world, B * N, ms_step)
    phase_ms = {"build": statistics.mean(ev_s[i].elapsed_time(ev_b[i]) for i in range(n))}
    for j, name in enumerate(phases):
        phase_ms[name] = statistics.mean(pisa.event_elapsed_ms(ev_p[i][j], ev_p[i][j + 1]) for i in range(n))

    # dominant kernel roofline (algorithmic work of that kernel / its event time)
    tf_peak = pk["bf16_tflops"]
    dom = max(("walk", "leaf"), key=lambda k: phase_ms.get(k, 0.0))
    fl = alg["leaf_flops"] if dom == "leaf" else alg["inter_flops"]
    achieved = fl / (phase_ms[dom] / 1e3) / 1e12
    roof = {"bound": "tensor", "achieved": achieved, "peak": tf_peak, "unit": "TFLOP/s",
            "frac": achieved / tf_peak, "traffic": ncu_traffic(dom, args.workload), "kernel": dom,
            "peak_source": f"{pk_kind} bf16 burst"}
    t_tensor = alg["flops"] / (tf_peak * 1e12) * 1e3
    t_hbm = alg["bytes"] / (pk["hbm_gbs"] * 1e9) * 1e3
    ms_stats = {"mean": ms_step, "median": statistics.median(ms), "min": min(ms), "runs": n}
    rates = {"query_rows_per_s": value, "kv_rows_per_s": value * Hkv, "head_rows_per_s": value * Hq}
    work = {"exps": alg["exps"], "leaf_row_gather_bytes": alg["leaf_row_gather_bytes"],
            "note": "the metric's work model (non-causal upper bound); leaf_row_gather_bytes = query rows "
                    "gathered once per (query, KV head, level-2 survivor)"}
    # informative third bound (not part of the metric's roofline): the work model's
    # exponentials at the exponential unit's rate measured on this GPU (ex2 ~29 per clock
    # per SM, 152 SMs at 2.07 GHz)
    t_exp = alg["exps"] / (MUFU_EX2_PER_CLK_SM * 152 * 2.07e9) * 1e3
    # and the leaf stage's query-row gathers at the measured L2 random-gather rate
    t_l2 = alg["leaf_row_gather_bytes"] / (L2_GATHER_TBS * 1e12) * 1e3
    pass_roof = {"flops": alg["flops"], "min_bytes": alg["bytes"], "t_tensor_ms": t_tensor, "t_hbm_ms": t_hbm,
                 "t_roofline_ms": max(t_tensor, t_hbm), "frac": max(t_tensor, t_hbm) / ms_step,
                 "peaks": f"{pk_kind}: {tf_peak} TFLOP/s bf16 burst, {pk['hbm_gbs']} GB/s",
                 "t_exp_ms": t_exp, "t_l2_gather_ms": t_l2,
                 "frac_with_exp_bound": max(t_tensor, t_hbm, t_exp) / ms_step}

    # end to end through the public API with host buffers (pinned): every step copies K and
    # Q in and the indices out (pisa_select_prefill_host overlaps the copies with the
    # selection, query chunk by query chunk), timed on the compute stream, which the call
    # orders after its last copy
    e2e = None
    if not args.no_e2e:
        qh = q.pin_memory()
        kh = k.pin_memory()
        idx_h = torch.empty(idx.shape, dtype=idx.dtype).pin_memory()

        def e2e_step():
            pisa.select_prefill_host(qh, kh, pyr, K, causal=True, idx_host=idx_h, q_dev=qd, idx_dev=idx,
                                     workspace=ws, stream=stream)

        # this box's plain pinned host->device rate (it differs between boxes), for the floor
        # that the transfers alone put under the end-to-end step
        qd.copy_(qh, non_blocking=True)
        torch.cuda.synchronize()
        hs, he = mk(), mk()
        hs.record(stream)
        for _ in range(3):
            qd.copy_(qh, non_blocking=True)
        he.record(stream)
        torch.cuda.synchronize()
        h2d_gbs = 3 * qh.numel() * 2 / (hs.elapsed_time(he) * 1e6)
        for _ in range(2):
            e2e_step()
        torch.cuda.synchronize()
        ne = max(3, min(n, 20))
        es, ee = mk(), mk()
        if dist:
            dist.barrier()
        torch.cuda.synchronize()
        t_wall = time.perf_counter()
        es.record(stream)
        for _ in range(ne):
            e2e_step()
        ee.record(stream)
        torch.cuda.synchronize()
        wall_ms = (time.perf_counter() - t_wall) * 1e3 / ne
        e_ms = max_over_ranks(es.elapsed_time(ee) / ne, dist, dev)
        e2e = {"value": job_rows_per_s(world, B * N, e_ms), "unit": UNIT, "ms_per_step": e_ms,
               "wall_ms_per_step": wall_ms, "api": "pisa_select_prefill_host",
               "h2d_gbs_measured": h2d_gbs,
               "transfer_floor_ms": (qh.numel() * 2 + kh.numel() * 2) / (h2d_gbs * 1e6),
               "h2d_bytes_per_step": qh.numel() * 2 + kh.numel() * 2,
               "d2h_bytes_per_step": idx_h.numel() * 4}

    decode = None
    if not args.no_decode and rank == 0:
        decode = bench_decode(torch, pisa, synth, dev, args)

    modes = None
    if args.modes and rank == 0:
        modes = {}
        for m in (1, 2):
            ms_m = []
            for i in range(max(3, min(n, 10)) + 2):
                flush.zero_()
                a, b = mk(), mk()
                a.record(stream)
                pisa.build_pyramid(pyr)
                pisa.select_prefill(qd, pyr, K, workspace=ws, out=(idx, None), with_scores=False, mode=m)
                b.record(stream)
                torch.cuda.synchronize()
                if i >= 2:
                    ms_m.append(a.elapsed_time(b))
            modes[["lse", "mean", "mean_half_var"][m]] = {"ms_median": statistics.median(ms_m),
                                                          "status": pisa.check_device_status(ws)}

    attention = None
    if args.attention and rank == 0:
        # stage two over this pass's selection, with seeded random values
        gv = torch.Generator().manual_seed(3)
        vd = torch.randn(B, N, Hkv, 64, generator=gv).to(torch.bfloat16).to(dev)
        att_out = torch.empty(B, N, Hq, 64, dtype=torch.float32, device=dev)
        step()
        ms_a = []
        for i in range(7):
            flush.zero_()
            a, b = mk(), mk()
            a.record(stream)
            pisa.sparse_attention(qd, kd, vd, idx, out=att_out)
            b.record(stream)
            torch.cuda.synchronize()
            if i >= 2:
                ms_a.append(a.elapsed_time(b))
        t_att = statistics.median(ms_a)
        fl = 4.0 * B * N * Hq * K * 64 * 64  # QK^T and PV over K full leaves (upper bound)
        attention = {"ms_median": t_att, "forward_ms": ms_step + t_att, "tflops_upper_bound": fl / t_att / 1e9,
                     "note": "stage two over the pass's idx, random bf16 V, fp32 output"}
        del vd, att_out

    per_config = None
    if args.configs and rank == 0:
        per_config = {}
        for name in args.configs.split(","):
            per_config[name] = bench_config(torch, pisa, synth, dev, name, pk, runs=20,
                                            cpu_s=0.0 if args.no_cpu_baseline else args.cfg_cpu_s)

    flat = None
    if args.flat and rank == 0:
        flat = [bench_flat(torch, pisa, synth, dev, name) for name in args.flat.split(",")]

    cpu = None
    if not args.no_cpu_baseline and rank == 0 and world == 1:
        cpu = oracle_rows_per_s(q, k, w, target_s=args.cpu_s)
        cpu.pop("seconds", None)
        cpu.pop("rows", None)

    if rank == 0:
        line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": n,
                "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
                "vs_baseline": None, "dtype": "bf16", "data": "synthetic", "config": cfg(w, args),
                "roofline": roof, "roofline_pass": pass_roof, "phases_ms": phase_ms, "ms_stats": ms_stats,
                "rates": rates, "work": work,
                "cpu_baseline": cpu, "e2e": e2e, "gpu_launches": launches, "clocks": clk,
                "device_status": device_status,
                "per_config": per_config, "decode": decode, "flat": flat, "score_modes": modes,
                "attention": attention}
        print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()
    return 0


def bench_config(torch, pisa, synth, dev, name, pk, runs, cpu_s):
    """One more workload of the metric's range: median / min ms of a full pass
    (pyramid build + selection, L2 flushed between passes), query-rows/s, the pass
    against its roofline, and the oracle on the host cores (all of them; also one
    thread up to 32K tokens) on a bounded sample of the same workload."""
    q, k, w = synth.make(name)
    B, N, Hq, Hkv, K = w["B"], w["N"], w["Hq"], w["Hkv"], w["K"]
    qd, kd = q.to(dev), k.to(dev)
    pyr = pisa.Pyramid.allocate(kd)
    ws = torch.empty(pisa.select_workspace_bytes(B, N, Hq, Hkv, K), dtype=torch.uint8, device=dev)
    idx = torch.empty(B, Hkv, N, K, dtype=torch.int32, device=dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()
    ms = []
    for i in range(runs + 3):
        flush.zero_()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        pisa.build_pyramid(pyr)
        pisa.select_prefill(qd, pyr, K, workspace=ws, out=(idx, None), with_scores=False)
        b.record(stream)
        torch.cuda.synchronize()
        if i >= 3:
            ms.append(a.elapsed_time(b))
    st = pisa.check_device_status(ws)
    alg = algorithmic(w)
    t_tensor = alg["flops"] / (pk["bf16_tflops"] * 1e12) * 1e3
    t_hbm = alg["bytes"] / (pk["hbm_gbs"] * 1e9) * 1e3
    med = statistics.median(ms)
    out = {"B": B, "N": N, "Hq": Hq, "Hkv": Hkv, "K": K, "ms_median": med, "ms_min": min(ms), "runs": runs,
           "query_rows_per_s": B * N / (med / 1e3), "status": st,
           "roofline_pass": {"t_tensor_ms": t_tensor, "t_hbm_ms": t_hbm, "t_roofline_ms": max(t_tensor, t_hbm),
                             "frac": max(t_tensor, t_hbm) / med}}
    del qd, kd, pyr, ws, idx, flush
    if cpu_s > 0:
        o = oracle_rows_per_s(q, k, w, target_s=cpu_s)
        out["oracle"] = {x: o[x] for x in ("value", "cores", "extrapolated", "rows_timed", "seconds_timed")}
        if N <= 32768:
            o1 = oracle_rows_per_s(q, k, w, target_s=cpu_s, threads=1)
            out["oracle_1thread"] = {x: o1[x] for x in ("value", "cores", "extrapolated", "rows_timed",
                                                        "seconds_timed")}
    return out


def bench_flat(torch, pisa, synth, dev, name, runs=5):
    """The flat selector (every eligible leaf scored exactly, the conventional
    baseline) against the pyramid pass on the same workload: ms per selection
    (build included for the pyramid), and the synthetic Recall@K of the pyramid's
    blocks in the flat selector's, over query positions with more than K eligible
    leaves (random inputs: not the pages' full-attention diagnostic)."""
    q, k, w = synth.make(name)
    B, N, Hq, Hkv, K = w["B"], w["N"], w["Hq"], w["Hkv"], w["K"]
    qd, kd = q.to(dev), k.to(dev)
    del q, k
    pyr = pisa.Pyramid.allocate(kd)
    ws = torch.empty(pisa.select_workspace_bytes(B, N, Hq, Hkv, K), dtype=torch.uint8, device=dev)
    wf = torch.empty(pisa.flat_workspace_bytes(B, N, Hq, Hkv, K), dtype=torch.uint8, device=dev)
    ip = torch.empty(B, Hkv, N, K, dtype=torch.int32, device=dev)
    iflat = torch.empty_like(ip)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()

    def timed(fn):
        out = []
        for i in range(runs + 2):
            flush.zero_()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            fn()
            b.record(stream)
            torch.cuda.synchronize()
            if i >= 2:
                out.append(a.elapsed_time(b))
        return statistics.median(out)

    def pyr_pass():
        pisa.build_pyramid(pyr)
        pisa.select_prefill(qd, pyr, K, workspace=ws, out=(ip, None), with_scores=False)

    t_pyr = timed(pyr_pass)
    t_flat = timed(lambda: pisa.select_flat(qd, pyr, K, workspace=wf, out=(iflat, None), with_scores=False))
    st = pisa.check_device_status(wf)
    a, b = ip.cpu(), iflat.cpu()
    t = torch.arange(N)
    rows = (t // 64 + 1) > K  # more than K eligible leaves
    hit = (a.unsqueeze(-1) == b.unsqueeze(-2)) & (a.unsqueeze(-1) >= 0)
    recall = hit.any(-1).sum(-1).float() / K  # [B, Hkv, N]
    return {"workload": name, "N": N, "K": K, "pyramid_ms": t_pyr, "flat_ms": t_flat,
            "flat_over_pyramid": t_flat / t_pyr, "recall_at_k": float(recall[:, :, rows].mean()),
            "recall_rows": int(rows.sum()) * B * Hkv, "status": st}


def bench_decode(torch, pisa, synth, dev, args):
    """µs per decode step: 16 sequences with a 131072-token cached pyramid,
    Hq=32, Hkv=2, K=8; each step appends one key per sequence and selects."""
    B, Hq, Hkv, K, n_ctx, steps = 16, 32, 2, 8, 131072, args.decode_steps
    n_cap = n_ctx + steps + 8
    cache, g = synth.decode_context(B, n_ctx, n_cap, Hkv, seed=2)
    pyr = pisa.Pyramid.allocate(cache.to(dev), with_lengths=True)
    del cache
    pisa.build_pyramid(pyr, N=n_ctx)
    qs, ks = [], []
    for _ in range(steps):
        a, b = synth.decode_step(g, B, Hq, Hkv)
        qs.append(a)
        ks.append(b)
    qd = torch.stack(qs).to(dev)
    kd = torch.stack(ks).to(dev)
    ws = torch.empty(pisa.decode_workspace_bytes(B, Hq, Hkv, K), dtype=torch.uint8, device=dev)
    idx = torch.empty(B, Hkv, K, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream()
    torch.cuda.synchronize()
    es, ee = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    es.record(stream)
    for s in range(steps):
        pisa.decode_append_and_select(qd[s], kd[s], pyr, K, workspace=ws, out=(idx, None), with_scores=False)
    ee.record(stream)
    torch.cuda.synchronize()
    st = pisa.check_device_status(ws)
    us_eager = es.elapsed_time(ee) * 1000.0 / steps
    # the same steps captured once in a CUDA graph and replayed (a fresh cache)
    cache, g = synth.decode_context(B, n_ctx, n_cap, Hkv, seed=2)
    pyr_g = pisa.Pyramid.allocate(cache.to(dev), with_lengths=True)
    del cache
    pisa.build_pyramid(pyr_g, N=n_ctx)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=side):
        for s in range(steps):
            pisa.decode_append_and_select(qd[s], kd[s], pyr_g, K, workspace=ws, out=(idx, None), with_scores=False)
    torch.cuda.synchronize()
    es.record(stream)
    graph.replay()
    ee.record(stream)
    torch.cuda.synchronize()
    # byte floor of a step: per (sequence, KV head) the keys of the 2K leaf candidates, the children
    # rows of 2K candidates at each scored level (fp32 summaries) and the path's siblings and new
    # means, at the HBM copy rate
    levels = len(level_sizes(n_ctx + 1))
    per_bh = 2 * K * kC_TOKENS * 64 * 2 + (levels - 2) * 2 * (2 * K) * 64 * 4 + 2 * levels * 64 * 4
    step_bytes = B * Hkv * per_bh
    return {"us_per_step": us_eager, "us_per_step_graph": es.elapsed_time(ee) * 1000.0 / steps, "steps": steps,
            "B": B, "n_ctx": n_ctx, "Hq": Hq, "Hkv": Hkv, "K": K, "status": st,
            "status_graph": pisa.check_device_status(ws),
            "bytes_per_step_model": step_bytes,
            "byte_floor_us": step_bytes / (peaks()[0]["hbm_gbs"] * 1e9) * 1e6}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="latency-256k")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-decode", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--attention", type=int, default=1, help="also time stage-two attention on the selection")
    ap.add_argument("--modes", type=int, default=1, help="also time the PISA-1 / PISA-2 score modes")
    ap.add_argument("--flat", default="latency-4k,latency-8k,latency-16k,latency-32k,latency-64k,latency-128k,"
                                      "latency-256k",
                    help="comma-separated workloads for the flat-selector comparison ('' to skip)")
    ap.add_argument("--configs", default="tiny-2k,latency-32k,latency-64k,latency-128k,ragged-16421",
                    help="comma-separated workloads also timed (per_config; '' to skip)")
    ap.add_argument("--cfg-cpu-s", type=float, default=3.0, help="seconds of oracle work per per_config entry")
    ap.add_argument("--cpu-s", type=float, default=12.0, help="seconds of oracle work for cpu_baseline")
    ap.add_argument("--ref-step-s", type=float, default=6.0, help="seconds of oracle work per reference step")
    ap.add_argument("--decode-steps", type=int, default=256)
    args = ap.parse_args()
    from pyramid_top_block_gb300 import synth
    if args.workload not in synth.WORKLOADS:
        raise SystemExit(f"unknown workload {args.workload}")
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
