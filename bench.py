#!/usr/bin/env python
"""Benchmark of the relative-position memory attention hot path.

Workload: one layer's forward + backward at B=16, H=16, L=512, M=512 (memory
full), d_h=64, bf16 inputs with fp32 accumulation; synthetic seeded inputs
with the distributions of that configuration. A step = rxl_attn_fwd +
rxl_attn_bwd over that batch.

Throughput counts algorithmic work only: visible pairs N = B*H*(L*m +
L(L+1)/2); forward 6*d_h = 384 flop per pair (three d_h-long products: the
content score, the position score, P.V), backward 12*d_h = 768 flop per pair
(dV, dP, dQ-content, dQ-position, dK, dR); recomputation is not counted.

Timing: W untimed warm-up steps, then K steps, each bracketed by CUDA events
on the launching stream, with the L2 flushed (a 256 MiB write) between steps
outside the events; barrier + synchronize around the timed region, max over
ranks. Under torchrun every rank runs its own copy of the workload (the
path's (b,h) units are independent: weak scaling, no collective).

--impl reference times the float64 CPU oracle on a bounded sample of the
same workload (the only comparison program this path has).
"""
from __future__ import annotations

import argparse
import json
import math
import os
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "rel-pos mem-attention fwd+bwd TFLOP/s & tokens/s vs bf16 tensor-core peak"
WORKLOAD = "cfg3_bf16_B16H16_L512M512_dh64_fwd+bwd"
B, H, L, M, DH = 16, 16, 512, 512, 64
SCALE = 1.0 / math.sqrt(DH)
FLOP_FWD_PAIR, FLOP_BWD_PAIR = 6 * DH, 12 * DH
# The backward main kernel's sources: a DRAM-traffic record in its profile
# summary counts only while these files are unchanged since the capture.
BWD_MAIN_SOURCES = ("long_context_lm_rel_gb300/csrc/attn_bwd_tc.cu", "long_context_lm_rel_gb300/csrc/tc_common.cuh",
                    "long_context_lm_rel_gb300/csrc/sm103.cuh")
BWD_MAIN_PROFILE = "profiles/bwd_main_kernel_B4H16L512M512.md"


def code_of(text):
    """C/CUDA source with its comments and blank space taken out (string
    literals kept), so that the hash below follows the code alone."""
    out, i, n = [], 0, len(text)
    while i < n:
        c = text[i]
        if c == '"':
            j = i + 1
            while j < n and text[j] != '"':
                j += 2 if text[j] == "\\" else 1
            out.append(text[i:j + 1])
            i = j + 1
        elif text.startswith("//", i):
            j = text.find("\n", i)
            i = n if j < 0 else j
        elif text.startswith("/*", i):
            j = text.find("*/", i + 2)
            i = n if j < 0 else j + 2
        else:
            out.append(c)
            i += 1
    return " ".join("".join(out).split())


def sources_sha256(paths):
    """sha256 of the code (comments and blank space aside) of `paths`."""
    import hashlib
    h = hashlib.sha256()
    for rel in paths:
        with open(os.path.join(ROOT, rel), encoding="utf-8") as f:
            h.update(code_of(f.read()).encode())
    return h.hexdigest()


def traffic_record(profile, sources):
    """(bytes per launch at the profile's batch, batch) from the profile's
    'traffic-record:' line if its source hash matches the current sources,
    else (None, reason)."""
    try:
        with open(os.path.join(ROOT, profile)) as f:
            lines = [ln for ln in f if ln.startswith("traffic-record:")]
    except OSError:
        return None, "no profile"
    if not lines:
        return None, "no traffic record in the profile"
    rec = dict(kv.split("=", 1) for kv in lines[-1].split(":", 1)[1].split())
    if rec.get("sha256") != sources_sha256(sources):
        return None, "the kernel changed since the capture"
    return (float(rec["bytes_per_launch"]), int(rec["batch"])), None


def visible_pairs(b, h, l, m):
    return b * h * (l * m + l * (l + 1) // 2)


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return float(p["bf16_tflops"]), float(p["hbm_gbs"]), "measured"
    except Exception:
        return 1900.0, 6800.0, "fallback"


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled during the timed region."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index, self.lines, self.proc = index, [], None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except Exception:
            self.proc = None
        time.sleep(0.3)
        return self

    def _read(self):
        for ln in self.proc.stdout:
            self.lines.append(ln.strip())

    def __exit__(self, *a):
        time.sleep(0.3)
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 8:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for n, v in zip(names, f[4:8]):
                if v.lower() in ("active", "1"):
                    reasons.add(n)
        sm.sort()
        return {"sm_mhz": sm[len(sm) // 2] if sm else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm)}


def make_inputs(seed=0):
    import dataclasses

    import rxl_inputs as gen
    w = dataclasses.replace(gen.CFG3, seed=seed, B=B)
    p, s, mem = gen.layer_params(w), gen.segment_inputs(w), gen.initial_memory(w)
    return dict(q=s["q"], k_mem=mem["k_mem"], k_cur=s["k_cur"], v_mem=mem["v_mem"], v_cur=s["v_cur"],
                u=p["u"], vb=p["vb"], r=p["r"], do=s["do"])


def cpu_sample(x, units_heads, nthreads):
    """Oracle fwd+bwd on the heads `units_heads` (all batch rows); returns
    (seconds, algorithmic flop of the sample)."""
    import numpy as np
    import oracle
    k = np.concatenate([x["k_mem"], x["k_cur"]], 2)
    v = np.concatenate([x["v_mem"], x["v_cur"]], 2)
    hs = slice(units_heads[0], units_heads[1])
    t0 = time.perf_counter()
    oracle.fwd(x["q"][:, hs], k[:, hs], v[:, hs], x["r"][hs], x["u"][hs], x["vb"][hs], SCALE, nthreads=nthreads)
    oracle.bwd(x["q"][:, hs], k[:, hs], v[:, hs], x["r"][hs], x["u"][hs], x["vb"][hs], x["do"][:, hs], SCALE,
               nthreads=nthreads)
    dt = time.perf_counter() - t0
    nh = units_heads[1] - units_heads[0]
    return dt, visible_pairs(B, nh, L, M) * (FLOP_FWD_PAIR + FLOP_BWD_PAIR)


def run_reference(args, rank, world):
    if rank != 0:
        return
    x = make_inputs()
    nthreads = os.cpu_count() or 1
    heads = (0, 1)                  # one head, all 16 batch rows: 16 (b,h) units per step
    for _ in range(args.warmup):
        cpu_sample(x, heads, nthreads)
    tot_s, tot_f = 0.0, 0.0
    for _ in range(args.steps):
        dt, fl = cpu_sample(x, heads, nthreads)
        tot_s += dt
        tot_f += fl
    value = tot_f / tot_s / 1e12
    pairs = visible_pairs(B, 1, L, M)
    sample = f"fwd+bwd of 1 head x {B} batch rows ({pairs} visible pairs) of the workload per step"
    out = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * tot_s / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "tokens_per_s": args.steps * B * L / 16 / tot_s,
        "config": {"workload": WORKLOAD, "B": B, "H": H, "L": L, "M": M, "dh": DH, "sample": sample},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": min(nthreads, B), "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(out), flush=True)


def run_ours(args, rank, world):
    import numpy as np
    import torch
    import torch.distributed as dist

    import long_context_lm_rel_gb300 as rxl
    from long_context_lm_rel_gb300.multirank import max_over_ranks, replica_seed, whole_job_rate
    from long_context_lm_rel_gb300.calls import AttnCall, place_kv

    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    rxl.lib()
    x = make_inputs(replica_seed(0, rank))   # one independent replica per rank
    cap = m = M
    c = AttnCall(x["q"], place_kv(x["k_mem"], x["k_cur"], cap, 0), place_kv(x["v_mem"], x["v_cur"], cap, 0),
                 x["r"], x["u"], x["vb"], cap=cap, m=m, head=0, dtype="bf16", scale=SCALE).alloc_bwd(x["do"])
    stream = torch.cuda.current_stream()
    flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")

    # the training pair: the forward keeps the low part of O for the backward
    def step():
        c.fwd_ex(stream)
        n = rxl.rxl_last_launch_count()
        c.bwd_ex(stream)
        return n + rxl.rxl_last_launch_count()

    for _ in range(max(args.warmup, 0)):
        step()
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    # One event pair per step and none inside it: an event recorded between
    # the forward and the backward would stop the backward's first kernel
    # from starting while the forward's last CTAs finish.
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(args.steps)]
    launches = 0
    with ClockSampler(local) as clk:
        torch.cuda.synchronize()
        for e in ev:
            flush.zero_()                 # L2 flush, outside the timed events
            e[0].record(stream)
            c.fwd_ex(stream)
            launches += rxl.rxl_last_launch_count()
            c.bwd_ex(stream)
            launches += rxl.rxl_last_launch_count()
            e[1].record(stream)
        torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    step_ms = [e[0].elapsed_time(e[1]) for e in ev]
    tot_ms = max_over_ranks(sum(step_ms), world, device="cuda")
    # the forward / backward split: the same steps again with an event
    # between the two calls (reported beside the headline, not part of it)
    ev3 = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    torch.cuda.synchronize()
    for e in ev3:
        flush.zero_()
        e[0].record(stream)
        c.fwd_ex(stream)
        e[1].record(stream)
        c.bwd_ex(stream)
        e[2].record(stream)
    torch.cuda.synchronize()
    fwd_ms = [e[0].elapsed_time(e[1]) for e in ev3]
    bwd_ms = [e[1].elapsed_time(e[2]) for e in ev3]

    pairs = visible_pairs(B, H, L, m)
    flop_step = pairs * (FLOP_FWD_PAIR + FLOP_BWD_PAIR)
    value = whole_job_rate(args.steps * flop_step, world, tot_ms * 1e-3) / 1e12
    tokens = whole_job_rate(args.steps * B * L, world, tot_ms * 1e-3)

    # end to end through the C ABI from pinned host buffers: inputs H2D, fwd,
    # bwd, every output D2H, each step
    host_in = {n: getattr(c, n).cpu().pin_memory() for n in ("q", "k", "v", "r", "u", "vb", "do")}
    host_out = {n: torch.empty_like(getattr(c, n), device="cpu").pin_memory()
                for n in ("o", "lse", "dq", "dk", "dv", "dr", "du", "dvb")}
    h2d = sum(t.numel() * t.element_size() for t in host_in.values())
    d2h = sum(t.numel() * t.element_size() for t in host_out.values())

    # End to end through the C ABI from pinned host buffers, every step:
    # inputs host -> device, fwd, bwd, every output device -> host. As an
    # input pipeline would, the steps overlap: step n+1's inputs are copied on
    # one copy stream while step n computes and step n-1's outputs are read
    # back on another; two device buffer sets (and two host output sets)
    # alternate. All of every step's copies are inside the timed region.
    sets = [c, AttnCall(x["q"], place_kv(x["k_mem"], x["k_cur"], cap, 0),
                        place_kv(x["v_mem"], x["v_cur"], cap, 0), x["r"], x["u"], x["vb"], cap=cap, m=m,
                        head=0, dtype="bf16", scale=SCALE).alloc_bwd(x["do"])]
    for cs in sets:
        cs.fwd_ex(stream)   # allocates the low part of O
    host_outs = [host_out, {n: torch.empty_like(t).pin_memory() for n, t in host_out.items()}]
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()

    def e2e_run(nsteps):
        start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        ev_in = [torch.cuda.Event() for _ in range(nsteps)]
        ev_comp = [torch.cuda.Event() for _ in range(nsteps)]
        ev_out = [torch.cuda.Event() for _ in range(nsteps)]
        torch.cuda.synchronize()
        start.record(stream)
        s_in.wait_event(start)
        s_out.wait_event(start)
        for n in range(nsteps):
            cs, ho = sets[n % 2], host_outs[n % 2]
            with torch.cuda.stream(s_in):
                if n >= 2:
                    s_in.wait_event(ev_comp[n - 2])   # this set's inputs are no longer read
                for name, t in host_in.items():
                    getattr(cs, name).copy_(t, non_blocking=True)
                ev_in[n].record(s_in)
            stream.wait_event(ev_in[n])
            if n >= 2:
                stream.wait_event(ev_out[n - 2])      # this set's outputs were read back
            cs.fwd_ex(stream)
            cs.bwd_ex(stream)
            ev_comp[n].record(stream)
            with torch.cuda.stream(s_out):
                s_out.wait_event(ev_comp[n])
                for name, t in ho.items():
                    t.copy_(getattr(cs, name), non_blocking=True)
                ev_out[n].record(s_out)
        stream.wait_event(ev_out[nsteps - 1])
        stream.wait_event(ev_in[nsteps - 1])
        end.record(stream)
        torch.cuda.synchronize()
        return start.elapsed_time(end)

    # the dominant kernel alone: the same steps again with the library's
    # event pairs around each launch of the forward kernel and of the
    # backward's main kernel (kept out of the headline pass: an event between
    # two kernels stops the second from overlapping the first one's tail)
    timed = {"rxl_fwd_tc_kernel": rxl.RXL_KERNEL_FWD, "rxl_bwd_main_kernel": rxl.RXL_KERNEL_BWD_MAIN,
             "bwd_prep": rxl.RXL_KERNEL_BWD_PREP, "bwd_dq_finish_kernel": rxl.RXL_KERNEL_BWD_FINISH}
    rxl.rxl_kernel_timing(True)
    for k in timed.values():
        rxl.rxl_kernel_timing_read(k)
    for _ in range(args.steps):
        flush.zero_()
        step()
    torch.cuda.synchronize()
    rxl.rxl_kernel_timing(False)
    kernel_ms = {}
    for name, k in timed.items():
        t_ms, n_launch = rxl.rxl_kernel_timing_read(k)
        kernel_ms[name] = t_ms / max(n_launch, 1)
    kernel_ms = {k: max_over_ranks(v, world, device="cuda") for k, v in kernel_ms.items()}

    # run-to-run variation of the backward: dQ/dR/du/dv are summed by
    # hardware reductions in a varying order (dK/dV are reproducible)
    ref = {n: getattr(c, n).float().clone() for n in ("dq", "dr", "du", "dvb", "dk", "dv")}
    step()
    torch.cuda.synchronize()
    variation = {n: {"max_abs_diff": (getattr(c, n).float() - t).abs().max().item(),
                     "max_abs": t.abs().max().item()} for n, t in ref.items()}

    e2e_value = None
    if not args.no_e2e:
        e2e_run(max(args.warmup, 2))
        e2e_ms = max_over_ranks(e2e_run(args.steps), world, device="cuda")
        e2e_value = whole_job_rate(args.steps * flop_step, world, e2e_ms * 1e-3) / 1e12

    if rank != 0:
        return
    peak_tf, _, peak_kind = peaks()
    bwd_avg = sum(bwd_ms) / len(bwd_ms)
    fwd_avg = sum(fwd_ms) / len(fwd_ms)
    kb = kernel_ms["rxl_bwd_main_kernel"]
    achieved = pairs * FLOP_BWD_PAIR / (kb * 1e-3) / 1e12
    rec, why = traffic_record(BWD_MAIN_PROFILE, BWD_MAIN_SOURCES)
    traffic = rec[0] * B / rec[1] if rec else None
    out = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": tot_ms / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "tokens_per_s": tokens, "fwd_ms": fwd_avg, "bwd_ms": bwd_avg,
        "split_note": "fwd_ms / bwd_ms from a second pass of the same steps with an event between the forward "
                      "and the backward; ms_per_step has no event inside a step",
        "fwd_tflops": pairs * FLOP_FWD_PAIR / (fwd_avg * 1e-3) / 1e12,
        "config": {"workload": WORKLOAD, "B": B, "H": H, "L": L, "M": M, "mem_len": m, "dh": DH,
                   "flop_per_step": flop_step, "l2": "flushed between steps (256 MiB write, outside events)",
                   "parallelism": f"{world} independent replicas (one per GPU)"},
        "roofline": {"bound": "tensor", "kernel": "rxl_bwd_main_kernel",
                     "achieved": achieved, "peak": peak_tf, "unit": "TFLOP/s", "frac": achieved / peak_tf,
                     "traffic": traffic,
                     "kernel_ms": kb, "algorithmic_flop_per_launch": pairs * FLOP_BWD_PAIR,
                     "traffic_note": (f"dram read+write per launch from the ncu record in {BWD_MAIN_PROFILE} "
                                      f"(batch {rec[1]}), scaled by the batch (the items scale with B)")
                     if rec else f"null: {why}",
                     "timing_note": "CUDA events around each launch of the kernel on its stream, in a second "
                                    "pass of the same steps (L2 flushed between steps)",
                     "peak_kind": f"{peak_kind} bf16 burst"},
        "kernels_ms": kernel_ms,
        "bwd_run_to_run": variation,
        "fwd_kernel_tflops": pairs * FLOP_FWD_PAIR / (kernel_ms["rxl_fwd_tc_kernel"] * 1e-3) / 1e12,
        "clocks": clk.summary(),
        "e2e": {"value": e2e_value, "unit": "TFLOP/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "note": "pinned host buffers; inputs of step n+1 and outputs of step n-1 are copied on two copy "
                        "streams while step n computes (double-buffered device and host sets)"},
        "gpu_launches": launches,
    }
    if world == 1 and not args.no_stream:
        stream, mu = stream_cfg5()
        out["stream_cfg5"] = stream
        out["mem_update_roofline"] = mem_update_hbm()
        out["mem_update_l2_resident"] = mu
        out["cfg2_stream"] = cfg2_stream(cpu=not args.no_cpu_baseline)
        out["cfg4_pair"] = cfg4_pair(cpu=not args.no_cpu_baseline)
        out["window_recompute"] = window_recompute()
        out["reset_cfg3"] = reset_cfg3()
        out["proj_cfg3"] = proj_cfg3()
        out["stack_cfg5"] = stack_cfg5()
    if world == 1 and not args.no_cpu_baseline:
        nthreads = os.cpu_count() or 1
        dt, fl = cpu_sample(x, (0, H), nthreads)
        out["cpu_baseline"] = {"value": fl / dt / 1e12, "unit": "TFLOP/s", "cores": min(nthreads, H * B),
                               "kind": "oracle",
                               "sample": f"fwd+bwd of the whole workload ({H * B} (b,h) units), {dt:.1f} s"}
    print(json.dumps(out), flush=True)


def stream_cfg5(segments=32, layers=16, reps_update=200):
    """The 16-layer evaluation stream (B4 H16 L128 M1600, fwd + ring update per
    layer and segment, memory empty at the start) and the memory-update kernel
    alone. Inputs: seeded device normals (timing only; parity is in tests)."""
    import torch
    import long_context_lm_rel_gb300 as rxl
    B5, H5, L5, M5 = 4, 16, 128, 1600
    kv = M5 + L5
    g = torch.Generator(device="cuda").manual_seed(5)
    bf = torch.bfloat16
    mk = lambda *s, std=0.125: (torch.randn(*s, generator=g, device="cuda") * std).to(bf)
    K = [mk(B5, H5, kv, DH) for _ in range(layers)]
    V = [mk(B5, H5, kv, DH) for _ in range(layers)]
    R = [mk(H5, kv, DH, std=0.7) for _ in range(layers)]
    U = [mk(H5, DH, std=0.02) for _ in range(layers)]
    VB = [mk(H5, DH, std=0.02) for _ in range(layers)]
    Q = mk(B5, H5, L5, DH)
    o = torch.empty(B5, H5, L5, DH, device="cuda", dtype=bf)
    lse = torch.empty(B5, H5, L5, device="cuda", dtype=torch.float32)
    cur = mk(B5, H5, L5, DH)
    rings = [[rxl.rxl_ring(t.data_ptr(), B5 * H5, M5, DH, kv * DH, rxl.RXL_DTYPE_BF16, 0, 0) for t in (K[n], V[n])]
             for n in range(layers)]
    def run_stream(st):
        """One pass of the stream from empty memory; returns (launches, visible pairs)."""
        rings = [[rxl.rxl_ring(t.data_ptr(), B5 * H5, M5, DH, kv * DH, rxl.RXL_DTYPE_BF16, 0, 0)
                  for t in (K[n], V[n])] for n in range(layers)]
        launches = pairs = 0
        for seg in range(segments):
            for n in range(layers):
                rk, rv = rings[n]
                K[n][:, :, M5:].copy_(cur)
                V[n][:, :, M5:].copy_(cur)
                m = rk.len
                pairs += B5 * H5 * (L5 * m + L5 * (L5 + 1) // 2)
                d = rxl.make_desc(B5, H5, L5, M5, m, rk.head, SCALE, rxl.RXL_DTYPE_BF16)
                rxl.rxl_attn_fwd(d, Q, K[n], V[n], R[n], U[n], VB[n], o, lse, st)
                launches += rxl.rxl_last_launch_count()
                rxl.rxl_mem_update_rings([rk, rv], [K[n].data_ptr() + M5 * DH * 2, V[n].data_ptr() + M5 * DH * 2],
                                         [kv * DH, kv * DH], L5, st)
                launches += rxl.rxl_last_launch_count()
        return launches, pairs

    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    # eager: the calls issued from Python one by one
    st = torch.cuda.current_stream()
    torch.cuda.synchronize()
    e0.record(st)
    launches, pairs = run_stream(st)
    e1.record(st)
    torch.cuda.synchronize()
    ms_eager = e0.elapsed_time(e1)
    # the same 32 x 16 sequence (same ring positions) captured once as a CUDA
    # graph and replayed: what the GPU takes without the host issuing every call
    graph = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        with torch.cuda.graph(graph, stream=side):
            run_stream(torch.cuda.current_stream())
    torch.cuda.current_stream().wait_stream(side)
    graph.replay()
    torch.cuda.synchronize()
    reps = 3
    e0.record(st)
    for _ in range(reps):
        graph.replay()
    e1.record(st)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / reps
    # the memory update alone at the stream's call size (K and V rings of a
    # layer in one launch, 2 MiB appended per ring): back-to-back calls on full
    # rings, replayed as a graph. The 28 MB of rings stay in L2 here.
    rk = rxl.rxl_ring(K[0].data_ptr(), B5 * H5, M5, DH, kv * DH, rxl.RXL_DTYPE_BF16, 0, M5)
    rv = rxl.rxl_ring(V[0].data_ptr(), B5 * H5, M5, DH, kv * DH, rxl.RXL_DTYPE_BF16, 0, M5)
    srcs = [K[0].data_ptr() + M5 * DH * 2, V[0].data_ptr() + M5 * DH * 2]
    for _ in range(10):
        rxl.rxl_mem_update_rings([rk, rv], srcs, [kv * DH] * 2, L5, st)
    torch.cuda.synchronize()
    g_up = torch.cuda.CUDAGraph()
    with torch.cuda.stream(side):
        with torch.cuda.graph(g_up, stream=side):
            for _ in range(reps_update):
                rxl.rxl_mem_update_rings([rk, rv], srcs, [kv * DH] * 2, L5, torch.cuda.current_stream())
    torch.cuda.current_stream().wait_stream(side)
    g_up.replay()
    torch.cuda.synchronize()
    e0.record(st)
    g_up.replay()
    e1.record(st)
    torch.cuda.synchronize()
    us = 1e3 * e0.elapsed_time(e1) / reps_update
    bytes_call = 2 * 2 * B5 * H5 * min(L5, M5) * DH * 2   # K and V: read + write of the appended rows
    return {"workload": "cfg5_bf16_B4H16_L128M1600_16layer_32seg_fwd", "segments": segments, "layers": layers,
            "ms": ms, "tokens_per_s": B5 * L5 * segments / (ms * 1e-3),
            "attn_tflops": pairs * FLOP_FWD_PAIR / (ms * 1e-3) / 1e12, "gpu_launches": launches,
            "ms_eager": ms_eager, "tokens_per_s_eager": B5 * L5 * segments / (ms_eager * 1e-3),
            "note": "per segment and layer: K/V current rows copied in (torch), rxl_attn_fwd, "
                    "rxl_mem_update_rings (K and V in one launch); ms = the whole stream captured once as a "
                    "CUDA graph and replayed, ms_eager = the same calls issued one by one from Python"}, \
           {"kernel": "mem_update_kernel", "residency": "l2", "unit": "GB/s", "us_per_call": us,
            "bytes_per_call": bytes_call, "achieved": bytes_call / (us * 1e-6) / 1e9,
            "note": f"cfg5 call size (K+V of a layer, 4 MiB appended), {reps_update} back-to-back calls as a "
                    "CUDA graph; the rings stay L2-resident, so this is launch/latency-bound, not an HBM figure"}


def mem_update_hbm(reps=10):
    """The memory-update kernel where HBM bounds it: the K and V rings of a
    B16 H16 layer (256 planes, 128-byte rows) with 8192 rows of memory,
    appending 4096 rows per ring per call (268 MB read + 268 MB written per
    call), the L2 flushed (256 MiB write) before each timed call."""
    import torch
    import long_context_lm_rel_gb300 as rxl
    planes, cap, Lm = 256, 8192, 4096
    bf = torch.bfloat16
    rings = [torch.zeros(planes, cap, DH, device="cuda", dtype=bf) for _ in range(2)]
    srcs = [torch.randn(planes, Lm, DH, device="cuda").to(bf) for _ in range(2)]
    flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
    st = torch.cuda.current_stream()
    rr = [rxl.rxl_ring(t.data_ptr(), planes, cap, DH, cap * DH, rxl.RXL_DTYPE_BF16, 0, cap) for t in rings]
    for _ in range(3):
        rxl.rxl_mem_update_rings(rr, srcs, [Lm * DH] * 2, Lm, st)
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(reps)]
    for e0, e1 in ev:
        flush.zero_()
        e0.record(st)
        rxl.rxl_mem_update_rings(rr, srcs, [Lm * DH] * 2, Lm, st)
        e1.record(st)
    torch.cuda.synchronize()
    us = 1e3 * sum(a.elapsed_time(b) for a, b in ev) / reps
    bytes_call = 2 * 2 * planes * Lm * DH * 2
    _, hbm, kind = peaks()
    gbs = bytes_call / (us * 1e-6) / 1e9
    return {"kernel": "mem_update_kernel", "residency": "hbm", "bound": "hbm", "unit": "GB/s",
            "us_per_call": us, "bytes_per_call": bytes_call, "achieved": gbs, "peak": hbm, "frac": gbs / hbm,
            "peak_kind": f"{kind} copy",
            "workload": "K and V rings, 256 planes x 8192 rows x 64 bf16, 4096 rows appended per ring per call",
            "note": "L2 flushed (256 MiB write) before each call, outside the events; bytes = read + write of the "
                    "appended rows"}


def pair_bytes(b, h, l, cap):
    """Compulsory HBM bytes of one fwd_ex + bwd_ex pair (bf16 tensors, fp32
    LSE and position gradients): every input read once, every output written
    once: forward Q, K, V, R in, O, O_lo, LSE out; backward Q, K, V, R, O,
    O_lo, LSE, dO in, dQ, dK, dV, dR, du, dv out."""
    q = b * h * l * DH * 2
    kv = b * h * (cap + l) * DH * 2
    r = h * (cap + l) * DH * 2
    lse = b * h * l * 4
    fwd = q + 2 * kv + r + 2 * q + lse
    bwd = (q + 2 * kv + r + 2 * q + lse + q) + (q + 2 * kv + 2 * r + 2 * h * DH * 4)
    return fwd, bwd


def timed_pairs(fwd, bwd, stream, flush, reps):
    """Per step (L2 flushed before it, outside the events): the whole step
    with one event pair and nothing between the two calls, then the same
    steps again with an event between them for the forward / backward split.
    Returns (step_ms, fwd_ms, bwd_ms), averages over reps."""
    import torch
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(reps)]
    for e in ev:
        flush.zero_()
        e[0].record(stream)
        fwd()
        bwd()
        e[1].record(stream)
    ev3 = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(reps)]
    for e in ev3:
        flush.zero_()
        e[0].record(stream)
        fwd()
        e[1].record(stream)
        bwd()
        e[2].record(stream)
    torch.cuda.synchronize()
    step_ms = sum(e[0].elapsed_time(e[1]) for e in ev) / reps
    fwd_ms = sum(e[0].elapsed_time(e[1]) for e in ev3) / reps
    bwd_ms = sum(e[1].elapsed_time(e[2]) for e in ev3) / reps
    return step_ms, fwd_ms, bwd_ms


def cfg4_pair(reps=10, cpu=True):
    """Configuration 4 (long memory, M = 5L): B8 H16 L256 M1280, the training
    pair (fwd_ex + bwd_ex), seeded inputs of the configuration's
    distributions, L2 flushed between steps. Near the ridge of the tensor and
    HBM roofs, so both fractions are reported; the oracle is timed on the
    whole workload on the host cores."""
    import numpy as np
    import torch
    import long_context_lm_rel_gb300 as rxl  # noqa: F401
    import rxl_inputs as gen
    from long_context_lm_rel_gb300.calls import AttnCall, place_kv
    w = gen.CFG4
    p, sg, mem = gen.layer_params(w), gen.segment_inputs(w), gen.initial_memory(w)
    cap = m = w.M
    c = AttnCall(sg["q"], place_kv(mem["k_mem"], sg["k_cur"], cap, 0), place_kv(mem["v_mem"], sg["v_cur"], cap, 0),
                 p["r"], p["u"], p["vb"], cap=cap, m=m, head=0, dtype="bf16", scale=w.scale)
    c.fwd_ex().alloc_bwd(sg["do"])
    st = torch.cuda.current_stream()
    flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
    for _ in range(3):
        c.fwd_ex(st).bwd_ex(st)
    torch.cuda.synchronize()
    step_ms, fwd_ms, bwd_ms = timed_pairs(lambda: c.fwd_ex(st), lambda: c.bwd_ex(st), st, flush, reps)
    pairs = visible_pairs(w.B, w.H, w.L, m)
    flop = pairs * (FLOP_FWD_PAIR + FLOP_BWD_PAIR)
    tot = step_ms * 1e-3
    peak_tf, hbm, kind = peaks()
    fb, bb = pair_bytes(w.B, w.H, w.L, cap)
    tf = flop / tot / 1e12
    out = {"workload": "cfg4_bf16_B8H16_L256M1280_dh64_fwd+bwd", "ms_per_step": step_ms, "fwd_ms": fwd_ms,
           "bwd_ms": bwd_ms,
           "tokens_per_s": w.B * w.L / tot, "tflops": tf, "visible_pairs": pairs,
           "roofline": {"tensor": {"achieved": tf, "peak": peak_tf, "unit": "TFLOP/s", "frac": tf / peak_tf,
                                   "peak_kind": f"{kind} bf16 burst"},
                        "hbm": {"achieved": (fb + bb) / tot / 1e9, "peak": hbm, "unit": "GB/s",
                                "frac": (fb + bb) / tot / 1e9 / hbm, "compulsory_bytes": fb + bb,
                                "peak_kind": f"{kind} copy"}},
           "note": "L2 flushed between steps; compulsory bytes = every input read and every output written once; "
                   "ms_per_step has no event inside a step, fwd_ms / bwd_ms come from a second pass with one"}
    if cpu:
        import oracle
        k = np.concatenate([mem["k_mem"], sg["k_cur"]], 2)
        v = np.concatenate([mem["v_mem"], sg["v_cur"]], 2)
        nthreads = os.cpu_count() or 1
        t0 = time.perf_counter()
        oracle.fwd(sg["q"], k, v, p["r"], p["u"], p["vb"], w.scale, nthreads=nthreads)
        oracle.bwd(sg["q"], k, v, p["r"], p["u"], p["vb"], sg["do"], w.scale, nthreads=nthreads)
        dt = time.perf_counter() - t0
        out["cpu_baseline"] = {"value": flop / dt / 1e12, "unit": "TFLOP/s", "seconds": dt, "kind": "oracle",
                               "cores": min(nthreads, w.B * w.H), "sample": "the whole workload, fwd+bwd"}
    return out


def cfg2_stream(reps=20, cpu=True):
    """Configuration 2: one layer over 4 consecutive segments, B8 H8 L128
    M128, memory empty at the start and rolled with Tail_M (K and V rings in
    one launch) after each segment; per segment the training pair (fwd_ex +
    bwd_ex). Device-generated normals (timing only; parity is in the tests).
    The whole workload is L2-resident and small (64 query tiles per call), so
    it is launch- and latency-bound: reported eager and as a CUDA graph."""
    import numpy as np
    import torch
    import long_context_lm_rel_gb300 as rxl
    B2, H2, L2, M2, segs = 8, 8, 128, 128, 4
    kv = M2 + L2
    g = torch.Generator(device="cuda").manual_seed(2)
    bf = torch.bfloat16
    mk = lambda *sh, std=0.125: (torch.randn(*sh, generator=g, device="cuda") * std).to(bf)
    K, V = mk(B2, H2, kv, DH), mk(B2, H2, kv, DH)
    R, U, VB = mk(H2, kv, DH, std=0.7), mk(H2, DH, std=0.02), mk(H2, DH, std=0.02)
    seg_in = [dict(q=mk(B2, H2, L2, DH), k=mk(B2, H2, L2, DH), v=mk(B2, H2, L2, DH), do=mk(B2, H2, L2, DH, std=1.0))
              for _ in range(segs)]
    o, o_lo = torch.empty(B2, H2, L2, DH, device="cuda", dtype=bf), torch.empty(B2, H2, L2, DH, device="cuda", dtype=bf)
    lse = torch.empty(B2, H2, L2, device="cuda", dtype=torch.float32)
    dq = torch.empty_like(o)
    dk, dv = torch.empty_like(K), torch.empty_like(V)
    dr = torch.empty(H2, kv, DH, device="cuda", dtype=torch.float32)
    du, dvb = torch.empty(H2, DH, device="cuda", dtype=torch.float32), torch.empty(H2, DH, device="cuda",
                                                                                  dtype=torch.float32)
    d0 = rxl.make_desc(B2, H2, L2, M2, M2, 0, SCALE, rxl.RXL_DTYPE_BF16)
    wsb = rxl.rxl_attn_bwd_workspace_bytes(d0)
    ws = torch.empty(wsb, device="cuda", dtype=torch.uint8)

    def run(st):
        rk = rxl.rxl_ring(K.data_ptr(), B2 * H2, M2, DH, kv * DH, rxl.RXL_DTYPE_BF16, 0, 0)
        rv = rxl.rxl_ring(V.data_ptr(), B2 * H2, M2, DH, kv * DH, rxl.RXL_DTYPE_BF16, 0, 0)
        pairs = launches = 0
        for x in seg_in:
            K[:, :, M2:].copy_(x["k"])
            V[:, :, M2:].copy_(x["v"])
            m = rk.len
            d = rxl.make_desc(B2, H2, L2, M2, m, rk.head, SCALE, rxl.RXL_DTYPE_BF16)
            rxl.rxl_attn_fwd_ex(d, x["q"], K, V, R, U, VB, o, o_lo, lse, st)
            launches += rxl.rxl_last_launch_count()
            rxl.rxl_attn_bwd_ex(d, x["q"], K, V, R, U, VB, o, o_lo, lse, x["do"], dq, dk, dv, dr, du, dvb, ws, wsb, st)
            launches += rxl.rxl_last_launch_count()
            rxl.rxl_mem_update_rings([rk, rv], [K.data_ptr() + M2 * DH * 2, V.data_ptr() + M2 * DH * 2],
                                     [kv * DH] * 2, L2, st)
            launches += rxl.rxl_last_launch_count()
            pairs += visible_pairs(B2, H2, L2, m)
        return pairs, launches

    st = torch.cuda.current_stream()
    for _ in range(3):
        run(st)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(st)
    for _ in range(reps):
        pairs, launches = run(st)
    e1.record(st)
    torch.cuda.synchronize()
    ms_eager = e0.elapsed_time(e1) / reps
    graph = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    side.wait_stream(st)
    with torch.cuda.stream(side):
        with torch.cuda.graph(graph, stream=side):
            run(torch.cuda.current_stream())
    st.wait_stream(side)
    graph.replay()
    torch.cuda.synchronize()
    e0.record(st)
    for _ in range(reps):
        graph.replay()
    e1.record(st)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / reps
    flop = pairs * (FLOP_FWD_PAIR + FLOP_BWD_PAIR)
    peak_tf, _, kind = peaks()
    tf = flop / (ms * 1e-3) / 1e12
    out = {"workload": "cfg2_bf16_B8H8_L128M128_4seg_fwd+bwd", "ms": ms, "ms_eager": ms_eager,
           "tokens_per_s": segs * B2 * L2 / (ms * 1e-3), "tflops": tf,
           "tflops_eager": flop / (ms_eager * 1e-3) / 1e12, "visible_pairs": pairs, "gpu_launches": launches,
           "roofline": {"bound": "tensor", "achieved": tf, "peak": peak_tf, "unit": "TFLOP/s", "frac": tf / peak_tf,
                        "peak_kind": f"{kind} bf16 burst"},
           "note": "4 segments from empty memory, per segment: K/V current rows copied in, fwd_ex, bwd_ex, K+V ring "
                   "update; ms = captured once as a CUDA graph and replayed, ms_eager = issued from Python; warm L2 "
                   "(the whole workload is ~10 MB)"}
    if cpu:
        import oracle
        import rxl_inputs as gen
        wk = gen.CFG2
        prm = gen.layer_params(wk)
        mk_, mv_ = np.zeros((wk.B, wk.H, 0, wk.dh)), np.zeros((wk.B, wk.H, 0, wk.dh))
        nthreads = os.cpu_count() or 1
        t_cpu = 0.0
        for sgi in range(wk.segments):
            x = gen.segment_inputs(wk, sgi)
            k = np.concatenate([mk_, x["k_cur"]], 2)
            v = np.concatenate([mv_, x["v_cur"]], 2)
            t0 = time.perf_counter()
            oracle.fwd(x["q"], k, v, prm["r"], prm["u"], prm["vb"], wk.scale, nthreads=nthreads)
            oracle.bwd(x["q"], k, v, prm["r"], prm["u"], prm["vb"], x["do"], wk.scale, nthreads=nthreads)
            mk_, mv_ = oracle.tail_m(mk_, x["k_cur"], wk.M), oracle.tail_m(mv_, x["v_cur"], wk.M)
            t_cpu += time.perf_counter() - t0
        out["cpu_baseline"] = {"value": flop / t_cpu / 1e12, "unit": "TFLOP/s", "seconds": t_cpu, "kind": "oracle",
                               "cores": min(nthreads, wk.B * wk.H), "sample": "the whole 4-segment stream, fwd+bwd"}
    return out


def reset_cfg3(reps=10):
    """The cfg3 training pair under a per-row document reset: a quarter of the
    batch rows has just started a new document (no memory), a quarter sees
    128, a quarter 384 and a quarter all 512 memory rows. Throughput counts
    the visible pairs of each row. L2 flushed between steps as in the main
    measurement."""
    import numpy as np
    import torch
    import long_context_lm_rel_gb300 as rxl
    from long_context_lm_rel_gb300.calls import AttnCall, place_kv
    x = make_inputs()
    cap = m = M
    mvis = [(0, 128, 384, 512)[b % 4] for b in range(B)]
    c = AttnCall(x["q"], place_kv(x["k_mem"], x["k_cur"], cap, 0), place_kv(x["v_mem"], x["v_cur"], cap, 0),
                 x["r"], x["u"], x["vb"], cap=cap, m=m, head=0, dtype="bf16", scale=SCALE)
    c.fwd_reset(mvis)
    c.alloc_bwd(x["do"])
    stream = torch.cuda.current_stream()
    flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
    for _ in range(3):
        c.fwd_reset(mvis, stream=stream)
        c.bwd_reset(stream)
    torch.cuda.synchronize()
    step_ms, fwd_ms, bwd_ms = timed_pairs(
        lambda: rxl.rxl_attn_fwd_reset(c.desc, c.mvis, c.q, c.k, c.v, c.r, c.u, c.vb, c.o, c.o_lo, c.lse, stream),
        lambda: c.bwd_reset(stream), stream, flush, reps)
    pairs = sum(H * (L * mb + L * (L + 1) // 2) for mb in mvis)
    flop = pairs * (FLOP_FWD_PAIR + FLOP_BWD_PAIR)
    return {"workload": "cfg3 with per-row reset, mem_visible = 0/128/384/512 by b mod 4",
            "ms_per_step": step_ms, "fwd_ms": fwd_ms, "bwd_ms": bwd_ms, "visible_pairs": pairs,
            "tflops": flop / (step_ms * 1e-3) / 1e12}


def proj_cfg3(reps=20):
    """The projection front-end at the cfg3 shape with a hidden-state memory:
    d = 1024, H*dh = 1024; Q from the 512 current rows, K and V from the 512
    memory + 512 current rows of each of the 16 batch rows (2 * 16 * (512 +
    2 * 1024) * 1024 * 1024 flop). Warm L2, back-to-back calls (the weights
    are 6 MB, the hidden states 32 MB)."""
    import torch
    import long_context_lm_rel_gb300 as rxl
    d, Hh = 1024, H
    g = torch.Generator(device="cuda").manual_seed(11)
    bf = torch.bfloat16
    mk = lambda *s, std=1.0: (torch.randn(*s, generator=g, device="cuda") * std).to(bf)
    hm, hc = mk(B, M, d), mk(B, L, d)
    w = [mk(d, Hh * DH, std=d ** -0.5) for _ in range(3)]
    q = torch.empty(B, Hh, L, DH, device="cuda", dtype=bf)
    k = torch.empty(B, Hh, M + L, DH, device="cuda", dtype=bf)
    v = torch.empty_like(k)
    desc = rxl.make_desc(B, Hh, L, M, M, 0, SCALE, rxl.RXL_DTYPE_BF16)
    st = torch.cuda.current_stream()
    for _ in range(3):
        rxl.rxl_qkv_proj(desc, d, hm, hc, *w, q, k, v, st)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(st)
    for _ in range(reps):
        rxl.rxl_qkv_proj(desc, d, hm, hc, *w, q, k, v, st)
    e1.record(st)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / reps
    flop = 2 * B * (L + 2 * (M + L)) * d * Hh * DH
    peak_tf, _, kind = peaks()
    tf = flop / (ms * 1e-3) / 1e12
    return {"workload": "cfg3 shape, d=1024, hidden-state memory of 512 rows; Q, K, V in one launch",
            "ms": ms, "tflops": tf, "roofline": {"bound": "tensor", "achieved": tf, "peak": peak_tf,
                                                  "unit": "TFLOP/s", "frac": tf / peak_tf,
                                                  "peak_kind": f"{kind} bf16 burst"},
            "note": "warm L2, back-to-back calls"}


def stack_cfg5(segments=3, layers=16):
    """The full evaluation stack at the cfg5 shape: 16 layers (d = 1024,
    d_ff = 4096, H = 16) over B4 L128 segments, each layer's hidden-state
    memory already holding M = 1600 rows (steady state; the ring head moves
    by L per segment). Per segment and layer: rxl_layer_fwd (projections of
    the 1728 memory + current rows, attention, W_O, two LayerNorms, the
    feed-forward sublayer) and rxl_mem_update of that layer's input states.
    Seeded device normals (timing only; parity is in the tests)."""
    import torch
    import long_context_lm_rel_gb300 as rxl
    B5, H5, L5, M5, d, dff = 4, 16, 128, 1600, 1024, 4096
    g = torch.Generator(device="cuda").manual_seed(13)
    bf = torch.bfloat16
    mk = lambda *s, std=1.0: (torch.randn(*s, generator=g, device="cuda") * std).to(bf)
    Ws, keep = [], []
    for _ in range(layers):
        t = dict(w_q=mk(d, H5 * DH, std=d ** -0.5), w_k=mk(d, H5 * DH, std=d ** -0.5),
                 w_v=mk(d, H5 * DH, std=d ** -0.5), w_o=mk(H5 * DH, d, std=(H5 * DH) ** -0.5),
                 r=mk(H5, M5 + L5, DH, std=0.7), u=mk(H5, DH, std=0.02), vbias=mk(H5, DH, std=0.02),
                 ln1_gamma=torch.ones(d, device="cuda", dtype=bf), ln1_beta=torch.zeros(d, device="cuda", dtype=bf),
                 w_1=mk(d, dff, std=d ** -0.5), b_1=mk(dff, std=0.1), w_2=mk(dff, d, std=dff ** -0.5),
                 b_2=mk(d, std=0.1), ln2_gamma=torch.ones(d, device="cuda", dtype=bf),
                 ln2_beta=torch.zeros(d, device="cuda", dtype=bf))
        keep.append(t)
        Ws.append(rxl.make_layer_weights(**t))
    rings = [mk(B5, M5, d) for _ in range(layers)]
    state = [rxl.rxl_ring(rings[n].data_ptr(), B5, M5, d, M5 * d, rxl.RXL_DTYPE_BF16, 0, M5)
             for n in range(layers)]
    hs = [mk(B5, L5, d) for _ in range(layers + 1)]
    desc0 = rxl.make_desc(B5, H5, L5, M5, M5, 0, SCALE, rxl.RXL_DTYPE_BF16)
    wsb = rxl.rxl_layer_fwd_workspace_bytes(desc0, d, dff)
    ws = torch.empty(wsb, device="cuda", dtype=torch.uint8)
    st = torch.cuda.current_stream()
    launches = 0

    def segment():
        nonlocal launches
        for n in range(layers):
            desc = rxl.make_desc(B5, H5, L5, M5, state[n].len, state[n].head, SCALE, rxl.RXL_DTYPE_BF16)
            rxl.rxl_layer_fwd(desc, d, dff, Ws[n], rings[n], hs[n], hs[n + 1], ws, wsb, st)
            launches += rxl.rxl_last_launch_count()
            rxl.rxl_mem_update(state[n], hs[n], L5 * d, L5, st)
            launches += rxl.rxl_last_launch_count()

    segment()
    torch.cuda.synchronize()
    launches = 0
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(st)
    for _ in range(segments):
        segment()
    e1.record(st)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / segments
    rows_kv = M5 + L5
    flop_layer = (2 * B5 * (L5 + 2 * rows_kv) * d * H5 * DH              # Q, K, V projections
                  + visible_pairs(B5, H5, L5, M5) * FLOP_FWD_PAIR           # attention
                  + 2 * B5 * L5 * H5 * DH * d                             # W_O
                  + 2 * 2 * B5 * L5 * d * dff)                            # feed-forward
    return {"workload": "cfg5 shape, 16-layer stack: B4 H16 L128, hidden-state memory 1600 rows, d 1024, d_ff 4096, fwd",
            "ms_per_segment": ms, "tokens_per_s": B5 * L5 / (ms * 1e-3),
            "tflops": layers * flop_layer / (ms * 1e-3) / 1e12, "gpu_launches_per_segment": launches // segments,
            "note": "steady state (memory full); each segment re-projects K/V of the 1728 memory + current rows per layer"}


def window_recompute(reps=20):
    """Evaluation with and without the memory, one layer (the reuse the pages
    credit for Transformer-XL's evaluation speed): the segment-recurrent step
    (L = 128 new queries over M = 1600 cached rows plus the segment) against
    recomputing causal attention over the whole window of M + L = 1728
    positions for every new position (m = 0), B4 H16 bf16, the same kernel.
    Speed-up per evaluated position = L * t_window / t_segment. Warm L2,
    back-to-back calls; parity of both shapes is in the GPU tests."""
    import torch
    import long_context_lm_rel_gb300 as rxl
    B5, H5, L5, M5 = 4, 16, 128, 1600
    W = M5 + L5
    g = torch.Generator(device="cuda").manual_seed(7)
    bf = torch.bfloat16
    mk = lambda *s, std=0.125: (torch.randn(*s, generator=g, device="cuda") * std).to(bf)
    st = torch.cuda.current_stream()

    def timed(Lq, cap, m):
        q, k, v = mk(B5, H5, Lq, DH), mk(B5, H5, cap + Lq, DH), mk(B5, H5, cap + Lq, DH)
        r, u, vb = mk(H5, cap + Lq, DH, std=0.7), mk(H5, DH, std=0.02), mk(H5, DH, std=0.02)
        o = torch.empty(B5, H5, Lq, DH, device="cuda", dtype=bf)
        lse = torch.empty(B5, H5, Lq, device="cuda", dtype=torch.float32)
        d = rxl.make_desc(B5, H5, Lq, cap, m, 0, SCALE, rxl.RXL_DTYPE_BF16)
        for _ in range(3):
            rxl.rxl_attn_fwd(d, q, k, v, r, u, vb, o, lse, st)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(st)
        for _ in range(reps):
            rxl.rxl_attn_fwd(d, q, k, v, r, u, vb, o, lse, st)
        e1.record(st)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / reps

    t_seg = timed(L5, M5, M5)
    t_win = timed(W, 0, 0)
    pairs_seg = visible_pairs(B5, H5, L5, M5)
    pairs_win = B5 * H5 * W * (W + 1) // 2
    return {"workload": "cfg5 shape, one layer: B4 H16, L128 over M1600 vs window 1728 recomputed, fwd",
            "segment_ms": t_seg, "window_ms": t_win,
            "segment_positions_per_s": B5 * L5 / (t_seg * 1e-3),
            "window_positions_per_s": B5 / (t_win * 1e-3),
            "speedup_per_position": L5 * t_win / t_seg,
            "segment_attn_tflops": pairs_seg * FLOP_FWD_PAIR / (t_seg * 1e-3) / 1e12,
            "window_attn_tflops": pairs_win * FLOP_FWD_PAIR / (t_win * 1e-3) / 1e12,
            "note": "attention of one layer only, warm L2; the pages' ~1800x refers to the whole model"}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-stream", action="store_true", help="skip the cfg5 stream / memory-update timing")
    ap.add_argument("--no-e2e", action="store_true", help="skip the end-to-end (host buffers) timing")
    ap.add_argument("--batch", type=int, default=16,
                    help="batch rows of the workload (16 = the benchmark; smaller = profiling case)")
    args = ap.parse_args()
    global B, WORKLOAD
    if args.batch != B:
        B = args.batch
        WORKLOAD = f"cfg3_shape_bf16_B{B}H16_L512M512_dh64_fwd+bwd (profiling case)"
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if world > 1 and args.impl == "ours":
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", "0")))
        dist.init_process_group("nccl")
    try:
        if args.impl == "reference":
            run_reference(args, rank, world)
        else:
            run_ours(args, rank, world)
    finally:
        if world > 1 and args.impl == "ours":
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
