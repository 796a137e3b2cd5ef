#!/usr/bin/env python
"""GMA forward throughput on one GB300: tokens*heads/s at K=256, bidirectional + causal.

One step = one bidirectional and one causal forward over the workload (both forms of the hot
path).  Prints ONE JSON line on rank 0.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl gma|reference]

--impl reference times the float64 CPU oracle (the only baseline that exists for this method)
on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import json
import os
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from gaussian_mixture_sequence_gma_gb300.inputs import bf16_bits, make_inputs, make_workload, workloads  # noqa: E402

WORKLOAD = "sweep_bf16_B1H8N131072K256"
METRIC = "GMA fwd tokens*heads/s at K=256 (bidir & causal)"
UNIT = "tokens*heads/s"
SWEEP = (4096, 16384, 65536, 131072)
CPU_SAMPLE_N = 65536      # positions of the workload the oracle baseline processes (a few s on 16 cores)


def flop_per_tokhead(K, d=64, dv=64):
    """Algorithmic FLOPs per token*head for both forms' shared work: logits for q and k
    (2 * 2*(2d)*K) plus write and read contractions with the normaliser column (2 * 2*K*(dv+1))."""
    return 8 * d * K + 4 * K * (dv + 1)


# Algorithmic FLOPs per token*head assigned to each kernel (every algorithmic op counted once;
# recomputation and the causal intra-chunk term are kernel overhead).
def kernel_flops(name, K, d=64, dv=64):
    half = 2 * 2 * d * K + 2 * K * (dv + 1)  # one side's logits + one of write/read
    table = {
        "simt_write": half, "simt_read": half, "simt_causal": half,
        "tc_bidir_write": half, "tc_bidir_read": half, "tc_causal_aggregate": half, "tc_causal_chunk": half,
    }
    return table.get(name, 0)


def kernel_bound(name):
    return "tensor" if name.startswith("tc_") else "alu"


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            j = json.load(f)
        return dict(hbm=j["hbm_gbs"], bf16=j["bf16_tflops"], bf16_sus=j.get("bf16_tflops_sustained"),
                    sm_max_mhz=j.get("sm_max_mhz", 2070.0), source="measured")
    return dict(hbm=6800.0, bf16=1900.0, bf16_sus=1700.0, sm_max_mhz=2070.0, source="fallback")


def kernel_source_hash():
    """Hash of the tensor-core kernel sources (a traffic figure is valid only for the code it was taken on)."""
    import hashlib
    src = os.path.join(ROOT, "gaussian_mixture_sequence_gma_gb300", "csrc")
    h = hashlib.sha256()
    for f in ("gma_tc.cu", "gma_tc_common.cuh", "gma_internal.h"):
        h.update(open(os.path.join(src, f), "rb").read())
    return h.hexdigest()[:16]


def traffic_for(name):
    """DRAM bytes per launch from the committed ncu summary, if taken on the current source."""
    p = os.path.join(ROOT, "profiles", "traffic.txt")
    if not os.path.exists(p):
        return None
    sha = kernel_source_hash()
    for line in open(p):
        parts = line.split()
        if len(parts) >= 3 and not line.startswith("#") and parts[0] == name and parts[2] == sha:
            return float(parts[1])
    return None


class ClockSampler:
    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.windows = []

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.FIELDS,
                                          "--format=csv,noheader,nounits", "-lms", "50"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.3)

    def mark(self, t0, t1):
        self.windows.append((t0, t1))

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        out, _ = self.proc.communicate(timeout=10)
        rows = []
        for line in out.splitlines():
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                ts = time.mktime(time.strptime(parts[0].split(".")[0], "%Y/%m/%d %H:%M:%S"))
                ts += float("0." + parts[0].split(".")[1]) if "." in parts[0] else 0.0
                rows.append((ts, float(parts[1]), float(parts[2]), parts[4:]))
            except (ValueError, IndexError):
                continue
        inside = [r for r in rows if any(t0 - 0.06 <= r[0] <= t1 + 0.06 for t0, t1 in self.windows)]
        use = inside if inside else rows
        if not use:
            return None
        names = ["active", "hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = set()
        for r in use:
            for n, v in zip(names[1:], r[3][1:]):
                if v.strip().lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": float(np.median([r[1] for r in use])), "sm_max_mhz": float(max(r[2] for r in use)),
                "reasons": sorted(reasons), "samples": len(use), "in_window": bool(inside)}


def max_over_ranks(x: float, world: int, device=None) -> float:
    """Maximum of a per-rank float over all ranks (identity for one rank)."""
    if world <= 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(units_per_rank: int, ms_per_step_max: float, world: int) -> float:
    """Whole-job throughput: every rank processes its own copy of the workload (weak scaling), and the
    job's step time is the slowest rank's."""
    return world * units_per_rank / (ms_per_step_max * 1e-3)


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def oracle_sample(inp, n_pos):
    """Float64 oracle over the first n_pos positions of every (b, h): bidirectional and causal.  The oracle
    parallelises over (b, h) units; the two forms run side by side, so up to 2 B H host threads are busy.
    Returns (seconds, token*heads processed, threads used, host cores)."""
    from concurrent.futures import ThreadPoolExecutor

    from oracle import oracle as orc
    sl = {k: np.ascontiguousarray(inp[k][:, :, :n_pos]) for k in ("Q", "K", "V")}
    B, H = sl["Q"].shape[:2]
    host = orc.default_threads()
    per_form = max(1, host // 2)

    def one(causal):
        orc.forward(sl["Q"], sl["K"], sl["V"], inp["mu"], inp["sigma2"], inp["log_pi"], 1e-6, causal=causal,
                    nthreads=per_form)

    t0 = time.perf_counter()
    with ThreadPoolExecutor(max_workers=2) as ex:  # the oracle call releases the interpreter lock
        list(ex.map(one, (False, True)))
    dt = time.perf_counter() - t0
    return dt, 2 * B * H * n_pos, 2 * min(per_form, B * H), host


def run_reference(args, world, rank):
    if rank != 0:
        return 0
    w = workloads()[args.workload]
    inp = make_workload(w)
    n_pos = min(args.ref_positions, w.N)
    for _ in range(args.warmup):
        oracle_sample(inp, n_pos)
    total_t, total_units, cores, host = 0.0, 0, 1, 1
    for _ in range(args.steps):
        dt, units, cores, host = oracle_sample(inp, n_pos)
        total_t += dt
        total_units += units
    value = total_units / total_t
    sample = "first %d positions of every (b,h) of %s, bidirectional + causal, float64 oracle" % (n_pos, w.name)
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total_t / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded; shapes and distributions of the workload)",
            "config": config_dict(w),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "host_cores": host, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def config_dict(w):
    return {"workload": w.name, "B": w.B, "H": w.H, "N": w.N, "K": w.K, "d": w.d, "dv": w.dv,
            "forms": "bidirectional + causal per step", "io_dtype": w.dtype,
            "l2": "inputs larger than L2 (Q,K,V = %.0f MB > 129 MB); no flush" % (3 * w.B * w.H * w.N * 64 * 2 / 1e6),
            "parallelism": "one process per GPU, independent replicas of the workload"}


def to_dev(inp, dev):
    import torch
    t = {k: torch.from_numpy(inp[k]).to(dev) for k in ("mu", "sigma2", "log_pi")}
    for k in ("Q", "K", "V"):
        if inp.get("dtype", "bf16") == "f32":
            t[k] = torch.from_numpy(np.ascontiguousarray(inp[k])).to(dev)
        else:
            t[k] = torch.from_numpy(bf16_bits(inp[k]).view(np.int16)).to(dev).view(torch.bfloat16)
    return t


def rel_err(O, ref):
    """max |O - O_ref| / max |O_ref| over the compared outputs (the parity measure of the tests)."""
    O = np.asarray(O, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    return float(np.abs(O - ref).max() / np.abs(ref).max())


def parity_rows(N, n=64, seed=0):
    """Rows compared against the oracle on a long sequence: both ends, tile boundaries, random rows."""
    r = np.random.Generator(np.random.PCG64(seed))
    fixed = [0, 1, N - 2, N - 1] + [b for b in (127, 128, 129, 4095, 4096, 65535, 65536) if b < N]
    return np.unique(np.concatenate([np.array(fixed, dtype=np.int64), r.integers(0, N, size=n, dtype=np.int64)]))


def run_gma(args, world, rank, local):
    import torch
    import torch.distributed as dist

    from gaussian_mixture_sequence_gma_gb300 import gma

    if world > 1:
        dist.init_process_group("nccl")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    peaks = load_peaks()
    mufu_rate = gma.probe_ex2_rate(dev)
    w = workloads()[args.workload]
    B, H, N, K = w.B, w.H, w.N, w.K
    inp = make_workload(w)
    t = to_dev(inp, dev)
    stream = torch.cuda.current_stream(dev)
    prob_b = gma.problem(B, H, N, K, torch.bfloat16, w.eps)
    ws_b = gma.alloc_workspace(prob_b, gma.OP_BIDIR, dev)
    ws_c = gma.alloc_workspace(prob_b, gma.OP_CAUSAL, dev)
    Ob = torch.empty((B, H, N, w.dv), dtype=torch.bfloat16, device=dev)
    Oc = torch.empty_like(Ob)

    def step(q, k, v):
        gma.forward_bidir(q, k, v, t["mu"], t["sigma2"], t["log_pi"], w.eps, out=Ob, workspace=ws_b)
        gma.forward_causal(q, k, v, t["mu"], t["sigma2"], t["log_pi"], w.eps, out=Oc, workspace=ws_c)

    def barrier():
        torch.cuda.synchronize(dev)
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize(dev)

    def timed(fn, n):
        barrier()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        w0 = time.time()
        e0.record(stream)
        for _ in range(n):
            fn()
        e1.record(stream)
        barrier()
        w1 = time.time()
        ms = max_over_ranks(e0.elapsed_time(e1), world, dev)
        return ms, (w0, w1)

    # per-call distribution: each call bracketed by its own events, with L2 flushed (a 2 x L2 buffer
    # written) outside the bracket before every call; returns [p10, median, p90] in ms
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    flush_buf = torch.empty(max(2 * l2, 1 << 20) // 4, dtype=torch.float32, device=dev)

    def timed_each(fn, n):
        barrier()
        ts = []
        for _ in range(n):
            flush_buf.zero_()
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record(stream)
            fn()
            b.record(stream)
            b.synchronize()
            ts.append(a.elapsed_time(b))
        return [float(x) for x in np.percentile(ts, [10, 50, 90])]

    clocks = ClockSampler(local)
    for _ in range(args.warmup):
        step(t["Q"], t["K"], t["V"])
    if gma.check_device_error(ws_b) != gma.GMA_OK or gma.check_device_error(ws_c) != gma.GMA_OK:
        raise RuntimeError("device wait timed out during warm-up")
    clocks.start()
    n0 = gma.launch_count()
    ms, win = timed(lambda: step(t["Q"], t["K"], t["V"]), args.steps)
    launches = gma.launch_count() - n0
    clocks.mark(*win)
    ms_per_step = ms / args.steps
    units_per_step = 2 * B * H * N
    value = whole_job_rate(units_per_step, ms_per_step, world)

    step_dist = timed_each(lambda: step(t["Q"], t["K"], t["V"]), args.steps)

    # per-kernel durations (events on the launch stream), same step loop
    gma.profile_enable(True)
    _, win = timed(lambda: step(t["Q"], t["K"], t["V"]), args.steps)
    gma.profile_enable(False)
    clocks.mark(*win)
    prof = gma.profile_read()

    # end to end through the public API with host buffers: H2D of Q,K,V and D2H of both outputs per step
    host = {k: torch.from_numpy(bf16_bits(inp[k]).view(np.int16)).view(torch.bfloat16).pin_memory()
            for k in ("Q", "K", "V")}
    dq, dk, dv_ = (torch.empty_like(t["Q"]), torch.empty_like(t["K"]), torch.empty_like(t["V"]))
    hb = torch.empty(Ob.shape, dtype=torch.bfloat16).pin_memory()
    hc = torch.empty(Oc.shape, dtype=torch.bfloat16).pin_memory()

    # pipelined over the B*H (batch, head) units: unit u's inputs go up on one stream while unit u-1
    # computes (one bidirectional and one causal call per unit, on the launch stream) and unit u-2's
    # outputs come down on a third; the step ends when the last output has landed in host memory
    U = B * H
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    prob_u = gma.problem(1, 1, N, K, torch.bfloat16, w.eps)
    ws_bu = gma.alloc_workspace(prob_u, gma.OP_BIDIR, dev)
    ws_cu = gma.alloc_workspace(prob_u, gma.OP_CAUSAL, dev)
    hv = {k: host[k].view(U, 1, 1, N, -1) for k in ("Q", "K", "V")}
    dvw = {"Q": dq.view(U, 1, 1, N, -1), "K": dk.view(U, 1, 1, N, -1), "V": dv_.view(U, 1, 1, N, -1)}
    obv, ocv = Ob.view(U, 1, 1, N, -1), Oc.view(U, 1, 1, N, -1)
    hbv, hcv = hb.view(U, 1, 1, N, -1), hc.view(U, 1, 1, N, -1)
    ev_in = [torch.cuda.Event() for _ in range(U)]
    ev_c = [torch.cuda.Event() for _ in range(U)]

    def e2e_step():
        s_in.wait_stream(stream)  # the previous step's calls have read the device inputs
        for u in range(U):
            with torch.cuda.stream(s_in):
                for k in ("Q", "K", "V"):
                    dvw[k][u].copy_(hv[k][u], non_blocking=True)
                ev_in[u].record(s_in)
            stream.wait_event(ev_in[u])
            hh = u % H
            pu = (t["mu"][hh:hh + 1], t["sigma2"][hh:hh + 1], t["log_pi"][hh:hh + 1])
            gma.forward_bidir(dvw["Q"][u], dvw["K"][u], dvw["V"][u], *pu, w.eps, out=obv[u], workspace=ws_bu)
            gma.forward_causal(dvw["Q"][u], dvw["K"][u], dvw["V"][u], *pu, w.eps, out=ocv[u], workspace=ws_cu)
            ev_c[u].record(stream)
            s_out.wait_event(ev_c[u])
            with torch.cuda.stream(s_out):
                hbv[u].copy_(obv[u], non_blocking=True)
                hcv[u].copy_(ocv[u], non_blocking=True)
        stream.wait_stream(s_out)

    for _ in range(2):
        e2e_step()
    e2e_ms, win = timed(e2e_step, args.steps)
    clocks.mark(*win)
    clk = clocks.stop()
    e2e_value = whole_job_rate(units_per_step, e2e_ms / args.steps, world)
    # the pipelined per-unit calls must give what the one batched call gives (up to the order of the
    # float32 reductions across CTAs)
    step(t["Q"], t["K"], t["V"])
    torch.cuda.synchronize(dev)
    for dev_o, host_o in ((Ob, hb), (Oc, hc)):
        ref_o = dev_o.float().cpu()
        if (host_o.float() - ref_o).abs().max().item() > 1e-2 * ref_o.abs().max().item():
            raise RuntimeError("end-to-end outputs differ from the device-resident step")
    h2d = sum(host[k].numel() * 2 for k in ("Q", "K", "V"))
    d2h = (hb.numel() + hc.numel()) * 2

    if gma.check_device_error(ws_b) != gma.GMA_OK or gma.check_device_error(ws_c) != gma.GMA_OK:
        raise RuntimeError("device wait timed out in the timed region")

    # roofline of the dominant kernel
    dom = max(prof.items(), key=lambda kv: kv[1][1]) if prof else None
    roof = None
    if dom:
        name, (cnt, tot_ms) = dom
        avg_s = tot_ms / cnt * 1e-3
        bound = kernel_bound(name)
        fl = kernel_flops(name, K) * B * H * N
        achieved = fl / avg_s / 1e12
        if bound == "tensor":
            peak, unit, src = peaks["bf16"], "TFLOP/s", "bf16 dense, %s (burst)" % peaks["source"]
        else:
            peak = 152 * 128 * 2 * peaks["sm_max_mhz"] * 1e6 / 1e12
            unit, src = "TFLOP/s", "fp32 FFMA: 152 SMs x 128 lanes x 2 flop x max SM clock (derived)"
        tr = traffic_for(name)
        roof = {"bound": bound, "achieved": achieved, "peak": peak, "unit": unit, "frac": achieved / peak,
                "traffic": tr, "kernel": name, "avg_launch_us": avg_s * 1e6, "peak_source": src}
        if bound == "tensor" and peaks.get("bf16_sus"):
            roof["frac_of_sustained"] = achieved / peaks["bf16_sus"]

    # whole-path roofline (spec definition): slowest of tensor, MUFU and HBM per token*head
    t_tensor = flop_per_tokhead(K) / (peaks["bf16"] * 1e12)
    t_mufu = 2 * K / mufu_rate
    t_hbm = 4 * 64 * 2 / (peaks["hbm"] * 1e9)
    bound_rate = 1.0 / max(t_tensor, t_mufu, t_hbm)
    path = {"bound_tok_heads_per_s": bound_rate, "frac": value / world / bound_rate,
            "binding": ["tensor", "mufu", "hbm"][int(np.argmax([t_tensor, t_mufu, t_hbm]))],
            "per_form_ms": {}}
    kernels = {k: {"launches": c, "total_ms": m, "avg_us": 1e3 * m / c} for k, (c, m) in prof.items()}

    # per-form times and the long-context sweep (time and peak memory vs N)
    sweep = {}
    if args.sweep and rank == 0 and world == 1:
        for n in SWEEP:
            wi = workloads()["sweep_bf16_B1H8N%dK256" % n]
            ii = make_workload(wi) if n != N else inp
            ti = to_dev(ii, dev) if n != N else t
            pb = gma.problem(wi.B, wi.H, n, wi.K, torch.bfloat16, wi.eps)
            entry = {}
            for form, op, fn in (("bidir", gma.OP_BIDIR, gma.forward_bidir), ("causal", gma.OP_CAUSAL, gma.forward_causal)):
                ws = gma.alloc_workspace(pb, op, dev)
                out = torch.empty((wi.B, wi.H, n, 64), dtype=torch.bfloat16, device=dev)
                for _ in range(3):
                    fn(ti["Q"], ti["K"], ti["V"], ti["mu"], ti["sigma2"], ti["log_pi"], wi.eps, out=out, workspace=ws)
                reps = max(3, min(50, int(2e6 // n)))
                m, _ = timed(lambda: fn(ti["Q"], ti["K"], ti["V"], ti["mu"], ti["sigma2"], ti["log_pi"], wi.eps,
                                        out=out, workspace=ws), reps)
                torch.cuda.synchronize(dev)
                torch.cuda.reset_peak_memory_stats(dev)
                base = torch.cuda.memory_allocated(dev)
                ws2 = gma.alloc_workspace(pb, op, dev)
                out2 = torch.empty_like(out)
                fn(ti["Q"], ti["K"], ti["V"], ti["mu"], ti["sigma2"], ti["log_pi"], wi.eps, out=out2, workspace=ws2)
                torch.cuda.synchronize(dev)
                peak_call = torch.cuda.max_memory_allocated(dev) - base
                inputs_b = 3 * wi.B * wi.H * n * 64 * 2
                dist_ms = timed_each(lambda: fn(ti["Q"], ti["K"], ti["V"], ti["mu"], ti["sigma2"], ti["log_pi"],
                                                wi.eps, out=out, workspace=ws), min(reps, 20))
                entry[form] = {"ms": m / reps, "tok_heads_per_s": wi.B * wi.H * n / (m / reps * 1e-3),
                               "ms_p10_median_p90_l2_flushed": dist_ms,
                               "workspace_bytes": ws.numel(), "call_peak_bytes_beyond_inputs": peak_call,
                               "inputs_bytes": inputs_b}
                del ws, out, ws2, out2
            sweep[str(n)] = entry
            if n == N:
                path["per_form_ms"] = {f: entry[f]["ms"] for f in entry}

    # widened rows: cross-attention (queries of one sequence reading the memory of another) and the
    # causal decode step (state resident between calls), each timed with CUDA events like the sweep
    extensions = None
    if args.sweep and rank == 0 and world == 1:
        extensions = {}
        from gaussian_mixture_sequence_gma_gb300.inputs import make_cross_inputs
        Bc, Hc, Nq, Nk, Kc = 1, 8, 16384, 131072, 256
        ci = to_dev(make_cross_inputs(Bc, Hc, Nq, Nk, Kc, dtype="bf16", seed=13), dev)
        pc = gma.problem(Bc, Hc, Nq, Kc, torch.bfloat16, 1e-6)
        wsc = gma.alloc_workspace(pc, gma.OP_CROSS, dev)
        outc = torch.empty((Bc, Hc, Nq, 64), dtype=torch.bfloat16, device=dev)
        call = lambda: gma.forward_cross(ci["Q"], ci["K"], ci["V"], ci["mu"], ci["sigma2"], ci["log_pi"], 1e-6,
                                         out=outc, workspace=wsc)
        for _ in range(3):
            call()
        m, _ = timed(call, 20)
        t_call = m / 20 * 1e-3
        flop = flop_per_tokhead(Kc) / 2 * Bc * Hc * (Nq + Nk)  # each query and each key: logits + read / write
        extensions["cross_bf16_B1H8_N16384_Nk131072_K256"] = {
            "ms": t_call * 1e3, "tok_heads_per_s": Bc * Hc * (Nq + Nk) / t_call,
            "tflops_algorithmic": flop / t_call / 1e12, "frac_of_bf16_peak": flop / t_call / 1e12 / peaks["bf16"]}
        del ci, wsc, outc
        Bd, Hd, Kd, N0 = 8, 12, 256, 2048
        di = to_dev(make_inputs(Bd, Hd, N0 + 64, Kd, dtype="bf16", seed=3, sigma_raw_std=0.5, projection=True), dev)
        sl = lambda x, a, b: x[:, :, a:b].contiguous()
        state = gma.causal_state(sl(di["K"], 0, N0), sl(di["V"], 0, N0), di["mu"], di["sigma2"], di["log_pi"])
        pd = gma.problem(Bd, Hd, 1, Kd, torch.bfloat16, 1e-6)
        wsd = gma.alloc_workspace(pd, gma.OP_CAUSAL_DECODE, dev)
        toks = [(sl(di["Q"], N0 + i, N0 + i + 1), sl(di["K"], N0 + i, N0 + i + 1), sl(di["V"], N0 + i, N0 + i + 1))
                for i in range(64)]
        outd = torch.empty((Bd, Hd, 1, 64), dtype=torch.bfloat16, device=dev)
        it = [0]

        def decode_step():
            q, k, v = toks[it[0] % 64]
            it[0] += 1
            gma.causal_decode(q, k, v, di["mu"], di["sigma2"], di["log_pi"], state, 1e-6, out=outd, workspace=wsd)
        for _ in range(5):
            decode_step()
        # 64 steps captured in one CUDA graph, so the device time per step is not hidden behind the
        # host-side cost of a Python call per token; eager timing if capture is not possible
        try:
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                for _ in range(64):
                    decode_step()
            g.replay()
            m, _ = timed(g.replay, 5)
            t_step = m / (5 * 64) * 1e-3
            how = "CUDA graph of 64 steps"
        except Exception as exc:  # noqa: BLE001
            m, _ = timed(decode_step, 200)
            t_step = m / 200 * 1e-3
            how = "eager (graph capture failed: %s)" % type(exc).__name__
        state_bytes = 2 * Bd * Hd * Kd * 65 * 4  # read + write of the resident state per step
        t_hbm = state_bytes / (peaks["hbm"] * 1e9)
        # the same steps with the parameters folded once (fixed parameters while decoding): one launch per
        # step instead of two
        wsp = gma.decode_prepare(di["mu"], di["sigma2"], di["log_pi"], dtype=torch.bfloat16)

        def decode_step_prepared():
            q, k, v = toks[it[0] % 64]
            it[0] += 1
            gma.causal_decode_prepared(q, k, v, state, wsp, 1e-6, out=outd)
        for _ in range(5):
            decode_step_prepared()
        try:
            g2 = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g2):
                for _ in range(64):
                    decode_step_prepared()
            g2.replay()
            m, _ = timed(g2.replay, 5)
            t_prep = m / (5 * 64) * 1e-3
        except Exception:  # noqa: BLE001
            m, _ = timed(decode_step_prepared, 200)
            t_prep = m / 200 * 1e-3
        extensions["decode_bf16_B8H12K256_1token"] = {
            "us_per_step": t_step * 1e6, "tok_heads_per_s": Bd * Hd / t_step, "state_bytes_per_step": state_bytes,
            "hbm_bound_us": t_hbm * 1e6, "frac_of_hbm_bound": t_hbm / t_step,
            "launches_per_step": 2, "timing": how,
            "prepared_us_per_step": t_prep * 1e6, "prepared_frac_of_hbm_bound": t_hbm / t_prep,
            "prepared_note": "parameters folded once (gma_decode_prepare), one launch per step"}
        del di, state, wsd, wsp, toks, outd
        # Transformer-block form at the language-model block shape: projection GEMM + layout + causal forward
        from gaussian_mixture_sequence_gma_gb300.inputs import make_projected_inputs
        Bp, Hp, Np, Kp_, dmp = 8, 12, 2048, 256, 768
        pi_ = make_projected_inputs(Bp, Hp, Np, Kp_, dm=dmp, dtype="bf16", seed=3)
        tp = {k: torch.from_numpy(np.ascontiguousarray(pi_[k])).to(dev) for k in ("mu", "sigma2", "log_pi", "bqkv")}
        for k in ("X", "Wqkv"):
            tp[k] = torch.from_numpy(bf16_bits(pi_[k]).view(np.int16)).to(dev).view(torch.bfloat16)
        pp_ = gma.problem(Bp, Hp, Np, Kp_, torch.bfloat16, 1e-6)
        wsp = gma.alloc_workspace(pp_, gma.OP_PROJECTED_CAUSAL, dev)
        outp = torch.empty((Bp, Hp, Np, 64), dtype=torch.bfloat16, device=dev)
        callp = lambda: gma.forward_projected(tp["X"], tp["Wqkv"], tp["bqkv"], tp["mu"], tp["sigma2"], tp["log_pi"],
                                              causal=True, out=outp, workspace=wsp)
        qkv = [torch.empty((Bp, Hp, Np, 64), dtype=torch.bfloat16, device=dev) for _ in range(3)]
        callu = lambda: gma.forward_causal(qkv[0], qkv[1], qkv[2], tp["mu"], tp["sigma2"], tp["log_pi"], 1e-6)
        for _ in range(3):
            callp()
            callu()
        mp, _ = timed(callp, 10)
        mu_, _ = timed(callu, 10)
        t_p = mp / 10 * 1e-3
        gemm_flop = 2.0 * Bp * Np * dmp * 3 * Hp * 64
        gma_flop = flop_per_tokhead(Kp_) * Bp * Hp * Np
        extensions["projected_causal_bf16_B8H12N2048K256_dm768"] = {
            "ms": t_p * 1e3, "tok_heads_per_s": Bp * Hp * Np / t_p, "forward_only_ms": mu_ / 10,
            "projection_ms": t_p * 1e3 - mu_ / 10, "tflops_algorithmic": (gemm_flop + gma_flop) / t_p / 1e12,
            "frac_of_bf16_peak": (gemm_flop + gma_flop) / t_p / 1e12 / peaks["bf16"],
            "note": "projection = one tcgen05 GEMM with bias and layout in its epilogue (bf16 Q, K, V round-trip HBM)"}
        del tp, wsp, outp, qkv
        # backward pass of the bidirectional form on the bidir bf16 workload shape
        wb = workloads()["bidir_bf16_B4H8N4096K128"]
        bi = to_dev(make_workload(wb), dev)
        gO = torch.randn((wb.B, wb.H, wb.N, 64), device=dev).to(torch.bfloat16)
        pbk = gma.problem(wb.B, wb.H, wb.N, wb.K, torch.bfloat16, wb.eps)
        wsb = gma.alloc_workspace(pbk, gma.OP_BACKWARD_BIDIR, dev)
        callb = lambda: gma.backward_bidir(bi["Q"], bi["K"], bi["V"], bi["mu"], bi["sigma2"], bi["log_pi"], gO, wb.eps,
                                           workspace=wsb)
        callf = lambda: gma.forward_bidir(bi["Q"], bi["K"], bi["V"], bi["mu"], bi["sigma2"], bi["log_pi"], wb.eps)
        for _ in range(2):
            callb()
            callf()
        mb, _ = timed(callb, 5)
        mf, _ = timed(callf, 5)
        extensions["backward_bidir_bf16_B4H8N4096K128"] = {
            "ms": mb / 5, "tok_heads_per_s": wb.B * wb.H * wb.N / (mb / 5 * 1e-3), "forward_ms": mf / 5,
            "backward_over_forward": mb / mf, "workspace_bytes": wsb.numel(),
            "note": "state and responsibilities by the tensor-core forward kernels; query, key and parameter passes in float32 on the CUDA cores"}
        del wsb
        pbc = gma.problem(wb.B, wb.H, wb.N, wb.K, torch.bfloat16, wb.eps)
        wsc = gma.alloc_workspace(pbc, gma.OP_BACKWARD_CAUSAL, dev)
        callc = lambda: gma.backward_causal(bi["Q"], bi["K"], bi["V"], bi["mu"], bi["sigma2"], bi["log_pi"], gO,
                                            wb.eps, workspace=wsc)
        callfc = lambda: gma.forward_causal(bi["Q"], bi["K"], bi["V"], bi["mu"], bi["sigma2"], bi["log_pi"], wb.eps)
        for _ in range(2):
            callc()
            callfc()
        mc, _ = timed(callc, 3)
        mfc, _ = timed(callfc, 5)
        extensions["backward_causal_bf16_B4H8N4096K128"] = {
            "ms": mc / 3, "tok_heads_per_s": wb.B * wb.H * wb.N / (mc / 3 * 1e-3), "forward_ms": mfc / 5,
            "backward_over_forward": (mc / 3) / (mfc / 5), "workspace_bytes": wsc.numel(),
            "note": "float32 CUDA-core kernels"}
        del bi, gO, wsc

    # CPU baseline: the oracle as it stands on a bounded sample of the same workload (rank 0 only).
    # The same leg measures parity: the timed step's outputs, and every listed workload's, against the
    # float64 oracle (max |O - O_ref| / max |O_ref|; sampled rows on the long sequences).
    cpu = None
    parity = None
    configs = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        from oracle import oracle as orc
        n_pos = min(CPU_SAMPLE_N, N)
        dt, units, cores, host = oracle_sample(inp, n_pos)
        cpu = {"value": units / dt, "unit": UNIT, "cores": cores, "host_cores": host, "kind": "oracle",
               "sample": "first %d positions of each of the %d (b,h) units, bidirectional + causal (%.1f s)"
                         % (n_pos, B * H, dt)}
        step(t["Q"], t["K"], t["V"])
        torch.cuda.synchronize(dev)
        rows = parity_rows(N, seed=N)
        parity = {"workload": w.name, "rows_per_head": int(len(rows)), "tolerance": 2e-2,
                  "measure": "max |O - O_ref| / max |O_ref| against the float64 oracle"}
        for form, O_dev, causal in (("bidir", Ob, False), ("causal", Oc, True)):
            ref = orc.forward(inp["Q"], inp["K"], inp["V"], inp["mu"], inp["sigma2"], inp["log_pi"], w.eps,
                              causal=causal, rows=rows)
            parity[form] = rel_err(O_dev.float().cpu().numpy()[:, :, rows], ref)
        # the listed workloads (configs 1-4): device time per call, fraction of the path roofline, parity
        configs = {}
        for name in ("bidir_f32_B1H1N1024K16", "bidir_bf16_B4H8N4096K128", "causal_bf16_B4H8N4096K128",
                     "causal_lm_bf16_B8H12N2048K256"):
            wc = workloads()[name]
            ic = make_workload(wc)
            tc_ = to_dev(ic, dev)
            fn = gma.forward_causal if wc.causal else gma.forward_bidir
            dt_ = torch.float32 if wc.dtype == "f32" else torch.bfloat16
            pc_ = gma.problem(wc.B, wc.H, wc.N, wc.K, dt_, wc.eps)
            wsx = gma.alloc_workspace(pc_, gma.OP_CAUSAL if wc.causal else gma.OP_BIDIR, dev)
            outx = torch.empty((wc.B, wc.H, wc.N, 64), dtype=dt_, device=dev)
            callx = lambda: fn(tc_["Q"], tc_["K"], tc_["V"], tc_["mu"], tc_["sigma2"], tc_["log_pi"], wc.eps, out=outx,
                               workspace=wsx)
            for _ in range(5):
                callx()
            reps = 50
            mx, _ = timed(callx, reps)
            t_call = mx / reps * 1e-3
            esz = 4 if wc.dtype == "f32" else 2
            t_bound = max(flop_per_tokhead(wc.K) / (peaks["bf16"] * 1e12), 2 * wc.K / mufu_rate,
                          4 * 64 * esz / (peaks["hbm"] * 1e9)) * wc.B * wc.H * wc.N
            rws = None if wc.B * wc.H * wc.N <= 131072 else parity_rows(wc.N, seed=7)
            ref = orc.forward(ic["Q"], ic["K"], ic["V"], ic["mu"], ic["sigma2"], ic["log_pi"], wc.eps,
                              causal=bool(wc.causal), rows=rws)
            got = outx.float().cpu().numpy()
            if rws is not None:
                got = got[:, :, rws]
            configs[name] = {"ms": t_call * 1e3, "tok_heads_per_s": wc.B * wc.H * wc.N / t_call,
                             "frac_of_path_roofline": t_bound / t_call, "parity_max_rel_err": rel_err(got, ref),
                             "parity_rows": "all" if rws is None else "%d per head" % len(rws),
                             "tolerance": 1e-3 if wc.dtype == "f32" else 2e-2}
            del wsx, outx, tc_

    if rank == 0:
        line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
                "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
                "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded; shapes and distributions of the workload)",
                "config": config_dict(w),
                "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
                "gpu_launches": int(launches), "roofline": roof, "cpu_baseline": cpu, "clocks": clk,
                "step_ms_p10_median_p90_l2_flushed": step_dist,
                "roofline_path": path, "kernels": kernels, "sweep": sweep or None, "extensions": extensions,
                "parity": parity, "configs": configs, "mufu_ex2_per_s": mufu_rate}
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["gma", "reference"], default="gma")
    ap.add_argument("--workload", default=WORKLOAD)
    ap.add_argument("--no-sweep", dest="sweep", action="store_false")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--ref-positions", type=int, default=2048)
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    world, rank, local = dist_setup()
    if args.impl == "reference":
        return run_reference(args, world, rank)
    return run_gma(args, world, rank, local)


if __name__ == "__main__":
    sys.exit(main())
