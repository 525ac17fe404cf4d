#!/usr/bin/env python3
"""Throughput of the chunked gated delta rule forward on GB300.

One step = one whole forward (chunk enumeration, prep, state scan, output) over
the packed 64k-token workload: 65536 tokens in segments of uniform random
length in [1, 8192] plus 16 trailing length-0 segments, H = 32 heads,
dk = dv = 128, bf16 q/k/v/beta, fp32 g, no initial or final state.  Inputs are
seeded synthetic tensors (q, k L2-normalised, v Gaussian, g = logsigmoid(N(3,1)),
beta = sigmoid(N(0,1))) resident in HBM before timing; they total 2.16 GB, more
than the 129 MB L2, so no flush is needed between steps.

Prints ONE JSON line (rank 0).  ``--impl reference`` times the fp64 CPU oracle
on the host cores instead (a deliberately slow baseline).
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "GDR chunk-fwd tokens/s (H=32, d=128, 64k packed) & % of tensor/HBM roofline"
WORKLOAD = "packed_64k_h32"
TRAFFIC_RECORD = os.path.join(ROOT, "profiles", "k_fused_traffic.json")


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=100)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--op", choices=["fwd", "bwd"], default="fwd",
                   help="fwd: the forward (the headline); bwd: the backward")
    p.add_argument("--path", choices=["auto", "fused", "staged", "fused_whole"], default="auto")
    p.add_argument("--workload", default=WORKLOAD)
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--cpu-seconds", type=float, default=12.0,
                   help="target CPU seconds for the oracle sample")
    p.add_argument("--record-traffic", metavar="NCU_CSV",
                   help="write the fused kernel's traffic record from an ncu CSV log of "
                        "dram__bytes_read.sum / dram__bytes_write.sum, then exit")
    p.add_argument("--traffic-out", default=None,
                   help="where --record-traffic writes (default: the committed record)")
    p.add_argument("--traffic-command", default="",
                   help="the capture command, stored in the record")
    return p.parse_args()


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        d = json.load(open(path))
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), "measured"
    except Exception:
        return 6800.0, 1900.0, "fallback"


def algorithmic_bytes(w) -> int:
    """q, k, v, o in bf16; g in fp32; beta in bf16; h0/ht in fp32 when present."""
    T, Hk, H, dk, dv = w.T, w.Hk, w.H, w.dk, w.dv
    b = T * (2 * dk * Hk * 2 + 2 * dv * H * 2 + 4 * H + 2 * H)
    state = w.n_seq * H * dk * dv * 4
    b += state * ((w.h0 is not None) + bool(w.want_ht))
    return int(b)


def algorithmic_flops(w) -> int:
    """Dense-tile FLOPs, 2 (5 c^2 d + 3 c d^2) per chunk of c tokens per value head."""
    d = w.dk
    f = 0
    for n in w.lengths():
        full, rem = divmod(n, 64)
        f += full * 2 * (5 * 64 * 64 * d + 3 * 64 * d * d)
        if rem:
            f += 2 * (5 * rem * rem * d + 3 * rem * d * d)
    return int(f * w.H)


# the sources the fused forward kernel is compiled from
KERNEL_SOURCES = ("gdr_fused.cu", "gdr_internal.cuh", "gdr_tc.cuh")


def kernel_sha() -> str:
    import hashlib
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "chunked_gated_delta_gdr_gb300", "csrc")
    for f in KERNEL_SOURCES:
        h.update(open(os.path.join(csrc, f), "rb").read())
    return h.hexdigest()[:16]


def read_traffic(expected_sha: str, workload: str):
    """DRAM bytes per launch of the fused kernel from the machine-written record of an
    ncu capture (``--record-traffic``), scaled to ``workload``; None unless the record
    was taken on the current kernel sources (same sha256) and names this workload."""
    try:
        rec = json.load(open(TRAFFIC_RECORD))
    except (OSError, ValueError):
        return None
    if rec.get("source_sha256") != expected_sha:
        return None
    scaled = rec.get("scaled", {}).get(workload)
    return None if scaled is None else float(scaled["dram_bytes_per_launch"])


def record_traffic(csv_path: str, case: str, out_path: str, command: str) -> int:
    """Write the traffic record from an ncu CSV log of dram__bytes_read.sum and
    dram__bytes_write.sum for k_fused launches of workload ``case``: bytes per launch
    (mean over the captured launches), the sha256 of the kernel sources computed here,
    and the figure scaled to the bench workload by algorithmic bytes (every token is
    streamed once, so traffic grows in proportion to the tokens processed)."""
    import csv
    from chunked_gated_delta_gdr_gb300.inputs import make_named
    launches = {}
    with open(csv_path) as f:
        rows = [ln for ln in f if ln.startswith('"')]
    for row in csv.DictReader(rows):
        if "k_fused" not in row["Kernel Name"]:
            continue
        m = row["Metric Name"]
        if m in ("dram__bytes_read.sum", "dram__bytes_write.sum"):
            val = float(row["Metric Value"].replace(",", ""))
            unit = row["Metric Unit"].lower()
            val *= {"byte": 1, "kbyte": 1e3, "mbyte": 1e6, "gbyte": 1e9}.get(unit, 1)
            launches.setdefault(row["ID"], {})[m] = val
    full = [v for v in launches.values() if len(v) == 2]
    if not full:
        print(f"no k_fused dram counters in {csv_path}", file=sys.stderr)
        return 1
    rd = sum(v["dram__bytes_read.sum"] for v in full) / len(full)
    wr = sum(v["dram__bytes_write.sum"] for v in full) / len(full)
    wc = make_named(case)
    alg_case = algorithmic_bytes(wc)
    rec = {"kernel": "k_fused", "source_sha256": kernel_sha(), "case": case,
           "launches": len(full), "dram_bytes_read": rd, "dram_bytes_write": wr,
           "dram_bytes_per_launch": rd + wr, "algorithmic_bytes": alg_case,
           "ratio_to_algorithmic": (rd + wr) / alg_case, "command": command, "scaled": {}}
    for name in (case, WORKLOAD):
        f = algorithmic_bytes(make_named(name)) / alg_case
        rec["scaled"][name] = {"factor": f, "dram_bytes_per_launch": (rd + wr) * f}
    with open(out_path, "w") as f:
        json.dump(rec, f, indent=1)
        f.write("\n")
    print(json.dumps(rec))
    return 0


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled while the timed region runs."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.path = os.path.join("/tmp", f"gdr_clocks_{os.getpid()}.csv")

    def start(self):
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.f.close()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for nm, val in zip(names, parts[5:9]):
                if val.lower() == "active":
                    reasons.add(nm)
        try:
            os.remove(self.path)
        except OSError:
            pass
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def cpu_oracle_sample(w, target_s: float):
    """Time the fp64 oracle on a head subset of the workload sized to ~target_s."""
    import oracle
    from chunked_gated_delta_gdr_gb300.inputs import Workload  # noqa: F401
    threads = oracle.max_threads()

    def run(heads):
        sel = lambda t: t[:, heads].contiguous()
        hk = [h // (w.H // w.Hk) for h in heads]
        t0 = time.perf_counter()
        oracle.recurrent(w.q[:, hk].contiguous(), w.k[:, hk].contiguous(), sel(w.v),
                         sel(w.g), sel(w.beta), w.scale,
                         None if w.h0 is None else w.h0[:, heads].contiguous(),
                         w.cu_seqlens, want_ht=w.want_ht)
        return time.perf_counter() - t0

    t1 = run([0])
    nh = max(1, min(w.H, int(target_s / max(t1, 1e-3))))
    heads = list(range(nh))
    el = run(heads)
    value = w.T * nh / w.H / el  # tokens/s of the whole-H workload
    return {"value": value, "unit": "tokens/s", "cores": threads, "kind": "oracle",
            "sample": f"fp64 token recurrence on {nh} of {w.H} heads of the full "
                      f"{w.name} workload ({w.T} tokens), {el:.1f} s; tokens/s scaled by "
                      f"{nh}/{w.H}"}


def max_over_ranks(x: float, dist, device="cpu") -> float:
    """The slowest rank's value (timings are reported as the max over ranks)."""
    if dist is None:
        return x
    import torch
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_tokens_per_s(world: int, tokens_per_rank: int, steps: int, max_ms: float) -> float:
    """Whole-job throughput: every rank processes its own copy of the workload."""
    return world * tokens_per_rank * steps / (max_ms / 1e3)


def dist_setup(args):
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if ws > 1:
        import torch.distributed as dist
        backend = "nccl" if os.environ.get("GDR_BENCH_BACKEND", "nccl") == "nccl" else "gloo"
        dist.init_process_group(backend)
        return dist, rank, ws
    return None, 0, 1


def bench_reference(args):
    dist, rank, ws = dist_setup(args)
    if rank != 0:
        return 0
    from chunked_gated_delta_gdr_gb300.inputs import make_named
    w = make_named(args.workload)
    # each step: the oracle on one head of the workload (a bounded sample)
    import oracle
    times = []
    heads = [0]
    for i in range(args.warmup + args.steps):
        h = [i % w.H]
        hk = [h[0] // (w.H // w.Hk)]
        t0 = time.perf_counter()
        oracle.recurrent(w.q[:, hk].contiguous(), w.k[:, hk].contiguous(),
                         w.v[:, h].contiguous(), w.g[:, h].contiguous(),
                         w.beta[:, h].contiguous(), w.scale,
                         None if w.h0 is None else w.h0[:, h].contiguous(), w.cu_seqlens,
                         want_ht=w.want_ht)
        if i >= args.warmup:
            times.append(time.perf_counter() - t0)
    per_step = sum(times) / len(times)
    value = w.T / w.H / per_step
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": per_step * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": w.name, "T": w.T, "H": w.H, "Hk": w.Hk, "d": w.dk,
                       "n_seq": w.n_seq, "step": "one value head of the workload"},
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": oracle.max_threads(),
                             "kind": "oracle",
                             "sample": "each step runs the fp64 token recurrence on one of the "
                                       f"{w.H} heads; tokens/s scaled by 1/{w.H}"},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def bench_ours(args):
    import torch
    dist, rank, ws = dist_setup(args)
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    from chunked_gated_delta_gdr_gb300 import api
    from chunked_gated_delta_gdr_gb300.inputs import make_named
    w = make_named(args.workload)
    wd = w.to(dev)
    T, H, D, N = w.T, w.H, w.dk, w.n_seq
    path = args.path
    o = torch.empty(T, H, D, dtype=torch.bfloat16, device=dev)
    ht = torch.empty(N, H, D, D, dtype=torch.float32, device=dev) if w.want_ht else None
    wsz = api.workspace_bytes(T, N, H, D, D, path)
    work = torch.empty(max(wsz, 256), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()

    def step():
        api.chunk_fwd(wd.q, wd.k, wd.v, wd.g, wd.beta, scale=w.scale, initial_state=wd.h0,
                      cu_seqlens=wd.cu_seqlens, output_final_state=w.want_ht, path=path,
                      workspace=work, out=o, final_state=ht)

    for _ in range(max(args.warmup, 3)):
        step()
    torch.cuda.synchronize()
    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.3)
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    t_wall = time.perf_counter()
    for a, b in ev:
        a.record(stream)
        step()
        b.record(stream)
    torch.cuda.synchronize()
    wall = time.perf_counter() - t_wall
    if dist is not None:
        dist.barrier()
    clocks = sampler.stop()
    per = [a.elapsed_time(b) for a, b in ev]  # ms, each step on the launching stream
    total_ms = max_over_ranks(sum(per), dist, dev)
    ms_per_step = total_ms / args.steps
    value = job_tokens_per_s(ws, T, args.steps, total_ms)
    fused = path in ("auto", "fused", "fused_whole") and _fused_available(api, wd, w)
    pieces = api.split_pieces(T, N, H) if path in ("auto", "fused") else 1
    if fused and pieces > 1:
        # chunk enumeration, split units, [empty-segment states], pass A, combine, pass B
        launches_per_step = 5 + bool(w.want_ht)
    elif fused:
        # chunk enumeration, work list, [empty-segment states], fused kernel
        launches_per_step = 3 + bool(w.want_ht)
    else:
        launches_per_step = 4
    hbm, tflops, peak_kind = peaks()
    alg_b = algorithmic_bytes(w)
    alg_f = algorithmic_flops(w)
    med_ms = statistics.median(per)
    achieved_gbs = alg_b / (med_ms / 1e3) / 1e9
    achieved_tfs = alg_f / (med_ms / 1e3) / 1e12
    line = {"metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": ws,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "bf16" if fused else "f32", "data": "synthetic",
            "config": {"workload": w.name, "T": T, "H": H, "Hk": w.Hk, "d": D, "n_seq": N,
                       "n_chunks": w.n_chunks(), "path": path, "split_pieces": pieces if fused else 1,
                       "l2": (f"inputs ({alg_b / 1e9:.2f} GB) exceed the 129 MB L2; "
                              "no flush between steps"),
                       "per_rank": "each rank runs its own copy of the workload"},
            "roofline": {"bound": "hbm", "achieved": achieved_gbs, "peak": hbm, "unit": "GB/s",
                         "frac": achieved_gbs / hbm, "peak_kind": f"{peak_kind} burst copy",
                         "traffic": read_traffic(kernel_sha(), w.name),
                         "algorithmic_bytes_per_launch": alg_b,
                         "tensor": {"achieved": achieved_tfs, "peak": tflops,
                                    "unit": "TFLOP/s", "frac": achieved_tfs / tflops,
                                    "algorithmic_flops_per_launch": alg_f},
                         "timed": "median CUDA-event time of the whole forward call per step "
                                  "(chunk enumeration included)"},
            "gpu_launches": launches_per_step * args.steps,
            "clocks": clocks,
            "wall_s_timed_region": wall}
    if not args.no_e2e:
        line["e2e"] = bench_e2e(args, api, w, dev, path, dist)
    if rank == 0 and not args.no_cpu_baseline and ws == 1:
        line["cpu_baseline"] = cpu_oracle_sample(w, args.cpu_seconds)
    if dist is not None:
        dist.destroy_process_group()
    if rank == 0:
        print(json.dumps(line), flush=True)
    return 0


def _fused_available(api, wd, w):
    try:
        api.chunk_fwd(wd.q[:64], wd.k[:64], wd.v[:64], wd.g[:64], wd.beta[:64],
                      cu_seqlens=wd.cu_seqlens.new_tensor([0, 64]), path="fused")
        return True
    except api.nat.GdrError:
        return False


def bench_e2e(args, api, w, dev, path, dist):
    """Same metric through the public API with pinned HOST inputs: every step
    copies q, k, v, g, beta (and h0) to the device, runs, and copies o (and ht)
    back; all inside the timed region."""
    import torch
    pin = lambda t: None if t is None else t.pin_memory()
    hq, hk, hv, hg, hb, hh0 = map(pin, (w.q, w.k, w.v, w.g, w.beta, w.h0))
    o_h = torch.empty(w.T, w.H, w.dv, dtype=torch.bfloat16).pin_memory()
    ht_h = (torch.empty(w.n_seq, w.H, w.dk, w.dv, dtype=torch.float32).pin_memory()
            if w.want_ht else None)
    work = torch.empty(max(api.workspace_bytes(w.T, w.n_seq, w.H, w.dk, w.dv, path), 256),
                       dtype=torch.uint8, device=dev)

    def step():
        api.chunk_fwd(hq, hk, hv, hg, hb, scale=w.scale, initial_state=hh0,
                      cu_seqlens=w.cu_seqlens, output_final_state=w.want_ht, path=path,
                      workspace=work, out=o_h, final_state=ht_h)

    for _ in range(2):
        step()
    torch.cuda.synchronize()
    steps = max(3, min(args.steps, 20))
    t0 = time.perf_counter()
    for _ in range(steps):
        step()
    torch.cuda.synchronize()
    el = max_over_ranks(time.perf_counter() - t0, dist, dev)
    ws = dist.get_world_size() if dist is not None else 1
    h2d = sum(t.numel() * t.element_size() for t in (hq, hk, hv, hg, hb, hh0, w.cu_seqlens)
              if t is not None)
    d2h = o_h.numel() * 2 + (ht_h.numel() * 4 if ht_h is not None else 0)
    return {"value": ws * w.T * steps / el, "unit": "tokens/s", "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "steps": steps,
            "timed": "host wall clock around the public chunk_fwd call on pinned host tensors"}


METRIC_BWD = "GDR chunk-bwd tokens/s (H=32, d=128, 64k packed) & % of tf32 tensor roofline"
TF32_PER_BF16 = 1.1 / 2.25


def algorithmic_flops_bwd(w) -> int:
    """Per chunk of c tokens and value head: the dense products of the chunk backward
    (6 c d^2 + 12 c^2 d + 2 c^3 multiply-adds: dV', dS_0, dQ, dK, dW, E, T^T dU, T^T dW,
    dT, dA, B K) plus the forward recompute (the forward's 5 c^2 d + 3 c d^2)."""
    d = w.dk
    cu = [int(x) for x in w.cu_seqlens.tolist()]
    tot = 0
    for s, e in zip(cu[:-1], cu[1:]):
        L = max(e - s, 0)
        for c0 in range(0, L, 64):
            c = min(64, L - c0)
            tot += 2 * (9 * c * d * d + 17 * c * c * d + 2 * c ** 3)
    return tot * w.H


def algorithmic_bytes_bwd(w) -> int:
    """Reads q, k, v, dout (bf16), g (fp32), beta (bf16), h0 and dht (fp32, if present);
    writes dq, dk, dv, dg, dbeta (fp32) and dh0 (fp32, if h0 is given)."""
    T, Hk, H, dk, dv = w.T, w.Hk, w.H, w.dk, w.dv
    b = T * (2 * dk * Hk * 2 + 2 * dv * H * 2 + 4 * H + 2 * H)
    b += T * (2 * dk * Hk * 4 + dv * H * 4 + 8 * H)
    states = w.n_seq * H * dk * dv * 4
    b += states * ((w.h0 is not None) * 2 + bool(w.want_ht))
    return b


def _upstream_bwd(w, dev):
    import torch
    gen = torch.Generator().manual_seed(4321)
    do = (0.1 * torch.randn(w.T, w.H, w.dv, generator=gen)).to(torch.bfloat16)
    dht = (0.1 * torch.randn(w.n_seq, w.H, w.dk, w.dv, generator=gen)) if w.want_ht else None
    return do, dht


def bench_ours_bwd(args):
    import torch
    dist, rank, ws = dist_setup(args)
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    from chunked_gated_delta_gdr_gb300 import api
    from chunked_gated_delta_gdr_gb300.inputs import make_named
    w = make_named(args.workload)
    wd = w.to(dev)
    do_h, dht_h = _upstream_bwd(w, dev)
    do, dht = do_h.to(dev), None if dht_h is None else dht_h.to(dev)
    want_dh0 = w.h0 is not None
    work = torch.empty(max(api.bwd_workspace_bytes(w.T, w.n_seq, w.Hk, w.H, w.dk, w.dv), 256),
                       dtype=torch.uint8, device=dev)

    def step():
        return api.chunk_bwd(wd.q, wd.k, wd.v, wd.g, wd.beta, do, scale=w.scale,
                             initial_state=wd.h0, cu_seqlens=wd.cu_seqlens, dht=dht,
                             want_dh0=want_dh0, workspace=work)

    for _ in range(max(args.warmup, 3)):
        step()
    torch.cuda.synchronize()
    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.3)
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    t_wall = time.perf_counter()
    for a, b in ev:
        a.record(stream)
        step()
        b.record(stream)
    torch.cuda.synchronize()
    wall = time.perf_counter() - t_wall
    if dist is not None:
        dist.barrier()
    clocks = sampler.stop()
    per = [a.elapsed_time(b) for a, b in ev]
    total_ms = max_over_ranks(sum(per), dist, dev)
    med_ms = statistics.median(per)
    flops = algorithmic_flops_bwd(w)
    byts = algorithmic_bytes_bwd(w)
    hbm, bf16_tf, peak_kind = peaks()
    # the dense products run as tf32 tensor-core tiles: the tf32 peak is the measured
    # bf16 peak times the nominal tf32 / bf16 ratio (1.1 / 2.25 PFLOP/s dense)
    peak = bf16_tf * TF32_PER_BF16
    achieved = flops / (med_ms / 1e3) / 1e12
    # chunk enumeration (2), forward recompute (2), five backward kernels, grouped heads
    launches = 2 + 2 + 5 + (w.H != w.Hk)
    line = {"metric": METRIC_BWD, "value": job_tokens_per_s(ws, w.T, args.steps, total_ms),
            "unit": "tokens/s", "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": total_ms / args.steps, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": {"workload": w.name, "op": "backward", "T": w.T, "H": w.H, "Hk": w.Hk,
                       "d": w.dk, "n_seq": w.n_seq, "n_chunks": w.n_chunks(),
                       "upstream": "dout = 0.1 N(0,1) bf16" + (", dht = 0.1 N(0,1)" if dht is not None else ""),
                       "l2": "inputs and fp32 gradients exceed the 129 MB L2; no flush between steps"},
            "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                         "frac": achieved / peak,
                         "peak_kind": f"{peak_kind} bf16 burst x nominal tf32/bf16 ratio 1.1/2.25",
                         "traffic": None, "algorithmic_flops_per_launch": flops,
                         "hbm": {"algorithmic_bytes_per_launch": byts,
                                 "achieved_gbs": byts / (med_ms / 1e3) / 1e9, "peak": hbm,
                                 "peak_kind": f"{peak_kind} burst copy"},
                         "timed": "median CUDA-event time of the whole backward call per step"},
            "gpu_launches": launches * args.steps, "clocks": clocks,
            "wall_s_timed_region": wall}
    if not args.no_e2e:
        hs = [t.pin_memory() for t in (w.q, w.k, w.v, w.g, w.beta, do_h)]
        hh0 = None if w.h0 is None else w.h0.pin_memory()
        hdht = None if dht_h is None else dht_h.pin_memory()

        f32 = dict(dtype=torch.float32, pin_memory=True)
        outs_h = (torch.empty(w.T, w.Hk, w.dk, **f32), torch.empty(w.T, w.Hk, w.dk, **f32),
                  torch.empty(w.T, w.H, w.dv, **f32), torch.empty(w.T, w.H, **f32),
                  torch.empty(w.T, w.H, **f32),
                  torch.empty(w.n_seq, w.H, w.dk, w.dv, **f32) if want_dh0 else None)

        def step_host():
            return api.chunk_bwd(*hs, scale=w.scale, initial_state=hh0, cu_seqlens=w.cu_seqlens,
                                 dht=hdht, want_dh0=want_dh0, workspace=work, out=outs_h)

        step_host()
        torch.cuda.synchronize()
        n = max(3, min(args.steps, 5))
        t0 = time.perf_counter()
        for _ in range(n):
            outs = step_host()
        el = max_over_ranks(time.perf_counter() - t0, dist, dev)
        h2d = sum(t.numel() * t.element_size() for t in hs + [hh0, hdht, w.cu_seqlens]
                  if t is not None)
        d2h = sum(t.numel() * t.element_size() for t in outs if t is not None)
        line["e2e"] = {"value": ws * w.T * n / el, "unit": "tokens/s",
                       "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": n,
                       "timed": "host wall clock around the public chunk_bwd call on pinned "
                                "host tensors"}
    if rank == 0 and not args.no_cpu_baseline and ws == 1:
        line["cpu_baseline"] = cpu_oracle_bwd_sample(w, do_h, dht_h, args.cpu_seconds)
    if dist is not None:
        dist.destroy_process_group()
    if rank == 0:
        print(json.dumps(line), flush=True)
    return 0


def _oracle_bwd_heads(w, do, dht, heads):
    import oracle
    hk = [h // (w.H // w.Hk) for h in heads]
    sel = lambda t: t[:, heads].contiguous()
    t0 = time.perf_counter()
    # one value head per key head taken: the key heads are selected alongside
    oracle.recurrent_bwd(w.q[:, hk].contiguous(), w.k[:, hk].contiguous(), sel(w.v), sel(w.g),
                         sel(w.beta), w.scale, None if w.h0 is None else sel(w.h0),
                         w.cu_seqlens, sel(do), None if dht is None else sel(dht))
    return time.perf_counter() - t0


def cpu_oracle_bwd_sample(w, do, dht, target_s: float):
    """Time the fp64 oracle's backward on a head subset of the workload (~target_s)."""
    import oracle
    t1 = _oracle_bwd_heads(w, do, dht, [0])
    nh = max(1, min(w.H, int(target_s / max(t1, 1e-3))))
    el = _oracle_bwd_heads(w, do, dht, list(range(nh)))
    return {"value": w.T * nh / w.H / el, "unit": "tokens/s", "cores": oracle.max_threads(),
            "kind": "oracle",
            "sample": f"fp64 backward of the token recurrence on {nh} of {w.H} heads of the "
                      f"full {w.name} workload ({w.T} tokens), {el:.1f} s; tokens/s scaled by "
                      f"{nh}/{w.H}"}


def bench_reference_bwd(args):
    dist, rank, ws = dist_setup(args)
    if rank != 0:
        return 0
    from chunked_gated_delta_gdr_gb300.inputs import make_named
    import oracle
    w = make_named(args.workload)
    do, dht = _upstream_bwd(w, None)
    times = []
    for i in range(args.warmup + args.steps):
        el = _oracle_bwd_heads(w, do, dht, [i % w.H])
        if i >= args.warmup:
            times.append(el)
    per_step = sum(times) / len(times)
    value = w.T / w.H / per_step
    line = {"impl": "reference", "metric": METRIC_BWD, "value": value, "unit": "tokens/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": per_step * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": w.name, "op": "backward", "T": w.T, "H": w.H, "Hk": w.Hk,
                       "d": w.dk, "n_seq": w.n_seq, "step": "one value head of the workload"},
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": oracle.max_threads(),
                             "kind": "oracle",
                             "sample": "each step runs the fp64 backward on one of the "
                                       f"{w.H} heads; tokens/s scaled by 1/{w.H}"},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def main():
    args = parse()
    if args.record_traffic:
        return record_traffic(args.record_traffic, args.workload,
                              args.traffic_out or TRAFFIC_RECORD, args.traffic_command)
    if args.op == "bwd":
        return bench_reference_bwd(args) if args.impl == "reference" else bench_ours_bwd(args)
    if args.impl == "reference":
        return bench_reference(args)
    return bench_ours(args)


if __name__ == "__main__":
    sys.exit(main())
