"""Benchmark of the fused GRPO loss (advantages + forward + recompute backward).

python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                [--workload NAME]

One step = one pass of the whole path over one batch: group advantages from
the rewards, grpo_loss_fwd (policy and reference log-probs, KL, loss) and
grpo_loss_bwd (dH of the policy hidden states; with --dW also the lm_head
gradient dW), on synthetic inputs shaped
like the Llama-3.1-8B head at 20K context with 8 generations unless
--workload says otherwise. Inputs are resident in HBM for `value`; `e2e`
repeats the step through the public Python API from pinned host buffers
(host-to-device copies of the step's inputs and the read-back of the loss
inside the timed region). Under torchrun every rank runs its own replica of
the workload (weak scaling, no collective on the data path).

--impl reference times the float64 CPU oracle on a bounded sample of rows
of the same workload (rank 0 only).
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from grpo_loss_gb300 import workloads as WL  # noqa: E402
from grpo_loss_gb300.dist import reduce_timing  # noqa: E402

METRIC = "GRPO loss fwd+bwd tokens/s at 1 GB300; % of bf16 dense tensor peak"
DEFAULT_WORKLOAD = WL.LLAMA31_8B_20K.name


def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as fh:
            p = json.load(fh)
        return {"bf16_tflops": p.get("bf16_tflops"), "bf16_tflops_sustained":
                p.get("bf16_tflops_sustained"), "hbm_gbs": p.get("hbm_gbs"), "source": "measured"}
    return {"bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "hbm_gbs": 6800.0,
            "source": "fallback"}


def kernel_source_hash() -> str:
    """sha256 over the library's CUDA/C++ sources and its public header: a
    DRAM traffic figure measured on other sources no longer applies."""
    import glob
    import hashlib
    h = hashlib.sha256()
    files = sorted(glob.glob(os.path.join(ROOT, "grpo_loss_gb300", "csrc", "*")))
    files.append(os.path.join(ROOT, "include", "grpo.h"))
    for f in files:
        h.update(os.path.basename(f).encode())
        with open(f, "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()


def measured_traffic(kernel: str, workload: str):
    """DRAM bytes per launch (dram__bytes_read.sum + dram__bytes_write.sum)
    of `kernel` on `workload`, from the ncu summary in profiles/, or None when
    there is none or it was taken on different kernel sources."""
    path = os.path.join(ROOT, "profiles", "traffic_%s_%s.txt" % (kernel, workload))
    if not os.path.exists(path):
        return None
    kv = {}
    with open(path) as fh:
        for line in fh:
            if ":" in line and not line.startswith("#"):
                k, v = line.split(":", 1)
                kv[k.strip()] = v.strip()
    if kv.get("source_sha256") != kernel_source_hash():
        return None
    try:
        return float(kv["dram_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples while the timed region runs."""
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.proc = None
        self.lines = []
        self.dev = device_index
        self.thread = None

    def start(self):
        try:
            uuid = str(torch.cuda.get_device_properties(self.dev).uuid)
            sel = ["-i", "GPU-" + uuid if not uuid.startswith("GPU-") else uuid]
        except Exception:
            sel = []
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "--query-gpu=" + self.FIELDS,
                                          "--format=csv,noheader,nounits", "-lms", "200"] + sel,
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                                         text=True)
        except (OSError, ValueError):
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=2)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                smax.append(float(parts[1]))
            except ValueError:
                continue
            for nm, val in zip(names, parts[4:8]):
                if val.lower().startswith("active"):
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def _flops(w, n_valid, dW=False, ref_given=False):
    # 2 N d V per logit GEMM: policy (+ reference) forward, policy recompute,
    # dH (and dW when requested)
    unit = 2.0 * n_valid * w.d * w.V
    sides = 1.0 if ref_given else 2.0
    return {"step": (sides + 2.0 + (1.0 if dW else 0.0)) * unit, "fwd_gemm_lse": sides * unit,
            "bwd_dz_gemm": unit, "bwd_dh_gemm": unit, "bwd_dw_gemm": unit}


def _dist():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def cpu_oracle_sample(w, inp, rows_target: int = 256, time_budget_s: float = 15.0):
    """Time the float64 oracle (as it stands) on a bounded sample of valid rows
    of the workload: both log-prob passes and the backward of those rows."""
    from oracle import grpo_oracle as O
    m = inp["mask"].numpy() > 0
    valid = np.nonzero(m)[0]
    rng = np.random.default_rng(11)
    A = (inp["adv"].double().numpy() if w.supplied_adv
         else O.advantages(inp["rewards"], w.G, w.eps, w.std_unbiased))
    t0 = time.perf_counter()
    Wf = O.to_f64(inp["W"])
    t_conv = time.perf_counter() - t0
    done, t_rows, n = 0, 0.0, 16
    while done < rows_target and t_rows < time_budget_s:
        rows = np.sort(rng.choice(valid, size=min(n, valid.size), replace=False))
        t1 = time.perf_counter()
        O.token_logprobs(inp["H_pol"], Wf, inp["ids"], rows=rows)
        O.token_logprobs(inp["H_ref"], Wf, inp["ids"], rows=rows)
        O.backward(inp["H_pol"], inp["H_ref"], Wf, inp["ids"], inp["mask"], A, w.B, w.T,
                   w.beta, rows=rows)
        t_rows += time.perf_counter() - t1
        done += rows.size
        n = min(2 * n, 128)
    try:
        from threadpoolctl import threadpool_info
        cores = max(int(i.get("num_threads", 1)) for i in threadpool_info()) if threadpool_info() else os.cpu_count()
    except Exception:
        cores = os.cpu_count()
    return {"value": done / t_rows, "unit": "tokens/s", "cores": cores, "kind": "oracle",
            "sample": "%d valid rows of %s (policy+reference log-probs and backward per row, "
                      "float64, full vocab), %.1f s; one-off W->float64 conversion %.1f s "
                      "excluded" % (done, w.name, t_rows, t_conv)}


class _RowView:
    """Rows of a matrix computed for a sample only (the oracle's per-row
    functions index just the rows they are asked for)."""

    def __init__(self, rows, data):
        self.pos = {int(r): i for i, r in enumerate(rows)}
        self.data = data

    def __getitem__(self, idx):
        return self.data[[self.pos[int(i)] for i in np.asarray(idx).reshape(-1)]]


def run_reference(args, w):
    ws, rank, _ = _dist()
    if rank != 0:
        return
    inp = WL.make_inputs(w)
    from oracle import grpo_oracle as O
    m = inp["mask"].numpy() > 0
    valid = np.nonzero(m)[0]
    A = (inp["adv"].double().numpy() if w.supplied_adv
         else O.advantages(inp["rewards"], w.G, w.eps, w.std_unbiased))
    t0 = time.perf_counter()
    if args.fp8:
        # the e4m3 problem: W quantized and dequantized once (excluded from the
        # timing like the float64 conversion); each step's rows inside the step
        Wf = np.empty((w.V, w.d))
        for r0 in range(0, w.V, 8192):
            Wf[r0:r0 + 8192] = O.dequantize_rows(*O.quantize_e4m3_rows(inp["W"][r0:r0 + 8192]))
    else:
        Wf = O.to_f64(inp["W"])
    t_setup = time.perf_counter() - t0
    rng = np.random.default_rng(5)
    rows_per_step = 32 if w.V * w.d > 1e8 else min(valid.size, 512)

    def step():
        rows = np.sort(rng.choice(valid, size=min(rows_per_step, valid.size), replace=False))
        Hp, Hr = inp["H_pol"], inp["H_ref"]
        if args.fp8:
            sel = torch.from_numpy(rows)
            Hp = _RowView(rows, O.dequantize_rows(*O.quantize_e4m3_rows(Hp[sel])))
            Hr = _RowView(rows, O.dequantize_rows(*O.quantize_e4m3_rows(Hr[sel])))
        O.token_logprobs(Hp, Wf, inp["ids"], rows=rows)
        O.token_logprobs(Hr, Wf, inp["ids"], rows=rows)
        O.backward(Hp, Hr, Wf, inp["ids"], inp["mask"], A, w.B, w.T, w.beta, rows=rows)
        return rows.size

    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    rows = sum(step() for _ in range(args.steps))
    dt = time.perf_counter() - t0
    value = rows / dt
    cores = os.cpu_count()
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
            "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1e3 * dt / args.steps, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": w.name, "tokens_per_step": rows_per_step,
                       "sample": "rows drawn from the valid tokens",
                       "operands": "e4m3 row-quantized by the oracle" if args.fp8 else w.dtype},
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                             "sample": "%d valid rows per step of %s, float64 full-vocab oracle"
                                       "%s; one-off W setup %.1f s excluded"
                                       % (rows_per_step, w.name,
                                          " on e4m3 operands (rows quantized in the step)"
                                          if args.fp8 else "", t_setup)},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def _gpu_numa_cpus(device_index: int):
    """(NUMA node, CPU ids) of the host node the GPU is attached to, from
    its PCI device in sysfs; (None, None) when that cannot be read."""
    try:
        uuid = str(torch.cuda.get_device_properties(device_index).uuid)
        sel = uuid if uuid.startswith("GPU-") else "GPU-" + uuid
        out = subprocess.run(["nvidia-smi", "--query-gpu=pci.bus_id", "--format=csv,noheader",
                              "-i", sel], capture_output=True, text=True, timeout=20)
        bus = out.stdout.strip().splitlines()[0].strip().lower()
        dom, rest = bus.split(":", 1)
        bus = "%04x:%s" % (int(dom, 16), rest)
        with open("/sys/bus/pci/devices/%s/numa_node" % bus) as fh:
            node = int(fh.read().strip())
        if node < 0:
            return None, None
        with open("/sys/devices/system/node/node%d/cpulist" % node) as fh:
            cpus = set()
            for part in fh.read().strip().split(","):
                a, _, b = part.partition("-")
                cpus.update(range(int(a), int(b or a) + 1))
        cpus &= os.sched_getaffinity(0)
        return (node, cpus) if cpus else (None, None)
    except Exception:
        return None, None


def replica_workload(w, rank: int):
    """Rank r's independent batch: the same recipe with its own seed."""
    return w if rank == 0 else WL.Workload(**{**w.__dict__, "seed": w.seed + 100 * rank})


def run_ours(args, w):
    import torch.distributed as dist

    import grpo_loss_gb300 as G

    ws, rank, local = _dist()
    if ws > 1:
        dist.init_process_group("nccl")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    w_r = replica_workload(w, rank)
    inp = WL.make_inputs(w_r)
    n_valid = int(inp["mask"].sum())
    dt = torch.float32 if w.dtype == "f32" else torch.bfloat16
    if args.fp8:
        # e4m3 operands: the step quantizes H_pol, H_ref and W row-wise first
        dt = torch.float8_e4m3fn

    eng = G.GRPOLoss(w.B, w.T, w.d, w.V, w.G, beta=w.beta, eps=w.eps,
                     std_unbiased=w.std_unbiased, dtype=dt, device=dev, compute_dW=args.dW,
                     token_level=args.token_level, softcap=args.softcap,
                     temperature=args.temperature, ref_logp_given=args.ref_given,
                     cluster_mode=args.cluster_mode)
    d_in = {k: (v.to(dev) if v is not None else None) for k, v in inp.items()}
    rewards = d_in["rewards"]
    adv_in = d_in["adv"]
    dH = (torch.empty(d_in["H_pol"].shape, dtype=torch.bfloat16, device=dev) if args.fp8
          else torch.empty_like(d_in["H_pol"]))
    stream = torch.cuda.current_stream()

    if args.ref_given:
        # reference log-probs a trainer kept from generation time; any float32
        # values serve for timing (the kernels' work does not depend on them)
        d_in["logp_ref"] = torch.full((w.N,), -12.0, dtype=torch.float32, device=dev)

    def step(d):
        adv = adv_in if w.supplied_adv else eng.advantages(d["rewards"])
        if args.ref_given:
            eng.forward(d["H_pol"], None, d["W"], d["ids"], d["mask"], adv,
                        logp_ref=d["logp_ref"])
        else:
            eng.forward(d["H_pol"], d["H_ref"], d["W"], d["ids"], d["mask"], adv)
        eng.backward(d["H_pol"], d["W"], d["ids"], d["mask"], adv, 1.0, dH=dH)

    # ---------------------------------------------------------- device-resident
    for _ in range(args.warmup):
        step(d_in)
    torch.cuda.synchronize()
    timed_step = step
    graph_launches_per_step = 0
    if args.graph:
        # kernels per step, counted on one eager step (a replay records none)
        G.profile_enable(True)
        G.profile_collect()
        step(d_in)
        torch.cuda.synchronize()
        graph_launches_per_step = int(sum(v[1] for v in G.profile_collect().values()))
        G.profile_enable(False)
        # the whole step captured once and replayed (the library's calls are
        # stream-ordered; the first call above set the kernel attributes)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            step(d_in)
        timed_step = lambda _d: graph.replay()  # noqa: E731
        for _ in range(args.warmup):
            timed_step(d_in)
        torch.cuda.synchronize()
    eng.check()
    if ws > 1:
        dist.barrier()
    G.profile_enable(True)
    G.profile_collect()
    clocks = ClockSampler(local) if rank == 0 else None
    if clocks:
        clocks.start()
        time.sleep(0.3)
    torch.cuda.synchronize()
    if ws > 1:
        dist.barrier()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev0.record(stream)
    for _ in range(args.steps):
        timed_step(d_in)
    ev1.record(stream)
    torch.cuda.synchronize()
    if ws > 1:
        dist.barrier()
    clk = clocks.stop() if clocks else None
    G.profile_enable(False)
    prof = G.profile_collect()
    eng.check()
    ms_max, total_valid = reduce_timing(ev0.elapsed_time(ev1), n_valid, device=dev)
    ms_step = ms_max / args.steps
    value = total_valid / (ms_step / 1e3)

    # --------------------------------------------------------------- end to end
    # Every step copies its inputs from pinned host memory and reads its loss
    # back, as a training loop would. Two device copies of the inputs let the
    # copies of step i + 1 run on a copy stream while step i computes.
    e2e_src = dict(inp, H_ref=None, logp_ref=d_in["logp_ref"].cpu()) if args.ref_given else inp
    # pin the host buffers on the NUMA node the GPU is attached to (the
    # pages come from the allocating thread's node), then restore affinity
    node, cpus = _gpu_numa_cpus(local)
    saved_aff = os.sched_getaffinity(0)
    if cpus:
        os.sched_setaffinity(0, cpus)
    try:
        host = {k: (v.pin_memory() if v is not None else None) for k, v in e2e_src.items()}
    finally:
        os.sched_setaffinity(0, saved_aff)
    bufs = [{k: (torch.empty_like(v, device=dev) if v is not None else None)
             for k, v in e2e_src.items()} for _ in range(2)]
    n_res = max(args.steps, args.warmup, 1)
    res_host = torch.empty(n_res, 2, dtype=torch.float32).pin_memory()
    h2d = sum(v.numel() * v.element_size() for k, v in host.items() if v is not None)
    d2h = 2 * res_host.element_size()
    copy_stream = torch.cuda.Stream(device=dev)
    copied = [torch.cuda.Event() for _ in range(2)]
    consumed = [torch.cuda.Event() for _ in range(2)]

    def issue_copy(i):
        b = i % 2
        copy_stream.wait_event(consumed[b])        # step i - 2 no longer reads buffer b
        with torch.cuda.stream(copy_stream):
            for k, v in host.items():
                if v is not None:
                    bufs[b][k].copy_(v, non_blocking=True)
        copied[b].record(copy_stream)

    def compute(i):
        b = i % 2
        stream.wait_event(copied[b])
        step(bufs[b])
        consumed[b].record(stream)
        res_host[i % n_res, 0:1].copy_(eng.loss, non_blocking=True)
        res_host[i % n_res, 1:2].copy_(eng.kl_mean, non_blocking=True)

    def e2e_run(k_steps):
        copy_stream.wait_stream(stream)
        issue_copy(0)
        for i in range(k_steps):
            if i + 1 < k_steps:
                issue_copy(i + 1)
            compute(i)

    e2e_run(max(1, args.warmup))
    torch.cuda.synchronize()
    if ws > 1:
        dist.barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    e2e_run(args.steps)
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms, _ = reduce_timing(e0.elapsed_time(e1), n_valid, device=dev)
    e2e_value = total_valid / (e2e_ms / args.steps / 1e3)
    eng.check()

    if rank == 0:
        peaks = _peaks()
        fl = _flops(w, n_valid, args.dW, args.ref_given)
        gemms = {k: prof[k] for k in ("fwd_gemm_lse", "bwd_dz_gemm", "bwd_dh_gemm",
                                      "bwd_dw_gemm") if prof[k][1]}
        peak = peaks["bf16_tflops_sustained"]
        # e4m3 contractions: the measured bf16 peak times the nominal e4m3 / bf16
        # dense ratio (4.5 / 2.25 PFLOP/s)
        fp8_kernels = ("fwd_gemm_lse", "bwd_dz_gemm") if args.fp8 else ()

        def kpeak(k):
            return peak * 2.0 if k in fp8_kernels else peak

        roofline = None
        if gemms:  # (a replayed CUDA graph records no per-kernel events)
            dom = max(gemms, key=lambda k: gemms[k][0])
            dom_ms, dom_launches = gemms[dom]
            per_launch_flops = fl[dom] * args.steps / dom_launches
            achieved = per_launch_flops / (dom_ms / dom_launches / 1e3) / 1e12
            roofline = {"bound": "tensor", "kernel": dom, "achieved": achieved,
                        "peak": kpeak(dom), "unit": "TFLOP/s", "frac": achieved / kpeak(dom),
                        "traffic": measured_traffic(dom, w.name + ("-e4m3" if args.fp8 else "")),
                        "peak_kind": ("e4m3 = 2 x bf16 sustained (%s)" if dom in fp8_kernels
                                      else "bf16 sustained (%s)") % peaks["source"]}
        launches = int(sum(v[1] for v in prof.values())) or graph_launches_per_step * args.steps
        kernels = {k: {"ms_per_step": v[0] / args.steps, "launches_per_step": v[1] / args.steps}
                   for k, v in prof.items() if v[1]}
        step_tflops = fl["step"] / (ms_step / 1e3) / 1e12
        # time the step's GEMM flops would take at their own peaks
        ideal_s = sum(fl[k] / (kpeak(k) * 1e12) for k in
                      ("fwd_gemm_lse", "bwd_dz_gemm", "bwd_dh_gemm") +
                      (("bwd_dw_gemm",) if args.dW else ()))
        cpu = cpu_oracle_sample(w, inp) if ws == 1 and not args.no_cpu_baseline else None
        line = {
            "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": ws,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": ("e4m3" if args.fp8 else "bf16" if w.dtype == "bf16" else "f32->bf16"),
            "data": "synthetic",
            "config": {"workload": w.name, "prompts": w.prompts, "generations": w.G,
                       "completion_len": w.T, "tokens": w.N, "valid_tokens": n_valid,
                       "hidden": w.d, "vocab": w.V, "beta": w.beta, "dW": bool(args.dW),
                       "variant": {"token_level": bool(args.token_level), "softcap": args.softcap,
                                   "temperature": args.temperature,
                                   "ref_logp_given": bool(args.ref_given),
                                   "cluster_mode": args.cluster_mode,
                                   "cuda_graph": bool(args.graph),
                                   "operands": ("e4m3 row-scaled H W^T GEMMs (quantized from "
                                                "bf16 inside the step); bf16 dH/dW GEMMs"
                                                if args.fp8 else w.dtype)},
                       "flops_per_step": fl["step"],
                       "parallelism": "replicas" if ws > 1 else "single",
                       "l2": "inputs larger than L2 (H_pol+H_ref+W = %.2f GB)"
                             % ((inp["H_pol"].numel() * 2 + inp["W"].numel()) *
                                inp["W"].element_size() / 1e9)},
            "tflops_per_step": step_tflops,
            # the same step without the backward's recompute GEMM in the count
            # (forward GEMMs, dH and dW only): what an implementation keeping
            # the logits would have to compute
            "model_tflops_per_step": (fl["step"] - fl["bwd_dz_gemm"]) / (ms_step / 1e3) / 1e12,
            # every row, padding included (value counts valid tokens only)
            "all_rows_per_s": ws * w.N / (ms_step / 1e3),
            "frac_of_peak": ideal_s / (ms_step / 1e3),
            "peak": {"bf16_tflops_sustained": peak, "source": peaks["source"]},
            "roofline": roofline,
            "kernels": kernels,
            "memory": {
                "fwd_workspace_bytes": eng.ws_fwd.numel(),
                "bwd_workspace_bytes": eng.ws_bwd.numel(),
                # what an unfused loss would hold: fp32 logits of policy and reference
                "unfused_fp32_logits_bytes": 2 * w.N * w.V * 4,
            },
            "gpu_launches": launches,
            "clocks": clk,
            "e2e": {"value": e2e_value, "unit": "tokens/s", "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h,
                    "mode": "pinned host inputs copied every step on a copy stream, "
                            "overlapping the previous step's compute; loss read back "
                            "every step",
                    "host_numa_node": node},
            "cpu_baseline": cpu,
        }
        print(json.dumps(line), flush=True)
    if ws > 1:
        dist.barrier()
        dist.destroy_process_group()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD,
                    choices=sorted(list(WL.FULL) + list(WL.SMALL)))
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--dW", action="store_true", help="also compute the lm_head gradient")
    ap.add_argument("--token-level", action="store_true", help="token-level loss aggregation")
    ap.add_argument("--softcap", type=float, default=0.0, help="logit softcap (0 = off)")
    ap.add_argument("--temperature", type=float, default=0.0, help="logit temperature (0 = off)")
    ap.add_argument("--graph", action="store_true",
                    help="time the step replayed from a CUDA graph")
    ap.add_argument("--cluster-mode", type=int, default=0, choices=[0, 1],
                    help="GEMM tiling: 0 one CTA per tile, 1 CTA pairs (cta_group::2)")
    ap.add_argument("--fp8", action="store_true",
                    help="e4m3 operands for the H W^T GEMMs (row-wise quantized in the step)")
    ap.add_argument("--ref-given", action="store_true",
                    help="reference log-probs supplied; skip the reference GEMM half")
    ap.add_argument("--seq-len", type=int, default=0,
                    help="shorter sequences of the same workload (a smaller case of the same "
                         "shapes for profiling; the workload is renamed <name>-T<len>)")
    args = ap.parse_args()
    w = WL.FULL.get(args.workload) or WL.SMALL[args.workload]
    if args.seq_len > 0:
        # same d, V and value recipe; padding bounds clipped to the new length
        w = w.scaled("%s-T%d" % (w.name, args.seq_len), T=args.seq_len,
                     pad_lo=min(w.pad_lo, args.seq_len), pad_hi=min(w.pad_hi, args.seq_len))
    if args.impl == "reference":
        run_reference(args, w)
    else:
        run_ours(args, w)


if __name__ == "__main__":
    main()
