"""Benchmark of the Muon optimizer step on one B300 per rank.

Headline workload: the GPT-2 124M hidden-matrix set, 12 layers x (4x 768x768
attention q/k/v/o, 768x3072, 3072x768 MLP), bf16 gradients N(0,1e-3) plus a
rank-4 spike x50, fp32 momentum with beta 0.95 and Nesterov, 5 cubic
Newton-Schulz iterations, bf16 parameters updated with lr 0.02 * max(1,r/c)^0.5.
One step = one muon_step call over all 72 matrices.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--workload NAME]

Prints one JSON line (rank 0). Under torchrun every rank runs its own replica
of the workload on its own GPU (weak scaling, no collective on the data path);
value = all ranks' steps / the slowest rank's time.
"""
from __future__ import annotations

import argparse
import hashlib
import re
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads as wl  # noqa: E402

METRIC = "Muon steps/sec at GPT-2 124M hidden-matrix shapes; % BF16 TC peak, HBM GB/s"
UNIT = "steps/s"
FALLBACK_PEAKS = {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0}
# Dense bf16 tensor rate per SM and clock: 2.25 PFLOP/s nominal = 148 SMs x 8192 flops x 1.86 GHz.
DENSE_FLOPS_PER_SM_CYCLE = 8192
SMS = 148

# DRAM bytes (read + write) per launch of a kernel on a workload, from one ncu capture, keyed by
# the hash of the kernel sources' code (comments excluded) they were taken with, then by workload
# and kernel kind. A stale hash, or a workload or kernel without a capture, gives null.
NCU_TRAFFIC = {
    "c0a396102587b97f": {
        # ncu --set full on the GPT-2 124M step: the persistent launch running all 5 iterations
        # (profiles/persistent_ns_gpt2_124m.md), 2.069 GB read + 1.242 GB written.
        "gpt2_124m_hidden": {"newton_schulz": 3.310e9},
        # ncu --set full on one per-phase combine and one Gram of the 4096 x 16384 matrix
        # (profiles/combine_gemm_illcond_4096x16384.md): 218.2 + 115.7 MB and 233.6 + 21.5 MB.
        "illcond_4096x16384": {"combine_ax_bx": 3.338e8, "gram_xxt": 2.551e8},
    },
}


def ncu_traffic(workload: str, kernel: str):
    """The captured DRAM bytes per launch of `kernel` on `workload` at the current sources, or None."""
    return NCU_TRAFFIC.get(source_hash(), {}).get(workload, {}).get(kernel)

KERNEL_SOURCES = ["muon_newton_schulz_09_b300/csrc/ns_gemm.cuh", "muon_newton_schulz_09_b300/csrc/elementwise.cuh",
                  "muon_newton_schulz_09_b300/csrc/ptx.cuh", "muon_newton_schulz_09_b300/csrc/muon_api.cu",
                  "muon_newton_schulz_09_b300/csrc/ns_fused.cuh"]


def code_text(src: str) -> str:
    """C++ source without its comments and blank lines: what a change to the kernels changes."""
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    src = re.sub(r"//[^\n]*", "", src)
    return "\n".join(line.rstrip() for line in src.splitlines() if line.strip())


def source_hash() -> str:
    """Hash of the kernel sources' code (comments excluded), keying the ncu traffic table."""
    h = hashlib.sha256()
    for f in KERNEL_SOURCES:
        with open(os.path.join(ROOT, f)) as fh:
            h.update(code_text(fh.read()).encode())
    return h.hexdigest()[:16]


# ----------------------------------------------------------------------------- distributed host logic

def dist_env() -> tuple:
    """(rank, local_rank, world_size) from the torchrun environment (defaults for a plain launch)."""
    return (int(os.environ.get("RANK", 0)), int(os.environ.get("LOCAL_RANK", 0)),
            int(os.environ.get("WORLD_SIZE", 1)))


def reduce_max(x: float) -> float:
    """Max of x over ranks (x itself without an initialised process group)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return x
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier():
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized():
        dist.barrier()


def whole_job_rate(steps_per_rank: int, world: int, max_elapsed_s: float) -> float:
    """Steps per second over the whole job: every rank's steps over the slowest rank's time."""
    return steps_per_rank * world / max_elapsed_s


# ----------------------------------------------------------------------------- work accounting

def workload_of(name: str) -> wl.Workload:
    return wl.WORKLOADS[name]


def oriented(shape) -> tuple:
    r, c = shape
    return min(r, c), max(r, c)


def kernel_work(w: wl.Workload, carry: bool = False) -> dict:
    """Algorithmic work of each kernel kind per STEP: ("flops" | "bytes", amount).

    Gram: n(n+1)m flops per iteration (upper triangle); combine: 2 n^2 m per
    iteration; A A pass (c != 0): n^2 (n+1) per iteration. Elementwise kernels:
    bytes each element must move once (momentum: g + buf read/write + u
    write; scale: u or input read + X0 write; update: O read + W read/write;
    copy: O read + out write). A kind may take several launches per step
    (one per iteration, or one per 128 matrices); throughput is the step's
    work over the kind's summed launch time. With the precise carry X0 and
    O move a bf16 low part as well (2 more bytes per element).
    """
    gb = 4 if w.dtype == "f32" else 2
    pb = 4 if w.param_dtype == "f32" else 2
    elems = w.elements()
    lo = 2 if carry else 0
    k = w.steps
    gram = sum(n * (n + 1) * m for n, m in map(oriented, w.shapes)) * k
    comb = sum(2 * n * n * m for n, m in map(oriented, w.shapes)) * k
    aa = sum(n * n * (n + 1) for n, m in map(oriented, w.shapes)) * k
    work = {"gram_xxt": ("flops", float(gram)), "combine_ax_bx": ("flops", float(comb)),
            "gram_aa": ("flops", float(aa)),
            "newton_schulz": ("flops", float(gram + comb + (aa if w.coeffs[2] != 0 else 0)))}
    if w.kind == "step":
        work.update({"momentum_norm": ("bytes", float(elems * (gb + 4 + 4 + 2 + lo))),
                     "scale_orient": ("bytes", float(elems * (2 + 2))),
                     "update": ("bytes", float(elems * (2 + lo + 2 * pb)))})
    else:
        work.update({"norm": ("bytes", float(elems * gb)),
                     "scale_orient": ("bytes", float(elems * (gb + 2 + lo))),
                     "copy_out": ("bytes", float(elems * (2 + lo + 4)))})
    return work


def step_flops(w: wl.Workload) -> float:
    a, b, c = w.coeffs
    per = sum(n * (n + 1) * m + 2 * n * n * m + (n * n * (n + 1) if c != 0 else 0) for n, m in map(oriented, w.shapes))
    return float(per * w.steps)


def resident_bytes(w: wl.Workload) -> int:
    """Bytes of the caller's tensors one step reads or writes: grads, momentum and params (step),
    or inputs and bf16 outputs (orthogonalize)."""
    gb = 4 if w.dtype == "f32" else 2
    pb = 4 if w.param_dtype == "f32" else 2
    per = gb + 4 + pb if w.kind == "step" else gb + 2
    return w.elements() * per


def config_of(w: wl.Workload, world: int, carry: bool) -> dict:
    """The workload's description, identical for both arms."""
    return {"workload": w.name, "description": w.notes, "matrices": w.count,
            "ns_steps": w.steps, "coeffs": list(w.coeffs), "kind": w.kind,
            "parallelism": f"replicas x{world} (one full step per GPU, no collective)",
            "l2": f"inputs larger than L2: {resident_bytes(w) / 1e6:.0f} MB resident per step",
            "precise_carry": carry,
            "alg_flops_per_step": step_flops(w)}


# ----------------------------------------------------------------------------- peaks and clocks

# A region shorter than this is timed against the burst tensor peak (a kernel timed alone); a
# longer one against the sustained peak measured over seconds under the power limit.
SUSTAINED_REGION_S = 1.0


def uses_sustained_peak(region_s: float) -> bool:
    return region_s >= SUSTAINED_REGION_S


def load_peaks() -> tuple:
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 200 ms during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.proc = None
        self.path = None
        self.device_index = device_index

    def __enter__(self):
        import tempfile
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "200",
                 "-i", str(self.device_index)], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self) -> dict:
        rows = []
        if self.path and os.path.exists(self.path):
            with open(self.path) as f:
                for line in f:
                    parts = [p.strip() for p in line.split(",")]
                    if len(parts) >= 9:
                        rows.append(parts)
            os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        pw = [float(r[3]) for r in rows if r[3].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower().startswith("active")})
        load = [s for s in sm if mx and s > 0.3 * max(mx)] or sm
        return {"sm_mhz": statistics.median(load) if load else None, "sm_max_mhz": max(mx) if mx else None,
                "power_w_max": max(pw) if pw else None, "reasons": reasons, "samples": len(rows)}


# ----------------------------------------------------------------------------- oracle timing (host cores)

def blas_threads() -> int:
    try:
        from threadpoolctl import threadpool_info
        n = [i.get("num_threads", 0) for i in threadpool_info() if i.get("user_api") == "blas"]
        if n:
            return int(max(n))
    except Exception:
        pass
    return os.cpu_count() or 1


def oracle_matrix_call(w: wl.Workload, j: int, inputs: dict):
    import oracle
    if w.kind == "step":
        g, m, p = inputs[j]
        return oracle.muon_step(p, g, m, w.lr, w.beta, w.nesterov, w.steps, w.coeffs, w.eps)
    (g,) = inputs[j]
    return oracle.orthogonalize(g, w.steps, w.coeffs, w.eps)


def oracle_inputs(w: wl.Workload, j: int) -> tuple:
    if w.kind == "step":
        return wl.gradient(w, j), wl.momentum_buffer(w, j), wl.parameter(w, j)
    return (wl.gradient(w, j),)


def matrix_fraction(w: wl.Workload) -> list:
    """Share of one full step's flops carried by each matrix."""
    f = [n * (n + 1) * m + 2 * n * n * m for n, m in map(oriented, w.shapes)]
    tot = float(sum(f))
    return [x / tot for x in f]


def distinct_matrices(w: wl.Workload) -> list:
    """One matrix index per distinct shape (a layer's worth for the GPT-2 sets)."""
    seen, out = set(), []
    for j, s in enumerate(w.shapes):
        if s not in seen:
            seen.add(s)
            out.append(j)
    return out


def time_oracle(w: wl.Workload, budget_s: float, min_calls: int = 1) -> dict:
    """Runs the oracle on matrices of the workload, cycling over its distinct shapes, for about budget_s.

    Returns the full-workload steps/s extrapolated by each matrix's flop share.
    """
    frac = matrix_fraction(w)
    pick = distinct_matrices(w)
    inputs = {j: oracle_inputs(w, j) for j in pick}
    done_frac, elapsed, calls = 0.0, 0.0, 0
    while calls < min_calls or elapsed < budget_s:
        j = pick[calls % len(pick)]
        t0 = time.perf_counter()
        oracle_matrix_call(w, j, inputs)
        elapsed += time.perf_counter() - t0
        done_frac += frac[j]
        calls += 1
        if calls >= 10 * len(pick) and elapsed >= 0.5 * budget_s:
            break
    return {"value": done_frac / elapsed, "calls": calls, "elapsed_s": elapsed, "fraction": done_frac,
            "shapes": [list(w.shapes[j]) for j in pick]}


# ----------------------------------------------------------------------------- device workload

class DeviceWorkload:
    """Flat device buffers holding every matrix of the workload (views per matrix)."""

    def __init__(self, w: wl.Workload, device: int):
        import torch
        self.w = w
        td = {"bf16": torch.bfloat16, "f32": torch.float32}
        n = w.elements()
        offs = np.cumsum([0] + [r * c for r, c in w.shapes])
        self.grads_flat = torch.empty(n, dtype=td[w.dtype], device=device)
        self.grads = [self.grads_flat[offs[j]:offs[j + 1]].view(*w.shapes[j]) for j in range(w.count)]
        for j in range(w.count):
            self.grads[j].copy_(torch.from_numpy(wl.gradient(w, j)))
        if w.kind == "step":
            self.mom_flat = torch.empty(n, dtype=torch.float32, device=device)
            self.params_flat = torch.empty(n, dtype=td[w.param_dtype], device=device)
            self.momentum = [self.mom_flat[offs[j]:offs[j + 1]].view(*w.shapes[j]) for j in range(w.count)]
            self.params = [self.params_flat[offs[j]:offs[j + 1]].view(*w.shapes[j]) for j in range(w.count)]
            for j in range(w.count):
                self.momentum[j].copy_(torch.from_numpy(wl.momentum_buffer(w, j)))
                self.params[j].copy_(torch.from_numpy(wl.parameter(w, j)))
        else:
            self.out_flat = torch.empty(n, dtype=torch.bfloat16, device=device)
            self.outs = [self.out_flat[offs[j]:offs[j + 1]].view(*w.shapes[j]) for j in range(w.count)]

    def resident_bytes(self) -> int:
        t = [self.grads_flat] + ([self.mom_flat, self.params_flat] if self.w.kind == "step" else [self.out_flat])
        return sum(x.numel() * x.element_size() for x in t)

    def run(self, muon, stream=None):
        w = self.w
        if w.kind == "step":
            muon.step(self.params, self.grads, self.momentum, lr=w.lr, beta=w.beta, nesterov=w.nesterov,
                      stream=stream)
        else:
            muon.orthogonalize(self.grads, self.outs, steps=w.steps, coeffs=w.coeffs, stream=stream)

    def prepared(self, muon, stream=None):
        """The same call with its descriptors built once (what a training loop would hold on to)."""
        w = self.w
        if w.kind == "step":
            return muon.prepare_step(self.params, self.grads, self.momentum, lr=w.lr, beta=w.beta,
                                     nesterov=w.nesterov, stream=stream)
        return muon.prepare_orthogonalize(self.grads, self.outs, steps=w.steps, coeffs=w.coeffs, stream=stream)

    def result_flat(self):
        return self.params_flat if self.w.kind == "step" else self.out_flat


# ----------------------------------------------------------------------------- end to end

def run_e2e(muon, dw, steps: int, stream) -> dict:
    """Steps with host->device gradients and device->host results inside the timed region."""
    import torch
    w = dw.w
    grads = [dw.grads_flat, torch.empty_like(dw.grads_flat)]
    offs = np.cumsum([0] + [r * c for r, c in w.shapes])
    views = [[g[offs[j]:offs[j + 1]].view(*w.shapes[j]) for j in range(w.count)] for g in grads]
    if w.kind == "step":
        calls = [muon.prepare_step(dw.params, v, dw.momentum, lr=w.lr, beta=w.beta, nesterov=w.nesterov,
                                   stream=stream) for v in views]
    else:
        calls = [muon.prepare_orthogonalize(v, dw.outs, steps=w.steps, coeffs=w.coeffs, stream=stream)
                 for v in views]
    result = dw.result_flat()
    h2d_src = dw.grads_flat.cpu().pin_memory()
    d2h_dst = torch.empty(result.shape, dtype=result.dtype).pin_memory()
    stage = torch.empty_like(result)
    s_h2d, s_d2h = torch.cuda.Stream(), torch.cuda.Stream()
    ev = lambda: torch.cuda.Event()
    loaded, used = [ev(), ev()], [ev(), ev()]
    staged, read_back = ev(), ev()

    def run(n):
        with torch.cuda.stream(s_h2d):
            grads[0].copy_(h2d_src, non_blocking=True)
            loaded[0].record(s_h2d)
        read_back.record(s_d2h)
        for k in range(n):
            b = k % 2
            if k + 1 < n:  # next step's gradients, into the buffer the previous step has finished with
                with torch.cuda.stream(s_h2d):
                    if k >= 1:
                        s_h2d.wait_event(used[1 - b])
                    grads[1 - b].copy_(h2d_src, non_blocking=True)
                    loaded[1 - b].record(s_h2d)
            stream.wait_event(loaded[b])
            calls[b]()
            used[b].record(stream)
            stream.wait_event(read_back)  # the stage buffer is free once the last read-back is done
            stage.copy_(result, non_blocking=True)
            staged.record(stream)
            with torch.cuda.stream(s_d2h):
                s_d2h.wait_event(staged)
                d2h_dst.copy_(stage, non_blocking=True)
                read_back.record(s_d2h)
        stream.wait_event(read_back)

    run(2)
    torch.cuda.synchronize()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    run(steps)
    t1.record(stream)
    torch.cuda.synchronize()
    return {"unit": UNIT, "h2d_bytes_per_step": h2d_src.numel() * h2d_src.element_size(),
            "d2h_bytes_per_step": d2h_dst.numel() * d2h_dst.element_size(), "steps": steps,
            "elapsed_s": t0.elapsed_time(t1) / 1e3}


# ----------------------------------------------------------------------------- arms

def run_ours(args) -> dict:
    import torch
    import torch.distributed as dist
    from muon_newton_schulz_09_b300 import Muon

    rank, local_rank, world = dist_env()
    torch.cuda.set_device(local_rank)
    if world > 1 and not dist.is_initialized():
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    w = workload_of(args.workload)
    dw = DeviceWorkload(w, local_rank)
    a, b, c = w.coeffs
    # The library default carries X as bf16 hi + lo exactly when c != 0; --precise-carry forces it.
    carry = bool(getattr(args, "precise_carry", False)) or c != 0
    muon = Muon(local_rank, steps=w.steps, a=a, b=b, c=c, eps=w.eps, scale_lr_by_shape=True,
                precise_carry=True if getattr(args, "precise_carry", False) else None)
    stream = torch.cuda.current_stream()
    step = dw.prepared(muon, stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    if muon.get_error() != 0:
        raise RuntimeError("device error flag raised during warm-up")

    # ---- timed region: inputs resident in HBM. Nothing but the steps is queued in it.
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    torch.cuda.synchronize()
    with ClockSampler(local_rank) as clk:
        start.record(stream)
        # Host cost per step, read over the first steps, before the launch queue fills and the
        # host starts waiting for the GPU.
        h_n = min(args.steps, 20)
        h0 = time.perf_counter()
        for i in range(args.steps):
            step()
            if i + 1 == h_n:
                host_s = (time.perf_counter() - h0) / h_n
        end.record(stream)
        torch.cuda.synchronize()
    barrier()
    elapsed_s = start.elapsed_time(end) / 1e3
    if muon.get_error() != 0:
        raise RuntimeError("device error flag raised during the timed region")
    max_s = reduce_max(elapsed_s)
    value = whole_job_rate(args.steps, world, max_s)

    # ---- the same steps again with every kernel bracketed by CUDA events on the launching
    # stream (the library's profiling hooks), for per-kernel durations. The events sit between
    # kernels, so this region runs slightly slower than the one above; its own step time is
    # reported as ms_per_step_profiled.
    muon.profile_read()
    muon.profile(True)
    p0, p1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    torch.cuda.synchronize()
    p0.record(stream)
    for _ in range(args.steps):
        step()
    p1.record(stream)
    torch.cuda.synchronize()
    barrier()
    muon.profile(False)
    prof = muon.profile_read()
    # The SM clock the GEMM kernels themselves saw: clock64 cycles over %globaltimer ns, summed over
    # their CTAs. nvidia-smi samples every 200 ms and misses the power-cap dips inside a step.
    device_mhz = muon.profile_clock()
    prof_s = p0.elapsed_time(p1) / 1e3
    if muon.get_error() != 0:
        raise RuntimeError("device error flag raised during the profiled region")

    # ---- end to end through the public API: every step uploads its gradients from pinned host
    # memory and reads the updated parameters (or the orthogonalised output) back to pinned host
    # memory. The copies are pipelined as a training loop would run them: the next step's
    # gradients upload on a copy stream into a second device buffer while this step computes,
    # and the result is staged on the device and read back on another copy stream.
    e2e = run_e2e(muon, dw, max(3, min(args.steps, 50)), stream)
    barrier()
    e2e_s = reduce_max(e2e.pop("elapsed_s"))
    e2e["value"] = whole_job_rate(e2e["steps"], world, e2e_s)

    # ---- roofline of the dominant kernel, from the per-kernel events of the timed region
    peaks, peak_src = load_peaks()
    clk = clk.summary()
    clk["sm_mhz_device"] = round(device_mhz, 1)
    sustained = uses_sustained_peak(prof_s)
    tc_peak = peaks["bf16_tflops_sustained" if sustained else "bf16_tflops"]
    work = kernel_work(w, carry)
    kernels = {}
    for name, (ms, n) in prof.items():
        if n == 0:
            continue
        kind, per_step = work[name]
        avg_ms = ms / n
        amount = per_step * args.steps / n  # work per launch
        if kind == "flops":
            ach = amount / (avg_ms * 1e-3) / 1e12
            kernels[name] = {"launches": n, "avg_us": avg_ms * 1e3, "share": 0.0, "bound": "tensor",
                             "achieved": ach, "unit": "TFLOP/s", "frac": ach / tc_peak,
                             "frac_burst": ach / peaks["bf16_tflops"],
                             "frac_sustained": ach / peaks["bf16_tflops_sustained"]}
            if device_mhz > 0:  # of the dense rate at the clock the kernels ran at
                kernels[name]["frac_per_cycle"] = ach / (DENSE_FLOPS_PER_SM_CYCLE * SMS * device_mhz * 1e6 / 1e12)
        else:
            ach = amount / (avg_ms * 1e-3) / 1e9
            kernels[name] = {"launches": n, "avg_us": avg_ms * 1e3, "share": 0.0, "bound": "hbm",
                             "achieved": ach, "unit": "GB/s", "frac": ach / peaks["hbm_gbs"]}
    total_ms = sum(ms for ms, n in prof.values())
    for name in kernels:
        kernels[name]["share"] = prof[name][0] / total_ms
    top = max(kernels, key=lambda k: prof[k][0])
    k = kernels[top]
    traffic = ncu_traffic(w.name, top)
    roofline = {"kernel": top, "bound": k["bound"], "achieved": round(k["achieved"], 2),
                "peak": tc_peak if k["bound"] == "tensor" else peaks["hbm_gbs"], "unit": k["unit"],
                "frac": round(k["frac"], 4), "traffic": traffic,
                "peak_source": f"{peak_src} ({'sustained' if sustained and k['bound'] == 'tensor' else 'burst'})"}
    if k["bound"] == "tensor":
        roofline["frac_sustained"] = round(k["frac_sustained"], 4)
        if "frac_per_cycle" in k:
            roofline["frac_per_cycle"] = round(k["frac_per_cycle"], 4)
    gpu_launches = int(sum(n for ms, n in prof.values()))
    gemm_ms = sum(prof[n][0] for n in ("gram_xxt", "gram_aa", "combine_ax_bx", "newton_schulz"))
    gemm_tflops = step_flops(w) * args.steps / (gemm_ms * 1e-3) / 1e12 if gemm_ms > 0 else None

    line = {
        "metric": METRIC, "value": round(value, 3), "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(max_s * 1e3 / args.steps, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded generators; random-init weights, no dataset)",
        "config": config_of(w, world, carry),
        "roofline": roofline,
        "gemm_tflops_per_step": round(gemm_tflops, 1) if gemm_tflops else None,
        "kernels": {n: {kk: (round(v, 4) if isinstance(v, float) else v) for kk, v in d.items()}
                    for n, d in kernels.items()},
        "e2e": {kk: (round(v, 3) if isinstance(v, float) else v) for kk, v in e2e.items()},
        "gpu_launches": gpu_launches,
        "host_submit_ms_per_step": round(host_s * 1e3, 4),
        "ms_per_step_profiled": round(prof_s * 1e3 / args.steps, 4),
        "kernel_ms_per_step": round(total_ms / args.steps, 4),
        "clocks": clk,
        "impl": "ours",
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        t = time_oracle(w, budget_s=args.cpu_budget)
        line["cpu_baseline"] = {"value": round(t["value"], 6), "unit": UNIT, "cores": blas_threads(),
                                "kind": "oracle",
                                "sample": (f"{t['calls']} single-matrix oracle calls cycling over shapes "
                                           f"{t['shapes']} ({t['elapsed_s']:.1f} s, {t['fraction']:.3f} of one "
                                           f"full step by flops), fp64 numpy, extrapolated to the full step")}
    muon.close()
    return line


def run_reference(args) -> dict:
    """The oracle (fp64, host cores) as the reference arm: each step is one matrix of the workload."""
    rank, _, world = dist_env()
    if rank != 0:
        return {}
    w = workload_of(args.workload)
    frac = matrix_fraction(w)
    pick = distinct_matrices(w)
    inputs = {j: oracle_inputs(w, j) for j in pick}
    for i in range(args.warmup):
        oracle_matrix_call(w, pick[i % len(pick)], inputs)
    done, t0 = 0.0, time.perf_counter()
    for i in range(args.steps):
        j = pick[i % len(pick)]
        oracle_matrix_call(w, j, inputs)
        done += frac[j]
    el = time.perf_counter() - t0
    value = done / el
    cores = blas_threads()
    sample = (f"each step: one matrix of {w.name}, cycling over shapes {[list(w.shapes[j]) for j in pick]}; "
              f"{done:.3f} of one full step by flops in {el:.1f} s; fp64 numpy")
    return {"metric": METRIC, "value": round(value, 6), "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(el * 1e3 / args.steps, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded generators)",
            "config": config_of(w, world, bool(getattr(args, "precise_carry", False)) or w.coeffs[2] != 0),
            "impl": "reference",
            "cpu_baseline": {"value": round(value, 6), "unit": UNIT, "cores": cores, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": round(value, 6), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def run_sharded(args) -> dict:
    """The step sharded over the ranks (--sharded): one in-place NCCL reduce-scatter of every
    rank's gradients, muon_step on each rank's own matrices, one in-place all-gather of the bf16
    parameters. One step advances the whole model once, whatever the number of ranks, so value =
    steps / the slowest rank's time (strong scaling)."""
    import torch
    import torch.distributed as dist
    from muon_newton_schulz_09_b300 import ShardedMuon

    rank, local_rank, world = dist_env()
    torch.cuda.set_device(local_rank)
    if not dist.is_initialized():
        if world > 1:
            dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
        else:
            dist.init_process_group("nccl", store=dist.HashStore(), rank=0, world_size=1,
                                    device_id=torch.device("cuda", local_rank))
    w = workload_of(args.workload)
    if w.kind != "step":
        raise SystemExit("--sharded runs muon_step workloads")
    a, b, c = w.coeffs
    sm = ShardedMuon(w.shapes, rank, world, local_rank, lr=w.lr, beta=w.beta, nesterov=w.nesterov,
                     steps=w.steps, a=a, b=b, c=c, eps=w.eps, scale_lr_by_shape=True)
    for j in range(w.count):  # every rank holds the same local gradients: the sum is world x them
        sm.params[j].copy_(torch.from_numpy(wl.parameter(w, j)))
        sm.grads[j].copy_(torch.from_numpy(wl.gradient(w, j)))
    for k, j in enumerate(sm.own):
        sm.momentum[k].copy_(torch.from_numpy(wl.momentum_buffer(w, j)))
    grads0 = sm.flat_grads.clone()
    lo, hi = rank * sm.layout.segment, (rank + 1) * sm.layout.segment
    stream = torch.cuda.current_stream()

    def step():
        # The reduce-scatter leaves the summed gradients in this rank's own segment; with more than
        # one rank that segment gets the local gradients back (a device copy standing in for the
        # backward pass that writes fresh ones). With one rank the reduce-scatter changes nothing.
        if world > 1:
            sm.flat_grads[lo:hi].copy_(grads0[lo:hi], non_blocking=True)
        sm.step()

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    torch.cuda.synchronize()
    with ClockSampler(local_rank) as clk:
        start.record(stream)
        for _ in range(args.steps):
            step()
        end.record(stream)
        torch.cuda.synchronize()
    barrier()
    if sm.muon.get_error() != 0:
        raise RuntimeError("device error flag raised during the timed region")
    max_s = reduce_max(start.elapsed_time(end) / 1e3)
    value = args.steps / max_s

    # end to end: each step uploads this rank's gradients from pinned host memory and reads the
    # replicated parameters back, around the same sharded step
    h_grads = grads0.cpu().pin_memory()
    h_params = torch.empty(sm.flat_params.shape, dtype=sm.flat_params.dtype).pin_memory()
    n_e2e = max(3, min(args.steps, 50))
    barrier()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(n_e2e):
        sm.flat_grads.copy_(h_grads, non_blocking=True)
        sm.step()
        h_params.copy_(sm.flat_params, non_blocking=True)
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_s = reduce_max(e0.elapsed_time(e1) / 1e3)
    cfg = config_of(w, world, False)
    cfg["parallelism"] = (f"sharded x{world}: whole matrices per rank, one reduce-scatter of gradients and "
                          f"one all-gather of parameters per step (NCCL)")
    cfg["owned_matrices"] = len(sm.own)
    cfg["load_balance"] = round(max(sm.layout.load) / (sum(sm.layout.load) / world), 4)
    line = {
        "metric": METRIC, "value": round(value, 3), "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(max_s * 1e3 / args.steps, 4), "higher_is_better": True,
        "scaling": "strong", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded generators; random-init weights, no dataset)", "config": cfg,
        "e2e": {"value": round(n_e2e / e2e_s, 3), "unit": UNIT,
                "h2d_bytes_per_step": h_grads.numel() * h_grads.element_size(),
                "d2h_bytes_per_step": h_params.numel() * h_params.element_size()},
        "clocks": clk.summary(), "impl": "ours-sharded",
    }
    sm.close()
    return line


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=500)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=wl.GPT2_124M.name, choices=sorted(wl.WORKLOADS))
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-budget", type=float, default=15.0, help="seconds of oracle work for cpu_baseline")
    ap.add_argument("--precise-carry", action="store_true",
                    help="carry X between iterations as bf16 hi + lo (the default does so only when c != 0)")
    ap.add_argument("--sharded", action="store_true",
                    help="shard whole matrices over the ranks between a reduce-scatter and an all-gather")
    args = ap.parse_args(argv)
    args.warmup = max(3, args.warmup)  # at least 3 untimed warm-up steps
    if args.impl == "reference":
        line = run_reference(args)
    else:
        line = run_sharded(args) if args.sharded else run_ours(args)
    if line and dist_env()[0] == 0:
        print(json.dumps(line), flush=True)
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized():
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
