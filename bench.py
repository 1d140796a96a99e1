"""Benchmark of the hot path: one step = the three contractions once each on
their full-size synthetic workloads, through the C ABI, on one stream:

  dense     C = A . B^T, M = N = K = 8192, bf16 in, fp32 accumulate, bf16 out
  grouped   MoE up-projection: 64 experts, 16384 tokens routed top-2,
            K = 4096, N = 1536 per expert, bf16 out
  ikbo      linear compression, 64 users x 128 candidates, U[64,256,128],
            C[8192,64,128], W[32,320], fp32 out

value = algorithmic FLOPs of the step / device time (TFLOP/s), whole job over
all ranks (each rank runs its own replica: weak scaling).  Inputs are larger
than L2 (129 MB), so L2 is not flushed between steps.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

--impl reference times the CPU oracle (fp64, all host cores) on a bounded
sample of the same workload, as the reference arm.

Besides the step, the JSON line carries `parity_workloads`: dense 256^3, the
skinny batched GEMM, the RMSNorm- and LayerNorm-fused GEMMs and IKBO attention,
each timed on
its own (`--only rmsnorm|layernorm|attention|skinny|dense256` times one of
them alone).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "bf16 TFLOP/s and % of GB300 dense tensor peak (GEMM, grouped, IKBO)"
UNIT = "TFLOP/s"
WORKLOAD = ("step = dense GEMM 8192x8192x8192 (bf16 out) + grouped MoE GEMM "
            "(64 experts, 16384 tokens top-2, K=4096, N=1536, bf16 out) + IKBO linear "
            "compression (64 users x 128 candidates, Du=256, Dc=64, D=128, O=32, fp32 out)")

# Algorithmic FLOPs (2 per multiply-add) and bytes (each input read once,
# each output written once) of the three workloads.
DENSE = dict(M=8192, N=8192, K=8192)
GROUPED = dict(M=32768, N=1536, K=4096, G=64)
IKBO = dict(users=64, cand=8192, Du=256, Dc=64, D=128, O=32)


def dense_flops(M, N, K, batch=1):
    return 2.0 * batch * M * N * K


def dense_bytes(M, N, K, batch=1, out_bytes=2, shared_b=False):
    return batch * (M * K * 2 + (0 if shared_b else N * K * 2) + M * N * out_bytes) + \
        (N * K * 2 if shared_b else 0)


def grouped_flops(M, N, K, G):
    return 2.0 * M * N * K


def grouped_bytes(M, N, K, G):
    return M * K * 2 + G * N * K * 2 + M * N * 2 + (G + 1) * 4


def ikbo_flops(users, cand, Du, Dc, D, O):
    # decomposed form: once per user for the user part, per candidate for the rest
    return 2.0 * (users * O * Du * D + cand * O * Dc * D)


def ikbo_bytes(users, cand, Du, Dc, D, O):
    return users * Du * D * 2 + cand * Dc * D * 2 + O * (Du + Dc) * 2 + cand * O * D * 4 + \
        (users + 1) * 4


def max_over_ranks(value: float, dist, device) -> float:
    """The largest value across ranks (every rank gets it); identity when
    dist is None.  Used for the timed region: the job is as slow as its
    slowest rank."""
    if dist is None:
        return float(value)
    import torch
    t = torch.tensor([float(value)], dtype=torch.float64,
                     device=device if dist.get_backend() == "nccl" else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(step_flops: float, steps: int, world: int, max_ms: float) -> float:
    """Whole-job TFLOP/s: every rank runs `steps` steps of `step_flops`."""
    return step_flops * steps * world / (max_ms * 1e-3) / 1e12


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return {"bf16_tflops": float(p["bf16_tflops"]),
                "bf16_tflops_sustained": float(p.get("bf16_tflops_sustained", p["bf16_tflops"])),
                "hbm_gbs": float(p["hbm_gbs"]), "source": "measured"}
    except Exception:
        return {"bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "hbm_gbs": 6800.0,
                "source": "fallback"}


KERNEL_SOURCES = {
    "dense": ["sm103.cuh", "wst_common.cuh", "gemm_ws.cuh", "gemm_dense.cu"],
    "grouped": ["sm103.cuh", "wst_common.cuh", "grouped_ws.cuh", "grouped_ws.cu"],
    "ikbo": ["sm103.cuh", "wst_common.cuh", "ikbo_ws.cuh", "ikbo_ws.cu"],
}


def kernel_source_digest(kernel: str):
    """Digest of one kernel's sources, to tell whether committed ncu counters
    still describe the kernel being timed."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "warp_specialized_tensor_gb300", "csrc")
    for f in KERNEL_SOURCES[kernel]:
        path = os.path.join(csrc, f)
        if os.path.exists(path):
            with open(path, "rb") as fh:
                h.update(f.encode() + b"\0" + fh.read())
    return h.hexdigest()[:16]


def committed_traffic(kernel: str):
    """DRAM bytes per launch from the committed ncu summary, or None if the
    kernel's sources changed since the counters were taken."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            t = json.load(f)
        e = t[kernel]
        if e.get("source_digest") != kernel_source_digest(kernel):
            return None
        return float(e["dram_bytes_per_launch"])
    except Exception:
        return None


# ----------------------------------------------------------------------------
# clocks sampler
# ----------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.dev = device_index
        self.samples = []
        self.proc = None
        self.thread = None
        self.window = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.dev), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "25"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.samples.append((time.time(), line.strip()))

    def mark(self, t0, t1):
        self.window = (t0, t1)

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
        if self.thread is not None:
            self.thread.join(timeout=2)

    def summary(self):
        rows = []
        for t, line in self.samples:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 7:
                continue
            try:
                rows.append((t, float(parts[0]), float(parts[1]), parts[3:7]))
            except ValueError:
                continue
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        inside = rows
        if self.window:
            w = [r for r in rows if self.window[0] - 0.05 <= r[0] <= self.window[1] + 0.05]
            if w:
                inside = w
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in inside for i, v in enumerate(r[3]) if v == "Active"})
        return {"sm_mhz": statistics.median(r[1] for r in inside),
                "sm_max_mhz": max(r[2] for r in inside), "reasons": reasons,
                "samples": len(inside)}


# ----------------------------------------------------------------------------
# our arm
# ----------------------------------------------------------------------------
def run_ours(args, rank, world, dist):
    import torch
    import synthetic
    import warp_specialized_tensor_gb300 as wst

    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    wst.load_library()
    peaks = load_peaks()

    extra_only = {"rmsnorm": "dense8192_rmsnorm", "layernorm": "dense8192_layernorm",
                  "attention": "ikbo_attention", "skinny": "skinny_batch",
                  "dense256": "dense256"}.get(args.only)
    if extra_only:
        need = ()
    else:
        need = (args.only,) if args.only else ("dense", "grouped", "ikbo")
    host = {}
    d = g = k = None
    if "dense" in need:
        d = synthetic.workload("dense8192")
        host.update({"dA": d["A"], "dB": d["B"]})
    if "grouped" in need:
        g = synthetic.workload("grouped_moe")
        host.update({"gA": g["A"], "gB": g["B"], "goff": g["offsets"]})
    if "ikbo" in need:
        k = synthetic.workload("ikbo")
        host.update({"kU": k["U"], "kC": k["C"], "kW": k["W"], "koff": k["user_offsets"]})
    dv = {n: t.to(dev) for n, t in host.items()}
    dC = torch.empty(8192, 8192, dtype=torch.bfloat16, device=dev) if d else None
    gC = torch.empty(GROUPED["M"], GROUPED["N"], dtype=torch.bfloat16, device=dev) if g else None
    kY = torch.empty(IKBO["cand"], IKBO["O"], IKBO["D"], dtype=torch.float32, device=dev) if k else None
    ws = wst.workspace(device=dev)
    wsk = wst.workspace(IKBO["users"], IKBO["O"], IKBO["D"], device=dev)
    stream = torch.cuda.current_stream(dev)

    def k_dense():
        wst.wst_gemm_bf16(dv["dA"], dv["dB"], dC, workspace=ws, stream=stream)

    def k_grouped():
        wst.wst_grouped_gemm_bf16(dv["gA"], dv["gB"], dv["goff"], gC, workspace=ws, stream=stream)

    def k_ikbo():
        wst.wst_ikbo_linear_compress(dv["kU"], dv["kC"], dv["kW"], dv["koff"], kY, wsk,
                                     stream=stream)

    kernels = [("dense", k_dense), ("grouped", k_grouped), ("ikbo", k_ikbo)]
    if args.only:
        kernels = [kv for kv in kernels if kv[0] == args.only]
    if extra_only:
        out = time_parity_workloads(wst, torch, dev, stream, peaks, ws, names=(extra_only,),
                                    iters=max(1, args.steps))
        return {"metric": "extra workload timing (profiling run; not a bench line)",
                "only": extra_only, "parity_workloads": out}
    flops = {"dense": dense_flops(**DENSE), "grouped": grouped_flops(**GROUPED),
             "ikbo": ikbo_flops(**IKBO)}
    nbytes = {"dense": dense_bytes(**DENSE), "grouped": grouped_bytes(**GROUPED),
              "ikbo": ikbo_bytes(**IKBO)}
    step_flops = sum(flops[n] for n, _ in kernels)

    # warm-up
    for _ in range(args.warmup):
        for _, fn in kernels:
            fn()
    torch.cuda.synchronize(dev)
    for w_ in (ws, wsk):
        st = wst.wst_sync_status(w_, stream)
        if st != 0:
            raise RuntimeError("device error during warm-up: %s" % wst.wst_status_string(st))

    # timed region: K steps, per-kernel events on the launching stream
    ev = {n: [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(args.steps)] for n, _ in kernels}
    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.4)  # let the sampler start before the timed region
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize(dev)
    t_begin = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    wall0 = time.time()
    t_begin.record(stream)
    for i in range(args.steps):
        for n, fn in kernels:
            a, b = ev[n][i]
            a.record(stream)
            fn()
            b.record(stream)
    t_end.record(stream)
    torch.cuda.synchronize(dev)
    wall1 = time.time()
    if dist is not None:
        dist.barrier()
    sampler.mark(wall0, wall1)
    time.sleep(0.15)
    sampler.stop()
    for w_ in (ws, wsk):
        st = wst.wst_sync_status(w_, stream)
        if st != 0:
            raise RuntimeError("device error in timed region: %s" % wst.wst_status_string(st))
    elapsed_ms = t_begin.elapsed_time(t_end)
    per_kernel_ms = {n: sum(a.elapsed_time(b) for a, b in ev[n]) / args.steps for n, _ in kernels}

    elapsed_ms = max_over_ranks(elapsed_ms, dist, dev)
    ms_per_step = elapsed_ms / args.steps
    value = job_throughput(step_flops, args.steps, world, elapsed_ms)

    # ---- e2e: the step through the public API from pinned host buffers, with
    # every step's uploads and its result readback inside the timed region.
    # Pipelined over two device buffer sets: step i+1's uploads (32 MB chunks
    # over four copy streams) and step i's readback (a fifth stream) overlap
    # step i's kernels.
    pinned = {n: t.pin_memory() for n, t in host.items()}
    outs0 = {n: t for n, t in (("dC", dC), ("gC", gC), ("kY", kY)) if t is not None}
    h2d = sum(t.numel() * t.element_size() for t in pinned.values())
    d2h = sum(t.numel() * t.element_size() for t in outs0.values())
    e2e_steps = max(3, min(args.steps, 20)) if not args.no_e2e else 0

    def run_step(src, dst):
        if "dense" in need:
            wst.wst_gemm_bf16(src["dA"], src["dB"], dst["dC"], workspace=ws, stream=stream)
        if "grouped" in need:
            wst.wst_grouped_gemm_bf16(src["gA"], src["gB"], src["goff"], dst["gC"], workspace=ws,
                                      stream=stream)
        if "ikbo" in need:
            wst.wst_ikbo_linear_compress(src["kU"], src["kC"], src["kW"], src["koff"], dst["kY"], wsk,
                                         stream=stream)

    e2e_ms = float("nan")
    if e2e_steps:
        ins = [dv, {n: torch.empty_like(t) for n, t in dv.items()}]
        outs = [outs0, {n: torch.empty_like(t) for n, t in outs0.items()}]
        out_host = [{n: torch.empty(t.shape, dtype=t.dtype).pin_memory() for n, t in outs0.items()}
                    for _ in range(2)]
        up = [torch.cuda.Stream(dev) for _ in range(4)]
        down = torch.cuda.Stream(dev)
        # (name, flat element range) chunks of ~32 MB, dealt round-robin to the streams
        chunks = []
        for n, t in pinned.items():
            step = max(1, (32 << 20) // t.element_size())
            for a in range(0, t.numel(), step):
                chunks.append((n, a, min(t.numel(), a + step)))

        def pipeline(nsteps, start_ev=None):
            kdone, rb = [], []
            for i in range(nsteps):
                b = i & 1
                ev_up = []
                for k, us in enumerate(up):
                    if start_ev is not None:
                        us.wait_event(start_ev)
                    if i >= 2:
                        us.wait_event(kdone[i - 2])    # set b no longer read
                    with torch.cuda.stream(us):
                        for n, a0, a1 in chunks[k::len(up)]:
                            ins[b][n].view(-1)[a0:a1].copy_(pinned[n].view(-1)[a0:a1], non_blocking=True)
                    e = torch.cuda.Event()
                    e.record(us)
                    ev_up.append(e)
                for e in ev_up:
                    stream.wait_event(e)
                if i >= 2:
                    stream.wait_event(rb[i - 2])       # outputs of set b read back
                run_step(ins[b], outs[b])
                e = torch.cuda.Event()
                e.record(stream)
                kdone.append(e)
                down.wait_event(e)
                with torch.cuda.stream(down):
                    for n, t in outs[b].items():
                        out_host[b][n].copy_(t, non_blocking=True)
                e = torch.cuda.Event()
                e.record(down)
                rb.append(e)
            stream.wait_event(rb[-1])

        pipeline(2)
        torch.cuda.synchronize(dev)
        if dist is not None:
            dist.barrier()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        pipeline(e2e_steps, start_ev=e0)
        e1.record(stream)
        torch.cuda.synchronize(dev)
        e2e_ms = e0.elapsed_time(e1)
    if e2e_steps:
        e2e_ms = max_over_ranks(e2e_ms, dist, dev)
    e2e_value = job_throughput(step_flops, e2e_steps, world, e2e_ms) if e2e_steps else None

    # ---- context: cuBLAS through torch.matmul on the dense workload (not the product)
    ctx = {}
    if not args.no_context and d is not None:
        Bt = dv["dB"].t()
        for _ in range(3):
            torch.matmul(dv["dA"], Bt)
        torch.cuda.synchronize(dev)
        c0 = torch.cuda.Event(enable_timing=True)
        c1 = torch.cuda.Event(enable_timing=True)
        c0.record(stream)
        for _ in range(10):
            torch.matmul(dv["dA"], Bt)
        c1.record(stream)
        torch.cuda.synchronize(dev)
        ctx["torch_matmul_dense_tflops"] = round(flops["dense"] * 10 / (c0.elapsed_time(c1) * 1e-3) / 1e12, 1)

    # ---- the extra workloads (parity cases and next rows), timed on their own
    extra = {}
    if not args.only and not args.no_extra:
        extra = time_parity_workloads(wst, torch, dev, stream, peaks, ws)

    variants = {}
    for n, _ in kernels:
        ms = per_kernel_ms[n]
        tf = flops[n] / (ms * 1e-3) / 1e12
        gbs = nbytes[n] / (ms * 1e-3) / 1e9
        t_flop = flops[n] / (peaks["bf16_tflops"] * 1e12)
        t_byte = nbytes[n] / (peaks["hbm_gbs"] * 1e9)
        variants[n] = {"ms": round(ms, 4), "tflops": round(tf, 1),
                       "frac_dense_peak": round(tf / peaks["bf16_tflops"], 4),
                       "gbs": round(gbs, 1),
                       "bound": "tensor" if t_flop >= t_byte else "hbm",
                       "frac_roofline": round(max(t_flop, t_byte) / (ms * 1e-3), 4),
                       "algorithmic_flops": flops[n], "algorithmic_bytes": nbytes[n]}

    dom = "dense" if "dense" in per_kernel_ms else kernels[0][0]
    ach = flops[dom] / (per_kernel_ms[dom] * 1e-3) / 1e12
    roofline = {"kernel": "k_gemm_ws (dense 8192^3)", "bound": "tensor", "achieved": round(ach, 1),
                "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                "frac": round(ach / peaks["bf16_tflops"], 4),
                "traffic": committed_traffic(dom),
                "peak_source": peaks["source"] + " (burst bf16, cuBLAS)",
                # context: the same kernel against the power-capped sustained figure
                "peak_sustained": peaks["bf16_tflops_sustained"],
                "frac_of_sustained": round(ach / peaks["bf16_tflops_sustained"], 4)}

    result = {
        "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded, shapes and distributions of the named workloads)",
        "config": {"workload": WORKLOAD, "l2": "inputs larger than L2 (no flush)",
                   "parallelism": "replicas" if world > 1 else "single GPU"},
        "roofline": roofline,
        "e2e": {"value": round(e2e_value, 2) if e2e_value else None, "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "steps": e2e_steps,
                "mode": "pipelined: step i+1's uploads (32 MB chunks on 4 copy streams) and step "
                        "i's readback overlap step i's kernels; two device buffer sets"},
        "gpu_launches": len(kernels) * args.steps,
        "clocks": sampler.summary(),
        "variants": variants,
        "parity_workloads": extra,
        "peaks": peaks,
        "context": ctx,
    }
    if rank == 0 and not args.no_cpu_baseline and not args.only:
        result["cpu_baseline"] = cpu_baseline(d, g, k, budget_s=args.cpu_seconds)
    return result


def time_parity_workloads(wst, torch, dev, stream, peaks, ws, iters: int = 20, names=None):
    """dense 256^3 (fp32 out; launch-latency bound), the skinny recsys batch
    (512 x 1024x256x512, bias+SiLU, bf16 out; HBM-bound; 940 MB > L2), the
    row-RMSNorm- and LayerNorm-fused GEMMs on the dense 8192^3 operands, and
    IKBO attention."""
    import synthetic
    out = {}
    extra_ws = [ws]

    def dense256():
        d1 = synthetic.workload("dense256")
        A1, B1 = d1["A"].to(dev), d1["B"].to(dev)
        C1 = torch.empty(256, 256, dtype=torch.float32, device=dev)
        return (lambda: wst.wst_gemm_bf16(A1, B1, C1, workspace=ws, stream=stream),
                dense_flops(256, 256, 256), dense_bytes(256, 256, 256, out_bytes=4))

    def skinny_batch():
        d5 = synthetic.workload("skinny_batch")
        A5, B5, b5 = d5["A"].to(dev), d5["B"].to(dev), d5["bias"].to(dev)
        C5 = torch.empty(512, 1024, 256, dtype=torch.bfloat16, device=dev)
        return (lambda: wst.wst_gemm_bf16(A5, B5, C5, bias=b5, epi="bias_silu", workspace=ws,
                                          stream=stream),
                dense_flops(1024, 256, 512, batch=512),
                dense_bytes(1024, 256, 512, batch=512) + 512 * 256 * 2)

    def dense8192_rmsnorm():
        # the row-RMSNorm GEMM on the dense 8192^3 operands: with room for
        # the row statistics the library takes them in a separate pass over
        # A (N > 1024), both kernels timed (A read twice)
        d2 = synthetic.workload("dense8192")
        A2, B2 = d2["A"].to(dev), d2["B"].to(dev)
        C2 = torch.empty(8192, 8192, dtype=torch.bfloat16, device=dev)
        ws2 = wst.norm_workspace(A2, B2, stream=stream)
        extra_ws.append(ws2)
        return (lambda: wst.wst_gemm_rmsnorm_bf16(A2, B2, C2, eps=1e-6, workspace=ws2, stream=stream),
                dense_flops(8192, 8192, 8192), dense_bytes(8192, 8192, 8192))

    def dense8192_layernorm():
        # the row-LayerNorm GEMM on the dense 8192^3 operands: the column-sum
        # kernel, the row-statistics pass and the GEMM, all timed (A and B
        # read twice)
        d3 = synthetic.workload("dense8192")
        A3, B3 = d3["A"].to(dev), d3["B"].to(dev)
        C3 = torch.empty(8192, 8192, dtype=torch.bfloat16, device=dev)
        ws3 = wst.norm_workspace(A3, B3, layernorm=True, stream=stream)
        extra_ws.append(ws3)
        return (lambda: wst.wst_gemm_layernorm_bf16(A3, B3, C3, eps=1e-5, workspace=ws3,
                                                    stream=stream),
                dense_flops(8192, 8192, 8192), dense_bytes(8192, 8192, 8192))

    def ikbo_attention():
        # 32 users x 256 candidates x 2 query rows, 4 heads, Dh 128, 2048
        # context rows per user; bf16 out.  FLOPs: QK^T and PV; bytes: Q, the
        # users' K and V once, O.
        d6 = synthetic.workload("ikbo_attention")
        Q6, K6, V6 = d6["Q"].to(dev), d6["K"].to(dev), d6["V"].to(dev)
        off6 = d6["user_offsets"].to(dev)
        O6 = torch.empty(Q6.shape, dtype=torch.bfloat16, device=dev)
        nq6, H6, Dh6 = Q6.shape
        Lkv6 = K6.shape[1]
        ws6 = wst.attention_workspace(device=dev, stream=stream)
        extra_ws.append(ws6)
        return (lambda: wst.wst_ikbo_attention_bf16(Q6, K6, V6, off6, O6, Lq=d6["Lq"],
                                                    workspace=ws6, stream=stream),
                4.0 * nq6 * Lkv6 * Dh6 * H6,
                2 * (2 * nq6 * H6 * Dh6) + 2 * (2 * K6.numel()))

    builders = [("dense256", dense256), ("skinny_batch", skinny_batch),
                ("dense8192_rmsnorm", dense8192_rmsnorm),
                ("dense8192_layernorm", dense8192_layernorm), ("ikbo_attention", ikbo_attention)]
    for name, build in builders:
        if names is not None and name not in names:
            continue
        fn, fl, by = build()
        for _ in range(3):
            fn()
        torch.cuda.synchronize(dev)
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        # Queue the timed calls behind a short device-side sleep so that the
        # host's per-call work (argument checks, tensor maps: about as long as
        # the smallest kernels here) does not leave the GPU idle between them.
        with torch.cuda.stream(stream):
            torch.cuda._sleep(8_000_000)
        e0.record(stream)
        for _ in range(iters):
            fn()
        e1.record(stream)
        torch.cuda.synchronize(dev)
        ms = e0.elapsed_time(e1) / iters
        t_flop = fl / (peaks["bf16_tflops"] * 1e12)
        t_byte = by / (peaks["hbm_gbs"] * 1e9)
        out[name] = {"ms": round(ms, 4), "tflops": round(fl / (ms * 1e-3) / 1e12, 1),
                     "gbs": round(by / (ms * 1e-3) / 1e9, 1),
                     "bound": "tensor" if t_flop >= t_byte else "hbm",
                     "frac_roofline": round(max(t_flop, t_byte) / (ms * 1e-3), 4)}
    for w in extra_ws:
        st = wst.wst_sync_status(w, stream)
        if st != 0:
            raise RuntimeError("device error in parity workloads: %s" % wst.wst_status_string(st))
    return out


# ----------------------------------------------------------------------------
# the oracle as CPU baseline / reference arm
# ----------------------------------------------------------------------------
def oracle_sample(d, g, k, scale: int):
    """One bounded sample of the step for the fp64 oracle: `scale` rows of the
    dense GEMM, `scale` rows of one expert, 4*`scale` IKBO candidates.
    Returns (flops done, seconds)."""
    import oracle
    t0 = time.time()
    rows = list(range(0, 8192, max(1, 8192 // scale)))[:scale]
    oracle.gemm(d["A"], d["B"], rows=rows)
    off = g["offsets"].tolist()
    e = 7
    r0, r1 = off[e], off[e + 1]
    sel = list(range(r0, min(r1, r0 + scale)))
    oracle.gemm(g["A"][sel], g["B"][e])
    cands = list(range(0, 8192, max(1, 8192 // (4 * scale))))[:4 * scale]
    oracle.ikbo(k["U"], k["C"], k["W"], k["user_offsets"], cands=cands)
    dt = time.time() - t0
    F = IKBO["Du"] + IKBO["Dc"]
    fl = 2.0 * len(rows) * 8192 * 8192 + 2.0 * len(sel) * 1536 * 4096 + \
        2.0 * len(cands) * IKBO["O"] * F * IKBO["D"]
    return fl, dt


def cpu_baseline(d, g, k, budget_s: float = 15.0):
    """Time the oracle, as it stands, on repeated bounded samples of the step
    until about budget_s seconds of CPU work are done."""
    import oracle
    scale = 64
    tot_fl, tot_dt, reps = 0.0, 0.0, 0
    while tot_dt < budget_s and reps < 1000:
        fl, dt = oracle_sample(d, g, k, scale)
        tot_fl += fl
        tot_dt += dt
        reps += 1
    return {"value": tot_fl / tot_dt / 1e12, "unit": UNIT, "cores": oracle.num_threads(),
            "kind": "oracle",
            "sample": "%d x (%d dense rows with all 8192 columns, %d rows of expert 7, %d IKBO "
                      "candidates); fp64 accumulation; %.1f s" % (reps, scale, scale, 4 * scale, tot_dt)}


def record_traffic(report: str, kernel_key: str, regex: str):
    """Write profiles/traffic.json[kernel_key] from an ncu report of one launch:
    dram__bytes_read.sum + dram__bytes_write.sum, stamped with the current
    kernel-source digest (so bench.py reports null once the kernels change)."""
    import csv
    import io
    out = subprocess.run(["ncu", "-i", report, "--page", "raw", "--csv"], capture_output=True,
                         text=True, check=True).stdout
    rows = list(csv.reader(io.StringIO(out)))
    hdr, units = rows[0], rows[1]
    import re
    scale = {"byte": 1, "Kbyte": 1e3, "Mbyte": 1e6, "Gbyte": 1e9}
    launches = []
    for r in rows[2:]:
        name = r[hdr.index("Kernel Name")]
        if not re.search(regex, name):
            continue
        tot = 0.0
        for m in ("dram__bytes_read.sum", "dram__bytes_write.sum"):
            i = hdr.index(m)
            tot += float(r[i]) * scale[units[i]]
        launches.append(tot)
    if not launches:
        raise SystemExit("no launch of %r in %s" % (regex, report))
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        data = json.load(open(path))
    except Exception:
        data = {}
    data[kernel_key] = {"dram_bytes_per_launch": sum(launches) / len(launches),
                        "launches": len(launches), "report": os.path.basename(report),
                        "source_digest": kernel_source_digest(kernel_key)}
    with open(path, "w") as f:
        json.dump(data, f, indent=1, sort_keys=True)
    print(json.dumps(data[kernel_key]))


def run_reference(args, rank, world):
    import oracle
    import synthetic
    oracle.build()
    d = synthetic.workload("dense8192")
    g = synthetic.workload("grouped_moe")
    k = synthetic.workload("ikbo")
    fl1, dt1 = oracle_sample(d, g, k, 1)
    per_unit = dt1
    budget = max(0.05, args.ref_seconds / max(1, args.steps + args.warmup))
    scale = max(1, int(budget / max(per_unit, 1e-6)))
    for _ in range(args.warmup):
        oracle_sample(d, g, k, scale)
    tot_fl, tot_dt = 0.0, 0.0
    for _ in range(args.steps):
        fl, dt = oracle_sample(d, g, k, scale)
        tot_fl += fl
        tot_dt += dt
    value = tot_fl / tot_dt / 1e12
    sample = ("per step: %d dense rows (all columns), %d rows of expert 7, %d IKBO candidates "
              "of the same workload; fp64 oracle on host cores" % (scale, scale, 4 * scale))
    return {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": tot_dt * 1e3 / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": {"workload": WORKLOAD, "l2": "n/a (CPU)",
                                        "parallelism": "single process"},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": oracle.num_threads(),
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-context", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-extra", action="store_true",
                    help="skip timing the extra workloads (parity cases and next rows)")
    ap.add_argument("--only", choices=["dense", "grouped", "ikbo", "rmsnorm", "layernorm", "attention",
                                       "skinny", "dense256"],
                    default=None,
                    help="time one kernel only (profiling runs); not a bench line. rmsnorm, "
                         "layernorm, attention, skinny and dense256 time that extra workload alone")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--ref-seconds", type=float, default=90.0)
    ap.add_argument("--record-traffic", nargs=3, metavar=("REPORT", "KEY", "REGEX"),
                    help="store DRAM bytes per launch from an ncu report in profiles/traffic.json")
    args = ap.parse_args()
    if args.record_traffic:
        record_traffic(*args.record_traffic)
        return 0
    if args.warmup < 3 and args.impl == "ours":
        args.warmup = 3

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    dist = None
    if args.impl == "reference":
        if rank != 0:
            return 0
        print(json.dumps(run_reference(args, rank, world)))
        return 0
    if world > 1:
        import torch
        import torch.distributed as tdist
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", "0")))
        tdist.init_process_group(backend)
        dist = tdist
    res = run_ours(args, rank, world, dist)
    if rank == 0:
        print(json.dumps(res))
    if dist is not None:
        dist.barrier()
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
