"""Throughput of the context-parallel zigzag ring attention hot path on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
                    [--impl ours|reference]

One step is the whole hot path over one batch of synthetic input resident in
HBM: zigzag-permute Q, K, V, dO into sharded order, ring forward (O, LSE),
ring backward (dQ, dK, dV from the saved LSE), unpermute O, LSE, dQ, dK, dV
back to natural order.  The default workload is the S=131072 forward+backward
one (B=1, H=32, Hkv=8, D=128, cp=16, zigzag, causal, bf16); the S=32768
forward on which the tensor-roofline target is quoted is timed in the same
run and reported under "c3_forward".

Metric: useful attention TFLOP/s -- 4*D flops per visible (query, key) pair
forward, 10*D backward (S(S+1)/2 visible pairs per head when causal; under
packed documents, the sum over documents).  Inputs are far larger than L2
(129 MB), so no flush is needed between steps.

The same run times the packed-document workload (S=131072, documents of mean
length 8192) forward and backward and reports it under "docs", and the
S=131072 workload through the all-gather K/V schedule (K/V gathered into
natural order, one pass per rank, gathered dK/dV returned to their owners)
under "allgather", through the Ulysses variant (all-to-all to head
ownership, full attention per head slice, all-to-all back) under "ulysses",
and through the hierarchical a2a+p2p schedule with level sizes [4, 4] under
"hierarchical"; the forwards of the other named workloads (S=256 float32,
S=8192 zigzag and contiguous with their kernel censuses, S=16384 full
attention at cp 1, 2, 4, 8) are timed alone under "named_forwards";
``--workload docs_bf16_s131072_fwdbwd`` makes it the main line (its step adds
the document-bounds kernel and uses the document-rule forward/backward).

Under torchrun (N > 1) each rank runs an independent replica on its own GPU
(the path itself runs on one GPU: "replicas only"); the reported value is the
work of all ranks over the slowest rank's time.

``--impl reference`` times the fp64 CPU oracle on the host cores instead, on a
bounded sample of the same workload (rank 0 only).
"""
import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from context_causal_attention_zigzag_gb300 import inputs  # noqa: E402

METRIC = "useful causal attention TFLOP/s on 1 GB300 (fwd, fwd+bwd) and % of BF16 tensor peak"
UNIT = "TFLOP/s"
ALL_WORKLOADS = {**inputs.WORKLOADS, **inputs.DOC_WORKLOADS}


# DRAM bytes per launch (dram__bytes_read.sum + dram__bytes_write.sum) of each
# kernel, one ncu capture per kernel on the S=16384 reduction of the
# S=131072 workload (same heads, head dim and layout; 1/8 of the tokens,
# 1/64 of the tile pairs).  The traffic does not grow in proportion to the
# work from there to the full size (compulsory bytes grow 8x, re-reads with
# the L2 miss rate), so the full-size roofline reports these figures beside
# a null traffic instead of a scaled guess.  Re-take them whenever a kernel
# changes.
REDUCED_CASE_TRAFFIC = {
    "workload": "S=16384 reduction (B1 H32 Hkv8 D128 cp4 zigzag causal, float32 gradients)",
    "bytes": {
        "tc_fwd_kernel": 276.1e6 + 96.0e6,
        "bwd_prep_kernel": 268.5e6 + 4.3e6,
        "dkdv_kernel": 484.7e6 + 485.9e6,
        "dq_kernel": 507.4e6 + 222.5e6,
        "grad_reduce_kernel": 536.9e6 + 117.2e6,
        "dkdvq_kernel": 1098.1e6 + 1038.3e6,
    },
}


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as fh:
            d = json.load(fh)
        return float(d["bf16_tflops"]), float(d.get("bf16_tflops_sustained", d["bf16_tflops"])), \
            float(d["hbm_gbs"]), "measured"
    return 1900.0, 1700.0, 6800.0, "fallback"


def max_over_ranks(x, ws, device):
    """The largest of x over all ranks (x itself for one rank); `device` is
    where the process group's backend wants the tensor (CUDA for NCCL)."""
    if ws == 1:
        return float(x)
    import torch.distributed as dist
    t = torch.tensor([float(x)], device=device, dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_value(step_flops, ws, ms_max):
    """TFLOP/s of the whole job: every rank's step over the slowest rank's time."""
    return step_flops * ws / (ms_max * 1e-3) / 1e12


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


# ---------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", self.gpu, f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=self.fh, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.fh.close()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as fh:
            for line in fh:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    mx.append(float(parts[2]))
                except ValueError:
                    continue
                for name, val in zip(names, parts[5:9]):
                    if val.lower() == "active":
                        reasons.add(name)
        os.unlink(self.path)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx),
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------

def run_ours(args):
    import context_causal_attention_zigzag_gb300 as cpa

    ws, rank, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    w = ALL_WORKLOADS[args.workload]
    peak, peak_sus, hbm, peak_kind = peaks()
    stream = torch.cuda.current_stream(dev)
    onepass = args.bwd == "onepass"

    q, k, v, do = inputs.generate(w)
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    dod = do.to(dev) if do is not None else None
    cp, layout, causal = w.cp, w.layout, w.causal
    B, S, H, Hkv, D = w.B, w.S, w.H, w.Hkv, w.D

    # Preallocated sharded buffers, outputs and workspace: the step allocates nothing.
    qs, ks, vs = torch.empty_like(qd), torch.empty_like(kd), torch.empty_like(vd)
    o = torch.empty_like(qd)
    lse = torch.empty((B, H, S), device=dev, dtype=torch.float32)
    o_nat, lse_nat = torch.empty_like(o), torch.empty_like(lse)
    if w.backward:
        # float32 gradients: the configuration the full-size parity test checks
        # (a bf16 dV element near the first key exceeds the 2e-2 bar by rounding).
        gdt = torch.float32
        dos = torch.empty_like(dod)
        dq = torch.empty(qd.shape, device=dev, dtype=gdt)
        dk = torch.empty(kd.shape, device=dev, dtype=gdt)
        dv = torch.empty(vd.shape, device=dev, dtype=gdt)
        dq_nat, dk_nat, dv_nat = torch.empty_like(dq), torch.empty_like(dk), torch.empty_like(dv)
        wsp = torch.empty(cpa.ring_bwd_workspace_bytes(B, H, Hkv, S, D, cpa.BF16 | cpa.GRAD_F32),
                          device=dev, dtype=torch.uint8)
    docs = w.doc_offsets()
    if docs is not None:
        cu_dev = torch.tensor(docs, dtype=torch.int32, device=dev)
        bounds = torch.empty((S, 2), dtype=torch.int32, device=dev)
    ev = {}

    def mark(name):
        e = torch.cuda.Event(enable_timing=True)
        e.record(stream)
        ev.setdefault(name, []).append(e)

    def step(timed=False, src=(qd, kd, vd, dod)):
        sq, sk, sv, sdo = src
        cpa.zigzag_permute(sq, cp, layout, out=qs)
        cpa.zigzag_permute(sk, cp, layout, out=ks)
        cpa.zigzag_permute(sv, cp, layout, out=vs)
        if w.backward:
            cpa.zigzag_permute(sdo, cp, layout, out=dos)
        if docs is not None:
            cpa.doc_bounds(cu_dev, S, out=bounds)
        if timed:
            mark("fwd0")
        if docs is None:
            cpa.ring_fwd(qs, ks, vs, cp, layout, causal, out=o, lse=lse)
        else:
            cpa.ring_fwd_docs(qs, ks, vs, cp, bounds, layout, causal, out=o, lse=lse)
        if timed:
            mark("fwd1")
        if w.backward:
            if docs is None:
                cpa.ring_bwd(qs, ks, vs, o, dos, lse, cp, layout, causal, dq=dq, dk=dk, dv=dv,
                             workspace=wsp, grad_dtype=gdt, onepass=onepass)
            else:
                cpa.ring_bwd_docs(qs, ks, vs, o, dos, lse, cp, bounds, layout, causal, dq=dq,
                                  dk=dk, dv=dv, workspace=wsp, grad_dtype=gdt, onepass=onepass)
            if timed:
                mark("bwd1")
        cpa.zigzag_unpermute(o, cp, layout, out=o_nat)
        cpa.zigzag_unpermute(lse, cp, layout, seq_dim=2, out=lse_nat)
        if w.backward:
            cpa.zigzag_unpermute(dq, cp, layout, out=dq_nat)
            cpa.zigzag_unpermute(dk, cp, layout, out=dk_nat)
            cpa.zigzag_unpermute(dv, cp, layout, out=dv_nat)

    bwd_path = cpa.plan(B, H, Hkv, S, D, cp, layout, causal, w.dtype, backward=True)[0] \
        if w.backward else None
    # permutes + forward + backward (pre-pass, kernel(s), finishing pass(es)) + unpermutes
    if not w.backward:
        bwd_launches = 0
    elif bwd_path != cpa.PATH_TCGEN05:
        bwd_launches = 3
    else:
        bwd_launches = 3 if onepass else 4   # one-pass: float32 dQ needs no conversion
    launches_per_step = ((4 if w.backward else 3) + 1 + bwd_launches + (5 if w.backward else 2)
                         + (1 if docs is not None else 0))
    fwd_flops = w.useful_flops(False)
    bwd_flops = w.useful_flops(True) if w.backward else 0.0
    step_flops = fwd_flops + bwd_flops

    def barrier():
        if ws > 1:
            import torch.distributed as dist
            dist.barrier()
        torch.cuda.synchronize(dev)

    for _ in range(args.warmup):
        step()
    barrier()
    try:
        gpu_id = "GPU-" + str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:
        gpu_id = str(local)
    clocks = ClockSampler(gpu_id)
    clocks.start()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    ev.clear()
    t0.record(stream)
    for _ in range(args.steps):
        step(timed=True)
    t1.record(stream)
    barrier()
    clk = clocks.stop()
    ms = t0.elapsed_time(t1) / args.steps
    fwd_ms = statistics.mean(a.elapsed_time(b) for a, b in zip(ev["fwd0"], ev["fwd1"]))
    bwd_ms = (statistics.mean(a.elapsed_time(b) for a, b in zip(ev["fwd1"], ev["bwd1"]))
              if w.backward else None)
    ms_max = max_over_ranks(ms, ws, dev)
    value = whole_job_value(step_flops, ws, ms_max)

    # End to end through the C ABI on host buffers (cpattn_attention_host):
    # pinned natural-order host inputs in, every result back in host memory.
    e2e = None
    e2e_api = None
    if rank == 0 or ws > 1:
        hq, hk, hv = q.pin_memory(), k.pin_memory(), v.pin_memory()
        hdo = do.pin_memory() if do is not None else None
        outs = [o_nat, lse_nat] + ([dq_nat, dk_nat, dv_nat] if w.backward else [])
        host_outs = [torch.empty(x.shape, dtype=x.dtype, pin_memory=True) for x in outs]
        h2d = sum(x.numel() * x.element_size() for x in (hq, hk, hv, hdo) if x is not None)
        d2h = sum(x.numel() * x.element_size() for x in outs)
        hcode = (cpa.BF16 if w.dtype == torch.bfloat16 else cpa.F32) | \
            (cpa.GRAD_F32 if w.backward else 0)
        hres = dict(zip(("out", "lse", "dq", "dk", "dv"), host_outs))
        if docs is None:
            e2e_api = "cpattn_attention_host"
            hws = torch.empty(cpa.attention_host_workspace_bytes(B, H, Hkv, S, D, cp, layout, hcode,
                                                                 w.backward),
                              device=dev, dtype=torch.uint8)

            def e2e_step():
                cpa.attention_host(hq, hk, hv, hdo, cp, layout, causal, workspace=hws,
                                   grad_dtype=gdt if w.backward else None, onepass=onepass,
                                   **hres)
        else:
            e2e_api = "cpattn_attention_host_docs"
            hws = torch.empty(cpa.attention_host_docs_workspace_bytes(B, H, Hkv, S, D, cp, layout,
                                                                      hcode, w.backward),
                              device=dev, dtype=torch.uint8)

            def e2e_step():
                cpa.attention_host_docs(hq, hk, hv, hdo, cp, docs, layout, causal, workspace=hws,
                                        grad_dtype=gdt if w.backward else None,
                                        onepass=onepass, **hres)

        e2e_step()
        barrier()
        n_e2e = max(1, min(args.steps, 5))
        e2e_clocks = ClockSampler(gpu_id)
        e2e_clocks.start()
        marks = [torch.cuda.Event(enable_timing=True) for _ in range(n_e2e + 1)]
        marks[0].record(stream)
        for i in range(n_e2e):
            e2e_step()
            marks[i + 1].record(stream)
        torch.cuda.synchronize(dev)
        e2e_clk = e2e_clocks.stop()
        per_call = [marks[i].elapsed_time(marks[i + 1]) for i in range(n_e2e)]
        e2e_ms = sum(per_call) / n_e2e
        e2e = {"value": step_flops / (e2e_ms * 1e-3) / 1e12, "unit": UNIT,
               "ms_per_step": e2e_ms, "ms_per_call": per_call, "h2d_bytes_per_step": int(h2d),
               "d2h_bytes_per_step": int(d2h), "api": e2e_api, "clocks": e2e_clk}
        e2e["head_parts"] = cpa.attention_host_parts(B, H, Hkv, S, D)
        e2e["host_link_gbs"] = host_link_gbs(dev, stream)

    # Roofline of the dominant kernel, from the live event timings.  The
    # kernels of the step are timed inside the multi-second loop of back-to-back
    # steps, so the denominator is the sustained bf16 figure; the burst one is
    # reported beside it.
    dom_ms, dom_flops, dom_name = (bwd_ms, bwd_flops, "ring_bwd") \
        if (w.backward and bwd_ms >= fwd_ms) else (fwd_ms, fwd_flops, "ring_fwd")
    achieved = dom_flops / (dom_ms * 1e-3) / 1e12
    tb = REDUCED_CASE_TRAFFIC["bytes"]
    if dom_name == "ring_bwd":
        parts = (["bwd_prep_kernel", "dkdvq_kernel", "grad_reduce_kernel"] if onepass else
                 ["bwd_prep_kernel", "dkdv_kernel", "dq_kernel", "grad_reduce_kernel"])
    else:
        parts = ["tc_fwd_kernel"]
    reduced = {"workload": REDUCED_CASE_TRAFFIC["workload"], "kernels": parts,
               "bytes_per_launch": sum(tb[p] for p in parts)}
    roofline = {"kernel": dom_name, "bound": "tensor", "achieved": achieved, "peak": peak_sus,
                "unit": "TFLOP/s", "frac": achieved / peak_sus, "traffic": None,
                "traffic_reduced_case": reduced,
                "peak_kind": f"{peak_kind} bf16 sustained (kernel timed inside the step loop)",
                "ms": dom_ms, "peak_burst": peak, "frac_of_burst": achieved / peak}
    fwd_info = {"ms": fwd_ms, "tflops": fwd_flops / (fwd_ms * 1e-3) / 1e12}
    fwd_info["frac"] = fwd_info["tflops"] / peak_sus
    fwd_info["frac_of_burst"] = fwd_info["tflops"] / peak
    if w.backward:
        fwd_info["bwd_ms"] = bwd_ms
        fwd_info["bwd_tflops"] = bwd_flops / (bwd_ms * 1e-3) / 1e12

    # The S=32768 forward (tensor-roofline target workload), timed alone.
    c3 = None
    if args.workload != "c3_bf16_s32768_gqa" and not args.no_c3:
        c3 = time_forward(cpa, inputs.WORKLOADS["c3_bf16_s32768_gqa"], dev, stream,
                          args.warmup, max(args.steps, 5), peak)
    # The packed-document workload, forward and backward timed alone.
    docs_info = None
    if docs is None and not args.no_docs:
        wd = inputs.DOC_WORKLOADS["docs_bf16_s131072_fwdbwd"]
        docs_info = time_docs(cpa, wd, dev, stream, args.warmup, max(args.steps, 5), peak)

    ag_info = None
    if docs is None and not args.no_allgather and w.backward:
        ag_info = time_allgather(cpa, w, dev, stream, args.warmup, max(args.steps, 5), peak,
                                 (qs, ks, vs, dos))
    hbm_info = None
    if not args.no_hbm:
        hbm_info = time_hbm_kernels(cpa, w, dev, stream, args.warmup, max(args.steps, 5), hbm)
    ul_info = None
    if docs is None and not args.no_ulysses and w.backward:
        ul_info = time_ulysses(cpa, w, dev, stream, args.warmup, max(args.steps, 5), peak,
                               (qs, ks, vs, dos))

    hier_info = None
    if docs is None and not args.no_hier and w.backward and cp == 16:
        hier_info = time_hier(cpa, w, dev, stream, args.warmup, max(args.steps, 5), peak,
                              (qs, ks, vs, dos), (4, 4))
    named = None
    if not args.no_named:
        named = time_named_forwards(cpa, dev, stream, args.warmup, max(args.steps, 10), peak)

    path, tile = cpa.plan(B, H, Hkv, S, D, cp, layout, causal, w.dtype)
    cpu = None
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(w, q, k, v, do, budget_s=args.cpu_seconds)

    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_max, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": w.dtype_name, "data": "synthetic",
        "config": {"workload": w.name, "B": B, "S": S, "H": H, "Hkv": Hkv, "D": D, "cp": cp,
                   "layout": "zigzag" if layout == 1 else "contiguous", "causal": causal,
                   "backward": w.backward, "seed": w.seed,
                   "parallelism": "replicas" if ws > 1 else "single_gpu",
                   "l2": "inputs larger than L2 (no flush)",
                   "fwd_path": "tcgen05" if path == 1 else "simt", "tile": tile,
                   "grad_dtype": "f32" if w.backward else None,
                   "bwd_path": (args.bwd if w.backward else None),
                   "documents": None if docs is None else len(docs) - 1,
                   "useful_tflop_per_step": step_flops / 1e12},
        "e2e": e2e, "gpu_launches": launches_per_step * args.steps, "clocks": clk,
        "roofline": roofline, "kernels": fwd_info, "c3_forward": c3, "docs": docs_info,
        "allgather": ag_info, "ulysses": ul_info, "hierarchical": hier_info,
        "named_forwards": named, "hbm_kernels": hbm_info,
        "cpu_baseline": cpu,
        "status": cpa.device_status(),
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def host_link_gbs(dev, stream, mib=256, reps=3):
    """The machine's host link as the end-to-end run sees it: a pinned 256 MiB
    copy up and one down, best of `reps`, CUDA events (context for the e2e
    figure, which depends on it)."""
    h = torch.empty(mib << 20, dtype=torch.uint8, pin_memory=True)
    d = torch.empty(mib << 20, dtype=torch.uint8, device=dev)
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    res = {}
    for name, dst, src in (("h2d", d, h), ("d2h", h, d)):
        best = None
        for _ in range(reps):
            a.record(stream)
            dst.copy_(src, non_blocking=True)
            b.record(stream)
            b.synchronize()
            ms = a.elapsed_time(b)
            best = ms if best is None else min(best, ms)
        res[name] = (mib << 20) / (best * 1e-3) / 1e9
    return res


def time_hbm_kernels(cpa, w, dev, stream, warmup, steps, hbm):
    """The HBM-bound kernels alone, on tensors larger than L2: the zigzag
    permute and unpermute of a query-sized tensor of the workload, and the
    LSE merge of two float32 step partials of it.  Algorithmic bytes: one
    read and one write of the tensor (permute); two partials and two LSE
    read, one of each written (merge).  Median of `steps` launches, CUDA
    events on the launching stream."""
    x = torch.randn((w.B, w.S, w.H, w.D), device=dev, dtype=torch.float32).to(w.dtype)
    y = torch.empty_like(x)
    o_a = torch.randn((w.B, w.S, w.H, w.D), device=dev, dtype=torch.float32)
    o_b = torch.randn_like(o_a)
    l_a = torch.randn((w.B, w.H, w.S), device=dev, dtype=torch.float32)
    l_b = torch.randn_like(l_a)
    o_out, l_out = torch.empty_like(o_a), torch.empty_like(l_a)
    calls = {
        "zigzag_permute": (lambda: cpa.zigzag_permute(x, w.cp, w.layout, out=y),
                           2 * x.numel() * x.element_size()),
        "zigzag_unpermute": (lambda: cpa.zigzag_unpermute(y, w.cp, w.layout, out=x),
                             2 * x.numel() * x.element_size()),
        "lse_merge": (lambda: cpa.lse_merge(o_a, l_a, o_b, l_b, o_out, l_out),
                      3 * (o_a.numel() + l_a.numel()) * 4),
    }
    res = {}
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    for name, (fn, nbytes) in calls.items():
        for _ in range(warmup):
            fn()
        torch.cuda.synchronize(dev)
        times = []
        for _ in range(steps):
            a.record(stream)
            fn()
            b.record(stream)
            b.synchronize()
            times.append(a.elapsed_time(b))
        ms = statistics.median(times)
        gbs = nbytes / (ms * 1e-3) / 1e9
        res[name] = {"ms_median": ms, "bytes": nbytes, "GB/s": gbs, "peak": hbm,
                     "frac": gbs / hbm}
    res["status"] = cpa.device_status()
    del x, y, o_a, o_b, l_a, l_b, o_out, l_out
    torch.cuda.empty_cache()
    return res


def time_forward(cpa, w, dev, stream, warmup, steps, peak):
    q, k, v, _ = inputs.generate(w, with_dout=False)
    qd, kd, vd = (x.to(dev) for x in (q, k, v))
    qs, ks, vs = (cpa.zigzag_permute(x, w.cp, w.layout) for x in (qd, kd, vd))
    o = torch.empty_like(qs)
    lse = torch.empty((w.B, w.H, w.S), device=dev, dtype=torch.float32)
    for _ in range(warmup):
        cpa.ring_fwd(qs, ks, vs, w.cp, w.layout, w.causal, out=o, lse=lse)
    torch.cuda.synchronize(dev)
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    times = []
    for _ in range(steps):
        a.record(stream)
        cpa.ring_fwd(qs, ks, vs, w.cp, w.layout, w.causal, out=o, lse=lse)
        b.record(stream)
        b.synchronize()
        times.append(a.elapsed_time(b))
    ms = statistics.median(times)
    tf = w.useful_flops(False) / (ms * 1e-3) / 1e12
    path, tile = cpa.plan(w.B, w.H, w.Hkv, w.S, w.D, w.cp, w.layout, w.causal, w.dtype)
    # Kernel census of the same call: per-step max/mean of tiles per rank.
    counts = torch.zeros((w.cp, w.cp), device=dev, dtype=torch.int64)
    cpa.ring_fwd(qs, ks, vs, w.cp, w.layout, w.causal, out=o, lse=lse, tiles_rt=counts)
    c = counts.cpu().numpy().astype(np.float64)
    imbalance = float(np.max(c.max(axis=0) / np.maximum(c.mean(axis=0), 1)))
    return {"workload": w.name, "ms_median": ms, "ms_min": min(times), "tflops": tf,
            "frac": tf / peak, "path": "tcgen05" if path == 1 else "simt", "tile": tile,
            "zigzag_step_imbalance_max_over_mean": imbalance}


def census_balance(counts):
    """Per-step balance of a kernel census tiles[r, t]: the worst step's
    max/mean over ranks, and the lockstep efficiency sum_t mean_t / sum_t
    max_t (the share of rank-steps doing work when every step waits for its
    slowest rank)."""
    c = np.asarray(counts, dtype=np.float64)
    mx, mean = c.max(axis=0), c.mean(axis=0)
    worst = float(np.max(np.where(mean > 0, mx / np.maximum(mean, 1e-30), 1.0)))
    return {"worst_step_max_over_mean": worst, "lockstep_efficiency": float(mean.sum() / mx.sum())}


def time_named_forwards(cpa, dev, stream, warmup, steps, peak):
    """The forward of every named workload that the main line does not time:
    the S=256 float32 one, the S=8192 one in both layouts (with the kernel's
    own census of each), and the S=16384 full-attention one at every ring
    size of its sweep.  Median of `steps` calls, CUDA events on the
    launching stream, clocks sampled over the whole section."""
    gpu_id = "GPU-" + str(torch.cuda.get_device_properties(dev).uuid)
    clk = ClockSampler(gpu_id)
    clk.start()
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)

    def timed(fn):
        for _ in range(warmup):
            fn()
        torch.cuda.synchronize(dev)
        times = []
        for _ in range(steps):
            a.record(stream)
            fn()
            b.record(stream)
            b.synchronize()
            times.append(a.elapsed_time(b))
        return statistics.median(times), min(times)

    def one(w, cp, layout):
        q, k, v, _ = inputs.generate(w, with_dout=False)
        qs, ks, vs = (cpa.zigzag_permute(x.to(dev), cp, layout) for x in (q, k, v))
        o = torch.empty_like(qs)
        lse = torch.empty((w.B, w.H, w.S), device=dev, dtype=torch.float32)
        ms, ms_min = timed(lambda: cpa.ring_fwd(qs, ks, vs, cp, layout, w.causal, out=o, lse=lse))
        tf = w.useful_flops(False) / (ms * 1e-3) / 1e12
        path, tile = cpa.plan(w.B, w.H, w.Hkv, w.S, w.D, cp, layout, w.causal, w.dtype)
        res = {"cp": cp, "layout": "zigzag" if layout == cpa.ZIGZAG else "contiguous",
               "ms_median": ms, "ms_min": ms_min, "tflops": tf, "frac": tf / peak,
               "path": "tcgen05" if path == cpa.PATH_TCGEN05 else "simt", "tile": tile}
        if w.causal:
            counts = torch.zeros((cp, cp), device=dev, dtype=torch.int64)
            cpa.ring_fwd(qs, ks, vs, cp, layout, w.causal, out=o, lse=lse, tiles_rt=counts)
            res["census"] = census_balance(counts.cpu().numpy())
        return res

    out = {}
    w1 = inputs.WORKLOADS["c1_fp32_s256"]
    out[w1.name] = one(w1, w1.cp, w1.layout)
    w2 = inputs.WORKLOADS["c2_bf16_s8192"]
    out[w2.name] = {"zigzag": one(w2, w2.cp, cpa.ZIGZAG),
                    "contiguous": one(w2, w2.cp, cpa.CONTIGUOUS)}
    w4 = inputs.WORKLOADS["c4_bf16_s16384_bidir"]
    out[w4.name] = {f"cp{cp}": one(w4, cp, w4.layout) for cp in w4.cp_sweep}
    out["clocks"] = clk.stop()
    out["status"] = cpa.device_status()
    torch.cuda.empty_cache()
    return out


def time_docs(cpa, w, dev, stream, warmup, steps, peak):
    """Forward and backward of a packed-document workload, each timed alone
    (median of `steps`), in sharded order with the bounds precomputed."""
    q, k, v, do = inputs.generate(w)
    cu = w.doc_offsets()
    qs, ks, vs, dos = (cpa.zigzag_permute(x.to(dev), w.cp, w.layout) for x in (q, k, v, do))
    del q, k, v, do
    bounds = cpa.doc_bounds(cu, w.S, dev)
    o = torch.empty_like(qs)
    lse = torch.empty((w.B, w.H, w.S), device=dev, dtype=torch.float32)
    g = [torch.empty(x.shape, device=dev, dtype=torch.float32) for x in (qs, ks, vs)]
    wsp = torch.empty(cpa.ring_bwd_workspace_bytes(w.B, w.H, w.Hkv, w.S, w.D,
                                                   cpa.BF16 | cpa.GRAD_F32),
                      device=dev, dtype=torch.uint8)

    def fwd():
        cpa.ring_fwd_docs(qs, ks, vs, w.cp, bounds, w.layout, w.causal, out=o, lse=lse)

    def bwd():
        cpa.ring_bwd_docs(qs, ks, vs, o, dos, lse, w.cp, bounds, w.layout, w.causal, dq=g[0],
                          dk=g[1], dv=g[2], workspace=wsp, grad_dtype=torch.float32)

    res = {}
    for name, fn in (("fwd", fwd), ("bwd", bwd)):
        for _ in range(warmup):
            fn()
        torch.cuda.synchronize(dev)
        times = []
        for _ in range(steps):
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record(stream)
            fn()
            b.record(stream)
            b.synchronize()
            times.append(a.elapsed_time(b))
        ms = statistics.median(times)
        tf = w.useful_flops(name == "bwd") / (ms * 1e-3) / 1e12
        res[name] = {"ms_median": ms, "ms_min": min(times), "tflops": tf, "frac": tf / peak}
    full = w.S * (w.S + 1) // 2
    return {"workload": w.name, "documents": len(cu) - 1, "doc_mean": w.doc_mean,
            "useful_pairs_vs_one_document": w.valid_pairs_per_head() / full,
            "forward": res["fwd"], "backward": res["bwd"], "grad_dtype": "f32",
            "status": cpa.device_status()}


def time_allgather(cpa, w, dev, stream, warmup, steps, peak, sharded):
    """The all-gather schedule on sharded inputs: gather K/V (natural order),
    forward, backward, reduce-scatter dK/dV to sharded order; each part timed
    with CUDA events (median of `steps`)."""
    qs, ks, vs, dos = sharded
    kf, vf = torch.empty_like(ks), torch.empty_like(vs)
    o = torch.empty_like(qs)
    lse = torch.empty((w.B, w.H, w.S), device=dev, dtype=torch.float32)
    g = [torch.empty(x.shape, device=dev, dtype=torch.float32) for x in (qs, ks, vs)]
    gs = [torch.empty_like(g[1]), torch.empty_like(g[2])]
    wsp = torch.empty(cpa.ring_bwd_workspace_bytes(w.B, w.H, w.Hkv, w.S, w.D,
                                                   cpa.BF16 | cpa.GRAD_F32),
                      device=dev, dtype=torch.uint8)
    parts = {
        "gather": lambda: cpa.kv_allgather(ks, vs, w.cp, w.layout, k_full=kf, v_full=vf),
        "fwd": lambda: cpa.allgather_fwd(qs, kf, vf, w.cp, w.layout, w.causal, out=o, lse=lse),
        "bwd": lambda: cpa.allgather_bwd(qs, kf, vf, o, dos, lse, w.cp, w.layout, w.causal,
                                         dq=g[0], dk_full=g[1], dv_full=g[2], workspace=wsp,
                                         grad_dtype=torch.float32),
        "scatter": lambda: (cpa.zigzag_permute(g[1], w.cp, w.layout, out=gs[0]),
                            cpa.zigzag_permute(g[2], w.cp, w.layout, out=gs[1])),
    }
    res = {}
    for name, fn in parts.items():
        for _ in range(warmup):
            fn()
        torch.cuda.synchronize(dev)
        times = []
        for _ in range(steps):
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record(stream)
            fn()
            b.record(stream)
            b.synchronize()
            times.append(a.elapsed_time(b))
        res[name] = statistics.median(times)
    fwd_tf = w.useful_flops(False) / (res["fwd"] * 1e-3) / 1e12
    bwd_tf = w.useful_flops(True) / (res["bwd"] * 1e-3) / 1e12
    total = sum(res.values())
    return {"workload": w.name, "schedule": "all-gather K/V", "ms": res,
            "forward": {"tflops": fwd_tf, "frac": fwd_tf / peak},
            "backward": {"tflops": bwd_tf, "frac": bwd_tf / peak},
            "fwd_bwd_with_gather_scatter_tflops":
                (w.useful_flops(False) + w.useful_flops(True)) / (total * 1e-3) / 1e12,
            "grad_dtype": "f32", "status": cpa.device_status()}


def time_ulysses(cpa, w, dev, stream, warmup, steps, peak, sharded):
    """The Ulysses variant on sharded inputs, forward and backward calls (each
    includes its all-to-alls), timed with CUDA events (median of `steps`)."""
    qs, ks, vs, dos = sharded
    o = torch.empty_like(qs)
    lse = torch.empty((w.B, w.H, w.S), device=dev, dtype=torch.float32)
    g = [torch.empty(x.shape, device=dev, dtype=torch.float32) for x in (qs, ks, vs)]
    code = cpa.BF16 if w.dtype == torch.bfloat16 else cpa.F32
    wf = torch.empty(cpa.ulysses_workspace_bytes(w.B, w.H, w.Hkv, w.S, w.D, w.cp, w.layout, code,
                                                 False), device=dev, dtype=torch.uint8)
    wb = torch.empty(cpa.ulysses_workspace_bytes(w.B, w.H, w.Hkv, w.S, w.D, w.cp, w.layout,
                                                 code | cpa.GRAD_F32, True),
                     device=dev, dtype=torch.uint8)
    parts = {
        "fwd": lambda: cpa.ulysses_fwd(qs, ks, vs, w.cp, w.layout, w.causal, out=o, lse=lse,
                                       workspace=wf),
        "bwd": lambda: cpa.ulysses_bwd(qs, ks, vs, o, dos, lse, w.cp, w.layout, w.causal,
                                       dq=g[0], dk=g[1], dv=g[2], workspace=wb,
                                       grad_dtype=torch.float32),
    }
    res = {}
    for name, fn in parts.items():
        for _ in range(warmup):
            fn()
        torch.cuda.synchronize(dev)
        times = []
        for _ in range(steps):
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record(stream)
            fn()
            b.record(stream)
            b.synchronize()
            times.append(a.elapsed_time(b))
        res[name] = statistics.median(times)
    fwd_tf = w.useful_flops(False) / (res["fwd"] * 1e-3) / 1e12
    bwd_tf = w.useful_flops(True) / (res["bwd"] * 1e-3) / 1e12
    hc, nkv = cpa._binding.ulysses_heads(w.H, w.Hkv, w.cp)
    return {"workload": w.name, "schedule": "Ulysses all-to-all", "ms": res,
            "heads_per_rank": hc, "kv_heads_per_rank": nkv,
            "forward": {"tflops": fwd_tf, "frac": fwd_tf / peak},
            "backward": {"tflops": bwd_tf, "frac": bwd_tf / peak},
            "fwd_bwd_tflops": (w.useful_flops(False) + w.useful_flops(True))
            / ((res["fwd"] + res["bwd"]) * 1e-3) / 1e12,
            "grad_dtype": "f32", "status": cpa.device_status()}


def time_hier(cpa, w, dev, stream, warmup, steps, peak, sharded, split):
    """The hierarchical (a2a+p2p) schedule on sharded inputs with level sizes
    `split` = (cp_a2a, cp_p2p), forward and backward calls (each includes its
    all-to-alls), timed with CUDA events (median of `steps`)."""
    A, P = split
    qs, ks, vs, dos = sharded
    o = torch.empty_like(qs)
    lse = torch.empty((w.B, w.H, w.S), device=dev, dtype=torch.float32)
    g = [torch.empty(x.shape, device=dev, dtype=torch.float32) for x in (qs, ks, vs)]
    code = cpa.BF16 if w.dtype == torch.bfloat16 else cpa.F32
    wf = torch.empty(cpa.hier_workspace_bytes(w.B, w.H, w.Hkv, w.S, w.D, A, P, w.layout, code,
                                              False), device=dev, dtype=torch.uint8)
    wb = torch.empty(cpa.hier_workspace_bytes(w.B, w.H, w.Hkv, w.S, w.D, A, P, w.layout,
                                              code | cpa.GRAD_F32, True),
                     device=dev, dtype=torch.uint8)
    parts = {
        "fwd": lambda: cpa.hier_fwd(qs, ks, vs, A, P, w.layout, w.causal, out=o, lse=lse,
                                    workspace=wf),
        "bwd": lambda: cpa.hier_bwd(qs, ks, vs, o, dos, lse, A, P, w.layout, w.causal,
                                    dq=g[0], dk=g[1], dv=g[2], workspace=wb,
                                    grad_dtype=torch.float32),
    }
    res = {}
    for name, fn in parts.items():
        for _ in range(warmup):
            fn()
        torch.cuda.synchronize(dev)
        times = []
        for _ in range(steps):
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record(stream)
            fn()
            b.record(stream)
            b.synchronize()
            times.append(a.elapsed_time(b))
        res[name] = statistics.median(times)
    fwd_tf = w.useful_flops(False) / (res["fwd"] * 1e-3) / 1e12
    bwd_tf = w.useful_flops(True) / (res["bwd"] * 1e-3) / 1e12
    hc, nkv = cpa._binding.ulysses_heads(w.H, w.Hkv, A)
    del wf, wb, g
    torch.cuda.empty_cache()
    return {"workload": w.name, "schedule": f"hierarchical a2a+p2p [{A}, {P}]", "ms": res,
            "heads_per_member": hc, "kv_heads_per_member": nkv,
            "forward": {"tflops": fwd_tf, "frac": fwd_tf / peak},
            "backward": {"tflops": bwd_tf, "frac": bwd_tf / peak},
            "fwd_bwd_tflops": (w.useful_flops(False) + w.useful_flops(True))
            / ((res["fwd"] + res["bwd"]) * 1e-3) / 1e12,
            "grad_dtype": "f32", "status": cpa.device_status()}


# ---------------------------------------------------------------------------
# the oracle on the host cores
# ---------------------------------------------------------------------------

def oracle_sample_rows(w, n, seed):
    rng = np.random.default_rng(seed)
    b = rng.integers(0, w.B, n)
    h = rng.integers(0, w.H, n)
    i = rng.integers(0, w.S, n)
    return np.stack([b, h, i], axis=1).astype(np.int64)


def oracle_flops(w, rows, backward):
    # Visible keys per sampled row; forward 4*D per pair, plus the dQ part of
    # the backward (recompute S, dP, dQ: 6*D per pair) when timed.
    cu = w.doc_offsets()
    if cu is None:
        keys = (rows[:, 2] + 1) if w.causal else np.full(len(rows), w.S)
    else:
        cu = np.asarray(cu)
        d = np.searchsorted(cu, rows[:, 2], side="right") - 1
        keys = (rows[:, 2] - cu[d] + 1) if w.causal else (cu[d + 1] - cu[d])
    per = 4 * w.D + (6 * w.D if backward else 0)
    return float(per) * float(keys.sum())


def oracle_step(w, qf, kf, vf, dof, rows):
    import oracle
    cu = w.doc_offsets()
    if cu is None:
        oracle.attn_fwd_rows(qf, kf, vf, rows, causal=w.causal)
        if dof is not None:
            oracle.attn_bwd_dq_rows(qf, kf, vf, dof, rows, causal=w.causal)
    else:
        oracle.attn_fwd_rows_docs(qf, kf, vf, rows, cu, causal=w.causal)
        if dof is not None:
            oracle.attn_bwd_dq_rows_docs(qf, kf, vf, dof, rows, cu, causal=w.causal)


def cpu_baseline(w, q, k, v, do, budget_s=12.0, seed=0):
    import oracle
    cores = len(os.sched_getaffinity(0))
    oracle.set_threads(cores)
    qf, kf, vf = (inputs.to_f32_numpy(x) for x in (q, k, v))
    dof = inputs.to_f32_numpy(do) if do is not None else None
    # Calibrate on a few rows, then size the sample to the budget.
    n = 2 * cores
    rows = oracle_sample_rows(w, n, seed)
    t = time.perf_counter()
    oracle_step(w, qf, kf, vf, dof, rows)
    dt = time.perf_counter() - t
    n = int(max(cores, min(1 << 16, n * max(1.0, budget_s / max(dt, 1e-3)))))
    rows = oracle_sample_rows(w, n, seed + 1)
    t = time.perf_counter()
    oracle_step(w, qf, kf, vf, dof, rows)
    dt = time.perf_counter() - t
    fl = oracle_flops(w, rows, dof is not None)
    return {"value": fl / dt / 1e12, "unit": UNIT, "cores": oracle.get_threads(),
            "kind": "oracle", "seconds": dt,
            "sample": f"{n} random query rows (b, h, i) of {w.name}: fp64 forward "
                      f"definition" + (" + row-local dQ" if dof is not None else "") +
                      "; useful flops 4*D (+6*D) per visible pair"}


def run_reference(args):
    ws, rank, local = dist_env()
    if rank != 0:
        return
    import oracle
    w = ALL_WORKLOADS[args.workload]
    q, k, v, do = inputs.generate(w)
    cores = len(os.sched_getaffinity(0))
    oracle.set_threads(cores)
    qf, kf, vf = (inputs.to_f32_numpy(x) for x in (q, k, v))
    dof = inputs.to_f32_numpy(do) if do is not None else None
    # Size each step to ~budget seconds of host work.
    per_step_s = max(0.5, args.cpu_seconds / max(1, args.steps + args.warmup))
    rows = oracle_sample_rows(w, 2 * cores, 0)
    t = time.perf_counter()
    oracle_step(w, qf, kf, vf, dof, rows)
    dt = time.perf_counter() - t
    n = int(max(cores, min(1 << 16, 2 * cores * max(1.0, per_step_s / max(dt, 1e-3)))))
    for i in range(args.warmup):
        oracle_step(w, qf, kf, vf, dof, oracle_sample_rows(w, n, 100 + i))
    total_t, total_f = 0.0, 0.0
    for i in range(args.steps):
        rows = oracle_sample_rows(w, n, 1000 + i)
        t = time.perf_counter()
        oracle_step(w, qf, kf, vf, dof, rows)
        total_t += time.perf_counter() - t
        total_f += oracle_flops(w, rows, dof is not None)
    value = total_f / total_t / 1e12
    sample = (f"{n} random query rows (b, h, i) per step of {w.name}: fp64 forward definition"
              + (" + row-local dQ" if dof is not None else "") +
              "; useful flops 4*D (+6*D) per visible pair")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
            "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": total_t / args.steps * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": w.name, "B": w.B, "S": w.S, "H": w.H, "Hkv": w.Hkv,
                       "D": w.D, "cp": w.cp, "causal": w.causal, "backward": w.backward,
                       "documents": (None if w.doc_offsets() is None
                                     else len(w.doc_offsets()) - 1)},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": oracle.get_threads(),
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--workload", default="c5_bf16_s131072_fwdbwd", choices=sorted(ALL_WORKLOADS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-c3", action="store_true")
    ap.add_argument("--no-docs", action="store_true")
    ap.add_argument("--no-allgather", action="store_true")
    ap.add_argument("--no-ulysses", action="store_true")
    ap.add_argument("--no-hbm", action="store_true")
    ap.add_argument("--no-hier", action="store_true")
    ap.add_argument("--bwd", default="two", choices=["two", "onepass"],
                    help="tensor-core backward of the main step: the deterministic two-kernel "
                         "path or the one-pass kernel (CPATTN_BWD_ONEPASS)")
    ap.add_argument("--no-named", action="store_true")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
