#!/usr/bin/env python
"""Benchmark of the EAGLE-3 TTT draft-step core on GB300.

One step = the whole hot path over one batch of synthetic input: for every TTT
step k of the workload, sparse-tree attention forward and backward, then the
in-place soft-CE over the workload's logits.  Inputs are resident in HBM when
the timed region starts; every timed step consumes its own fresh copy of the
logits (the soft-CE overwrites them).

Prints ONE JSON line (rank 0).  `value` is the attention fwd+bwd useful
TFLOP/s (only unmasked score entries, 4*D flops forward and 10*D backward);
`soft_ce` carries the soft-CE's algorithmic GB/s.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload llama8b]
  python bench.py --impl reference ...   # the CPU oracle, timed on host cores
"""

from __future__ import annotations

import argparse
import csv
import hashlib
import io
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

from speculative_decoding_draft_eagle_gb300 import metrics, workloads as wl  # noqa: E402

PEAKS_FILE = os.path.join(ROOT, "MEASURED_PEAKS.json")
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "traffic.json")
CSRC = os.path.join(ROOT, "speculative_decoding_draft_eagle_gb300", "csrc")
METRIC = "TTT-attn fwd+bwd useful TFLOP/s; in-place soft-CE GB/s (1×GB300)"

# kernel id -> (source file, roofline bound)
KERNELS = {1: ("soft_ce.cu", "hbm"), 2: ("soft_ce.cu", "hbm"), 3: ("attn_fwd.cu", "tensor"),
           4: ("attn_bwd.cu", "hbm"), 5: ("attn_bwd.cu", "tensor")}


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=30)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="llama8b", choices=[n for n in wl.WORKLOADS if n != "tiny"])
    ap.add_argument("--e2e-steps", type=int, default=3)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    return ap.parse_args()


# ------------------------------------------------------------ distributed --
def dist_env():
    return int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")), int(
        os.environ.get("LOCAL_RANK", "0"))


def dist_init(backend):
    rank, world, _ = dist_env()
    if world > 1:
        import torch.distributed as dist
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        dist.init_process_group(backend=backend)
    return rank, world


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def allreduce_max(x: float, world, device) -> float:
    if world == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def allreduce_sum(x: float, world, device) -> float:
    if world == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


# ------------------------------------------------------------------ peaks --
def peaks():
    try:
        d = json.load(open(PEAKS_FILE))
        return {"hbm": float(d["hbm_gbs"]), "bf16": float(d["bf16_tflops"]),
                "bf16_sustained": float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                "src": "measured"}
    except Exception:
        return {"hbm": 6800.0, "bf16": 1900.0, "bf16_sustained": 1700.0, "src": "fallback"}


def source_hash(fname):
    h = hashlib.sha256()
    for f in (fname, "attn_common.cuh", "ptx.cuh"):
        p = os.path.join(CSRC, f)
        if os.path.exists(p):
            h.update(open(p, "rb").read())
    return h.hexdigest()[:16]


def traffic_for(kernel_name, src_file, workload):
    """DRAM bytes per launch from a committed ncu capture, if the kernel's source
    is unchanged since the capture (else None)."""
    try:
        d = json.load(open(TRAFFIC_FILE))
        e = d[workload][kernel_name]
        if e.get("source_hash") != source_hash(src_file):
            return None
        return float(e["dram_bytes_per_launch"])
    except Exception:
        return None


# ------------------------------------------------------------------ clocks --
class ClockSampler:
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self):
        self.proc = None
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.Q}", "--format=csv",
                                          "-lms", "50"], stdout=subprocess.PIPE,
                                         stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.12)
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out, _ = self.proc.communicate()
        rows = [r for r in csv.reader(io.StringIO(out)) if r and not r[0].startswith("index")]
        mhz, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            try:
                mhz.append(float(r[1].split()[0]))
                mx = float(r[2].split()[0])
                for n, v in zip(names, r[5:9]):
                    if "Active" in v and "Not" not in v:
                        reasons.add(n)
            except Exception:
                continue
        if not mhz:
            return None
        return {"sm_mhz": statistics.median(mhz), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(mhz)}


# ------------------------------------------------------------- our arm -----
def run_ours(a):
    rank, world = dist_init("nccl")
    _, _, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    from speculative_decoding_draft_eagle_gb300 import build, ops, _lib
    if rank == 0:
        build.build()
    barrier(world)
    L = _lib.lib()

    w = wl.WORKLOADS[a.workload]
    sh, sc = w.attn, w.soft_ce
    seed = w.seed + 7919 * rank  # independent problem per rank (weak scaling)
    T, Ks, Vs, qs, dOs = wl.attn_inputs(sh, dev, seed)
    z0, p, g = wl.soft_ce_inputs(sc, dev, seed, T=T, Q_LEN=sh.Q_LEN)
    n_z = a.warmup + a.steps
    zs = [torch.empty_like(z0) for _ in range(n_z)]
    for z in zs:
        z.copy_(z0)
    nb = sh.n_blocks
    out = torch.empty_like(qs[sh.steps[0]])
    lse = torch.empty((sh.B, sh.H, sh.Q_LEN), device=dev, dtype=torch.float32)
    dq = torch.empty(out.shape, device=dev, dtype=torch.float32)
    dk = [torch.empty(Ks[0].shape, device=dev, dtype=torch.float32) for _ in range(nb)]
    dv = [torch.empty(Ks[0].shape, device=dev, dtype=torch.float32) for _ in range(nb)]
    ws = torch.empty(ops.stt_attn_bwd_workspace_size(sh.B, sh.H, sh.H_kv, sh.D, sh.Q_LEN, nb - 1),
                     device=dev, dtype=torch.uint8)
    ce_ws = torch.empty(ops.soft_ce_workspace_size(sc.N, sc.V), device=dev, dtype=torch.uint8)
    loss = torch.empty(1, device=dev, dtype=torch.float32)
    row_loss = torch.empty(sc.N, device=dev, dtype=torch.float32)
    stream = torch.cuda.current_stream()

    def step(i, ev=None):
        for k in sh.steps:
            if ev is not None:
                ev["a0"][k].record(stream)
            ops.stt_attn_fwd(qs[k], Ks[: k + 1], Vs[: k + 1], T, sh.scale, out=out, lse=lse,
                             stream=stream)
            ops.stt_attn_bwd(qs[k], Ks[: k + 1], Vs[: k + 1], T, out, dOs[k], lse, sh.scale, dq=dq,
                             dk_blocks=dk[: k + 1], dv_blocks=dv[: k + 1], workspace=ws,
                             stream=stream)
            if ev is not None:
                ev["a1"][k].record(stream)
        if ev is not None:
            ev["c0"].record(stream)
        ops.soft_ce_fwd_bwd_inplace(zs[i], p, g, row_loss=row_loss, loss=loss, workspace=ce_ws,
                                    stream=stream)
        if ev is not None:
            ev["c1"].record(stream)

    for i in range(a.warmup):
        step(i)
    torch.cuda.synchronize()

    evs = [{"a0": {k: torch.cuda.Event(enable_timing=True) for k in sh.steps},
            "a1": {k: torch.cuda.Event(enable_timing=True) for k in sh.steps},
            "c0": torch.cuda.Event(enable_timing=True), "c1": torch.cuda.Event(enable_timing=True)}
           for _ in range(a.steps)]
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    launches_per_step = len(sh.steps) * 3 + 2  # fwd, bwd prep, bwd causal; soft-CE + loss sum
    cap = launches_per_step * a.steps + 16
    clk = ClockSampler() if rank == 0 else None
    time.sleep(0.1 if clk else 0)
    barrier(world)
    torch.cuda.synchronize()
    _lib.check("stt_profile_start", L.stt_profile_start(cap))
    t0.record(stream)
    for i in range(a.steps):
        step(a.warmup + i, evs[i])
    t1.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    import ctypes
    n = ctypes.c_int(0)
    ids = (ctypes.c_int * cap)()
    ms = (ctypes.c_float * cap)()
    _lib.check("stt_profile_stop", L.stt_profile_stop(ctypes.byref(n), ids, ms, cap))
    clocks = clk.stop() if clk else None
    assert ops.stt_device_error(stream) == 0

    total_ms = allreduce_max(t0.elapsed_time(t1), world, dev)
    attn_ms = sum(e["a0"][k].elapsed_time(e["a1"][k]) for e in evs for k in sh.steps)
    ce_ms = sum(e["c0"].elapsed_time(e["c1"]) for e in evs)
    attn_ms_max = allreduce_max(attn_ms, world, dev)
    ce_ms_max = allreduce_max(ce_ms, world, dev)

    ff, fb = metrics.attn_useful_flops(sh, T)
    flops_all = allreduce_sum(float(ff + fb) * a.steps, world, dev)
    ce_bytes = metrics.soft_ce_algorithmic_bytes(sc.N, sc.V, g)
    ce_bytes_all = allreduce_sum(float(ce_bytes) * a.steps, world, dev)
    value = flops_all / (attn_ms_max * 1e-3) / 1e12
    ce_gbs = ce_bytes_all / (ce_ms_max * 1e-3) / 1e9

    # per-kernel shares and the roofline of the dominant kernel
    per = {}
    for i in range(n.value):
        per.setdefault(int(ids[i]), []).append(float(ms[i]))
    pk = peaks()
    kinfo = kernel_algorithmic(sh, sc, T, g)
    kern_rows = {}
    tot_k = sum(sum(v) for v in per.values())
    for kid, v in per.items():
        name = L.stt_kernel_name(kid).decode()
        units = kinfo.get(name)
        ent = {"launches": len(v), "total_ms": round(sum(v), 4), "share": round(sum(v) / tot_k, 4)}
        if units:
            amount, unit = units
            rate = amount * a.steps / (sum(v) * 1e-3)
            ent["achieved"] = round(rate / (1e12 if unit == "TFLOP/s" else 1e9), 2)
            ent["unit"] = unit
        kern_rows[name] = ent
    dom_id = max(per, key=lambda kk: sum(per[kk]))
    dom = L.stt_kernel_name(dom_id).decode()
    src, bound = KERNELS[dom_id]
    if bound == "tensor":
        peak, unit = pk["bf16_sustained"], "TFLOP/s"
    else:
        peak, unit = pk["hbm"], "GB/s"
    achieved = kern_rows[dom].get("achieved")
    roofline = {"kernel": dom, "bound": bound, "achieved": achieved, "peak": peak, "unit": unit,
                "frac": round(achieved / peak, 4) if achieved else None,
                "traffic": traffic_for(dom, src, a.workload),
                "peak_src": pk["src"] + (" sustained" if bound == "tensor" else " copy")}

    e2e = (run_e2e(a, sh, sc, T, Ks, Vs, qs, dOs, z0, p, g, ops, dev, stream, ff + fb, world)
           if a.e2e_steps > 0 else None)

    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "TFLOP/s", "n_gpus": world,
        "steps": a.steps, "warmup": a.warmup, "ms_per_step": round(total_ms / a.steps, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": a.workload, "B": sh.B, "H": sh.H, "H_kv": sh.H_kv, "D": sh.D,
                   "Q_LEN": sh.Q_LEN, "T": T if len(T) <= 16 else f"{len(T)} values",
                   "ttt_steps": list(sh.steps), "soft_ce_N": sc.N, "soft_ce_V": sc.V,
                   "parallelism": f"replicas x{world}",
                   "l2": "inputs > L2: each step streams a fresh logits copy (> 129 MB) "
                         "through the soft-CE, flushing L2 between steps"},
        "soft_ce": {"metric": "in-place soft-CE algorithmic GB/s", "value": round(ce_gbs, 1),
                    "unit": "GB/s", "frac_of_measured_hbm": round(ce_gbs / pk["hbm"], 4),
                    "ms_per_step": round(ce_ms_max / a.steps, 4)},
        "attn_ms_per_step": round(attn_ms_max / a.steps, 4),
        "roofline": roofline,
        "kernels": kern_rows,
        # every launch of the library's kernels in the timed region (the profiler
        # records the soft-CE row kernel and its loss sum as one unit)
        "gpu_launches": launches_per_step * a.steps,
        "e2e": e2e,
        "clocks": clocks,
    }
    if rank == 0 and world == 1 and not a.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(a.workload, samples=1)
    if rank == 0:
        print(json.dumps(line), flush=True)
    barrier(world)


def kernel_algorithmic(sh, sc, T, g):
    """Algorithmic work per step of each kernel (amount, unit)."""
    D, H = sh.D, sh.H
    causal = sum(t * (t + 1) // 2 + (sh.Q_LEN - t) * t for t in T) * H * len(sh.steps)
    suffix = sum(k * t for t in T for k in sh.steps) * H
    bpe = 2
    nq = sh.B * H * sh.Q_LEN
    nkv = sh.B * sh.H_kv * sh.Q_LEN
    # rows with suffix keys (q < T): only they need q, K_j and V_j, j >= 1
    vq = sum(T) * H
    vkv = sum(T) * sh.H_kv
    prep_bytes = 0
    for k in sh.steps:
        prep_bytes += 2 * nq * D * bpe + 4 * nq + 4 * nq             # O, dO; lse; Delta
        prep_bytes += (vq * D * bpe if k > 0 else 0)                 # q
        prep_bytes += 2 * k * vkv * D * bpe                          # K_j, V_j, j >= 1
        prep_bytes += 4 * nq * D + 2 * (k + 1) * nkv * D * 4         # dq init; dK_j, dV_j
    return {
        "attn_fwd": (4 * D * (causal + suffix), "TFLOP/s"),
        "attn_bwd_causal": (10 * D * causal, "TFLOP/s"),
        "attn_bwd_prep": (prep_bytes, "GB/s"),
        "soft_ce": (metrics.soft_ce_algorithmic_bytes(sc.N, sc.V, g), "GB/s"),
    }


def run_e2e(a, sh, sc, T, Ks, Vs, qs, dOs, z0, p, g, ops, dev, stream, flops, world):
    """The same metric through the public API with HOST buffers: every step copies
    its inputs from pinned host memory and reads its results back."""
    pin = lambda t: t.detach().cpu().pin_memory()  # noqa: E731
    hK = [pin(x) for x in Ks]
    hV = [pin(x) for x in Vs]
    hq = {k: pin(qs[k]) for k in sh.steps}
    hd = {k: pin(dOs[k]) for k in sh.steps}
    hz, hp, hg = pin(z0), pin(p), pin(g)
    nb = sh.n_blocks
    dK = [torch.empty_like(x) for x in Ks]
    dV = [torch.empty_like(x) for x in Vs]
    dq_ = {k: torch.empty_like(qs[k]) for k in sh.steps}
    ddo = {k: torch.empty_like(dOs[k]) for k in sh.steps}
    dz, dp_, dg = torch.empty_like(z0), torch.empty_like(p), torch.empty_like(g)
    o_h = torch.empty(qs[sh.steps[0]].shape, dtype=torch.bfloat16).pin_memory()
    lse_h = torch.empty((sh.B, sh.H, sh.Q_LEN), dtype=torch.float32).pin_memory()
    dq_h = torch.empty(qs[sh.steps[0]].shape, dtype=torch.float32).pin_memory()
    dkv_h = [torch.empty(Ks[0].shape, dtype=torch.float32).pin_memory() for _ in range(2 * nb)]
    z_h = torch.empty(z0.shape, dtype=torch.float32).pin_memory()
    loss_h = torch.empty(1, dtype=torch.float32).pin_memory()
    h2d = sum(x.numel() * x.element_size() for x in hK + hV + list(hq.values()) + list(hd.values()))
    h2d += sum(x.numel() * x.element_size() for x in (hz, hp, hg))
    d2h = 0
    for k in sh.steps:
        d2h += o_h.numel() * 2 + lse_h.numel() * 4 + dq_h.numel() * 4 + 2 * (k + 1) * dkv_h[0].numel() * 4
    d2h += z_h.numel() * 4 + 4

    def one():
        for j in range(nb):
            dK[j].copy_(hK[j], non_blocking=True)
            dV[j].copy_(hV[j], non_blocking=True)
        for k in sh.steps:
            dq_[k].copy_(hq[k], non_blocking=True)
            ddo[k].copy_(hd[k], non_blocking=True)
        dz.copy_(hz, non_blocking=True)
        dp_.copy_(hp, non_blocking=True)
        dg.copy_(hg, non_blocking=True)
        for k in sh.steps:
            o, l = ops.stt_attn_fwd(dq_[k], dK[: k + 1], dV[: k + 1], T, sh.scale, stream=stream)
            gq, gk, gv = ops.stt_attn_bwd(dq_[k], dK[: k + 1], dV[: k + 1], T, o, ddo[k], l,
                                          sh.scale, stream=stream)
            o_h.copy_(o, non_blocking=True)
            lse_h.copy_(l, non_blocking=True)
            dq_h.copy_(gq, non_blocking=True)
            for j in range(k + 1):
                dkv_h[j].copy_(gk[j], non_blocking=True)
                dkv_h[nb + j].copy_(gv[j], non_blocking=True)
        lo, _ = ops.soft_ce_fwd_bwd_inplace(dz, dp_, dg, want_row_loss=False, stream=stream)
        z_h.copy_(dz, non_blocking=True)
        loss_h.copy_(lo, non_blocking=True)

    one()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize()
    e0.record(stream)
    for _ in range(a.e2e_steps):
        one()
    e1.record(stream)
    torch.cuda.synchronize()
    ms_ = allreduce_max(e0.elapsed_time(e1), world, dev)
    tot = allreduce_sum(float(flops) * a.e2e_steps, world, dev)
    return {"value": round(tot / (ms_ * 1e-3) / 1e12, 3), "unit": "TFLOP/s",
            "ms_per_step": round(ms_ / a.e2e_steps, 3), "h2d_bytes_per_step": int(h2d),
            "d2h_bytes_per_step": int(d2h)}


# ------------------------------------------------------ oracle on the CPU --
def cpu_baseline(workload, samples=1):
    """The fp64 oracle, as it stands, on a bounded sample of the workload: one
    query head (b=0, h=0) at the last TTT step, forward and backward, plus the
    soft-CE on 256 rows.  Returns the attention useful TFLOP/s of the sample."""
    import oracle
    w = wl.WORKLOADS[workload]
    sh, sc = w.attn, w.soft_ce
    T = wl.draw_T(sh, w.seed)
    k = sh.steps[-1]
    Kb = [wl.kv_block(sh, "K", j, "cpu", w.seed)[0, 0].float().numpy().astype(np.float64)
          for j in range(k + 1)]
    Vb = [wl.kv_block(sh, "V", j, "cpu", w.seed)[0, 0].float().numpy().astype(np.float64)
          for j in range(k + 1)]
    q = wl.step_query(sh, k, "cpu", w.seed)[0, 0].float().numpy().astype(np.float64)
    dO = wl.step_dout(sh, k, "cpu", w.seed)[0, 0].float().numpy().astype(np.float64)
    ent = metrics.useful_entries(T[0], sh.Q_LEN, k)
    flops = 14 * sh.D * ent
    t_attn = 0.0
    for _ in range(samples):
        t0 = time.perf_counter()
        O, l = oracle.attention.head_forward_keyset(q, Kb, Vb, T[0], sh.scale)
        oracle.attention.head_backward_keyset(q, Kb, Vb, T[0], sh.scale, dO, O, l)
        t_attn += time.perf_counter() - t0
    rows = 256
    g0 = torch.Generator().manual_seed(w.seed)
    z = (torch.randn((rows, sc.V), generator=g0) * sc.z_std).numpy()
    lg = torch.randn((rows, sc.V), generator=g0) * sc.p_std
    pp = torch.softmax(lg / sc.p_temp, dim=1).numpy()
    gg = np.full(rows, 1.0 / sc.N, dtype=np.float32)
    t0 = time.perf_counter()
    oracle.soft_ce.soft_ce(z, pp, gg)
    t_ce = time.perf_counter() - t0
    return {"value": round(flops * samples / t_attn / 1e12, 6), "unit": "TFLOP/s",
            "cores": os.cpu_count(), "kind": "oracle",
            "sample": f"{workload}: query head (b=0,h=0) at TTT step k={k}, T={T[0]}, fwd+bwd in fp64 "
                      f"({t_attn / samples:.2f} s); soft-CE oracle on {rows} rows of V={sc.V} "
                      f"({t_ce:.2f} s)",
            "soft_ce_gbs": round(12 * rows * sc.V / t_ce / 1e9, 4),
            "threads_note": "NumPy BLAS at its default thread count (all cores); element-wise "
                            "steps single-threaded"}


def run_reference(a):
    rank, world, _ = dist_env()
    if rank != 0:
        return
    w = wl.WORKLOADS[a.workload]
    sh = w.attn
    times = []
    cb = None
    for i in range(a.warmup + a.steps):
        t0 = time.perf_counter()
        cb = cpu_baseline(a.workload, samples=1)
        if i >= a.warmup:
            times.append(time.perf_counter() - t0)
    ms = 1e3 * sum(times) / len(times)
    line = {"impl": "reference", "metric": METRIC, "value": cb["value"], "unit": "TFLOP/s",
            "n_gpus": world, "steps": a.steps, "warmup": a.warmup, "ms_per_step": round(ms, 2),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic",
            "config": {"workload": a.workload, "B": sh.B, "H": sh.H, "H_kv": sh.H_kv, "D": sh.D,
                       "Q_LEN": sh.Q_LEN, "ttt_steps": list(sh.steps)},
            "cpu_baseline": cb,
            "e2e": {"value": cb["value"], "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    a = parse()
    if a.impl == "reference":
        run_reference(a)
    else:
        run_ours(a)


if __name__ == "__main__":
    main()
