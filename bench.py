#!/usr/bin/env python
"""Benchmark of the EAGLE-3 TTT draft-step core on GB300.

One step = the whole hot path over one batch of synthetic input: for every TTT
step k of the workload, sparse-tree attention forward and backward, then the
in-place soft-CE over the workload's logits.  Inputs are resident in HBM when
the timed region starts; every timed step consumes its own fresh copy of the
logits (the soft-CE overwrites them), refilled outside the timed region.

Prints ONE JSON line (rank 0).  `value` is the attention fwd+bwd useful
TFLOP/s (only unmasked score entries, 4*D flops forward and 10*D backward) of
the headline workload (long_ttt: B1 H32 Hkv8 D128 Q_LEN 8192, TTT steps
0..12, the largest single-GPU workload); `soft_ce` carries the soft-CE's
algorithmic GB/s; `other_workloads` the same figures for the other full-size
workloads (fewer steps).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload long_ttt]
  python bench.py --impl reference ...   # the CPU oracle, timed on host cores
"""

from __future__ import annotations

import argparse
import dataclasses
import csv
import hashlib
import io
import json
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
HEADLINE = "long_ttt"
Z_BUDGET = 40e9  # bytes of device memory for fresh logits copies

# kernel name -> (source file, roofline bound)
KERNELS = {"soft_ce": ("soft_ce.cu", "hbm"), "attn_fwd": ("attn_fwd.cu", "tensor"),
           "attn_bwd_prep": ("attn_bwd.cu", "hbm"), "attn_bwd_causal": ("attn_bwd.cu", "tensor")}


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=HEADLINE, choices=[n for n in wl.WORKLOADS if n != "tiny"])
    ap.add_argument("--e2e-steps", type=int, default=6)
    ap.add_argument("--copy-streams", type=int, default=2,
                    help="e2e: copy streams per direction (pieces of <= 64 MB alternate them)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-other-workloads", action="store_true")
    ap.add_argument("--other-steps", type=int, default=5)
    ap.add_argument("--no-extras", action="store_true")
    ap.add_argument("--profile", choices=["attn", "lm_head", "verify", "soft_ce"], default=None,
                    help="small profiling case (a few GB): 2 calls of one row and exit")
    ap.add_argument("--profile-step", type=int, default=None,
                    help="with --profile attn: the TTT step (default: the workload's last)")
    a = ap.parse_args()
    if a.warmup < 0 or a.steps < 1:
        ap.error("--steps must be >= 1 and --warmup >= 0")
    return a


# ------------------------------------------------------------ distributed --
def dist_env():
    return int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")), int(
        os.environ.get("LOCAL_RANK", "0"))


def check_world(a):
    _, world, _ = dist_env()
    if a.gpus != world:
        raise SystemExit(f"--gpus {a.gpus} but WORLD_SIZE={world}: launch N > 1 with "
                         f"torch.distributed.run --nproc-per-node {a.gpus}")


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


def allreduce(x: float, world, device, op) -> float:
    if world == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX if op == "max" else dist.ReduceOp.SUM)
    return float(t.item())


# ------------------------------------------------------------------ peaks --
def peaks():
    try:
        d = json.load(open(PEAKS_FILE))
        return {"hbm": float(d["hbm_gbs"]), "bf16": float(d["bf16_tflops"]), "src": "measured"}
    except Exception:
        return {"hbm": 6800.0, "bf16": 1900.0, "src": "fallback"}


def source_hash(fname):
    h = hashlib.sha256()
    for f in (fname, "attn_common.cuh", "ptx.cuh"):
        p = os.path.join(CSRC, f)
        if os.path.exists(p):
            h.update(open(p, "rb").read())
    return h.hexdigest()[:16]


def traffic_for(kernel_name, workload):
    """DRAM bytes per launch from a committed ncu capture, if the kernel's source
    is unchanged since the capture (else None)."""
    try:
        e = json.load(open(TRAFFIC_FILE))[workload][kernel_name]
        if e.get("source_hash") != source_hash(KERNELS[kernel_name][0]):
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
class Workbench:
    """Device-resident inputs and outputs of one workload, and one step of the path."""

    def __init__(self, name, dev, seed, n_steps):
        from speculative_decoding_draft_eagle_gb300 import ops
        self.ops = ops
        self.name = name
        w = wl.WORKLOADS[name]
        self.sh, self.sc = sh, sc = w.attn, w.soft_ce
        self.T, self.Ks, self.Vs, self.qs, self.dOs = wl.attn_inputs(sh, dev, seed)
        self.z0, self.p, self.g = wl.soft_ce_inputs(sc, dev, seed, T=self.T, Q_LEN=sh.Q_LEN)
        zbytes = self.z0.numel() * 4
        self.R = int(max(1, min(n_steps, Z_BUDGET // zbytes)))
        self.zs = [torch.empty_like(self.z0) for _ in range(self.R)]
        nb = sh.n_blocks
        self.out = torch.empty_like(self.qs[sh.steps[0]])
        self.lse = torch.empty((sh.B, sh.H, sh.Q_LEN), device=dev, dtype=torch.float32)
        self.dq = torch.empty(self.out.shape, device=dev, dtype=torch.float32)
        self.dk = [torch.empty(self.Ks[0].shape, device=dev, dtype=torch.float32) for _ in range(nb)]
        self.dv = [torch.empty(self.Ks[0].shape, device=dev, dtype=torch.float32) for _ in range(nb)]
        self.ws = torch.empty(ops.stt_attn_bwd_workspace_size(sh.B, sh.H, sh.H_kv, sh.D, sh.Q_LEN,
                                                              nb - 1), device=dev, dtype=torch.uint8)
        self.ce_ws = torch.empty(ops.soft_ce_workspace_size(sc.N, sc.V), device=dev, dtype=torch.uint8)
        self.loss = torch.empty(1, device=dev, dtype=torch.float32)
        self.row_loss = torch.empty(sc.N, device=dev, dtype=torch.float32)
        self.launches_per_step = len(sh.steps) * 3 + 2  # fwd, prep, causal; soft-CE row + loss sum

    def refill(self):
        for z in self.zs:
            z.copy_(self.z0)

    def step(self, i, stream, ev=None):
        sh, ops = self.sh, self.ops
        for k in sh.steps:
            if ev is not None:
                ev["a0"][k].record(stream)
            ops.stt_attn_fwd(self.qs[k], self.Ks[: k + 1], self.Vs[: k + 1], self.T, sh.scale,
                             out=self.out, lse=self.lse, stream=stream)
            ops.stt_attn_bwd(self.qs[k], self.Ks[: k + 1], self.Vs[: k + 1], self.T, self.out,
                             self.dOs[k], self.lse, sh.scale, dq=self.dq,
                             dk_blocks=self.dk[: k + 1], dv_blocks=self.dv[: k + 1],
                             workspace=self.ws, stream=stream)
            if ev is not None:
                ev["a1"][k].record(stream)
        if ev is not None:
            ev["c0"].record(stream)
        ops.soft_ce_fwd_bwd_inplace(self.zs[i], self.p, self.g, row_loss=self.row_loss,
                                    loss=self.loss, workspace=self.ce_ws, stream=stream)
        if ev is not None:
            ev["c1"].record(stream)

    def kernel_work(self):
        """Algorithmic work per step of each kernel (amount, unit)."""
        sh, sc, T = self.sh, self.sc, self.T
        D, H = sh.D, sh.H
        causal = sum(t * (t + 1) // 2 + (sh.Q_LEN - t) * t for t in T) * H * len(sh.steps)
        suffix = sum(k * t for t in T for k in sh.steps) * H
        nq = sh.B * H * sh.Q_LEN
        nkv = sh.B * sh.H_kv * sh.Q_LEN
        vq = sum(T) * H          # query rows with suffix keys (q < T)
        vkv = sum(T) * sh.H_kv
        prep = 0
        for k in sh.steps:
            prep += 2 * nq * D * 2 + 4 * nq + 4 * nq              # O, dO; lse; Delta
            prep += (vq * D * 2 if k > 0 else 0)                  # q
            prep += 2 * k * vkv * D * 2                           # K_j, V_j, j >= 1
            prep += 4 * nq * D + 2 * (k + 1) * nkv * D * 4        # dq init; dK_j, dV_j
        return {
            "attn_fwd": (4 * D * (causal + suffix), "TFLOP/s"),
            "attn_bwd_causal": (10 * D * causal, "TFLOP/s"),
            "attn_bwd_prep": (prep, "GB/s"),
            "soft_ce": (metrics.soft_ce_algorithmic_bytes(sc.N, sc.V, self.g), "GB/s"),
        }


def timed_run(wb, steps, warmup, stream, L, _lib, clocks=False):
    """W warm-up steps, then exactly `steps` timed steps in segments of at most
    wb.R steps (the logits copies are refilled between segments, outside the
    timed region).  Returns device-event times and the per-launch profile."""
    import ctypes
    sh = wb.sh
    done = 0
    while done < warmup:
        wb.refill()
        n = min(wb.R, warmup - done)
        for i in range(n):
            wb.step(i, stream)
        done += n
    torch.cuda.synchronize()
    evs = [{"a0": {k: torch.cuda.Event(enable_timing=True) for k in sh.steps},
            "a1": {k: torch.cuda.Event(enable_timing=True) for k in sh.steps},
            "c0": torch.cuda.Event(enable_timing=True), "c1": torch.cuda.Event(enable_timing=True)}
           for _ in range(steps)]
    cap = wb.launches_per_step * steps + 16
    clk = ClockSampler() if clocks else None
    if clk:
        time.sleep(0.1)
    seg_ms = 0.0
    _lib.check("stt_profile_start", L.stt_profile_start(cap))
    done = 0
    while done < steps:
        wb.refill()
        torch.cuda.synchronize()
        n = min(wb.R, steps - done)
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t0.record(stream)
        for i in range(n):
            wb.step(i, stream, evs[done + i])
        t1.record(stream)
        torch.cuda.synchronize()
        seg_ms += t0.elapsed_time(t1)
        done += n
    n_rec = ctypes.c_int(0)
    ids = (ctypes.c_int * cap)()
    ms = (ctypes.c_float * cap)()
    _lib.check("stt_profile_stop", L.stt_profile_stop(ctypes.byref(n_rec), ids, ms, cap))
    clocks_rec = clk.stop() if clk else None
    attn_ms = sum(e["a0"][k].elapsed_time(e["a1"][k]) for e in evs for k in sh.steps)
    ce_ms = sum(e["c0"].elapsed_time(e["c1"]) for e in evs)
    per = {}
    for i in range(n_rec.value):
        per.setdefault(L.stt_kernel_name(int(ids[i])).decode(), []).append(float(ms[i]))
    return {"total_ms": seg_ms, "attn_ms": attn_ms, "ce_ms": ce_ms, "per": per,
            "launches": n_rec.value, "clocks": clocks_rec}


def kernel_rows(wb, per, steps, pk):
    rows = {}
    tot = sum(sum(v) for v in per.values())
    work = wb.kernel_work()
    for name, v in per.items():
        ent = {"launches": len(v), "total_ms": round(sum(v), 4), "share": round(sum(v) / tot, 4)}
        if name in work:
            amount, unit = work[name]
            rate = amount * steps / (sum(v) * 1e-3)
            ach = rate / (1e12 if unit == "TFLOP/s" else 1e9)
            peak = pk["bf16"] if unit == "TFLOP/s" else pk["hbm"]
            ent.update({"achieved": round(ach, 2), "unit": unit, "peak": peak,
                        "frac": round(ach / peak, 4)})
        rows[name] = ent
    return rows


def run_ours(a):
    check_world(a)
    rank, world = dist_init("nccl")
    _, _, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    from speculative_decoding_draft_eagle_gb300 import build, ops, _lib
    if rank == 0:
        build.build()
    barrier(world)
    L = _lib.lib()
    stream = torch.cuda.current_stream()
    pk = peaks()

    name = a.workload
    seed = wl.WORKLOADS[name].seed + 7919 * rank  # an independent problem per rank (weak scaling)
    wb = Workbench(name, dev, seed, a.warmup + a.steps)
    T = wb.T
    launches = wb.launches_per_step * a.steps
    barrier(world)
    torch.cuda.synchronize()
    r = timed_run(wb, a.steps, a.warmup, stream, L, _lib, clocks=(rank == 0))
    barrier(world)
    assert ops.stt_device_error(stream) == 0
    sh, sc = wb.sh, wb.sc

    total_ms = allreduce(r["total_ms"], world, dev, "max")
    attn_ms = allreduce(r["attn_ms"], world, dev, "max")
    ce_ms = allreduce(r["ce_ms"], world, dev, "max")
    ff, fb = metrics.attn_useful_flops(sh, wb.T)
    flops_all = allreduce(float(ff + fb) * a.steps, world, dev, "sum")
    ce_bytes = metrics.soft_ce_algorithmic_bytes(sc.N, sc.V, wb.g)
    ce_all = allreduce(float(ce_bytes) * a.steps, world, dev, "sum")
    value = flops_all / (attn_ms * 1e-3) / 1e12
    ce_gbs = ce_all / (ce_ms * 1e-3) / 1e9

    krows = kernel_rows(wb, r["per"], a.steps, pk)
    dom = max(r["per"], key=lambda kk: sum(r["per"][kk]))
    bound = KERNELS[dom][1]
    d = krows[dom]
    roofline = {"kernel": dom, "bound": bound, "achieved": d.get("achieved"), "peak": d.get("peak"),
                "unit": d.get("unit"), "frac": d.get("frac"), "traffic": traffic_for(dom, name),
                "peak_src": pk["src"] + (" bf16 dense burst (kernel timed alone, seconds-short "
                                         "timed region at max SM clock)" if bound == "tensor"
                                         else " HBM copy bandwidth")}

    e2e = (run_e2e(a, wb, dev, stream, ff + fb, world) if a.e2e_steps > 0 else None)

    others = {}
    if not a.no_other_workloads:
        del wb
        torch.cuda.empty_cache()
        for on in ("llama8b", "varlen", "llama70b", "long_ttt"):
            if on == name:
                continue
            ob = Workbench(on, dev, wl.WORKLOADS[on].seed + 7919 * rank, 3 + a.other_steps)
            ro = timed_run(ob, a.other_steps, 3, stream, L, _lib)
            assert ops.stt_device_error(stream) == 0
            off, ofb = metrics.attn_useful_flops(ob.sh, ob.T)
            o_attn = allreduce(ro["attn_ms"], world, dev, "max")
            o_ce = allreduce(ro["ce_ms"], world, dev, "max")
            o_fl = allreduce(float(off + ofb) * a.other_steps, world, dev, "sum")
            o_cb = allreduce(float(metrics.soft_ce_algorithmic_bytes(ob.sc.N, ob.sc.V, ob.g))
                             * a.other_steps, world, dev, "sum")
            kr = kernel_rows(ob, ro["per"], a.other_steps, pk)
            others[on] = {"steps": a.other_steps, "warmup": 3,
                          "attn_tflops": round(o_fl / (o_attn * 1e-3) / 1e12, 2),
                          "attn_frac_of_bf16_burst": round(o_fl / (o_attn * 1e-3) / 1e12 / pk["bf16"], 4),
                          "soft_ce_gbs": round(o_cb / (o_ce * 1e-3) / 1e9, 1),
                          "kernels": {kn: {x: kv[x] for x in ("achieved", "unit", "frac", "share")
                                           if x in kv} for kn, kv in kr.items()}}
            del ob
            torch.cuda.empty_cache()

    extras = None
    if not a.no_extras:
        extras = measure_extras(dev, stream, pk, ops)
        assert ops.stt_device_error(stream) == 0

    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "TFLOP/s", "n_gpus": world,
        "steps": a.steps, "warmup": a.warmup, "ms_per_step": round(total_ms / a.steps, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": name, "B": sh.B, "H": sh.H, "H_kv": sh.H_kv, "D": sh.D,
                   "Q_LEN": sh.Q_LEN, "T": T if len(T) <= 16 else f"{len(T)} values in [{min(T)}, {max(T)}]", "ttt_steps": list(sh.steps),
                   "soft_ce_N": sc.N, "soft_ce_V": sc.V, "parallelism": f"replicas x{world}",
                   "l2": "inputs > L2: each step streams a fresh logits copy (> 129 MB) "
                         "through the soft-CE, flushing L2 between steps"},
        "attn_frac_of_bf16_burst": round(value / pk["bf16"], 4),
        "soft_ce": {"metric": "in-place soft-CE algorithmic GB/s", "value": round(ce_gbs, 1),
                    "unit": "GB/s", "frac_of_measured_hbm": round(ce_gbs / pk["hbm"], 4),
                    "ms_per_step": round(ce_ms / a.steps, 4)},
        "attn_ms_per_step": round(attn_ms / a.steps, 4),
        "roofline": roofline,
        "kernels": krows,
        # every launch of the library's kernels in the timed region (the profiler
        # records the soft-CE row kernel and its loss sum as one unit)
        "gpu_launches": launches,
        "gpu_launches_recorded": r["launches"],
        "e2e": e2e,
        "clocks": r["clocks"],
        "other_workloads": others or None,
        "extras": extras,
    }
    if rank == 0 and world == 1 and not a.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(name)
    if rank == 0:
        print(json.dumps(line), flush=True)
    barrier(world)


def _time_calls(fn, n, warmup, stream, before=None):
    """Device time (ms) of n calls of fn(i) after `warmup` untimed ones; before(i),
    if given, runs outside the timed events (input refill, L2 flush)."""
    for i in range(warmup):
        if before:
            before(i)
        fn(i)
    torch.cuda.synchronize()
    tot = 0.0
    for i in range(n):
        if before:
            before(warmup + i)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        fn(warmup + i)
        e1.record(stream)
        torch.cuda.synchronize()
        tot += e0.elapsed_time(e1)
    return tot


def measure_extras(dev, stream, pk, ops, steps=10, warmup=3):
    """The rows beyond the attention + soft-CE step, each timed alone with CUDA
    events (inputs larger than L2, or L2 flushed between calls)."""
    out = {}
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)  # > L2 (129 MB)

    # fused draft LM head + soft-CE (Llama-8B draft shape)
    ls = wl.LM_HEAD
    h, W, p, g = wl.lm_head_inputs(ls, dev, 1002)
    dh = torch.empty((ls.N, ls.Hd), device=dev)
    dW = torch.empty((ls.V, ls.Hd), device=dev)
    rl = torch.empty(ls.N, device=dev)
    lo = torch.empty(1, device=dev)
    ws = torch.empty(int(ops.lib().stt_lm_head_ce_workspace_size(ls.N, ls.Hd, ls.V)),
                     device=dev, dtype=torch.uint8)
    ms = _time_calls(lambda i: ops.stt_lm_head_ce(h, W, p, g, dh=dh, dW=dW, row_loss=rl, loss=lo,
                                                  workspace=ws, stream=stream),
                     steps, warmup, stream) / steps
    fl = 4 * 2.0 * ls.N * ls.V * ls.Hd  # z (twice: statistics, then per chunk), dh, dW
    ach = fl / (ms * 1e-3) / 1e12
    out["lm_head_ce"] = {"workload": f"N {ls.N}, Hd {ls.Hd}, V {ls.V} (Llama-3.1-8B draft head)",
                         "ms_per_call": round(ms, 4), "achieved": round(ach, 1), "unit": "TFLOP/s",
                         "flops_counted": "4 GEMMs of 2 N V Hd: z for the statistics, z again "
                                          "per chunk for dz, dh = dz W, dW = dz^T h",
                         "peak": pk["bf16"], "frac": round(ach / pk["bf16"], 4),
                         "logits_bytes_avoided": int(ls.N * ls.V * 4)}
    del h, W, p, g, dh, dW, ws
    torch.cuda.empty_cache()

    # rejection-sampling verification
    vs = wl.VERIFY
    p_t, p_d, toks, ua, us = wl.verify_inputs(vs, dev, 1006)
    n_acc = torch.empty(vs.B, device=dev, dtype=torch.int32)
    o_t = torch.empty((vs.B, vs.gamma), device=dev, dtype=torch.int32)
    ops.stt_verify(p_t, p_d, toks, ua, us, n_accepted=n_acc, out_tokens=o_t, stream=stream)
    torch.cuda.synchronize()
    na = n_acc.cpu()
    rejected = int((na < vs.gamma).sum())
    tested = int(torch.clamp(na + 1, max=vs.gamma).sum())
    vbytes = tested * 8 + rejected * 2 * vs.V * 4 + vs.B * (vs.gamma * 12 + 8)
    ms = _time_calls(lambda i: ops.stt_verify(p_t, p_d, toks, ua, us, n_accepted=n_acc,
                                              out_tokens=o_t, stream=stream),
                     steps, warmup, stream, before=lambda i: flush.fill_(i & 255)) / steps
    out["verify"] = {"workload": f"B {vs.B}, gamma {vs.gamma}, V {vs.V}; {rejected} sequences "
                                 f"with a rejection, mean accepted {float(na.float().mean()):.2f}",
                     "ms_per_call": round(ms, 5), "sequences_per_s": round(vs.B / (ms * 1e-3)),
                     "achieved": round(vbytes / (ms * 1e-3) / 1e9, 1), "unit": "GB/s",
                     "algorithmic_bytes": vbytes, "peak": pk["hbm"],
                     "frac": round(vbytes / (ms * 1e-3) / 1e9 / pk["hbm"], 4),
                     "l2": "flushed (256 MB write) before every call"}
    del p_t, p_d, toks, ua, us
    torch.cuda.empty_cache()

    # soft-CE variants on the Llama-8B soft-CE shape
    sc = wl.WORKLOADS["llama8b"].soft_ce
    z0, pp, g = wl.soft_ce_inputs(sc, dev, 1002)
    gr = torch.Generator(device=dev).manual_seed(5)
    G = (torch.rand(z0.shape, generator=gr, device=dev) < 0.8).float() / sc.N
    nz = int((g != 0).sum())
    for tag, zdt, gel in (("bf16_z_p", torch.bfloat16, False), ("per_element_g", torch.float32, True)):
        zb = z0.to(zdt)
        pb = pp.to(zdt)
        gg = G if gel else g
        R = 4
        zs = [torch.empty_like(zb) for _ in range(R)]
        wsc = torch.empty(ops.soft_ce_workspace_size(sc.N, sc.V), device=dev, dtype=torch.uint8)
        lo = torch.empty(1, device=dev)
        rl = torch.empty(sc.N, device=dev)

        def refill(i, zs=zs, zb=zb):
            zs[i % R].copy_(zb)

        ms = _time_calls(lambda i, zs=zs, pb=pb, gg=gg: ops.soft_ce_fwd_bwd_inplace_ex(
            zs[i % R], pb, gg, row_loss=rl, loss=lo, workspace=wsc, stream=stream),
            steps, warmup, stream, before=refill) / steps
        es = zb.element_size()
        if gel:
            vb = sc.N * sc.V * (3 * es + 4) + 8 * sc.N
        else:
            vb = nz * sc.V * 3 * es + (sc.N - nz) * sc.V * es + 8 * sc.N
        ach = vb / (ms * 1e-3) / 1e9
        out[f"soft_ce_{tag}"] = {"workload": f"N {sc.N}, V {sc.V}", "ms_per_call": round(ms, 4),
                                 "achieved": round(ach, 1), "unit": "GB/s",
                                 "peak": pk["hbm"], "frac": round(ach / pk["hbm"], 4)}
        del zs, zb, pb
    del z0, pp, g, G, flush
    torch.cuda.empty_cache()
    return out


def run_e2e(a, wb, dev, stream, flops, world):
    """The same metric through the public API with HOST buffers: every step copies
    all its inputs from pinned host memory and reads all its results back (O,
    lse, dq, dK_j and dV_j of every TTT step, the soft-CE gradient and loss).

    Arranged as a user streaming batches from host memory would: copies run on
    --copy-streams streams per direction in pieces of at most 64 MB, so that
    several copy engines work in both directions at once; the attention's inputs
    go first and its results leave while the soft-CE's inputs (the largest) are
    still coming in (the reverse order measured 143 against 108 ms per long_ttt
    step); each TTT step's kernels wait only for that step's inputs, and its
    results leave while the later steps compute.  Consecutive steps use two sets
    of device buffers, so a step's copies in overlap the previous step's copies
    out; a step's copies in wait only for the step before the previous one (the
    last user of its set) to be done."""
    ops, sh = wb.ops, wb.sh
    pin = lambda t: t.detach().cpu().pin_memory()  # noqa: E731
    nb = sh.n_blocks
    steps = list(sh.steps)
    # host inputs (pinned, read by every step)
    hK = [pin(x) for x in wb.Ks]
    hV = [pin(x) for x in wb.Vs]
    hq = {k: pin(wb.qs[k]) for k in steps}
    hd = {k: pin(wb.dOs[k]) for k in steps}
    hz, hp, hg = pin(wb.z0), pin(wb.p), pin(wb.g)

    def device_set():
        """Device inputs and results of one step."""
        d = {"K": [torch.empty_like(x) for x in wb.Ks], "V": [torch.empty_like(x) for x in wb.Vs],
             "q": {k: torch.empty_like(wb.qs[k]) for k in steps},
             "dO": {k: torch.empty_like(wb.dOs[k]) for k in steps},
             "z": torch.empty_like(wb.z0), "p": torch.empty_like(wb.p), "g": torch.empty_like(wb.g),
             "o": {k: torch.empty_like(wb.out) for k in steps},
             "lse": {k: torch.empty((sh.B, sh.H, sh.Q_LEN), device=dev, dtype=torch.float32)
                     for k in steps},
             "gq": {k: torch.empty(wb.out.shape, device=dev, dtype=torch.float32) for k in steps},
             "gk": {k: [torch.empty(wb.Ks[0].shape, device=dev, dtype=torch.float32)
                        for _ in range(k + 1)] for k in steps},
             "gv": {k: [torch.empty(wb.Ks[0].shape, device=dev, dtype=torch.float32)
                        for _ in range(k + 1)] for k in steps},
             "loss": torch.empty(1, device=dev, dtype=torch.float32)}
        return d

    sets = [device_set(), device_set()]
    ws = torch.empty(ops.stt_attn_bwd_workspace_size(sh.B, sh.H, sh.H_kv, sh.D, sh.Q_LEN, max(steps)),
                     device=dev, dtype=torch.uint8)
    ce_ws = torch.empty(ops.soft_ce_workspace_size(*wb.z0.shape), device=dev, dtype=torch.uint8)
    ns = max(1, a.copy_streams)
    # pinned host results: per copy-out stream (a stream's copies are ordered),
    # and the soft-CE gradient per device set (its pieces alternate streams)
    o_h = [torch.empty(wb.out.shape, dtype=torch.bfloat16).pin_memory() for _ in range(ns)]
    lse_h = [torch.empty((sh.B, sh.H, sh.Q_LEN), dtype=torch.float32).pin_memory() for _ in range(ns)]
    dq_h = [torch.empty(wb.out.shape, dtype=torch.float32).pin_memory() for _ in range(ns)]
    dkv_h = [[torch.empty(wb.Ks[0].shape, dtype=torch.float32).pin_memory() for _ in range(2 * nb)]
             for _ in range(ns)]
    z_h = [torch.empty(wb.z0.shape, dtype=torch.float32).pin_memory() for _ in range(2)]
    loss_h = [torch.empty(1, dtype=torch.float32).pin_memory() for _ in range(2)]
    h2d = sum(x.numel() * x.element_size() for x in hK + hV + list(hq.values()) + list(hd.values()))
    h2d += sum(x.numel() * x.element_size() for x in (hz, hp, hg))
    d2h = 0
    for k in steps:
        d2h += o_h[0].numel() * 2 + lse_h[0].numel() * 4 + dq_h[0].numel() * 4
        d2h += 2 * (k + 1) * dkv_h[0][0].numel() * 4
    d2h += z_h[0].numel() * 4 + 4

    s_in = [torch.cuda.Stream(device=dev) for _ in range(ns)]
    s_out = [torch.cuda.Stream(device=dev) for _ in range(ns)]
    s_join = torch.cuda.Stream(device=dev)
    piece = 64 << 20
    turn = {"in": 0, "out": 0}

    def copy(dst, src, kind):
        """dst <- src in pieces of at most 64 MB, alternating the kind's streams."""
        ss = s_in if kind == "in" else s_out
        fd, fs = dst.view(-1), src.view(-1)
        step = max(1, piece // src.element_size())
        for i in range(0, fs.numel(), step):
            st = ss[turn[kind]]
            turn[kind] = (turn[kind] + 1) % len(ss)
            with torch.cuda.stream(st):
                fd[i:i + step].copy_(fs[i:i + step], non_blocking=True)

    def mark(ss):
        """An event per stream of a pair, for a consumer to wait on both."""
        evs = []
        for st in ss:
            e = torch.cuda.Event()
            e.record(st)
            evs.append(e)
        return evs

    def wait(st, evs):
        for e in evs:
            st.wait_event(e)

    def one(n, set_free):
        """Step n on device set n % 2; set_free: the event after which the set's
        previous step is done with it (None: free)."""
        d = sets[n % 2]
        if set_free is not None:
            for st in s_in:
                st.wait_event(set_free)
        ready = {}
        blocks_in = 0
        for k in steps:
            while blocks_in <= k:   # the blocks this step sees, first time needed
                copy(d["K"][blocks_in], hK[blocks_in], "in")
                copy(d["V"][blocks_in], hV[blocks_in], "in")
                blocks_in += 1
            copy(d["q"][k], hq[k], "in")
            copy(d["dO"][k], hd[k], "in")
            ready[k] = mark(s_in)
        copy(d["z"], hz, "in")
        copy(d["p"], hp, "in")
        copy(d["g"], hg, "in")
        ce_ready = mark(s_in)
        for i, k in enumerate(steps):
            wait(stream, ready[k])
            o, l = ops.stt_attn_fwd(d["q"][k], d["K"][: k + 1], d["V"][: k + 1], wb.T, sh.scale,
                                    out=d["o"][k], lse=d["lse"][k], stream=stream)
            ops.stt_attn_bwd(d["q"][k], d["K"][: k + 1], d["V"][: k + 1], wb.T, o, d["dO"][k], l,
                             sh.scale, dq=d["gq"][k], dk_blocks=d["gk"][k], dv_blocks=d["gv"][k],
                             workspace=ws, stream=stream)
            done = torch.cuda.Event()
            done.record(stream)
            so = s_out[i % ns]   # each copy-out stream reuses only its own host buffers
            so.wait_event(done)
            with torch.cuda.stream(so):
                hb = i % ns
                o_h[hb].copy_(d["o"][k], non_blocking=True)
                lse_h[hb].copy_(d["lse"][k], non_blocking=True)
                dq_h[hb].copy_(d["gq"][k], non_blocking=True)
                for j in range(k + 1):
                    dkv_h[hb][j].copy_(d["gk"][k][j], non_blocking=True)
                    dkv_h[hb][nb + j].copy_(d["gv"][k][j], non_blocking=True)
        wait(stream, ce_ready)
        ops.soft_ce_fwd_bwd_inplace(d["z"], d["p"], d["g"], loss=d["loss"], workspace=ce_ws,
                                    want_row_loss=False, stream=stream)
        ce_done = torch.cuda.Event()
        ce_done.record(stream)
        for st in s_out:
            st.wait_event(ce_done)
        copy(z_h[n % 2], d["z"], "out")
        with torch.cuda.stream(s_out[0]):
            loss_h[n % 2].copy_(d["loss"], non_blocking=True)
        # the step ends when every copy out has landed (recorded on a stream of
        # its own, so the next step's kernels need not wait for these copies)
        wait(s_join, mark(s_out))
        end = torch.cuda.Event()
        end.record(s_join)
        return end

    one(0, None)  # untimed: first touch of every buffer
    one(1, None)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize()
    e0.record(stream)
    ends = [e0, e0]
    for n in range(a.e2e_steps):
        ends[n % 2] = one(n, ends[n % 2])
    wait(stream, [ends[(a.e2e_steps - 1) % 2], ends[a.e2e_steps % 2]])
    e1.record(stream)
    torch.cuda.synchronize()
    ms_ = allreduce(e0.elapsed_time(e1), world, dev, "max")
    tot = allreduce(float(flops) * a.e2e_steps, world, dev, "sum")
    return {"value": round(tot / (ms_ * 1e-3) / 1e12, 3), "unit": "TFLOP/s",
            "ms_per_step": round(ms_ / a.e2e_steps, 3), "h2d_bytes_per_step": int(h2d),
            "d2h_bytes_per_step": int(d2h), "copy_streams_per_direction": ns,
            "device_buffer_sets": 2}


# ------------------------------------------------------ oracle on the CPU --
def _oracle_head_task(workload, b, h, k):
    """Oracle forward + backward of one query head at TTT step k (inputs drawn
    with the workload's CPU generator); returns the seconds the oracle took."""
    import oracle
    w = wl.WORKLOADS[workload]
    sh = w.attn
    T = wl.draw_T(sh, w.seed)
    g = h // (sh.H // sh.H_kv)
    f = lambda t: t.float().numpy().astype(np.float64)  # noqa: E731
    Kb = [f(wl.kv_block(sh, "K", j, "cpu", w.seed)[b, g]) for j in range(k + 1)]
    Vb = [f(wl.kv_block(sh, "V", j, "cpu", w.seed)[b, g]) for j in range(k + 1)]
    q = f(wl.step_query(sh, k, "cpu", w.seed)[b, h])
    dO = f(wl.step_dout(sh, k, "cpu", w.seed)[b, h])
    t0 = time.perf_counter()
    O, l = oracle.attention.head_forward_keyset(q, Kb, Vb, T[b], sh.scale)
    oracle.attention.head_backward_keyset(q, Kb, Vb, T[b], sh.scale, dO, O, l)
    return time.perf_counter() - t0


def _pool_units(workload, n):
    """The first n units of the sampled plan: batch 0, KV group 0 with all its
    query heads, TTT steps spread from the last to the first."""
    sh = wl.WORKLOADS[workload].attn
    G = sh.H // sh.H_kv
    ks = sorted(sh.steps, reverse=True)
    n_steps = max(1, n // G)
    pick = [ks[round(i * (len(ks) - 1) / max(1, n_steps - 1))] for i in range(n_steps)] \
        if n_steps > 1 else [ks[0]]
    return [(0, h, k) for k in dict.fromkeys(pick) for h in range(G)]


def cpu_baseline(workload, mode="pool"):
    """The fp64 oracle, as it stands, on a bounded sample of the workload.

    mode "pool": one wave of concurrent single-threaded oracle tasks, one per
    host core, over the sampled units (batch 0, KV group 0 with all its query
    heads, TTT steps spread over 0..K-1); value = their useful FLOPs / wall
    time of the wave.  mode "one": one query head (b=0, h=0) at the last TTT
    step in this process, NumPy BLAS at its default thread count.
    Plus the soft-CE oracle on 256 rows."""
    import concurrent.futures as cf
    import multiprocessing as mp
    w = wl.WORKLOADS[workload]
    sh, sc = w.attn, w.soft_ce
    T = wl.draw_T(sh, w.seed)
    cores = os.cpu_count() or 1
    if mode == "pool":
        units = _pool_units(workload, cores)
        saved = {v: os.environ.get(v) for v in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS")}
        for v in saved:
            os.environ[v] = "1"
        try:
            with cf.ProcessPoolExecutor(max_workers=len(units),
                                        mp_context=mp.get_context("spawn")) as ex:
                t0 = time.perf_counter()
                secs = list(ex.map(_oracle_head_task, *zip(*[(workload,) + u for u in units])))
                wall_all = time.perf_counter() - t0
        finally:
            for v, val in saved.items():
                if val is None:
                    os.environ.pop(v, None)
                else:
                    os.environ[v] = val
        used = len(units)
        wall = max(secs)  # the tasks run concurrently, one per core
        sample = (f"{workload}: {len(units)} concurrent single-threaded oracle tasks (fwd+bwd of one "
                  f"query head each: b=0, KV group 0, heads 0..{sh.H // sh.H_kv - 1}, TTT steps "
                  f"{sorted({u[2] for u in units})}); oracle time of the slowest task {wall:.1f} s "
                  f"(wave wall time with worker start-up and input generation {wall_all:.1f} s)")
    else:
        units = [(0, 0, sh.steps[-1])]
        t0 = time.perf_counter()
        _oracle_head_task(workload, *units[0])
        wall = time.perf_counter() - t0
        used = cores
        sample = (f"{workload}: one query head (b=0, h=0) at TTT step k={sh.steps[-1]}, fwd+bwd, "
                  f"NumPy BLAS at its default thread count, {wall:.1f} s")
    flops = sum(14 * sh.D * metrics.useful_entries(T[b], sh.Q_LEN, k) for b, _, k in units)
    full = metrics.attn_useful_flops(sh, T)
    rows = 256
    g0 = torch.Generator().manual_seed(w.seed)
    z = (torch.randn((rows, sc.V), generator=g0) * sc.z_std).numpy()
    lg = torch.randn((rows, sc.V), generator=g0) * sc.p_std
    pp = torch.softmax(lg / sc.p_temp, dim=1).numpy()
    gg = np.full(rows, 1.0 / sc.N, dtype=np.float32)
    import oracle
    t0 = time.perf_counter()
    oracle.soft_ce.soft_ce(z, pp, gg)
    t_ce = time.perf_counter() - t0
    value = flops / wall / 1e12
    return {"value": round(value, 6), "unit": "TFLOP/s", "cores": used, "kind": "oracle",
            "sample": sample + f"; soft-CE oracle on {rows} rows of V={sc.V} ({t_ce:.2f} s)",
            "full_config_s_extrapolated": round(sum(full) / (value * 1e12), 1),
            "soft_ce_gbs": round(12 * rows * sc.V / t_ce / 1e9, 4),
            "host_cores": cores}


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
        cb = cpu_baseline(a.workload, mode="one")
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


def run_profile_case(a):
    """Two calls of one row on bounded memory, for ncu captures: the attention
    forward + backward at one TTT step of the workload (inputs of that step
    only), the workload's soft-CE on 1024 of its rows, the fused LM head, or the
    verifier.  Prints nothing measured."""
    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    from speculative_decoding_draft_eagle_gb300 import build, ops
    build.build()
    if a.profile == "attn":
        w = wl.WORKLOADS[a.workload]
        sh = w.attn
        k = sh.steps[-1] if a.profile_step is None else a.profile_step
        T = wl.draw_T(sh, w.seed)
        Ks = [wl.kv_block(sh, "K", j, dev, w.seed) for j in range(k + 1)]
        Vs = [wl.kv_block(sh, "V", j, dev, w.seed) for j in range(k + 1)]
        q, dO = wl.step_query(sh, k, dev, w.seed), wl.step_dout(sh, k, dev, w.seed)
        for _ in range(2):
            out, lse = ops.stt_attn_fwd(q, Ks, Vs, T, sh.scale)
            ops.stt_attn_bwd(q, Ks, Vs, T, out, dO, lse, sh.scale)
    elif a.profile == "soft_ce":
        # the workload's soft-CE rows, 1024 of them (its vocabulary, so the same
        # slice layout as the full call; about 1.2 GB of z and p)
        sc = wl.WORKLOADS[a.workload].soft_ce
        z0, p, g = wl.soft_ce_inputs(dataclasses.replace(sc, N=1024, mask_beyond_T=False), dev, 1007)
        for _ in range(2):
            ops.soft_ce_fwd_bwd_inplace(z0.clone(), p, g)
    elif a.profile == "lm_head":
        h, W, p, g = wl.lm_head_inputs(wl.LM_HEAD, dev, 1002)
        for _ in range(2):
            ops.stt_lm_head_ce(h, W, p, g)
    else:
        args = wl.verify_inputs(wl.VERIFY, dev, 1006)
        for _ in range(2):
            ops.stt_verify(*args)
    torch.cuda.synchronize()
    assert ops.stt_device_error() == 0
    print(f"profile case {a.profile} done", flush=True)


def main():
    a = parse()
    if a.profile:
        run_profile_case(a)
    elif a.impl == "reference":
        run_reference(a)
    else:
        run_ours(a)


if __name__ == "__main__":
    main()
