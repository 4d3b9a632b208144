#!/usr/bin/env python
"""Benchmark of broadcasting elementwise binary ops (forward + fused
backward) on GB300: effective HBM GB/s against the HBM roofline.

One step = every op of the five seeded synthetic workloads (forward chain,
then fused backward with sum-to-shape), issued through the C ABI on
device-resident inputs:

  c1  mul      [32,64,128] * [64,1]
  c2  bias add [4096,1024] + [1024]
  c3  affine   ([16,1024,768] * [768]) + [768]
  c4  scores   ([8,12,1024,1024] + causal mask [1,1,1024,1024]) / [8.0]
  c5a sub      transposed view [128,256,512] - [1,256,1]
  c5b div      [4,1,8,1,16,1,32,64] / [1,6,1,12,1,10,1,64]

value = algorithmic bytes of the step (each op reads every input once and
writes every output once) / device time of the step (CUDA events, L2
flushed before each step).  ``--impl reference`` times the CPU oracle on a
bounded sample of the same workload instead.

Launch: ``python bench.py --gpus N --steps K --warmup W``; for N > 1 under
torchrun, every rank runs its own replica of the step (weak scaling, no
collective on the data path) and rank 0 prints the line.
"""
from __future__ import annotations

import argparse
import ctypes
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads  # noqa: E402

METRIC = "effective HBM GB/s (and % of GB300 peak) for broadcast binary fwd+bwd"
NOMINAL_HBM_GBS = 8000.0
FALLBACK_HBM_GBS = 6800.0
SUITE = ["c1", "c2", "c3", "c4", "c5a", "c5b"]
WORKLOAD_DESC = ("five-workload suite c1..c5b (c1 mul [32,64,128]x[64,1]; c2 bias add "
                 "[4096,1024]+[1024]; c3 affine [16,1024,768]; c4 causal-mask add + /8 on "
                 "[8,12,1024,1024]; c5a transposed-view sub [128,256,512]-[1,256,1]; c5b 8-d div "
                 "to [4,6,8,12,16,10,32,64]) fwd+bwd")
KERNEL_SOURCES = ["broadcast_elementwise_shape_gb300/csrc/zr_kernels.cuh",
                  "broadcast_elementwise_shape_gb300/csrc/zr_sab.cuh",
                  "broadcast_elementwise_shape_gb300/csrc/zr_internal.h",
                  "broadcast_elementwise_shape_gb300/csrc/zr_plan.cpp"]


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=300)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", choices=["zr", "reference"], default="zr")
    p.add_argument("--workload", default="suite", help="suite or one of " + ",".join(workloads.NAMES))
    p.add_argument("--dims", default=None,
                   help="JSON size overrides for a single --workload (see workloads.DEFAULT_DIMS), "
                        "e.g. for a smaller profiling case")
    p.add_argument("--e2e-steps", type=int, default=None,
                   help="timed end-to-end steps (default: --steps, at least 10 and at most 50)")
    p.add_argument("--config-reps", type=int, default=20,
                   help="timed runs per workload phase in the per-config pass (0: skip)")
    p.add_argument("--breakdown-steps", type=int, default=20,
                   help="steps of the untimed per-op breakdown pass")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--ref-procs", type=int, default=0,
                   help="processes of the reference arm's oracle pool (0: one per host core)")
    p.add_argument("--no-e2e", action="store_true")
    a = p.parse_args()
    if a.warmup < 3:
        p.error("--warmup must be >= 3")
    return a


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def max_over_ranks(ms, world, device=None):
    """The slowest rank's timed total: with N replicas (one per GPU, no
    collective on the data path) the job takes as long as its slowest rank."""
    if world == 1:
        return ms
    import torch
    import torch.distributed as dist
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_gbs(world, step_bytes, steps, total_ms):
    """Whole-job throughput: every rank moves step_bytes per step (weak
    scaling), over the slowest rank's time."""
    return world * step_bytes * steps / (total_ms * 1e-3) / 1e9


def _code_only(text):
    """C++ source without comments, blank lines and spacing (a change to a
    comment or to layout leaves the compiled kernels, and so their measured
    traffic, as they are)."""
    import re
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    text = re.sub(r"//[^\n]*", "", text)
    return "\n".join(" ".join(line.split()) for line in text.splitlines() if line.strip())


def kernel_hash():
    """Hash of the code of the kernel sources: profiles/traffic.json holds the
    ncu-measured traffic under the hash of the code it was measured on."""
    h = hashlib.sha256()
    for f in KERNEL_SOURCES:
        with open(os.path.join(ROOT, f), encoding="utf-8") as fh:
            h.update(_code_only(fh.read()).encode())
    return h.hexdigest()[:16]


def measured_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


# ------------------------------------------------------------------ op list

def chain_reads(op1, op2):
    """Inputs (a, b, c) the full chain backward reads: t = a op1 b when op2's
    grad_c needs it (mul, div); b for grad_a and a for grad_b when op1 is mul
    or div (div's grad_b also b); c when op2 is mul or div."""
    need_t = op2 in ("mul", "div")
    ra = need_t or op1 in ("mul", "div")
    rb = need_t or op1 in ("mul", "div")
    rc = op2 in ("mul", "div")
    return ra, rb, rc


def op_bytes(step, shapes, es=4):
    """Algorithmic bytes of one op: read each input once, write each output
    once (es bytes per element)."""
    return es * op_elems(step, shapes)


def op_elems(step, shapes):
    """Elements the op reads and writes (its algorithmic bytes / element size)."""
    if step[0] == "ufwd":
        _, op, alpha, xn, on = step
        return (shapes[xn] + shapes[on])
    if step[0] == "ubwd":
        _, op, alpha, gn, xn, gxn = step
        return (shapes[gn] + (shapes[xn] if op == "gelu" else 0) + shapes[gxn])
    if step[0] == "cfwd":
        _, op1, op2, an, bn, cn, on = step
        return (shapes[an] + shapes[bn] + shapes[cn] + shapes[on])
    if step[0] == "cbwd":
        _, op1, op2, gn, an, bn, cn, gan, gbn, gcn = step
        ra, rb, rc = chain_reads(op1, op2)
        return (shapes[gn] + ra * shapes[an] + rb * shapes[bn] + rc * shapes[cn]
                    + shapes[gan] + shapes[gbn] + shapes[gcn])
    if step[0] == "fwd":
        _, op, an, bn, on = step
        return (shapes[an] + shapes[bn] + shapes[on])
    _, op, gn, an, bn, gan, gbn = step
    reads_a = op in ("mul", "div")
    reads_b = op in ("mul", "div")
    return (shapes[gn] + (shapes[an] if reads_a else 0) + (shapes[bn] if reads_b else 0)
                + shapes[gan] + shapes[gbn])


def numel(shape):
    n = 1
    for s in shape:
        n *= int(s)
    return n


def shape_table(name, host):
    """Element counts of every tensor named in a workload's steps."""
    sizes = {k: v.numel() for k, v in host.items()}
    shapes = {k: tuple(v.shape) for k, v in host.items()}
    import numpy as np
    for step in workloads.STEPS[name]:
        if step[0] in ("ufwd", "ubwd"):
            src, dst = step[-2], step[-1]
            shapes[dst], sizes[dst] = shapes[src], sizes[src]
        elif step[0] == "cfwd":
            _, op1, op2, an, bn, cn, on = step
            shapes[on] = tuple(np.broadcast_shapes(shapes[an], shapes[bn], shapes[cn]))
            sizes[on] = numel(shapes[on])
        elif step[0] == "cbwd":
            _, op1, op2, gn, an, bn, cn, gan, gbn, gcn = step
            for src, dst in ((an, gan), (bn, gbn), (cn, gcn)):
                shapes[dst], sizes[dst] = shapes[src], sizes[src]
        elif step[0] == "fwd":
            _, op, an, bn, on = step
            shapes[on] = tuple(np.broadcast_shapes(shapes[an], shapes[bn]))
            sizes[on] = numel(shapes[on])
        else:
            _, op, gn, an, bn, gan, gbn = step
            shapes[gan], shapes[gbn] = shapes[an], shapes[bn]
            sizes[gan], sizes[gbn] = sizes[an], sizes[bn]
    return sizes, shapes


# ------------------------------------------------------------------ clocks

class ClockSampler:
    """nvidia-smi sampling (every 100 ms) stamped with host time."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, uuid=None):
        self.samples = []
        self.proc = None
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
               "-lms", "100"]
        if uuid:
            cmd += ["-i", uuid]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                                         text=True)
        except Exception:
            self.proc = None
            return
        self.th = threading.Thread(target=self._read, daemon=True)
        self.th.start()

    def _read(self):
        for line in self.proc.stdout:
            self.samples.append((time.monotonic(), [x.strip() for x in line.split(",")]))

    def stop(self):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self, t0, t1):
        if not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"],
                    "samples": 0}
        win = [s for t, s in self.samples if t0 <= t <= t1]
        if not win:  # very short timed region: nearest samples
            win = [min(self.samples, key=lambda ts: abs(ts[0] - (t0 + t1) / 2))[1]]
        sm = [float(s[1]) for s in win if s[1].replace(".", "").isdigit()]
        smax = [float(s[2]) for s in win if s[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for s in win for i in range(4)
                          if len(s) > 5 + i and s[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None, "reasons": reasons,
                "samples": len(win)}


# ------------------------------------------------------------------ zr arm

class Suite:
    """Device tensors, preallocated outputs/workspaces and prepared C-ABI
    calls for the chosen workloads."""

    def __init__(self, names, device, dims=None):
        import torch
        import broadcast_elementwise_shape_gb300 as zr
        from broadcast_elementwise_shape_gb300 import ZrTensor
        self.zr = zr
        self.L = zr.lib()
        self.torch = torch
        self.device = device
        self.calls = []       # (config, kind, op, bytes, launches, fn, elements)
        self.host = {}
        self.dev = {}
        self.in_names = {}
        self.out_names = {}
        self._keep = []
        i64p = ctypes.POINTER(ctypes.c_int64)
        L = self.L
        L.zr_test_describe_bwd.argtypes = [ctypes.c_int, ZrTensor, ZrTensor, ZrTensor,
                                           ctypes.c_void_p, ctypes.c_void_p, ctypes.c_char_p,
                                           ctypes.c_size_t]
        L.zr_test_describe_fwd.argtypes = [ctypes.c_int, ZrTensor, ZrTensor, ctypes.c_void_p,
                                           i64p, ctypes.c_char_p, ctypes.c_size_t]
        L.zr_test_describe_bwd_t.argtypes = [ctypes.c_int, ctypes.c_int, ZrTensor, ZrTensor,
                                             ZrTensor, ctypes.c_void_p, ctypes.c_void_p,
                                             ctypes.c_char_p, ctypes.c_size_t]
        self.es = {}
        for name in names:
            host = workloads.make_inputs(name, **(dims or {}))
            sizes, shapes = shape_table(name, host)
            self.es[name] = 2 if name in workloads.BF16 else 4
            dt = torch.bfloat16 if self.es[name] == 2 else torch.float32
            env = {}
            for k, v in host.items():
                env[k] = self._to_dev(v).to(dt)
            outs = []
            for step in workloads.STEPS[name]:
                if step[0] in ("fwd", "cfwd", "ufwd", "ubwd"):
                    on = step[-1]
                    env[on] = torch.empty(shapes[on], dtype=dt, device=device)
                    outs.append(on)
                else:
                    for gname in (step[7:10] if step[0] == "cbwd" else step[5:7]):
                        env[gname] = torch.empty(shapes[gname], dtype=dt, device=device)
                        outs.append(gname)
            self.host[name] = host
            self.dev[name] = env
            self.in_names[name] = list(host)
            self.out_names[name] = outs
            for step in workloads.STEPS[name]:
                self.calls.append(self._prepare(name, step, env, sizes))

    def _to_dev(self, v):
        """Device copy keeping strides and storage offset (views included)."""
        torch = self.torch
        st = v.untyped_storage()
        flat = torch.empty(0, dtype=v.dtype).set_(st, 0, (st.nbytes() // v.element_size(),), (1,))
        return flat.to(self.device).as_strided(v.shape, v.stride(), v.storage_offset())

    def _desc(self, t):
        d, keep = self.zr._desc(t)
        self._keep.append(keep)
        return d

    def _prepare_chain(self, name, step, env, sizes, stream_of):
        zr, L, torch = self.zr, self.L, self.torch
        nbytes = op_bytes(step, sizes)
        op1, op2 = zr.OPS[step[1]], zr.OPS[step[2]]
        if step[0] == "cfwd":
            _, _, _, an, bn, cn, on = step
            da, db, dc = self._desc(env[an]), self._desc(env[bn]), self._desc(env[cn])
            out = env[on]
            ost = zr._i64(out.stride())
            self._keep.append(ost)
            ptr = out.data_ptr()

            def fn(da=da, db=db, dc=dc, ptr=ptr, ost=ost):
                rc = L.zr_chain_fwd(op1, op2, da, db, dc, ptr, ost, stream_of())
                if rc:
                    raise zr.ZrError(rc, f"{name} chain fwd")
            return (name, "fwd", f"{step[1]}+{step[2]}", nbytes, 1, fn, sizes[on])
        _, _, _, gn, an, bn, cn, gan, gbn, gcn = step
        dg, da, db, dc = (self._desc(env[k]) for k in (gn, an, bn, cn))
        ptrs = [env[k].data_ptr() for k in (gan, gbn, gcn)]
        need = ctypes.c_size_t(0)
        assert L.zr_chain_bwd(op1, op2, dg, da, db, dc, *ptrs, None, ctypes.byref(need), None) == 0
        ws = torch.empty(max(16, need.value), dtype=torch.uint8, device=self.device)
        self._keep.append(ws)
        L.zr_test_describe_chain_bwd.argtypes = [ctypes.c_int, ctypes.c_int] + [type(dg)] * 4 + [
            ctypes.c_void_p] * 3 + [ctypes.c_char_p, ctypes.c_size_t]
        buf = ctypes.create_string_buffer(8192)
        assert L.zr_test_describe_chain_bwd(op1, op2, dg, da, db, dc, *ptrs, buf, 8192) == 0
        desc = json.loads(buf.value.decode())
        if desc["route"] == "fused":
            p = desc["plans"][0]
            launches = 1 + (p["nslots"] > 1) + ((p["ctas"] > 1) if p["c_scalar"] else (p["nslots"] > 1))
        else:
            launches = 0  # composed route: counted as one op of several launches
        wsz = ws.numel()

        def fn(dg=dg, da=da, db=db, dc=dc, ptrs=ptrs, wsp=ws.data_ptr(), wsz=wsz):
            n = ctypes.c_size_t(wsz)
            rc = L.zr_chain_bwd(op1, op2, dg, da, db, dc, *ptrs, wsp, ctypes.byref(n), stream_of())
            if rc:
                raise zr.ZrError(rc, f"{name} chain bwd")
        return (name, "bwd", f"{step[1]}+{step[2]} ({desc['route']})", nbytes, launches, fn,
                sizes[gn])

    def _prepare_unary(self, name, step, env, sizes, stream_of):
        zr, L = self.zr, self.L
        es = self.es[name]
        dtc = zr.ZR_BF16 if es == 2 else zr.ZR_F32
        nbytes = op_bytes(step, sizes, es)
        uop, alpha = zr.UNARY[step[1]], float(step[2])
        out = env[step[-1]]
        ost = zr._i64(out.stride())
        self._keep.append(ost)
        ptr = out.data_ptr()
        if step[0] == "ufwd":
            dx = self._desc(env[step[3]])

            def fn(dx=dx, ptr=ptr, ost=ost):
                rc = L.zr_unary_fwd_t(dtc, uop, alpha, dx, ptr, ost, stream_of())
                if rc:
                    raise zr.ZrError(rc, f"{name} unary fwd")
            return (name, "fwd", step[1], nbytes, 1, fn, sizes[step[-1]])
        dg, dx = self._desc(env[step[3]]), self._desc(env[step[4]])

        def fn(dg=dg, dx=dx, ptr=ptr, ost=ost):
            rc = L.zr_unary_bwd_t(dtc, uop, alpha, dg, dx, ptr, ost, stream_of())
            if rc:
                raise zr.ZrError(rc, f"{name} unary bwd")
        return (name, "bwd", step[1], nbytes, 1, fn, sizes[step[-1]])

    def _prepare(self, name, step, env, sizes):
        zr, L, torch = self.zr, self.L, self.torch
        stream_of = lambda: ctypes.c_void_p(torch.cuda.current_stream(self.device).cuda_stream)
        if step[0] in ("cfwd", "cbwd"):
            return self._prepare_chain(name, step, env, sizes, stream_of)
        if step[0] in ("ufwd", "ubwd"):
            return self._prepare_unary(name, step, env, sizes, stream_of)
        opc = zr.OPS[step[1]]
        es = self.es[name]
        dtc = zr.ZR_BF16 if es == 2 else zr.ZR_F32
        nbytes = op_bytes(step, sizes, es)
        if step[0] == "fwd":
            _, op, an, bn, on = step
            da, db = self._desc(env[an]), self._desc(env[bn])
            out = env[on]
            ost = zr._i64(out.stride())
            self._keep.append(ost)
            ptr = out.data_ptr()
            launches = 1
            if es == 4:  # the plan description hooks plan float storage
                buf = ctypes.create_string_buffer(2048)
                assert L.zr_test_describe_fwd(opc, da, db, ptr, ost, buf, 2048) == 0
                launches = 0 if json.loads(buf.value.decode()).get("kernel") == "none" else 1

            def fn(da=da, db=db, ptr=ptr, ost=ost):
                rc = L.zr_binary_fwd_t(dtc, opc, da, db, ptr, ost, stream_of())
                if rc:
                    raise zr.ZrError(rc, f"{name} fwd {op}")
            return (name, "fwd", op, nbytes, launches, fn, sizes[on])
        _, op, gn, an, bn, gan, gbn = step
        dg, da, db = self._desc(env[gn]), self._desc(env[an]), self._desc(env[bn])
        pa, pb = env[gan].data_ptr(), env[gbn].data_ptr()
        need = ctypes.c_size_t(0)
        rc = L.zr_binary_bwd_t(dtc, opc, dg, da, db, pa, pb, None, ctypes.byref(need), None)
        assert rc == 0, rc
        ws = torch.empty(max(16, need.value), dtype=torch.uint8, device=self.device)
        self._keep.append(ws)
        buf = ctypes.create_string_buffer(8192)
        assert L.zr_test_describe_bwd_t(dtc, opc, dg, da, db, pa, pb, buf, 8192) == 0
        desc = json.loads(buf.value.decode())
        plans = desc.get("plans", [])
        if plans and plans[0].get("kernel") == "sab":
            launches = 3  # fused pass + one combine per gradient
        else:
            launches = sum(1 + (p.get("nslots", 1) > 1) for p in plans)
        wsz = ws.numel()

        def fn(dg=dg, da=da, db=db, pa=pa, pb=pb, wsp=ws.data_ptr(), wsz=wsz):
            n = ctypes.c_size_t(wsz)
            rc = L.zr_binary_bwd_t(dtc, opc, dg, da, db, pa, pb, wsp, ctypes.byref(n), stream_of())
            if rc:
                raise zr.ZrError(rc, f"{name} bwd {op}")
        return (name, "bwd", op, nbytes, launches, fn, sizes[gn])

    def step_bytes(self):
        return sum(c[3] for c in self.calls)

    def launches(self):
        return sum(c[4] for c in self.calls)


def run_zr(args, rank, world, local):
    import torch
    import torch.distributed as dist

    import __graft_entry__
    __graft_entry__.build()
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA device (no CPU fallback)")
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    if world > 1:
        dist.init_process_group("nccl", device_id=device)
    names = SUITE if args.workload == "suite" else [args.workload]
    dims = json.loads(args.dims) if args.dims else None
    if dims and args.workload == "suite":
        raise SystemExit("--dims needs a single --workload")
    suite = Suite(names, device, dims)
    nbytes = suite.step_bytes()
    l2 = torch.cuda.get_device_properties(device).L2_cache_size
    nflush = max(2 * l2, 256 << 20) // 4
    flush_w = torch.empty(nflush, dtype=torch.float32, device=device)
    flush_r = torch.zeros(nflush, dtype=torch.float32, device=device)

    def flush():
        # Write a buffer of 2x L2, then read another one of 2x L2: the second
        # pass evicts the first one's dirty lines, so their write-back happens
        # here and not inside the next timed region.
        flush_w.fill_(0.0)
        flush_r.sum()
    stream = torch.cuda.current_stream(device)

    ncalls = len(suite.calls)

    def one_step(events=None, only=None):
        for i, c in enumerate(suite.calls):
            timed = events is not None and (only is None or i == only)
            if timed:
                events[i if only is None else 0][0].record(stream)
            c[5]()
            if timed:
                events[i if only is None else 0][1].record(stream)

    def new_events(n):
        return [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                for _ in range(n)]

    for _ in range(args.warmup):
        flush()
        one_step()
    torch.cuda.synchronize()

    # Per-op breakdown (outside the timed region): events around every op.
    # An event between two ops keeps the second op's first kernel from being
    # scheduled while the first op's last kernel drains, so these per-op
    # times add up to a little more than a step of the timed loop.
    nb = max(1, min(args.steps, args.breakdown_steps))
    bd_ev = [new_events(ncalls) for _ in range(nb)]
    for k in range(nb):
        flush()
        one_step(bd_ev[k])
    torch.cuda.synchronize()
    op_ms = [[bd_ev[k][i][0].elapsed_time(bd_ev[k][i][1]) for k in range(nb)]
             for i in range(ncalls)]
    dom = max(range(ncalls), key=lambda i: statistics.fmean(op_ms[i]))

    uuid = None
    try:
        uuid = str(torch.cuda.get_device_properties(device).uuid)
        if not uuid.startswith("GPU-"):
            uuid = "GPU-" + uuid
    except Exception:
        uuid = None
    sampler = ClockSampler(uuid) if rank == 0 else None
    if sampler:
        time.sleep(0.35)
        if not sampler.samples and uuid:
            sampler.stop()
            sampler = ClockSampler(None)
            time.sleep(0.35)
    # Timed loop: events around each whole step and around the dominant op
    # (for its roofline), nothing between the other ops.
    steps_ev = new_events(args.steps)
    dom_ev = [new_events(1) for _ in range(args.steps)]
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    t0 = time.monotonic()
    for k in range(args.steps):
        flush()
        steps_ev[k][0].record(stream)
        one_step(dom_ev[k], only=dom)
        steps_ev[k][1].record(stream)
    torch.cuda.synchronize()
    t1 = time.monotonic()
    if world > 1:
        dist.barrier()
    step_ms = [s.elapsed_time(e) for s, e in steps_ev]
    total_ms = max_over_ranks(sum(step_ms), world, device)
    dom_ms = [dom_ev[k][0][0].elapsed_time(dom_ev[k][0][1]) for k in range(args.steps)]
    clocks = sampler.summary(t0, t1) if sampler else None

    per_config = per_op_alone = None
    if rank == 0 and args.config_reps > 0:
        extra = ([Suite(["x1", "c3f", "c4f", "u1", "c4h", "u1h"], device)]
                 if args.workload == "suite" else [])
        per_config, per_op_alone = run_per_config([suite] + extra, flush, stream, args.config_reps)
    e2e = None
    if not args.no_e2e:
        # Every rank runs its replica end to end; the job takes as long as the
        # slowest rank, and moves every rank's bytes.
        if world > 1:
            dist.barrier()
        e2e = run_e2e(args, suite, flush, stream, nbytes, measure_link=rank == 0)
        ms = max_over_ranks(e2e["ms_per_step"], world, device)
        e2e["value"] = round(job_gbs(world, nbytes, 1, ms), 1)
        e2e["ms_per_step"] = round(ms, 3)
        e2e["h2d_bytes_per_step"] *= world
        e2e["d2h_bytes_per_step"] *= world
    if sampler:
        sampler.stop()

    if rank == 0:
        peak, peak_kind = measured_peak()
        value = job_gbs(world, nbytes, args.steps, total_ms)
        per_op = []
        for i, c in enumerate(suite.calls):
            mean = statistics.fmean(op_ms[i])
            med = statistics.median(op_ms[i])
            per_op.append({"config": c[0], "kind": c[1], "op": c[2], "bytes": c[3],
                           "launches": c[4], "ms_mean": round(mean, 5), "ms_median": round(med, 5),
                           "gbs": round(c[3] / (mean * 1e-3) / 1e9, 1)})
        dom_gbs = suite.calls[dom][3] / (statistics.fmean(dom_ms) * 1e-3) / 1e9
        traffic = read_traffic(suite.calls[dom])
        roofline = {"bound": "hbm", "achieved": round(dom_gbs, 1), "peak": peak, "unit": "GB/s",
                    "frac": round(dom_gbs / peak, 4), "traffic": traffic,
                    "kernel": f"{suite.calls[dom][0]} {suite.calls[dom][1]} {suite.calls[dom][2]}",
                    "peak_kind": peak_kind}
        cpu = None
        if not args.no_cpu_baseline and world == 1:
            cpu = cpu_baseline()
        line = {
            "metric": METRIC, "value": round(value, 1), "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(total_ms / args.steps, 5), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": {"workload": WORKLOAD_DESC if args.workload == "suite" else
                       (args.workload + (" " + json.dumps(dims) if dims else "")),
                       "bytes_per_step": nbytes,
                       "l2": "flushed before every step, outside the timed events: 2x L2 written, "
                             "then another 2x L2 buffer read (clean, cold L2 at step start)",
                       "pct_of_measured_hbm": round(value / world / peak, 4),
                       "pct_of_nominal_8000": round(value / world / NOMINAL_HBM_GBS, 4)},
            "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e,
            "gpu_launches": suite.launches() * args.steps, "clocks": clocks, "per_op": per_op,
            "per_op_pass": f"untimed breakdown, {nb} steps with events around every op",
            "per_config": per_config,
            "per_op_alone": per_op_alone,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def run_per_config(suites, flush, stream, reps, warm=5):
    """Each workload's forward chain and backward chain, and each op, timed on
    its own: the median of ``reps`` CUDA-event timings after ``warm`` untimed
    runs, with L2 flushed before every run.  GB/s = algorithmic bytes over
    that median; elements/s = elements of the broadcast shape (per op) over
    it.  The supplementary contiguous add ``x1`` is timed here only."""
    import torch
    peak, _ = measured_peak()

    def time_calls(calls):
        ev = []
        for r in range(warm + reps):
            flush()
            s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            s.record(stream)
            for c in calls:
                c[5]()
            e.record(stream)
            if r >= warm:
                ev.append((s, e))
        torch.cuda.synchronize()
        return statistics.median(s.elapsed_time(e) for s, e in ev)

    def record(nbytes, nelem, ms):
        gbs = nbytes / (ms * 1e-3) / 1e9
        return {"bytes": nbytes, "ms_median": round(ms, 5), "gbs": round(gbs, 1),
                "elems_per_s": float(f"{nelem / (ms * 1e-3):.4g}"),
                "pct_of_measured_hbm": round(gbs / peak, 4),
                "pct_of_nominal_8000": round(gbs / NOMINAL_HBM_GBS, 4)}

    per_config, per_op = {}, []
    for suite in suites:
        for name in dict.fromkeys(c[0] for c in suite.calls):
            for kind in ("fwd", "bwd"):
                calls = [c for c in suite.calls if c[0] == name and c[1] == kind]
                ms = time_calls(calls)
                per_config.setdefault(name, {})[kind] = record(
                    sum(c[3] for c in calls), sum(c[6] for c in calls), ms)
                for c in calls:
                    rec = record(c[3], c[6], time_calls([c]) if len(calls) > 1 else ms)
                    per_op.append({"config": c[0], "kind": c[1], "op": c[2], **rec})
    return per_config, per_op


def last_readers(steps):
    """For each name a workload's steps read: the index of the last step that
    reads it (the next step's upload of that buffer must wait for it)."""
    last = {}
    for i, step in enumerate(steps):
        for k in step_io(step)[0]:
            last[k] = i
    return last


def step_io(step):
    """Names a workload step reads and writes."""
    kind = step[0]
    if kind == "fwd":
        return list(step[2:4]), [step[4]]
    if kind == "bwd":
        return list(step[2:5]), list(step[5:7])
    if kind == "cfwd":
        return list(step[3:6]), [step[6]]
    if kind == "cbwd":
        return list(step[3:7]), list(step[7:10])
    if kind == "ufwd":
        return [step[3]], [step[4]]
    return list(step[3:5]), [step[5]]


def link_rates(device, nbytes=1 << 30, reps=5):
    """Copy rates of the host link in GB/s (median of `reps`): pinned host to
    device, device to pinned host, and both directions at once on two
    streams (their total).  The ceiling for the end-to-end measurement."""
    import torch
    n = nbytes // 4
    h_src = torch.ones(n, dtype=torch.float32).pin_memory()
    h_dst = torch.empty(n, dtype=torch.float32).pin_memory()
    d_dst = torch.empty(n, dtype=torch.float32, device=device)
    d_src = torch.ones(n, dtype=torch.float32, device=device)
    cur = torch.cuda.current_stream(device)
    s1, s2 = torch.cuda.Stream(device=device), torch.cuda.Stream(device=device)

    def up():
        d_dst.copy_(h_src, non_blocking=True)

    def down():
        h_dst.copy_(d_src, non_blocking=True)

    def both():
        e0 = cur.record_event()
        s1.wait_event(e0)
        s2.wait_event(e0)
        with torch.cuda.stream(s1):
            up()
        with torch.cuda.stream(s2):
            down()
        cur.wait_event(s1.record_event())
        cur.wait_event(s2.record_event())

    # The library's own forward reading its input straight from pinned host
    # memory (the C ABI takes a pinned pointer the device addresses as is):
    # out = h_src + 0 into device memory; rate = host bytes read per second.
    import broadcast_elementwise_shape_gb300 as zr
    zero = torch.zeros(1, dtype=torch.float32, device=device)
    da, ka = zr._desc(h_src.view(1, n), need_data=False)
    da.data = h_src.data_ptr()
    db, kb = zr._desc(zero)

    def zero_copy():
        rc = zr.lib().zr_binary_fwd(0, da, db, ctypes.c_void_p(d_dst.data_ptr()), None,
                                    ctypes.c_void_p(cur.cuda_stream))
        if rc:
            raise zr.ZrError(rc, "zero-copy forward")

    out = {}
    for key, fn, moved in (("h2d", up, nbytes), ("d2h", down, nbytes), ("both", both, 2 * nbytes),
                           ("kernel_reads_host", zero_copy, nbytes)):
        fn()
        torch.cuda.synchronize(device)
        ts = []
        for _ in range(reps):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(cur)
            fn()
            b.record(cur)
            torch.cuda.synchronize(device)
            ts.append(a.elapsed_time(b))
        out[key] = round(moved / (statistics.median(ts) * 1e-3) / 1e9, 1)
    del h_src, h_dst, d_dst, d_src
    return out


def run_e2e(args, suite, flush, stream, nbytes, measure_link=True):
    """Same metric with host buffers: every step copies each input from
    pinned host memory and every output back, inside the timed region.  The
    copies are scheduled per op: an input is uploaded (on an upload stream)
    just before the first op that reads it, the op runs on the caller's
    stream once its uploads are in, and each output is downloaded (on a
    third stream) as soon as its op has written it.  Uploads thus run ahead
    of the ops and downloads behind them, so the host link carries both
    directions at once for most of the step (a forward whose inputs are
    small starts its large download while the next op's large input is
    still arriving).  Steps follow one another as a training loop's would:
    the next step's uploads start while this step's last downloads are still
    running, each waiting only for what it overwrites (an input buffer for
    the previous step's last op that read it, an op's outputs for the
    previous step's download of them).  The inputs (4 GB) are far larger
    than L2, so no flush is needed between the steps.  The step time is the
    median interval between consecutive steps' ends, an end being an event
    recorded after the step's last download."""
    import torch
    h2d = d2h = 0
    plan = []  # per op: (uploads [(dst, src)], call, downloads [(dst, src)], last readers)
    for name in suite.dev:
        env = suite.dev[name]
        host_in = set(suite.in_names[name])
        written = set(suite.out_names[name])
        calls = [c for c in suite.calls if c[0] == name]
        steps = workloads.STEPS[name]
        assert len(calls) == len(steps)
        uploaded = {}
        first = len(plan)
        for i, (step, call) in enumerate(zip(steps, calls)):
            reads, writes = step_io(step)
            ups, downs = [], []
            for k in reads:
                if k in host_in and k not in uploaded:
                    uploaded[k] = len(ups)
                    # Copy the operand's whole storage (views keep their
                    # layout); the pinned host buffer holds the same bytes
                    # in the device's element type.
                    t = env[k]
                    ds = t.untyped_storage()
                    dflat = torch.empty(0, dtype=t.dtype, device=t.device).set_(
                        ds, 0, (ds.nbytes() // t.element_size(),), (1,))
                    hp = torch.empty(dflat.numel(), dtype=t.dtype).pin_memory()
                    hp.copy_(dflat)
                    ups.append((dflat, hp, k))
                    h2d += hp.numel() * hp.element_size()
            for k in writes:
                if k in written:
                    t = env[k]
                    hp = torch.empty(t.shape, dtype=t.dtype).pin_memory()
                    downs.append((hp, t))
                    d2h += hp.numel() * hp.element_size()
            plan.append([ups, call, downs, reads])
        # For each upload: the op of this workload that reads it last.
        last = last_readers(steps)
        for i in range(first, len(plan)):
            plan[i][3] = [first + last[k] for _dst, _src, k in plan[i][0]]
    s_in = torch.cuda.Stream(device=stream.device)
    s_out = torch.cuda.Stream(device=stream.device)
    steps = args.e2e_steps if args.e2e_steps else min(50, max(10, args.steps))
    steps = max(1, steps)
    n = len(plan)

    def run(nsteps):
        """nsteps pipelined steps; returns the start event and, per step, an
        event on the download stream after its last download (so after all
        of the step's work)."""
        s = torch.cuda.Event(enable_timing=True)
        s.record(stream)
        s_in.wait_event(s)
        s_out.wait_event(s)
        ends = []
        done_call = [None] * n  # previous step's events, per op
        done_down = [None] * n
        for _ in range(nsteps):
            call_ev, down_ev = [None] * n, [None] * n
            for i, (ups, call, downs, last) in enumerate(plan):
                if ups:
                    for j in set(last):
                        if done_call[j] is not None:
                            s_in.wait_event(done_call[j])
                    with torch.cuda.stream(s_in):
                        for dst, src, _k in ups:
                            dst.copy_(src, non_blocking=True)
                    stream.wait_event(s_in.record_event())
                if done_down[i] is not None:
                    stream.wait_event(done_down[i])
                call[5]()
                call_ev[i] = stream.record_event()
                if downs:
                    s_out.wait_event(call_ev[i])
                    with torch.cuda.stream(s_out):
                        for dst, src in downs:
                            dst.copy_(src, non_blocking=True)
                    down_ev[i] = s_out.record_event()
            done_call, done_down = call_ev, down_ev
            s_out.wait_event(stream.record_event())
            s_out.wait_event(s_in.record_event())
            e = torch.cuda.Event(enable_timing=True)
            e.record(s_out)
            ends.append(e)
        stream.wait_event(ends[-1])
        return s, ends

    flush()
    run(1)  # warm-up
    torch.cuda.synchronize()
    flush()
    s, ends = run(steps)
    torch.cuda.synchronize()
    # The step time is the median interval between consecutive steps' ends
    # (the loop's period once it runs; robust to a late copy in one step).
    marks = [s] + ends
    ms = statistics.median(a.elapsed_time(b) for a, b in zip(marks[:-1], marks[1:]))
    moved = (h2d + d2h) / (ms * 1e-3) / 1e9
    out = {"value": round(nbytes / (ms * 1e-3) / 1e9, 1), "unit": "GB/s",
           "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": ms,
           "steps": steps, "copied_gbs": round(moved, 1),
           "copies": "per op: uploads ahead on one stream, ops on the caller's stream, "
                     "downloads behind on a third stream; steps pipelined"}
    if measure_link:  # this process's own host link (rank 0's at N > 1)
        link = link_rates(stream.device)
        out["link_gbs"] = link
        out["frac_of_link_both"] = round(moved / link["both"], 3) if link["both"] else None
    return out


def read_traffic(call):
    """DRAM bytes (read + write, summed over the op's launches) of the
    dominant op from the committed ncu summary (profiles/traffic.json), if
    it was taken on the current kernel sources; otherwise None."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            t = json.load(f)
    except Exception:
        return None
    if t.get("kernel_hash") != kernel_hash():
        return None
    key = f"{call[0]} {call[1]} {call[2]}"
    v = t.get("per_op_dram_bytes", {}).get(key)
    return v


# ------------------------------------------------------------------ oracle (CPU)

def oracle_steps(name, host):
    """The oracle over every step of one workload (forward chain, then
    backward); returns (algorithmic bytes, op-elements)."""
    import oracle
    sizes, _ = shape_table(name, host)
    env = dict(host)
    total_bytes = elems = 0
    for step in workloads.STEPS[name]:
        total_bytes += op_bytes(step, sizes)
        if step[0] == "fwd":
            _, op, an, bn, on = step
            env[on] = oracle.binary_fwd(op, env[an], env[bn])
            elems += sizes[on]
        else:
            _, op, gn, an, bn, gan, gbn = step
            ga, gb, _, _ = oracle.binary_bwd(op, env[gn], env[an], env[bn])
            env[gan], env[gbn] = ga, gb
            elems += sizes[gn]
    return total_bytes, elems


# The host baseline's sample: the complete fwd+bwd of c1, c2 and c3 at full
# size, and of c5a and c5b at reduced sizes that keep their structure (a
# transposed view; an 8-d division with both gradients reduced), so that the
# oracle's strided and 8-d paths are timed too.  (name, size overrides).
CPU_SAMPLE = (("c1", {}), ("c2", {}), ("c3", {}), ("c5a", {"P": 16}),
              ("c5b", {"a": (4, 1, 8, 1, 4, 1, 8, 64), "b": (1, 6, 1, 12, 1, 10, 1, 64)}))
# The reference arm's per-step sample (smaller: K + W steps in minutes).
REF_SAMPLE = (("c1", {}), ("c2", {}), ("c5a", {"P": 4}),
              ("c5b", {"a": (4, 1, 8, 1, 4, 1, 2, 64), "b": (1, 6, 1, 12, 1, 10, 1, 64)}))


def _items(sample):
    """(name, dims) pairs from workload names or (name, dims) pairs."""
    return [(x, {}) if isinstance(x, str) else (x[0], dict(x[1])) for x in sample]


def sample_label(sample):
    """Readable name of a sample: c5a[P=16] for a workload at reduced sizes."""
    out = []
    for name, dims in _items(sample):
        if dims:
            dd = ",".join(f"{k}={'x'.join(map(str, v)) if isinstance(v, (tuple, list)) else v}"
                          for k, v in dims.items())
            out.append(f"{name}[{dd}]")
        else:
            out.append(name)
    return out


def oracle_sample(sample):
    """Run the oracle over the complete fwd+bwd of the sample's workloads in
    this process; returns (seconds, algorithmic bytes, output elements)."""
    import oracle
    oracle.build()
    total_bytes = elems = 0
    t_total = 0.0
    for name, dims in _items(sample):
        host = workloads.make_inputs(name, **dims)
        t = time.perf_counter()
        b, e = oracle_steps(name, host)
        t_total += time.perf_counter() - t
        total_bytes += b
        elems += e
    return t_total, total_bytes, elems


def _oracle_worker(sample, cmd, res):
    """One process of OraclePool: builds its own inputs, reports ready, then
    runs the whole sample each time it is told to."""
    import torch
    torch.set_num_threads(1)  # one core per process; torch only draws the inputs
    import oracle
    oracle.build()
    items = _items(sample)
    inputs = [workloads.make_inputs(n, **d) for n, d in items]
    res.put("ready")
    while cmd.get() is not None:
        t0 = time.time()
        nbytes = elems = 0
        for (n, _), host in zip(items, inputs):
            b, e = oracle_steps(n, host)
            nbytes += b
            elems += e
        res.put((t0, time.time(), nbytes, elems))


class OraclePool:
    """The oracle on every host core: one spawned process per core (the
    oracle itself is single-threaded and unchanged), each with its own copy
    of the sample's inputs.  Independent problems on separate cores is how
    the path shards, so the pool's throughput is the processes' total bytes
    over the wall time from the first start to the last finish.  Spawned,
    not forked, so that no process inherits a CUDA context.  ``sample``:
    workload names, or (name, size overrides) pairs."""

    def __init__(self, sample, procs=None):
        import multiprocessing as mp
        import oracle
        oracle.build()  # once, before the processes load it
        ctx = mp.get_context("spawn")
        self.n = procs or len(os.sched_getaffinity(0))
        self.res = ctx.Queue()
        self.cmd = [ctx.Queue() for _ in range(self.n)]
        sample = _items(sample)
        self.procs = [ctx.Process(target=_oracle_worker, args=(sample, q, self.res),
                                  daemon=True) for q in self.cmd]
        for p in self.procs:
            p.start()
        for _ in range(self.n):
            assert self.res.get(timeout=600) == "ready"

    def run(self):
        """One pass of every process; returns (wall seconds, bytes, elements)."""
        for q in self.cmd:
            q.put(1)
        out = [self.res.get(timeout=600) for _ in range(self.n)]
        span = max(o[1] for o in out) - min(o[0] for o in out)
        return span, sum(o[2] for o in out), sum(o[3] for o in out)

    def close(self):
        for q in self.cmd:
            q.put(None)
        for p in self.procs:
            p.join(timeout=60)


def cpu_baseline(sample=CPU_SAMPLE, runs=3, procs=None):
    """The oracle on the machine's host cores: `runs` passes of the pool (one
    process per core, each computing the complete fwd+bwd of the sample),
    median wall time; plus the same sample on one core for reference."""
    secs1, nbytes1, elems1 = oracle_sample(sample)
    pool = OraclePool(sample, procs)
    try:
        passes = [pool.run() for _ in range(runs)]
    finally:
        pool.close()
    span = statistics.median(p[0] for p in passes)
    nbytes, elems = passes[0][1], passes[0][2]
    return {"value": round(nbytes / span / 1e9, 4), "unit": "GB/s", "cores": pool.n,
            "kind": "oracle",
            "sample": f"complete fwd+bwd of {', '.join(sample_label(sample))} in each of "
                      f"{pool.n} processes (single-thread C++ oracle, binary64 accumulation, one "
                      f"process per host core; c5a and c5b at the reduced sizes given, with their "
                      f"transposed-view and 8-d structure); {elems} op-elements per pass, median "
                      f"of {runs} passes, {span:.2f} s",
            "seconds": round(span, 3),
            "single_core": {"value": round(nbytes1 / secs1 / 1e9, 4), "cores": 1,
                            "seconds": round(secs1, 3)}}


def run_reference(args, rank, world):
    if rank != 0:
        return
    # Each step is one pass of the oracle on every host core over a bounded
    # sample of the suite, sized so that K + W steps stay within a few
    # minutes.
    sample = list(REF_SAMPLE) if args.steps + args.warmup <= 40 else [("c1", {})]
    names = sample_label(sample)
    pool = OraclePool(sample, args.ref_procs or None)
    try:
        for _ in range(args.warmup):
            pool.run()
        times, nbytes = [], 0
        for _ in range(args.steps):
            s, b, _ = pool.run()
            times.append(s)
            nbytes = b
    finally:
        pool.close()
    total = sum(times)
    value = nbytes * len(times) / total / 1e9
    sample = (f"complete fwd+bwd of {' and '.join(names)} per step in each of {pool.n} "
              "processes (single-thread C++ oracle, one process per host core)")
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(1e3 * total / len(times), 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": "a sample of the suite by design (the oracle is a deliberately "
                               "plain CPU program): complete fwd+bwd of " + ", ".join(names)
                               + f" per step on {pool.n} host cores"},
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": pool.n,
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    args = parse()
    rank, world, local = dist_env()
    if args.gpus > 1 and world == 1:
        raise SystemExit("--gpus > 1 needs torchrun (one process per GPU)")
    if args.impl == "reference":
        run_reference(args, rank, world)
        return
    run_zr(args, rank, world, local)


if __name__ == "__main__":
    main()
