#!/usr/bin/env python
"""Throughput benchmark of the chunked gated delta rule forward on one GB300 per rank.

Workload (one "step"): the long-context bf16 case -- one packed sequence of T = 65536
tokens, 16 key heads shared by 32 value heads, K = V = 128, C = 64, fp32 state, h0 = 0,
synthetic seeded inputs -- run through all three phases (segment summaries, prefix scan,
re-emit) with P segments.  Metric: tokens/s (whole job, all ranks).  Inputs plus output are
1.63 GB, far larger than the 129 MB L2, so no flush is needed between steps.

Prints ONE JSON line (rank 0).  ``--impl reference`` times the fp64 CPU oracle instead on a
bounded sample of the same workload.  Multi-GPU (torchrun): by default every rank runs its own
independent sequence (weak scaling, no collective on the data path); ``--mode seq`` splits one
sequence over the ranks instead (strong scaling: each rank summarises its contiguous range, one
all_gather exchanges the fp32 segment summaries, every rank scans them in order and re-emits
its own range).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

T_FULL, HK, HV, KD, VD, C = 65536, 16, 32, 128, 128, 64
METRIC = "GDN fwd tokens/s at T=65536, Hv=32, K=V=128; % of roofline (tensor pipe)"
# Algorithmic work per token (independent of P): 2*[C(3K+2V) + 3KV + C^2/6] FLOP per value
# head, and q + k + v + out (bf16) + g + beta (fp32) bytes.
FLOP_PER_TOKEN = 2 * (C * (3 * KD + 2 * VD) + 3 * KD * VD + C * C / 6) * HV
BYTES_PER_TOKEN = HK * KD * 2 * 2 + HV * VD * 2 * 2 + HV * 4 * 2
# what each phase-1 kernel must read per token: k, v, g, beta (U half); k, g, beta (M half)
SUM_U_BYTES_PER_TOKEN = HK * KD * 2 + HV * VD * 2 + HV * 4 * 2
SUM_M_BYTES_PER_TOKEN = HK * KD * 2 + HV * 4 * 2
# backward (state recurrences and triangular factors on fp32 CUDA cores, products on TF32 tensor
# cores): FLOPs per token of what it computes -- per chunk and value head 6 CKV + 6 C^2 K +
# 3 C^2 V products and two C x C triangular solves over V columns, per token and value head the
# two state-column recurrences (2 KV + 3 KV multiply-adds)
BWD_FLOP_PER_TOKEN = HV * (2 * (6 * C * KD * VD + 6 * C * C * KD + 3 * C * C * VD
                                 + C * (C - 1) * VD) / C + 2 * 5 * KD * VD)
# fp32 FMA peak of the CUDA cores: 152 SMs x 128 lanes x 2 FLOP x 2.07 GHz (maximum SM clock)
FP32_ALU_TFLOPS = 152 * 128 * 2 * 2.07e9 / 1e12
BWD_STEPS = 5
# prologue: bytes per token it must move (x read, q, k, v written in bf16; a, b read in bf16;
# g, beta written in fp32); W = 4 taps, SiLU
CH = 2 * HK * KD + HV * VD
PRO_BYTES_PER_TOKEN = CH * 2 * 2 + HV * 2 * 2 + HV * 4 * 2
# decode: requests per step, slots in the state pool, timed steps; bytes one step must move
# (each request's fp32 state read and written once per value head, q, k, v, out, g, beta, slot)
DEC_B, DEC_SLOTS, DEC_STEPS = 256, 256, 200
DEC_BYTES = (DEC_B * HV * KD * VD * 4 * 2 + DEC_B * HK * KD * 2 * 2 + DEC_B * HV * VD * 2 * 2
             + DEC_B * HV * 4 * 2 + DEC_B * 4)


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), float(
            d.get("bf16_tflops_sustained", d["bf16_tflops"])), "measured"
    except (OSError, KeyError, ValueError):
        return 6800.0, 1900.0, 1700.0, "fallback"


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


class Clocks:
    """Samples the SM clock and the clock-event (throttle) reasons of the benchmark's GPU while the
    timed region runs.  Read-only NVML queries through ctypes every ~2 ms in a thread (so that a
    short timed region still gets many samples); `nvidia-smi -lms 20` when NVML cannot be
    loaded."""

    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}

    def __init__(self, index, period_s=0.002):
        self.index = index
        self.period = period_s
        self.samples = []      # (sm_mhz, reasons bitmask)
        self.max_mhz = None
        self.source = None
        self.proc = None
        self._thread = None
        self._stop = None

    def _nvml_handle(self):
        import ctypes
        lib = ctypes.CDLL("libnvidia-ml.so.1")
        if lib.nvmlInit_v2() != 0:
            raise OSError("nvmlInit failed")
        dev = ctypes.c_void_p()
        try:  # the CUDA device's PCI address names the same GPU in NVML
            import torch
            pr = torch.cuda.get_device_properties(self.index)
            bus = f"{pr.pci_domain_id:08x}:{pr.pci_bus_id:02x}:{pr.pci_device_id:02x}.0".encode()
            if lib.nvmlDeviceGetHandleByPciBusId_v2(bus, ctypes.byref(dev)) != 0:
                raise OSError("no NVML device at " + bus.decode())
        except (AttributeError, OSError):
            if lib.nvmlDeviceGetHandleByIndex_v2(self.index, ctypes.byref(dev)) != 0:
                raise OSError("no NVML device")
        return lib, dev

    def __enter__(self):
        import ctypes
        import threading
        try:
            lib, dev = self._nvml_handle()
            mx = ctypes.c_uint()
            if lib.nvmlDeviceGetMaxClockInfo(dev, 1, ctypes.byref(mx)) == 0:
                self.max_mhz = float(mx.value)
            reasons_fn = getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
                lib.nvmlDeviceGetCurrentClocksThrottleReasons
            self._stop = threading.Event()

            def run():
                mhz, rs = ctypes.c_uint(), ctypes.c_ulonglong()
                while not self._stop.is_set():
                    if (lib.nvmlDeviceGetClockInfo(dev, 1, ctypes.byref(mhz)) == 0 and
                            reasons_fn(dev, ctypes.byref(rs)) == 0):
                        self.samples.append((float(mhz.value), int(rs.value)))
                    time.sleep(self.period)

            self._thread = threading.Thread(target=run, daemon=True)
            self._thread.start()
            self.source = "nvml"
        except (OSError, AttributeError):
            try:
                self.proc = subprocess.Popen(
                    ["nvidia-smi", f"--id={self.index}",
                     "--query-gpu=clocks.sm,clocks.max.sm,clocks_event_reasons.hw_slowdown,"
                     "clocks_event_reasons.hw_thermal_slowdown,"
                     "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap",
                     "--format=csv,noheader,nounits", "-lms", "20"],
                    stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
                self.source = "nvidia-smi"
            except OSError:
                self.proc = None
        return self

    def __exit__(self, *exc):
        if self._thread is not None:
            self._stop.set()
            self._thread.join(timeout=2)
        if self.proc is not None:
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            bits = (0x8, 0x40, 0x20, 0x4)
            for ln in out.splitlines():
                f = [x.strip() for x in ln.split(",")]
                if len(f) < 6:
                    continue
                try:
                    self.max_mhz = float(f[1])
                    mask = sum(b for b, v in zip(bits, f[2:6]) if v.lower() == "active")
                    self.samples.append((float(f[0]), mask))
                except ValueError:
                    continue
        return False

    def summary(self):
        if not self.samples:
            return None
        reasons = sorted({name for _, m in self.samples for bit, name in self.REASONS.items()
                          if m & bit})
        return {"sm_mhz": statistics.median(x for x, _ in self.samples),
                "sm_max_mhz": self.max_mhz, "samples": len(self.samples), "reasons": reasons,
                "source": self.source}


def make_inputs(T, device, seed):
    from gated_delta_rule_07_gb300 import inputs
    inp = inputs.make(inputs.long_bf16(T=T, seed=seed))
    return inp


TC5_SOURCES = ("gdn_tc5.cu", "gdn_tc5_util.cuh", "gdn_sm100.cuh", "gdn_common.cuh",
               "gdn_warp_mma.cuh")


def source_hash(names=TC5_SOURCES):
    h = hashlib.sha256()
    for name in names:
        with open(os.path.join(ROOT, "gated_delta_rule_07_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def stored_traffic(kernel):
    """DRAM bytes per token (decode: per request) of `kernel` from the committed ncu summary,
    if the kernel's sources have not changed since it was captured (else None)."""
    try:
        with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
            d = json.load(f)
        e = d[kernel]
        if e.get("source_sha") != source_hash(tuple(e.get("sources", TC5_SOURCES))):
            return None
        return float(e["dram_bytes_per_token"])
    except (OSError, KeyError, ValueError):
        return None


# ------------------------------------------------------------------------------ our arm

def run_seq_sharded(args, ws, rank, local):
    """One T-token sequence split by sequence over the ranks (strong scaling): each rank
    summarises its contiguous range (P segments), one NCCL all_gather exchanges the fp32
    summaries, every rank scans all ranks' segments in order and re-emits its own range."""
    import torch
    import torch.distributed as dist
    from gated_delta_rule_07_gb300 import build, sharding
    build.build()
    from gated_delta_rule_07_gb300 import gdn

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    dist.init_process_group("nccl", device_id=dev)
    T = args.T
    P = args.P or 4
    inp = make_inputs(T, dev, seed=0)
    t0, t1 = sharding.sequence_partition(T, ws, rank)
    d = {n: getattr(inp, n)[t0:t1].to(dev).contiguous() for n in ("q", "k", "v", "g", "beta")}
    summary, scan, emit = sharding.gpu_steps(gdn)

    def step():
        return sharding.sequence_parallel_forward(d["q"], d["k"], d["v"], d["g"], d["beta"], None,
                                                  summary=summary, scan=scan, emit=emit,
                                                  P_local=P)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    dist.barrier()
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with Clocks(local) as clk:
        e0.record(stream)
        for _ in range(args.steps):
            step()
        e1.record(stream)
        torch.cuda.synchronize()
    dist.barrier()
    ms = torch.tensor([e0.elapsed_time(e1) / args.steps], device=dev)
    dist.all_reduce(ms, op=dist.ReduceOp.MAX)
    ms = float(ms.item())
    if rank != 0:
        return None
    return {"metric": METRIC, "value": T / (ms / 1e3), "unit": "tokens/s", "n_gpus": ws,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
            "higher_is_better": True, "scaling": "strong", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic (seeded, as the default mode)",
            "config": {"workload": f"long-context bf16 T={T} Hk={HK} Hv={HV} K=V={KD} C={C}",
                       "segments_per_rank": P, "batch": 1, "seq_len": T,
                       "parallelism": f"sequence-sharded x{ws} (all_gather of fp32 segment "
                                      f"summaries, {sharding.exchange_bytes(HV, KD, VD, P)} B "
                                      f"per rank)"},
            "gpu_launches": None, "e2e": None, "clocks": clk.summary()}


def run_ours(args, ws, rank, local):
    import torch
    from gated_delta_rule_07_gb300 import build
    build.build()
    from gated_delta_rule_07_gb300 import gdn

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    T = args.T
    inp = make_inputs(T, dev, seed=rank)
    d = {n: getattr(inp, n).to(dev).contiguous() for n in ("q", "k", "v", "g", "beta")}
    out = torch.empty_like(d["v"])
    hf = torch.empty(1, HV, KD, VD, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream()

    def barrier():
        torch.cuda.synchronize()
        if ws > 1:
            import torch.distributed as dist
            dist.barrier()
        torch.cuda.synchronize()

    def timed_forward(P, steps, warmup):
        p = gdn.problem_for(d["q"], d["v"], None, P=P)
        wsb = gdn.workspace_for(p, dev)
        for _ in range(warmup):
            gdn.gdn_forward(p, d["q"], d["k"], d["v"], d["g"], d["beta"], None, None, out, hf,
                            wsb)
        barrier()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(steps):
            gdn.gdn_forward(p, d["q"], d["k"], d["v"], d["g"], d["beta"], None, None, out, hf,
                            wsb)
        e1.record(stream)
        barrier()
        st = gdn.gdn_device_status(wsb)
        if st != 0:
            raise gdn.GdnError(st, "device status")
        return e0.elapsed_time(e1) / steps

    # P sweep (short), then the timed run at the chosen P
    sweep = {}
    Ps = [args.P] if args.P else [1, 2, 3, 4, 5, 6, 8, 16, 64]
    for P in Ps:
        ms = timed_forward(P, steps=3 if len(Ps) > 1 else 1, warmup=1)
        sweep[P] = ms
    P_best = args.P or min(sweep, key=sweep.get)

    with Clocks(local) as clk:
        ms = timed_forward(P_best, args.steps, args.warmup)
    if ws > 1:
        import torch.distributed as dist
        t = torch.tensor([ms], device=dev)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        ms = float(t.item())

    # per-phase times of the forward itself: CUDA events between its launches
    p = gdn.problem_for(d["q"], d["v"], None, P=P_best)
    wsp = gdn.workspace_for(p, dev)
    phase_ms = {"summary": [], "scan": [], "emit": [], "summary_first": []}
    for it in range(args.warmup + args.steps):
        sm_, sc_, em_, s1_ = gdn.gdn_forward_timed(p, d["q"], d["k"], d["v"], d["g"], d["beta"],
                                                   None, None, out, hf, wsp, stream=stream)
        if it >= args.warmup:
            phase_ms["summary"].append(sm_)
            phase_ms["scan"].append(sc_)
            phase_ms["emit"].append(em_)
            phase_ms["summary_first"].append(s1_)
    ph = {k: statistics.mean(v) for k, v in phase_ms.items()}

    # end to end through the C ABI with host buffers: every step copies its inputs in from
    # pinned host memory, runs the forward and reads its outputs back.  Steps are pipelined over
    # two sets of device buffers: the input copies on two streams (q, k, g, beta and v, about
    # half the bytes each, so that two copy engines work at once), the forward on its own, the
    # output copies in two halves on two more, so one step's copies overlap its neighbours'
    # work.
    host = {n: d[n].cpu().pin_memory() for n in d}
    out_h = [torch.empty(out.shape, dtype=out.dtype).pin_memory() for _ in range(2)]
    hf_h = [torch.empty(hf.shape, dtype=hf.dtype).pin_memory() for _ in range(2)]
    h2d = sum(t.numel() * t.element_size() for t in host.values())
    d2h = out_h[0].numel() * out_h[0].element_size() + hf_h[0].numel() * hf_h[0].element_size()
    pe = gdn.problem_for(d["q"], d["v"], None, P=P_best)
    wse = gdn.workspace_for(pe, dev)
    dd = [{n: torch.empty_like(d[n]) for n in d} for _ in range(2)]
    outs = [torch.empty_like(out) for _ in range(2)]
    hfs = [torch.empty_like(hf) for _ in range(2)]
    groups = (("q", "k", "g", "beta"), ("v",))
    s_in = [torch.cuda.Stream() for _ in groups]
    s_out = [torch.cuda.Stream() for _ in range(2)]
    ev_in = [[torch.cuda.Event() for _ in s_in] for _ in range(2)]    # inputs on the device
    ev_cmp = [torch.cuda.Event() for _ in range(2)]                   # forward done
    ev_out = [[torch.cuda.Event() for _ in s_out] for _ in range(2)]  # outputs on the host
    half = out.shape[0] // 2

    def e2e_step(i):
        b = i & 1
        for s, names, ev in zip(s_in, groups, ev_in[b]):
            with torch.cuda.stream(s):
                s.wait_event(ev_cmp[b])  # the forward two steps back has read these buffers
                for n in names:
                    dd[b][n].copy_(host[n], non_blocking=True)
                ev.record(s)
        for ev in ev_in[b] + ev_out[b]:  # (its outputs two steps back have been read out)
            stream.wait_event(ev)
        gdn.gdn_forward(pe, dd[b]["q"], dd[b]["k"], dd[b]["v"], dd[b]["g"], dd[b]["beta"], None,
                        None, outs[b], hfs[b], wse, stream=stream)
        ev_cmp[b].record(stream)
        for k, s in enumerate(s_out):
            with torch.cuda.stream(s):
                s.wait_event(ev_cmp[b])
                rows = slice(0, half) if k == 0 else slice(half, out.shape[0])
                out_h[b][rows].copy_(outs[b][rows], non_blocking=True)
                if k == 1:
                    hf_h[b].copy_(hfs[b], non_blocking=True)
                ev_out[b][k].record(s)

    for i in range(args.warmup):
        e2e_step(i)
    torch.cuda.synchronize()
    barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for s in s_in:
        s.wait_event(e0)
    for i in range(args.steps):
        e2e_step(args.warmup + i)
    for evs in ev_out:
        for ev in evs:
            stream.wait_event(ev)
    e1.record(stream)
    torch.cuda.synchronize()
    barrier()
    e2e_ms = e0.elapsed_time(e1) / args.steps

    # the decode step: one token per request over a pool of per-slot states (every step reads
    # and writes each named slot's fp32 state once; the pool is larger than L2)
    from gated_delta_rule_07_gb300 import inputs as inputs_mod
    dec = inputs_mod.decode_batch(DEC_B, DEC_SLOTS, HK, HV, KD, VD, seed=rank)
    dd_ = {n: getattr(dec, n).to(dev).contiguous() for n in ("q", "k", "v", "g", "beta", "slot",
                                                              "state")}
    dec_out = torch.empty_like(dd_["v"])
    dec_st = torch.zeros(1, dtype=torch.int32, device=dev)
    dp = gdn.decode_problem_for(dd_["q"], dd_["v"], dd_["state"])

    def dec_step():
        gdn.gdn_decode_step(dp, dd_["q"], dd_["k"], dd_["v"], dd_["g"], dd_["beta"], dd_["slot"],
                            dd_["state"], dec_out, dec_st, stream=stream)

    for _ in range(max(args.warmup, 3)):
        dec_step()
    barrier()
    e0.record(stream)
    for _ in range(DEC_STEPS):
        dec_step()
    e1.record(stream)
    barrier()
    dec_us = e0.elapsed_time(e1) / DEC_STEPS * 1e3
    st = gdn.gdn_device_status(dec_st)
    if st != 0:
        raise gdn.GdnError(st, "decode device status")
    del dd_

    # the backward at the same workload: gradients of <dout, out> through the forward
    gen = torch.Generator().manual_seed(100 + rank)
    dout = torch.randn(d["v"].shape, generator=gen).to(torch.bfloat16).to(dev)
    pb = gdn.problem_for(d["q"], d["v"], None)
    bws = torch.empty(gdn.gdn_backward_workspace_size(pb), dtype=torch.uint8, device=dev)
    bo = [torch.empty_like(d["q"]), torch.empty_like(d["k"]), torch.empty_like(d["v"]),
          torch.empty_like(d["g"]), torch.empty_like(d["beta"])]

    def bwd_step():
        gdn.gdn_backward(pb, d["q"], d["k"], d["v"], d["g"], d["beta"], None, None, dout, None,
                         *bo, None, bws, stream=stream)

    bwd_step()
    barrier()
    e0.record(stream)
    for _ in range(BWD_STEPS):
        bwd_step()
    e1.record(stream)
    barrier()
    bwd_ms = e0.elapsed_time(e1) / BWD_STEPS
    st = gdn.gdn_device_status(bws)
    if st != 0:
        raise gdn.GdnError(st, "backward device status")
    del bws, bo, dout

    # the prologue at the same workload: q, k, v, g, beta from projection-shaped inputs
    gen = torch.Generator().manual_seed(200 + rank)
    px = torch.randn(T, CH, generator=gen).to(torch.bfloat16).to(dev)
    pw = (torch.randn(CH, 4, generator=gen) * 0.5).to(dev)
    pab = torch.randn(2, T, HV, generator=gen).to(torch.bfloat16).to(dev)
    pal = torch.full((HV,), -2.3, device=dev)
    pdt = torch.zeros(HV, device=dev)
    pp = gdn.PrologueProblem(T, 1, HK, HV, KD, VD, 4, 1, gdn.GDN_BF16)
    po = [torch.empty_like(d["q"]), torch.empty_like(d["k"]), torch.empty_like(d["v"]),
          torch.empty_like(d["g"]), torch.empty_like(d["beta"])]

    def pro_step():
        gdn.gdn_prologue(pp, px, pw, None, pab[0], pab[1], pal, pdt, None, *po, None,
                         stream=stream)

    for _ in range(3):
        pro_step()
    barrier()
    e0.record(stream)
    for _ in range(20):
        pro_step()
    e1.record(stream)
    barrier()
    pro_ms = e0.elapsed_time(e1) / 20
    del px, pab, po

    if rank != 0:
        return None
    hbm, tf, tf_sus, src = peaks()
    tokens = T * ws
    # the launches of one forward, their times and what each must move (algorithmic bytes)
    kern_ms = {"emit": ph["emit"]}
    if P_best > 1:  # phase 1 = the U half (writes the factor records), then the M half
        kern_ms["sum_u"] = ph["summary_first"]
        kern_ms["sum_m"] = ph["summary"] - ph["summary_first"]
    kern_bytes = {
        "emit": BYTES_PER_TOKEN * T + (P_best * HV + HV) * KD * VD * 4,
        "sum_u": SUM_U_BYTES_PER_TOKEN * T + P_best * HV * KD * VD * 4,
        "sum_m": SUM_M_BYTES_PER_TOKEN * T * (P_best - 1) // P_best + (P_best - 1) * HV * KD * KD * 4,
    }
    kern_name = {
        "emit": ("chunk kernel <emit from records> (phase 3: attn_i + chain + output)"
                 if P_best > 1 else "chunk kernel <emit> (prepare + chain + output)"),
        "sum_u": "chunk kernel <U summary> (phase 1: prepare + U chain + factor records)",
        "sum_m": "chunk kernel <M summary from records> (phase 1: M chain)",
    }
    kern_traffic_key = {"emit": "emit_records" if P_best > 1 else "emit",
                        "sum_u": "sum_u_records", "sum_m": "sum_m_records"}
    dom = max(kern_ms, key=kern_ms.get)
    emit_bytes = kern_bytes[dom]
    emit_s = kern_ms[dom] / 1e3
    achieved_gbs = emit_bytes / emit_s / 1e9
    tr = stored_traffic(kern_traffic_key[dom])
    t_bound = max(BYTES_PER_TOKEN * T / (hbm * 1e9), FLOP_PER_TOKEN * T / (tf * 1e12))
    launches_per_step = 4 if P_best > 1 else 1  # summary (M and U halves), scan, emit
    res = {
        "metric": METRIC,
        "value": tokens / (ms / 1e3),
        "unit": "tokens/s",
        "n_gpus": ws,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": ms,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic (seeded; q,k L2-normalised N(0,1), v N(0,1), g=-softplus(N)*0.1, "
                "beta=sigmoid(N), h0=0)",
        "config": {"workload": f"long-context bf16 T={T} Hk={HK} Hv={HV} K=V={KD} C={C}",
                   "segments_per_seq": P_best, "batch": 1, "seq_len": T,
                   "parallelism": f"replicas x{ws} (independent sequences)",
                   "l2": f"inputs+output {BYTES_PER_TOKEN * T / 1e9:.2f} GB vs 129 MB L2" + ("; no flush" if BYTES_PER_TOKEN * T > 129e6 else "; L2-resident"),
                   "kernel_family": args.family},
        "sweep_ms_per_step": {f"P={k}": round(v, 4) for k, v in sweep.items()},
        "phase_ms": {k: round(v, 4) for k, v in ph.items()},
        "gpu_launches": launches_per_step * args.steps,
        "kernels_ms": {k: round(v, 4) for k, v in kern_ms.items()},
        "roofline": {
            "kernel": kern_name[dom] + " -- the longest launch of the step",
            "bound": "hbm", "achieved": achieved_gbs, "peak": hbm, "unit": "GB/s",
            "frac": achieved_gbs / hbm, "peak_source": src,
            "traffic": None if tr is None else tr * T,
            "algorithmic_bytes_per_launch": emit_bytes},
        "roofline_by_kernel": {
            k: {"ms": round(kern_ms[k], 4), "algorithmic_bytes": kern_bytes[k],
                "achieved_gbs": kern_bytes[k] / (kern_ms[k] / 1e3) / 1e9,
                "frac": kern_bytes[k] / (kern_ms[k] / 1e3) / 1e9 / hbm}
            for k in kern_ms},
        "path_roofline": {"bound_us": t_bound * 1e6, "step_us": ms * 1e3,
                          "frac": t_bound / (ms / 1e3),
                          "note": "max(FLOP/bf16 peak, bytes/HBM) over the whole step, of "
                                  + src},
        "e2e": {"value": tokens / (e2e_ms / 1e3), "unit": "tokens/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms,
                "pipelining": "copies in on two streams, the forward, copies out on two more, "
                              "over two buffer sets"},
        "clocks": clk.summary(),
        "backward": {
            "workload": f"long-context bf16 T={T} Hk={HK} Hv={HV} K=V={KD}: gradients of q, k, "
                        "v, g, beta, h0 for a random dout",
            "ms_per_step": bwd_ms, "tokens_per_s": T / (bwd_ms / 1e3), "steps": BWD_STEPS,
            "gpu_launches_per_step": 3,
            "roofline": {"bound": "alu", "unit": "TFLOP/s",
                         "achieved": BWD_FLOP_PER_TOKEN * T / (bwd_ms / 1e3) / 1e12,
                         "peak": FP32_ALU_TFLOPS,
                         "frac": BWD_FLOP_PER_TOKEN * T / (bwd_ms / 1e3) / 1e12 / FP32_ALU_TFLOPS,
                         "peak_source": "fp32 FMA units x maximum SM clock (not measured)",
                         "algorithmic_flop_per_step": BWD_FLOP_PER_TOKEN * T,
                         "traffic": None}},
        "prologue": {
            "workload": f"conv (4 taps, SiLU) + L2 norm + g, beta: T={T}, {CH} channels, "
                        f"Hk={HK} Hv={HV} K=V={KD} bf16",
            "ms_per_step": pro_ms, "tokens_per_s": T / (pro_ms / 1e3), "steps": 20,
            "gpu_launches_per_step": 1,
            "roofline": {"kernel": "prologue_kernel", "bound": "hbm",
                         "achieved": PRO_BYTES_PER_TOKEN * T / (pro_ms / 1e3) / 1e9,
                         "peak": hbm, "unit": "GB/s",
                         "frac": PRO_BYTES_PER_TOKEN * T / (pro_ms / 1e3) / 1e9 / hbm,
                         "peak_source": src,
                         "algorithmic_bytes_per_launch": PRO_BYTES_PER_TOKEN * T,
                         "traffic": (None if stored_traffic("prologue") is None
                                     else stored_traffic("prologue") * T)}},
        "decode": {
            "workload": f"decode bf16 B={DEC_B} requests, pool of {DEC_SLOTS} slots, Hk={HK} "
                        f"Hv={HV} K=V={KD}; fp32 state pool "
                        f"{DEC_SLOTS * HV * KD * VD * 4 / 2**20:.0f} MiB (> L2)",
            "us_per_step": dec_us, "tokens_per_s": DEC_B / (dec_us / 1e6), "steps": DEC_STEPS,
            "gpu_launches_per_step": 1,
            "roofline": {"kernel": "decode_kernel (one CTA per request and value head)",
                         "bound": "hbm", "achieved": DEC_BYTES / (dec_us / 1e6) / 1e9,
                         "peak": hbm, "unit": "GB/s",
                         "frac": DEC_BYTES / (dec_us / 1e6) / 1e9 / hbm, "peak_source": src,
                         "algorithmic_bytes_per_launch": DEC_BYTES,
                         "traffic": (None if stored_traffic("decode") is None
                                     else stored_traffic("decode") * DEC_B)}},
    }
    if not args.no_cpu_baseline:
        res["cpu_baseline"] = cpu_baseline(args.cpu_seconds, inp=inp)
    return res


# ------------------------------------------------------------------------ oracle arm

def cpu_baseline(seconds=12.0, T=None, inp=None):
    """Times the fp64 oracle (as it stands) on a bounded sample of the workload: the first
    Ts tokens, all 32 value heads, sized from a short calibration to ~`seconds` of work."""
    import oracle
    if inp is None:
        inp = make_inputs(T_FULL if T is None else T, "cpu", seed=0)
    threads = os.cpu_count() or 1

    def run(n):
        sl = {nm: getattr(inp, nm)[:n] for nm in ("q", "k", "v", "g", "beta")}
        t0 = time.perf_counter()
        oracle.token(**sl, nthreads=threads)
        return time.perf_counter() - t0

    cal = 256
    dt = run(cal)
    Ts = int(min(inp.q.shape[0], max(cal, cal * seconds / max(dt, 1e-6))))
    Ts = max(64, Ts // 64 * 64)
    dt = run(Ts)
    return {"value": Ts / dt, "unit": "tokens/s", "cores": threads, "kind": "oracle",
            "sample": f"first {Ts} tokens of the T=65536 stream, all 32 value heads, fp64 "
                      f"per-token recurrence ({dt:.1f} s)"}


def run_reference(args, ws, rank):
    if rank != 0:
        return None
    import oracle
    inp = make_inputs(T_FULL, "cpu", seed=0)
    threads = os.cpu_count() or 1
    Ts = args.ref_tokens
    sl = {nm: getattr(inp, nm)[:Ts] for nm in ("q", "k", "v", "g", "beta")}
    for _ in range(args.warmup):
        oracle.token(**sl, nthreads=threads)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.token(**sl, nthreads=threads)
    dt = (time.perf_counter() - t0) / args.steps
    v = Ts / dt
    return {"impl": "reference", "metric": METRIC, "value": v, "unit": "tokens/s",
            "n_gpus": ws, "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (same recipe and seed as our arm)",
            "config": {"workload": f"long-context bf16 T={T_FULL} Hk={HK} Hv={HV} K=V={KD} "
                                   f"C={C}", "sample_tokens": Ts},
            "cpu_baseline": {"value": v, "unit": "tokens/s", "cores": threads, "kind": "oracle",
                             "sample": f"first {Ts} tokens, all 32 value heads, per step"},
            "e2e": {"value": v, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--P", type=int, default=0, help="segments per sequence (0 = sweep)")
    ap.add_argument("--T", type=int, default=T_FULL)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--ref-tokens", type=int, default=2048)
    ap.add_argument("--mode", default="replicas", choices=["replicas", "seq"],
                    help="with several ranks: independent sequences (weak scaling) or one "
                         "sequence split by sequence over the ranks (strong scaling)")
    args = ap.parse_args()
    args.family = "tcgen05 (TMEM accumulators, fp16 operands, fp32 state)"
    if args.warmup < 3:
        args.warmup = 3
    ws, rank, local = dist_env()
    if args.impl == "reference":
        res = run_reference(args, ws, rank)
    else:
        res = (run_seq_sharded(args, ws, rank, local) if args.mode == "seq" and ws > 1
               else run_ours(args, ws, rank, local))
    if res is not None:
        print(json.dumps(res), flush=True)


if __name__ == "__main__":
    main()
