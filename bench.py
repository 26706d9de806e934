#!/usr/bin/env python3
"""Benchmark of the packed FP8 QKV projection, forward + backward, on GB300.

One step = one pass of the whole hot path over one batch: the per-update bank
refresh of the layer (amax + dual-layout quantisation, on a side stream beside
the x quantisation, which it does not depend on), the forward (x amax and
quantisation, packed GEMM with the fused split/RMSNorm/RoPE epilogue) and
the backward (dY amax, dY quantisation, dX GEMM, dW GEMM with its split reduction).
Workload: 6 sequences x 8192 tokens (T = 49152), D = 768, H = 6, d_qk = 96,
d_v = 128, synthetic seeded inputs.

Prints one JSON line (rank 0).  `--impl reference` times the plain CPU oracle
on the host cores instead, each step one bounded sample of the same workload.
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

import torch  # noqa: E402

import synth  # noqa: E402

METRIC = "packed-QKV fwd+bwd tokens/s"
KERNELS = ["bank_refresh", "x_quant", "fwd_gemm", "dy_amax", "dy_quant", "dx_gemm", "dw_gemm"]
# event index pairs bracketing each kernel (see qkvp_set_timing_events); the
# bank refresh runs on a side stream beside the x quantisation
SPANS = [(0, 1), (2, 3), (4, 5), (6, 7), (7, 8), (8, 9), (9, 10)]
EVENTS_PER_STEP = 11


def algorithmic_work(s: synth.Shape):
    """Bytes (HBM-bound kernels) or FLOPs (GEMMs) one launch must move or do."""
    T, D, H, dqk, dv, N = s.T, s.D, s.H, s.d_qk, s.d_v, s.N
    bank = N * D * 2
    q_bytes = H * T * dqk * 2
    v_bytes = H * T * dv * 2
    rstd = 2 * H * T * 4
    bwd_in = 2 * q_bytes + v_bytes + 2 * q_bytes + rstd + T * 4
    flops = 2.0 * T * D * N
    return {
        # the bf16 bank read once, both code layouts written
        "bank_refresh": ("hbm", bank + 2 * N * D),
        # amax and codes in one launch: a per-tensor scale needs every value
        # before the first code, so the method reads x twice (amax, codes)
        # and writes x8, as the two passes of the kernel do
        "x_quant": ("hbm", 2 * T * D * 2 + T * D),
        "fwd_gemm": ("tensor", flops),
        "dy_amax": ("hbm", bwd_in),
        "dy_quant": ("hbm", bwd_in + T * N),
        "dx_gemm": ("tensor", flops),
        "dw_gemm": ("tensor", flops),
    }


# DRAM traffic (dram__bytes_read.sum + dram__bytes_write.sum) per launch from
# ncu captures of the kernels (one kernel per capture), taken at T =
# TRAFFIC["T"] tokens and scaled to the workload by its tokens (no scaling at
# the training shape).  Each figure describes the device code of its
# kernel as it was captured (the digest of the kernel's source file and the
# shared device headers) and is reported as null for any other.
KERNEL_SOURCES = {"bwd": "bwd.cu", "gemm": "gemm.cu", "quant": "quant.cu"}
TRAFFIC = {
    "T": 49152,
    "sources_sha256": {"bwd": "1777f6c32b295348ded47b18b2f2b9085109759253829ccc4ab6266348dc5e1f",
                       "gemm": "c9de075080dc23a9d5634eeef7ed9d35df6004e98cdbcb2d6a71d068e2d946c9",
                       "quant": "270726eee5aada0c53740ecf87baf9304a5be421b85aac7ae31ba42d03c9339b"},
    # mean of two launches of the full-size step; dw_gemm: the GEMM and its
    # split-reduction kernel (one span); bank_refresh: the one-layer refresh
    # of the step
    "bytes": {"dy_amax": ("bwd", 3.099e+08), "dy_quant": ("bwd", 3.811e+08),
              "fwd_gemm": ("gemm", 1.751e+08), "dx_gemm": ("gemm", 1.318e+08),
              "dw_gemm": ("gemm", 1.515e+08), "x_quant": ("quant", 7.901e+07),
              "bank_refresh": ("quant", 2.98e+06)},
}


def sources_sha256(unit: str) -> str:
    """Digest of one kernel source file with the device headers it includes."""
    import hashlib
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "fp8_packed_reduced_gb300", "csrc")
    for path in (os.path.join(csrc, KERNEL_SOURCES[unit]), os.path.join(csrc, "common.cuh"),
                 os.path.join(csrc, "kernels.cuh")):
        h.update(os.path.basename(path).encode())
        h.update(open(path, "rb").read())
    return h.hexdigest()


def traffic_for(kernel: str, T: int):
    entry = TRAFFIC["bytes"].get(kernel)
    if entry is None:
        return None
    unit, b = entry
    if sources_sha256(unit) != TRAFFIC["sources_sha256"][unit]:
        return None
    return round(b * T / TRAFFIC["T"])


def max_over_ranks(x: float, world: int, device) -> float:
    """The largest of the ranks' values of x (the job's time is its slowest rank's)."""
    if world <= 1:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def job_tokens_per_s(tokens_per_rank: int, world: int, ms_per_step: float) -> float:
    """Whole-job throughput: every rank's tokens over the slowest rank's step time."""
    return tokens_per_rank * world / (ms_per_step * 1e-3)


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        p = json.load(open(path))
        return dict(hbm=float(p["hbm_gbs"]), bf16=float(p["bf16_tflops"]),
                    bf16_sus=float(p["bf16_tflops_sustained"]), source="measured")
    except Exception:
        return dict(hbm=6800.0, bf16=1900.0, bf16_sus=1700.0, source="fallback")


class ClockSampler:
    """nvidia-smi clock and throttle-reason samples while the timed region runs."""
    Q = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.t0 = self.t1 = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu=timestamp,{self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None

    def mark(self, which):
        setattr(self, which, time.time())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.1)
        self.proc.terminate()
        out, _ = self.proc.communicate(timeout=10)
        rows = []
        for line in out.strip().splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 8:
                continue
            try:
                rows.append(dict(sm=float(f[1]), smax=float(f[2]), power=float(f[3]),
                                 hw=f[4], hwt=f[5], swt=f[6], pcap=f[7]))
            except ValueError:
                continue
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        busy = [r for r in rows if r["power"] > 0] or rows
        reasons = set()
        for r in busy:
            for key, name in (("hw", "hw_slowdown"), ("hwt", "hw_thermal_slowdown"),
                              ("swt", "sw_thermal_slowdown"), ("pcap", "sw_power_cap")):
                if r[key].lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(r["sm"] for r in busy), "sm_max_mhz": max(r["smax"] for r in busy),
                "samples": len(busy), "reasons": sorted(reasons)}


# ----------------------------------------------------------------------------
# CUDA path
# ----------------------------------------------------------------------------

class Step:
    """Inputs resident in HBM, preallocated outputs and workspace: one call of
    step() runs the whole hot path once on the current stream."""

    def __init__(self, s: synth.Shape, dev):
        import fp8_packed_reduced_gb300 as qk
        self.qk, self.s, self.dev = qk, s, dev
        inp = synth.forward_inputs(s, seed=0, device=dev)
        g = synth.backward_inputs(s, seed=0, device=dev)
        self.layers = [(inp["Wq"], inp["Wk"], inp["Wv"])]
        self.x, self.pos = inp["x"], inp["pos"]
        self.dq, self.dk, self.dv = g["dq"], g["dk"], g["dv"]
        self.table = qk.build_rope_table(s.seq_len, s.d_qk, 10000.0, dev)
        shp = qk.Shape(s.T, s.D, s.H, s.d_qk, s.d_v)
        self.ws = qk.new_workspace(shp, dev)
        N, T, D, H = s.N, s.T, s.D, s.H
        u8, bf = dict(dtype=torch.uint8, device=dev), dict(dtype=torch.bfloat16, device=dev)
        self.bank = (torch.empty((1, N, D), **u8), torch.empty((1, D, N), **u8),
                     torch.empty((1,), dtype=torch.float32, device=dev))
        self.fwd_out = dict(q=torch.empty((H, T, s.d_qk), **bf), k=torch.empty((H, T, s.d_qk), **bf),
                            v=torch.empty((H, T, s.d_v), **bf),
                            rstd=torch.empty((2, H, T), dtype=torch.float32, device=dev),
                            x8=torch.empty((T, D), **u8),
                            x_scale=torch.empty((1,), dtype=torch.float32, device=dev))
        self.bwd_out = dict(dx=torch.empty((T, D), **bf), dW=torch.empty((N, D), **bf),
                            dY8=torch.empty((T, N), **u8),
                            dy_scale=torch.empty((1,), dtype=torch.float32, device=dev))
        self.side = torch.cuda.Stream(dev)
        self.fork, self.bank_done = torch.cuda.Event(), torch.cuda.Event()

    def step(self):
        """Bank refresh on a side stream, concurrently with the quantisation
        of x (the two are independent); the forward GEMM waits for both."""
        qk = self.qk
        main = torch.cuda.current_stream(self.dev)
        self.fork.record(main)
        self.side.wait_event(self.fork)
        with torch.cuda.stream(self.side):
            W8, W8T, ws_ = qk.quantize_bank(self.layers, self.s.H, self.s.d_qk, self.s.d_v, out=self.bank)
            self.bank_done.record(self.side)
        x8, sx = qk.quantize_activation(self.x, self.ws, out=(self.fwd_out["x8"], self.fwd_out["x_scale"]))
        main.wait_event(self.bank_done)
        q, k, v, saved = qk.forward_quantized(x8, sx, self.pos, W8[0], ws_[0:1], self.s.H, self.table, self.s.d_qk,
                                              self.s.d_v, ws=self.ws, out=self.fwd_out)
        qk.backward(self.dq, self.dk, self.dv, saved, W8T[0], ws_[0:1], self.table, ws=self.ws, out=self.bwd_out)


def fp8_peak(peaks):
    """Dense E4M3 peak (TFLOP/s): the burst cuBLAS bf16 figure x 2, the nominal
    E4M3/bf16 ratio.  The burst figure fits a timed region of milliseconds;
    the sustained one is for kernels timed inside seconds-long loops."""
    return 2.0 * peaks["bf16"]


def kernel_table(per, work, peaks):
    """Per-kernel mean time, achieved algorithmic rate and fraction of the
    measured peak (HBM copy GB/s, or burst bf16 x 2 for E4M3 GEMMs)."""
    fp8 = fp8_peak(peaks)
    kern = {}
    for name, (bound, amount) in work.items():
        t = per[name] * 1e-3
        if bound == "hbm":
            ach = amount / t / 1e9
            kern[name] = dict(ms=round(per[name], 5), bound="hbm", achieved=round(ach, 1), unit="GB/s",
                              frac=round(ach / peaks["hbm"], 4))
        else:
            ach = amount / t / 1e12
            kern[name] = dict(ms=round(per[name], 5), bound="tensor", achieved=round(ach, 1), unit="TFLOP/s",
                              frac=round(ach / fp8, 4))
    return kern


def run_ours(args, rank, world):
    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    from fp8_packed_reduced_gb300 import build as b
    b.build()
    import fp8_packed_reduced_gb300 as qk
    if args.cta_pairs is not None:
        qk.set_cta_pairs(args.cta_pairs)
    pairs = qk.set_cta_pairs(0)          # read the mask back
    qk.set_cta_pairs(pairs)
    s = synth.Shape(T=args.T, D=args.D, H=args.H, d_qk=args.dqk, d_v=128, seq_len=args.seq_len)
    st = Step(s, dev)
    stream = torch.cuda.current_stream(dev)

    def barrier():
        if world > 1:
            torch.distributed.barrier()

    for _ in range(args.warmup):
        st.step()
    torch.cuda.synchronize()
    code, where = qk.poll_device_status(st.ws)
    if code != 0:
        raise RuntimeError(f"device status {qk.STATUS.get(code)} from kernel {where}")

    # per-kernel events for every timed step
    events = [[torch.cuda.Event(enable_timing=True) for _ in range(EVENTS_PER_STEP)] for _ in range(args.steps)]
    for ev in events:               # torch creates the CUDA event on its first record
        for e in ev:
            e.record(stream)
    torch.cuda.synchronize()
    assert all(e.cuda_event for ev in events for e in ev)
    # The K timed steps are captured once into one CUDA graph (as a training
    # loop would run them), so host launch overhead stays out of the timing.
    # A second graph of the same K steps has the library record kernel-boundary
    # events between its launches: replayed after the timed region, it gives
    # the per-kernel breakdown.  (Event nodes between kernels break the
    # back-to-back launch of dependent kernels, about 3 us each, so the timed
    # graph has none.)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        for i in range(args.steps):
            st.step()
    graph_ev = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph_ev):
        for i in range(args.steps):
            qk.set_timing_events(events[i])
            st.step()
        qk.set_timing_events([])
    torch.cuda.synchronize()
    graph.replay()                  # one untimed replay each: a graph's first launch uploads it
    graph_ev.replay()
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream(dev)
    sampler = ClockSampler(dev.index)
    sampler.start()
    time.sleep(0.3)
    for _ in range(max(3, args.warmup)):      # keep the GPU busy while the sampler starts
        st.step()
    barrier()
    torch.cuda.synchronize()
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    sampler.mark("t0")
    t_start.record(stream)
    graph.replay()
    t_end.record(stream)
    barrier()
    torch.cuda.synchronize()
    sampler.mark("t1")
    clocks = sampler.stop()
    ms = max_over_ranks(t_start.elapsed_time(t_end) / args.steps, world, dev)
    graph_ev.replay()                # the per-kernel breakdown, after the timed region
    torch.cuda.synchronize()
    code, where = qk.poll_device_status(st.ws)
    if code != 0:
        raise RuntimeError(f"device status {qk.STATUS.get(code)} from kernel {where}")

    # per-kernel average durations (ms)
    per = {k: 0.0 for k in KERNELS}
    for ev in events:
        for name, (a, b_) in zip(KERNELS, SPANS):
            per[name] += ev[a].elapsed_time(ev[b_]) / args.steps
    work = algorithmic_work(s)
    peaks = load_peaks()
    fp8 = fp8_peak(peaks)
    kern = kernel_table(per, work, peaks)
    for name in kern:                # DRAM bytes per launch from the ncu captures (null if not this build's)
        kern[name]["traffic"] = traffic_for(name, s.T)
    dom = max(KERNELS, key=lambda k: per[k])
    bound, amount = work[dom]
    roofline = dict(kernel=dom, bound=bound, achieved=kern[dom]["achieved"],
                    peak=peaks["hbm"] if bound == "hbm" else round(fp8, 1),
                    unit=kern[dom]["unit"], frac=kern[dom]["frac"], traffic=traffic_for(dom, s.T),
                    peak_source=(f"{peaks['source']} HBM copy GB/s" if bound == "hbm" else
                                 f"{peaks['source']} burst bf16 x 2 (E4M3 nominal ratio)"),
                    algorithmic=amount)

    e2e = run_e2e(st, args, dev, world)
    line = {
        "metric": METRIC, "value": round(job_tokens_per_s(s.T, world, ms), 1), "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 5), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "e4m3 GEMMs, fp32 accumulate, bf16 I/O",
        "data": "synthetic (seeded N(0,1) activations and gradients, N(0,1/D) weights)",
        "config": {"workload": f"packed QKV fwd+bwd, T={s.T} ({s.T // s.seq_len}x{s.seq_len}), D={s.D}, "
                               f"H={s.H}, d_qk={s.d_qk}, d_v={s.d_v}, bank refresh per step",
                   "T": s.T, "D": s.D, "H": s.H, "d_qk": s.d_qk, "d_v": s.d_v, "parallelism": f"replicas{world}",
                   "l2": "no flush; one step touches ~1.3 GB, 10x the 129 MB L2",
                   "gemm_cta_pairs": pairs},
        "roofline": roofline, "kernels": kern,
        "gpu_launches": (len(KERNELS) + 1) * args.steps,   # + the dW split reduction kernel
        "launch": "the K timed steps replayed as one captured CUDA graph",
        "kernel_timing": "per-kernel means from a second replay of the same K steps with kernel-boundary events "
                         "(each event node adds about 3 us to the span it ends)",
        "clocks": clocks, "e2e": e2e,
    }
    if not args.no_next_rows:
        line["bank_refresh"] = run_bank_refresh(args, dev, load_peaks())
        line["next_rows"] = {"oproj": run_oproj(args, dev, world), "mlp": run_mlp(args, dev, world)}
    if not args.no_sweep:
        line["sweep"] = run_sweep(args, dev, world)
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(s, args.cpu_sample)
    return line


def time_in_graph(step, n_events, steps, warmup, dev, world, ws_list):
    """Run `step` warmup times, capture `steps` calls in one CUDA graph (timed)
    and again with the library's kernel-boundary events (n_events per call;
    replayed after the timed region for the per-kernel breakdown).  Returns
    (ms per step, max over ranks; list of per-call event lists)."""
    import fp8_packed_reduced_gb300 as qk
    for _ in range(max(3, warmup)):
        step()
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream(dev)
    events = [[torch.cuda.Event(enable_timing=True) for _ in range(n_events)] for _ in range(steps)]
    for ev in events:
        for e in ev:
            e.record(stream)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        for i in range(steps):
            step()
    graph_ev = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph_ev):
        for i in range(steps):
            qk.set_timing_events(events[i])
            step()
        qk.set_timing_events([])
    torch.cuda.synchronize()
    graph.replay()
    graph_ev.replay()
    torch.cuda.synchronize()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    graph.replay()
    t1.record(stream)
    torch.cuda.synchronize()
    ms = max_over_ranks(t0.elapsed_time(t1) / steps, world, dev)
    graph_ev.replay()
    torch.cuda.synchronize()
    for ws in ws_list:
        code, where = qk.poll_device_status(ws)
        if code != 0:
            raise RuntimeError(f"device status {qk.STATUS.get(code)} from kernel {where}")
    return ms, events


def span_means(events, kernels, spans):
    per = {k: 0.0 for k in kernels}
    for ev in events:
        for name, (a, b_) in zip(kernels, spans):
            per[name] += ev[a].elapsed_time(ev[b_]) / len(events)
    return per


OPROJ_KERNELS = ["w_refresh", "a_quant", "out_gemm", "g_quant", "da_gemm", "dwo_gemm"]
OPROJ_SPANS = [(0, 1), (2, 3), (3, 4), (5, 6), (6, 7), (7, 8)]
OPROJ_EVENTS = 9


def run_oproj(args, dev, world):
    """The output projection over the V/O bank (weight refresh + forward +
    backward) on the same token count, D = K = H * d_v, timed like the main
    step: K steps captured in one CUDA graph, per-kernel events inside it."""
    import fp8_packed_reduced_gb300 as qk
    T, D, K = args.T, args.D, args.H * 128
    inp = synth.oproj_inputs(T, D, K, seed=0, device=dev)
    u8, bf, f = (dict(dtype=torch.uint8, device=dev), dict(dtype=torch.bfloat16, device=dev),
                 dict(dtype=torch.float32, device=dev))
    wbuf = (torch.empty((1, D, K), **u8), torch.empty((1, K, D), **u8), torch.empty((1,), **f))
    fo = dict(out=torch.empty((T, D), **bf), a8=torch.empty((T, K), **u8), a_scale=torch.empty((1,), **f))
    bo = dict(da=torch.empty((T, K), **bf), dWo=torch.empty((D, K), **bf), dout8=torch.empty((T, D), **u8),
              dout_scale=torch.empty((1,), **f))
    ws = qk.new_oproj_workspace(T, D, K, dev)

    def step():
        W8, W8T, so = qk.quantize_weight([inp["Wo"]], out=wbuf)
        _, a8, sa = qk.oproj_forward(inp["a"], W8[0], so[0:1], ws=ws, out=fo)
        qk.oproj_backward(inp["dout"], W8T[0], so[0:1], a8, sa, ws=ws, out=bo)

    steps = max(3, min(args.steps, 100))
    ms, events = time_in_graph(step, OPROJ_EVENTS, steps, args.warmup, dev, world, [ws])
    per = span_means(events, OPROJ_KERNELS, OPROJ_SPANS)
    flops = 2.0 * T * D * K
    work = {"w_refresh": ("hbm", D * K * 4), "a_quant": ("hbm", T * K * 5),
            "out_gemm": ("tensor", flops), "g_quant": ("hbm", T * D * 5), "da_gemm": ("tensor", flops),
            "dwo_gemm": ("tensor", flops)}
    kern = kernel_table(per, work, load_peaks())
    return {"workload": f"output projection over the V/O bank fwd+bwd, T={T}, D={D}, K=H*d_v={K}, "
                        "weight refresh per step",
            "value": round(job_tokens_per_s(T, world, ms), 1), "unit": "tokens/s", "ms_per_step": round(ms, 5),
            "steps": steps, "kernels": kern, "gpu_launches": (len(OPROJ_KERNELS) + 1) * steps}


MLP_KERNELS = ["w1_refresh", "w2_refresh", "x_quant", "fc_gemm", "h_quant", "proj_gemm",
               "g_quant", "dh_gemm", "dpre_quant", "dx_gemm", "dw1_gemm", "dw2_gemm"]
MLP_SPANS = [(0, 1), (2, 3), (4, 5), (5, 6), (6, 7), (7, 8), (9, 10), (10, 11), (11, 12), (12, 13), (13, 14),
             (14, 15)]
MLP_EVENTS = 16


def run_mlp(args, dev, world):
    """The FP8 ReLU-squared MLP (both weight refreshes + forward + backward) on
    the same token count, hidden width F = 4 D, timed like the main step."""
    import fp8_packed_reduced_gb300 as qk
    T, D = args.T, args.D
    F_ = 4 * D
    inp = synth.mlp_inputs(T, D, F_, seed=0, device=dev)
    u8, f = dict(dtype=torch.uint8, device=dev), dict(dtype=torch.float32, device=dev)
    w1 = (torch.empty((1, F_, D), **u8), torch.empty((1, D, F_), **u8), torch.empty((1,), **f))
    w2 = (torch.empty((1, D, F_), **u8), torch.empty((1, F_, D), **u8), torch.empty((1,), **f))
    ws = qk.new_mlp_workspace(T, D, F_, dev)
    W1_8, W1_8T, s1 = qk.quantize_weight([inp["W1"]], out=w1)
    W2_8, W2_8T, s2 = qk.quantize_weight([inp["W2"]], out=w2)
    fo = qk.mlp_forward(inp["x"], W1_8[0], s1[0:1], W2_8[0], s2[0:1], ws=ws)
    bo = qk.mlp_backward(inp["dout"], W1_8T[0], s1[0:1], W2_8T[0], s2[0:1], fo, ws=ws)

    def step():
        qk.quantize_weight([inp["W1"]], out=w1)
        qk.quantize_weight([inp["W2"]], out=w2)
        qk.mlp_forward(inp["x"], W1_8[0], s1[0:1], W2_8[0], s2[0:1], ws=ws, out=fo)
        qk.mlp_backward(inp["dout"], W1_8T[0], s1[0:1], W2_8T[0], s2[0:1], fo, ws=ws, out=bo)

    steps = max(3, min(args.steps, 50))
    ms, events = time_in_graph(step, MLP_EVENTS, steps, args.warmup, dev, world, [ws])
    per = span_means(events, MLP_KERNELS, MLP_SPANS)
    fl = 2.0 * T * D * F_
    work = {"w1_refresh": ("hbm", F_ * D * 4), "w2_refresh": ("hbm", F_ * D * 4), "x_quant": ("hbm", T * D * 5),
            "fc_gemm": ("tensor", fl), "h_quant": ("hbm", T * F_ * 3), "proj_gemm": ("tensor", fl),
            "g_quant": ("hbm", T * D * 5), "dh_gemm": ("tensor", fl),
            "dpre_quant": ("hbm", T * F_ * 3), "dx_gemm": ("tensor", fl), "dw1_gemm": ("tensor", fl),
            "dw2_gemm": ("tensor", fl)}
    kern = kernel_table(per, work, load_peaks())
    return {"workload": f"FP8 ReLU-squared MLP fwd+bwd, T={T}, D={D}, F={F_}, both weight refreshes per step",
            "value": round(job_tokens_per_s(T, world, ms), 1), "unit": "tokens/s", "ms_per_step": round(ms, 5),
            "steps": steps, "kernels": kern, "gpu_launches": (len(MLP_KERNELS) + 2) * steps}


def run_sweep(args, dev, world, steps=20):
    """The width / scale sweep: the whole step (bank refresh, forward,
    backward) at T tokens for d_qk in {64, 96, 128} (d_v = 128: 256, 320 and
    384 packed columns per head) and D in {768, 1024, 2048} with H = D / 128,
    each timed as `steps` steps replayed from one CUDA graph.  Per D, the
    step-time ratios of the reduced widths against the 384-column layout are
    reported beside the column-count ratios (the work the GEMMs do scales with
    the columns; the bandwidth-bound passes read and write the q, k, v and dY
    columns)."""
    points = []
    for D in (768, 1024, 2048):
        for dqk in (64, 96, 128):
            s = synth.Shape(T=args.T, D=D, H=D // 128, d_qk=dqk, d_v=128, seq_len=args.seq_len)
            st = Step(s, dev)
            stream = torch.cuda.Stream(dev)
            with torch.cuda.stream(stream):
                for _ in range(3):
                    st.step()
            torch.cuda.synchronize()
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph, stream=stream):
                for _ in range(steps):
                    st.step()
            graph.replay()
            torch.cuda.synchronize()
            cur = torch.cuda.current_stream(dev)   # the stream the replays run on
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(cur)
            graph.replay()
            b.record(cur)
            torch.cuda.synchronize()
            code, where = st.qk.poll_device_status(st.ws)
            if code != 0:
                raise RuntimeError(f"device status {st.qk.STATUS.get(code)} from kernel {where}")
            ms = max_over_ranks(a.elapsed_time(b) / steps, world, dev)
            flops = 3 * 2.0 * s.T * s.D * s.N
            points.append({"D": D, "H": s.H, "d_qk": dqk, "cols_per_head": 2 * dqk + 128,
                           "ms_per_step": round(ms, 5), "tokens_per_s": round(job_tokens_per_s(s.T, world, ms), 1),
                           "gemm_tflops_per_step": round(flops / (ms * 1e-3) / 1e12, 1)})
            del graph, st
            torch.cuda.empty_cache()
    ratios = []
    for D in (768, 1024, 2048):
        t = {p_["d_qk"]: p_["ms_per_step"] for p_ in points if p_["D"] == D}
        ratios.append({"D": D, "t320_over_t384": round(t[96] / t[128], 4), "cols_320_over_384": round(320 / 384, 4),
                       "t256_over_t384": round(t[64] / t[128], 4), "cols_256_over_384": round(256 / 384, 4)})
    return {"workload": f"whole step at T={args.T}: d_qk in 64/96/128 (d_v 128), D in 768/1024/2048, H = D/128",
            "steps_per_point": steps, "points": points, "ratios": ratios}


def run_bank_refresh(args, dev, peaks, L=12, copies=8, repeats=32):
    """The weight-bank workload: L layers of the packed bank [N, D] refreshed
    from their bf16 sources in one call (amax, then both code layouts),
    alternating between the weights and a perturbed copy of them (an optimizer
    update).  `repeats` refreshes run back to back in one CUDA graph over
    `copies` separate copies of the bank, each with its own outputs (8 x 70.8
    MB at the default shape, 4.4 x L2), so no refresh finds its inputs in L2:
    every refresh reads its bank from HBM and pays for the write-back of the
    codes earlier refreshes left in L2.  Time per refresh = the graph's time
    over `repeats` (CUDA events on the launching stream)."""
    import fp8_packed_reduced_gb300 as qk
    H, D, dqk, dv = args.H, args.D, args.dqk, 128
    N = H * (2 * dqk + dv)
    u8 = dict(dtype=torch.uint8, device=dev)
    banks, outs = [], []
    for c in range(copies):
        banks.append(synth.bank_layers(L, H, D, dqk, dv, perturb=1e-3 if c % 2 else 0.0, device=dev))
        outs.append((torch.empty((L, N, D), **u8), torch.empty((L, D, N), **u8),
                     torch.empty((L,), dtype=torch.float32, device=dev)))
    stream = torch.cuda.Stream(dev)    # warm-up and capture on one stream: its scratch is made before capture
    with torch.cuda.stream(stream):
        for c in range(copies):
            qk.quantize_bank(banks[c], H, dqk, dv, out=outs[c])
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        for r in range(repeats):
            qk.quantize_bank(banks[r % copies], H, dqk, dv, out=outs[r % copies])
    graph.replay()
    torch.cuda.synchronize()
    cur = torch.cuda.current_stream(dev)   # the stream the replays run on
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(cur)
    graph.replay()
    b.record(cur)
    torch.cuda.synchronize()
    ms = a.elapsed_time(b) / repeats
    moved = L * (N * D * 2 + 2 * N * D)   # bf16 sources read once, both code layouts written
    gbs = moved / (ms * 1e-3) / 1e9
    return {"workload": f"bank refresh, {L} layers x [{N}, {D}] (copies alternating with a perturbed copy)",
            "ms_per_refresh": round(ms, 5), "bytes": moved, "achieved": round(gbs, 1), "unit": "GB/s",
            "frac": round(gbs / peaks["hbm"], 4), "repeats": repeats,
            "l2": f"{repeats} refreshes back to back in one CUDA graph over {copies} copies of the bank with their "
                  f"own outputs ({copies * 2 * moved / 1e6:.0f} MB, more than L2)",
            "gpu_launches": repeats}


def run_e2e(st: Step, args, dev, world):
    """Same metric through the public API with pinned host buffers: every step
    copies the step's inputs host->device and its results device->host.  As an
    input pipeline would, the copies overlap the neighbouring steps' compute:
    two sets of device buffers, the uploads on one stream, the step on a
    second, the downloads on a third, ordered by events (step i's uploads wait
    until step i-2 has finished with that buffer set, its downloads until step
    i has computed)."""
    qk = st.qk
    sets = [st, Step(st.s, dev)]
    torch.cuda.synchronize()   # the second set is built on the default stream
    h = dict(x=st.x.cpu().pin_memory(), dq=st.dq.cpu().pin_memory(), dk=st.dk.cpu().pin_memory(),
             dv=st.dv.cpu().pin_memory(), pos=st.pos.cpu().pin_memory())
    res = dict(q=torch.empty_like(st.fwd_out["q"], device="cpu").pin_memory(),
               k=torch.empty_like(st.fwd_out["k"], device="cpu").pin_memory(),
               v=torch.empty_like(st.fwd_out["v"], device="cpu").pin_memory(),
               dx=torch.empty_like(st.bwd_out["dx"], device="cpu").pin_memory(),
               dW=torch.empty_like(st.bwd_out["dW"], device="cpu").pin_memory())
    h2d = sum(t.numel() * t.element_size() for t in h.values())
    d2h = sum(t.numel() * t.element_size() for t in res.values())
    s_in, s_c, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev = {k: [torch.cuda.Event(), torch.cuda.Event()] for k in ("in", "comp", "out")}

    def one(i):
        b, j = sets[i % 2], i % 2
        with torch.cuda.stream(s_in):
            if i >= 2:
                s_in.wait_event(ev["comp"][j])      # step i-2 is done with these inputs
            b.x.copy_(h["x"], non_blocking=True)
            b.pos.copy_(h["pos"], non_blocking=True)
            b.dq.copy_(h["dq"], non_blocking=True)
            b.dk.copy_(h["dk"], non_blocking=True)
            b.dv.copy_(h["dv"], non_blocking=True)
            ev["in"][j].record(s_in)
        with torch.cuda.stream(s_c):
            s_c.wait_event(ev["in"][j])
            if i >= 2:
                s_c.wait_event(ev["out"][j])        # step i-2's results have been read out
            b.step()
            ev["comp"][j].record(s_c)
        with torch.cuda.stream(s_out):
            s_out.wait_event(ev["comp"][j])
            res["q"].copy_(b.fwd_out["q"], non_blocking=True)
            res["k"].copy_(b.fwd_out["k"], non_blocking=True)
            res["v"].copy_(b.fwd_out["v"], non_blocking=True)
            res["dx"].copy_(b.bwd_out["dx"], non_blocking=True)
            res["dW"].copy_(b.bwd_out["dW"], non_blocking=True)
            ev["out"][j].record(s_out)

    steps = max(3, min(args.steps, 50))
    for i in range(4):
        one(i)
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    # three timed runs of `steps` steps each; the median run is reported (the
    # host link is shared with the machine's other GPUs, and single runs have
    # varied by up to 60 %)
    runs = []
    for _ in range(3):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(s_in)
        for i in range(steps):
            one(i)
        b.record(s_out)
        torch.cuda.synchronize()
        runs.append(a.elapsed_time(b) / steps)
    for b_ in sets:
        code, where = qk.poll_device_status(b_.ws)
        if code != 0:
            raise RuntimeError(f"device status {qk.STATUS.get(code)} from kernel {where}")
    ms = max_over_ranks(sorted(runs)[1], world, dev)
    return {"value": round(job_tokens_per_s(st.s.T, world, ms), 1), "unit": "tokens/s", "ms_per_step": round(ms, 4),
            "steps": steps, "runs_ms_per_step": [round(r, 4) for r in runs], "reported": "median of the three runs",
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "overlap": "uploads, compute and downloads of neighbouring steps on three streams"}


# ----------------------------------------------------------------------------
# CPU oracle (the reference arm and the cpu_baseline leg)
# ----------------------------------------------------------------------------

def oracle_step(s: synth.Shape, inp, g):
    import oracle
    f = synth.to_numpy_f32
    W8, W8T, sw = oracle.quantize_bank(f(inp["Wq"]), f(inp["Wk"]), f(inp["Wv"]))
    pos = inp["pos"].numpy()
    fw = oracle.forward(f(inp["x"]), W8, sw, pos, s.H, s.d_qk, s.d_v)
    oracle.backward(f(g["dq"]), f(g["dk"]), f(g["dv"]), fw["q"], fw["k"], fw["rstd"], pos, W8, sw, fw["x8"],
                    fw["x_scale"], s.H, s.d_qk, s.d_v)


def cpu_baseline(s: synth.Shape, sample_T: int):
    sub = synth.Shape(T=sample_T, D=s.D, H=s.H, d_qk=s.d_qk, d_v=s.d_v, seq_len=s.seq_len)
    inp, g = synth.forward_inputs(sub, 0), synth.backward_inputs(sub, 0)
    t0 = time.perf_counter()
    oracle_step(sub, inp, g)
    dt = time.perf_counter() - t0
    return {"value": round(sample_T / dt, 2), "unit": "tokens/s", "cores": os.cpu_count(), "kind": "oracle",
            "sample": f"first {sample_T} tokens of the workload (bank refresh + fwd + bwd), float64 NumPy, "
                      f"{dt:.2f} s"}


def run_reference(args, rank, world):
    s = synth.Shape(T=args.T, D=args.D, H=args.H, d_qk=args.dqk, d_v=128, seq_len=args.seq_len)
    sub = synth.Shape(T=args.ref_sample, D=s.D, H=s.H, d_qk=s.d_qk, d_v=s.d_v, seq_len=s.seq_len)
    inp, g = synth.forward_inputs(sub, 0), synth.backward_inputs(sub, 0)
    for _ in range(args.warmup):
        oracle_step(sub, inp, g)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle_step(sub, inp, g)
    dt = (time.perf_counter() - t0) / args.steps
    v = round(sub.T / dt, 2)
    sample = f"{sub.T} of the {s.T} tokens per step (bank refresh + fwd + bwd), float64 NumPy"
    return {
        "impl": "reference", "metric": METRIC, "value": v, "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(dt * 1e3, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64 (e4m3 codes emulated)", "data": "synthetic",
        "config": {"workload": f"packed QKV fwd+bwd, T={s.T} ({s.T // s.seq_len}x{s.seq_len}), D={s.D}, "
                               f"H={s.H}, d_qk={s.d_qk}, d_v={s.d_v}, bank refresh per step",
                   "T": s.T, "D": s.D, "H": s.H, "d_qk": s.d_qk, "d_v": s.d_v},
        "cpu_baseline": {"value": v, "unit": "tokens/s", "cores": os.cpu_count(), "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": v, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--T", type=int, default=49152)
    ap.add_argument("--D", type=int, default=768)
    ap.add_argument("--H", type=int, default=6)
    ap.add_argument("--dqk", type=int, default=96)
    ap.add_argument("--seq-len", type=int, default=8192)
    ap.add_argument("--cpu-sample", type=int, default=8192, help="tokens the oracle times for cpu_baseline")
    ap.add_argument("--ref-sample", type=int, default=1024, help="tokens per reference-arm step")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-next-rows", action="store_true",
                    help="skip the bank-refresh, output-projection and MLP measurements")
    ap.add_argument("--no-sweep", action="store_true", help="skip the width / scale sweep")
    ap.add_argument("--cta-pairs", type=int, default=None,
                    help="GEMMs on 2-CTA clusters: bit 0 forward, bit 1 dX, bit 2 dW (default: the library's)")
    args = ap.parse_args()

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args, rank, world)), flush=True)
        return
    if world > 1:
        torch.distributed.init_process_group("nccl")
    line = run_ours(args, rank, world)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
