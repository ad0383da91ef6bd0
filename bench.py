#!/usr/bin/env python3
"""Benchmark of the width-6 speculative-verifier hot path on one GB300.

One step = one pass of every hot-path call over one batch of synthetic input
(weights resident in HBM, seeded synthetic data shaped like the pages'
workloads):
  1. quantize_q8_1   x [6, 5120] -> Q8_1          (shared by gate and up)
  2. qgemv_q4_0_pair gate and up, M=6 K=5120 N=17408 each, one launch on
                     the one Q8_1 activation
  3. quantize_q8_1   h [6, 17408]
  4. qgemv_q4_0      down  M=6 K=17408 N=5120
  5. lmhead_q6_k_top1  draft rows 1..5 of [6, 5120] against the Q6_K
                     [5120, 248320] LM-head -> 5 token ids, no logits
                     (a Q8_1 pre-pass, then the MMVQ with the top-1 epilogue)
  6. quantize_q8_1   target hidden [6, 5120]
  7. qgemv_q6_k      target LM-head M=6 N=248320 (logits)
  8. argmax_f32_rows the 6 target rows -> 6 token ids
About 2.2 GB of weights stream from HBM per step, far more than L2 (129 MB),
so no call finds its weights in L2.

value = effective GB/s: bytes of quantized weights plus activations read by
the calls / step time.  Per-kernel figures (CUDA events on the launching
stream) give the M=6 MMVQ GB/s, the fused LM-head microseconds and the
roofline of the dominant kernel.  `--impl reference` times the CPU oracle on a
bounded sample of the same step instead.
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

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "effective weight GB/s (% of GB300 HBM peak) for M=6 MMVQ; µs per fused LM-head top-1"
UNIT = "GB/s"
K_H, N_FF, N_V = 5120, 17408, 248320
M_T = 6
FALLBACK_HBM_GBS = 6800.0

WORKLOAD = ("width-6 verifier step: Q4_0 gate/up M=6 K=5120 N=17408 (shared Q8_1), Q4_0 down M=6 K=17408 N=5120, "
            "fused Q6_K draft LM-head top-1 rows 1..5 K=5120 N=248320, target Q6_K LM-head M=6 N=248320 + argmax")


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=1000)
    p.add_argument("--warmup", type=int, default=20)
    p.add_argument("--impl", default="native", choices=["native", "reference"])
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--eager", action="store_true",
                   help="launch the step's calls one by one in the timed regions instead of replaying a CUDA graph "
                        "captured from them")
    p.add_argument("--cpu-seconds", type=float, default=12.0, help="bounded oracle sample length")
    p.add_argument("--sweep", action="store_true",
                   help="instead of the step: time qgemv_<format> over M in {1,2,4,6,9,12,17}, K=5120, "
                        "N in {5120, 17408, 248320} for Q4_0, Q6_K, Q8_0, Q4_K, Q5_K (one JSON line per shape)")
    p.add_argument("--sweep-formats", default="q4_0,q6_k,q8_0,q4_k,q5_k", help="sweep: comma-separated formats")
    p.add_argument("--sweep-m", default="1,2,4,6,9,12,17", help="sweep: comma-separated row counts M")
    p.add_argument("--sweep-n", default="5120,17408,248320", help="sweep: comma-separated output sizes N")
    p.add_argument("--sweep-k", type=int, default=5120, help="sweep: the reduction size K")
    p.add_argument("--profile", choices=["mlp", "heads", "topk"], default=None,
                   help="for a profiler: run only the verifier MLP projections (gate/up pair, down), only the "
                        "LM heads (target qgemv_q6_k M=6, fused top-1 M=5, and the tensor-core qgemv_q6_k at M=8), "
                        "or the fused top-1 and top-8 of rows 1..5, --steps times each with an L2 flush between "
                        "calls; prints per-call times, not a bench line")
    return p.parse_args()


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        d = json.load(open(path))
        return float(d["hbm_gbs"]), "measured"
    return FALLBACK_HBM_GBS, "fallback"


# ---------------------------------------------------------------- inputs


def make_inputs(seed_base: int = 0):
    from block_quantized_gemv_quantize_gb300 import synth

    c1 = synth.WORKLOADS["verifier_gate_up"]
    c2 = synth.WORKLOADS["verifier_down"]
    c3 = synth.WORKLOADS["lmhead_q6_k"]
    return dict(
        w_gate=synth.q4_0_weights(N_FF, K_H, seed=c1["seed"]),
        w_up=synth.q4_0_weights(N_FF, K_H, seed=c1["seed"] + 10),
        w_down=synth.q4_0_weights(K_H, N_FF, seed=c2["seed"]),
        w_vocab=synth.q6_k_weights(N_V, K_H, seed=c3["seed"]),
        x=synth.activations(M_T, K_H, seed=c1["seed"] + 100, outlier_frac=0.01),
        h=synth.activations(M_T, N_FF, seed=c2["seed"] + 100, outlier_frac=0.01),
        x_draft=synth.activations(6, K_H, seed=c3["seed"] + 100),
        x_target=synth.activations(M_T, K_H, seed=c3["seed"] + 200),
    )


def step_bytes():
    """Algorithmic bytes read per call (quantized weights + activations)."""
    from block_quantized_gemv_quantize_gb300 import ops

    q4 = ops.q4_0_pack_bytes(N_FF, K_H)
    q6 = ops.q6_k_pack_bytes(N_V, K_H)
    return {
        "quantize_x": M_T * K_H * 4,
        "gate_up": 2 * q4 + ops.q8_1_bytes(M_T, K_H),
        "quantize_h": M_T * N_FF * 4,
        "down": ops.q4_0_pack_bytes(K_H, N_FF) + ops.q8_1_bytes(M_T, N_FF),
        "lmhead_top1": q6 + 5 * K_H * 4,
        "quantize_t": M_T * K_H * 4,
        "target_head": q6 + ops.q8_1_bytes(M_T, K_H),
        "argmax": M_T * N_V * 4,
    }


# ---------------------------------------------------------------- clocks


class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int, interval_ms: int = 20):
        self.index = index
        self.interval_ms = interval_ms
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", str(self.interval_ms)],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *a):
        self.lines = []
        if self.proc is not None:
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [ln for ln in out.splitlines() if ln.strip()]

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in getattr(self, "lines", []):
            parts = [p.strip() for p in ln.split(",")]
            try:
                sm.append(float(parts[0]))
                mx = float(parts[1])
            except (ValueError, IndexError):
                continue
            for nm, v in zip(names, parts[3:7]):
                if v.lower().startswith("active"):
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_min_mhz": min(sm) if sm else None,
                "sm_max_mhz": mx, "reasons": sorted(reasons), "samples": len(sm), "interval_ms": self.interval_ms,
                "window": "the whole GPU part of the native run (warm-up, timed steps, per-call, e2e, A/B and chain "
                          "measurements)"}


# ---------------------------------------------------------------- ranks


def max_over_ranks(ms: float, world: int) -> float:
    """The slowest rank's time: every rank of a replicas run ends its timed
    region at a barrier, and the job is as fast as its slowest replica."""
    if world <= 1:
        return ms
    import torch
    import torch.distributed as dist

    dev = torch.device("cuda", torch.cuda.current_device()) if dist.get_backend() == "nccl" else torch.device("cpu")
    t = torch.tensor([ms], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_gbs(world: int, bytes_per_step: int, ms_per_step: float) -> float:
    """Whole-job effective GB/s: the bytes every replica streams per step,
    over the (slowest rank's) step time."""
    return world * bytes_per_step / (ms_per_step * 1e-3) / 1e9


# ---------------------------------------------------------------- native arm


def run_native(args, rank, world):
    import torch
    import torch.distributed as dist

    from block_quantized_gemv_quantize_gb300 import build

    build.build()
    from block_quantized_gemv_quantize_gb300 import ops

    from block_quantized_gemv_quantize_gb300 import synth

    local = int(os.environ.get("LOCAL_RANK", 0))
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    inp = make_inputs()
    c_sweep_seed = synth.WORKLOADS["lmhead_q6_k"]["seed"] + 300

    def up(a):
        return torch.from_numpy(np.ascontiguousarray(a)).to(dev)

    w = {}
    for name, fmt, n, k in (("w_gate", "q4_0", N_FF, K_H), ("w_up", "q4_0", N_FF, K_H), ("w_down", "q4_0", K_H, N_FF),
                            ("w_vocab", "q6_k", N_V, K_H)):
        canon = up(inp[name])
        w[name] = (ops.qpack_q4_0 if fmt == "q4_0" else ops.qpack_q6_k)(canon, n, k)
        del canon
    torch.cuda.synchronize()
    torch.cuda.empty_cache()

    # resident activations, outputs and Q8_1 buffers
    x, h, xd, xt = up(inp["x"]), up(inp["h"]), up(inp["x_draft"]), up(inp["x_target"])
    xq1 = torch.empty(ops.q8_1_bytes(M_T, K_H), dtype=torch.uint8, device=dev)
    xq2 = torch.empty(ops.q8_1_bytes(M_T, N_FF), dtype=torch.uint8, device=dev)
    xq3 = torch.empty(ops.q8_1_bytes(M_T, K_H), dtype=torch.uint8, device=dev)
    y_gate = torch.empty((M_T, N_FF), device=dev)
    y_up = torch.empty((M_T, N_FF), device=dev)
    y_down = torch.empty((M_T, K_H), device=dev)
    logits = torch.empty((M_T, N_V), device=dev)
    ids_d = torch.empty(5, dtype=torch.int32, device=dev)
    ids_t = torch.empty(M_T, dtype=torch.int32, device=dev)
    ws1 = torch.zeros(ops.lmhead_q6_k_top1_workspace_bytes(5, K_H, N_V), dtype=torch.uint8, device=dev)
    ws2 = torch.zeros(ops.argmax_f32_rows_workspace_bytes(M_T, N_V), dtype=torch.uint8, device=dev)
    xd_rows = xd[1:6]

    names = ["quantize_x", "gate_up", "quantize_h", "down", "lmhead_top1", "quantize_t", "target_head", "argmax"]
    kernels_per_call = {"lmhead_top1": 2}  # the fused head: Q8_1 pre-pass + MMVQ with the top-1 epilogue
    calls = [
        lambda: ops.quantize_q8_1(x, out=xq1),
        lambda: ops.qgemv_q4_0_pair(w["w_gate"], w["w_up"], xq1, M_T, K_H, N_FF, N_FF, y_a=y_gate, y_b=y_up),
        lambda: ops.quantize_q8_1(h, out=xq2),
        lambda: ops.qgemv_q4_0(w["w_down"], xq2, M_T, N_FF, K_H, y=y_down),
        lambda: ops.lmhead_q6_k_top1(w["w_vocab"], xd_rows, K_H, N_V, ids=ids_d, ws=ws1),
        lambda: ops.quantize_q8_1(xt, out=xq3),
        lambda: ops.qgemv_q6_k(w["w_vocab"], xq3, M_T, K_H, N_V, y=logits),
        lambda: ops.argmax_f32_rows(logits, ids=ids_t, ws=ws2),
    ]
    stream = torch.cuda.current_stream(dev)

    def step(evs=None):
        for i, c in enumerate(calls):
            if evs is not None:
                evs[i][0].record(stream)
            c()
            if evs is not None:
                evs[i][1].record(stream)

    def barrier():
        if world > 1:
            dist.barrier()

    # clocks are sampled over the whole GPU part of the run (the timed region
    # alone can be a few milliseconds, shorter than nvidia-smi's interval)
    clk = ClockSampler(dev.index if dev.index is not None else 0)
    clk.__enter__()
    for _ in range(max(args.warmup, 3)):
        step()
    torch.cuda.synchronize()

    # The timed regions replay CUDA graphs captured from the library calls
    # (the same kernels, arguments and buffers, without the per-call host
    # work); --eager launches the calls one by one instead.
    def capture(fn):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            fn()
        torch.cuda.synchronize()
        return g

    g_step = None if args.eager else capture(step)
    if g_step is not None:
        for _ in range(3):
            g_step.replay()
        torch.cuda.synchronize()

    # timed region: K steps bracketed by two events
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    torch.cuda.synchronize()
    t0.record(stream)
    for _ in range(args.steps):
        if g_step is not None:
            g_step.replay()
        else:
            step()
    t1.record(stream)
    torch.cuda.synchronize()
    barrier()
    total_ms = max_over_ranks(t0.elapsed_time(t1), world)
    ms_per_step = total_ms / args.steps

    # per-call breakdown: a second timed region with an event pair around every call
    n_break = max(3, min(args.steps, 200))
    per = [[[torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)] for _ in calls]
           for _ in range(n_break)]
    torch.cuda.synchronize()
    for s_ in range(n_break):
        step(per[s_])
    torch.cuda.synchronize()
    call_ms = {n: statistics.mean(per[s_][i][0].elapsed_time(per[s_][i][1]) for s_ in range(n_break))
               for i, n in enumerate(names)}
    call_spread = {}  # median, p10, p90 of each call over the n_break steps (us)
    for i, n in enumerate(names):
        v = [per[s_][i][0].elapsed_time(per[s_][i][1]) * 1e3 for s_ in range(n_break)]
        q = statistics.quantiles(v, n=10)
        call_spread[n] = {"median": round(statistics.median(v), 2), "p10": round(q[0], 2), "p90": round(q[-1], 2)}

    nbytes = step_bytes()
    step_total = sum(nbytes.values())
    value = job_gbs(world, step_total, ms_per_step)

    # e2e: the same step through the public API with host buffers: per step the
    # activations are copied in from pinned host memory and the results
    # (both id vectors and the MLP output) are copied back.
    host_in = {k: torch.from_numpy(np.ascontiguousarray(inp[k])).pin_memory() for k in ("x", "h", "x_draft", "x_target")}
    dev_in = {"x": x, "h": h, "x_draft": xd, "x_target": xt}
    host_out = {"ids_d": torch.empty(5, dtype=torch.int32).pin_memory(),
                "ids_t": torch.empty(M_T, dtype=torch.int32).pin_memory(),
                "y_down": torch.empty((M_T, K_H)).pin_memory()}
    dev_out = {"ids_d": ids_d, "ids_t": ids_t, "y_down": y_down}
    h2d = sum(t.numel() * t.element_size() for t in host_in.values())
    d2h = sum(t.numel() * t.element_size() for t in host_out.values())

    def e2e_step():
        for k, t in host_in.items():
            dev_in[k].copy_(t, non_blocking=True)
        step()
        for k, t in host_out.items():
            t.copy_(dev_out[k], non_blocking=True)

    for _ in range(3):
        e2e_step()
    torch.cuda.synchronize()
    g_e2e = None if args.eager else capture(e2e_step)
    if g_e2e is not None:
        for _ in range(3):
            g_e2e.replay()
        torch.cuda.synchronize()
    barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        if g_e2e is not None:
            g_e2e.replay()
        else:
            e2e_step()
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1) / args.steps, world)
    e2e_value = job_gbs(world, step_total, e2e_ms)

    # fused vs unfused LM-head on identical inputs (rows 1..5), interleaved A/B
    y5 = torch.empty((5, N_V), device=dev)
    xq5 = torch.empty(ops.q8_1_bytes(5, K_H), dtype=torch.uint8, device=dev)
    ids_u = torch.empty(5, dtype=torch.int32, device=dev)

    def fused():
        ops.lmhead_q6_k_top1(w["w_vocab"], xd_rows, K_H, N_V, ids=ids_d, ws=ws1)

    def unfused():
        ops.quantize_q8_1(xd_rows, out=xq5)
        ops.qgemv_q6_k(w["w_vocab"], xq5, 5, K_H, N_V, y=y5)
        ops.argmax_f32_rows(y5, ids=ids_u, ws=ws2)

    cand = ids_d.clone()  # the verifier's candidate-max on the same rows, candidates = the draft's ids

    def candmax():
        ops.lmhead_q6_k_candmax(w["w_vocab"], xd_rows, K_H, N_V, cand, ws=ws1)

    # the top-8 form of the candidate-max on the same rows and candidates
    ws_k = torch.zeros(ops.lmhead_q6_k_topk_workspace_bytes(5, K_H, N_V, 8), dtype=torch.uint8, device=dev)
    ids_k = torch.empty((5, 8), dtype=torch.int32, device=dev)
    vals_k = torch.empty((5, 8), device=dev)
    cv_k = torch.empty(5, device=dev)

    def topk8():
        ops.lmhead_q6_k_topk(w["w_vocab"], xd_rows, K_H, N_V, 8, cand=cand, ws=ws_k, ids=ids_k, vals=vals_k,
                             cand_vals=cv_k)

    # the target side with all six rows fused (no logits) against the step's
    # unfused target head (quantize + qgemv_q6_k + argmax), same inputs
    ws6 = torch.zeros(ops.lmhead_q6_k_top1_workspace_bytes(M_T, K_H, N_V), dtype=torch.uint8, device=dev)
    ids_tf = torch.empty(M_T, dtype=torch.int32, device=dev)

    def target_fused():
        ops.lmhead_q6_k_top1(w["w_vocab"], xt, K_H, N_V, ids=ids_tf, ws=ws6)

    def target_unfused():
        ops.quantize_q8_1(xt, out=xq3)
        ops.qgemv_q6_k(w["w_vocab"], xq3, M_T, K_H, N_V, y=logits)
        ops.argmax_f32_rows(logits, ids=ids_t, ws=ws2)

    # RMSNorm fused into the Q8_1 quantizer against the quantizer alone, on
    # the gate/up input rows [6, 5120]
    gamma = torch.linspace(0.5, 1.5, K_H, device=dev)

    def rms_q8():
        ops.rmsnorm_quantize_q8_1(x, gamma, 1e-6, out=xq1)

    def q8_only():
        ops.quantize_q8_1(x, out=xq1)

    ab = {"fused": [], "unfused": [], "candmax": [], "topk8": [], "target_fused": [], "target_unfused": [],
          "rms_q8": [], "q8_only": []}
    ab_rounds = 20  # interleaved A/B rounds of 10 calls each
    for _ in range(ab_rounds):
        for name, fn in (("fused", fused), ("unfused", unfused), ("candmax", candmax), ("topk8", topk8),
                         ("target_fused", target_fused), ("target_unfused", target_unfused), ("rms_q8", rms_q8),
                         ("q8_only", q8_only)):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            for _ in range(10):
                fn()
            b.record(stream)
            torch.cuda.synchronize()
            ab[name].append(a.elapsed_time(b) * 1e3 / 10)
    same_ids = ids_d.cpu().tolist() == ids_u.cpu().tolist()
    same_ids_t = ids_tf.cpu().tolist() == ids_t.cpu().tolist()
    topk_first_is_top1 = ids_k[:, 0].cpu().tolist() == ids_d.cpu().tolist()

    # Fused against unfused LM-head over the M sweep (the unfused control
    # writes the full fp32 logits and runs a separate argmax): for each M,
    # rows 0..M-1 of a [17, 5120] activation, the fused top-1 against
    # quantize + qgemv_q6_k + argmax_f32_rows on the same inputs, interleaved
    # rounds of 10 calls each.
    xs = up(synth.activations(17, K_H, seed=c_sweep_seed))
    ys = torch.empty((17, N_V), device=dev)
    xqs = torch.empty(ops.q8_1_bytes(17, K_H), dtype=torch.uint8, device=dev)
    ws17 = torch.zeros(ops.lmhead_q6_k_top1_workspace_bytes(17, K_H, N_V), dtype=torch.uint8, device=dev)
    m_sweep = {}
    for Ms in (1, 2, 4, 6, 9, 12, 17):
        xm = xs[:Ms]
        idf = torch.empty(Ms, dtype=torch.int32, device=dev)
        idu = torch.empty(Ms, dtype=torch.int32, device=dev)
        fm = (lambda xm=xm, idf=idf: ops.lmhead_q6_k_top1(w["w_vocab"], xm, K_H, N_V, ids=idf, ws=ws17))

        def um(xm=xm, idu=idu, Ms=Ms):
            ops.quantize_q8_1(xm, out=xqs[: ops.q8_1_bytes(Ms, K_H)])
            ops.qgemv_q6_k(w["w_vocab"], xqs[: ops.q8_1_bytes(Ms, K_H)], Ms, K_H, N_V, y=ys[:Ms])
            ops.argmax_f32_rows(ys[:Ms], ids=idu, ws=ws2)

        tf, tu = [], []
        for _ in range(8):
            for lst, fn in ((tf, fm), (tu, um)):
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record(stream)
                for _ in range(10):
                    fn()
                b.record(stream)
                torch.cuda.synchronize()
                lst.append(a.elapsed_time(b) * 1e3 / 10)
        diff = [u_ - f_ for f_, u_ in zip(tf, tu)]
        m_sweep[str(Ms)] = {"fused_us": round(statistics.median(tf), 2), "unfused_us": round(statistics.median(tu), 2),
                            "diff_median_us": round(statistics.median(diff), 2), "diff_min_us": round(min(diff), 2),
                            "diff_max_us": round(max(diff), 2),
                            "same_ids": idf.cpu().tolist() == idu.cpu().tolist()}
    del ys, xqs

    # The verifier MLP projections as a layer stack runs them: the gate/up
    # pair and the down projection of L layers with distinct weights (so no
    # call finds its weights in L2), back to back on the stream, the
    # activations quantized once beforehand; events around the whole chain.
    L_LAYERS = 4
    lw = [(w["w_gate"], w["w_up"], w["w_down"])]
    for i in range(1, L_LAYERS):
        g_ = torch.randint(0, 256, (w["w_gate"].numel(),), dtype=torch.uint8, device=dev)
        u_ = torch.randint(0, 256, (w["w_up"].numel(),), dtype=torch.uint8, device=dev)
        d_ = torch.randint(0, 256, (w["w_down"].numel(),), dtype=torch.uint8, device=dev)
        lw.append((g_, u_, d_))
    ops.quantize_q8_1(x, out=xq1)
    ops.quantize_q8_1(h, out=xq2)

    def mlp_chain():
        for wg_, wu_, wd_ in lw:
            ops.qgemv_q4_0_pair(wg_, wu_, xq1, M_T, K_H, N_FF, N_FF, y_a=y_gate, y_b=y_up)
            ops.qgemv_q4_0(wd_, xq2, M_T, N_FF, K_H, y=y_down)

    for _ in range(3):
        mlp_chain()
    torch.cuda.synchronize()
    chain_rounds = 25
    c0, c1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    c0.record(stream)
    for _ in range(chain_rounds):
        mlp_chain()
    c1.record(stream)
    torch.cuda.synchronize()
    chain_us_layer = c0.elapsed_time(c1) * 1e3 / (chain_rounds * L_LAYERS)
    del lw
    clk.__exit__(None, None, None)

    def ab_pair(a_name, b_name, keys, extra):
        """Medians of two interleaved arms, and the median, p10 and p90 of
        their per-round difference (b - a, us)."""
        diff = [y - x for x, y in zip(ab[a_name], ab[b_name])]
        q = statistics.quantiles(diff, n=10)
        out = {keys[0]: round(statistics.median(ab[a_name]), 2), keys[1]: round(statistics.median(ab[b_name]), 2),
               "diff_median": round(statistics.median(diff), 2), "diff_p10": round(q[0], 2),
               "diff_p90": round(q[-1], 2), "rounds": ab_rounds}
        out.update(extra)
        return out

    peak, peak_kind = peaks()
    dominant = max(("lmhead_top1", "target_head", "gate_up", "down"), key=lambda n: call_ms[n])
    achieved = nbytes[dominant] / (call_ms[dominant] * 1e-3) / 1e9
    traffic = load_traffic(dominant)
    mmvq_names = ("gate_up", "down")
    mmvq_bytes = sum(nbytes[n] for n in mmvq_names)
    mmvq_lone_gbs = mmvq_bytes / (sum(call_ms[n] for n in mmvq_names) * 1e-3) / 1e9
    mmvq_gbs = mmvq_bytes / (chain_us_layer * 1e-6) / 1e9

    result = None
    if rank == 0:
        clocks = clk.summary()
        run_native.inputs = inp
        result = {
            "metric": METRIC,
            "value": round(value, 1),
            "unit": UNIT,
            "n_gpus": world,
            "steps": args.steps,
            "warmup": args.warmup,
            "ms_per_step": round(ms_per_step, 4),
            "higher_is_better": True,
            "scaling": "weak",
            "vs_baseline": None,
            "dtype": "int8 x int4/int6 -> int32 block dots, fp32 accumulate",
            "data": "synthetic (seeded; Q4_0/Q6_K/Q8_1 shapes and distributions of the pages' workloads)",
            "config": {"workload": WORKLOAD, "bytes_per_step": step_total,
                       "l2": "inputs larger than L2: ~2.2 GB of weights streamed per step, no flush needed",
                       "replicas": world},
            "mmvq_m6_q4_0": {"gbs": round(mmvq_gbs, 1), "frac_of_hbm_peak": round(mmvq_gbs / peak, 4),
                             "timing": f"back-to-back chain of the gate/up pair and the down projection of "
                                       f"{L_LAYERS} layers with distinct weights, {chain_rounds} rounds, events "
                                       "around the chain",
                             "us_per_layer": round(chain_us_layer, 2), "bytes_per_layer": mmvq_bytes,
                             "lone_call": {"gbs": round(mmvq_lone_gbs, 1),
                                           "frac_of_hbm_peak": round(mmvq_lone_gbs / peak, 4),
                                           "us": {n: round(call_ms[n] * 1e3, 2) for n in mmvq_names},
                                           "timing": "an event pair around each call inside the step"}},
            "lmhead_top1_us": round(call_ms["lmhead_top1"] * 1e3, 2),
            "fused_vs_unfused_us": ab_pair("fused", "unfused", ("fused", "unfused"), {"same_ids": same_ids}),
            "candmax_us": round(statistics.median(ab["candmax"]), 2),
            "topk8_vs_top1_us": ab_pair("fused", "topk8", ("top1", "topk8"),
                                        {"rows": "1..5", "k": 8, "with_candidate_scores": True,
                                         "rank0_equals_top1": topk_first_is_top1}),
            "rmsnorm_q8_1_vs_quantize_us": ab_pair("q8_only", "rms_q8", ("quantize_q8_1", "rmsnorm_q8_1"), {}),
            "target_m6_fused_vs_unfused_us": ab_pair("target_fused", "target_unfused", ("fused", "unfused"),
                                                     {"same_ids": same_ids_t}),
            "fused_vs_unfused_m_sweep_us": m_sweep,
            "per_call_us": {n: round(call_ms[n] * 1e3, 2) for n in names},
            "per_call_us_spread": call_spread,
            "per_call_gbs": {n: round(nbytes[n] / (call_ms[n] * 1e-3) / 1e9, 1) for n in names},
            "roofline": {"kernel": dominant, "bound": "hbm", "achieved": round(achieved, 1), "peak": peak,
                         "peak_kind": peak_kind, "unit": "GB/s", "frac": round(achieved / peak, 4),
                         "traffic": traffic, "algorithmic_bytes": nbytes[dominant]},
            "e2e": {"value": round(e2e_value, 1), "unit": UNIT, "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h, "ms_per_step": round(e2e_ms, 4)},
            "gpu_launches": sum(kernels_per_call.get(n, 1) for n in names) * args.steps,
            "launch": "eager" if args.eager else "cuda_graph (captured from the library calls, replayed per step)",
            "breakdown_steps": n_break,
            "clocks": clocks,
        }
    return result


def _source_digest() -> str:
    """A digest of the sources that decide what a kernel reads and writes:
    every header (kernels, launch plans) and every translation unit that
    defines a kernel or instantiates one; the host-only entry layer (argument
    checks, status words) is left out."""
    csrc = os.path.join(ROOT, "block_quantized_gemv_quantize_gb300", "csrc")
    h = hashlib.sha256()
    for f in sorted(os.listdir(csrc)):
        if f.endswith((".cu", ".cuh")) and f != "api.cu":
            h.update(f.encode())
            h.update(open(os.path.join(csrc, f), "rb").read())
    return h.hexdigest()[:16]


def load_traffic(kernel: str):
    """DRAM bytes per launch from the committed ncu summary, or None when the
    kernels changed since it was captured."""
    path = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    if not os.path.exists(path):
        return None
    d = json.load(open(path))
    if d.get("source_digest") != _source_digest():
        return None
    return d.get("per_launch_dram_bytes", {}).get(kernel)


# ---------------------------------------------------------------- M sweep


def run_sweep(args):
    """Per-call time and effective GB/s of the MMVQ over the M sweep, each
    call timed alone (CUDA events) right after an L2 flush that is not timed,
    on random packed weights (timing does not depend on the bytes)."""
    import torch

    from block_quantized_gemv_quantize_gb300 import build

    build.build()
    from block_quantized_gemv_quantize_gb300 import ops

    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    g = torch.Generator(device="cpu").manual_seed(0)
    flush = torch.empty(256 * 2**20, dtype=torch.uint8, device=dev)  # twice the L2
    reps = max(3, min(args.steps, 20))
    peak, _ = peaks()
    pack_bytes = {"q4_0": ops.q4_0_pack_bytes, "q6_k": ops.q6_k_pack_bytes, "q8_0": ops.q8_0_pack_bytes,
                  "q4_k": ops.q4_k_pack_bytes, "q5_k": ops.q5_k_pack_bytes}
    gemv = {"q4_0": ops.qgemv_q4_0, "q6_k": ops.qgemv_q6_k, "q8_0": ops.qgemv_q8_0, "q4_k": ops.qgemv_q4_k,
            "q5_k": ops.qgemv_q5_k}
    canonical = {"q4_k": 144, "q5_k": 176}  # bytes per 256 values
    K = args.sweep_k
    for fmt in args.sweep_formats.split(","):
        for N in (int(v) for v in args.sweep_n.split(",")):
            nbytes_w = pack_bytes[fmt](N, K)
            # algorithmic bytes: the canonical size (the Q4_K / Q5_K packs carry
            # 148 / 180 B per 256 values against 144 / 176; the others are equal)
            nbytes_alg = N * (K // 256) * canonical[fmt] if fmt in canonical else nbytes_w
            w = torch.randint(0, 256, (nbytes_w,), dtype=torch.uint8, generator=g).to(dev)
            for M in (int(v) for v in args.sweep_m.split(",")):
                x = torch.randn(M, K, generator=g).to(dev)
                xq = ops.quantize_q8_1(x)
                y = torch.empty((M, N), device=dev)
                call = (lambda f=gemv[fmt]: f(w, xq, M, K, N, y=y))
                try:
                    call()
                except ops.QgemvError as e:  # a shape the library declines: recorded, not timed
                    print(json.dumps({"sweep": fmt, "M": M, "K": K, "N": N, "unsupported": str(e)}), flush=True)
                    continue
                for _ in range(3):
                    call()
                ts = []
                for _ in range(reps):
                    flush.fill_(1)
                    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                    a.record()
                    call()
                    b.record()
                    torch.cuda.synchronize()
                    ts.append(a.elapsed_time(b))
                us = statistics.median(ts) * 1e3
                nbytes = nbytes_alg + ops.q8_1_bytes(M, K)
                gbs = nbytes / (us * 1e-6) / 1e9
                print(json.dumps({"sweep": fmt, "M": M, "K": K, "N": N, "us": round(us, 2),
                                  "gbs": round(gbs, 1), "frac_of_hbm_peak": round(gbs / peak, 4),
                                  "l2": "flushed before every call"}), flush=True)
            del w
            torch.cuda.empty_cache()


# ---------------------------------------------------------------- CPU oracle


def oracle_sample_step(inp, frac: float, nthreads: int):
    """One step of the oracle over the first `frac` of every weight's rows;
    returns (seconds, algorithmic bytes of the sample)."""
    import oracle

    def rows(a):
        return a[: max(1, int(round(a.shape[0] * frac)))]

    t = time.perf_counter()
    nbytes = 0
    xq1 = oracle.quantize_q8_1(inp["x"])
    for name in ("w_gate", "w_up"):
        wr = rows(inp[name])
        oracle.qgemv_q4_0(wr, xq1, nthreads)
        nbytes += wr.nbytes
    nbytes += xq1.nbytes  # gate and up read one activation
    xq2 = oracle.quantize_q8_1(inp["h"])
    wr = rows(inp["w_down"])
    oracle.qgemv_q4_0(wr, xq2, nthreads)
    nbytes += wr.nbytes + xq2.nbytes
    wv = rows(inp["w_vocab"])
    y5, _ = oracle.qgemv_q6_k(wv, oracle.quantize_q8_1(inp["x_draft"][1:6]), nthreads)
    oracle.top1(y5)
    nbytes += wv.nbytes + 5 * K_H * 4
    yt, _ = oracle.qgemv_q6_k(wv, oracle.quantize_q8_1(inp["x_target"]), nthreads)
    oracle.top1(yt)
    nbytes += wv.nbytes + xq1.nbytes + yt.size * 4
    nbytes += (inp["x"].nbytes + inp["h"].nbytes + inp["x_target"].nbytes)
    return time.perf_counter() - t, nbytes


def cpu_model() -> str:
    """The host CPU's model name (lscpu, else /proc/cpuinfo), with the
    architecture."""
    import platform

    name = None
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for ln in out.splitlines():
            if ln.split(":")[0].strip() == "Model name":
                name = ln.split(":", 1)[1].strip()
                break
    except (OSError, subprocess.SubprocessError):
        pass
    if not name:
        try:
            for ln in open("/proc/cpuinfo"):
                if ln.lower().startswith("model name"):
                    name = ln.split(":", 1)[1].strip()
                    break
        except OSError:
            pass
    return f"{name or 'unknown'} ({platform.machine()})"


def calibrate_fraction(inp, seconds: float, nthreads: int) -> float:
    dt, _ = oracle_sample_step(inp, 0.002, nthreads)
    return min(1.0, max(0.0005, 0.002 * seconds / max(dt, 1e-3)))


def cpu_baseline(inp, seconds: float):
    """The oracle on the host cores: whole oracle steps (or a row fraction of
    one, if a step is longer than `seconds`) repeated until `seconds` pass."""
    import oracle

    n = oracle.default_threads()
    frac = calibrate_fraction(inp, seconds, n)
    total_t, total_b, reps = 0.0, 0, 0
    while total_t < seconds or reps == 0:
        dt, nb = oracle_sample_step(inp, frac, n)
        total_t += dt
        total_b += nb
        reps += 1
    # the same oracle on one core, on a smaller row fraction (about a quarter
    # of the time above), for the single-thread figure
    frac1 = calibrate_fraction(inp, seconds / 4, 1)
    t1, b1 = oracle_sample_step(inp, frac1, 1)
    return {"value": round(total_b / total_t / 1e9, 4), "unit": UNIT, "cores": n, "kind": "oracle",
            "cpu_model": cpu_model(),
            "sample": f"{reps} oracle step(s) over the first {frac:.2%} of the rows of every weight "
                      f"({total_t:.1f} s, {total_b / 1e6:.0f} MB)",
            "single_core": {"value": round(b1 / t1 / 1e9, 4), "unit": UNIT, "cores": 1,
                            "sample": f"one oracle step over the first {frac1:.2%} of the rows ({t1:.1f} s)"}}


def run_reference(args):
    import oracle

    inp = make_inputs()
    n = oracle.default_threads()
    per_step_s = max(1.0, min(6.0, 150.0 / max(1, args.steps + args.warmup)))
    frac = calibrate_fraction(inp, per_step_s, n)
    for _ in range(args.warmup):
        oracle_sample_step(inp, frac, n)
    times, nb = [], 0
    for _ in range(args.steps):
        dt, nb = oracle_sample_step(inp, frac, n)
        times.append(dt)
    total = sum(times)
    value = nb * args.steps / total / 1e9
    sample = f"first {frac:.4%} of the rows of every weight per step"
    return {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(1e3 * total / args.steps, 2),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "int32 block dots, fp64 accumulate (CPU oracle)",
        "data": "synthetic (seeded; same inputs as the native arm)",
        "config": {"workload": WORKLOAD, "sampled": sample},
        "cpu_baseline": {"value": round(value, 4), "unit": UNIT, "cores": n, "kind": "oracle", "sample": sample,
                         "cpu_model": cpu_model()},
        "e2e": {"value": round(value, 4), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def run_profile(args):
    """A few calls of one part of the step, each after an L2 flush, on the
    step's own seeded inputs; a small device footprint for a profiler.  Prints
    the median event time of each call."""
    import torch

    from block_quantized_gemv_quantize_gb300 import build, synth

    build.build()
    from block_quantized_gemv_quantize_gb300 import ops

    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)

    def up(a):
        return torch.from_numpy(np.ascontiguousarray(a)).to(dev)

    def pack(fmt, canon, n, k):
        c = up(canon)
        return (ops.qpack_q4_0 if fmt == "q4_0" else ops.qpack_q6_k)(c, n, k)

    flush = torch.empty(256 * 2**20, dtype=torch.uint8, device=dev)
    if args.profile == "mlp":
        c1, c2 = synth.WORKLOADS["verifier_gate_up"], synth.WORKLOADS["verifier_down"]
        wg = pack("q4_0", synth.q4_0_weights(N_FF, K_H, seed=c1["seed"]), N_FF, K_H)
        wu = pack("q4_0", synth.q4_0_weights(N_FF, K_H, seed=c1["seed"] + 10), N_FF, K_H)
        wd = pack("q4_0", synth.q4_0_weights(K_H, N_FF, seed=c2["seed"]), K_H, N_FF)
        xq = ops.quantize_q8_1(up(synth.activations(M_T, K_H, seed=c1["seed"] + 100, outlier_frac=0.01)))
        hq = ops.quantize_q8_1(up(synth.activations(M_T, N_FF, seed=c2["seed"] + 100, outlier_frac=0.01)))
        yg, yu, yd = (torch.empty((M_T, n), device=dev) for n in (N_FF, N_FF, K_H))
        calls = {"gate_up": lambda: ops.qgemv_q4_0_pair(wg, wu, xq, M_T, K_H, N_FF, N_FF, y_a=yg, y_b=yu),
                 "down": lambda: ops.qgemv_q4_0(wd, hq, M_T, N_FF, K_H, y=yd)}
    elif args.profile == "topk":
        c3 = synth.WORKLOADS["lmhead_q6_k"]
        wv = pack("q6_k", synth.q6_k_weights(N_V, K_H, seed=c3["seed"]), N_V, K_H)
        xd = up(synth.activations(6, K_H, seed=c3["seed"] + 100))
        ids5 = torch.empty(5, dtype=torch.int32, device=dev)
        idk = torch.empty((5, 8), dtype=torch.int32, device=dev)
        vk = torch.empty((5, 8), dtype=torch.float32, device=dev)
        calls = {"lmhead_top1": lambda: ops.lmhead_q6_k_top1(wv, xd[1:6], K_H, N_V, ids=ids5),
                 "lmhead_top8": lambda: ops.lmhead_q6_k_topk(wv, xd[1:6], K_H, N_V, 8, ids=idk, vals=vk)}
    else:
        c3 = synth.WORKLOADS["lmhead_q6_k"]
        wv = pack("q6_k", synth.q6_k_weights(N_V, K_H, seed=c3["seed"]), N_V, K_H)
        xd = up(synth.activations(6, K_H, seed=c3["seed"] + 100))
        xq = ops.quantize_q8_1(up(synth.activations(M_T, K_H, seed=c3["seed"] + 200)))
        logits = torch.empty((M_T, N_V), device=dev)
        x8 = up(synth.activations(8, K_H, seed=c3["seed"] + 300))
        xq8 = ops.quantize_q8_1(x8)
        logits8 = torch.empty((8, N_V), device=dev)

        def tc_m8():
            # the tensor-core Q6_K kernel at M = 8, for comparison with the dp4a heads
            prev = ops.set_q6_k_tensor_cores(2)
            ops.qgemv_q6_k(wv, xq8, 8, K_H, N_V, y=logits8)
            ops.set_q6_k_tensor_cores(prev)

        calls = {"target_head": lambda: ops.qgemv_q6_k(wv, xq, M_T, K_H, N_V, y=logits),
                 "lmhead_top1": lambda: ops.lmhead_q6_k_top1(wv, xd[1:6], K_H, N_V),
                 "q6_k_tc_m8": tc_m8}
    torch.cuda.synchronize()
    times = {n: [] for n in calls}
    for _ in range(max(1, args.steps)):
        for n, f in calls.items():
            flush.fill_(1)
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            f()
            b.record()
            torch.cuda.synchronize()
            times[n].append(a.elapsed_time(b) * 1e3)
    print(json.dumps({"profile": args.profile, "calls": args.steps,
                      "median_us": {n: round(statistics.median(v), 2) for n, v in times.items()},
                      "l2": "flushed before every call"}), flush=True)


def main():
    args = parse()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args)), flush=True)
        return
    if args.sweep:
        if rank == 0:
            run_sweep(args)
        return
    if args.profile:
        if rank == 0:
            run_profile(args)
        return
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl")
    result = run_native(args, rank, world)
    if rank == 0:
        if world == 1 and not args.no_cpu_baseline:
            result["cpu_baseline"] = cpu_baseline(run_native.inputs, args.cpu_seconds)
        print(json.dumps(result), flush=True)
    if world > 1:
        import torch.distributed as dist

        dist.destroy_process_group()


if __name__ == "__main__":
    main()
