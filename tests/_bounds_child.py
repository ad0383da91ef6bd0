"""Child process of test_gpu_bounds_check (run with QGEMV_BOUNDS_CHECK=1, so
that the binding loads the bounds-checking library): every entry point on
small and odd shapes against the oracle, each followed by a read of the
bounds records, then one planted out-of-extent store.  Prints one JSON line.
Test code only."""
import json
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import torch  # noqa: E402

import oracle  # noqa: E402
from block_quantized_gemv_quantize_gb300 import ops, synth  # noqa: E402
from tests import _cases as C  # noqa: E402

DEV = "cuda:0"


def t_(a):
    return torch.from_numpy(np.ascontiguousarray(a)).to(DEV)


def n_(x):
    torch.cuda.synchronize()
    return x.cpu().numpy()


def main():
    res = {"bounds_build": ops.qgemv_bounds_check_build(), "cases": [], "fail": []}
    ops.qgemv_take_bounds_errors()

    def record(name, ok, detail=""):
        cnt, site = ops.qgemv_take_bounds_errors()
        res["cases"].append(name)
        if not ok or cnt:
            res["fail"].append([name, bool(ok), cnt, site, str(detail)[:300]])

    # Q8_1 quantizer (bit for bit), RMSNorm quantizer (within its bounds)
    for M, K, ldx in ((1, 32, 32), (3, 96, 100), (17, 1024, 1056)):
        x = synth.activations(M, ldx, seed=M + K)
        got = n_(ops.quantize_q8_1(t_(x), K)).reshape(M, K // 32, 36)
        record(f"quantize {M}x{K}", np.array_equal(got, oracle.quantize_q8_1(x, K)))
    x = synth.activations(2, 160, seed=5)
    gamma = np.linspace(0.5, 1.5, 160).astype(np.float32)
    ref, xh = oracle.rmsnorm_quantize_q8_1(x, gamma, 1e-6, K=160, with_xh=True)
    got = n_(ops.rmsnorm_quantize_q8_1(t_(x), t_(gamma), 1e-6, K=160)).reshape(2, 5, 36)
    record("rmsnorm 2x160", C.check_q8_1_near(got, ref, xh, 160)["ok"])

    def gemv_case(name, fmt, M, K, N, seed, mode=None):
        wgen = {"q4_0": synth.q4_0_weights, "q6_k": synth.q6_k_weights, "q8_0": synth.q8_0_weights,
                "q4_k": synth.q4_k_weights, "q5_k": synth.q5_k_weights}[fmt]
        w = wgen(N, K, seed=seed)
        x = synth.activations(M, K, seed=seed + 1)
        xq_ref = oracle.quantize_q8_1(x)
        xq = ops.quantize_q8_1(t_(x))
        pack = getattr(ops, "qpack_" + fmt)(t_(w), N, K)
        y = n_(getattr(ops, "qgemv_" + fmt)(pack, xq, M, K, N))
        y_ref, S = getattr(oracle, "qgemv_" + fmt)(w, xq_ref)
        r = C.check_close(y, y_ref, S)
        record(f"{name} {fmt} M={M} K={K} N={N} mode={mode}", r["ok"], r)

    for mode in (0, 1, 2):
        prev = ops.set_q4_0_tensor_cores(mode)
        for M, K, N in ((1, 32, 1), (5, 96, 7), (9, 1056, 33), (17, 256, 5), (6, 1024, 48), (12, 1024, 48),
                        (6, 17408, 64), (3, 5120, 80)):
            gemv_case("gemv", "q4_0", M, K, N, seed=M * 100 + N, mode=mode)
        ops.set_q4_0_tensor_cores(prev)
    for mode in (0, 2):
        prev = ops.set_q6_k_tensor_cores(mode)
        for M, K, N in ((1, 256, 5), (2, 768, 33), (12, 1024, 48), (6, 1024, 48), (17, 2048, 16)):
            gemv_case("gemv", "q6_k", M, K, N, seed=M * 100 + N + 1, mode=mode)
        ops.set_q6_k_tensor_cores(prev)
    for fmt in ("q8_0", "q4_k", "q5_k"):
        for M, K, N in ((3, 256, 17), (9, 512, 40), (6, 5120, 48)):
            gemv_case("gemv", fmt, M, K, N, seed=M * 10 + N + 2)

    # pair and residual (Q4_0)
    for mode in (0, 1):
        prev = ops.set_q4_0_tensor_cores(mode)
        M, K, Na, Nb = 6, 1024, 48, 32
        wa, wb = synth.q4_0_weights(Na, K, seed=11), synth.q4_0_weights(Nb, K, seed=12)
        x = synth.activations(M, K, seed=13)
        xq_ref = oracle.quantize_q8_1(x)
        ya, yb = ops.qgemv_q4_0_pair(ops.qpack_q4_0(t_(wa), Na, K), ops.qpack_q4_0(t_(wb), Nb, K),
                                     ops.quantize_q8_1(t_(x)), M, K, Na, Nb)
        ok = all(C.check_close(n_(y), *oracle.qgemv_q4_0(w, xq_ref))["ok"] for y, w in ((ya, wa), (yb, wb)))
        record(f"pair mode={mode}", ok)
        ops.set_q4_0_tensor_cores(prev)
    M, K, N = 3, 96, 7
    w = synth.q4_0_weights(N, K, seed=14)
    x = synth.activations(M, K, seed=15)
    r_ = synth.activations(M, N, seed=16)
    y = n_(ops.qgemv_q4_0_residual(ops.qpack_q4_0(t_(w), N, K), ops.quantize_q8_1(t_(x)), t_(r_), M, K, N))
    y_ref, S = oracle.qgemv_q4_0(w, oracle.quantize_q8_1(x))
    want = y_ref + r_.astype(np.float64)  # the MMVQ's gate plus one fp32 rounding of the sum
    tol = 1e-5 * np.maximum(np.abs(y_ref), S) + 2.0 ** -23 * np.abs(want)
    record("residual", bool(np.all(np.abs(y.astype(np.float64) - want) <= tol)))

    # integer block dots (bit for bit)
    M, K, N = 2, 256, 5
    w4, w6 = synth.q4_0_weights(N, K, seed=17), synth.q6_k_weights(N, K, seed=18)
    x = synth.activations(M, K, seed=19)
    xq_ref = oracle.quantize_q8_1(x)
    xq = ops.quantize_q8_1(t_(x))
    record("block dots q4_0", np.array_equal(n_(ops.qgemv_block_dots_q4_0(ops.qpack_q4_0(t_(w4), N, K), xq, M, K, N)),
                                             oracle.block_dots_q4_0(w4, xq_ref)))
    record("block dots q6_k", np.array_equal(n_(ops.qgemv_block_dots_q6_k(ops.qpack_q6_k(t_(w6), N, K), xq, M, K, N)),
                                             oracle.block_dots_q6_k(w6, xq_ref)))

    # the LM-head family: top-1 (ring and lock-step), candidate-max, top-k,
    # the no-allocation entry, and the unfused argmax
    for M, K, N in ((5, 512, 301), (1, 256, 7), (17, 17408, 64)):
        w = synth.q6_k_weights(N, K, seed=M + N)
        x = synth.activations(M, K, seed=K + M)
        ids_ref, y_ref, S = oracle.lmhead_q6_k_top1(w, x)
        wp = ops.qpack_q6_k(t_(w), N, K)
        xd = t_(x)
        record(f"top1 {M}x{K}x{N}", C.check_top1(n_(ops.lmhead_q6_k_top1(wp, xd, K, N)), y_ref) == [])
        record(f"noalloc {M}x{K}x{N}", C.check_top1(n_(ops.lmhead_q6_k_top1_noalloc(wp, xd, K, N)), y_ref) == [])
        cand = torch.zeros(M, dtype=torch.int32, device=DEV)
        ids, tv, cv = ops.lmhead_q6_k_candmax(wp, xd, K, N, cand)
        record(f"candmax {M}x{K}x{N}", C.check_top1(n_(ids), y_ref) == [])
        if M * K <= 5 * 5120:  # the top-k takes the ring kernel's shapes only
            k = min(8, N)
            ids, vals, _ = ops.lmhead_q6_k_topk(wp, xd, K, N, k)
            record(f"topk {M}x{K}x{N}", C.check_topk(n_(ids), n_(vals), y_ref, S) == [])
    y = synth.activations(3, 1001, seed=20)
    record("argmax", n_(ops.argmax_f32_rows(t_(y))).tolist() == oracle.top1(y).tolist())

    # a planted store past its extent: skipped and recorded (site 620, the ring
    # kernel's plain store), the context still usable
    prev = ops.set_q6_k_tensor_cores(0)
    M, K, N = 2, 256, 64
    w = synth.q6_k_weights(N, K, seed=21)
    x = synth.activations(M, K, seed=22)
    wp, xq = ops.qpack_q6_k(t_(w), N, K), ops.quantize_q8_1(t_(x))
    ops.qgemv_take_bounds_errors()
    ops.qgemv_debug_plant_bad_store()
    ops.qgemv_q6_k(wp, xq, M, K, N)
    res["planted"] = list(ops.qgemv_take_bounds_errors())
    y = n_(ops.qgemv_q6_k(wp, xq, M, K, N))
    y_ref, S = oracle.qgemv_q6_k(w, oracle.quantize_q8_1(x))
    res["after_planted_ok"] = C.check_close(y, y_ref, S)["ok"]
    res["after_planted_records"] = list(ops.qgemv_take_bounds_errors())
    ops.set_q6_k_tensor_cores(prev)
    res["timeouts"] = ops.qgemv_take_wait_timeouts()
    print(json.dumps(res), flush=True)


if __name__ == "__main__":
    main()
