"""Parity at the full workload sizes the benchmark times (same launch
configuration: the library picks it from M, K, N), against the CPU oracle.

  * tiny Q4_0 GEMV exactly as configured (M=1, K=256, N=512, seed 0): every
    output, and the row argmax with lowest-index ties;
  * width-6 verifier MMVQ, Q4_0: gate/up M=6 K=5120 N=17408, down M=6 K=17408
    N=5120 (1% outlier channels x20) -- every output checked;
  * fused Q6_K LM-head top-1, K=5120 N=248320, rows 1..5 of a [6, 5120] block
    -- ids against the full oracle, and against the unfused path;
  * M sweep {1,2,4,6,9,12,17} for Q4_0 and Q6_K at K=5120, N in {5120, 17408,
    248320} -- sampled rows (first 64, last 64 and 1024 random rows); the
    further formats Q8_0, Q4_K, Q5_K at M in {1, 6, 9, 17}, N in {17408,
    248320}, the same way;
  * adversarial top-1 at K=5120 N=248320 M=5: all-zero weights, planted exact
    ties at (1,256), (255,256), (0,248319), a planted near tie.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = [pytest.mark.gpu, pytest.mark.slow]

import oracle  # noqa: E402
from block_quantized_gemv_quantize_gb300 import synth  # noqa: E402

from . import _cases as C  # noqa: E402

DEV = "cuda:0"
K_H, N_V = 5120, 248320


@pytest.fixture(scope="module")
def ops():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from block_quantized_gemv_quantize_gb300 import build

    build.build()
    from block_quantized_gemv_quantize_gb300 import ops as o

    return o


def _t(a):
    return torch.from_numpy(np.ascontiguousarray(a)).to(DEV)


def _np(t):
    torch.cuda.synchronize()
    return t.cpu().numpy()


def test_tiny_q4_0_as_configured(ops):
    c = synth.WORKLOADS["tiny_q4_0"]
    M, K, N = c["M"], c["K"], c["N"]
    w, x = synth.tiny_q4_0_inputs()
    xq_ref = oracle.quantize_q8_1(x)
    y_ref, S = oracle.qgemv_q4_0(w, xq_ref)
    xq = ops.quantize_q8_1(_t(x))
    assert np.array_equal(_np(xq).reshape(xq_ref.shape), xq_ref)
    yd = ops.qgemv_q4_0(ops.qpack_q4_0(_t(w), N, K), xq, M, K, N)
    y = _np(yd)
    r = C.check_close(y, y_ref, S)
    print("tiny_q4_0", r)
    assert r["ok"], r
    # the argmax: on the GPU's own fp32 output, the oracle's lowest-index
    # rule bit for bit; against the fp64 oracle values, the gap rule
    ids = _np(ops.argmax_f32_rows(yd))
    assert np.array_equal(ids, oracle.top1(y.astype(np.float32)))
    assert not C.check_top1(ids, y_ref)


@pytest.mark.parametrize("name", ["verifier_gate_up", "verifier_down"])
def test_verifier_mmvq_full(ops, name):
    c = synth.WORKLOADS[name]
    M, K, N = c["M"], c["K"], c["N"]
    w = synth.q4_0_weights(N, K, seed=c["seed"])
    x = synth.activations(M, K, seed=c["seed"] + 100, outlier_frac=c["outlier_frac"])
    xq_ref = oracle.quantize_q8_1(x)
    y_ref, S = oracle.qgemv_q4_0(w, xq_ref)
    xq = ops.quantize_q8_1(_t(x))
    assert np.array_equal(_np(xq).reshape(xq_ref.shape), xq_ref)
    y = _np(ops.qgemv_q4_0(ops.qpack_q4_0(_t(w), N, K), xq, M, K, N))
    r = C.check_close(y, y_ref, S)
    print(name, r)
    assert r["ok"], r


@pytest.fixture(scope="module")
def vocab(ops):
    c = synth.WORKLOADS["lmhead_q6_k"]
    w = synth.q6_k_weights(N_V, K_H, seed=c["seed"])
    x6 = synth.activations(6, K_H, seed=c["seed"] + 100)
    wd = _t(w)
    wp = ops.qpack_q6_k(wd, N_V, K_H)
    torch.cuda.synchronize()
    y_ref, S = oracle.qgemv_q6_k(w, oracle.quantize_q8_1(x6[1:6]))
    return dict(w=w, x6=x6, wd=wd, wp=wp, y_ref=y_ref, S=S)


def test_verifier_gate_up_pair_full(ops):
    # gate and up in one launch, as the benchmark runs them
    c = synth.WORKLOADS["verifier_gate_up"]
    M, K, N = c["M"], c["K"], c["N"]
    wg = synth.q4_0_weights(N, K, seed=c["seed"])
    wu = synth.q4_0_weights(N, K, seed=c["seed"] + 1)
    x = synth.activations(M, K, seed=c["seed"] + 100, outlier_frac=c["outlier_frac"])
    xq_ref = oracle.quantize_q8_1(x)
    yg, yu = ops.qgemv_q4_0_pair(ops.qpack_q4_0(_t(wg), N, K), ops.qpack_q4_0(_t(wu), N, K),
                                 ops.quantize_q8_1(_t(x)), M, K, N, N)
    for y, w in ((yg, wg), (yu, wu)):
        y_ref, S = oracle.qgemv_q4_0(w, xq_ref)
        r = C.check_close(_np(y), y_ref, S)
        print("pair", r)
        assert r["ok"], r


def test_lmhead_top1_full(ops, vocab):
    x6d = _t(vocab["x6"])
    ids = _np(ops.lmhead_q6_k_top1(vocab["wp"], x6d[1:6], K_H, N_V))
    assert C.check_top1(ids, vocab["y_ref"]) == []
    # unfused: full logits, then argmax; same ids, and the logits pass the gate
    y = ops.qgemv_q6_k(vocab["wp"], ops.quantize_q8_1(x6d[1:6]), 5, K_H, N_V)
    assert _np(ops.argmax_f32_rows(y)).tolist() == ids.tolist()
    r = C.check_close(_np(y), vocab["y_ref"], vocab["S"])
    print("lmhead logits", r)
    assert r["ok"], r
    # repeatable (workspace reset, order-independent reduction)
    assert _np(ops.lmhead_q6_k_top1(vocab["wp"], x6d[1:6], K_H, N_V)).tolist() == ids.tolist()


def test_lmhead_candmax_full(ops, vocab):
    # rows 1..5 at the full vocabulary: greedy ids and values, and candidate
    # logits equal to the unfused logits (both kernels take K whole here)
    x6d = _t(vocab["x6"])
    y_ref = vocab["y_ref"]
    ids_ref = y_ref.argmax(axis=1)
    cand = np.array([ids_ref[0], 0, N_V - 1, 123456, ids_ref[4]], dtype=np.int32)
    ids, top_vals, cand_vals = (_np(t) for t in ops.lmhead_q6_k_candmax(vocab["wp"], x6d[1:6], K_H, N_V, _t(cand)))
    assert C.check_top1(ids, y_ref) == []
    y = _np(ops.qgemv_q6_k(vocab["wp"], ops.quantize_q8_1(x6d[1:6]), 5, K_H, N_V))
    S = vocab["S"]
    for m in range(5):
        assert top_vals[m] == y[m, ids[m]]
        assert cand_vals[m] == y[m, cand[m]]
        assert abs(float(cand_vals[m]) - y_ref[m, cand[m]]) <= 1e-5 * max(abs(y_ref[m, cand[m]]), S[m, cand[m]])
    assert cand_vals[0] == top_vals[0] and cand_vals[4] == top_vals[4]


def test_lmhead_topk_full(ops, vocab):
    # rows 1..5 at the full vocabulary, k = 8: the oracle's ranking within the
    # top-k gate, and exactly the ranking of the unfused fp32 logits (both
    # kernels take K whole here, so the values are equal bit for bit)
    x6d = _t(vocab["x6"])
    y_ref, S = vocab["y_ref"], vocab["S"]
    ids_ref = y_ref.argmax(axis=1)
    cand = np.array([ids_ref[0], 0, N_V - 1, 123456, ids_ref[4]], dtype=np.int32)
    ids, vals, cv = ops.lmhead_q6_k_topk(vocab["wp"], x6d[1:6], K_H, N_V, 8, cand=_t(cand))
    ids, vals, cv = _np(ids), _np(vals), _np(cv)
    errs = C.check_topk(ids, vals, y_ref, S)
    assert errs == [], errs[:5]
    print("top-8 ranks equal to the oracle's:", int((ids == oracle.topk(y_ref, 8)[0]).sum()), "of", ids.size)
    y = _np(ops.qgemv_q6_k(vocab["wp"], ops.quantize_q8_1(x6d[1:6]), 5, K_H, N_V))
    assert np.array_equal(vals, np.take_along_axis(y, ids.astype(np.int64), axis=1))
    assert ids.tolist() == np.argsort(-y, axis=1, kind="stable")[:, :8].tolist()
    assert ids[:, 0].tolist() == _np(ops.lmhead_q6_k_top1(vocab["wp"], x6d[1:6], K_H, N_V)).tolist()
    for m in range(5):
        assert cv[m] == y[m, cand[m]]
    assert np.array_equal(_np(ops.lmhead_q6_k_topk(vocab["wp"], x6d[1:6], K_H, N_V, 8)[0]), ids)


def test_lmhead_topk_target_six_rows_full(ops, vocab):
    # the target side's six rows: the ranking of the unfused fp32 logits
    x6d = _t(vocab["x6"])
    ids, vals, _ = ops.lmhead_q6_k_topk(vocab["wp"], x6d, K_H, N_V, 8)
    ids, vals = _np(ids), _np(vals)
    y = _np(ops.qgemv_q6_k(vocab["wp"], ops.quantize_q8_1(x6d), 6, K_H, N_V))
    assert ids.tolist() == np.argsort(-y, axis=1, kind="stable")[:, :8].tolist()
    assert np.array_equal(vals, np.take_along_axis(y, ids.astype(np.int64), axis=1))


def _sample_rows(N, seed=0):
    g = np.random.default_rng(seed)
    return np.unique(np.concatenate([np.arange(min(64, N)), np.arange(max(0, N - 64), N),
                                     g.choice(N, size=min(1024, N), replace=False)]))


@pytest.mark.parametrize("fmt", ["q4_0", "q6_k"])
@pytest.mark.parametrize("N", [5120, 17408, 248320])
def test_m_sweep_sampled(ops, fmt, N):
    K = K_H
    w = synth.q4_0_weights(N, K, seed=N + 1) if fmt == "q4_0" else synth.q6_k_weights(N, K, seed=N + 2)
    wp = ops.qpack_q4_0(_t(w), N, K) if fmt == "q4_0" else ops.qpack_q6_k(_t(w), N, K)
    rows = _sample_rows(N)
    for M in (1, 2, 4, 6, 9, 12, 17):
        x = synth.activations(M, K, seed=1000 + M, outlier_frac=0.01)
        xq_ref = oracle.quantize_q8_1(x)
        xq = ops.quantize_q8_1(_t(x))
        y = _np((ops.qgemv_q4_0 if fmt == "q4_0" else ops.qgemv_q6_k)(wp, xq, M, K, N))
        f = oracle.qgemv_q4_0 if fmt == "q4_0" else oracle.qgemv_q6_k
        y_ref, S = f(w[rows], xq_ref)
        r = C.check_close(y[:, rows], y_ref, S)
        assert r["ok"], (M, r)
    del wp
    torch.cuda.empty_cache()


@pytest.mark.parametrize("fmt", ["q8_0", "q4_k", "q5_k"])
@pytest.mark.parametrize("N", [17408, 248320])
def test_further_formats_sweep_sampled(ops, fmt, N):
    # the M sweep's shapes for the further formats (their tensor-core kernel,
    # the launch configuration the sweep times), on sampled rows
    K = K_H
    w = getattr(synth, fmt + "_weights")(N, K, seed=N + 3)
    wp = getattr(ops, "qpack_" + fmt)(_t(w), N, K)
    rows = _sample_rows(N)
    for M in (1, 6, 9, 17):
        x = synth.activations(M, K, seed=2000 + M, outlier_frac=0.01)
        xq_ref = oracle.quantize_q8_1(x)
        xq = ops.quantize_q8_1(_t(x))
        y = _np(getattr(ops, "qgemv_" + fmt)(wp, xq, M, K, N))
        y_ref, S = getattr(oracle, "qgemv_" + fmt)(w[rows], xq_ref)
        r = C.check_close(y[:, rows], y_ref, S)
        assert r["ok"], (M, r)
    del wp
    torch.cuda.empty_cache()


def _set_rows(ops, vocab, rows, data):
    """Overwrite canonical rows on the device and re-pack the whole weight."""
    for r, d in zip(rows, data):
        vocab["wd"][r] = _t(d)
    ops.qpack_q6_k(vocab["wd"], N_V, K_H, out=vocab["wp"])


def test_adversarial_all_zero_weights(ops):
    w = torch.zeros((N_V, K_H // 256, 210), dtype=torch.uint8, device=DEV)
    wp = ops.qpack_q6_k(w, N_V, K_H)
    x = _t(synth.activations(6, K_H, seed=5))
    assert _np(ops.lmhead_q6_k_top1(wp, x[1:6], K_H, N_V)).tolist() == [0] * 5
    y = ops.qgemv_q6_k(wp, ops.quantize_q8_1(x[1:6]), 5, K_H, N_V)
    assert _np(ops.argmax_f32_rows(y)).tolist() == [0] * 5


@pytest.mark.parametrize("pair", [(1, 256), (255, 256), (0, 248319)])
def test_adversarial_planted_ties(ops, vocab, pair):
    x5 = vocab["x6"][1:6]
    win = C.winner_q6_k_row(x5)
    yw, _ = oracle.qgemv_q6_k(win.reshape(1, -1, 210), oracle.quantize_q8_1(x5))
    others = np.delete(vocab["y_ref"], list(pair), axis=1).max(axis=1)
    assert np.all(yw[:, 0] - others > C.TOP1_TOL * np.abs(yw[:, 0]))  # a clear winner for every row
    saved = [vocab["w"][p].copy() for p in pair]
    try:
        _set_rows(ops, vocab, pair, [win, win])
        x6d = _t(vocab["x6"])
        ids = _np(ops.lmhead_q6_k_top1(vocab["wp"], x6d[1:6], K_H, N_V))
        assert ids.tolist() == [min(pair)] * 5
        y = ops.qgemv_q6_k(vocab["wp"], ops.quantize_q8_1(x6d[1:6]), 5, K_H, N_V)
        assert _np(ops.argmax_f32_rows(y)).tolist() == [min(pair)] * 5
    finally:
        _set_rows(ops, vocab, pair, saved)


def test_adversarial_near_tie(ops, vocab):
    x5 = vocab["x6"][1:6]
    xq = oracle.quantize_q8_1(x5)
    win = C.winner_q6_k_row(x5)
    # change one code by one step at the channel with the smallest nonzero
    # activation magnitude over the five rows
    qa = np.abs(xq[:, :, 4:].view(np.int8).astype(np.int64).reshape(5, -1)).max(axis=0)
    i = int(np.argmin(np.where(qa > 0, qa, 1 << 20)))
    codes = np.zeros(K_H, dtype=np.int64)
    wf = win.reshape(-1)
    for j in range(K_H):  # decode the winner's codes (sequential packing)
        sb, t = divmod(j, 256)
        lo = (int(wf[sb * 210 + (t >> 1)]) >> (4 * (t & 1))) & 0xF
        hi = (int(wf[sb * 210 + 128 + (t >> 2)]) >> (2 * (t & 3))) & 3
        codes[j] = lo | (hi << 4)
    codes[i] += -1 if codes[i] == 63 else 1
    sc = np.full((1, K_H // 16), 63, dtype=np.int8)
    d = np.array([[1e-3] * (K_H // 256)], dtype=np.float32).astype(np.float16).view(np.uint16)
    near = C.q6_k_from_codes(codes.reshape(1, -1), sc, d)[0]
    pair = (1000, 2000)
    saved = [vocab["w"][p].copy() for p in pair]
    try:
        _set_rows(ops, vocab, pair, [near, win])
        y_ref = vocab["y_ref"].copy()
        yp, _ = oracle.qgemv_q6_k(np.stack([near, win]), xq)
        y_ref[:, list(pair)] = yp
        gap = np.abs(yp[:, 0] - yp[:, 1]) / np.abs(yp[:, 1])
        print("planted relative gaps", gap)
        x6d = _t(vocab["x6"])
        ids = _np(ops.lmhead_q6_k_top1(vocab["wp"], x6d[1:6], K_H, N_V))
        assert C.check_top1(ids, y_ref) == []
        assert set(ids.tolist()) <= set(pair)
        assert _np(ops.lmhead_q6_k_top1(vocab["wp"], x6d[1:6], K_H, N_V)).tolist() == ids.tolist()
    finally:
        _set_rows(ops, vocab, pair, saved)


def test_no_wait_timeouts(ops):
    assert ops.qgemv_take_wait_timeouts() == 0
