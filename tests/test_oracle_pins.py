"""Pins for the CPU oracle: each test checks it against something other than
itself (IEEE binary16 via numpy, hand-worked blocks, an independent numpy
dequantizer, algebraic invariants, the pages' byte count, planted ties)."""
import json
import os

import numpy as np
import pytest

import oracle
from block_quantized_gemv_quantize_gb300 import synth

GOLDEN = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "single_blocks.json")))


def _q4_0_block(d: float, codes) -> np.ndarray:
    codes = np.asarray(codes, dtype=np.uint8)
    blk = np.zeros(18, dtype=np.uint8)
    blk[0:2] = np.array([d], dtype=np.float16).view(np.uint8)
    blk[2:18] = (codes[:16] & 0x0F) | ((codes[16:] & 0x0F) << 4)
    return blk


def _q6_k_superblock(d: float, sc, codes) -> np.ndarray:
    codes = np.asarray(codes, dtype=np.int64)
    sb = np.zeros(210, dtype=np.uint8)
    for i in range(256):
        sb[i >> 1] |= (codes[i] & 0x0F) << (4 * (i & 1))
        sb[128 + (i >> 2)] |= ((codes[i] >> 4) & 3) << (2 * (i & 3))
    sb[192:208] = np.asarray(sc, dtype=np.int8).view(np.uint8)
    sb[208:210] = np.array([d], dtype=np.float16).view(np.uint8)
    return sb


# ---------------------------------------------------------------- binary16

def test_f32_to_f16_matches_ieee_rne():
    g = np.random.default_rng(1)
    vals = np.concatenate([
        g.standard_normal(3000).astype(np.float32) * np.float32(10.0) ** g.integers(-9, 6, 3000).astype(np.float32),
        np.array([0.0, -0.0, 65504.0, 65519.0, 65520.0, 1e6, -1e6, 2.0 ** -14, 2.0 ** -24, 2.0 ** -25,
                  3 * 2.0 ** -26, 2.0 ** -26, 1.0 + 2.0 ** -11, 1.0 + 3 * 2.0 ** -11, 6.1e-5, 5.96e-8,
                  np.inf, -np.inf], dtype=np.float32),
    ])
    mine = oracle.f32_to_f16_bits(vals)
    with np.errstate(over="ignore"):
        ref = vals.astype(np.float16).view(np.uint16)
    assert np.array_equal(mine, ref)


def test_f16_decode_exact():
    bits = np.arange(0, 65536, dtype=np.uint32).astype(np.uint16)
    bits = bits[(bits & 0x7C00) != 0x7C00]  # finite only
    mine = oracle.f16_bits_to_f64(bits)
    ref = bits.view(np.float16).astype(np.float64)
    assert np.array_equal(mine, ref)


# ---------------------------------------------------------------- Q8_1

def test_q8_1_hand_block():
    g = GOLDEN["q8_1_all_ones"]
    xq = oracle.quantize_q8_1(np.ones((1, 32), dtype=np.float32))
    d16 = int(xq[0, 0, 0]) | (int(xq[0, 0, 1]) << 8)
    s16 = int(xq[0, 0, 2]) | (int(xq[0, 0, 3]) << 8)
    assert d16 == int(g["d16_bits"], 16)
    assert s16 == int(g["s16_bits"], 16)
    assert np.all(xq[0, 0, 4:].view(np.int8) == g["q"])


def test_q8_1_rounds_half_away_from_zero():
    # amax = 127 makes d = 1 exactly, so x/d is x itself: the ties are exact.
    x = np.zeros((1, 32), dtype=np.float32)
    x[0, 0] = 127.0
    x[0, 1:7] = [2.5, -2.5, 0.5, -0.5, 3.5, 126.5]
    xq = oracle.quantize_q8_1(x)
    q = xq[0, 0, 4:].view(np.int8)
    assert q[:7].tolist() == [127, 3, -3, 1, -1, 4, 127]


def test_q8_1_divides_by_fp32_scale_not_fp16():
    # amax = 1: fp32 d = 1/127, its fp16 rounding is 1032/131072.  x = 0.05118
    # gives 6 with the fp32 d and 7 with the fp16 one.
    x = np.zeros((1, 32), dtype=np.float32)
    x[0, 0] = 1.0
    x[0, 1] = np.float32(0.05118)
    q = oracle.quantize_q8_1(x)[0, 0, 4:].view(np.int8)
    d32 = np.float32(1.0) / np.float32(127.0)
    assert q[1] == int(np.floor(x[0, 1] / d32 + np.float32(0.5)))
    assert q[1] == 6


def test_q8_1_properties():
    x = synth.activations(4, 512, seed=7, outlier_frac=0.02)
    xq = oracle.quantize_q8_1(x)
    q = xq[:, :, 4:].view(np.int8).astype(np.int64)
    xb = x.reshape(4, 16, 32)
    amax = np.abs(xb).max(axis=2)
    # the largest |x| of each block maps to +-127, and |q| <= 127
    arg = np.abs(xb).argmax(axis=2)
    assert np.all(np.abs(np.take_along_axis(q, arg[..., None], 2)) == 127)
    assert np.all(np.abs(q) <= 127)
    # q = round(x / d) with the fp32 d = amax/127: |x/d - q| <= 1/2
    d32 = (amax / np.float32(127.0)).astype(np.float32)
    r = xb / d32[..., None]
    assert np.all(np.abs(r - q) <= 0.5)
    # stored fp16 d is the RNE rounding of d; s is fp16(d * sum q)
    d16 = xq[:, :, 0:2].copy().view(np.float16)[..., 0]
    assert np.array_equal(d16, d32.astype(np.float16))
    s16 = xq[:, :, 2:4].copy().view(np.float16)[..., 0]
    assert np.array_equal(s16, (d32 * q.sum(axis=2).astype(np.float32)).astype(np.float16))
    # sign symmetry
    xq_neg = oracle.quantize_q8_1(-x)
    assert np.array_equal(xq_neg[:, :, 4:].view(np.int8), -xq[:, :, 4:].view(np.int8))
    assert np.array_equal(xq_neg[:, :, 0:2], xq[:, :, 0:2])


def test_q8_1_zero_block_and_power_of_two_scaling():
    x = synth.activations(2, 256, seed=3)
    x[1, 64:96] = 0.0
    xq = oracle.quantize_q8_1(x)
    assert np.all(xq[1, 2] == 0)
    for k in (-3, 4):
        xs = (x * np.float32(2.0 ** k)).astype(np.float32)
        xqs = oracle.quantize_q8_1(xs)
        assert np.array_equal(xqs[:, :, 4:], xq[:, :, 4:])
        d = xq[:, :, 0:2].copy().view(np.float16).astype(np.float64)
        ds = xqs[:, :, 0:2].copy().view(np.float16).astype(np.float64)
        nz = d != 0
        assert np.array_equal(ds[nz], d[nz] * 2.0 ** k)


# ---------------------------------------------------------------- hand blocks

def test_q4_0_hand_block():
    g = GOLDEN["q4_0_block_times_ones"]
    w = _q4_0_block(1.0, [9] * 32).reshape(1, 1, 18)
    xq = oracle.quantize_q8_1(np.ones((1, 32), dtype=np.float32))
    assert oracle.block_dots_q4_0(w, xq)[0, 0, 0] == g["I"]
    y, S = oracle.qgemv_q4_0(w, xq)
    assert y[0, 0] == g["y"]
    assert S[0, 0] == g["y"]


def test_q6_k_hand_superblock():
    g = GOLDEN["q6_k_superblock_times_ones"]
    w = _q6_k_superblock(2.0 ** -10, [1] * 16, [33] * 256).reshape(1, 1, 210)
    xq = oracle.quantize_q8_1(np.ones((1, 256), dtype=np.float32))
    assert np.all(oracle.block_dots_q6_k(w, xq) == g["J_per_block"])
    y, _ = oracle.qgemv_q6_k(w, xq)
    assert y[0, 0] == g["y"]


def test_q6_k_codes_subscales_and_offsets_hand():
    # distinct codes and subscales: the dot against a one-hot activation reads
    # back exactly one weight value d * sc * (q - 32)
    g = np.random.default_rng(5)
    codes = g.integers(0, 64, 256)
    sc = g.integers(-64, 64, 16)
    w = _q6_k_superblock(2.0 ** -8, sc, codes).reshape(1, 1, 210)
    for i in (0, 1, 15, 16, 17, 31, 100, 129, 255):
        x = np.zeros((1, 256), dtype=np.float32)
        x[0, i] = 1.0
        xq = oracle.quantize_q8_1(x)
        y, _ = oracle.qgemv_q6_k(w, xq)
        expect = 2.0 ** -8 * sc[i >> 4] * (codes[i] - 32) * 127 * (1032 / 131072)
        assert y[0, 0] == expect, i


def test_q4_0_codes_one_hot():
    g = np.random.default_rng(6)
    codes = g.integers(0, 16, 32)
    w = _q4_0_block(0.5, codes).reshape(1, 1, 18)
    for i in range(32):
        x = np.zeros((1, 32), dtype=np.float32)
        x[0, i] = -1.0
        y, _ = oracle.qgemv_q4_0(w, oracle.quantize_q8_1(x))
        assert y[0, 0] == 0.5 * (codes[i] - 8) * -127 * (1032 / 131072), i


# ---------------------------------------------------------------- brute force

@pytest.mark.parametrize("M", [1, 2, 3])
@pytest.mark.parametrize("K", [32, 64, 256, 512])
@pytest.mark.parametrize("N", [1, 2, 3, 7, 33])
def test_q4_0_int_dots_match_fp64_dequant_matmul(M, K, N):
    w = synth.q4_0_weights(N, K, seed=100 + K + N)
    xq = oracle.quantize_q8_1(synth.activations(M, K, seed=200 + M))
    y, S = oracle.qgemv_q4_0(w, xq)
    ref = oracle.dequant_q8_1_np(xq) @ oracle.dequant_q4_0_np(w).T
    assert np.all(np.abs(y - ref) <= 1e-12 * np.maximum(S, 1e-300))


@pytest.mark.parametrize("M", [1, 2, 3])
@pytest.mark.parametrize("K", [256, 512])
@pytest.mark.parametrize("N", [1, 2, 3, 7, 33])
def test_q6_k_int_dots_match_fp64_dequant_matmul(M, K, N):
    w = synth.q6_k_weights(N, K, seed=300 + K + N)
    xq = oracle.quantize_q8_1(synth.activations(M, K, seed=400 + M))
    y, S = oracle.qgemv_q6_k(w, xq)
    ref = oracle.dequant_q8_1_np(xq) @ oracle.dequant_q6_k_np(w).T
    assert np.all(np.abs(y - ref) <= 1e-12 * np.maximum(S, 1e-300))


def test_c_and_numpy_dequantizers_agree():
    w4 = synth.q4_0_weights(5, 256, seed=1)
    w6 = synth.q6_k_weights(5, 512, seed=2)
    out4 = np.zeros((5, 256))
    out6 = np.zeros((5, 512))
    lib = oracle.oracle._load()
    lib.oracle_dequant_q4_0(w4.ctypes.data, 5, 256, out4.ctypes.data)
    lib.oracle_dequant_q6_k(w6.ctypes.data, 5, 512, out6.ctypes.data)
    assert np.array_equal(out4, oracle.dequant_q4_0_np(w4))
    assert np.array_equal(out6, oracle.dequant_q6_k_np(w6))


def test_block_dots_sum_to_output():
    w = synth.q4_0_weights(9, 512, seed=4)
    xq = oracle.quantize_q8_1(synth.activations(2, 512, seed=5))
    I = oracle.block_dots_q4_0(w, xq).astype(np.float64)
    dw = w[:, :, 0:2].copy().view(np.float16)[..., 0].astype(np.float64)
    da = xq[:, :, 0:2].copy().view(np.float16)[..., 0].astype(np.float64)
    y = (I * dw[None, :, :] * da[:, None, :]).sum(axis=2)
    ref, _ = oracle.qgemv_q4_0(w, xq)
    assert np.allclose(y, ref, rtol=1e-13, atol=0)


def _q6_k_decode_numpy(w: np.ndarray):
    """Codes, subscales and d of canonical Q6_K superblocks [N, ns, 210],
    decoded in numpy from the documented byte layout (ql[128], qh[64], int8
    sc[16], fp16 d; value i: low 4 bits = nibble (i & 1) of ql[i >> 1], high 2
    bits = bits 2 (i & 3) of qh[i >> 2]; subscale i >> 4)."""
    i = np.arange(256)
    lo = (w[..., i >> 1] >> (4 * (i & 1))) & 0x0F
    hi = (w[..., 128 + (i >> 2)] >> (2 * (i & 3))) & 0x03
    q = (lo | (hi << 4)).astype(np.int64)
    sc = w[..., 192:208].copy().view(np.int8).astype(np.int64)
    d = w[..., 208:210].copy().view(np.float16)[..., 0].astype(np.float64)
    return q, sc, d


def test_q6_k_block_dots_match_per_block_dequant():
    # random superblocks: each J[m, n, b], scaled by d6 of its superblock and
    # d_a of its block, is the fp64 dot of block b's dequantized weights and
    # activations; a slip in the (superblock, block) index or in the
    # [m][n][b] layout breaks the match at once
    M, K, N = 3, 1024, 7
    w = synth.q6_k_weights(N, K, seed=21)
    xq = oracle.quantize_q8_1(synth.activations(M, K, seed=22))
    J = oracle.block_dots_q6_k(w, xq).astype(np.float64)
    assert J.shape == (M, N, K // 32)
    q, sc, d = _q6_k_decode_numpy(w)
    wdq = (d[:, :, None] * sc[:, :, np.arange(256) >> 4] * (q - 32)).reshape(N, K)
    da = xq[:, :, 0:2].copy().view(np.float16)[..., 0].astype(np.float64)
    qa = xq[:, :, 4:].copy().view(np.int8).astype(np.float64)
    adq = (da[:, :, None] * qa).reshape(M, K)
    per_block = np.einsum("mbi,nbi->mnb", adq.reshape(M, K // 32, 32), wdq.reshape(N, K // 32, 32))
    d6 = np.repeat(d, 8, axis=1)  # the superblock scale of each block
    got = J * d6[None, :, :] * da[:, None, :]
    assert np.allclose(got, per_block, rtol=1e-13, atol=1e-300)
    y, _ = oracle.qgemv_q6_k(w, xq)
    assert np.allclose(got.sum(axis=2), y, rtol=1e-12, atol=0)


def test_q6_k_block_dots_one_hot_per_half():
    # a one-hot activation at value i of superblock s reads back, in block
    # 8 s + (i mod 256) // 32 only, sc[(i mod 256) // 16] * (q_i - 32) * 127
    # (the one-hot's code); every other block dot is 0
    N, K = 2, 512
    g = np.random.default_rng(23)
    codes = g.integers(0, 64, (N, 2, 256))
    sc = g.integers(-64, 64, (N, 2, 16))
    w = np.stack([np.stack([_q6_k_superblock(2.0 ** -9, sc[n, s], codes[n, s]) for s in range(2)])
                  for n in range(N)])
    for i in (0, 15, 16, 31, 32, 47, 200, 255, 256, 271, 300, 511):
        x = np.zeros((1, K), dtype=np.float32)
        x[0, i] = 1.0
        J = oracle.block_dots_q6_k(w, oracle.quantize_q8_1(x))
        s, v = i // 256, i % 256
        for n in range(N):
            want = np.zeros(K // 32, dtype=np.int64)
            want[8 * s + v // 32] = sc[n, s, v // 16] * (codes[n, s, v] - 32) * 127
            assert np.array_equal(J[0, n], want), (i, n)


def test_threads_do_not_change_results():
    w = synth.q6_k_weights(37, 512, seed=8)
    xq = oracle.quantize_q8_1(synth.activations(3, 512, seed=9))
    y1, s1 = oracle.qgemv_q6_k(w, xq, nthreads=1)
    y4, s4 = oracle.qgemv_q6_k(w, xq, nthreads=4)
    assert np.array_equal(y1, y4) and np.array_equal(s1, s4)


# ---------------------------------------------------------------- invariants

def test_invariants_zero_row_permutation_scaling():
    K, N = 512, 40
    w = synth.q4_0_weights(N, K, seed=11)
    x = synth.activations(3, K, seed=12)
    x[1] = 0.0
    xq = oracle.quantize_q8_1(x)
    y, _ = oracle.qgemv_q4_0(w, xq)
    assert np.all(y[1] == 0.0)
    perm = np.random.default_rng(0).permutation(N)
    yp, _ = oracle.qgemv_q4_0(w[perm], xq)
    assert np.array_equal(yp, y[:, perm])
    ys, _ = oracle.qgemv_q4_0(w, oracle.quantize_q8_1(x * np.float32(4.0)))
    assert np.array_equal(ys, 4.0 * y)


# ---------------------------------------------------------------- byte counts

def test_pages_expanded_pack_byte_count():
    g = GOLDEN["q6_k_expanded_pack_bytes"]
    ns = g["K"] // 256
    # expanded: 256 int8 quants + 16 int8 subscales + one fp16 scale per superblock
    assert g["N"] * ns * (256 + 16 + 2) == g["expanded_bytes"]
    # canonical 6-bit superblock
    assert synth.Q6_K_BYTES == 256 * 6 // 8 + 16 + 2
    assert g["N"] * ns * synth.Q6_K_BYTES == g["canonical_bytes"]
    assert synth.Q4_0_BYTES == 32 * 4 // 8 + 2


# ---------------------------------------------------------------- top-1

def test_top1_ties_and_specials():
    y = np.zeros((6, 300))
    y[1, [1, 256]] = 5.0
    y[2, [255, 256]] = 5.0
    y[3, [0, 299]] = 5.0
    y[4, :] = np.nan
    y[5, 10] = -0.0
    y[5, :] = -1.0
    y[5, 7] = 0.0
    y[5, 3] = -0.0
    assert oracle.top1(y).tolist() == [0, 1, 255, 0, 0, 3]
    z = np.full((2, 10), -np.inf)
    z[0, 4] = np.inf
    z[0, 6] = np.inf
    z[1, 2] = np.nan
    assert oracle.top1(z).tolist() == [4, 0]
    assert oracle.top1(y.astype(np.float32)).tolist() == [0, 1, 255, 0, 0, 3]


def test_top1_all_zero_weights_give_token_0():
    w = np.zeros((64, 1, 210), dtype=np.uint8)
    ids, y, _ = oracle.lmhead_q6_k_top1(w, synth.activations(5, 256, seed=1))
    assert np.all(y == 0.0) and ids.tolist() == [0] * 5


def test_top1_matches_brute_force_argmax():
    w = synth.q6_k_weights(300, 512, seed=21)
    x = synth.activations(4, 512, seed=22)
    ids, y, _ = oracle.lmhead_q6_k_top1(w, x)
    ref = oracle.dequant_q8_1_np(oracle.quantize_q8_1(x)) @ oracle.dequant_q6_k_np(w).T
    assert ids.tolist() == np.argmax(ref, axis=1).tolist()


def _topk_by_repeated_max(row, k):
    """Brute force, a different procedure from the oracle's sort: k passes,
    each taking the first (lowest-index) strict maximum among the unused
    non-NaN entries."""
    used, ids, vals = set(), [], []
    for _ in range(k):
        best = None
        for n, v in enumerate(row):
            if n in used or v != v:
                continue
            if best is None or v > row[best]:
                best = n
        if best is None:
            ids.append(-1)
            vals.append(float("nan"))
        else:
            used.add(best)
            ids.append(best)
            vals.append(float(row[best]))
    return ids, vals


def test_topk_hand_example():
    y = np.array([[1.0, 5.0, 3.0, 5.0, np.nan, -2.0, 3.0],
                  [np.nan, np.nan, 2.0, np.nan, np.nan, np.nan, np.nan],
                  [-0.0, 0.0, -1.0, np.inf, -np.inf, 0.0, -0.0]])
    ids, vals = oracle.topk(y, 4)
    assert ids.tolist() == [[1, 3, 2, 6], [2, -1, -1, -1], [3, 0, 1, 5]]
    assert vals[0].tolist() == [5.0, 5.0, 3.0, 3.0]
    assert vals[1, 0] == 2.0 and np.isnan(vals[1, 1:]).all()
    assert vals[2].tolist() == [np.inf, 0.0, 0.0, 0.0]


def test_topk_matches_repeated_max_brute_force():
    g = np.random.default_rng(5)
    for trial in range(40):
        N = int(g.integers(1, 40))
        # few distinct values, so that ties are common; some NaN
        y = g.integers(-3, 4, size=(3, N)).astype(np.float64)
        y[g.random((3, N)) < 0.15] = np.nan
        k = int(g.integers(1, 9))
        ids, vals = oracle.topk(y, k)
        for m in range(3):
            bi, bv = _topk_by_repeated_max(y[m].tolist(), k)
            assert ids[m].tolist() == bi, (trial, m)
            np.testing.assert_array_equal(vals[m], np.array(bv))


def test_topk_first_entry_is_top1():
    y = synth.activations(6, 1000, seed=31).astype(np.float64)
    y[2, 17] = y[2, 400] = y[2].max() + 1.0  # an exact tie for the maximum
    ids, _ = oracle.topk(y, 5)
    assert ids[:, 0].tolist() == oracle.top1(y).tolist()


def test_lmhead_topk_matches_fp64_dequant_matmul():
    w = synth.q6_k_weights(300, 512, seed=23)
    x = synth.activations(4, 512, seed=24)
    ids, vals, y, _ = oracle.lmhead_q6_k_topk(w, x, 8)
    ref = oracle.dequant_q8_1_np(oracle.quantize_q8_1(x)) @ oracle.dequant_q6_k_np(w).T
    assert ids.tolist() == np.argsort(-ref, axis=1, kind="stable")[:, :8].tolist()
    np.testing.assert_allclose(vals, np.take_along_axis(ref, ids.astype(np.int64), axis=1), rtol=1e-12, atol=1e-12)


# ---------------------------------------------------------------- pack layout model (test helpers)

@pytest.mark.parametrize("N,K", [(3, 32), (2, 96), (5, 256), (4, 1056), (3, 5120), (8, 2048)])
def test_pack_q4_0_model_round_trip(N, K):
    from tests import _cases as C

    w = synth.q4_0_weights(N, K, seed=K)
    p = C.pack_q4_0(w)
    if K % 256 == 0:
        assert p.size == w.size
    assert np.array_equal(C.unpack_q4_0(p, N, K), w)


@pytest.mark.parametrize("N,K", [(3, 256), (2, 768), (4, 5120), (9, 1024), (5, 2048)])
def test_pack_q6_k_model_round_trip(N, K):
    from tests import _cases as C

    w = synth.q6_k_weights(N, K, seed=K)
    p = C.pack_q6_k(w)
    if N % 4 == 0 and K % 1024 == 0:
        assert p.size == w.size
    assert np.array_equal(C.unpack_q6_k(p, N, K), w)


# ---------------------------------------------------------------- Q8_0 (a further format)

def test_q8_0_hand_block():
    # one block: d = 0.5, q = (i - 16) for i = 0..31, against a Q8_1 block of
    # all 2s with d = 1/64 (stored exactly): y = 0.5 * (1/64) * 2 * sum(i - 16)
    w = np.zeros((1, 1, 34), dtype=np.uint8)
    w[0, 0, 0:2] = np.array([0.5], dtype=np.float16).view(np.uint8)
    w[0, 0, 2:] = (np.arange(32) - 16).astype(np.int8).view(np.uint8)
    xq = np.zeros((1, 1, 36), dtype=np.uint8)
    xq[0, 0, 0:2] = np.array([1.0 / 64], dtype=np.float16).view(np.uint8)
    xq[0, 0, 4:] = 2
    y, S = oracle.qgemv_q8_0(w, xq)
    assert y[0, 0] == 0.5 * (1.0 / 64) * 2 * float(np.sum(np.arange(32) - 16)) == -0.25
    assert S[0, 0] == 0.25


@pytest.mark.parametrize("M,K,N", [(1, 32, 1), (3, 256, 7), (2, 512, 33), (5, 1024, 16)])
def test_q8_0_matches_fp64_dequant_matmul(M, K, N):
    w = synth.q8_0_weights(N, K, seed=300 + K + N)
    xq = oracle.quantize_q8_1(synth.activations(M, K, seed=400 + M))
    y, S = oracle.qgemv_q8_0(w, xq)
    ref = oracle.dequant_q8_1_np(xq) @ oracle.dequant_q8_0_np(w).T
    assert np.all(np.abs(y - ref) <= 1e-12 * np.maximum(S, 1e-300))
    assert np.array_equal(oracle.dequant_q8_0(w), oracle.dequant_q8_0_np(w))


def test_q8_0_code_sign_and_position():
    # a single code +1 at position i of block b must pick activation value (b, i)
    # with its sign; -1 flips it (no offset in Q8_0, unlike Q4_0's q - 8)
    K, N = 128, 1
    x = synth.activations(1, K, seed=5)
    xq = oracle.quantize_q8_1(x)
    xd = oracle.dequant_q8_1_np(xq)[0]
    for b, i, s in ((0, 0, 1), (1, 31, -1), (3, 17, 1)):
        w = np.zeros((N, K // 32, 34), dtype=np.uint8)
        w[0, b, 0:2] = np.array([1.0], dtype=np.float16).view(np.uint8)
        w[0, b, 2 + i] = np.int8(s).view(np.uint8)
        y, _ = oracle.qgemv_q8_0(w, xq)
        assert y[0, 0] == s * xd[32 * b + i]


# ---------------------------------------------------------------- Q4_K (a further format)

# Twelve scale bytes chosen to exercise every field of the packing, with the
# (scale, min) pairs worked out by hand from the llama.cpp layout:
#   j < 4:  scale = byte j & 63, min = byte j + 4 & 63
#   j >= 4: scale = (byte j + 4 & 15) | (byte j - 4 >> 6) << 4,
#           min   = (byte j + 4 >> 4) | (byte j >> 6) << 4
Q4_K_SCALE_BYTES = [0x41, 0x02, 0xC3, 0x04, 0x85, 0x46, 0x07, 0xC8, 0x9A, 0x0B, 0xFC, 0x3D]
Q4_K_HAND_SC = [1, 2, 3, 4, 26, 11, 60, 13]   # e.g. j = 4: 0x9A & 15 = 10, 0x41 >> 6 = 1 -> 26
Q4_K_HAND_M = [5, 6, 7, 8, 41, 16, 15, 51]    # e.g. j = 7: 0x3D >> 4 = 3, 0xC8 >> 6 = 3 -> 51


def _q4_k_superblock(d: float, dmin: float, scale_bytes, qs) -> np.ndarray:
    sb = np.zeros(144, dtype=np.uint8)
    sb[0:2] = np.array([d], dtype=np.float16).view(np.uint8)
    sb[2:4] = np.array([dmin], dtype=np.float16).view(np.uint8)
    sb[4:16] = np.asarray(scale_bytes, dtype=np.uint8)
    sb[16:144] = np.asarray(qs, dtype=np.uint8)
    return sb


def test_q4_k_scale_min_hand_table():
    # every code 1 (qs bytes 0x11), d = dmin = 1: value = sc_j - m_j per 32-value sub-block
    w = _q4_k_superblock(1.0, 1.0, Q4_K_SCALE_BYTES, np.full(128, 0x11))[None, None]
    expect = np.repeat(np.array(Q4_K_HAND_SC, dtype=np.float64) - np.array(Q4_K_HAND_M), 32)
    assert np.array_equal(oracle.dequant_q4_k(w)[0], expect)
    assert np.array_equal(oracle.dequant_q4_k_np(w)[0], expect)
    # codes 0 leave -dmin * m; codes 15 give 15 sc - m
    w0 = _q4_k_superblock(1.0, 0.5, Q4_K_SCALE_BYTES, np.zeros(128))[None, None]
    assert np.array_equal(oracle.dequant_q4_k(w0)[0], np.repeat(-0.5 * np.array(Q4_K_HAND_M, dtype=np.float64), 32))
    w15 = _q4_k_superblock(1.0, 1.0, Q4_K_SCALE_BYTES, np.full(128, 0xFF))[None, None]
    assert np.array_equal(oracle.dequant_q4_k(w15)[0],
                          np.repeat(15.0 * np.array(Q4_K_HAND_SC) - np.array(Q4_K_HAND_M), 32))


def test_q4_k_code_order_hand_example():
    # qs[0] = 0x21 and qs[37] = 0x0A, every other byte 0; unit scales, no mins:
    # value 0 = 1 (low nibble of qs[0]), value 32 = 2 (its high nibble);
    # qs[37] sits in the second 32-byte group, so value 64 + 5 = 10 and value
    # 64 + 32 + 5 = 0; everything else is 0
    unit = [1, 1, 1, 1, 0, 0, 0, 0, 0x01, 0x01, 0x01, 0x01]
    qs = np.zeros(128, dtype=np.uint8)
    qs[0], qs[37] = 0x21, 0x0A
    v = oracle.dequant_q4_k(_q4_k_superblock(1.0, 0.0, unit, qs)[None, None])[0]
    expect = np.zeros(256)
    expect[0], expect[32], expect[69] = 1.0, 2.0, 10.0
    assert np.array_equal(v, expect)
    assert np.array_equal(oracle.dequant_q4_k_np(_q4_k_superblock(1.0, 0.0, unit, qs)[None, None])[0], expect)


@pytest.mark.parametrize("M,K,N", [(1, 256, 1), (3, 256, 7), (2, 512, 33), (5, 1024, 16)])
def test_q4_k_matches_fp64_dequant_matmul(M, K, N):
    w = synth.q4_k_weights(N, K, seed=500 + K + N)
    xq = oracle.quantize_q8_1(synth.activations(M, K, seed=600 + M))
    y, S = oracle.qgemv_q4_k(w, xq)
    ref = oracle.dequant_q8_1_np(xq) @ oracle.dequant_q4_k_np(w).T
    assert np.all(np.abs(y - ref) <= 1e-12 * np.maximum(S, 1e-300))
    assert np.array_equal(oracle.dequant_q4_k(w), oracle.dequant_q4_k_np(w))


def test_q4_k_min_term_closed_form():
    # all codes 0, every min 1 (scale bytes 0x00 x4, 0x01 x4, then 0x10 x4), dmin = 2:
    # y = -2 * sum of the (dequantized) activation values
    K, N = 512, 1
    mins = [0, 0, 0, 0, 1, 1, 1, 1, 0x10, 0x10, 0x10, 0x10]
    w = np.stack([_q4_k_superblock(0.25, 2.0, mins, np.zeros(128)) for _ in range(K // 256)])[None]
    x = synth.activations(2, K, seed=7)
    xq = oracle.quantize_q8_1(x)
    y, _ = oracle.qgemv_q4_k(w, xq)
    assert np.allclose(y[:, 0], -2.0 * oracle.dequant_q8_1_np(xq).sum(axis=1), rtol=1e-13, atol=0)


# ---------------------------------------------------------------- Q5_K (a further format)

def _q5_k_superblock(d: float, dmin: float, scale_bytes, qh, qs) -> np.ndarray:
    sb = np.zeros(176, dtype=np.uint8)
    sb[0:2] = np.array([d], dtype=np.float16).view(np.uint8)
    sb[2:4] = np.array([dmin], dtype=np.float16).view(np.uint8)
    sb[4:16] = np.asarray(scale_bytes, dtype=np.uint8)
    sb[16:48] = np.asarray(qh, dtype=np.uint8)
    sb[48:176] = np.asarray(qs, dtype=np.uint8)
    return sb


def test_q5_k_fifth_bit_hand_example():
    # unit scales, no mins; qh[0] = 0x81 sets the fifth bit of value 0 (bit 0:
    # sub-block 0, position 0) and of value 224 (bit 7: sub-block 7, position 0);
    # qh[3] = 0x04 that of value 67 (sub-block 2, position 3); qs[0] = 0x0F adds
    # 15 to value 0: values 0 = 31, 67 = 16, 224 = 16, all others 0
    unit = [1, 1, 1, 1, 0, 0, 0, 0, 0x01, 0x01, 0x01, 0x01]
    qh = np.zeros(32, dtype=np.uint8)
    qh[0], qh[3] = 0x81, 0x04
    qs = np.zeros(128, dtype=np.uint8)
    qs[0] = 0x0F
    w = _q5_k_superblock(1.0, 0.0, unit, qh, qs)[None, None]
    expect = np.zeros(256)
    expect[0], expect[67], expect[224] = 31.0, 16.0, 16.0
    assert np.array_equal(oracle.dequant_q5_k(w)[0], expect)
    assert np.array_equal(oracle.dequant_q5_k_np(w)[0], expect)


@pytest.mark.parametrize("M,K,N", [(1, 256, 1), (3, 256, 7), (2, 512, 33), (5, 1024, 16)])
def test_q5_k_matches_fp64_dequant_matmul(M, K, N):
    w = synth.q5_k_weights(N, K, seed=700 + K + N)
    xq = oracle.quantize_q8_1(synth.activations(M, K, seed=800 + M))
    y, S = oracle.qgemv_q5_k(w, xq)
    ref = oracle.dequant_q8_1_np(xq) @ oracle.dequant_q5_k_np(w).T
    assert np.all(np.abs(y - ref) <= 1e-12 * np.maximum(S, 1e-300))
    assert np.array_equal(oracle.dequant_q5_k(w), oracle.dequant_q5_k_np(w))


def test_q5_k_without_fifth_bits_is_q4_k():
    # with every qh bit clear a Q5_K superblock is the Q4_K superblock of the
    # same d, dmin, scales and codes
    K, N = 1024, 9
    w5 = synth.q5_k_weights(N, K, seed=31)
    w5[:, :, 16:48] = 0
    w4 = np.concatenate([w5[:, :, 0:16], w5[:, :, 48:176]], axis=2)
    xq = oracle.quantize_q8_1(synth.activations(3, K, seed=32))
    y5, S5 = oracle.qgemv_q5_k(w5, xq)
    y4, S4 = oracle.qgemv_q4_k(w4, xq)
    assert np.array_equal(y5, y4) and np.array_equal(S5, S4)
