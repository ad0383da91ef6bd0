"""Pins of the oracle's fused RMSNorm -> Q8_1 (CPU only).

The oracle is the plain definition (fp64 RMSNorm, then the fp32 Q8_1
quantizer).  These pins tie it to the mathematics: closed forms whose stored
scale exposes a misplaced eps, a missing gamma or a wrong mean; hand-worked
codes that expose a gamma read at the wrong index, a sign slip or a partial
sum of squares; exact invariance under power-of-two scaling; and agreement
with an fp64 RMSNorm within half a quantization step."""
import numpy as np
import pytest

import oracle

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


def _d(xq):
    return xq[:, :, 0:2].copy().view(np.float16).astype(np.float64)[:, :, 0]


def _q(xq):
    return xq[:, :, 4:].copy().view(np.int8).astype(np.float64)


def test_closed_form_eps_gamma_mean():
    # x = 1, gamma = 2, eps = 3: r = 1 / sqrt(1 + 3) = 0.5 and xh = 1 exactly,
    # so every block is 127 with d = fp16(1/127)
    K = 32
    xq = oracle.rmsnorm_quantize_q8_1(np.ones((2, K), np.float32), np.full(K, 2.0, np.float32), 3.0)
    assert np.all(_q(xq) == 127)
    d_ok = np.float16(np.float32(1.0) / np.float32(127.0))
    assert np.all(xq[:, :, 0:2].copy().view(np.uint16) == d_ok.view(np.uint16))
    # what the plausible mistakes would store: eps outside the root
    # (xh = 2 / (1 + 3)), gamma dropped (xh = 0.5), the mean over K - 1
    # (xh = 2 / sqrt(K / (K - 1) + 3)): all differ from d_ok in fp16
    for xh in (0.5, 0.5, 2.0 / np.sqrt(K / (K - 1) + 3.0)):
        assert np.float16(np.float32(xh) / np.float32(127.0)) != d_ok


def test_power_of_two_scaling_is_exact():
    g = np.random.default_rng(1)
    x = g.standard_normal((3, 2048)).astype(np.float32)
    gamma = g.uniform(0.5, 1.5, 2048).astype(np.float32)
    base = oracle.rmsnorm_quantize_q8_1(x, gamma, 0.0)
    for s in (0.25, 8.0, 1024.0):
        assert np.array_equal(oracle.rmsnorm_quantize_q8_1(x * np.float32(s), gamma, 0.0), base)


@pytest.mark.parametrize("M,K,ldx,eps", [(1, 32, 32, 1e-6), (6, 5120, 5128, 1e-5), (3, 17408, 17408, 1e-6),
                                         (5, 96, 128, 0.0)])
def test_matches_fp64_rmsnorm(M, K, ldx, eps):
    g = np.random.default_rng(M + K)
    x = (g.standard_normal((M, ldx)) * g.uniform(0.1, 10.0, (M, 1))).astype(np.float32)
    gamma = g.uniform(-2.0, 2.0, K).astype(np.float32)
    xq = oracle.rmsnorm_quantize_q8_1(x, gamma, eps, K=K)
    x64 = x[:, :K].astype(np.float64)
    ref = x64 / np.sqrt(np.mean(x64 * x64, axis=1, keepdims=True) + eps) * gamma.astype(np.float64)
    deq = (_d(xq)[:, :, None] * _q(xq)).reshape(M, K)
    step = np.repeat(_d(xq), 32, axis=1)
    # half a step of rounding, the fp16 rounding of d (1/2048 of a code's
    # value), and the fp32 normalization
    tol = 0.5 * step + np.abs(ref) * (2.0 ** -10) + 1e-6 * np.abs(ref).max()
    assert np.all(np.abs(deq - ref) <= tol)


def test_gamma_index_pattern():
    # x = 1 everywhere and eps = 3 give r = 1/2 exactly; gamma_k = 2^(k mod 4)
    # makes xh_k = 0.5, 1, 2, 4 repeating, so every block has max 4, d =
    # 4/127 and codes round(127 xh / 4) = 16, 32, 64, 127 (15.875, 31.75 and
    # 63.5, the last rounded half away from zero).  A gamma read at the wrong
    # index, or the pattern applied per block instead of per value, moves
    # them; the second row is the first negated (sign handling).
    K = 64
    x = np.ones((2, K), np.float32)
    x[1] = -1.0
    gamma = (2.0 ** (np.arange(K) % 4)).astype(np.float32)
    xq = oracle.rmsnorm_quantize_q8_1(x, gamma, 3.0)
    want = np.tile([16, 32, 64, 127], K // 4)
    assert np.array_equal(_q(xq)[0].reshape(-1), want)
    assert np.array_equal(_q(xq)[1].reshape(-1), -want)
    d = np.float16(np.float32(4.0) / np.float32(127.0))
    assert np.all(xq[:, :, 0:2].copy().view(np.uint16) == d.view(np.uint16))


def test_sum_of_squares_over_the_whole_row():
    # row [1]*16 + [3]*16 (K = 32): mean of squares (16 + 144) / 32 = 5, so
    # eps = 4 gives r = 1/3 and, with gamma = 3, xh = x: codes round(127/3) =
    # 42 for the ones and 127 for the threes, d = 3/127.  Summing over part of
    # the row, or the squares of the wrong values, changes r and d.
    K = 32
    x = np.array([[1.0] * 16 + [3.0] * 16], np.float32)
    xq, xh = oracle.rmsnorm_quantize_q8_1(x, np.full(K, 3.0, np.float32), 4.0, with_xh=True)
    assert np.array_equal(_q(xq)[0, 0], [42] * 16 + [127] * 16)
    assert np.allclose(xh[0], x[0].astype(np.float64), rtol=0, atol=1e-15)
    d = np.float16(np.float32(3.0) / np.float32(127.0))
    assert xq[0, 0, 0:2].copy().view(np.uint16)[0] == d.view(np.uint16)
