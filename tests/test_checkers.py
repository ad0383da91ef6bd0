"""The tolerance checkers of the parity tests, on the CPU: they accept the
oracle's own output and reject a planted mistake (in a copy of the oracle's
output) away from the stated boundaries."""
import numpy as np

import oracle
from tests import _cases as C


def _rms_case(K=1024, M=3, seed=0):
    g = np.random.default_rng(seed)
    x = (g.standard_normal((M, K)) * g.uniform(0.1, 10.0, (M, 1))).astype(np.float32)
    gamma = g.uniform(-2.0, 2.0, K).astype(np.float32)
    return oracle.rmsnorm_quantize_q8_1(x, gamma, 1e-6, with_xh=True)


def test_q8_1_near_accepts_the_oracle():
    ref, xh = _rms_case()
    r = C.check_q8_1_near(ref.copy(), ref, xh, 1024)
    assert r["ok"] and r["codes_off_by_one"] == 0 and r["scales_off_by_one"] == 0, r


def test_q8_1_near_rejects_a_code_off_by_one_away_from_a_boundary():
    ref, xh = _rms_case(seed=1)
    delta, _ = C.rmsnorm_q8_1_bounds(1024)
    d32 = (np.abs(xh.astype(np.float32)).reshape(3, 32, 32).max(axis=2) / np.float32(127)).astype(np.float64)
    t = np.abs(xh.reshape(3, 32, 32) / d32[:, :, None])
    far = np.abs(t - np.floor(t) - 0.5) > 10 * delta
    m, b, i = np.argwhere(far & (np.abs(ref[:, :, 4:].view(np.int8)) < 100))[0]
    bad = ref.copy()
    bad[m, b, 4 + i] = np.uint8((int(bad[m, b, 4 + i].view(np.int8)) + 1) & 0xFF)
    r = C.check_q8_1_near(bad, ref, xh, 1024)
    assert not r["ok"] and r["bad_codes"] == 1, r


def test_q8_1_near_rejects_a_wrong_scale():
    ref, xh = _rms_case(seed=2)
    bad = ref.copy()
    d = bad[1, 5, 0:2].copy().view(np.uint16)
    bad[1, 5, 0:2] = (d + 3).view(np.uint8)
    r = C.check_q8_1_near(bad, ref, xh, 1024)
    assert not r["ok"] and r["bad_scales"] == 1, r
