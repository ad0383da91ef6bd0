"""Parity of the CUDA path (through the C ABI) with the CPU oracle.

Gates: Q8_1 and the int32 block dots bit-exact; fp32 outputs within
|err| <= 1e-5 * max(|y_oracle|, S) with S = sum_b |d_w d_a I_b|; top-1 ids exact
where the oracle's top-2 gap exceeds 1e-4 * |top1| (otherwise any id within
that tolerance), planted exact ties resolved to the lower id; argmax over the
GPU's own fp32 logits bit-exact."""
import ctypes

import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import oracle  # noqa: E402
from block_quantized_gemv_quantize_gb300 import synth  # noqa: E402

from . import _cases as C  # noqa: E402


@pytest.fixture(scope="module")
def ops():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from block_quantized_gemv_quantize_gb300 import build

    build.build()
    from block_quantized_gemv_quantize_gb300 import ops as o

    return o


DEV = "cuda:0"


def _t(a):
    return torch.from_numpy(np.ascontiguousarray(a)).to(DEV)


def _np(t):
    torch.cuda.synchronize()
    return t.cpu().numpy()


# ---------------------------------------------------------------- A1 quantize

@pytest.mark.parametrize("M,K,ldx", [(1, 32, 32), (1, 256, 256), (5, 5120, 5120), (6, 5120, 5200),
                                     (6, 17408, 17408), (17, 1024, 1056), (3, 64, 64)])
def test_quantize_q8_1_bit_exact(ops, M, K, ldx):
    x = synth.activations(M, ldx, seed=K + M, outlier_frac=0.01)
    x[0, :32] = 0.0                      # an all-zero block
    x[-1, 32:64] *= np.float32(1e-30)    # tiny (fp32-subnormal after division) values
    ref = oracle.quantize_q8_1(x, K)
    got = _np(ops.quantize_q8_1(_t(x), K)).reshape(ref.shape)
    assert np.array_equal(got, ref)


# ---------------------------------------------------------------- A2 pack

@pytest.mark.parametrize("N,K", [(1, 32), (3, 96), (7, 256), (5, 1056), (300, 5120)])
def test_qpack_q4_0_layout(ops, N, K):
    w = synth.q4_0_weights(N, K, seed=N)
    p = _np(ops.qpack_q4_0(_t(w), N, K))
    assert p.size == ops.q4_0_pack_bytes(N, K)
    assert np.array_equal(p, C.pack_q4_0(w))
    assert np.array_equal(C.unpack_q4_0(p, N, K), w)


@pytest.mark.parametrize("N,K", [(1, 256), (7, 512), (3, 768), (300, 5120), (6, 1024)])
def test_qpack_q6_k_layout(ops, N, K):
    w = synth.q6_k_weights(N, K, seed=N)
    p = _np(ops.qpack_q6_k(_t(w), N, K))
    assert p.size == ops.q6_k_pack_bytes(N, K)
    assert np.array_equal(p, C.pack_q6_k(w))
    assert np.array_equal(C.unpack_q6_k(p, N, K), w)


# ---------------------------------------------------------------- block dots bit-exact

@pytest.mark.parametrize("M,K,N", [(1, 256, 5), (6, 512, 33), (17, 1024, 9)])
def test_block_dots_bit_exact(ops, M, K, N):
    x = synth.activations(M, K, seed=1, outlier_frac=0.05)
    xq = oracle.quantize_q8_1(x)
    w4 = synth.q4_0_weights(N, K, seed=2)
    w6 = synth.q6_k_weights(N, K, seed=3)
    xqd = _t(xq.reshape(M, -1))
    got4 = _np(ops.qgemv_block_dots_q4_0(ops.qpack_q4_0(_t(w4), N, K), xqd, M, K, N))
    got6 = _np(ops.qgemv_block_dots_q6_k(ops.qpack_q6_k(_t(w6), N, K), xqd, M, K, N))
    assert np.array_equal(got4, oracle.block_dots_q4_0(w4, xq))
    assert np.array_equal(got6, oracle.block_dots_q6_k(w6, xq))


# ---------------------------------------------------------------- A3 / A4 small shapes

GEMV_SHAPES = [(M, K, N) for M in (1, 2, 3, 5, 6, 8, 9, 12, 16, 17)
               for (K, N) in ((256, 1), (256, 37), (512, 130), (1024, 1001), (5120, 611))]


def _gemv_case(ops, fmt, M, K, N, seed):
    x = synth.activations(M, K, seed=seed, outlier_frac=0.01)
    xq_ref = oracle.quantize_q8_1(x)
    xq = ops.quantize_q8_1(_t(x))
    if fmt == "q4_0":
        w = synth.q4_0_weights(N, K, seed=seed + 1)
        y_ref, S = oracle.qgemv_q4_0(w, xq_ref)
        y = ops.qgemv_q4_0(ops.qpack_q4_0(_t(w), N, K), xq, M, K, N)
    else:
        w = synth.q6_k_weights(N, K, seed=seed + 1)
        y_ref, S = oracle.qgemv_q6_k(w, xq_ref)
        y = ops.qgemv_q6_k(ops.qpack_q6_k(_t(w), N, K), xq, M, K, N)
    return _np(y), y_ref, S


@pytest.mark.parametrize("M,K,N", GEMV_SHAPES + [(M, K, N) for M in (1, 6, 17) for (K, N) in ((32, 5), (96, 37),
                                                                                           (1056, 129))])
def test_qgemv_q4_0_matches_oracle(ops, M, K, N):
    y, y_ref, S = _gemv_case(ops, "q4_0", M, K, N, seed=10 * M + K)
    r = C.check_close(y, y_ref, S)
    assert r["ok"], r


@pytest.mark.parametrize("M,K,N", GEMV_SHAPES)
def test_qgemv_q6_k_matches_oracle(ops, M, K, N):
    y, y_ref, S = _gemv_case(ops, "q6_k", M, K, N, seed=10 * M + K + 7)
    r = C.check_close(y, y_ref, S)
    assert r["ok"], r


@pytest.mark.parametrize("M,K,Na,Nb", [(1, 256, 512, 512), (6, 512, 37, 64), (6, 1024, 4096, 130),
                                       (17, 256, 9, 11), (3, 3072, 1, 5), (6, 5120, 1536, 1539),
                                       (2, 17408, 64, 63)])
def test_qgemv_q4_0_pair_matches_oracle(ops, M, K, Na, Nb):
    # two weights of the same K against one activation in one launch (their
    # row groups are dealt out as one range): each output as its own qgemv
    x = synth.activations(M, K, seed=M + K, outlier_frac=0.01)
    xq_ref = oracle.quantize_q8_1(x)
    xq = ops.quantize_q8_1(_t(x))
    wa = synth.q4_0_weights(Na, K, seed=Na + 3)
    wb = synth.q4_0_weights(Nb, K, seed=Nb + 4)
    ya, yb = ops.qgemv_q4_0_pair(ops.qpack_q4_0(_t(wa), Na, K), ops.qpack_q4_0(_t(wb), Nb, K), xq, M, K, Na, Nb)
    for y, w in ((ya, wa), (yb, wb)):
        y_ref, S = oracle.qgemv_q4_0(w, xq_ref)
        r = C.check_close(_np(y), y_ref, S)
        assert r["ok"], r


# Tensor-core Q4_0 path: shapes it takes (N, N_b multiples of 16, K of 1024),
# over several tiles per CTA, warp ranges that cut tiles, clusters that split
# K (large K or few tiles), and M across the 8-row MMA tiles; each against the
# oracle in the three kernel modes: 1 = the small-M kernel up to M = 16 (the
# general one above), 2 = the general tensor-core kernel, 0 = SIMT only.
TC_SHAPES = [(5, 1024, 16), (6, 1024, 48), (7, 2048, 160), (6, 5120, 2448), (8, 3072, 512), (9, 1024, 4096),
             (12, 5120, 336), (16, 2048, 1040), (17, 5120, 272), (6, 17408, 320), (5, 17408, 64), (5, 9216, 784),
             (7, 1024, 9728)]


@pytest.mark.parametrize("tc", [1, 2, 0])
@pytest.mark.parametrize("M,K,N", TC_SHAPES)
def test_qgemv_q4_0_tensor_core_shapes(ops, M, K, N, tc):
    prev = ops.set_q4_0_tensor_cores(tc)
    try:
        plan = ops.qgemv_q4_0_plan(M, K, N)
        assert plan["tensor_cores"] == bool(tc)
        if tc == 2 or (tc == 1 and M > 16):
            assert plan["kernel"] == "tc"
        y, y_ref, S = _gemv_case(ops, "q4_0", M, K, N, seed=3 * M + K + N)
    finally:
        ops.set_q4_0_tensor_cores(prev)
    r = C.check_close(y, y_ref, S)
    assert r["ok"], r


def test_qgemv_q4_0_tensor_core_plans(ops):
    # the shapes above reach K split over clusters (2 and 4 CTAs) and one CTA
    p = ops.qgemv_q4_0_plan(6, 5120, 17408, 17408)
    assert p["tensor_cores"] and p["cluster"] == 1
    assert ops.qgemv_q4_0_plan(6, 17408, 5120)["cluster"] > 1
    assert ops.qgemv_q4_0_plan(5, 17408, 64)["cluster"] >= 4
    assert not ops.qgemv_q4_0_plan(4, 5120, 17408)["tensor_cores"]  # M < 5: the SIMT kernels
    # ... except on large weights, where the small-M kernel streams faster
    assert ops.qgemv_q4_0_plan(2, 5120, 248320)["kernel"] == "tc_small_m"
    assert ops.qgemv_q4_0_plan(4, 5120, 32768)["kernel"] == "simt"
    assert not ops.qgemv_q4_0_plan(6, 5120, 17400)["tensor_cores"]  # N % 16
    assert not ops.qgemv_q4_0_plan(6, 5056, 17408)["tensor_cores"]  # K % 1024
    for M, K, N in TC_SHAPES:
        p = ops.qgemv_q4_0_plan(M, K, N)
        assert p["tensor_cores"] and p["grid"] % p["cluster"] == 0 and p["stages"] >= 2, (M, K, N, p)


@pytest.mark.parametrize("M,K,Na,Nb", [(5, 1024, 16, 32), (6, 5120, 1536, 1552), (6, 17408, 64, 128),
                                       (17, 2048, 256, 80), (8, 3072, 4096, 16), (12, 5120, 256, 128),
                                       (16, 1024, 48, 32)])
def test_qgemv_q4_0_pair_tensor_cores(ops, M, K, Na, Nb):
    assert ops.qgemv_q4_0_plan(M, K, Na, Nb)["tensor_cores"]
    x = synth.activations(M, K, seed=M + K + 1, outlier_frac=0.01)
    xq_ref = oracle.quantize_q8_1(x)
    xq = ops.quantize_q8_1(_t(x))
    wa = synth.q4_0_weights(Na, K, seed=Na + 13)
    wb = synth.q4_0_weights(Nb, K, seed=Nb + 14)
    ya, yb = ops.qgemv_q4_0_pair(ops.qpack_q4_0(_t(wa), Na, K), ops.qpack_q4_0(_t(wb), Nb, K), xq, M, K, Na, Nb)
    for y, w in ((ya, wa), (yb, wb)):
        y_ref, S = oracle.qgemv_q4_0(w, xq_ref)
        r = C.check_close(_np(y), y_ref, S)
        assert r["ok"], r


def _unit_scale_case(M, K, N, seed):
    """Q4_0 weights with d = 1 and integer activations whose every block holds
    a 127 (so d_a = 1 and q_a = x): every output is an exact integer below
    2^24, so any correct fp32 path must reproduce the oracle bit for bit."""
    w = synth.q4_0_weights(N, K, seed=seed, d_lo=1.0, d_hi=1.0)
    g = np.random.default_rng(seed + 1)
    x = g.integers(-127, 128, size=(M, K)).astype(np.float32)
    x[:, ::32] = np.where(g.integers(0, 2, size=(M, K // 32)) == 1, 127.0, -127.0).astype(np.float32)
    return w, x


@pytest.mark.parametrize("tc", [1, 2, 0])
@pytest.mark.parametrize("M,K,N", [(6, 5120, 64), (5, 1024, 4096), (9, 2048, 48), (17, 1024, 32), (6, 8192, 64),
                                   (12, 5120, 64), (16, 2048, 96)])
def test_qgemv_q4_0_unit_scales_exact(ops, M, K, N, tc):
    # pins the exactness of the block dots on both paths: with unit scales the
    # output is the integer sum of the exact block dots (|y| <= K * 8 * 127 < 2^24)
    w, x = _unit_scale_case(M, K, N, seed=M * 31 + K + N)
    xq_ref = oracle.quantize_q8_1(x)
    assert np.all(xq_ref[:, :, 0:2].view(np.float16) == 1.0)
    y_ref, _ = oracle.qgemv_q4_0(w, xq_ref)
    assert np.all(y_ref == np.round(y_ref))
    prev = ops.set_q4_0_tensor_cores(tc)
    try:
        assert ops.qgemv_q4_0_plan(M, K, N)["tensor_cores"] == (tc > 0 and M >= 5)
        y = _np(ops.qgemv_q4_0(ops.qpack_q4_0(_t(w), N, K), ops.quantize_q8_1(_t(x)), M, K, N))
    finally:
        ops.set_q4_0_tensor_cores(prev)
    assert np.array_equal(y.astype(np.float64), y_ref)


@pytest.mark.parametrize("M", [6, 12])
def test_qgemv_q4_0_pair_unit_scales_exact(ops, M):
    K, Na, Nb = 4096, 48, 80
    wa, x = _unit_scale_case(M, K, Na, seed=5)
    wb, _ = _unit_scale_case(M, K, Nb, seed=6)
    xq_ref = oracle.quantize_q8_1(x)
    ya, yb = ops.qgemv_q4_0_pair(ops.qpack_q4_0(_t(wa), Na, K), ops.qpack_q4_0(_t(wb), Nb, K),
                                 ops.quantize_q8_1(_t(x)), M, K, Na, Nb)
    for y, w in ((ya, wa), (yb, wb)):
        y_ref, _ = oracle.qgemv_q4_0(w, xq_ref)
        assert np.array_equal(_np(y).astype(np.float64), y_ref)


# ---------------------------------------------------------------- Q6_K on the tensor cores
Q6_TC_SHAPES = [(7, 1024, 16), (8, 2048, 160), (9, 5120, 336), (12, 1024, 4096), (16, 2048, 1040),
                (17, 5120, 272), (9, 17408, 320), (12, 17408, 64), (7, 9216, 784), (17, 1024, 48)]


@pytest.mark.parametrize("mode", [2, 0])  # 2: the tensor cores for every shape they take; 0: dp4a
@pytest.mark.parametrize("M,K,N", Q6_TC_SHAPES)
def test_qgemv_q6_k_tensor_core_shapes(ops, M, K, N, mode):
    prev = ops.set_q6_k_tensor_cores(mode)
    try:
        assert ops.qgemv_q6_k_plan(M, K, N)["tensor_cores"] == (mode == 2)
        y, y_ref, S = _gemv_case(ops, "q6_k", M, K, N, seed=5 * M + K + N)
    finally:
        ops.set_q6_k_tensor_cores(prev)
    r = C.check_close(y, y_ref, S)
    assert r["ok"], r


def test_qgemv_q6_k_tensor_core_plans(ops):
    # default mode: only where they measured faster (the dp4a kernel splits K:
    # N < 16 row groups per SM; and M >= 12 or K >= 16384)
    assert ops.qgemv_q6_k_plan(7, 17408, 5120)["tensor_cores"]
    assert ops.qgemv_q6_k_plan(9, 17408, 5120)["cluster"] > 1
    assert ops.qgemv_q6_k_plan(12, 5120, 5120)["tensor_cores"]
    assert not ops.qgemv_q6_k_plan(9, 5120, 5120)["tensor_cores"]
    assert not ops.qgemv_q6_k_plan(12, 5120, 17408)["tensor_cores"]
    assert not ops.qgemv_q6_k_plan(17, 5120, 248320)["tensor_cores"]
    assert not ops.qgemv_q6_k_plan(6, 17408, 5120)["tensor_cores"]  # M < 7: the dp4a kernel
    prev = ops.set_q6_k_tensor_cores(2)
    try:
        assert not ops.qgemv_q6_k_plan(9, 5120, 17400)["tensor_cores"]  # N % 16
        assert not ops.qgemv_q6_k_plan(9, 5376, 17408)["tensor_cores"]  # K % 1024
        assert not ops.qgemv_q6_k_plan(6, 5120, 248320)["tensor_cores"]  # M < 7
        assert ops.qgemv_q6_k_plan(17, 5120, 248320)["tensor_cores"]
        for M, K, N in Q6_TC_SHAPES:
            p = ops.qgemv_q6_k_plan(M, K, N)
            assert p["tensor_cores"] and p["stages"] >= 2 and p["grid"] % p["cluster"] == 0
    finally:
        ops.set_q6_k_tensor_cores(prev)


def _q6_k_unit_case(M, K, N, seed, sc_lo, sc_hi):
    """Q6_K weights with d6 = 1 and subscales in [sc_lo, sc_hi], integer
    activations in [-2, 2] whose every block holds a +-127 (d_a = 1): every
    output is an integer sum of exact block dots."""
    w = synth.q6_k_weights(N, K, seed=seed, d_lo=1.0, d_hi=1.0)
    g = np.random.default_rng(seed + 1)
    w[:, :, 192:208] = g.integers(sc_lo, sc_hi + 1, size=(N, K // 256, 16)).astype(np.int8).view(np.uint8)
    x = g.integers(-2, 3, size=(M, K)).astype(np.float32)
    x[:, ::32] = np.where(g.integers(0, 2, size=(M, K // 32)) == 1, 127.0, -127.0).astype(np.float32)
    return w, x


@pytest.mark.parametrize("mode", [2, 0])
@pytest.mark.parametrize("M,K,N,sc", [(9, 1024, 48, (-3, 3)), (17, 2048, 32, (-3, 3)), (12, 1024, 64, (-128, -127)),
                                      (8, 1024, 32, (126, 127))])
def test_qgemv_q6_k_unit_scales_exact(ops, M, K, N, sc, mode):
    # with d6 = 1 and d_a = 1 every partial sum is an integer below 2^24 (S
    # bounds them), so both paths must reproduce the oracle bit for bit,
    # including the subscale extremes -128 and 127
    w, x = _q6_k_unit_case(M, K, N, M + K + N, *sc)
    xq_ref = oracle.quantize_q8_1(x)
    assert np.all(xq_ref[:, :, 0:2].view(np.float16) == 1.0)
    y_ref, S = oracle.qgemv_q6_k(w, xq_ref)
    assert np.all(S < 2.0 ** 24) and np.all(y_ref == np.round(y_ref))
    prev = ops.set_q6_k_tensor_cores(mode)
    try:
        assert ops.qgemv_q6_k_plan(M, K, N)["tensor_cores"] == (mode == 2)
        y = _np(ops.qgemv_q6_k(ops.qpack_q6_k(_t(w), N, K), ops.quantize_q8_1(_t(x)), M, K, N))
    finally:
        ops.set_q6_k_tensor_cores(prev)
    assert np.array_equal(y.astype(np.float64), y_ref)


def test_qgemv_q6_k_tensor_cores_stride(ops):
    M, K, N, ldy = 9, 2048, 96, 112
    w = synth.q6_k_weights(N, K, seed=25)
    x = synth.activations(M, K, seed=26)
    prev = ops.set_q6_k_tensor_cores(2)
    try:
        assert ops.qgemv_q6_k_plan(M, K, N)["tensor_cores"]
        y = torch.full((M, ldy), 5.0, device=DEV)
        ops.qgemv_q6_k(ops.qpack_q6_k(_t(w), N, K), ops.quantize_q8_1(_t(x)), M, K, N, y=y[:, :N])
    finally:
        ops.set_q6_k_tensor_cores(prev)
    yy = _np(y)
    y_ref, S = oracle.qgemv_q6_k(w, oracle.quantize_q8_1(x))
    assert C.check_close(yy[:, :N], y_ref, S)["ok"]
    assert np.all(yy[:, N:] == 5.0)
    assert ops.qgemv_take_wait_timeouts() == 0


def test_qgemv_q4_0_tensor_cores_stride_and_padding(ops):
    M, K, N, ldy = 6, 2048, 96, 112
    w = synth.q4_0_weights(N, K, seed=15)
    x = synth.activations(M, K, seed=16)
    y = torch.full((M, ldy), 7.0, device=DEV)
    ops.qgemv_q4_0(ops.qpack_q4_0(_t(w), N, K), ops.quantize_q8_1(_t(x)), M, K, N, y=y[:, :N])
    yy = _np(y)
    y_ref, S = oracle.qgemv_q4_0(w, oracle.quantize_q8_1(x))
    assert C.check_close(yy[:, :N], y_ref, S)["ok"]
    assert np.all(yy[:, N:] == 7.0)
    assert ops.qgemv_take_wait_timeouts() == 0


def test_qgemv_q4_0_pair_padding_untouched_and_errors(ops):
    M, K, Na, Nb, ldy = 6, 512, 70, 33, 80
    x = synth.activations(M, K, seed=8)
    xq = ops.quantize_q8_1(_t(x))
    wa = ops.qpack_q4_0(_t(synth.q4_0_weights(Na, K, seed=1)), Na, K)
    wb = ops.qpack_q4_0(_t(synth.q4_0_weights(Nb, K, seed=2)), Nb, K)
    ya = torch.full((M, ldy), 3.0, device=DEV)
    yb = torch.full((M, ldy), 5.0, device=DEV)
    ops.qgemv_q4_0_pair(wa, wb, xq, M, K, Na, Nb, y_a=ya[:, :Na], y_b=yb[:, :Nb])
    assert np.all(_np(ya)[:, Na:] == 3.0) and np.all(_np(yb)[:, Nb:] == 5.0)
    L = ops.LIB
    p = lambda t: ctypes.c_void_p(t.data_ptr())  # noqa: E731
    assert L.qgemv_q4_0_pair(p(wa), None, p(xq), p(ya), p(yb), ldy, M, K, Na, Nb, None) == -1
    assert L.qgemv_q4_0_pair(p(wa), p(wb), p(xq), p(ya), p(yb), 50, M, K, Na, Nb, None) == -1  # ldy < N_a
    assert L.qgemv_q4_0_pair(p(wa), p(wb), p(xq), p(ya), p(yb), ldy, 18, K, Na, Nb, None) == -2


@pytest.mark.parametrize("M,K,N,inplace", [(6, 5120, 2448, False), (6, 5120, 2448, True), (6, 17408, 320, True),
                                           (3, 1024, 1001, False), (8, 2048, 96, True), (17, 17408, 64, False)])
def test_qgemv_q4_0_residual_epilogue(ops, M, K, N, inplace):
    # y = W x + r: the MMVQ within the fp32 gate, then one fp32 addition
    x = synth.activations(M, K, seed=M + K, outlier_frac=0.01)
    w = synth.q4_0_weights(N, K, seed=N + 7)
    r = (synth.activations(M, N, seed=N + 9) * 3.0).astype(np.float32)
    xq_ref = oracle.quantize_q8_1(x)
    y_ref, S = oracle.qgemv_q4_0(w, xq_ref)
    ldr = N + 8
    rt = torch.zeros((M, ldr), device=DEV)
    rt[:, :N] = _t(r)
    wp, xq = ops.qpack_q4_0(_t(w), N, K), ops.quantize_q8_1(_t(x))
    if inplace:
        y = ops.qgemv_q4_0_residual(wp, xq, rt[:, :N], M, K, N, y=rt[:, :N])
    else:
        y = ops.qgemv_q4_0_residual(wp, xq, rt[:, :N], M, K, N)
    yy = _np(y).astype(np.float64)
    want = y_ref + r.astype(np.float64)
    tol = 1e-5 * np.maximum(np.abs(y_ref), S) + 2.0 ** -23 * np.abs(want)
    assert np.all(np.abs(yy - want) <= tol), float(np.max(np.abs(yy - want) - tol))
    if inplace:
        assert np.all(_np(rt)[:, N:] == 0.0)


def test_qgemv_q4_0_residual_errors(ops):
    M, K, N = 6, 1024, 64
    wp = ops.qpack_q4_0(_t(synth.q4_0_weights(N, K, seed=1)), N, K)
    xq = ops.quantize_q8_1(_t(synth.activations(M, K, seed=2)))
    buf = torch.zeros((2 * M, 2 * N), device=DEV)
    L = ops.LIB
    p = lambda t: ctypes.c_void_p(t.data_ptr())  # noqa: E731
    y, r = buf[:M, :N], buf[M:, :N]
    ld = buf.stride(0)
    assert L.qgemv_q4_0_residual(p(wp), p(xq), p(r), ld, p(y), ld, M, K, N, None) == 0
    assert L.qgemv_q4_0_residual(p(wp), p(xq), None, ld, p(y), ld, M, K, N, None) == -1
    assert L.qgemv_q4_0_residual(p(wp), p(xq), p(r), N - 1, p(y), ld, M, K, N, None) == -1  # ldr < N
    assert L.qgemv_q4_0_residual(p(wp), p(xq), p(buf[1:, :N]), ld, p(y), ld, M, K, N, None) == -1  # overlap
    assert L.qgemv_q4_0_residual(p(wp), p(xq), p(y), N, p(y), ld, M, K, N, None) == -1  # alias, ldr != ldy
    torch.cuda.synchronize()


@pytest.mark.parametrize("M,K,ldx,eps", [(1, 32, 32, 1e-6), (6, 5120, 5120, 1e-5), (6, 17408, 17416, 1e-6),
                                         (17, 1024, 1024, 0.0), (3, 96, 100, 1e-3), (17, 5120, 5120, 1e-6)])
def test_rmsnorm_quantize_q8_1_matches_plain_definition(ops, M, K, ldx, eps):
    """Against the oracle's plain definition (fp64 RMSNorm, then the fp32
    quantizer): codes and scales equal except at the stated boundaries, where
    they may be one apart; the counts are printed.  Two calls give the same
    bytes (the kernel's fixed reduction order)."""
    g = np.random.default_rng(M * 7 + K)
    x = (g.standard_normal((M, ldx)) * g.uniform(0.1, 10.0, (M, 1))).astype(np.float32)
    gamma = g.uniform(-2.0, 2.0, K).astype(np.float32)
    ref, xh = oracle.rmsnorm_quantize_q8_1(x, gamma, eps, K=K, with_xh=True)
    got = _np(ops.rmsnorm_quantize_q8_1(_t(x), _t(gamma), eps, K=K)).reshape(M, K // 32, 36)
    again = _np(ops.rmsnorm_quantize_q8_1(_t(x), _t(gamma), eps, K=K)).reshape(M, K // 32, 36)
    r = C.check_q8_1_near(got, ref, xh, K)
    print("rmsnorm_quantize_q8_1", (M, K), r)
    assert r["ok"], r
    assert np.array_equal(got, again)


def test_rmsnorm_quantize_q8_1_errors(ops):
    x, gamma = torch.zeros((2, 64), device=DEV), torch.ones(64, device=DEV)
    xq = torch.empty(ops.q8_1_bytes(2, 64), dtype=torch.uint8, device=DEV)
    L = ops.LIB
    p = lambda t: ctypes.c_void_p(t.data_ptr())  # noqa: E731
    assert L.rmsnorm_quantize_q8_1(p(x), 64, p(gamma), 1e-6, p(xq), 2, 64, None) == 0
    assert L.rmsnorm_quantize_q8_1(p(x), 64, None, 1e-6, p(xq), 2, 64, None) == -1
    assert L.rmsnorm_quantize_q8_1(p(x), 32, p(gamma), 1e-6, p(xq), 2, 64, None) == -1  # ldx < K
    assert L.rmsnorm_quantize_q8_1(p(x), 64, p(gamma), -1.0, p(xq), 2, 64, None) == -1  # eps < 0
    assert L.rmsnorm_quantize_q8_1(p(x), 64, p(gamma), 1e-6, p(xq), 18, 64, None) == -2  # M > 17
    assert L.rmsnorm_quantize_q8_1(p(x), 64, p(gamma), 1e-6, p(xq), 2, 48, None) == -2  # K % 32
    torch.cuda.synchronize()
    # the accepted call: zero rows with eps > 0 normalize to zero, the
    # quantizer's all-zero blocks
    assert np.all(_np(xq) == 0)


# ---------------------------------------------------------------- Q8_0 (tensor cores)

@pytest.mark.parametrize("N,K", [(1, 256), (16, 512), (37, 1024), (130, 5120)])
def test_qpack_q8_0_layout(ops, N, K):
    w = synth.q8_0_weights(N, K, seed=N + K)
    got = _np(ops.qpack_q8_0(_t(w), N, K))
    assert np.array_equal(got, C.pack_q8_0(w))


Q8_0_SHAPES = [(M, K, N) for M in (1, 2, 5, 6, 8, 9, 12, 16, 17) for (K, N) in ((256, 1), (512, 37), (5120, 611))] + [
    (6, 17408, 320), (2, 17408, 64), (6, 5120, 4096), (1, 8192, 16), (17, 17408, 64), (16, 17408, 80)]


@pytest.mark.parametrize("M,K,N", Q8_0_SHAPES)
def test_qgemv_q8_0_matches_oracle(ops, M, K, N):
    x = synth.activations(M, K, seed=M + 5 * K, outlier_frac=0.01)
    w = synth.q8_0_weights(N, K, seed=N + 3 * K)
    y_ref, S = oracle.qgemv_q8_0(w, oracle.quantize_q8_1(x))
    y = _np(ops.qgemv_q8_0(ops.qpack_q8_0(_t(w), N, K), ops.quantize_q8_1(_t(x)), M, K, N))
    r = C.check_close(y, y_ref, S)
    assert r["ok"], r


@pytest.mark.parametrize("M,K,N", [(6, 5120, 64), (1, 1024, 33), (17, 2048, 48), (6, 8192, 16)])
def test_qgemv_q8_0_unit_scales_exact(ops, M, K, N):
    # d_w = 1 and integer activations whose blocks hold +-127 (d_a = 1): the
    # output is the integer sum of the exact block dots (|y| <= K * 127^2 < 2^24
    # for K <= 1024; for larger K the random sums stay far below it)
    w = synth.q8_0_weights(N, K, seed=M + K, d_lo=1.0, d_hi=1.0)
    g = np.random.default_rng(M + N)
    x = g.integers(-127, 128, size=(M, K)).astype(np.float32)
    x[:, ::32] = 127.0
    xq_ref = oracle.quantize_q8_1(x)
    y_ref, _ = oracle.qgemv_q8_0(w, xq_ref)
    assert np.all(np.abs(y_ref) < 2.0 ** 24)
    y = _np(ops.qgemv_q8_0(ops.qpack_q8_0(_t(w), N, K), ops.quantize_q8_1(_t(x)), M, K, N))
    assert np.array_equal(y.astype(np.float64), y_ref)


# ---------------------------------------------------------------- Q4_K (tensor cores)
@pytest.mark.parametrize("N,K", [(16, 256), (37, 512), (5, 1024)])
def test_qpack_q4_k_layout(ops, N, K):
    w = synth.q4_k_weights(N, K, seed=N + K)
    got = _np(ops.qpack_q4_k(_t(w), N, K))
    assert np.array_equal(got, C.pack_q4_k(w))


Q4_K_SHAPES = [(M, K, N) for M in (1, 2, 5, 6, 8, 9, 12, 16, 17) for (K, N) in ((256, 1), (512, 37), (5120, 611))] + [
    (6, 17408, 320), (2, 17408, 64), (6, 5120, 4096), (1, 8192, 16), (17, 17408, 64), (12, 5120, 17408),
    (6, 768, 48), (13, 2304, 80)]


@pytest.mark.parametrize("M,K,N", Q4_K_SHAPES)
def test_qgemv_q4_k_matches_oracle(ops, M, K, N):
    x = synth.activations(M, K, seed=M + 7 * K, outlier_frac=0.01)
    w = synth.q4_k_weights(N, K, seed=N + 5 * K)
    y_ref, S = oracle.qgemv_q4_k(w, oracle.quantize_q8_1(x))
    y = _np(ops.qgemv_q4_k(ops.qpack_q4_k(_t(w), N, K), ops.quantize_q8_1(_t(x)), M, K, N))
    r = C.check_close(y, y_ref, S)
    assert r["ok"], r


@pytest.mark.parametrize("M,K,N", [(6, 2048, 64), (1, 1024, 33), (17, 2048, 48), (9, 4096, 16)])
def test_qgemv_q4_k_unit_scales_exact(ops, M, K, N):
    # d = dmin = 1 with random 6-bit scales and mins, integer activations whose
    # blocks hold +-127 (d_a = 1): both terms are integers and every partial
    # sum stays below 2^24 (S bounds them), so the output must equal the
    # oracle's bit for bit -- a wrong nibble order, scale/min unpacking or
    # accumulator start cannot hide in the fp32 tolerance
    w = synth.q4_k_weights(N, K, seed=M + K, d_lo=1.0, d_hi=1.0, dmin_lo=1.0, dmin_hi=1.0)
    g = np.random.default_rng(M + N)
    x = g.integers(-3, 4, size=(M, K)).astype(np.float32)
    x[:, ::32] = np.where(g.integers(0, 2, size=(M, K // 32)) == 1, 127.0, -127.0).astype(np.float32)
    xq_ref = oracle.quantize_q8_1(x)
    assert np.all(xq_ref[:, :, 0:2].view(np.float16) == 1.0)
    y_ref, S = oracle.qgemv_q4_k(w, xq_ref)
    assert np.all(S < 2.0 ** 24)
    y = _np(ops.qgemv_q4_k(ops.qpack_q4_k(_t(w), N, K), ops.quantize_q8_1(_t(x)), M, K, N))
    assert np.array_equal(y.astype(np.float64), y_ref)


def test_qgemv_q4_k_stride_errors_and_plans(ops):
    M, K, N, ldy = 6, 1024, 40, 48
    w = synth.q4_k_weights(N, K, seed=19)
    x = synth.activations(M, K, seed=20)
    wp, xq = ops.qpack_q4_k(_t(w), N, K), ops.quantize_q8_1(_t(x))
    y = torch.full((M, ldy), 7.0, device=DEV)
    ops.qgemv_q4_k(wp, xq, M, K, N, y=y[:, :N])
    yy = _np(y)
    y_ref, S = oracle.qgemv_q4_k(w, oracle.quantize_q8_1(x))
    assert C.check_close(yy[:, :N], y_ref, S)["ok"]
    assert np.all(yy[:, N:] == 7.0)
    L = ops.LIB
    p = lambda t: ctypes.c_void_p(t.data_ptr())  # noqa: E731
    assert L.qgemv_q4_k(p(wp), p(xq), p(y), ldy, M, 384, N, None) == -2  # K % 256
    assert L.qgemv_q4_k(p(wp), p(xq), p(y), ldy, M, 96, N, None) == -1  # K < 256
    assert L.qgemv_q4_k(p(wp), p(xq), p(y), ldy, 18, K, N, None) == -2  # M > 17
    assert L.qgemv_q4_k(None, p(xq), p(y), ldy, M, K, N, None) == -1
    assert ops.qgemv_take_wait_timeouts() == 0
    for M2, K2, N2 in Q4_K_SHAPES + [(17, 5120, 248320), (6, 5120, 248320)]:
        pl = ops.qgemv_q4_k_plan(M2, K2, N2)
        assert pl["tensor_cores"] and pl["stages"] >= 2 and pl["grid"] % pl["cluster"] == 0
        assert pl["job_blocks"] in (8, 16) and (K2 // 32) % pl["job_blocks"] == 0  # whole jobs only
    assert ops.qgemv_q4_k_plan(6, 5120, 17408)["job_blocks"] == 16  # two superblocks per copy
    assert ops.qgemv_q4_k_plan(6, 768, 48)["job_blocks"] == 8  # 24 blocks: 8-block jobs
    assert ops.qgemv_q4_k_plan(12, 5120, 17408)["job_blocks"] == 8  # M > 8: 8-block jobs


# ---------------------------------------------------------------- Q5_K (tensor cores)
@pytest.mark.parametrize("N,K", [(16, 256), (37, 512), (5, 1024)])
def test_qpack_q5_k_layout(ops, N, K):
    w = synth.q5_k_weights(N, K, seed=N + K + 1)
    got = _np(ops.qpack_q5_k(_t(w), N, K))
    assert np.array_equal(got, C.pack_q5_k(w))


Q5_K_SHAPES = [(M, K, N) for M in (1, 5, 6, 9, 12, 17) for (K, N) in ((256, 1), (512, 37), (5120, 611))] + [
    (6, 17408, 320), (17, 17408, 64), (6, 5120, 4096), (12, 5120, 17408), (6, 768, 48), (13, 2304, 80)]


@pytest.mark.parametrize("M,K,N", Q5_K_SHAPES)
def test_qgemv_q5_k_matches_oracle(ops, M, K, N):
    x = synth.activations(M, K, seed=M + 9 * K, outlier_frac=0.01)
    w = synth.q5_k_weights(N, K, seed=N + 7 * K)
    y_ref, S = oracle.qgemv_q5_k(w, oracle.quantize_q8_1(x))
    y = _np(ops.qgemv_q5_k(ops.qpack_q5_k(_t(w), N, K), ops.quantize_q8_1(_t(x)), M, K, N))
    r = C.check_close(y, y_ref, S)
    assert r["ok"], r


@pytest.mark.parametrize("M,K,N", [(6, 2048, 64), (1, 1024, 33), (17, 2048, 48), (9, 4096, 16)])
def test_qgemv_q5_k_unit_scales_exact(ops, M, K, N):
    # as the Q4_K case: d = dmin = 1, d_a = 1, every partial sum an integer
    # below 2^24, so the fifth bits must land exactly
    w = synth.q5_k_weights(N, K, seed=M + K + 3, d_lo=1.0, d_hi=1.0, dmin_lo=1.0, dmin_hi=1.0)
    g = np.random.default_rng(M + N + 3)
    x = g.integers(-3, 4, size=(M, K)).astype(np.float32)
    x[:, ::32] = np.where(g.integers(0, 2, size=(M, K // 32)) == 1, 127.0, -127.0).astype(np.float32)
    xq_ref = oracle.quantize_q8_1(x)
    assert np.all(xq_ref[:, :, 0:2].view(np.float16) == 1.0)
    y_ref, S = oracle.qgemv_q5_k(w, xq_ref)
    assert np.all(S < 2.0 ** 24)
    y = _np(ops.qgemv_q5_k(ops.qpack_q5_k(_t(w), N, K), ops.quantize_q8_1(_t(x)), M, K, N))
    assert np.array_equal(y.astype(np.float64), y_ref)


def test_qgemv_q5_k_errors_and_plans(ops):
    M, K, N = 6, 1024, 40
    w = synth.q5_k_weights(N, K, seed=21)
    x = synth.activations(M, K, seed=22)
    wp, xq = ops.qpack_q5_k(_t(w), N, K), ops.quantize_q8_1(_t(x))
    y = torch.empty((M, N), device=DEV)
    L = ops.LIB
    p = lambda t: ctypes.c_void_p(t.data_ptr())  # noqa: E731
    assert L.qgemv_q5_k(p(wp), p(xq), p(y), N, M, 384, N, None) == -2  # K % 256
    assert L.qgemv_q5_k(p(wp), p(xq), p(y), N, 18, K, N, None) == -2  # M > 17
    assert L.qgemv_q5_k(None, p(xq), p(y), N, M, K, N, None) == -1
    assert ops.qgemv_take_wait_timeouts() == 0
    for M2, K2, N2 in Q5_K_SHAPES + [(17, 5120, 248320), (6, 5120, 248320)]:
        pl = ops.qgemv_q5_k_plan(M2, K2, N2)
        assert pl["tensor_cores"] and pl["stages"] >= 2 and pl["grid"] % pl["cluster"] == 0
        assert pl["job_blocks"] in (8, 16) and (K2 // 32) % pl["job_blocks"] == 0


def test_qgemv_q8_0_plans(ops):
    # 8-block jobs where two stages of them fit, 4-block jobs (half a pack
    # region) where they do not; very large N launches clusters in waves
    sms = torch.cuda.get_device_properties(DEV).multi_processor_count
    p = ops.qgemv_q8_0_plan(6, 5120, 17408)
    assert p["tensor_cores"] and p["job_blocks"] == 8
    assert ops.qgemv_q8_0_plan(17, 17408, 64)["job_blocks"] == 4
    assert ops.qgemv_q8_0_plan(17, 5120, 611)["job_blocks"] == 4
    p = ops.qgemv_q8_0_plan(17, 5120, 248320)
    assert p["cluster"] > 1 and p["grid"] > sms
    for M, K, N in Q8_0_SHAPES + [(17, 5120, 17408), (17, 17408, 5120), (17, 5120, 40000)]:
        p = ops.qgemv_q8_0_plan(M, K, N)
        assert p["stages"] >= 2 and p["grid"] % p["cluster"] == 0 and p["job_blocks"] in (4, 8)
    with pytest.raises(ops.QgemvError):
        ops.qgemv_q8_0_plan(18, 5120, 64)


@pytest.mark.parametrize("fmt,M,N", [("q8_0", 17, 40000), ("q8_0", 12, 40000), ("q4_0", 17, 40000),
                                     ("q4_0", 12, 40000), ("q6_k", 17, 40000), ("q6_k", 12, 40000),
                                     ("q4_k", 17, 40000), ("q5_k", 17, 40000)])
def test_large_n_wave_plans_sampled_rows(ops, fmt, M, N):
    # more clusters than are resident (the combine area holds a wave's tiles
    # only): outputs checked on a sample of rows, which the oracle computes
    # row by row
    K = 5120
    x = synth.activations(M, K, seed=M + N, outlier_frac=0.01)
    xq = ops.quantize_q8_1(_t(x))
    if fmt == "q8_0":
        w = synth.q8_0_weights(N, K, seed=N + M)
        y = _np(ops.qgemv_q8_0(ops.qpack_q8_0(_t(w), N, K), xq, M, K, N))
        ref = oracle.qgemv_q8_0
    elif fmt == "q5_k":
        w = synth.q5_k_weights(N, K, seed=N + M)
        y = _np(ops.qgemv_q5_k(ops.qpack_q5_k(_t(w), N, K), xq, M, K, N))
        ref = oracle.qgemv_q5_k
    elif fmt == "q4_k":
        w = synth.q4_k_weights(N, K, seed=N + M)
        y = _np(ops.qgemv_q4_k(ops.qpack_q4_k(_t(w), N, K), xq, M, K, N))
        ref = oracle.qgemv_q4_k
    elif fmt == "q6_k":
        w = synth.q6_k_weights(N, K, seed=N + M)
        prev = ops.set_q6_k_tensor_cores(2)  # large N: taken only when forced
        try:
            assert ops.qgemv_q6_k_plan(M, K, N)["tensor_cores"]
            y = _np(ops.qgemv_q6_k(ops.qpack_q6_k(_t(w), N, K), xq, M, K, N))
        finally:
            ops.set_q6_k_tensor_cores(prev)
        ref = oracle.qgemv_q6_k
    else:
        assert ops.qgemv_q4_0_plan(M, K, N)["tensor_cores"]
        w = synth.q4_0_weights(N, K, seed=N + M)
        y = _np(ops.qgemv_q4_0(ops.qpack_q4_0(_t(w), N, K), xq, M, K, N))
        ref = oracle.qgemv_q4_0
    rows = np.unique(np.concatenate([np.arange(0, N, 97), np.arange(N - 40, N)]))
    y_ref, S = ref(w[rows], oracle.quantize_q8_1(x))
    r = C.check_close(y[:, rows], y_ref, S)
    assert r["ok"], r
    assert np.isfinite(y).all()


@pytest.mark.parametrize("wq,xv", [(127, 127), (-127, 127), (127, -127), (-128, 127), ("alt", 127), ("alt", -127)])
def test_qgemv_q8_0_extreme_codes_exact(ops, wq, xv):
    # the largest products and accumulator starts the tensor-core path sees
    # (codes at the int8 extremes, activations all +-127, d_w = d_a = 1): the
    # block dots and their sum over K = 256 (|y| <= 8 * 32 * 128 * 127) are
    # integers below 2^24, so the output must equal the oracle's exactly;
    # "alt" alternates +-127 so that the products cancel against the start
    M, K, N = 9, 256, 32
    w = synth.q8_0_weights(N, K, seed=1, d_lo=1.0, d_hi=1.0)
    codes = np.full(32, wq, dtype=np.int64) if wq != "alt" else np.tile([127, -127], 16)
    w[:, :, 2:] = codes.astype(np.int8).view(np.uint8)
    x = np.full((M, K), float(xv), dtype=np.float32)
    xq_ref = oracle.quantize_q8_1(x)
    y_ref, _ = oracle.qgemv_q8_0(w, xq_ref)
    y = _np(ops.qgemv_q8_0(ops.qpack_q8_0(_t(w), N, K), ops.quantize_q8_1(_t(x)), M, K, N))
    assert np.array_equal(y.astype(np.float64), y_ref)


def test_qgemv_q8_0_stride_padding_and_errors(ops):
    M, K, N, ldy = 6, 1024, 40, 48
    w = synth.q8_0_weights(N, K, seed=9)
    x = synth.activations(M, K, seed=10)
    wp, xq = ops.qpack_q8_0(_t(w), N, K), ops.quantize_q8_1(_t(x))
    y = torch.full((M, ldy), 7.0, device=DEV)
    ops.qgemv_q8_0(wp, xq, M, K, N, y=y[:, :N])
    yy = _np(y)
    y_ref, S = oracle.qgemv_q8_0(w, oracle.quantize_q8_1(x))
    assert C.check_close(yy[:, :N], y_ref, S)["ok"]
    assert np.all(yy[:, N:] == 7.0)
    L = ops.LIB
    p = lambda t: ctypes.c_void_p(t.data_ptr())  # noqa: E731
    assert L.qgemv_q8_0(p(wp), p(xq), p(y), ldy, M, 384, N, None) == -2  # K % 256
    assert L.qgemv_q8_0(p(wp), p(xq), p(y), ldy, M, 96, N, None) == -1  # K < 256
    assert L.qgemv_q8_0(p(wp), p(xq), p(y), ldy, 18, K, N, None) == -2  # M > 17
    assert L.qgemv_q8_0(None, p(xq), p(y), ldy, M, K, N, None) == -1
    assert ops.qgemv_take_wait_timeouts() == 0


def test_qgemv_output_stride_and_untouched_padding(ops):
    M, K, N, ldy = 6, 512, 100, 128
    w = synth.q4_0_weights(N, K, seed=5)
    x = synth.activations(M, K, seed=6)
    y = torch.full((M, ldy), 7.0, device=DEV)
    ops.qgemv_q4_0(ops.qpack_q4_0(_t(w), N, K), ops.quantize_q8_1(_t(x)), M, K, N, y=y[:, :N])
    yy = _np(y)
    y_ref, S = oracle.qgemv_q4_0(w, oracle.quantize_q8_1(x))
    assert C.check_close(yy[:, :N], y_ref, S)["ok"]
    assert np.all(yy[:, N:] == 7.0)


def test_chunked_k_matches_single_chunk(ops):
    # M = 17 at K = 17408 does not fit in shared memory at once: K is staged in
    # chunks.  The lane-to-block map and summation order are the same, so the
    # result must match the oracle under the same gate.
    M, K, N = 17, 17408, 97
    y, y_ref, S = _gemv_case(ops, "q4_0", M, K, N, seed=77)
    assert C.check_close(y, y_ref, S)["ok"]
    y6, y6_ref, S6 = _gemv_case(ops, "q6_k", M, K, N, seed=78)
    assert C.check_close(y6, y6_ref, S6)["ok"]


# ---------------------------------------------------------------- dependent launches

def test_dependent_chain_without_host_sync(ops):
    # Every kernel of the library starts while the previous one drains and
    # waits for it before touching its inputs (programmatic dependent
    # launch).  Chain calls whose inputs are the previous calls' outputs, with
    # no host synchronization in between, then check every link against the
    # oracle applied to the GPU's own previous output.
    M, K, N = 6, 1024, 1024
    w = synth.q4_0_weights(N, K, seed=31)
    wp = ops.qpack_q4_0(_t(w), N, K)
    wv = synth.q6_k_weights(3000, K, seed=32)
    wvp = ops.qpack_q6_k(_t(wv), 3000, K)
    x0 = synth.activations(M, K, seed=33)
    ys = [torch.empty((M, N), device=DEV) for _ in range(4)]
    xqs = [torch.empty(ops.q8_1_bytes(M, K), dtype=torch.uint8, device=DEV) for _ in range(4)]
    ids = [torch.empty(M, dtype=torch.int32, device=DEV) for _ in range(4)]
    cur = _t(x0)
    for i in range(4):
        ops.quantize_q8_1(cur, out=xqs[i])
        ops.qgemv_q4_0(wp, xqs[i], M, K, N, y=ys[i])
        ops.lmhead_q6_k_top1(wvp, ys[i], K, 3000, ids=ids[i])  # reads the GEMV output directly
        cur = ys[i]
    torch.cuda.synchronize()
    prev = x0
    for i in range(4):
        xq_ref = oracle.quantize_q8_1(prev)
        assert np.array_equal(_np(xqs[i]).reshape(xq_ref.shape), xq_ref), i
        y_ref, S = oracle.qgemv_q4_0(w, xq_ref)
        yi = _np(ys[i])
        assert C.check_close(yi, y_ref, S)["ok"], i
        ids_ref, y6, S6 = oracle.lmhead_q6_k_top1(wv, yi)
        assert C.check_top1(_np(ids[i]), y6) == [], i
        prev = yi


# ---------------------------------------------------------------- position independence, determinism

def test_duplicated_and_permuted_rows_bit_identical(ops):
    M, K, N = 6, 1024, 700
    w = synth.q6_k_weights(N, K, seed=9)
    w[256] = w[1]
    w[255] = w[1]
    w[699] = w[0]
    x = synth.activations(M, K, seed=10)
    xq = ops.quantize_q8_1(_t(x))
    y = _np(ops.qgemv_q6_k(ops.qpack_q6_k(_t(w), N, K), xq, M, K, N))
    assert np.array_equal(y[:, 256], y[:, 1]) and np.array_equal(y[:, 255], y[:, 1])
    assert np.array_equal(y[:, 699], y[:, 0])
    perm = np.random.default_rng(3).permutation(N)
    yp = _np(ops.qgemv_q6_k(ops.qpack_q6_k(_t(w[perm]), N, K), xq, M, K, N))
    assert np.array_equal(yp, y[:, perm])
    y2 = _np(ops.qgemv_q6_k(ops.qpack_q6_k(_t(w), N, K), xq, M, K, N))
    assert np.array_equal(y2, y)


# ---------------------------------------------------------------- A6 argmax

def test_argmax_f32_rows_bit_exact(ops):
    g = np.random.default_rng(0)
    M, N = 9, 100003
    y = g.standard_normal((M, N)).astype(np.float32)
    y[1, [5, 70000]] = 50.0
    y[2, :] = np.nan
    y[3, :] = -np.inf
    y[3, 17] = np.nan
    y[4, :] = 0.0
    y[4, :10] = -0.0
    y[5, [3, 99999]] = np.inf
    y[6, :] = -0.0
    y[6, 9] = 0.0
    y[7, 100002] = 1e30
    ids = _np(ops.argmax_f32_rows(_t(y)))
    assert ids.tolist() == oracle.top1(y).tolist()
    # twice in a row: the workspace is left reset
    assert _np(ops.argmax_f32_rows(_t(y))).tolist() == ids.tolist()


# ---------------------------------------------------------------- A5 fused top-1 (small)

@pytest.mark.parametrize("M,K,N", [(1, 256, 1), (5, 512, 1000), (6, 1024, 4099), (17, 256, 300)])
def test_lmhead_small_matches_oracle_and_unfused(ops, M, K, N):
    w = synth.q6_k_weights(N, K, seed=M + N)
    x = synth.activations(M, K, seed=K)
    ids_ref, y_ref, _ = oracle.lmhead_q6_k_top1(w, x)
    wp = ops.qpack_q6_k(_t(w), N, K)
    xd = _t(x)
    ids = _np(ops.lmhead_q6_k_top1(wp, xd, K, N))
    assert C.check_top1(ids, y_ref) == []
    y = ops.qgemv_q6_k(wp, ops.quantize_q8_1(xd), M, K, N)
    assert _np(ops.argmax_f32_rows(y)).tolist() == ids.tolist()


@pytest.mark.parametrize("M,K,N", [(5, 1024, 3001), (6, 2048, 777), (1, 256, 64), (17, 512, 1025)])
def test_lmhead_candmax_matches_oracle_and_logits(ops, M, K, N):
    # greedy id and value of each row plus the logit of a candidate id, within
    # the fp32 gate of the oracle's logits (qgemv_q6_k may split K differently
    # at these small shapes, so it is not compared bit for bit here)
    w = synth.q6_k_weights(N, K, seed=M + N + 1)
    x = synth.activations(M, K, seed=K + 1)
    ids_ref, y_ref, S = oracle.lmhead_q6_k_top1(w, x)
    wp = ops.qpack_q6_k(_t(w), N, K)
    xd = _t(x)
    rng = np.random.default_rng(M * N)
    cand = rng.integers(0, N, size=M).astype(np.int32)
    cand[0] = ids_ref[0]                  # the greedy token itself
    if M > 1:
        cand[1] = N + 5                   # out of range -> NaN
    if M > 2:
        cand[2] = N - 1                   # last row, possibly in a partial group
    ids, top_vals, cand_vals = (_np(t) for t in ops.lmhead_q6_k_candmax(wp, xd, K, N, _t(cand)))
    assert C.check_top1(ids, y_ref) == []

    def close(v, m, n):
        return abs(float(v) - y_ref[m, n]) <= 1e-5 * max(abs(y_ref[m, n]), S[m, n])

    for m in range(M):
        assert close(top_vals[m], m, ids[m]), m
        if 0 <= cand[m] < N:
            assert close(cand_vals[m], m, cand[m]), m
        else:
            assert np.isnan(cand_vals[m]), m
    assert cand_vals[0] == top_vals[0]  # the same sum, bit for bit


# ---------------------------------------------------------------- errors

def test_errors_are_reported_before_launch(ops):
    x = torch.zeros((18, 64), device=DEV)
    with pytest.raises(ops.QgemvError) as e:
        ops.quantize_q8_1(x)
    assert e.value.status == -2
    with pytest.raises(ops.QgemvError) as e:
        ops.quantize_q8_1(torch.zeros((2, 48), device=DEV))
    assert e.value.status == -2
    w = torch.zeros(1000, dtype=torch.uint8, device=DEV)
    xq = torch.zeros(1000, dtype=torch.uint8, device=DEV)
    with pytest.raises(ops.QgemvError) as e:
        ops.qgemv_q6_k(w, xq, 2, 320, 5)
    assert e.value.status == -2
    with pytest.raises(ops.QgemvError) as e:
        ops.lmhead_q6_k_top1(w, torch.zeros((2, 256), device=DEV), 256, 5,
                             ws=torch.zeros(8, dtype=torch.uint8, device=DEV))
    assert e.value.status == -4


def test_no_wait_timeouts(ops):
    # every bounded wait for a weight copy in this process completed
    assert ops.qgemv_take_wait_timeouts() == 0
