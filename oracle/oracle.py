"""ctypes wrapper around the C oracle (``qgemv_oracle.c``) plus an independent
numpy dequantizer used as its brute-force pin.

TEST INFRASTRUCTURE ONLY (see the package docstring).  Parity for the choices
of byte layout, rounding and Q8_1 storage precision is unpinned by the pages:
they name the formats without defining them; the readings are listed in the
C file's header.

Shapes and byte layouts:
  canonical Q4_0 weights: uint8 [N, K/32, 18]   = {fp16 d, qs[16]}
  canonical Q6_K weights: uint8 [N, K/256, 210] = {ql[128], qh[64], sc[16], fp16 d}
  Q8_1 activations:       uint8 [M, K/32, 36]   = {fp16 d, fp16 s, int8 q[32]}
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "qgemv_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle_qgemv.so")
_lock = threading.Lock()
_lib = None

CFLAGS = ["-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared", "-pthread"]


def build(force: bool = False) -> str:
    """Compile the C oracle with the system C compiler; returns the .so path."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.run(["cc", *CFLAGS, "-o", tmp, _SRC, "-lm"], check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            P = ctypes.c_void_p
            I = ctypes.c_int
            L = ctypes.c_int64
            lib.oracle_f32_to_f16.argtypes = [ctypes.c_float]
            lib.oracle_f32_to_f16.restype = ctypes.c_uint16
            lib.oracle_f16_to_f64.argtypes = [ctypes.c_uint16]
            lib.oracle_f16_to_f64.restype = ctypes.c_double
            lib.oracle_quantize_q8_1.argtypes = [P, L, I, I, P]
            lib.oracle_rmsnorm_quantize_q8_1.argtypes = [P, L, P, ctypes.c_float, I, I, P, P]
            for name in ("oracle_dequant_q4_0", "oracle_dequant_q6_k", "oracle_dequant_q8_1", "oracle_dequant_q8_0",
                         "oracle_dequant_q4_k", "oracle_dequant_q5_k"):
                getattr(lib, name).argtypes = [P, I, I, P]
            for name in ("oracle_block_dots_q4_0", "oracle_block_dots_q6_k"):
                getattr(lib, name).argtypes = [P, P, I, I, I, P]
            for name in ("oracle_qgemv_q4_0", "oracle_qgemv_q6_k", "oracle_qgemv_q8_0", "oracle_qgemv_q4_k",
                         "oracle_qgemv_q5_k"):
                getattr(lib, name).argtypes = [P, P, I, I, I, P, P, I]
            lib.oracle_top1_f64.argtypes = [P, L, I, I, P]
            lib.oracle_top1_f32.argtypes = [P, L, I, I, P]
            _lib = lib
    return _lib


def _ptr(a: np.ndarray) -> int:
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data


def default_threads() -> int:
    return max(1, len(os.sched_getaffinity(0)))


# --------------------------------------------------------------------------
# scalar helpers
# --------------------------------------------------------------------------

def f32_to_f16_bits(x) -> np.ndarray:
    """binary16 bits of each fp32 value (IEEE round to nearest even)."""
    lib = _load()
    a = np.asarray(x, dtype=np.float32).ravel()
    out = np.array([lib.oracle_f32_to_f16(float(v)) for v in a], dtype=np.uint16)
    return out.reshape(np.shape(x))


def f16_bits_to_f64(h) -> np.ndarray:
    lib = _load()
    a = np.asarray(h, dtype=np.uint16).ravel()
    out = np.array([lib.oracle_f16_to_f64(int(v)) for v in a], dtype=np.float64)
    return out.reshape(np.shape(h))


# --------------------------------------------------------------------------
# the path's steps
# --------------------------------------------------------------------------

def quantize_q8_1(x: np.ndarray, K: int | None = None) -> np.ndarray:
    """fp32 x [M, >=K] -> Q8_1 uint8 [M, K/32, 36]."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    M, ldx = x.shape
    K = ldx if K is None else K
    assert K % 32 == 0 and K <= ldx
    out = np.zeros((M, K // 32, 36), dtype=np.uint8)
    _load().oracle_quantize_q8_1(_ptr(x), ldx, M, K, _ptr(out))
    return out


def rmsnorm_quantize_q8_1(x: np.ndarray, gamma: np.ndarray, eps: float, K: int | None = None,
                          with_xh: bool = False):
    """Q8_1 of RMSNorm(x) * gamma by the plain definition (fp64 sum of squares
    in increasing k, r = 1 / sqrt(S / K + eps), xh = (x r) gamma in fp64, then
    xh rounded to fp32 and quantized): uint8 [M, K/32, 36]; with_xh: also the
    fp64 xh [M, K]."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    M, ldx = x.shape
    K = ldx if K is None else K
    g = np.ascontiguousarray(gamma, dtype=np.float32)
    assert K % 32 == 0 and K <= ldx and g.shape[0] >= K
    out = np.zeros((M, K // 32, 36), dtype=np.uint8)
    xh = np.zeros((M, K), dtype=np.float64)
    _load().oracle_rmsnorm_quantize_q8_1(_ptr(x), ldx, _ptr(g), ctypes.c_float(eps), M, K, _ptr(out), _ptr(xh))
    return (out, xh) if with_xh else out


def qgemv_q4_0(w: np.ndarray, xq: np.ndarray, nthreads: int | None = None):
    """canonical Q4_0 w [N, K/32, 18], Q8_1 xq [M, K/32, 36] -> (y, S) fp64 [M, N].

    y[m, n] = sum_b d_w * d_a * I_b (I_b exact integer block dots), and
    S[m, n] = sum_b |d_w * d_a * I_b| (the scale of the fp32 rounding error).
    """
    w = np.ascontiguousarray(w, dtype=np.uint8)
    xq = np.ascontiguousarray(xq, dtype=np.uint8)
    N, nb = w.shape[0], w.shape[1]
    M = xq.shape[0]
    assert xq.shape[1] == nb and w.shape[2] == 18
    y = np.zeros((M, N), dtype=np.float64)
    S = np.zeros((M, N), dtype=np.float64)
    _load().oracle_qgemv_q4_0(_ptr(w), _ptr(xq), M, nb * 32, N, _ptr(y), _ptr(S),
                              nthreads or default_threads())
    return y, S


def qgemv_q8_0(w: np.ndarray, xq: np.ndarray, nthreads: int | None = None):
    """canonical Q8_0 w [N, K/32, 34] = {fp16 d, int8 q[32]}, Q8_1 xq [M, K/32, 36]
    -> (y, S) fp64 [M, N]: y = sum_b d_w * d_a * sum_i q_w q_a."""
    w = np.ascontiguousarray(w, dtype=np.uint8)
    xq = np.ascontiguousarray(xq, dtype=np.uint8)
    N, nb, _ = w.shape
    M = xq.shape[0]
    K = nb * 32
    y = np.zeros((M, N), dtype=np.float64)
    S = np.zeros((M, N), dtype=np.float64)
    _load().oracle_qgemv_q8_0(_ptr(w), _ptr(xq), M, K, N, _ptr(y), _ptr(S), nthreads or default_threads())
    return y, S


def dequant_q8_0(w: np.ndarray) -> np.ndarray:
    """[N, K/32, 34] -> fp64 [N, K] (the C dequantizer)."""
    w = np.ascontiguousarray(w, dtype=np.uint8)
    N, nb, _ = w.shape
    out = np.zeros((N, nb * 32), dtype=np.float64)
    _load().oracle_dequant_q8_0(_ptr(w), N, nb * 32, _ptr(out))
    return out


def qgemv_q4_k(w: np.ndarray, xq: np.ndarray, nthreads: int | None = None):
    """canonical Q4_K w [N, K/256, 144] = {fp16 d, fp16 dmin, scales[12], qs[128]},
    Q8_1 xq [M, K/32, 36] -> (y, S) fp64 [M, N]:
    y = sum_b (d sc_b d_a I_b - dmin m_b d_a A_b), I_b = sum q_w q_a, A_b = sum q_a;
    S = sum_b (|first term| + |second term|)."""
    w = np.ascontiguousarray(w, dtype=np.uint8)
    xq = np.ascontiguousarray(xq, dtype=np.uint8)
    N, ns = w.shape[0], w.shape[1]
    M = xq.shape[0]
    assert xq.shape[1] == ns * 8 and w.shape[2] == 144
    y = np.zeros((M, N), dtype=np.float64)
    S = np.zeros((M, N), dtype=np.float64)
    _load().oracle_qgemv_q4_k(_ptr(w), _ptr(xq), M, ns * 256, N, _ptr(y), _ptr(S),
                              nthreads or default_threads())
    return y, S


def dequant_q4_k(w: np.ndarray) -> np.ndarray:
    """[N, K/256, 144] -> fp64 [N, K] (the C dequantizer)."""
    w = np.ascontiguousarray(w, dtype=np.uint8)
    N, ns, _ = w.shape
    out = np.zeros((N, ns * 256), dtype=np.float64)
    _load().oracle_dequant_q4_k(_ptr(w), N, ns * 256, _ptr(out))
    return out


def qgemv_q5_k(w: np.ndarray, xq: np.ndarray, nthreads: int | None = None):
    """canonical Q5_K w [N, K/256, 176] = {fp16 d, fp16 dmin, scales[12], qh[32], qs[128]},
    Q8_1 xq [M, K/32, 36] -> (y, S) fp64 [M, N], the formula of qgemv_q4_k with 5-bit codes."""
    w = np.ascontiguousarray(w, dtype=np.uint8)
    xq = np.ascontiguousarray(xq, dtype=np.uint8)
    N, ns = w.shape[0], w.shape[1]
    M = xq.shape[0]
    assert xq.shape[1] == ns * 8 and w.shape[2] == 176
    y = np.zeros((M, N), dtype=np.float64)
    S = np.zeros((M, N), dtype=np.float64)
    _load().oracle_qgemv_q5_k(_ptr(w), _ptr(xq), M, ns * 256, N, _ptr(y), _ptr(S),
                              nthreads or default_threads())
    return y, S


def dequant_q5_k(w: np.ndarray) -> np.ndarray:
    """[N, K/256, 176] -> fp64 [N, K] (the C dequantizer)."""
    w = np.ascontiguousarray(w, dtype=np.uint8)
    N, ns, _ = w.shape
    out = np.zeros((N, ns * 256), dtype=np.float64)
    _load().oracle_dequant_q5_k(_ptr(w), N, ns * 256, _ptr(out))
    return out


def qgemv_q6_k(w: np.ndarray, xq: np.ndarray, nthreads: int | None = None):
    """canonical Q6_K w [N, K/256, 210], Q8_1 xq [M, K/32, 36] -> (y, S) fp64 [M, N]."""
    w = np.ascontiguousarray(w, dtype=np.uint8)
    xq = np.ascontiguousarray(xq, dtype=np.uint8)
    N, ns = w.shape[0], w.shape[1]
    M = xq.shape[0]
    assert xq.shape[1] == ns * 8 and w.shape[2] == 210
    y = np.zeros((M, N), dtype=np.float64)
    S = np.zeros((M, N), dtype=np.float64)
    _load().oracle_qgemv_q6_k(_ptr(w), _ptr(xq), M, ns * 256, N, _ptr(y), _ptr(S),
                              nthreads or default_threads())
    return y, S


def block_dots_q4_0(w: np.ndarray, xq: np.ndarray) -> np.ndarray:
    """Exact integer block dots I[m, n, b] = sum_i (q_w - 8) * q_a."""
    w = np.ascontiguousarray(w, dtype=np.uint8)
    xq = np.ascontiguousarray(xq, dtype=np.uint8)
    N, nb = w.shape[0], w.shape[1]
    M = xq.shape[0]
    out = np.zeros((M, N, nb), dtype=np.int32)
    _load().oracle_block_dots_q4_0(_ptr(w), _ptr(xq), M, nb * 32, N, _ptr(out))
    return out


def block_dots_q6_k(w: np.ndarray, xq: np.ndarray) -> np.ndarray:
    """Exact integer block dots J[m, n, b] = sum_subblocks sc * sum_i (q - 32) * q_a."""
    w = np.ascontiguousarray(w, dtype=np.uint8)
    xq = np.ascontiguousarray(xq, dtype=np.uint8)
    N, ns = w.shape[0], w.shape[1]
    M = xq.shape[0]
    out = np.zeros((M, N, ns * 8), dtype=np.int32)
    _load().oracle_block_dots_q6_k(_ptr(w), _ptr(xq), M, ns * 256, N, _ptr(out))
    return out


def top1(y: np.ndarray) -> np.ndarray:
    """Lowest index attaining each row's maximum (NaN never wins; all-NaN -> 0)."""
    y = np.ascontiguousarray(y)
    M, N = y.shape
    ids = np.zeros(M, dtype=np.int32)
    if y.dtype == np.float64:
        _load().oracle_top1_f64(_ptr(y), N, M, N, _ptr(ids))
    elif y.dtype == np.float32:
        _load().oracle_top1_f32(_ptr(y), N, M, N, _ptr(ids))
    else:
        raise TypeError(y.dtype)
    return ids


def lmhead_q6_k_top1(w: np.ndarray, x: np.ndarray, nthreads: int | None = None):
    """Fused LM-head top-1, step by step: quantize the rows of x to Q8_1, project
    them through the Q6_K weight, take the lowest-ID argmax of each row.
    Returns (ids, y, S) so that callers can decide near-ties."""
    xq = quantize_q8_1(x)
    y, S = qgemv_q6_k(w, xq, nthreads)
    return top1(y), y, S


def topk(y: np.ndarray, k: int):
    """The k largest values of each row with their indices, larger first,
    exactly equal values by lower index (-0 == +0), NaN never ranked; a row
    with fewer than k non-NaN values fills its last places with -1 / NaN.
    The top-k form of the candidate-max precheck ("Qwen3.6 27B AutoRound
    Handoff", Current next-execution plan: true top ids and values).  Plain
    definition: a stable sort of (-value, index) over the non-NaN entries.
    Returns (ids int32 [M, k], vals float64 [M, k])."""
    y = np.asarray(y, dtype=np.float64)
    M, N = y.shape
    ids = np.full((M, k), -1, dtype=np.int32)
    vals = np.full((M, k), np.nan)
    for m in range(M):
        idx = np.flatnonzero(~np.isnan(y[m]))
        order = idx[np.lexsort((idx, -y[m, idx]))][:k]
        ids[m, : order.size] = order
        vals[m, : order.size] = y[m, order]
    return ids, vals


def lmhead_q6_k_topk(w: np.ndarray, x: np.ndarray, k: int, nthreads: int | None = None):
    """Fused LM-head top-k, step by step: quantize the rows of x to Q8_1,
    project them through the Q6_K weight, rank each row's logits (topk).
    Returns (ids, vals, y, S) so that callers can decide near-ties."""
    xq = quantize_q8_1(x)
    y, S = qgemv_q6_k(w, xq, nthreads)
    ids, vals = topk(y, k)
    return ids, vals, y, S


# --------------------------------------------------------------------------
# independent numpy dequantization (the brute-force pin for the C decoder)
# --------------------------------------------------------------------------

def _f16(bits: np.ndarray) -> np.ndarray:
    return np.ascontiguousarray(bits).view(np.float16).astype(np.float64)


def dequant_q4_0_np(w: np.ndarray) -> np.ndarray:
    """[N, K/32, 18] -> fp64 [N, K]: d * (q - 8), low nibbles first."""
    N, nb, _ = w.shape
    d = _f16(w[:, :, 0:2].copy()).reshape(N, nb, 1)
    qs = w[:, :, 2:18].astype(np.int64)
    q = np.concatenate([qs & 0x0F, qs >> 4], axis=2)
    return (d * (q - 8)).reshape(N, nb * 32)


def dequant_q6_k_np(w: np.ndarray) -> np.ndarray:
    """[N, K/256, 210] -> fp64 [N, K]: d * sc * (q - 32)."""
    N, ns, _ = w.shape
    ql = w[:, :, 0:128].astype(np.int64)
    qh = w[:, :, 128:192].astype(np.int64)
    sc = w[:, :, 192:208].view(np.int8).astype(np.float64)
    d = _f16(w[:, :, 208:210].copy()).reshape(N, ns, 1)
    lo = np.stack([ql & 0x0F, ql >> 4], axis=3).reshape(N, ns, 256)
    hi = np.stack([(qh >> s) & 3 for s in (0, 2, 4, 6)], axis=3).reshape(N, ns, 256)
    q = lo | (hi << 4)
    scale = np.repeat(sc, 16, axis=2)
    return (d * scale * (q - 32)).reshape(N, ns * 256)


def dequant_q8_0_np(w: np.ndarray) -> np.ndarray:
    """[N, K/32, 34] -> fp64 [N, K]: d * q (numpy, independent of the C code)."""
    d = _f16(w[:, :, 0:2].copy().view(np.uint16)[:, :, 0])
    q = w[:, :, 2:34].copy().view(np.int8).astype(np.float64)
    return (d[:, :, None] * q).reshape(w.shape[0], -1)


def dequant_q4_k_np(w: np.ndarray) -> np.ndarray:
    """[N, K/256, 144] -> fp64 [N, K] (numpy, written apart from the C code):
    the eight (scale, min) pairs unpacked with array bit operations, the codes
    as 4 chunks x (32 low nibbles, then the 32 high nibbles)."""
    N, ns, _ = w.shape
    d = _f16(w[:, :, 0:2].copy().view(np.uint16)[:, :, 0])
    dmin = _f16(w[:, :, 2:4].copy().view(np.uint16)[:, :, 0])
    s = w[:, :, 4:16].astype(np.int64)
    sc = np.concatenate([s[:, :, 0:4] & 63, (s[:, :, 8:12] & 15) | ((s[:, :, 0:4] >> 6) << 4)], axis=2)
    mn = np.concatenate([s[:, :, 4:8] & 63, (s[:, :, 8:12] >> 4) | ((s[:, :, 4:8] >> 6) << 4)], axis=2)
    qs = w[:, :, 16:144].astype(np.int64).reshape(N, ns, 4, 32)
    q = np.stack([qs & 15, qs >> 4], axis=3).reshape(N, ns, 8, 32)  # sub-block 2c: low, 2c + 1: high
    v = d[:, :, None, None] * sc[:, :, :, None] * q - dmin[:, :, None, None] * mn[:, :, :, None]
    return v.reshape(N, ns * 256)


def dequant_q5_k_np(w: np.ndarray) -> np.ndarray:
    """[N, K/256, 176] -> fp64 [N, K] (numpy, written apart from the C code):
    the Q4_K decode of scales, mins and nibbles (the codes after the 32 qh
    bytes), plus 16 x bit j of qh[l] for value l of sub-block j."""
    N, ns, _ = w.shape
    base = dequant_q4_k_np(np.concatenate([w[:, :, 0:16], w[:, :, 48:176]], axis=2))
    d = _f16(w[:, :, 0:2].copy().view(np.uint16)[:, :, 0])
    s = w[:, :, 4:16].astype(np.int64)
    sc = np.concatenate([s[:, :, 0:4] & 63, (s[:, :, 8:12] & 15) | ((s[:, :, 0:4] >> 6) << 4)], axis=2)
    qh = w[:, :, 16:48].astype(np.int64)  # [N, ns, 32]
    bits = (qh[:, :, None, :] >> np.arange(8)[None, None, :, None]) & 1  # [N, ns, sub-block j, l]
    return base + (16.0 * d[:, :, None, None] * sc[:, :, :, None] * bits).reshape(N, ns * 256)


def dequant_q8_1_np(xq: np.ndarray) -> np.ndarray:
    """[M, K/32, 36] -> fp64 [M, K]: d * q (the stored fp16 d)."""
    M, nb, _ = xq.shape
    d = _f16(xq[:, :, 0:2].copy()).reshape(M, nb, 1)
    q = xq[:, :, 4:36].view(np.int8).astype(np.float64)
    return (d * q).reshape(M, nb * 32)
