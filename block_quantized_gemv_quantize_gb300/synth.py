"""Seeded synthetic inputs shaped like the pages' workloads.

This module only draws random numbers and lays them out as canonical block
bytes; it holds none of the method's arithmetic (no quantization, no dot
products, no decoding).  Both the CPU oracle's tests and the CUDA path's tests
and benchmark take their inputs from here.

Recipe (every tensor gets its own child stream of one ``SeedSequence``):
  * Q4_0 weights: fp16 scale d ~ U(0.001, 0.02) drawn in fp32 and rounded
    to the nearest fp16; 4-bit codes uniform on 0..15 (uniform random bytes).
  * Q6_K weights: fp16 superblock scale d ~ U(1e-4, 1e-3); 16 int8 subscales
    ~ U{-64..63}; 6-bit codes uniform on 0..63 (uniform random ql/qh bytes).
  * Activations: fp32 ~ N(0, 1); optionally a fraction of the K channels,
    chosen by a seeded permutation, scaled by a factor in every row (outliers).
"""
from __future__ import annotations

import numpy as np

Q4_0_BYTES = 18
Q6_K_BYTES = 210


def streams(seed: int, n: int) -> list[np.random.Generator]:
    """n independent PCG64 generators spawned from SeedSequence(seed)."""
    return [np.random.Generator(np.random.PCG64(s)) for s in np.random.SeedSequence(seed).spawn(n)]


def _f16_bits(g: np.random.Generator, lo: float, hi: float, shape) -> np.ndarray:
    vals = g.uniform(lo, hi, size=shape).astype(np.float32).astype(np.float16)
    return vals.view(np.uint16)


def _random_bytes(g: np.random.Generator, shape) -> np.ndarray:
    return g.integers(0, 256, size=shape, dtype=np.uint8)


def q4_0_weights(N: int, K: int, seed: int, d_lo: float = 0.001, d_hi: float = 0.02) -> np.ndarray:
    """Canonical Q4_0 bytes uint8 [N, K/32, 18] = {fp16 d (little endian), qs[16]}."""
    assert K % 32 == 0
    nb = K // 32
    g_d, g_q = streams(seed, 2)
    out = np.empty((N, nb, Q4_0_BYTES), dtype=np.uint8)
    out[:, :, 0:2] = _f16_bits(g_d, d_lo, d_hi, (N, nb)).view(np.uint8).reshape(N, nb, 2)
    out[:, :, 2:18] = _random_bytes(g_q, (N, nb, 16))
    return out


def q8_0_weights(N: int, K: int, seed: int, d_lo: float = 0.0005, d_hi: float = 0.005) -> np.ndarray:
    """Canonical Q8_0 bytes uint8 [N, K/32, 34] = {fp16 d, int8 q[32]}, q ~ U{-127..127}."""
    assert K % 32 == 0
    nb = K // 32
    g_d, g_q = streams(seed, 2)
    out = np.empty((N, nb, 34), dtype=np.uint8)
    out[:, :, 0:2] = _f16_bits(g_d, d_lo, d_hi, (N, nb)).view(np.uint8).reshape(N, nb, 2)
    out[:, :, 2:34] = g_q.integers(-127, 128, size=(N, nb, 32), dtype=np.int8).view(np.uint8)
    return out


def q4_k_weights(N: int, K: int, seed: int, d_lo: float = 2e-4, d_hi: float = 2e-3, dmin_lo: float = 1e-4,
                 dmin_hi: float = 1e-3) -> np.ndarray:
    """Canonical Q4_K bytes uint8 [N, K/256, 144] = {fp16 d, fp16 dmin, scales[12], qs[128]};
    the 12 scale bytes and the codes uniform random."""
    assert K % 256 == 0
    ns = K // 256
    g_q, g_d, g_m = streams(seed, 3)
    out = np.empty((N, ns, 144), dtype=np.uint8)
    out[:, :, 0:2] = _f16_bits(g_d, d_lo, d_hi, (N, ns)).view(np.uint8).reshape(N, ns, 2)
    out[:, :, 2:4] = _f16_bits(g_m, dmin_lo, dmin_hi, (N, ns)).view(np.uint8).reshape(N, ns, 2)
    out[:, :, 4:144] = _random_bytes(g_q, (N, ns, 140))
    return out


def q5_k_weights(N: int, K: int, seed: int, d_lo: float = 1e-4, d_hi: float = 1e-3, dmin_lo: float = 1e-4,
                 dmin_hi: float = 1e-3) -> np.ndarray:
    """Canonical Q5_K bytes uint8 [N, K/256, 176] = {fp16 d, fp16 dmin, scales[12], qh[32], qs[128]};
    the scale, high-bit and code bytes uniform random."""
    assert K % 256 == 0
    ns = K // 256
    g_q, g_d, g_m = streams(seed, 3)
    out = np.empty((N, ns, 176), dtype=np.uint8)
    out[:, :, 0:2] = _f16_bits(g_d, d_lo, d_hi, (N, ns)).view(np.uint8).reshape(N, ns, 2)
    out[:, :, 2:4] = _f16_bits(g_m, dmin_lo, dmin_hi, (N, ns)).view(np.uint8).reshape(N, ns, 2)
    out[:, :, 4:176] = _random_bytes(g_q, (N, ns, 172))
    return out


def q6_k_weights(N: int, K: int, seed: int, d_lo: float = 1e-4, d_hi: float = 1e-3) -> np.ndarray:
    """Canonical Q6_K bytes uint8 [N, K/256, 210] = {ql[128], qh[64], int8 sc[16], fp16 d}."""
    assert K % 256 == 0
    ns = K // 256
    g_q, g_s, g_d = streams(seed, 3)
    out = np.empty((N, ns, Q6_K_BYTES), dtype=np.uint8)
    out[:, :, 0:192] = _random_bytes(g_q, (N, ns, 192))
    out[:, :, 192:208] = g_s.integers(-64, 64, size=(N, ns, 16), dtype=np.int8).view(np.uint8)
    out[:, :, 208:210] = _f16_bits(g_d, d_lo, d_hi, (N, ns)).view(np.uint8).reshape(N, ns, 2)
    return out


def activations(M: int, K: int, seed: int, outlier_frac: float = 0.0, outlier_scale: float = 20.0) -> np.ndarray:
    """fp32 [M, K] ~ N(0, 1), with round(outlier_frac * K) channels scaled in every row."""
    g_x, g_p = streams(seed, 2)
    x = g_x.standard_normal(size=(M, K), dtype=np.float32)
    n_out = int(round(outlier_frac * K))
    if n_out:
        ch = g_p.permutation(K)[:n_out]
        x[:, ch] *= np.float32(outlier_scale)
    return x


# Named workloads (shapes and distributions of the pages' configurations).
WORKLOADS = {
    "tiny_q4_0": dict(fmt="q4_0", M=1, K=256, N=512, seed=0),
    "verifier_gate_up": dict(fmt="q4_0", M=6, K=5120, N=17408, seed=1, outlier_frac=0.01),
    "verifier_down": dict(fmt="q4_0", M=6, K=17408, N=5120, seed=2, outlier_frac=0.01),
    "lmhead_q6_k": dict(fmt="q6_k", M=5, K=5120, N=248320, seed=3, rows_from=1, x_rows=6),
}


def tiny_q4_0_inputs():
    """The tiny Q4_0 workload exactly as configured: M = 1, K = 256, N = 512,
    seed 0.  The one seed is split into independent child seeds, the first
    for the weights, the second for the activation."""
    c = WORKLOADS["tiny_q4_0"]
    sw, sx = (int(ch.generate_state(1)[0]) for ch in np.random.SeedSequence(c["seed"]).spawn(2))
    return q4_0_weights(c["N"], c["K"], seed=sw), activations(c["M"], c["K"], seed=sx)
