"""Test helpers: the documented pack layouts undone on the CPU, the parity
gates, and the adversarial top-1 inputs.  Test code only."""
from __future__ import annotations

import numpy as np

# ---------------------------------------------------------------- pack layouts (inverse, numpy)


CHUNK = 32   # blocks per chunk
GROUP = 4    # rows per group


def _pad16(v: int) -> int:
    return (v + 15) & ~15


def _chunks(nb: int):
    """(first block, blocks) of each 32-block chunk of a row."""
    return [(c, min(CHUNK, nb - c)) for c in range(0, nb, CHUNK)]


def _groups(N: int):
    return [(g, min(GROUP, N - g)) for g in range(0, N, GROUP)]


def pack_q4_0(w: np.ndarray) -> np.ndarray:
    """Canonical Q4_0 [N, K/32, 18] -> the documented layout: groups of 4 rows;
    per (group, 32-block chunk): the 16-byte code blocks [row][block], then the
    fp16 scales [block][row], zero-padded to 16 bytes."""
    N, nb, _ = w.shape
    out = []
    for g0, rows in _groups(N):
        for c0, n in _chunks(nb):
            nib = w[g0:g0 + rows, c0:c0 + n, 2:18].reshape(-1)
            d = w[g0:g0 + rows, c0:c0 + n, 0:2].transpose(1, 0, 2).reshape(-1)
            out += [nib, d, np.zeros(_pad16(d.size) - d.size, dtype=np.uint8)]
    return np.concatenate(out)


def pack_q8_0(w: np.ndarray) -> np.ndarray:
    """Canonical Q8_0 [N, K/32, 34] -> the documented tensor-core pack: per
    16-row tile, per job of 8 blocks, codes [block p][lane 4g + t][16 B] (values
    2t, 2t+1, 2t+8, 2t+9, 16+2t, 17+2t, 24+2t, 25+2t of row g, then of row
    g + 8, each as q + 128) and the fp16 scales [block p][row r]; rows past N
    are zero."""
    N, nb, _ = w.shape
    T = (N + 15) // 16
    wp = np.zeros((T * 16, nb, 34), dtype=np.uint8)
    wp[:N] = w
    q = (wp[:, :, 2:].view(np.int8).astype(np.int16) + 128).astype(np.uint8)  # [rows, nb, 32]
    d = wp[:, :, 0:2]
    out = np.zeros((T, nb // 8, 4352), dtype=np.uint8)
    for tau in range(T):
        for j in range(nb // 8):
            reg = out[tau, j]
            for p in range(8):
                b = 8 * j + p
                for g in range(8):
                    for t in range(4):
                        e = [2 * t, 2 * t + 1, 2 * t + 8, 2 * t + 9, 16 + 2 * t, 17 + 2 * t, 24 + 2 * t, 25 + 2 * t]
                        o = (p * 32 + 4 * g + t) * 16
                        reg[o:o + 8] = q[16 * tau + g, b, e]
                        reg[o + 8:o + 16] = q[16 * tau + g + 8, b, e]
                for r in range(16):
                    reg[4096 + (p * 16 + r) * 2:4096 + (p * 16 + r) * 2 + 2] = d[16 * tau + r, b]
    return out.reshape(-1)


def pack_q4_k(w: np.ndarray) -> np.ndarray:
    """Canonical Q4_K [N, K/256, 144] -> the documented tensor-core pack: per
    16-row tile and superblock a 2368-byte region = codes [block p][lane 4g + t]
    8 B (word t of row g's then of row g + 8's 16 code bytes, byte k = value k
    | value k + 16 << 4 of block p), then [row r][p] {scale, min}, then [row]
    {d, dmin} bits; rows past N are zero."""
    N, ns, _ = w.shape
    T = (N + 15) // 16
    wp = np.zeros((T * 16, ns, 144), dtype=np.uint8)
    wp[:N] = w
    qs = wp[:, :, 16:144].astype(np.int64).reshape(T * 16, ns, 4, 32)
    vals = np.stack([qs & 15, qs >> 4], axis=3).reshape(T * 16, ns, 8, 32)  # [row, sb, block, value]
    code16 = (vals[..., :16] | (vals[..., 16:] << 4)).astype(np.uint8)  # [row, sb, block, 16 bytes]
    sb = wp[:, :, 4:16].astype(np.int64)
    sc = np.concatenate([sb[..., 0:4] & 63, (sb[..., 8:12] & 15) | ((sb[..., 0:4] >> 6) << 4)], axis=2)
    mn = np.concatenate([sb[..., 4:8] & 63, (sb[..., 8:12] >> 4) | ((sb[..., 4:8] >> 6) << 4)], axis=2)
    out = np.zeros((T, ns, 2368), dtype=np.uint8)
    for tau in range(T):
        rows = slice(16 * tau, 16 * tau + 16)
        c = code16[rows]  # [16, ns, 8, 16]
        for p in range(8):
            for g in range(8):
                for t in range(4):
                    o = p * 256 + (4 * g + t) * 8
                    out[tau, :, o:o + 4] = c[g, :, p, 4 * t:4 * t + 4]
                    out[tau, :, o + 4:o + 8] = c[g + 8, :, p, 4 * t:4 * t + 4]
            for r in range(16):
                out[tau, :, 2048 + r * 16 + 2 * p] = sc[16 * tau + r, :, p]
                out[tau, :, 2048 + r * 16 + 2 * p + 1] = mn[16 * tau + r, :, p]
        out[tau, :, 2304:2368] = wp[rows, :, 0:4].transpose(1, 0, 2).reshape(ns, 64)
    return out.reshape(-1)


def pack_q5_k(w: np.ndarray) -> np.ndarray:
    """Canonical Q5_K [N, K/256, 176] -> the documented tensor-core pack: the
    Q4_K pack of the same d, dmin, scales and nibbles, with a [block p][row]
    4-byte word of fifth bits (byte k, bit s = the fifth bit of value k + 4s of
    block p = bit p of qh[k + 4s]) inserted after the 2048 code bytes."""
    N, ns, _ = w.shape
    T = (N + 15) // 16
    q4 = pack_q4_k(np.concatenate([w[:, :, 0:16], w[:, :, 48:176]], axis=2)).reshape(T, ns, 2368)
    wp = np.zeros((T * 16, ns, 176), dtype=np.uint8)
    wp[:N] = w
    out = np.zeros((T, ns, 2880), dtype=np.uint8)
    out[:, :, 0:2048] = q4[:, :, 0:2048]
    out[:, :, 2560:2880] = q4[:, :, 2048:2368]
    qh = wp[:, :, 16:48].astype(np.int64)  # [rows, ns, 32]
    for p in range(8):
        for k in range(4):
            byte = np.zeros((T * 16, ns), dtype=np.int64)
            for s2 in range(8):
                byte |= ((qh[:, :, k + 4 * s2] >> p) & 1) << s2
            for tau in range(T):
                for r in range(16):
                    out[tau, :, 2048 + (p * 16 + r) * 4 + k] = byte[16 * tau + r]
    return out.reshape(-1)


def unpack_q4_0(pack: np.ndarray, N: int, K: int) -> np.ndarray:
    """Inverse of pack_q4_0."""
    nb = K // 32
    out = np.zeros((N, nb, 18), dtype=np.uint8)
    off = 0
    for g0, rows in _groups(N):
        for c0, n in _chunks(nb):
            out[g0:g0 + rows, c0:c0 + n, 2:18] = pack[off:off + 16 * n * rows].reshape(rows, n, 16)
            off += 16 * n * rows
            out[g0:g0 + rows, c0:c0 + n, 0:2] = pack[off:off + 2 * n * rows].reshape(n, rows, 2).transpose(1, 0, 2)
            off += _pad16(2 * n * rows)
    assert off == pack.size
    return out


def _q6_k_codes(w: np.ndarray) -> np.ndarray:
    """Canonical Q6_K [N, K/256, 210] -> codes [N, K] (sequential packing)."""
    N, ns, _ = w.shape
    ql = w[:, :, 0:128].astype(np.int64)
    qh = w[:, :, 128:192].astype(np.int64)
    lo = np.stack([ql & 0x0F, ql >> 4], axis=3).reshape(N, ns, 256)
    hi = np.stack([(qh >> s) & 3 for s in (0, 2, 4, 6)], axis=3).reshape(N, ns, 256)
    return (lo | (hi << 4)).reshape(N, ns * 256)


def pack_q6_k(w: np.ndarray) -> np.ndarray:
    """Canonical Q6_K -> the documented layout: groups of 4 rows; per
    (group, 32-block chunk) each row's tile = P (16 bytes, byte t = q_t |
    high2(q_16+t) << 6), Q (8 bytes, byte u = low4(q_16+u) | low4(q_24+u) <<
    4), sc (the block's two subscales); then the chunk's fp16 scales
    d[rows][blocks / 8], zero padded to 16 bytes."""
    N, ns, _ = w.shape
    nb = ns * 8
    q = _q6_k_codes(w).reshape(N, nb, 32)
    ql = (q[:, :, 0:16] | ((q[:, :, 16:32] >> 4) << 6)).astype(np.uint8)
    qh = ((q[:, :, 16:24] & 0x0F) | ((q[:, :, 24:32] & 0x0F) << 4)).astype(np.uint8)
    sc = w[:, :, 192:208].reshape(N, nb, 2)
    d = w[:, :, 208:210]  # [N, ns, 2]
    out = []
    for g0, rows in _groups(N):
        for c0, n in _chunks(nb):
            for r in range(rows):
                out += [ql[g0 + r, c0:c0 + n].reshape(-1), qh[g0 + r, c0:c0 + n].reshape(-1),
                        sc[g0 + r, c0:c0 + n].reshape(-1)]
            dpart = d[g0:g0 + rows, c0 // 8:(c0 + n) // 8].reshape(-1)
            out += [dpart, np.zeros(_pad16(dpart.size) - dpart.size, dtype=np.uint8)]
    return np.concatenate(out)


def unpack_q6_k(pack: np.ndarray, N: int, K: int) -> np.ndarray:
    """Inverse of pack_q6_k."""
    nb, ns = K // 32, K // 256
    ql = np.zeros((N, nb, 16), dtype=np.int64)
    qh = np.zeros((N, nb, 8), dtype=np.int64)
    sc = np.zeros((N, nb, 2), dtype=np.uint8)
    d = np.zeros((N, ns, 2), dtype=np.uint8)
    off = 0
    for g0, rows in _groups(N):
        for c0, n in _chunks(nb):
            for r in range(rows):
                ql[g0 + r, c0:c0 + n] = pack[off:off + 16 * n].reshape(n, 16)
                qh[g0 + r, c0:c0 + n] = pack[off + 16 * n:off + 24 * n].reshape(n, 8)
                sc[g0 + r, c0:c0 + n] = pack[off + 24 * n:off + 26 * n].reshape(n, 2)
                off += 26 * n
            dn = rows * (n // 8) * 2
            d[g0:g0 + rows, c0 // 8:(c0 + n) // 8] = pack[off:off + dn].reshape(rows, n // 8, 2)
            off += _pad16(dn)
    assert off == pack.size
    q = np.zeros((N, nb, 32), dtype=np.int64)
    q[:, :, 0:16] = ql & 0x3F
    q[:, :, 16:24] = (qh & 0x0F) | ((ql[:, :, 0:8] >> 6) << 4)
    q[:, :, 24:32] = (qh >> 4) | ((ql[:, :, 8:16] >> 6) << 4)
    return q6_k_from_codes(q.reshape(N, K), sc.reshape(N, K // 16).view(np.int8),
                           d.copy().view(np.uint16).reshape(N, ns))


def q6_k_from_codes(codes: np.ndarray, sc: np.ndarray, d16_bits: np.ndarray) -> np.ndarray:
    """Canonical Q6_K bytes from codes [N, K] (0..63), subscales [N, K/16]
    (int8) and fp16 scale bits [N, K/256]."""
    N, K = codes.shape
    ns = K // 256
    q = codes.reshape(N, ns, 256).astype(np.int64)
    out = np.zeros((N, ns, 210), dtype=np.uint8)
    lo = (q & 0x0F).reshape(N, ns, 128, 2)
    out[:, :, 0:128] = (lo[..., 0] | (lo[..., 1] << 4)).astype(np.uint8)
    hi = (q >> 4).reshape(N, ns, 64, 4)
    out[:, :, 128:192] = (hi[..., 0] | (hi[..., 1] << 2) | (hi[..., 2] << 4) | (hi[..., 3] << 6)).astype(np.uint8)
    out[:, :, 192:208] = sc.reshape(N, ns, 16).astype(np.int8).view(np.uint8)
    out[:, :, 208:210] = np.asarray(d16_bits, dtype=np.uint16).reshape(N, ns, 1).view(np.uint8)
    return out


# ---------------------------------------------------------------- gates

REL_TOL = 1e-5   # fp32 outputs: |err| <= 1e-5 * max(|y_oracle|, S)
TOP1_TOL = 1e-4  # top-1: exact where the oracle gap exceeds 1e-4 * |top1|


def check_close(y: np.ndarray, y_ref: np.ndarray, S: np.ndarray, rel: float = REL_TOL) -> dict:
    """Parity gate for fp32 outputs against the fp64 oracle.  The error of an
    fp32 accumulation scales with S = sum_b |d_w d_a I_b|, so the gate is
    |err| <= rel * max(|y_ref|, S); the literal per-output relative error is
    reported too."""
    y = np.asarray(y, dtype=np.float64)
    err = np.abs(y - y_ref)
    bound = rel * np.maximum(np.abs(y_ref), S)
    bad = err > bound
    with np.errstate(divide="ignore", invalid="ignore"):
        lit = np.where(y_ref != 0, err / np.abs(y_ref), np.where(err == 0, 0.0, np.inf))
    return dict(ok=not bad.any(), n_bad=int(bad.sum()), max_err_over_S=float((err / np.maximum(S, 1e-300)).max()),
                max_literal_rel=float(lit.max()), n_literal_over=int((err > rel * np.abs(y_ref)).sum()),
                n=int(y.size))


def check_top1(ids, y_ref: np.ndarray, tol: float = TOP1_TOL) -> list[str]:
    """Rule: the id must equal the oracle's where the oracle's top-2 gap exceeds
    tol * |top1|; otherwise any id whose oracle value is within tol * |top1| of
    the maximum is accepted.  Returns a list of violations."""
    ids = np.asarray(ids)
    errs = []
    for m in range(y_ref.shape[0]):
        row = y_ref[m]
        order = np.argsort(-row, kind="stable")
        top1 = row[order[0]]
        top2 = row[order[1]] if row.size > 1 else -np.inf
        best = int(np.flatnonzero(row == top1)[0])
        if top1 - top2 > tol * abs(top1):
            if int(ids[m]) != best:
                errs.append(f"row {m}: id {int(ids[m])} != oracle {best} (gap {top1 - top2:.3g})")
        else:
            if not (0 <= int(ids[m]) < row.size) or row[int(ids[m])] < top1 - tol * abs(top1):
                errs.append(f"row {m}: id {int(ids[m])} not within tolerance of the max")
    return errs


def check_topk(ids, vals, y_ref: np.ndarray, S: np.ndarray, tol: float = TOP1_TOL, rel: float = REL_TOL) -> list[str]:
    """Rule for a top-k [M][k] against the fp64 oracle logits y_ref [M][N]
    (S: the per-output magnitude sums of the fp32 gate).  Per row: the id at
    rank r has an oracle value within tol * |max| of the oracle's r-th largest
    (so set and order are the oracle's wherever its gaps exceed that), ids are
    distinct, each value is within the fp32 gate of its id's oracle logit,
    values never increase and equal values come by increasing id; past the
    row's non-NaN count, id -1 and NaN.  Returns a list of violations."""
    ids, vals = np.asarray(ids), np.asarray(vals, dtype=np.float64)
    errs = []
    M, k = ids.shape
    for m in range(M):
        row = y_ref[m]
        srt = np.sort(row[~np.isnan(row)])[::-1]
        top = abs(srt[0]) if srt.size else 0.0
        seen = set()
        for r in range(k):
            i, v = int(ids[m, r]), vals[m, r]
            if r >= srt.size:
                if i != -1 or not np.isnan(v):
                    errs.append(f"row {m} rank {r}: ({i}, {v}) past the non-NaN logits")
                continue
            if not 0 <= i < row.size or i in seen:
                errs.append(f"row {m} rank {r}: id {i} out of range or repeated")
                continue
            seen.add(i)
            if abs(row[i] - srt[r]) > tol * top:
                errs.append(f"row {m} rank {r}: id {i} has oracle value {row[i]:.6g}, rank value {srt[r]:.6g}")
            if not abs(v - row[i]) <= rel * max(abs(row[i]), S[m, i]):
                errs.append(f"row {m} rank {r}: value {v:.8g} vs oracle {row[i]:.8g}")
            if r > 0 and 0 <= int(ids[m, r - 1]):
                pv, pi = vals[m, r - 1], int(ids[m, r - 1])
                if v > pv or (v == pv and i < pi):
                    errs.append(f"row {m} rank {r}: ({i}, {v}) out of order after ({pi}, {pv})")
    return errs


# ---------------------------------------------------------------- adversarial top-1


def winner_q6_k_row(x_rows: np.ndarray) -> np.ndarray:
    """A Q6_K row that scores far above random rows for every row of x: the
    sign pattern of v = sum_m x_m / |x_m| at the largest codes, subscales and
    scale the workload's distributions allow (q in {1, 63}, sc = 63, d = 1e-3)."""
    K = x_rows.shape[1]
    v = (x_rows / np.linalg.norm(x_rows, axis=1, keepdims=True)).sum(axis=0)
    codes = np.where(v >= 0, 63, 1).reshape(1, K)
    sc = np.full((1, K // 16), 63, dtype=np.int8)
    d = np.array([[1e-3] * (K // 256)], dtype=np.float32).astype(np.float16).view(np.uint16)
    return q6_k_from_codes(codes, sc, d)[0]


def rmsnorm_q8_1_bounds(K: int):
    """The stated bounds of rmsnorm_quantize_q8_1 against the exact RMSNorm
    (include/qgemv.h): a code may differ by one where the exact x / d lies
    within `delta` of a half-integer, the fp16 scale may be the neighbouring
    one where d lies within a relative `drel` of a rounding midpoint.  Both
    follow from the fp32 sum of squares' relative error, (K / 512 + 9) 2^-24,
    plus the few roundings after it, with a margin of four."""
    e = (K / 512 + 16) * 2.0 ** -24
    return 4 * 127 * e, 4 * e


def check_q8_1_near(got: np.ndarray, ref: np.ndarray, xh: np.ndarray, K: int) -> dict:
    """Compare Q8_1 bytes (uint8 [M, K/32, 36]) from the GPU against the
    oracle's plain-definition bytes, allowing the near-boundary differences of
    rmsnorm_q8_1_bounds; returns counts and 'ok'."""
    delta, drel = rmsnorm_q8_1_bounds(K)
    M, NB = ref.shape[0], ref.shape[1]
    got = got.reshape(M, NB, 36)
    dg = got[:, :, 0:2].copy().view(np.float16)[:, :, 0]
    dr = ref[:, :, 0:2].copy().view(np.float16)[:, :, 0]
    sg = got[:, :, 2:4].copy().view(np.float16)[:, :, 0].astype(np.float64)
    qg = got[:, :, 4:].copy().view(np.int8).astype(np.int64)
    qr = ref[:, :, 4:].copy().view(np.int8).astype(np.int64)
    x32 = xh.astype(np.float32).reshape(M, NB, 32)
    d32 = (np.max(np.abs(x32), axis=2) / np.float32(127.0)).astype(np.float32)
    # codes: exact, or one apart where the exact xh / d is near a half-integer
    with np.errstate(divide="ignore", invalid="ignore"):
        t = np.abs(xh.reshape(M, NB, 32) / d32.astype(np.float64)[:, :, None])
    frac = t - np.floor(t)
    near_q = np.isfinite(t) & (np.abs(frac - 0.5) < delta)
    dq = np.abs(qg - qr)
    codes_ok = (dq == 0) | (near_q & (dq == 1))
    # scales: exact, or the neighbouring fp16 value where d is near a midpoint
    lo = dr.astype(np.float64) - np.spacing(dr).astype(np.float64) / 2
    hi = dr.astype(np.float64) + np.spacing(dr).astype(np.float64) / 2
    d64 = d32.astype(np.float64)
    near_d = (np.abs(d64 - lo) <= drel * d64) | (np.abs(d64 - hi) <= drel * d64)
    dd = np.abs(dg.view(np.int16).astype(np.int64) - dr.view(np.int16).astype(np.int64))
    d_ok = (dd == 0) | (near_d & (dd == 1))
    # s: the fp16 of d * sum(q) for the GPU's own codes, within one fp16 step
    s_ref = (d32.astype(np.float64) * qg.sum(axis=2)).astype(np.float32).astype(np.float16).astype(np.float64)
    s_ok = np.abs(sg - s_ref) <= np.spacing(np.abs(s_ref).astype(np.float16)).astype(np.float64) * 1.001
    return {"ok": bool(codes_ok.all() and d_ok.all() and s_ok.all()), "codes_off_by_one": int((dq == 1).sum()),
            "near_half_integer": int(near_q.sum()), "scales_off_by_one": int((dd == 1).sum()),
            "near_fp16_midpoint": int(near_d.sum()), "bad_codes": int((~codes_ok).sum()),
            "bad_scales": int((~d_ok).sum()), "bad_sums": int((~s_ok).sum()),
            "blocks": int(M * NB), "values": int(M * NB * 32), "delta": delta, "drel": drel}
