"""The fused LM-head top-k (candidate-max with the true top ids and values,
"Qwen3.6 27B AutoRound Handoff", Current next-execution plan) against the
oracle's ranking of its fp64 logits, through the C ABI.  Gate: check_topk
(ranks within 1e-4 * |max| of the oracle's, values within the fp32 gate, the
order and tie rule exact); planted exact ties and NaN logits decided exactly."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import oracle  # noqa: E402
from block_quantized_gemv_quantize_gb300 import synth  # noqa: E402

from . import _cases as C  # noqa: E402

DEV = "cuda:0"


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


@pytest.mark.parametrize("M,K,N,k", [(1, 256, 7, 7), (2, 256, 9, 8), (3, 512, 100, 1), (4, 768, 4096, 8),
                                     (5, 5120, 20011, 8), (6, 1024, 3001, 5), (9, 2048, 4099, 8),
                                     (17, 1024, 3001, 8),
                                     # the CTAs' lists (17 rows x 152 CTAs x 8 keys) do not fit the
                                     # freed shared memory next to this activation: the last CTA
                                     # picks from global memory
                                     (17, 6144, 2003, 8)])
def test_topk_matches_oracle(ops, M, K, N, k):
    w = synth.q6_k_weights(N, K, seed=M * 7 + N)
    x = synth.activations(M, K, seed=K + M)
    ids_ref, vals_ref, y_ref, S = oracle.lmhead_q6_k_topk(w, x, k)
    wp = ops.qpack_q6_k(_t(w), N, K)
    g = np.random.default_rng(M + N)
    cand = g.integers(0, N, size=M).astype(np.int32)
    cand[0] = ids_ref[0, -1]  # the k-th ranked token
    if M > 1:
        cand[1] = -3          # out of range -> NaN
    ids, vals, cv = ops.lmhead_q6_k_topk(wp, _t(x), K, N, k, cand=_t(cand))
    ids, vals, cv = _np(ids), _np(vals), _np(cv)
    errs = C.check_topk(ids, vals, y_ref, S)
    assert errs == [], errs[:5]
    agree = int((ids == ids_ref).sum())
    print(f"M={M} K={K} N={N} k={k}: {agree}/{ids.size} ranks equal to the oracle's")
    for m in range(M):
        if 0 <= cand[m] < N:
            n = int(cand[m])
            assert abs(float(cv[m]) - y_ref[m, n]) <= 1e-5 * max(abs(y_ref[m, n]), S[m, n]), m
        else:
            assert np.isnan(cv[m]), m
    hit = np.flatnonzero(ids[0] == cand[0])
    if hit.size:
        assert cv[0] == vals[0, hit[0]]  # the same fp32 sum, bit for bit
    # deterministic, and the first rank is the top-1 call's id
    again = _np(ops.lmhead_q6_k_topk(wp, _t(x), K, N, k)[0])
    assert np.array_equal(again, ids)
    assert ids[:, 0].tolist() == _np(ops.lmhead_q6_k_top1(wp, _t(x), K, N)).tolist()


def test_topk_planted_ties_and_nan_rows(ops):
    M, K, N, k = 3, 1024, 3001, 8
    x = synth.activations(M, K, seed=77)
    w = synth.q6_k_weights(N, K, seed=78)
    win = C.winner_q6_k_row(x)
    for r in (2999, 5, 700):
        w[r] = win                        # three exactly equal logits, far above the rest
    for r in (10, 11, 3000):
        w[r, :, 208:210] = [0x00, 0x7E]   # fp16 NaN scale: NaN logits, never ranked
    ids_ref, _, y_ref, S = oracle.lmhead_q6_k_topk(w, x, k)
    assert ids_ref[:, :3].tolist() == [[5, 700, 2999]] * M
    ids, vals, _ = ops.lmhead_q6_k_topk(ops.qpack_q6_k(_t(w), N, K), _t(x), K, N, k)
    ids, vals = _np(ids), _np(vals)
    assert ids[:, :3].tolist() == [[5, 700, 2999]] * M
    assert np.all(vals[:, 0] == vals[:, 1]) and np.all(vals[:, 1] == vals[:, 2])
    assert not np.isin(ids, [10, 11, 3000]).any()
    assert C.check_topk(ids, vals, y_ref, S) == []


def test_topk_fewer_finite_logits_than_k(ops):
    M, K, N, k = 2, 256, 6, 5
    x = synth.activations(M, K, seed=79)
    w = synth.q6_k_weights(N, K, seed=80)
    for r in (1, 3, 4):
        w[r, :, 208:210] = [0x00, 0x7E]
    _, _, y_ref, S = oracle.lmhead_q6_k_topk(w, x, k)
    ids, vals, _ = ops.lmhead_q6_k_topk(ops.qpack_q6_k(_t(w), N, K), _t(x), K, N, k)
    ids, vals = _np(ids), _np(vals)
    assert sorted(ids[:, :3].ravel().tolist()) == sorted([0, 2, 5] * M)
    assert (ids[:, 3:] == -1).all() and np.isnan(vals[:, 3:]).all()
    assert C.check_topk(ids, vals, y_ref, S) == []


def test_topk_rejects_bad_arguments(ops):
    K, N = 256, 64
    wp = torch.zeros(ops.q6_k_pack_bytes(N, K), dtype=torch.uint8, device=DEV)
    x = torch.zeros((2, K), device=DEV)
    for n, k in ((N, 0), (N, 9), (5, 6)):  # k outside 1..8, or above N
        with pytest.raises(ops.QgemvError) as e:
            ops.lmhead_q6_k_topk(wp, x, K, n, k)
        assert e.value.status == -1, (n, k)
    small = torch.zeros(256, dtype=torch.uint8, device=DEV)
    with pytest.raises(ops.QgemvError) as e:
        ops.lmhead_q6_k_topk(wp, x, K, N, 8, ws=small)
    assert e.value.status == -4
    # the top-k runs on the ring kernel only: an activation of 17 rows of
    # 17408 values does not fit next to its rings
    Kb = 17408
    wb = torch.zeros(ops.q6_k_pack_bytes(N, Kb), dtype=torch.uint8, device=DEV)
    with pytest.raises(ops.QgemvError) as e:
        ops.lmhead_q6_k_topk(wb, torch.zeros((17, Kb), device=DEV), Kb, N, 8)
    assert e.value.status == -2
