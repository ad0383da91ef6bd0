"""Thin ctypes binding of libqgemv.so (argument marshalling only).

Every function here has the name of the C entry point it calls, takes torch
tensors (device memory) plus sizes, passes raw pointers and the current CUDA
stream, and raises ``QgemvError`` on a non-zero status.  All computation runs
in the library's CUDA kernels; there is no other code path.  If the shared
library is missing, importing this module raises: build it first
(``python -m block_quantized_gemv_quantize_gb300.build``).
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

from . import build as _build

_P = ctypes.c_void_p
_I = ctypes.c_int
_L = ctypes.c_int64
_S = ctypes.c_size_t

# name -> (restype, argtypes)
SIGNATURES = {
    "qgemv_status_string": (ctypes.c_char_p, [_I]),
    "q8_1_bytes": (_S, [_I, _I]),
    "q4_0_pack_bytes": (_S, [_I, _I]),
    "q6_k_pack_bytes": (_S, [_I, _I]),
    "lmhead_q6_k_top1_workspace_bytes": (_S, [_I, _I, _I]),
    "argmax_f32_rows_workspace_bytes": (_S, [_I, _I]),
    "quantize_q8_1": (_I, [_P, _L, _P, _I, _I, _P]),
    "qpack_q4_0": (_I, [_P, _P, _I, _I, _P]),
    "qpack_q6_k": (_I, [_P, _P, _I, _I, _P]),
    "qgemv_q4_0": (_I, [_P, _P, _P, _L, _I, _I, _I, _P]),
    "qgemv_q6_k": (_I, [_P, _P, _P, _L, _I, _I, _I, _P]),
    "qgemv_q4_0_pair": (_I, [_P, _P, _P, _P, _P, _L, _I, _I, _I, _I, _P]),
    "lmhead_q6_k_top1": (_I, [_P, _P, _L, _P, _P, _S, _I, _I, _I, _P]),
    "lmhead_q6_k_candmax": (_I, [_P, _P, _L, _P, _P, _P, _P, _P, _S, _I, _I, _I, _P]),
    "lmhead_q6_k_topk_workspace_bytes": (_S, [_I, _I, _I, _I]),
    "lmhead_q6_k_topk": (_I, [_P, _P, _L, _I, _P, _P, _P, _P, _P, _S, _I, _I, _I, _P]),
    "argmax_f32_rows": (_I, [_P, _L, _P, _P, _S, _I, _I, _P]),
    "qgemv_block_dots_q4_0": (_I, [_P, _P, _P, _I, _I, _I, _P]),
    "qgemv_block_dots_q6_k": (_I, [_P, _P, _P, _I, _I, _I, _P]),
    "qgemv_take_wait_timeouts": (_I, [ctypes.POINTER(ctypes.c_uint)]),
    "qgemv_debug_drop_next_copy": (_I, []),
    "qgemv_debug_fail_fused": (_I, [_I]),
    "qgemv_bounds_check_build": (_I, []),
    "qgemv_take_bounds_errors": (_I, [ctypes.POINTER(ctypes.c_uint), ctypes.POINTER(ctypes.c_uint)]),
    "qgemv_debug_plant_bad_store": (_I, []),
    "qgemv_set_q4_0_tensor_cores": (_I, [_I]),
    "qgemv_set_q6_k_tensor_cores": (_I, [_I]),
    "q8_0_pack_bytes": (_S, [_I, _I]),
    "q4_k_pack_bytes": (_S, [_I, _I]),
    "q5_k_pack_bytes": (_S, [_I, _I]),
    "qpack_q5_k": (_I, [_P, _P, _I, _I, _P]),
    "qgemv_q5_k": (_I, [_P, _P, _P, _L, _I, _I, _I, _P]),
    "qgemv_q5_k_plan": (_I, [_I, _I, _I, ctypes.POINTER(ctypes.c_int)]),
    "qpack_q4_k": (_I, [_P, _P, _I, _I, _P]),
    "qgemv_q4_k": (_I, [_P, _P, _P, _L, _I, _I, _I, _P]),
    "qgemv_q4_k_plan": (_I, [_I, _I, _I, ctypes.POINTER(ctypes.c_int)]),
    "qpack_q8_0": (_I, [_P, _P, _I, _I, _P]),
    "qgemv_q8_0": (_I, [_P, _P, _P, _L, _I, _I, _I, _P]),
    "rmsnorm_quantize_q8_1": (_I, [_P, _L, _P, ctypes.c_float, _P, _I, _I, _P]),
    "qgemv_q4_0_residual": (_I, [_P, _P, _P, _L, _P, _L, _I, _I, _I, _P]),
    "qgemv_q4_0_plan": (_I, [_I, _I, _I, _I, ctypes.POINTER(ctypes.c_int)]),
    "qgemv_q8_0_plan": (_I, [_I, _I, _I, ctypes.POINTER(ctypes.c_int)]),
    "qgemv_q6_k_plan": (_I, [_I, _I, _I, ctypes.POINTER(ctypes.c_int)]),
    "lmhead_q6_k_top1_plan": (_I, [_I, _I, _I, ctypes.POINTER(ctypes.c_int)]),
    "lmhead_q6_k_top1_noalloc": (_I, [_P, _P, _L, _P, _I, _I, _I, _P]),
}


class QgemvError(RuntimeError):
    def __init__(self, name: str, status: int):
        super().__init__(f"{name} failed with status {status}: {status_string(status)}")
        self.status = status


BOUNDS_CHECK = os.environ.get("QGEMV_BOUNDS_CHECK", "0") == "1"


def _load() -> ctypes.CDLL:
    path = _build.LIB_DEBUG if BOUNDS_CHECK else _build.LIB
    if not os.path.exists(path):
        raise ImportError(f"{path} is missing: build the CUDA library first "
                          f"(python -m block_quantized_gemv_quantize_gb300.build"
                          f"{' --debug' if BOUNDS_CHECK else ''})")
    lib = ctypes.CDLL(path)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    return lib


LIB = _load()
LIB_PATH = _build.LIB_DEBUG if BOUNDS_CHECK else _build.LIB


def status_string(status: int) -> str:
    return LIB.qgemv_status_string(status).decode()


def _check(name: str, status: int) -> None:
    if status != 0:
        raise QgemvError(name, status)


def _stream(t: torch.Tensor) -> int:
    return torch.cuda.current_stream(t.device).cuda_stream


def _dev(t: torch.Tensor, what: str) -> int:
    if not t.is_cuda:
        raise ValueError(f"{what} must be a CUDA tensor")
    return t.data_ptr()


# ---------------------------------------------------------------- sizes

def q8_1_bytes(M: int, K: int) -> int:
    return LIB.q8_1_bytes(M, K)


def q4_0_pack_bytes(N: int, K: int) -> int:
    return LIB.q4_0_pack_bytes(N, K)


def q6_k_pack_bytes(N: int, K: int) -> int:
    return LIB.q6_k_pack_bytes(N, K)


def lmhead_q6_k_top1_workspace_bytes(M: int, K: int, N: int) -> int:
    return LIB.lmhead_q6_k_top1_workspace_bytes(M, K, N)


def argmax_f32_rows_workspace_bytes(M: int, N: int) -> int:
    return LIB.argmax_f32_rows_workspace_bytes(M, N)


def lmhead_q6_k_topk_workspace_bytes(M: int, K: int, N: int, k: int) -> int:
    return LIB.lmhead_q6_k_topk_workspace_bytes(M, K, N, k)


# ---------------------------------------------------------------- workspaces

_ws_lock = threading.Lock()
_ws_cache: dict[tuple, torch.Tensor] = {}


def workspace(device: torch.device, nbytes: int, key: str = "top1") -> torch.Tensor:
    """A zero-filled device workspace, one per (device, stream, key); the
    kernels leave it zero-filled after every call."""
    device = torch.device(device)
    stream = torch.cuda.current_stream(device).cuda_stream
    k = (device.index, stream, key)
    with _ws_lock:
        ws = _ws_cache.get(k)
        if ws is None or ws.numel() < nbytes:
            ws = torch.zeros(max(nbytes, 256), dtype=torch.uint8, device=device)
            _ws_cache[k] = ws
    return ws


# ---------------------------------------------------------------- the calls

def quantize_q8_1(x: torch.Tensor, K: int | None = None, out: torch.Tensor | None = None) -> torch.Tensor:
    """fp32 x [M, ldx] (row stride = x.stride(0)) -> Q8_1 uint8 [M, K/32*36]."""
    assert x.dtype == torch.float32 and x.dim() == 2 and x.stride(1) == 1
    M = x.shape[0]
    K = x.shape[1] if K is None else K
    if out is None:
        out = torch.empty((M, q8_1_bytes(1, K)), dtype=torch.uint8, device=x.device)
    _check("quantize_q8_1", LIB.quantize_q8_1(_dev(x, "x"), x.stride(0), _dev(out, "xq"), M, K, _stream(x)))
    return out


def rmsnorm_quantize_q8_1(x: torch.Tensor, gamma: torch.Tensor, eps: float, K: int | None = None,
                          out: torch.Tensor | None = None) -> torch.Tensor:
    """fp32 x [M, ldx] -> Q8_1 of RMSNorm(x) * gamma, uint8 [M, K/32*36]."""
    assert x.dtype == torch.float32 and x.dim() == 2 and x.stride(1) == 1
    assert gamma.dtype == torch.float32 and gamma.is_contiguous()
    M = x.shape[0]
    K = x.shape[1] if K is None else K
    if out is None:
        out = torch.empty((M, q8_1_bytes(1, K)), dtype=torch.uint8, device=x.device)
    _check("rmsnorm_quantize_q8_1", LIB.rmsnorm_quantize_q8_1(_dev(x, "x"), x.stride(0), _dev(gamma, "gamma"), eps,
                                                              _dev(out, "xq"), M, K, _stream(x)))
    return out


def qpack_q4_0(w_canon: torch.Tensor, N: int, K: int, out: torch.Tensor | None = None) -> torch.Tensor:
    if out is None:
        out = torch.empty(q4_0_pack_bytes(N, K), dtype=torch.uint8, device=w_canon.device)
    _check("qpack_q4_0", LIB.qpack_q4_0(_dev(w_canon, "w_canon"), _dev(out, "w_pack"), N, K, _stream(w_canon)))
    return out


def qpack_q6_k(w_canon: torch.Tensor, N: int, K: int, out: torch.Tensor | None = None) -> torch.Tensor:
    if out is None:
        out = torch.empty(q6_k_pack_bytes(N, K), dtype=torch.uint8, device=w_canon.device)
    _check("qpack_q6_k", LIB.qpack_q6_k(_dev(w_canon, "w_canon"), _dev(out, "w_pack"), N, K, _stream(w_canon)))
    return out


def _gemv(name: str, w_pack, xq, M, K, N, y):
    if y is None:
        y = torch.empty((M, N), dtype=torch.float32, device=xq.device)
    assert y.dtype == torch.float32 and y.stride(1) == 1
    fn = getattr(LIB, name)
    _check(name, fn(_dev(w_pack, "w_pack"), _dev(xq, "xq"), _dev(y, "y"), y.stride(0), M, K, N, _stream(xq)))
    return y


def qgemv_q4_0(w_pack: torch.Tensor, xq: torch.Tensor, M: int, K: int, N: int,
               y: torch.Tensor | None = None) -> torch.Tensor:
    """y [M, N] fp32 = Q4_0 weight (packed) x Q8_1 activation."""
    return _gemv("qgemv_q4_0", w_pack, xq, M, K, N, y)


def q8_0_pack_bytes(N: int, K: int) -> int:
    return LIB.q8_0_pack_bytes(N, K)


def qpack_q8_0(w_canon: torch.Tensor, N: int, K: int, out: torch.Tensor | None = None) -> torch.Tensor:
    """canonical Q8_0 bytes [N, K/32, 34] -> the tensor-core pack."""
    if out is None:
        out = torch.empty(q8_0_pack_bytes(N, K), dtype=torch.uint8, device=w_canon.device)
    _check("qpack_q8_0", LIB.qpack_q8_0(_dev(w_canon, "w_canon"), _dev(out, "w_pack"), N, K, _stream(w_canon)))
    return out


def qgemv_q8_0(w_pack: torch.Tensor, xq: torch.Tensor, M: int, K: int, N: int,
               y: torch.Tensor | None = None) -> torch.Tensor:
    """y [M, N] fp32 = Q8_0 weight (packed) x Q8_1 activation."""
    return _gemv("qgemv_q8_0", w_pack, xq, M, K, N, y)


def q4_k_pack_bytes(N: int, K: int) -> int:
    return LIB.q4_k_pack_bytes(N, K)


def qpack_q4_k(w_canon: torch.Tensor, N: int, K: int, out: torch.Tensor | None = None) -> torch.Tensor:
    """canonical Q4_K bytes [N, K/256, 144] -> the tensor-core pack."""
    if out is None:
        out = torch.empty(q4_k_pack_bytes(N, K), dtype=torch.uint8, device=w_canon.device)
    _check("qpack_q4_k", LIB.qpack_q4_k(_dev(w_canon, "w_canon"), _dev(out, "w_pack"), N, K, _stream(w_canon)))
    return out


def qgemv_q4_k(w_pack: torch.Tensor, xq: torch.Tensor, M: int, K: int, N: int,
               y: torch.Tensor | None = None) -> torch.Tensor:
    """y [M, N] fp32 = Q4_K weight (packed) x Q8_1 activation."""
    return _gemv("qgemv_q4_k", w_pack, xq, M, K, N, y)


def q5_k_pack_bytes(N: int, K: int) -> int:
    return LIB.q5_k_pack_bytes(N, K)


def qpack_q5_k(w_canon: torch.Tensor, N: int, K: int, out: torch.Tensor | None = None) -> torch.Tensor:
    """canonical Q5_K bytes [N, K/256, 176] -> the tensor-core pack."""
    if out is None:
        out = torch.empty(q5_k_pack_bytes(N, K), dtype=torch.uint8, device=w_canon.device)
    _check("qpack_q5_k", LIB.qpack_q5_k(_dev(w_canon, "w_canon"), _dev(out, "w_pack"), N, K, _stream(w_canon)))
    return out


def qgemv_q5_k(w_pack: torch.Tensor, xq: torch.Tensor, M: int, K: int, N: int,
               y: torch.Tensor | None = None) -> torch.Tensor:
    """y [M, N] fp32 = Q5_K weight (packed) x Q8_1 activation."""
    return _gemv("qgemv_q5_k", w_pack, xq, M, K, N, y)


def qgemv_q4_0_residual(w_pack: torch.Tensor, xq: torch.Tensor, residual: torch.Tensor, M: int, K: int, N: int,
                        y: torch.Tensor | None = None) -> torch.Tensor:
    """y [M, N] fp32 = Q4_0 weight x Q8_1 activation + residual (fp32 [M, >= N],
    row stride residual.stride(0)); y may be the residual itself (in-place add)."""
    assert residual.dtype == torch.float32 and residual.dim() == 2 and residual.stride(1) == 1
    if y is None:
        y = torch.empty((M, N), dtype=torch.float32, device=residual.device)
    _check("qgemv_q4_0_residual",
           LIB.qgemv_q4_0_residual(_dev(w_pack, "w_pack"), _dev(xq, "xq"), _dev(residual, "residual"),
                                   residual.stride(0), _dev(y, "y"), y.stride(0), M, K, N, _stream(y)))
    return y


def qgemv_q4_0_pair(w_a: torch.Tensor, w_b: torch.Tensor, xq: torch.Tensor, M: int, K: int, N_a: int, N_b: int,
                    y_a: torch.Tensor | None = None, y_b: torch.Tensor | None = None):
    """(y_a, y_b) = (W_a x, W_b x) for two packed Q4_0 weights of the same K, in one launch."""
    if y_a is None:
        y_a = torch.empty((M, max(N_a, N_b)), dtype=torch.float32, device=xq.device)[:, :N_a]
    if y_b is None:
        y_b = torch.empty((M, y_a.stride(0)), dtype=torch.float32, device=xq.device)[:, :N_b]
    assert y_a.dtype == torch.float32 and y_b.dtype == torch.float32 and y_a.stride(1) == 1 and y_b.stride(1) == 1
    assert y_a.stride(0) == y_b.stride(0), "y_a and y_b share one row stride"
    _check("qgemv_q4_0_pair", LIB.qgemv_q4_0_pair(_dev(w_a, "w_pack_a"), _dev(w_b, "w_pack_b"), _dev(xq, "xq"),
                                                  _dev(y_a, "y_a"), _dev(y_b, "y_b"), y_a.stride(0), M, K, N_a,
                                                  N_b, _stream(xq)))
    return y_a, y_b


def qgemv_q6_k(w_pack: torch.Tensor, xq: torch.Tensor, M: int, K: int, N: int,
               y: torch.Tensor | None = None) -> torch.Tensor:
    """y [M, N] fp32 = Q6_K weight (packed) x Q8_1 activation."""
    return _gemv("qgemv_q6_k", w_pack, xq, M, K, N, y)


def lmhead_q6_k_top1(w_pack: torch.Tensor, x: torch.Tensor, K: int, N: int, ids: torch.Tensor | None = None,
                     ws: torch.Tensor | None = None) -> torch.Tensor:
    """Greedy token id of each row of fp32 x [M, >=K] (row stride x.stride(0))."""
    assert x.dtype == torch.float32 and x.dim() == 2 and x.stride(1) == 1
    M = x.shape[0]
    if ids is None:
        ids = torch.empty(M, dtype=torch.int32, device=x.device)
    nb = lmhead_q6_k_top1_workspace_bytes(M, K, N)
    if ws is None:
        ws = workspace(x.device, nb)
    _check("lmhead_q6_k_top1", LIB.lmhead_q6_k_top1(_dev(w_pack, "w_pack"), _dev(x, "x"), x.stride(0),
                                                    _dev(ids, "ids"), _dev(ws, "workspace"), ws.numel(),
                                                    M, K, N, _stream(x)))
    return ids


def lmhead_top1_or_unfused(w_pack: torch.Tensor, x: torch.Tensor, K: int, N: int, ids: torch.Tensor | None = None,
                           ws: torch.Tensor | None = None):
    """The greedy ids of the rows of x through the fused LM-head, falling back
    to the ordinary path (quantize_q8_1, qgemv_q6_k with the logits written,
    argmax_f32_rows) when the fused call does not go through ("Q6_K M=6 fused
    DFlash top-1 production record", Exactness and safety contracts: the
    ordinary argmax is skipped only once the fused enqueue has succeeded).
    Returns (ids, "fused" or "ordinary"); a refused call enqueued nothing, so
    the fallback starts from the same inputs."""
    M = x.shape[0]
    if ids is None:
        ids = torch.empty(M, dtype=torch.int32, device=x.device)
    try:
        lmhead_q6_k_top1(w_pack, x, K, N, ids=ids, ws=ws)
        return ids, "fused"
    except QgemvError as e:
        if e.status in (-1, -3, -6):  # bad arguments, misaligned, a pending timeout: the ordinary path fails too
            raise
    y = qgemv_q6_k(w_pack, quantize_q8_1(x, K=K), M, K, N)
    argmax_f32_rows(y, ids=ids)
    return ids, "ordinary"


def lmhead_q6_k_candmax(w_pack: torch.Tensor, x: torch.Tensor, K: int, N: int, cand: torch.Tensor,
                        ws: torch.Tensor | None = None):
    """(ids, top_vals, cand_vals): the greedy id of each row of fp32 x, its
    logit, and the logit of the row's candidate id cand[m] (int32 [M])."""
    assert x.dtype == torch.float32 and x.dim() == 2 and x.stride(1) == 1
    assert cand.dtype == torch.int32 and cand.numel() == x.shape[0]
    M = x.shape[0]
    ids = torch.empty(M, dtype=torch.int32, device=x.device)
    top_vals = torch.empty(M, dtype=torch.float32, device=x.device)
    cand_vals = torch.empty(M, dtype=torch.float32, device=x.device)
    nb = lmhead_q6_k_top1_workspace_bytes(M, K, N)
    if ws is None:
        ws = workspace(x.device, nb)
    _check("lmhead_q6_k_candmax", LIB.lmhead_q6_k_candmax(_dev(w_pack, "w_pack"), _dev(x, "x"), x.stride(0),
                                                          _dev(cand, "cand"), _dev(ids, "ids"),
                                                          _dev(top_vals, "top_vals"), _dev(cand_vals, "cand_vals"),
                                                          _dev(ws, "workspace"), ws.numel(), M, K, N, _stream(x)))
    return ids, top_vals, cand_vals


def lmhead_q6_k_topk(w_pack: torch.Tensor, x: torch.Tensor, K: int, N: int, k: int,
                     cand: torch.Tensor | None = None, ws: torch.Tensor | None = None, ids: torch.Tensor | None = None,
                     vals: torch.Tensor | None = None, cand_vals: torch.Tensor | None = None):
    """(ids [M][k], vals [M][k], cand_vals [M] or None): the k largest logits
    of each row of fp32 x with their ids, larger first, exactly equal values
    by lower id (id -1 / NaN where a row has fewer than k non-NaN logits),
    and, given cand (int32 [M]), each row's candidate logit."""
    assert x.dtype == torch.float32 and x.dim() == 2 and x.stride(1) == 1
    M = x.shape[0]
    if ids is None:
        ids = torch.empty((M, k), dtype=torch.int32, device=x.device)
    if vals is None:
        vals = torch.empty((M, k), dtype=torch.float32, device=x.device)
    assert ids.shape == (M, k) and ids.is_contiguous() and vals.shape == (M, k) and vals.is_contiguous()
    if cand is None:
        cand_vals = None
    else:
        assert cand.dtype == torch.int32 and cand.numel() == M
        if cand_vals is None:
            cand_vals = torch.empty(M, dtype=torch.float32, device=x.device)
    nb = lmhead_q6_k_topk_workspace_bytes(M, K, N, k)
    if ws is None:
        ws = workspace(x.device, nb)
    _check("lmhead_q6_k_topk", LIB.lmhead_q6_k_topk(_dev(w_pack, "w_pack"), _dev(x, "x"), x.stride(0), k,
                                                    None if cand is None else _dev(cand, "cand"), _dev(ids, "ids"),
                                                    _dev(vals, "vals"),
                                                    None if cand_vals is None else _dev(cand_vals, "cand_vals"),
                                                    _dev(ws, "workspace"), ws.numel(), M, K, N, _stream(x)))
    return ids, vals, cand_vals


def lmhead_q6_k_top1_noalloc(w_pack: torch.Tensor, x: torch.Tensor, K: int, N: int,
                             ids: torch.Tensor | None = None) -> torch.Tensor:
    """As lmhead_q6_k_top1, with the library's fixed device scratch instead of
    a caller workspace (for callers that cannot allocate; calls on one device
    must not overlap)."""
    assert x.dtype == torch.float32 and x.dim() == 2 and x.stride(1) == 1
    M = x.shape[0]
    if ids is None:
        ids = torch.empty(M, dtype=torch.int32, device=x.device)
    _check("lmhead_q6_k_top1_noalloc", LIB.lmhead_q6_k_top1_noalloc(_dev(w_pack, "w_pack"), _dev(x, "x"),
                                                                    x.stride(0), _dev(ids, "ids"), M, K, N,
                                                                    _stream(x)))
    return ids


def argmax_f32_rows(y: torch.Tensor, N: int | None = None, ids: torch.Tensor | None = None,
                    ws: torch.Tensor | None = None) -> torch.Tensor:
    assert y.dtype == torch.float32 and y.dim() == 2 and y.stride(1) == 1
    M = y.shape[0]
    N = y.shape[1] if N is None else N
    if ids is None:
        ids = torch.empty(M, dtype=torch.int32, device=y.device)
    if ws is None:
        ws = workspace(y.device, argmax_f32_rows_workspace_bytes(M, N), key="argmax")
    _check("argmax_f32_rows", LIB.argmax_f32_rows(_dev(y, "y"), y.stride(0), _dev(ids, "ids"),
                                                  _dev(ws, "workspace"), ws.numel(), M, N, _stream(y)))
    return ids


def qgemv_block_dots_q4_0(w_pack: torch.Tensor, xq: torch.Tensor, M: int, K: int, N: int) -> torch.Tensor:
    out = torch.empty((M, N, K // 32), dtype=torch.int32, device=xq.device)
    _check("qgemv_block_dots_q4_0", LIB.qgemv_block_dots_q4_0(_dev(w_pack, "w_pack"), _dev(xq, "xq"),
                                                              out.data_ptr(), M, K, N, _stream(xq)))
    return out


def qgemv_block_dots_q6_k(w_pack: torch.Tensor, xq: torch.Tensor, M: int, K: int, N: int) -> torch.Tensor:
    out = torch.empty((M, N, K // 32), dtype=torch.int32, device=xq.device)
    _check("qgemv_block_dots_q6_k", LIB.qgemv_block_dots_q6_k(_dev(w_pack, "w_pack"), _dev(xq, "xq"),
                                                              out.data_ptr(), M, K, N, _stream(xq)))
    return out


def set_q4_0_tensor_cores(mode) -> int:
    """Kernel family of qgemv_q4_0 / qgemv_q4_0_pair: 1 or True (default) the
    tensor cores where the shape allows (the small-M kernel for M <= 8), 2 the
    general tensor-core kernel for every such M, 0 or False the SIMT kernels
    only; returns the previous setting."""
    return int(LIB.qgemv_set_q4_0_tensor_cores(int(mode)))


def set_q6_k_tensor_cores(mode: int) -> int:
    """qgemv_q6_k's kernel family: 1 = the tensor cores where they measured
    faster (default), 2 = wherever the shape allows, 0 = never (dp4a);
    returns the previous mode."""
    return int(LIB.qgemv_set_q6_k_tensor_cores(int(mode)))


def lmhead_q6_k_top1_plan(M: int, K: int, N: int) -> dict:
    """The kernel the fused LM-head calls would launch for this shape."""
    info = (ctypes.c_int * 4)()
    _check("lmhead_q6_k_top1_plan", LIB.lmhead_q6_k_top1_plan(M, K, N, info))
    return {"ring": bool(info[0]), "grid": info[1], "warps": info[2], "stages": info[3]}


def qgemv_q4_0_plan(M: int, K: int, N: int, N_b: int = 0) -> dict:
    """The kernel qgemv_q4_0 (N_b = 0) or the pair call would launch."""
    info = (ctypes.c_int * 4)()
    _check("qgemv_q4_0_plan", LIB.qgemv_q4_0_plan(M, K, N, N_b, info))
    return {"tensor_cores": bool(info[0]), "kernel": {0: "simt", 1: "tc", 2: "tc_small_m"}[info[0]],
            "cluster": info[1], "grid": info[2], "stages": info[3]}


def qgemv_q6_k_plan(M: int, K: int, N: int) -> dict:
    """The kernel qgemv_q6_k would launch for this shape."""
    info = (ctypes.c_int * 4)()
    _check("qgemv_q6_k_plan", LIB.qgemv_q6_k_plan(M, K, N, info))
    return {"tensor_cores": bool(info[0]), "cluster": info[1], "grid": info[2], "stages": info[3]}


def qgemv_q8_0_plan(M: int, K: int, N: int) -> dict:
    """The launch qgemv_q8_0 would make for this shape."""
    info = (ctypes.c_int * 5)()
    _check("qgemv_q8_0_plan", LIB.qgemv_q8_0_plan(M, K, N, info))
    return {"tensor_cores": bool(info[0]), "cluster": info[1], "grid": info[2], "stages": info[3],
            "job_blocks": info[4]}


def qgemv_q4_k_plan(M: int, K: int, N: int) -> dict:
    """The launch qgemv_q4_k would make for this shape."""
    info = (ctypes.c_int * 5)()
    _check("qgemv_q4_k_plan", LIB.qgemv_q4_k_plan(M, K, N, info))
    return {"tensor_cores": bool(info[0]), "cluster": info[1], "grid": info[2], "stages": info[3],
            "job_blocks": info[4]}


def qgemv_q5_k_plan(M: int, K: int, N: int) -> dict:
    """The launch qgemv_q5_k would make for this shape."""
    info = (ctypes.c_int * 5)()
    _check("qgemv_q5_k_plan", LIB.qgemv_q5_k_plan(M, K, N, info))
    return {"tensor_cores": bool(info[0]), "cluster": info[1], "grid": info[2], "stages": info[3],
            "job_blocks": info[4]}


def qgemv_take_wait_timeouts() -> int:
    """Warps that gave up waiting for their data since the last call; reads and
    clears the count (synchronizes the device first), after which calls are
    accepted again."""
    torch.cuda.synchronize()
    c = ctypes.c_uint(0)
    _check("qgemv_take_wait_timeouts", LIB.qgemv_take_wait_timeouts(ctypes.byref(c)))
    return c.value


def qgemv_debug_fail_fused(count: int) -> int:
    """Test only: the next `count` fused LM-head calls fail before enqueueing."""
    return int(LIB.qgemv_debug_fail_fused(int(count)))


def qgemv_bounds_check_build() -> bool:
    """Whether the loaded library is the bounds-checking build."""
    return bool(LIB.qgemv_bounds_check_build())


def qgemv_take_bounds_errors() -> tuple[int, int]:
    """(failed checks, site number of the first) since the last call, after a
    device synchronize; (0, 0) always in the release build."""
    count, site = ctypes.c_uint(0), ctypes.c_uint(0)
    _check("qgemv_take_bounds_errors", LIB.qgemv_take_bounds_errors(ctypes.byref(count), ctypes.byref(site)))
    return count.value, site.value


def qgemv_debug_plant_bad_store() -> int:
    """Test hook of the bounds-checking build: the next ring-kernel MMVQ
    launch moves its first stores out of their extent, which its checks skip
    and record.  Returns the previous request (QGEMV_UNSUPPORTED_SHAPE in the
    release build, where it does nothing)."""
    return LIB.qgemv_debug_plant_bad_store()


def qgemv_debug_drop_next_copy() -> int:
    """Test only: the next small-M tensor-core Q4_0 launch skips one copy, so
    one warp's bounded wait runs out (see include/qgemv.h)."""
    return int(LIB.qgemv_debug_drop_next_copy())
