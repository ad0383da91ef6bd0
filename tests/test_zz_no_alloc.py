"""The allocation-free fused top-1 entry point, called through the C ABI.

lmhead_q6_k_top1_noalloc serves callers that cannot allocate device memory
(their host's pool owns the device, or cudaMalloc could stall a latency
path), so it keeps its reduction scratch in a fixed array inside the library.
It must return exactly the ids of lmhead_q6_k_top1 (the entry point that takes
a caller workspace) on the same inputs, call after call, since every call
reuses the same scratch; and, since it quantizes the activation inside the
MMVQ kernel (no Q8_1 pre-pass), its ids are also checked against the CPU
oracle, on both kernel forms: the ring kernel, and the lock-step kernel that
stages K in chunks when the activation tile does not fit in shared memory.
This file is collected last on purpose, and passes both alone in a fresh
process and after the other tests."""
import ctypes

import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import oracle  # noqa: E402
from block_quantized_gemv_quantize_gb300 import synth  # noqa: E402

from . import _cases as C  # noqa: E402


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from block_quantized_gemv_quantize_gb300 import build

    build.build()
    from block_quantized_gemv_quantize_gb300 import ops

    return ops


def _noalloc(ops, wp, x, K, N, ids):
    fn = ops.LIB.lmhead_q6_k_top1_noalloc
    return fn(ctypes.c_void_p(wp.data_ptr()), ctypes.c_void_p(x.data_ptr()), x.stride(0),
              ctypes.c_void_p(ids.data_ptr()), x.shape[0], K, N,
              ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


# (5, 5120, 20011) and (6, 5120, 20011): the verifier's draft and target row
# counts at the LM-head's K; (17, 17408, 64): an activation tile of 370 KB,
# which the lock-step kernel stages in chunks
@pytest.mark.parametrize("M,K,N,ring", [(5, 5120, 20011, True), (6, 5120, 20011, True), (17, 1024, 3001, True),
                                        (1, 256, 7, True), (17, 17408, 64, False)])
def test_noalloc_matches_workspace_entry_point_and_oracle_twice(lib, M, K, N, ring):
    dev = torch.device("cuda:0")
    assert lib.lmhead_q6_k_top1_plan(M, K, N)["ring"] == ring
    w = synth.q6_k_weights(N, K, seed=N)
    xh = synth.activations(M + 1, K, seed=M)
    x = torch.from_numpy(xh).to(dev)[1:]
    wp = lib.qpack_q6_k(torch.from_numpy(w).to(dev), N, K)
    ref = lib.lmhead_q6_k_top1(wp, x, K, N).cpu()
    _, y_ref, _ = oracle.lmhead_q6_k_top1(w, xh[1:])
    lib.qgemv_take_wait_timeouts()
    for _ in range(2):  # the scratch keeps the previous call's contents
        ids = torch.full((M,), -1, dtype=torch.int32, device=dev)
        assert _noalloc(lib, wp, x, K, N, ids) == 0
        torch.cuda.synchronize()
        assert ids.cpu().tolist() == ref.tolist()
        assert C.check_top1(ids.cpu().numpy(), y_ref) == []
    assert lib.qgemv_take_wait_timeouts() == 0


def test_noalloc_rejects_rows_beyond_the_fixed_scratch(lib):
    dev = torch.device("cuda:0")
    wp = torch.zeros(lib.q6_k_pack_bytes(8, 256), dtype=torch.uint8, device=dev)
    x = torch.zeros((18, 256), device=dev)
    ids = torch.zeros(18, dtype=torch.int32, device=dev)
    assert _noalloc(lib, wp, x, 256, 8, ids) == -2
