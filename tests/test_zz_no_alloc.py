"""The allocation-free fused top-1 entry point, called through the C ABI.

lmhead_q6_k_top1_noalloc serves callers that cannot allocate device memory
(their host's pool owns the device, or cudaMalloc could stall a latency
path), so it keeps its reduction scratch in a fixed array inside the library.
It must return exactly the ids of lmhead_q6_k_top1 (the entry point that takes
a caller workspace) on the same inputs, call after call, since every call
reuses the same scratch.  This file is collected last on purpose, and passes
both alone in a fresh process and after the other tests."""
import ctypes

import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

from block_quantized_gemv_quantize_gb300 import synth  # noqa: E402


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


@pytest.mark.parametrize("M,K,N", [(5, 5120, 20011), (17, 1024, 3001), (1, 256, 7)])
def test_noalloc_matches_workspace_entry_point_twice(lib, M, K, N):
    dev = torch.device("cuda:0")
    w = synth.q6_k_weights(N, K, seed=N)
    x = torch.from_numpy(synth.activations(M + 1, K, seed=M)).to(dev)[1:]
    wp = lib.qpack_q6_k(torch.from_numpy(w).to(dev), N, K)
    ref = lib.lmhead_q6_k_top1(wp, x, K, N).cpu()
    for _ in range(2):  # the scratch keeps the previous call's contents
        ids = torch.full((M,), -1, dtype=torch.int32, device=dev)
        assert _noalloc(lib, wp, x, K, N, ids) == 0
        torch.cuda.synchronize()
        assert ids.cpu().tolist() == ref.tolist()


def test_noalloc_rejects_rows_beyond_the_fixed_scratch(lib):
    dev = torch.device("cuda:0")
    wp = torch.zeros(lib.q6_k_pack_bytes(8, 256), dtype=torch.uint8, device=dev)
    x = torch.zeros((18, 256), device=dev)
    ids = torch.zeros(18, dtype=torch.int32, device=dev)
    assert _noalloc(lib, wp, x, 256, 8, ids) == -2
