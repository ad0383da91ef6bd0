"""The fail-closed fused LM-head ("Q6_K M=6 fused DFlash top-1 production
record", Exactness and safety contracts): when the fused call does not go
through, the binding runs the ordinary path (quantize, qgemv_q6_k with the
logits written, argmax_f32_rows) on the same inputs, and the refused call
enqueued nothing.  The failure is made on the host, by the test-only hook."""
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


@pytest.mark.parametrize("M,K,N", [(5, 5120, 4099), (6, 1024, 777)])
def test_refused_fused_call_falls_back_to_the_ordinary_path(ops, M, K, N):
    w = synth.q6_k_weights(N, K, seed=N + 7)
    x = synth.activations(M, K, seed=K + 7)
    _, y_ref, _ = oracle.lmhead_q6_k_top1(w, x)
    wp = ops.qpack_q6_k(torch.from_numpy(w).to(DEV), N, K)
    xd = torch.from_numpy(x).to(DEV)
    ws = torch.zeros(ops.lmhead_q6_k_top1_workspace_bytes(M, K, N), dtype=torch.uint8, device=DEV)

    assert ops.qgemv_debug_fail_fused(1) == 0
    ids, path = ops.lmhead_top1_or_unfused(wp, xd, K, N, ws=ws)
    torch.cuda.synchronize()
    assert path == "ordinary"
    assert ops.qgemv_debug_fail_fused(0) == 0
    # the refused fused call enqueued nothing: its workspace (the Q8_1 copy
    # and the top-1 keys it would have written) is still all zero
    assert int(ws.count_nonzero()) == 0
    assert C.check_top1(ids.cpu().numpy(), y_ref) == []

    ids2, path2 = ops.lmhead_top1_or_unfused(wp, xd, K, N, ws=ws)
    torch.cuda.synchronize()
    assert path2 == "fused"
    assert ids2.cpu().tolist() == ids.cpu().tolist()
    assert np.array_equal(ws[:256].cpu().numpy(), np.zeros(256, np.uint8))  # left zeroed after the call
