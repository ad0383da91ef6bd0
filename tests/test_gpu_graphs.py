"""The library's calls can be captured in a CUDA graph and replayed: the
replays give the eager results bit for bit (the kernels' programmatic
dependent launches become graph edges; the top-1 workspace is left zeroed by
every call, so each replay starts clean)."""
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


def test_step_replays_as_a_graph(ops):
    M, K, N, NV = 6, 1024, 2048, 3001
    wq = synth.q4_0_weights(N, K, seed=41)
    wv = synth.q6_k_weights(NV, K, seed=42)
    x = _t(synth.activations(M, K, seed=43))
    wqp, wvp = ops.qpack_q4_0(_t(wq), N, K), ops.qpack_q6_k(_t(wv), NV, K)
    xq = torch.empty(ops.q8_1_bytes(M, K), dtype=torch.uint8, device=DEV)
    y = torch.empty((M, N), device=DEV)
    ids = torch.empty(M, dtype=torch.int32, device=DEV)
    idk = torch.empty((M, 4), dtype=torch.int32, device=DEV)
    vk = torch.empty((M, 4), device=DEV)
    ws = torch.zeros(ops.lmhead_q6_k_topk_workspace_bytes(M, K, NV, 4), dtype=torch.uint8, device=DEV)
    ws2 = torch.zeros(ops.lmhead_q6_k_top1_workspace_bytes(M, K, NV), dtype=torch.uint8, device=DEV)

    def step():
        ops.quantize_q8_1(x, out=xq)
        ops.qgemv_q4_0(wqp, xq, M, K, N, y=y)
        ops.lmhead_q6_k_top1(wvp, x, K, NV, ids=ids, ws=ws2)
        ops.lmhead_q6_k_topk(wvp, x, K, NV, 4, ws=ws, ids=idk, vals=vk)

    step()
    torch.cuda.synchronize()
    eager = [t.clone() for t in (xq, y, ids, idk, vk)]
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    for t in (xq, y, ids, idk, vk):
        t.zero_()
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    for got, want in zip((xq, y, ids, idk, vk), eager):
        assert torch.equal(got, want)
    # and the replayed results are the oracle's
    ids_ref, y_ref, S = oracle.lmhead_q6_k_top1(wv, x.cpu().numpy())
    assert C.check_top1(ids.cpu().numpy(), y_ref) == []
    yq_ref, Sq = oracle.qgemv_q4_0(wq, oracle.quantize_q8_1(x.cpu().numpy()))
    assert C.check_close(y.cpu().numpy(), yq_ref, Sq)["ok"]
    assert ops.qgemv_take_wait_timeouts() == 0
