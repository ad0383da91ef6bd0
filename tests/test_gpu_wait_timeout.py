"""The bounded waits' failure path, made to happen without any GPU fault.

A test-only switch makes the small-M tensor-core Q4_0 kernel issue no copy
for one warp's first job, so that warp's bounded wait (about a second) runs
out with no copy in flight for it.  The kernel counts the timeout and the
warp stops; the rest of the launch completes and the context stays usable.
Then every call that would enqueue work is refused with QGEMV_WAIT_TIMEOUT,
before enqueueing anything, until the count has been taken; after that the
same call runs and gives the right result again."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

from block_quantized_gemv_quantize_gb300 import synth  # noqa: E402

DEV = "cuda:0"
QGEMV_WAIT_TIMEOUT = -6


@pytest.fixture(scope="module")
def ops():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from block_quantized_gemv_quantize_gb300 import build

    build.build()
    from block_quantized_gemv_quantize_gb300 import ops as o

    return o


def test_wait_timeout_is_counted_and_refuses_calls_until_taken(ops):
    M, K, N = 6, 5120, 256
    w = synth.q4_0_weights(N, K, seed=31)
    x = synth.activations(M, K, seed=32)
    wp = ops.qpack_q4_0(torch.from_numpy(w).to(DEV), N, K)
    xq = ops.quantize_q8_1(torch.from_numpy(x).to(DEV))
    assert ops.qgemv_q4_0_plan(M, K, N)["kernel"] == "tc_small_m"
    y_ok = ops.qgemv_q4_0(wp, xq, M, K, N)
    assert ops.qgemv_take_wait_timeouts() == 0

    assert ops.qgemv_debug_drop_next_copy() == 0
    ops.qgemv_q4_0(wp, xq, M, K, N)  # one warp's wait runs out
    torch.cuda.synchronize()

    # refused before anything is enqueued: the output keeps its sentinel
    y = torch.full((M, N), float("nan"), device=DEV)
    with pytest.raises(ops.QgemvError) as e:
        ops.qgemv_q4_0(wp, xq, M, K, N, y=y)
    assert e.value.status == QGEMV_WAIT_TIMEOUT
    with pytest.raises(ops.QgemvError):
        ops.quantize_q8_1(torch.from_numpy(x).to(DEV))
    torch.cuda.synchronize()
    assert torch.isnan(y).all()

    assert ops.qgemv_take_wait_timeouts() >= 1
    assert ops.qgemv_take_wait_timeouts() == 0
    y2 = ops.qgemv_q4_0(wp, xq, M, K, N)
    torch.cuda.synchronize()
    assert torch.equal(y2, y_ok)
    assert np.isfinite(y2.cpu().numpy()).all()
