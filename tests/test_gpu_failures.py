"""Failure paths, exercised without faulting the GPU.

- An injected launch failure (a host-side test hook) makes qmm_matmul return
  QMM_ERR_CUDA before any CUDA call: the output is left untouched and the
  next call works.
- An injected stall: the decode kernel's first block withholds its weight
  stages from one stage on, so that block's consumers wait for a copy that
  never comes.  With the bounded waits' limit lowered to 2^22 SM clocks (a few
  milliseconds), the wait gives up, the block drains the copies it did issue
  and exits; qmm_last_device_error reports QMM_ERR_TIMEOUT, and the context
  stays usable: the same call afterwards matches the oracle.
"""
import numpy as np
import pytest

import qmm_synth

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

QMM_ERR_CUDA, QMM_ERR_TIMEOUT = 6, 7


@pytest.fixture(scope="module")
def qmm():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from gguf_block_quantized_qmatmul_gb300 import build
    build.build()
    import gguf_block_quantized_qmatmul_gb300 as q
    return q


def _case(orc, wtype, M, N, K):
    wq_h = orc.quantize(wtype, qmm_synth.weights(N, K, seed=5))
    x_h = qmm_synth.activations(M, K, seed=6)
    return wq_h, x_h, torch.from_numpy(wq_h).cuda(), torch.from_numpy(x_h).cuda()


def _within(orc, wtype, mode, wq_h, x_h, y):
    y_orc, T = orc.matmul(wtype, mode, wq_h, x_h)
    assert np.all(np.abs(y.cpu().numpy().astype(np.float64) - y_orc) <= 1e-5 * T + 1e-6)


def test_injected_launch_failure_touches_nothing(qmm, orc):
    wtype, mode, M, N, K = "q8_0", "int8_act", 2, 512, 4096
    wq_h, x_h, wq, x = _case(orc, wtype, M, N, K)
    y = torch.full((M, N), float("nan"), device="cuda")
    torch.cuda.synchronize()
    qmm.test_inject("launch_failure", 1)
    try:
        with pytest.raises(qmm.QmmError) as e:
            qmm.matmul(wq, x, wtype, mode, N=N, out=y)
        assert e.value.status == QMM_ERR_CUDA
    finally:
        qmm.test_inject("off")
    torch.cuda.synchronize()
    assert torch.isnan(y).all()          # nothing was launched
    qmm.matmul(wq, x, wtype, mode, N=N, out=y)
    _within(orc, wtype, mode, wq_h, x_h, y)
    assert qmm.last_device_error() == 0


# (weight type, form, M, N, K): a decode call whose activations are prepared in
# the launch, and one whose activations are prepared by their own launch and
# fetched by the decode blocks (weights over 32 MB, M above 2)
STALL_CASES = [("q8_0", "int8_act", 2, 8192, 4096), ("q4_k", "f32_act", 4, 8192, 8192)]


@pytest.mark.parametrize("wtype,mode,M,N,K", STALL_CASES)
def test_injected_stall_times_out_and_recovers(qmm, orc, wtype, mode, M, N, K):
    wq_h, x_h, wq, x = _case(orc, wtype, M, N, K)
    y = torch.empty((M, N), device="cuda")
    assert qmm.matmul_launches(wtype, mode, M, N, K) >= 1
    assert qmm.last_device_error() == 0
    torch.cuda.synchronize()
    qmm.test_set_wait_limit(22)
    try:
        qmm.test_inject("stall", 1, 1)   # block 0 issues its first weight stage only
        qmm.matmul(wq, x, wtype, mode, N=N, out=y)
        torch.cuda.synchronize()         # the call ends: every wait is bounded
        assert qmm.last_device_error() == QMM_ERR_TIMEOUT
    finally:
        qmm.test_inject("off")
        qmm.test_set_wait_limit(0)
    assert qmm.last_device_error() == 0  # the error word was cleared by the read
    qmm.matmul(wq, x, wtype, mode, N=N, out=y)
    _within(orc, wtype, mode, wq_h, x_h, y)
    assert qmm.last_device_error() == 0
