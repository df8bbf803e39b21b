"""qmm_matmul_static_workspace: the matmul for callers that cannot allocate.

Callers such as a host engine that owns every device allocation, or a
latency-critical loop that must not touch the allocator, cannot hand
qmm_matmul a workspace.  This entry point uses the library's own device array
instead.  Here it is called through the C ABI and compared with the CPU oracle
and with qmm_matmul (whose workspace the test allocates), on two calls in a
row, with the same bound the parity tests use, on each kernel that can need a
workspace; a shape whose workspace exceeds the array must be refused before
any launch.  This file is collected last on purpose.
"""
import ctypes

import numpy as np
import pytest

import qmm_synth

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def qmm():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from gguf_block_quantized_qmatmul_gb300 import build
    build.build()
    import gguf_block_quantized_qmatmul_gb300 as q
    return q


def _entry(q):
    lib = ctypes.CDLL(q._build.LIB)
    f = lib.qmm_matmul_static_workspace
    i64, p = ctypes.c_int64, ctypes.c_void_p
    f.argtypes = [ctypes.c_int, ctypes.c_int, p, p, p, i64, i64, i64, p]
    f.restype = ctypes.c_int
    return f


# Shapes whose workspace the entry point takes from its own array: the decode
# kernel with K split (partial sums only), the tcgen05 GEMM with K split (its
# arrival counters must start at zero on every call; Q6_K also repacks its
# weights there), the exact Q8_0 prefill GEMM (activation codes) and the
# streaming kernel with K split (arrival counters cleared by a memset).
STATIC_CASES = [("q8_0", "f32_act", 8, 100, 8192), ("q8_0", "f32_act", 64, 300, 4096),
                ("q4_k", "f32_act", 37, 256, 2048), ("q6_k", "f32_act", 37, 64, 4096),
                ("q8_0", "int8_act", 64, 300, 4096), ("q6_k", "int8_act", 37, 64, 4096)]


@pytest.mark.parametrize("wtype,mode,M,N,K", STATIC_CASES)
def test_static_workspace_matches_qmm_matmul(qmm, orc, wtype, mode, M, N, K):
    f = _entry(qmm)
    need = qmm.matmul_workspace(wtype, mode, M, N, K)
    assert 0 < need <= 8 << 20        # a workspace is really used, and it fits the array
    wq_h = orc.quantize(wtype, qmm_synth.weights(N, K, seed=21))
    wq = torch.from_numpy(wq_h).cuda()
    stream = torch.cuda.current_stream().cuda_stream
    for call in range(2):             # two calls in a row: the array keeps the last call's contents
        x_h = qmm_synth.activations(M, K, seed=30 + call, outlier_channels=4 if M >= 16 else 0)
        x = torch.from_numpy(x_h).cuda()
        y_ref = qmm.matmul(wq, x, wtype, mode, N=N)
        y = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
        st = f(qmm.TYPES[wtype], qmm.MODES[mode], wq.data_ptr(), x.data_ptr(), y.data_ptr(), M, N, K, stream)
        assert st == 0, qmm._lib().qmm_status_string(st)
        torch.cuda.synchronize()
        y_orc, T = orc.matmul(wtype, mode, wq_h, x_h)
        bound = 1e-5 * T + 1e-6
        got = y.cpu().numpy().astype(np.float64)
        # against the oracle, and against qmm_matmul with a caller's workspace
        assert np.all(np.abs(got - y_orc) <= bound)
        assert np.all(np.abs(got - y_ref.cpu().numpy()) <= bound)
    assert qmm.last_device_error() == 0


def test_static_workspace_refuses_too_large_shapes(qmm):
    f = _entry(qmm)
    wtype, mode, M, N, K = "q8_0", "f32_act", 1024, 14336, 4096
    assert qmm.matmul_workspace(wtype, mode, M, N, K) > 8 << 20
    # real buffers of the full size, so that nothing could run out of bounds even if the check failed
    wq = torch.zeros((N, qmm.row_bytes(wtype, K)), dtype=torch.uint8, device="cuda")
    x = torch.zeros((M, K), dtype=torch.float32, device="cuda")
    y = torch.zeros((M, N), dtype=torch.float32, device="cuda")
    st = f(qmm.TYPES[wtype], qmm.MODES[mode], wq.data_ptr(), x.data_ptr(), y.data_ptr(), M, N, K,
           torch.cuda.current_stream().cuda_stream)
    assert st == 5                    # QMM_ERR_WORKSPACE
