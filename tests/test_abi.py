"""The C-ABI library builds, loads and exports every declared symbol; host-side
argument checks (no GPU needed: every call here returns before touching the
device)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def qmm():
    from gguf_block_quantized_qmatmul_gb300 import build
    build.build()
    import gguf_block_quantized_qmatmul_gb300 as q
    return q


def header_functions():
    src = open(os.path.join(ROOT, "include", "qmm.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(qmm_[a-z0-9_]+)\s*\(", src)))


def test_exports_every_declared_symbol(qmm):
    lib = ctypes.CDLL(qmm._build.LIB)
    names = header_functions()
    assert len(names) >= 11
    for n in names:
        assert hasattr(lib, n), n
    assert sorted(qmm.EXPORTS) == names


def test_block_sizes(qmm):
    assert (qmm.block_values("q8_0"), qmm.block_bytes("q8_0")) == (32, 34)
    assert (qmm.block_values("q4_k"), qmm.block_bytes("q4_k")) == (256, 144)
    assert (qmm.block_values("q8_k"), qmm.block_bytes("q8_k")) == (256, 292)
    assert (qmm.block_values("q4_0"), qmm.block_bytes("q4_0")) == (32, 18)
    assert (qmm.block_values("q5_0"), qmm.block_bytes("q5_0")) == (32, 22)
    assert (qmm.block_values("q6_k"), qmm.block_bytes("q6_k")) == (256, 210)
    assert qmm.row_bytes("q6_k", 1536) == 1260    # half of the downloaded file's ffn_down
    assert qmm.row_bytes("q6_k", 576) == 0        # a K-quant: K % 256
    assert qmm.row_bytes("q5_0", 576) == 396      # the 576-wide SmolLM2 matrices take Q5_0
    assert qmm.row_bytes("q8_0", 576) == 612
    assert qmm.row_bytes("q4_k", 1536) == 864
    assert qmm.row_bytes("q4_k", 576) == 0        # the K-quant shape error
    assert qmm.row_bytes("q8_0", 33) == 0
    assert qmm.block_bytes(99) == 0


def test_row_bytes_agree_with_oracle(qmm, orc):
    for t in ("q8_0", "q4_k", "q8_k", "q4_0", "q5_0", "q6_k"):
        for K in (256, 512, 4096, 8192):
            assert qmm.row_bytes(t, K) == orc.row_bytes(t, K)


def _lib(qmm):
    return qmm._lib()


def test_argument_errors_return_before_launch(qmm):
    L = _lib(qmm)
    Q8_0, Q4_K, Q8_K, F32 = qmm.QMM_Q8_0, qmm.QMM_Q4_K, qmm.QMM_Q8_K, qmm.QMM_F32
    # wrong weight / activation types
    assert L.qmm_quantize_weights(Q8_K, 16, 4, 256, 16, None) == 3
    assert L.qmm_quantize_weights(F32, 16, 4, 256, 16, None) == 3
    assert L.qmm_quantize_act(Q4_K, 16, 4, 256, 16, None) == 3
    assert L.qmm_quantize_act(qmm.QMM_Q5_0, 16, 4, 256, 16, None) == 3   # Q5_0 weights take Q8_0 activations
    assert L.qmm_quantize_act(qmm.QMM_Q6_K, 16, 4, 256, 16, None) == 3   # Q6_K weights take Q8K activations
    assert L.qmm_matmul(qmm.QMM_Q6_K, 0, 16, 16, 16, 1, 1, 576, None, 0, None) == 2   # K % 256
    assert L.qmm_matmul(qmm.QMM_Q4_0, 0, 16, 16, 16, 1, 1, 100, None, 0, None) == 2
    assert L.qmm_matmul(Q8_K, 0, 16, 16, 16, 1, 1, 256, None, 0, None) == 3
    assert L.qmm_matmul(Q8_0, 7, 16, 16, 16, 1, 1, 256, None, 0, None) == 3
    assert L.qmm_dequantize(F32, 16, 1, 256, 16, None) == 3
    # K not a multiple of the block: the Q4K shape error on 576-wide rows
    assert L.qmm_quantize_weights(Q4_K, 16, 576, 576, 16, None) == 2
    assert L.qmm_matmul(Q4_K, 0, 16, 16, 16, 1, 576, 576, None, 0, None) == 2
    assert L.qmm_matmul(Q8_0, 0, 16, 16, 16, 1, 1, 100, None, 0, None) == 2
    assert L.qmm_matmul(Q8_0, 0, 16, 16, 16, -1, 1, 256, None, 0, None) == 2
    assert L.qmm_block_sums(Q8_0, 16, 16, 1, -3, 256, 16, None) == 2
    # NULL pointers
    assert L.qmm_quantize_weights(Q8_0, None, 4, 256, 16, None) == 1
    assert L.qmm_matmul(Q8_0, 0, None, 16, 16, 1, 1, 256, None, 0, None) == 1
    assert L.qmm_matmul(Q8_0, 1, 16, 16, None, 1, 1, 256, None, 0, None) == 1
    assert L.qmm_dequantize(Q8_0, 16, 1, 256, None, None) == 1
    # misaligned pointers
    assert L.qmm_matmul(Q8_0, 0, 18, 16, 16, 1, 1, 256, None, 0, None) == 4
    assert L.qmm_matmul(Q8_0, 0, 16, 20, 16, 1, 1, 256, None, 0, None) == 4
    assert L.qmm_matmul(Q8_0, 0, 16, 16, 18, 1, 1, 256, None, 0, None) == 4
    assert L.qmm_quantize_weights(Q4_K, 16, 4, 256, 8, None) == 4
    # empty problems are no-ops, even with NULL pointers
    assert L.qmm_matmul(Q8_0, 0, None, None, None, 0, 5, 256, None, 0, None) == 0
    assert L.qmm_matmul(Q4_K, 1, None, None, None, 3, 0, 256, None, 0, None) == 0
    assert L.qmm_quantize_act(Q8_K, None, 0, 256, None, None) == 0
    for s in range(8):
        assert L.qmm_status_string(s)


def test_batch_argument_errors_return_before_launch(qmm):
    L = _lib(qmm)
    D = qmm.MatmulDesc
    ok = D(16, 16, 16, 1, 8, 64)

    def call(wtype, mode, items):
        arr = (D * max(len(items), 1))(*items)
        return L.qmm_matmul_batch(wtype, mode, ctypes.cast(arr, ctypes.c_void_p), len(items), None)

    assert call(qmm.QMM_Q8_K, 0, [ok]) == 3                  # weight types only
    assert call(qmm.QMM_F32, 0, [ok]) == 3
    assert call(qmm.QMM_Q4_K, 0, [ok]) == 2                  # K % 256
    assert call(qmm.QMM_Q6_K, 1, [ok, D(16, 16, 16, 1, 8, 700)]) == 2     # K % 256
    assert call(qmm.QMM_Q8_0, 5, [ok]) == 3
    assert call(qmm.QMM_Q8_0, 0, [ok, D(16, 16, 16, 9, 8, 64)]) == 2      # M > QMM_BATCH_MAX_M
    assert call(qmm.QMM_Q8_0, 0, [ok, D(16, 16, 16, 2, 8, 16384)]) == 2   # M * K > QMM_BATCH_MAX_MK
    assert call(qmm.QMM_Q5_0, 1, [D(16, 16, 16, 1, 8, 100)]) == 2         # K % 32
    assert call(qmm.QMM_Q4_0, 0, [D(None, 16, 16, 1, 8, 64)]) == 1
    assert call(qmm.QMM_Q8_0, 0, [D(18, 16, 16, 1, 8, 64)]) == 4
    assert call(qmm.QMM_Q8_0, 0, [D(None, None, None, 0, 8, 64)]) == 0   # empty items are skipped
    assert L.qmm_matmul_batch(qmm.QMM_Q8_0, 0, None, 0, None) == 0
    assert L.qmm_matmul_batch(qmm.QMM_Q8_0, 0, None, 3, None) == 1


def test_typed_batch_argument_errors_return_before_launch(qmm):
    L = _lib(qmm)
    D = qmm.TypedMatmulDesc
    ok = D(qmm.QMM_Q8_0, 16, 16, 16, 1, 8, 64)

    def call(mode, items):
        arr = (D * max(len(items), 1))(*items)
        return L.qmm_matmul_batch_typed(mode, ctypes.cast(arr, ctypes.c_void_p), len(items), None)

    assert call(5, [ok]) == 3
    assert call(0, [ok, D(qmm.QMM_Q8_K, 16, 16, 16, 1, 8, 256)]) == 3      # an item's type
    assert call(0, [ok, D(qmm.QMM_Q4_K, 16, 16, 16, 1, 8, 64)]) == 2       # K % 256 for Q4_K
    assert call(1, [ok, D(qmm.QMM_Q6_K, 16, 16, 16, 9, 8, 256)]) == 2      # M > QMM_BATCH_MAX_M
    assert call(0, [ok, D(qmm.QMM_Q4_K, 16, 16, 16, 2, 8, 8448 + 8192)]) == 2  # M * K > QMM_BATCH_MAX_MK
    assert call(0, [ok, D(qmm.QMM_Q5_0, None, 16, 16, 1, 8, 64)]) == 1
    assert call(0, [ok, D(qmm.QMM_Q6_K, 24, 16, 16, 1, 8, 256)]) == 4
    assert call(0, [D(qmm.QMM_Q4_K, None, None, None, 0, 8, 256)]) == 0  # empty items are skipped
    assert L.qmm_matmul_batch_typed(0, None, 0, None) == 0
    assert L.qmm_matmul_batch_typed(0, None, 2, None) == 1


def test_binding_raises_on_error_status(qmm):
    with pytest.raises(qmm.QmmError) as e:
        qmm._check(2, "qmm_matmul")
    assert e.value.status == 2 and "QMM_ERR_SHAPE" in str(e.value)


def test_product_package_never_imports_the_oracle():
    pkg = os.path.join(ROOT, "gguf_block_quantized_qmatmul_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h", ".cpp")):
                txt = open(os.path.join(dirpath, f), encoding="utf-8").read()
                assert "import oracle" not in txt and "from oracle" not in txt and "qmm_oracle" not in txt, f


def test_injected_launch_failure_needs_no_device(qmm):
    """The failure-test hook: an armed launch failure makes the next call
    return QMM_ERR_CUDA before any CUDA call (this host has no GPU, so any
    CUDA call would fail differently or hang nothing), and arguments of the
    hooks themselves are checked on the host."""
    L = _lib(qmm)
    assert L.qmm_test_inject(1, 2, 0) == 0
    for _ in range(2):   # valid, aligned arguments: only the injection stops the call
        assert L.qmm_matmul(qmm.QMM_Q8_0, 0, 16, 16, 16, 1, 1, 256, None, 0, None) == 6
    assert L.qmm_test_inject(0, 0, 0) == 0
    assert L.qmm_test_inject(9, 1, 0) == 3            # unknown kind
    assert L.qmm_test_inject(1, -1, 0) == 2           # negative count
    assert L.qmm_test_set_wait_limit(5) == 2          # below 2^16 clocks
    assert L.qmm_test_set_wait_limit(40) == 2
