"""Parity of the CUDA path (through the C ABI) with the CPU oracle.

Codes, packed scales, dequantized values and integer block sums: bit-exact.
Float outputs: |y_gpu - y_oracle| <= 1e-5 * T + 1e-6 per element, with T the
sum of |scaled block terms| the oracle returns beside y.
"""
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


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def host(t):
    torch.cuda.synchronize()
    return t.cpu().numpy()


def assert_within_bound(y_gpu, y_orc, T, what=""):
    err = np.abs(y_gpu.astype(np.float64) - y_orc)
    bound = 1e-5 * T + 1e-6
    worst = np.max(err / bound) if err.size else 0.0
    assert np.all(err <= bound), f"{what}: worst err/bound = {worst:.3g}"
    return worst


def check_device_error(qmm):
    assert qmm.last_device_error() == 0


# Canaries: outputs are views into a larger buffer whose guard words before
# and after hold a NaN bit pattern; a write outside the output shows.  The
# output itself starts as that NaN, so an element left unwritten fails too.
CANARY = 0x7FBADBAD
GUARD = 64  # 4-byte words on each side


def guarded_out(M, N):
    buf = torch.full((M * N + 2 * GUARD,), CANARY, dtype=torch.int32, device="cuda")
    return buf, buf[GUARD:GUARD + M * N].view(torch.float32).view(M, N)


def check_guards(buf, what=""):
    b = host(buf)
    assert (b[:GUARD] == CANARY).all() and (b[-GUARD:] == CANARY).all(), f"{what}: write outside the output"


def matmul_checked(qmm, wq, x, wtype, mode, N, **kw):
    """qmm.matmul into a guarded output; returns y on the host."""
    M = x.shape[0]
    buf, y = guarded_out(M, N)
    qmm.matmul(wq, x, wtype, mode, N=N, out=y, **kw)
    out = host(y).copy()
    check_guards(buf, f"{wtype} {mode} M{M} N{N}")
    return out


# ---------------------------------------------------------------------------
# quantizers and dequantization: bit-exact
# ---------------------------------------------------------------------------

WEIGHT_CASES = [("q8_0", 576, 576), ("q8_0", 37, 96), ("q8_0", 61, 608), ("q8_0", 5, 8192),
                ("q4_k", 576, 1536), ("q4_k", 37, 256), ("q4_k", 19, 8192),
                ("q4_0", 576, 576), ("q4_0", 37, 96), ("q5_0", 576, 576), ("q5_0", 1536, 576), ("q5_0", 7, 8192),
                ("q6_k", 576, 1536), ("q6_k", 37, 256), ("q6_k", 19, 8192)]


@pytest.mark.parametrize("wtype,N,K", WEIGHT_CASES)
def test_quantize_weights_bit_exact(qmm, orc, wtype, N, K):
    w = np.concatenate([qmm_synth.weights(N, K, seed=N + K), qmm_synth.special_block_rows(K)])
    q = host(qmm.quantize_weights(dev(w), wtype))
    ref = orc.quantize(wtype, w)
    assert np.array_equal(q, ref)
    check_device_error(qmm)


@pytest.mark.parametrize("atype,M,K", [("q8_0", 8, 576), ("q8_0", 3, 8192), ("q8_k", 8, 1536), ("q8_k", 5, 8192)])
def test_quantize_act_bit_exact(qmm, orc, atype, M, K):
    x = np.concatenate([qmm_synth.activations(M, K, outlier_channels=4), qmm_synth.special_block_rows(K)])
    q = host(qmm.quantize_act(dev(x), atype))
    assert np.array_equal(q, orc.quantize(atype, x))


@pytest.mark.parametrize("t,K", [("q8_0", 576), ("q4_k", 1536), ("q8_k", 1024), ("q4_0", 576), ("q5_0", 576),
                                 ("q6_k", 1536)])
def test_dequantize_bit_exact(qmm, orc, t, K):
    w = np.concatenate([qmm_synth.weights(40, K), qmm_synth.special_block_rows(K)])
    q = orc.quantize(t, w)
    out = host(qmm.dequantize(dev(q), t, K))
    ref = orc.dequantize(t, q, K)
    assert np.array_equal(out.view(np.uint32), ref.view(np.uint32))


# ---------------------------------------------------------------------------
# integer block sums of the int8_act kernel: bit-exact
# ---------------------------------------------------------------------------

SUM_CASES = [("q8_0", 1, 33, 576), ("q8_0", 8, 576, 576), ("q8_0", 5, 40, 4096), ("q8_0", 13, 17, 1536),
             ("q8_0", 37, 24, 96), ("q4_k", 1, 33, 1536), ("q4_k", 8, 64, 2048), ("q4_k", 19, 20, 4096),
             ("q4_0", 1, 33, 576), ("q4_0", 13, 40, 1536), ("q5_0", 1, 192, 576), ("q5_0", 8, 33, 576),
             ("q5_0", 37, 24, 4096), ("q6_k", 1, 33, 1536), ("q6_k", 8, 64, 2048), ("q6_k", 19, 20, 4096),
             ("q4_k", 16, 40, 2048), ("q4_0", 12, 50, 1536), ("q8_0", 16, 33, 4096)]


@pytest.mark.parametrize("wtype,M,N,K", SUM_CASES)
def test_block_sums_bit_exact(qmm, orc, wtype, M, N, K):
    w = qmm_synth.weights(N, K, seed=3)
    w[0] = 1.0                    # all codes at the extreme
    x = qmm_synth.activations(M, K, seed=4, outlier_channels=4)
    x[0] = -1.0
    wq = orc.quantize(wtype, w)
    s = host(qmm.block_sums(dev(wq), dev(x), wtype, N=N))
    xq = orc.quantize("q8_k" if wtype in ("q4_k", "q6_k") else "q8_0", x)
    ref = orc.block_sums(wtype, wq, xq, M, N, K)
    assert np.array_equal(s, ref)
    check_device_error(qmm)


# ---------------------------------------------------------------------------
# matmul: both forms against the oracle's bound
# ---------------------------------------------------------------------------

MATMUL_CASES = [
    ("q8_0", 1, 576, 576),        # SmolLM2 q/o projection, single-token decode
    ("q8_0", 1, 192, 576),
    ("q8_0", 1, 576, 1536),       # ffn_down
    ("q8_0", 1, 1536, 576),
    ("q4_k", 1, 576, 1536),       # ffn_down in Q4_K, batches 1, 2, 4, 8
    ("q4_k", 2, 576, 1536),
    ("q4_k", 4, 576, 1536),
    ("q4_k", 8, 576, 1536),
    ("q8_0", 5, 37, 608),         # ragged tile, odd number of blocks
    ("q8_0", 8, 100, 8192),       # f32_act splits K here
    ("q4_k", 8, 100, 8192),
    ("q8_0", 16, 70, 4096),
    ("q8_0", 37, 64, 4096),       # prefill, ragged M
    ("q4_k", 37, 64, 4096),
    ("q8_0", 64, 33, 1024),
    ("q4_k", 100, 48, 1024),
    ("q8_0", 300, 260, 2048),     # prefill tiles: 3 x 3 with ragged edges in both
    ("q4_k", 200, 300, 1024),
    ("q8_0", 256, 384, 2048),     # 256-row activation tiles, one accumulator
    ("q4_k", 520, 130, 1024),     # three activation tiles of 176 rows, ragged weight tile
    ("q4_k", 9, 1000, 512),       # smallest prefill M (16-row activation tile)
    ("q5_0", 1, 576, 576),        # SmolLM2 Q5_0 projections (K = 576 rules out K-quants)
    ("q5_0", 1, 1536, 576),
    ("q5_0", 4, 192, 576),
    ("q5_0", 8, 576, 1536),
    ("q5_0", 37, 300, 576),       # prefill, ragged
    ("q4_0", 1, 576, 576),
    ("q4_0", 2, 100, 8192),       # K split across CTAs
    ("q4_0", 64, 130, 1024),      # prefill on tcgen05 (K % 256 = 0)
    ("q5_0", 256, 200, 1536),
    ("q4_0", 300, 260, 2048),
    ("q4_k", 13, 300, 4096),      # 9..16 rows on the warp-MMA kernel: f32 four column sets, K split
    ("q8_0", 12, 2050, 8192),     # ragged tile, activations prepared in the kernel
    ("q4_0", 16, 600, 4096),
    ("q5_0", 11, 333, 1536),
    ("q8_0", 16, 4100, 8192),     # 35.6 MB of weights: activations prepared once, then the decode kernel
    ("q6_k", 1, 576, 1536),       # the downloaded file's Q6K ffn_down, decode batches 1 and 8
    ("q6_k", 8, 576, 1536),
    ("q6_k", 3, 37, 8192),        # ragged tile, long rows
    ("q6_k", 2, 100, 8192),
    ("q6_k", 37, 64, 4096),       # prefill, ragged M
    ("q6_k", 200, 130, 1024),
    ("q4_k", 8, 40, 65536),       # long rows: activations split over K, 256 raw stages
    ("q8_0", 24, 24, 65536),
]


@pytest.mark.parametrize("mode", ["int8_act", "f32_act"])
@pytest.mark.parametrize("wtype,M,N,K", MATMUL_CASES)
def test_matmul_within_bound(qmm, orc, wtype, M, N, K, mode):
    w = qmm_synth.weights(N, K, seed=N * 7 + K)
    x = qmm_synth.activations(M, K, seed=M + 11, outlier_channels=4 if M >= 16 else 0)
    wq = orc.quantize(wtype, w)
    y = matmul_checked(qmm, dev(wq), dev(x), wtype, mode, N)
    y_orc, T = orc.matmul(wtype, mode, wq, x)
    assert_within_bound(y, y_orc, T, f"{wtype} {mode} M{M} N{N} K{K}")
    check_device_error(qmm)


@pytest.mark.parametrize("mode", ["int8_act", "f32_act"])
@pytest.mark.parametrize("wtype,K", [("q8_0", 1024), ("q4_k", 1024), ("q4_0", 1024), ("q5_0", 1024)])
def test_prefill_special_rows(qmm, orc, wtype, K, mode):
    """Prefill (M > 8) with the adversarial rows in both operands: zeros,
    constants, one-hot, ties, magnitudes from 1e-9 to 3e3 (each operand row is
    scaled by its own power of two before the f16 split)."""
    w = np.concatenate([qmm_synth.weights(100, K, seed=5), qmm_synth.special_block_rows(K)])
    x = np.concatenate([qmm_synth.activations(20, K, seed=6, outlier_channels=4), qmm_synth.special_block_rows(K)])
    wq = orc.quantize(wtype, w)
    y = host(qmm.matmul(dev(wq), dev(x), wtype, mode, N=w.shape[0]))
    y_orc, T = orc.matmul(wtype, mode, wq, x)
    assert_within_bound(y, y_orc, T, f"{wtype} {mode} special rows")
    check_device_error(qmm)


# ---------------------------------------------------------------------------
# adversarial rows (zeros, constants, one-hot, rounding ties, all-negative and
# all-positive blocks, magnitudes from the bottom of the f32 range to 3e3,
# +-127 and integer blocks) in both operands, through every matmul kernel
# ---------------------------------------------------------------------------

def edge_operands(wtype, K, M, n_plain=20, seed=0):
    """Weights: plain rows followed by the adversarial rows.  Activations: M
    rows cycling through the adversarial rows from a per-M offset (plain rows
    fill in past them)."""
    sp = qmm_synth.special_block_rows(K)
    w = np.concatenate([qmm_synth.weights(n_plain, K, seed=seed + 1), sp])
    plain = qmm_synth.activations(max(M, 1), K, seed=seed + 2)
    x = np.stack([sp[(5 * m + M) % len(sp)] if m < len(sp) else plain[m] for m in range(M)]).astype(np.float32)
    return w, x


DECODE_EDGE = [(t, M) for t in ("q8_0", "q4_k", "q4_0", "q5_0", "q6_k") for M in (2, 4, 8, 16)]


@pytest.mark.parametrize("mode", ["int8_act", "f32_act"])
@pytest.mark.parametrize("wtype,M", DECODE_EDGE)
def test_decode_kernel_edge_rows(qmm, orc, wtype, M, mode):
    """The 16-row warp-MMA decode kernel (activations prepared in the launch):
    every weight type, 2..16 activation rows, both forms, adversarial rows in
    both operands; outputs guarded by canaries."""
    K = 1536
    w, x = edge_operands(wtype, K, M)
    wq = orc.quantize(wtype, w)
    y = matmul_checked(qmm, dev(wq), dev(x), wtype, mode, w.shape[0])
    y_orc, T = orc.matmul(wtype, mode, wq, x)
    assert_within_bound(y, y_orc, T, f"{wtype} {mode} M{M} edge rows")
    check_device_error(qmm)


@pytest.mark.parametrize("mode", ["int8_act", "f32_act"])
@pytest.mark.parametrize("wtype", ["q8_0", "q4_k", "q4_0", "q5_0", "q6_k"])
def test_single_row_edge_rows(qmm, orc, wtype, mode):
    """M = 1 (the dp4a GEMV for Q8_0 int8_act, the warp-MMA decode kernel
    otherwise): each adversarial row alone as the activation."""
    K = 1536
    sp = qmm_synth.special_block_rows(K)
    w = np.concatenate([qmm_synth.weights(20, K, seed=9), sp])
    wq = orc.quantize(wtype, w)
    wq_d = dev(wq)
    for i in range(len(sp)):
        x = sp[i:i + 1]
        y = matmul_checked(qmm, wq_d, dev(x), wtype, mode, w.shape[0])
        y_orc, T = orc.matmul(wtype, mode, wq, x)
        assert_within_bound(y, y_orc, T, f"{wtype} {mode} adversarial row {i}")
    check_device_error(qmm)


@pytest.mark.parametrize("mode", ["int8_act", "f32_act"])
@pytest.mark.parametrize("wtype,N,M", [("q8_0", 4100, 8), ("q8_0", 4100, 16), ("q4_k", 8192, 4), ("q4_k", 8192, 8),
                                       ("q6_k", 5000, 8)])
def test_prepared_activations_edge_rows(qmm, orc, wtype, N, M, mode):
    """Weights over 32 MB with more than a few rows: the activations are
    prepared once by their own launch, then fetched by every decode block;
    adversarial rows in both operands (the weights' last rows)."""
    K = 8192
    w, x = edge_operands(wtype, K, M, n_plain=N - len(qmm_synth.special_block_rows(K)), seed=40)
    assert qmm.matmul_launches(wtype, mode, M, N, K) >= 2
    wq = orc.quantize(wtype, w)
    y = matmul_checked(qmm, dev(wq), dev(x), wtype, mode, N)
    y_orc, T = orc.matmul(wtype, mode, wq, x)
    assert_within_bound(y, y_orc, T, f"{wtype} {mode} M{M} N{N} prepared activations, edge rows")
    check_device_error(qmm)


@pytest.mark.parametrize("mode", ["int8_act", "f32_act"])
@pytest.mark.parametrize("wtype,M,K", [("q8_0", 37, 576), ("q5_0", 37, 576), ("q4_0", 20, 576), ("q8_0", 300, 96),
                                       ("q6_k", 37, 1536), ("q6_k", 37, 8192), ("q6_k", 300, 512)])
def test_prefill_kernels_edge_rows(qmm, orc, wtype, M, K, mode):
    """Prefill above 16 rows: the streaming warp-MMA kernel (32-value blocks
    with K % 256 != 0) and the tcgen05 GEMM on Q6_K (super-blocks repacked
    into 16-byte aligned slots), with and without a K split: adversarial rows
    in both operands."""
    w, x = edge_operands(wtype, K, M, n_plain=50, seed=60)
    wq = orc.quantize(wtype, w)
    y = matmul_checked(qmm, dev(wq), dev(x), wtype, mode, w.shape[0])
    y_orc, T = orc.matmul(wtype, mode, wq, x)
    assert_within_bound(y, y_orc, T, f"{wtype} {mode} M{M} K{K} streaming, edge rows")
    check_device_error(qmm)


@pytest.mark.parametrize("wtype,M,K", [("q8_0", 1, 576), ("q8_0", 8, 1536), ("q4_k", 8, 1536), ("q4_0", 4, 576),
                                       ("q5_0", 16, 576), ("q6_k", 8, 1536), ("q6_k", 37, 1536), ("q8_0", 37, 576),
                                       ("q4_k", 37, 1536)])
def test_block_sums_edge_rows_bit_exact(qmm, orc, wtype, M, K):
    """Integer block sums with adversarial rows in both operands: bit-exact
    (decode kernel, GEMV and streaming kernel)."""
    w, x = edge_operands(wtype, K, M, n_plain=20, seed=80)
    wq = orc.quantize(wtype, w)
    N = w.shape[0]
    s = host(qmm.block_sums(dev(wq), dev(x), wtype, N=N))
    xq = orc.quantize("q8_k" if wtype in ("q4_k", "q6_k") else "q8_0", x)
    assert np.array_equal(s, orc.block_sums(wtype, wq, xq, M, N, K))
    check_device_error(qmm)


@pytest.mark.parametrize("mode", ["int8_act", "f32_act"])
@pytest.mark.parametrize("wtype", ["q8_0", "q4_0", "q5_0", "q4_k", "q6_k"])
def test_matmul_batch_edge_rows(qmm, orc, wtype, mode):
    """qmm_matmul_batch with adversarial rows in the weights and activation
    rows of its items (M = 1..8, K = 576 or 256 and 1536); guarded outputs."""
    items, refs, guards = [], [], []
    k0 = 256 if wtype in ("q4_k", "q6_k") else 576
    for i, (M, K) in enumerate([(1, k0), (2, k0), (8, 1536), (4, 1536), (1, 1536), (8, k0)]):
        w, x = edge_operands(wtype, K, M, n_plain=7 + i, seed=100 + i)
        wq = orc.quantize(wtype, w)
        buf, y = guarded_out(M, w.shape[0])
        items.append((dev(wq), dev(x), y))
        refs.append(orc.matmul(wtype, mode, wq, x))
        guards.append(buf)
    qmm.matmul_batch(items, wtype, mode)
    for (wq, x, y), (y_orc, T), buf in zip(items, refs, guards):
        assert_within_bound(host(y), y_orc, T, f"batch {wtype} {mode} edge rows M{x.shape[0]}")
        check_guards(buf, "batch item")
    check_device_error(qmm)


@pytest.mark.parametrize("wtype,M,N,K", [("q8_0", 64, 300, 4096), ("q4_k", 256, 200, 2048), ("q4_k", 37, 200, 2048)])
def test_prefill_split_k_is_deterministic(qmm, orc, wtype, M, N, K):
    """Few output tiles split K across CTAs; the tile's last unit sums the
    partial tiles in slice order, so repeated calls agree bit for bit."""
    w = qmm_synth.weights(N, K, seed=3)
    x = dev(qmm_synth.activations(M, K, seed=4, outlier_channels=4))
    wq = dev(orc.quantize(wtype, w))
    for mode in ("int8_act", "f32_act"):
        ys = [host(qmm.matmul(wq, x, wtype, mode, N=N)) for _ in range(3)]
        assert np.array_equal(ys[0], ys[1]) and np.array_equal(ys[0], ys[2])
    check_device_error(qmm)


@pytest.mark.parametrize("wtype,M,N,K", [("q8_0", 40, 25600, 512), ("q4_k", 40, 25600, 512), ("q6_k", 40, 25600, 512),
                                        ("q5_0", 40, 25600, 512), ("q8_0", 200, 12800, 512), ("q4_k", 200, 12800, 512)])
def test_prefill_ctas_take_several_tiles(qmm, orc, wtype, M, N, K):
    """More output tiles than SMs (200 tiles of 128 weight rows): the
    persistent tcgen05 CTAs take several tiles each, so the accumulator and
    stage rings (and their barrier phases) carry over from one tile to the
    next, at 64- and 128-row activation tiles, in both forms."""
    w = qmm_synth.weights(N, K, seed=5)
    x_np = qmm_synth.activations(M, K, seed=6, outlier_channels=4)
    wq_h = orc.quantize(wtype, w)
    wq, x = dev(wq_h), dev(x_np)
    for mode in ("int8_act", "f32_act"):
        y = matmul_checked(qmm, wq, x, wtype, mode, N)
        y_orc, T = orc.matmul(wtype, mode, wq_h, x_np)
        assert_within_bound(y, y_orc, T, f"{wtype} {mode} M{M} N{N} K{K}")
    check_device_error(qmm)


def test_gap_ordering(qmm, orc):
    """The CPU form's distance to the dequantized-f32 product is far larger
    than the Metal form's (the activation-quantization error; the pages put
    the ratio at about 30 on model logits)."""
    for wtype, N, K in (("q8_0", 576, 576), ("q4_k", 576, 1536)):
        wq = orc.quantize(wtype, qmm_synth.weights(N, K))
        x = qmm_synth.activations(8, K)
        y_deq, _ = orc.matmul(wtype, "f32_act", wq, x)
        yi = host(qmm.matmul(dev(wq), dev(x), wtype, "int8_act", N=N)).astype(np.float64)
        yf = host(qmm.matmul(dev(wq), dev(x), wtype, "f32_act", N=N)).astype(np.float64)
        gap_cpu = np.abs(yi - y_deq).max()
        gap_metal = np.abs(yf - y_deq).max()
        assert gap_cpu >= 30 * gap_metal, (wtype, gap_cpu, gap_metal)


def test_batch_rows_are_independent(qmm, orc):
    """Row m's codes and integer block sums do not depend on the other rows of
    the batch (bit-exact); its output agrees within the bound (a batch of 8
    and a single row may run on different kernel paths, which sum in a
    different order)."""
    K, N = 1536, 96
    for wtype in ("q8_0", "q4_k"):
        wq_h = orc.quantize(wtype, qmm_synth.weights(N, K))
        wq = dev(wq_h)
        x = qmm_synth.activations(8, K)
        x[3] *= 40.0
        _, T = orc.matmul(wtype, "int8_act", wq_h, x)
        yb = host(qmm.matmul(wq, dev(x), wtype, "int8_act", N=N))
        sb = host(qmm.block_sums(wq, dev(x), wtype, N=N))
        for m in range(8):
            y1 = host(qmm.matmul(wq, dev(x[m:m + 1]), wtype, "int8_act", N=N))
            s1 = host(qmm.block_sums(wq, dev(x[m:m + 1]), wtype, N=N))
            assert np.array_equal(s1[0], sb[m])
            assert np.all(np.abs(y1[0].astype(np.float64) - yb[m]) <= 1e-5 * T[m] + 1e-6)


def test_one_hot_f32_act_is_exact(qmm, orc):
    """x = e_k: the Metal form returns column k of the dequantized weights."""
    for wtype, K in (("q8_0", 576), ("q4_k", 1536), ("q6_k", 1536)):
        wq = orc.quantize(wtype, qmm_synth.weights(64, K))
        W = orc.dequantize(wtype, wq, K)
        x = np.zeros((4, K), np.float32)
        for i, k in enumerate((0, 33, K // 2, K - 1)):
            x[i, k] = 1.0
        y = host(qmm.matmul(dev(wq), dev(x), wtype, "f32_act", N=64))
        for i, k in enumerate((0, 33, K // 2, K - 1)):
            assert np.array_equal(y[i], W[:, k])


@pytest.mark.parametrize("wtype,M,N,K", [("q8_0", 64, 300, 4096), ("q4_k", 37, 256, 2048), ("q5_0", 16, 96, 576),
                                         ("q6_k", 8, 100, 1536)])
def test_dequantize_all_form_matches_f32_act(qmm, orc, wtype, M, N, K):
    """The dequantize-all serving form (the weights dequantized once by the
    library, then a dense f32 GEMM with TF32 off) has the f32_act definition:
    it lies within the same bound of the oracle's f32_act output."""
    w = qmm_synth.weights(N, K, seed=N + 3 * K)
    x = qmm_synth.activations(M, K, seed=M + 5, outlier_channels=4)
    wq = orc.quantize(wtype, w)
    W = qmm.dequantize(dev(wq), wtype, K)
    assert np.array_equal(host(W), orc.dequantize(wtype, wq, K))
    tf32 = torch.backends.cuda.matmul.allow_tf32
    torch.backends.cuda.matmul.allow_tf32 = False
    try:
        y = host(torch.matmul(dev(x), W.t()))
    finally:
        torch.backends.cuda.matmul.allow_tf32 = tf32
    y_orc, T = orc.matmul(wtype, "f32_act", wq, x)
    assert_within_bound(y, y_orc, T, f"dequantize-all {wtype} M{M} N{N} K{K}")


def test_launch_counts(qmm):
    """qmm_matmul_launches mirrors the dispatch (decode: optional activation
    preparation + decode kernel + optional K-split reduction)."""
    assert qmm.matmul_launches("q8_0", "int8_act", 1, 100, 8192) == 1     # per-thread GEMV
    assert qmm.matmul_launches("q8_0", "f32_act", 1, 100, 8192) == 1      # small: prepared in-kernel
    assert qmm.matmul_launches("q8_0", "f32_act", 1, 28672, 8192) == 1    # large, M <= 4: each CTA prepares its slice
    assert qmm.matmul_launches("q4_k", "f32_act", 4, 28672, 8192) == 2    # large, M > 2: preparing kernel first
    assert qmm.matmul_launches("q4_k", "int8_act", 2, 28672, 8192) == 1
    assert qmm.matmul_launches("q4_k", "int8_act", 8, 28672, 8192) == 2
    assert qmm.matmul_launches("q8_0", "f32_act", 8, 28672, 8192) == 3    # K split: reduction after
    assert qmm.matmul_launches("q8_0", "int8_act", 256, 4096, 4096) == 2  # exact prefill: activation codes + GEMM
    assert qmm.matmul_launches("q8_0", "f32_act", 256, 4096, 4096) == 2   # tcgen05: operand pieces + GEMM
    assert qmm.matmul_launches("q4_k", "int8_act", 256, 4096, 4096) == 2  # exact tcgen05: activation codes + GEMM
    assert qmm.matmul_launches("q4_k", "f32_act", 64, 4096, 4096) == 2    # code GEMM: activation pieces + GEMM
    assert qmm.matmul_launches("q6_k", "f32_act", 64, 4096, 4096) == 3    # code GEMM: pieces, repack, GEMM
    assert qmm.matmul_launches("q5_0", "int8_act", 64, 4096, 4096) == 2   # exact tcgen05: activation codes + GEMM
    assert qmm.matmul_launches("q6_k", "int8_act", 256, 4096, 4096) == 3  # exact tcgen05: codes, repack, GEMM
    assert qmm.matmul_launches("q6_k", "int8_act", 16, 4096, 4096) == 1   # up to 16 rows: the decode kernel
    assert qmm.matmul_launches("q8_0", "int8_act", 1, 100, 100) == 0      # K not a multiple of 32
    assert qmm.matmul_launches("q5_0", "int8_act", 1, 576, 576) == 1      # Q4_0 / Q5_0 decode: the MMA kernel
    assert qmm.matmul_launches("q4_0", "f32_act", 8, 28672, 8192) == 3    # large: preparing kernel, K split
    assert qmm.matmul_launches("q4_0", "f32_act", 64, 4096, 4096) == 2     # prefill, K % 256 = 0: tcgen05
    assert qmm.matmul_launches("q5_0", "int8_act", 64, 576, 576) == 1     # K = 576: the streaming kernel
    assert qmm.matmul_launches("q6_k", "int8_act", 1, 576, 1536) == 1     # Q6_K decode: the MMA kernel
    assert qmm.matmul_launches("q6_k", "f32_act", 256, 4096, 4096) == 2   # Q6_K prefill: tcgen05 (repack + GEMM)
    assert qmm.matmul_launches("q5_0", "f32_act", 256, 576, 576) == 1     # K % 256 != 0: the streaming kernel


CHAIN_SHAPES = {"q8_0": [(8192, 8192), (576, 8192), (8192, 576), (8192, 8192)],
                "q4_k": [(8192, 8192), (512, 8192), (8192, 512), (8192, 8192)]}
PREFILL_CHAIN_SHAPES = [(1024, 1024), (768, 1024), (1024, 768), (1024, 1024)]


def run_chain(qmm, orc, wtype, mode, M, shapes):
    """Each call's x is the previous call's y, with no host synchronisation
    between calls and one workspace shared by all of them.  Grids are launched
    programmatically and read weights before the previous grid has finished;
    every output must still be the oracle's product of the weights with the
    previous (complete) output.  The outputs start as NaN, so a read of an
    unfinished output shows; so does a workspace overwritten too early."""
    shapes = shapes * 2
    wqs = {}
    for N, K in set(shapes):
        wqs[(N, K)] = orc.quantize(wtype, qmm_synth.weights(N, K, seed=N + 3 * K) * np.float32(50.0 / np.sqrt(K)))
    wq_dev = {k: dev(v) for k, v in wqs.items()}
    x0 = dev(qmm_synth.activations(M, shapes[0][1], seed=5))
    ys = [torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda") for N, _ in shapes]
    ws = torch.empty(max(max(qmm.matmul_workspace(wtype, mode, M, N, K) for N, K in shapes), 16), dtype=torch.uint8,
                     device="cuda")
    launches = [qmm.matmul_launches(wtype, mode, M, N, K) for N, K in shapes]
    torch.cuda.synchronize()
    x = x0
    for (N, K), y in zip(shapes, ys):
        qmm.matmul(wq_dev[(N, K)], x, wtype, mode, N=N, out=y, workspace=ws)
        x = y
    outs = [host(y) for y in ys]
    xin = host(x0)
    for i, ((N, K), y) in enumerate(zip(shapes, outs)):
        y_orc, T = orc.matmul(wtype, mode, wqs[(N, K)], xin)
        assert_within_bound(y, y_orc, T, f"{wtype} {mode} M{M} call {i} N{N} K{K}")
        xin = y
    check_device_error(qmm)
    return launches


@pytest.mark.parametrize("M", [1, 5])
@pytest.mark.parametrize("mode", ["int8_act", "f32_act"])
@pytest.mark.parametrize("wtype", ["q8_0", "q4_k"])
def test_chained_calls_wait_for_the_previous_output(qmm, orc, wtype, mode, M):
    launches = run_chain(qmm, orc, wtype, mode, M, CHAIN_SHAPES[wtype])
    if M > 4:  # the 8192 x 8192 calls prepare their activations in a launch of their own
        assert max(launches) >= 2


@pytest.mark.parametrize("M", [37, 300])
@pytest.mark.parametrize("mode", ["int8_act", "f32_act"])
@pytest.mark.parametrize("wtype", ["q8_0", "q4_k"])
def test_chained_prefill_calls_wait_for_the_previous_output(qmm, orc, wtype, mode, M):
    """The same chain on the prefill kernels: the tcgen05 GEMM (f32_act),
    whose preparing grid reads the weights' row scales before the previous
    GEMM has finished, the exact Q8_0 prefill GEMM and the streaming kernel
    (int8_act)."""
    launches = run_chain(qmm, orc, wtype, mode, M, PREFILL_CHAIN_SHAPES)
    # operand preparation + GEMM, except the single-launch streaming kernel (Q4_K int8_act)
    assert min(launches) == 2


def test_error_statuses_on_device(qmm, orc):
    wq = dev(orc.quantize("q8_0", qmm_synth.weights(100, 8192)))
    x = dev(qmm_synth.activations(8, 8192))
    need = qmm.matmul_workspace("q8_0", "f32_act", 8, 100, 8192)
    assert need > 0
    small = torch.empty(need - 16, dtype=torch.uint8, device="cuda")
    with pytest.raises(qmm.QmmError) as e:
        qmm.matmul(wq, x, "q8_0", "f32_act", N=100, workspace=small)
    assert e.value.status == 5
    assert qmm.matmul_workspace("q8_0", "int8_act", 8, 100, 8192) == 0
    # a workspace reused across calls needs no clearing by the caller
    ws = torch.empty(need, dtype=torch.uint8, device="cuda").fill_(0xAB)
    y1 = host(qmm.matmul(wq, x, "q8_0", "f32_act", N=100, workspace=ws))
    y2 = host(qmm.matmul(wq, x, "q8_0", "f32_act", N=100, workspace=ws))
    assert np.array_equal(y1, y2)
    check_device_error(qmm)


# ---------------------------------------------------------------------------
# full-size workloads, in the launch configuration the benchmark times:
# every output element against the oracle (run on all host cores)
# ---------------------------------------------------------------------------

FULL = [("q4_k", 28672, 8192, 8), ("q8_0", 28672, 8192, 8), ("q6_k", 28672, 8192, 8),  # decode kernel
        ("q8_0", 28672, 8192, 1),                                                       # dp4a GEMV (int8_act)
        ("q4_k", 28672, 8192, 1),
        ("q8_0", 14336, 4096, 1024), ("q4_k", 14336, 4096, 1024),                       # tcgen05 GEMM
        ("q8_0", 14336, 4096, 256), ("q4_k", 4096, 4096, 256), ("q5_0", 14336, 4096, 256),
        ("q4_k", 14336, 4096, 37), ("q8_0", 14336, 4096, 64),
        ("q6_k", 14336, 4096, 256), ("q6_k", 4096, 4096, 1024),                        # tcgen05, Q6_K repacked
        ("q6_k", 14336, 4096, 37),                                                      # exact / code GEMM, 64-row tiles
        ("q5_0", 49152, 576, 64),                                                       # streaming kernel (K % 256 != 0)
        ("q8_0", 4096, 4096, 16), ("q8_0", 49152, 576, 1), ("q5_0", 49152, 576, 1)]


@pytest.mark.slow
@pytest.mark.parametrize("wtype,N,K,M", FULL)
def test_full_size_full_outputs(qmm, orc, wtype, N, K, M):
    g = torch.Generator(device="cuda").manual_seed(0)
    w = torch.randn((N, K), generator=g, device="cuda") * 0.02
    wq = qmm.quantize_weights(w, wtype)
    del w
    x_np = qmm_synth.activations(M, K, outlier_channels=4 if M >= 16 else 0)
    x = dev(x_np)
    wq_h = host(wq)
    for mode in ("int8_act", "f32_act"):
        y = matmul_checked(qmm, wq, x, wtype, mode, N)
        y_orc, T = orc.matmul(wtype, mode, wq_h, x_np)
        assert_within_bound(y, y_orc, T, f"{wtype} {mode} N{N} K{K} M{M}")
    check_device_error(qmm)


@pytest.mark.parametrize("M", [1, 16])
def test_weights_beyond_2gb_use_64_bit_offsets(qmm, orc, M):
    """A Q8_0 weight buffer of 262144 x 8192 (2.28 GB > 2^31 bytes): decode and
    prefill outputs for rows near the end of the buffer match the oracle, so
    no byte offset wraps in 32 bits."""
    N, K = 262144, 8192
    g = torch.Generator(device="cuda").manual_seed(1)
    wq = torch.empty((N, qmm.row_bytes("q8_0", K)), dtype=torch.uint8, device="cuda")
    for r0 in range(0, N, 32768):  # quantize in slices (8 GB of f32 weights at once is not needed)
        w = torch.randn((32768, K), generator=g, device="cuda") * 0.02
        wq[r0:r0 + 32768] = qmm.quantize_weights(w, "q8_0")
        del w
    assert wq.numel() > 2 ** 31
    x_np = qmm_synth.activations(M, K, outlier_channels=4 if M >= 16 else 0)
    rows = np.unique(np.concatenate([np.arange(4), np.random.default_rng(3).choice(N, 12, replace=False),
                                     np.arange(N - 20, N)]))
    wq_rows = wq[torch.from_numpy(rows).cuda()].cpu().numpy()
    for mode in ("int8_act", "f32_act"):
        y = host(qmm.matmul(wq, dev(x_np), "q8_0", mode, N=N))
        y_orc, T = orc.matmul("q8_0", mode, wq_rows, x_np)
        assert_within_bound(y[:, rows], y_orc, T, f"q8_0 {mode} N{N} K{K} M{M}")
    del wq
    torch.cuda.empty_cache()
    check_device_error(qmm)


@pytest.mark.parametrize("wtype", ["q8_0", "q4_0", "q5_0", "q4_k", "q6_k"])
@pytest.mark.parametrize("mode", ["int8_act", "f32_act"])
def test_matmul_batch_items_within_bound(qmm, orc, wtype, mode):
    """qmm_matmul_batch: items of different N, K and M (<= 8), some sharing
    one x, each within the bound of its own oracle product."""
    if wtype in ("q4_k", "q6_k"):
        shapes = [(1, 576, 1536), (1, 192, 512), (1, 1536, 256), (1, 576, 14336), (4, 100, 2048), (8, 33, 256),
                  (2, 4097, 256), (3, 1, 768), (1, 576, 1536), (2, 300, 8192)]
    else:
        shapes = [(1, 576, 576), (1, 192, 576), (1, 1536, 576), (1, 576, 1536), (4, 100, 2048), (8, 33, 64),
                  (2, 4097, 256), (3, 1, 32), (1, 576, 576)]
    items, ref = [], []
    xs = {}
    for i, (M, N, K) in enumerate(shapes):
        w = qmm_synth.weights(N, K, seed=40 + i)
        wq = orc.quantize(wtype, w)
        if (M, K) not in xs:                 # items with the same (M, K) share x
            xs[(M, K)] = qmm_synth.activations(M, K, seed=60 + i)
        x = xs[(M, K)]
        items.append((dev(wq), dev(x), torch.full((M, N), float("nan"), device="cuda")))
        ref.append(orc.matmul(wtype, mode, wq, x))
    qmm.matmul_batch(items, wtype, mode)
    for (wq, x, y), (y_orc, T), s in zip(items, ref, shapes):
        assert_within_bound(host(y), y_orc, T, f"batch {wtype} {mode} {s}")
    check_device_error(qmm)


@pytest.mark.parametrize("mode", ["int8_act", "f32_act"])
def test_matmul_batch_many_items_empty_items_and_largest_rows(qmm, orc, mode):
    """More items than one launch takes (300: two launches of <= 256), empty
    items (M = 0 or N = 0) among them, and items at the largest M x K
    (8 x 2048 and 1 x 16384, where f32_act fits only two ring slots)."""
    shapes = []
    for i in range(300):
        shapes.append([(1, 3 + i % 7, 32 * (1 + i % 5)), (0, 8, 64), (2, 0, 64)][0 if i % 50 else 1 + (i // 50) % 2])
    shapes[17] = (8, 40, 2048)
    shapes[260] = (1, 50, 16384)
    items, ref = [], []
    for i, (M, N, K) in enumerate(shapes):
        w = qmm_synth.weights(max(N, 1), K, seed=300 + i)[:N]
        x = qmm_synth.activations(M, K, seed=700 + i) if M else np.zeros((0, K), np.float32)
        wq = orc.quantize("q8_0", w) if N else np.zeros((0, K // 32 * 34), np.uint8)
        y = torch.full((M, N), float("nan"), device="cuda")
        items.append((dev(wq) if N else torch.empty(16, dtype=torch.uint8, device="cuda"),
                      dev(x) if M else torch.empty((0, K), device="cuda"), y))
        ref.append(orc.matmul("q8_0", mode, wq, x) if M and N else None)
    qmm.matmul_batch(items, "q8_0", mode)
    for (_, _, y), r, sh in zip(items, ref, shapes):
        if r is not None:
            assert_within_bound(host(y), r[0], r[1], f"batch item {sh}")
    check_device_error(qmm)


def test_matmul_batch_smollm2_step_matches_single_calls(qmm, orc):
    """The 211 linears of the SmolLM2-135M-shaped decode step in one batch:
    every output element of every item against the oracle (outputs NaN-filled
    before each form, so an unwritten row fails)."""
    lins = qmm_synth.smollm2_linears()
    xs = {K: dev(qmm_synth.activations(1, K, seed=K)) for K in (576, 1536)}
    items = []
    for i, (_, N, K) in enumerate(lins):
        g = torch.Generator(device="cuda").manual_seed(1000 + i)
        w = torch.randn((N, K), generator=g, device="cuda") * 0.02
        items.append((qmm.quantize_weights(w, "q8_0"), xs[K], torch.full((1, N), float("nan"), device="cuda")))
    hosts = [(host(wq), host(x)) for wq, x, _ in items]
    for mode in ("int8_act", "f32_act"):
        for _, _, y in items:
            y.fill_(float("nan"))
        qmm.matmul_batch(items, "q8_0", mode)
        for i, ((wq_h, x_h), (_, _, y)) in enumerate(zip(hosts, items)):
            y_orc, T = orc.matmul("q8_0", mode, wq_h, x_h)
            assert_within_bound(host(y), y_orc, T, f"smollm2 item {i} {mode}")
    check_device_error(qmm)


def test_matmul_batch_typed_q4_k_m_step(qmm, orc):
    """The 211 linears of a SmolLM2-135M decode step with the weight types of
    its Q4_K_M file (Q5_0, Q8_0, Q4_K, Q6_K) in one qmm_matmul_batch_typed
    launch: every output element of every item against the oracle, both forms
    (outputs NaN-filled before each form, so an unwritten row fails)."""
    lins = qmm_synth.smollm2_q4_k_m_linears()
    xs = {K: qmm_synth.activations(1, K, seed=K) for K in (576, 1536)}
    xd = {K: dev(x) for K, x in xs.items()}
    items, hosts = [], []
    for i, (_, N, K, t) in enumerate(lins):
        g = torch.Generator(device="cuda").manual_seed(2000 + i)
        w = torch.randn((N, K), generator=g, device="cuda") * 0.02
        wq = qmm.quantize_weights(w, t)
        items.append((t, wq, xd[K], torch.full((1, N), float("nan"), device="cuda")))
        hosts.append(host(wq))
    for mode in ("int8_act", "f32_act"):
        for *_, y in items:
            y.fill_(float("nan"))
        qmm.matmul_batch_typed(items, mode)
        for i, ((t, _, x, y), wq_h) in enumerate(zip(items, hosts)):
            y_orc, T = orc.matmul(t, mode, wq_h, xs[x.shape[1]])
            assert_within_bound(host(y), y_orc, T, f"q4_k_m item {i} {t} {mode}")
    check_device_error(qmm)


@pytest.mark.parametrize("mode", ["int8_act", "f32_act"])
def test_matmul_batch_typed_mixed_items(qmm, orc, mode):
    """qmm_matmul_batch_typed with every weight type interleaved: items of
    M = 1..8 that share one x across types (the staged activations change
    form between Q8_0 and Q8K for the same x), adversarial rows, ragged N,
    guarded outputs; 300 items (two launches) with empty items among them."""
    types = ["q8_0", "q4_k", "q5_0", "q6_k", "q4_0"]
    xs = {}
    for M, K in ((1, 1536), (3, 512), (8, 2048), (2, 256), (1, 8192)):
        _, x = edge_operands("q8_0", K, M, n_plain=1, seed=M * 7 + K)
        xs[(M, K)] = x
    keys = list(xs)
    items, refs, guards = [], [], []
    for i in range(300):
        t = types[i % 5]
        M, K = keys[(i // 5 + i) % len(keys)]
        if i % 97 == 40:  # an empty item
            items.append((t, torch.empty(16, dtype=torch.uint8, device="cuda"), dev(xs[(M, K)]),
                          torch.empty((M, 0), device="cuda")))
            refs.append(None), guards.append(None)
            continue
        N = 5 + (i * 37) % 60
        w, _ = edge_operands(t, K, 1, n_plain=N, seed=500 + i)
        wq = orc.quantize(t, w)
        buf, y = guarded_out(M, w.shape[0])
        items.append((t, dev(wq), dev(xs[(M, K)]), y))
        refs.append(orc.matmul(t, mode, wq, xs[(M, K)]))
        guards.append(buf)
    qmm.matmul_batch_typed(items, mode)
    for (t, _, x, y), r, buf in zip(items, refs, guards):
        if r is None:
            continue
        assert_within_bound(host(y), r[0], r[1], f"typed batch {t} {mode} M{x.shape[0]} K{x.shape[1]}")
        check_guards(buf, "typed batch item")
    check_device_error(qmm)


SB_CANCEL = [(t, M, K) for t in ("q4_k", "q6_k") for (M, K) in ((1, 512), (2, 512), (8, 512), (1, 4096),
                                                                 (4, 4096), (16, 512), (37, 4096), (256, 4096))]


@pytest.mark.parametrize("wtype,M,K", SB_CANCEL)
def test_int8_superblock_sums_are_whole(qmm, orc, wtype, M, K):
    """int8_act on super-blocks whose exact sum is 0 while its four 64-value
    pieces are large and unequal (tests/superblock_cancel.py): T = 0, so every
    output must be within 1e-6 of 0, which only whole int32 super-block sums
    reach (per-piece f32 terms leave residues near 0.5).  Decode, streaming
    and prefill paths through qmm_matmul, and the batch kernel for M <= 8."""
    import superblock_cancel as sc
    N = 70
    wq = sc.weights(wtype, N, K)
    x = sc.activations(M, K)
    y_orc, T = orc.matmul(wtype, "int8_act", wq, x)
    y = matmul_checked(qmm, dev(wq), dev(x), wtype, "int8_act", N)
    assert_within_bound(y, y_orc, T, f"{wtype} M{M} K{K} zero-sum super-blocks")
    if M <= 8 and M * K <= 16384:
        buf, yb = guarded_out(M, N)
        qmm.matmul_batch([(dev(wq), dev(x), yb)], wtype, "int8_act")
        assert_within_bound(host(yb), y_orc, T, f"batch {wtype} M{M} K{K} zero-sum super-blocks")
        check_guards(buf, "batch zero-sum item")
    check_device_error(qmm)
