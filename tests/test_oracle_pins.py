"""Pins of the CPU oracle against facts that the pages or mathematics fix.

Nothing here calls the CUDA library.  Each test names the fact it checks and
the kind of mistake it catches.
"""
import json
import os

import numpy as np
import pytest

import qmm_synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ---------------------------------------------------------------------------
# An independent Python reading of the block layouts (written from the field
# description, not from the C oracle): used to cross-check unpacking.
# ---------------------------------------------------------------------------

def py_f16(bits):
    return np.asarray(bits, dtype=np.uint16).view(np.float16).astype(np.float32)


def py_decode_q8_0(row: np.ndarray, K: int):
    blocks = row.reshape(K // 32, 34)
    d = py_f16(blocks[:, 0].astype(np.uint16) | (blocks[:, 1].astype(np.uint16) << 8))
    q = blocks[:, 2:].view(np.int8).astype(np.int64)
    return d, q


def py_decode_q8_k(row: np.ndarray, K: int):
    blocks = row.reshape(K // 256, 292)
    d = blocks[:, 0:4].copy().view(np.float32).ravel()
    q = blocks[:, 4:260].view(np.int8).astype(np.int64)
    bs = blocks[:, 260:292].copy().view(np.int16).astype(np.int64)
    return d, q, bs


def py_decode_q4_k(row: np.ndarray, K: int):
    blocks = row.reshape(K // 256, 144)
    D = py_f16(blocks[:, 0].astype(np.uint16) | (blocks[:, 1].astype(np.uint16) << 8))
    Dm = py_f16(blocks[:, 2].astype(np.uint16) | (blocks[:, 3].astype(np.uint16) << 8))
    sc = np.zeros((K // 256, 8), np.int64)
    mn = np.zeros((K // 256, 8), np.int64)
    s = blocks[:, 4:16].astype(np.int64)
    for j in range(8):
        if j < 4:
            sc[:, j] = s[:, j] & 63
            mn[:, j] = s[:, j + 4] & 63
        else:
            sc[:, j] = (s[:, j + 4] & 0xF) | ((s[:, j - 4] >> 6) << 4)
            mn[:, j] = (s[:, j + 4] >> 4) | ((s[:, j] >> 6) << 4)
    qs = blocks[:, 16:].astype(np.int64)          # [nsb, 128]
    q = np.zeros((K // 256, 256), np.int64)
    for c in range(4):
        q[:, 64 * c: 64 * c + 32] = qs[:, 32 * c: 32 * c + 32] & 0xF
        q[:, 64 * c + 32: 64 * c + 64] = qs[:, 32 * c: 32 * c + 32] >> 4
    return D, Dm, sc, mn, q


def py_decode_q6_k(row: np.ndarray, K: int):
    """Q6_K super-block: ql[128] (low 4 bits), qh[64] (high 2 bits), 16 int8
    group scales, f16 d.  Value i: half h = i // 128, w = i % 128, quarter
    q = w // 32, l = w % 32; low bits = nibble q // 2 of ql[64h + 32 (q % 2)
    + l], high bits = bits 2q..2q+1 of qh[32h + l]; code = 6 bits - 32."""
    blocks = row.reshape(K // 256, 210)
    ql = blocks[:, 0:128].astype(np.int64)
    qh = blocks[:, 128:192].astype(np.int64)
    sc = blocks[:, 192:208].view(np.int8).astype(np.int64)
    D = py_f16(blocks[:, 208].astype(np.uint16) | (blocks[:, 209].astype(np.uint16) << 8))
    q = np.zeros((K // 256, 256), np.int64)
    for i in range(256):
        h, w = divmod(i, 128)
        qq, l = divmod(w, 32)
        lo = (ql[:, 64 * h + 32 * (qq % 2) + l] >> (4 * (qq // 2))) & 15
        hi = (qh[:, 32 * h + l] >> (2 * qq)) & 3
        q[:, i] = (lo | (hi << 4)) - 32
    return D, sc, q


# ---------------------------------------------------------------------------
# f16 conversion
# ---------------------------------------------------------------------------

@pytest.mark.slow
def test_f16_exhaustive_against_compiler_cast(orc):
    """All 2^32 f32 bit patterns: the oracle's hand-written f32->f16 (RNE with
    subnormals) equals the compiler's _Float16 conversion."""
    step = 1 << 28
    bad = sum(orc.f16_check_range(lo, lo + step) for lo in range(0, 1 << 32, step))
    assert bad == 0


def test_f16_against_numpy(orc):
    """A second independent reference: numpy's float16 conversion, on random
    bit patterns and on every half value (f16 -> f32 is exact)."""
    rng = np.random.default_rng(3)
    bits = rng.integers(0, 1 << 32, size=1 << 21, dtype=np.uint64).astype(np.uint32)
    x = bits.view(np.float32)
    finite = np.isfinite(x)
    with np.errstate(over="ignore"):
        ref = x[finite].astype(np.float16).view(np.uint16)
    got = orc.f32_to_f16_bits(x[finite])
    assert np.array_equal(got, ref)
    allh = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    f = orc.f16_bits_to_f32(allh)
    ref32 = allh.view(np.float16).astype(np.float32)
    assert (np.isnan(ref32) == np.isnan(f)).all()
    fin = ~np.isnan(ref32)
    assert np.array_equal(f[fin].view(np.uint32), ref32[fin].view(np.uint32))


# ---------------------------------------------------------------------------
# Sizes printed on the pages
# ---------------------------------------------------------------------------

def test_block_bytes_match_page_tensor_sizes(orc):
    """Per-tensor byte counts printed on the pages fix 34 B per 32 values
    (Q8_0), 144 B per 256 values (Q4K) and 22 B per 32 values (Q5_0)."""
    g = json.load(open(os.path.join(GOLDEN, "page_sizes.json")))
    for e in g["tensor_groups"]:
        N, K = e["shape"]
        assert e["tensors"] * N * orc.row_bytes(e["type"], K) == e["bytes"], e["what"]


def test_file_sizes_close_with_block_bytes(orc):
    """Whole-file sizes on the pages: every own file = header + 61 F32 norms
    + its matrices at the type's bytes per value, with ONE header size for all
    of them; Q8_0, Q4K, Q5_0 and Q4_0 bytes per value come from the oracle;
    Q6K at 210 B / 256 closes the downloaded Q4_K_M."""
    g = json.load(open(os.path.join(GOLDEN, "page_sizes.json")))
    files = {e["what"]: e["bytes"] for e in g["files"]}
    q5_bpv = orc.block_bytes("q5_0") / orc.block_values("q5_0")     # 22 / 32
    q8_bpv = orc.block_bytes("q8_0") / orc.block_values("q8_0")
    q4k_bpv = orc.block_bytes("q4_k") / orc.block_values("q4_k")
    lin = qmm_synth.smollm2_linears()[:-1]                            # 210 layer linears
    emb = qmm_synth.VOCAB * qmm_synth.HIDDEN                          # token_embd (lm_head is tied)
    norms = g["f32_norm_tensors"]["value"] * qmm_synth.HIDDEN * 4
    vals = sum(n * k for _, n, k in lin) + emb
    header = files["own F32 GGUF"] - norms - 4 * vals
    assert 0 < header < 65536
    assert header + norms + vals * q8_bpv == files["own Q8_0 GGUF"]
    assert header + norms + vals * orc.block_bytes("q4_0") / orc.block_values("q4_0") == files["own Q4_0 GGUF"]
    down = [(n, k) for name, n, k in lin if "ffn_down" in name]
    other = vals - sum(n * k for n, k in down)
    assert header + norms + sum(n * k for n, k in down) * q4k_bpv + other * q5_bpv == \
        files["own Q4K GGUF (ffn_down Q4K, other matrices Q5_0)"]
    meta = g["metadata_difference_bytes"]["value"]
    assert files["own Q8_0 GGUF"] + meta == files["downloaded Q8_0 GGUF"]
    # downloaded Q4_K_M: token_embd Q8_0; ffn_down 16 Q4K + 14 Q6K; attn_v 16 Q5_0 + 14 Q8_0; rest Q5_0
    size = header + meta + norms + emb * q8_bpv
    size += 16 * 576 * 1536 * q4k_bpv + 14 * 576 * 1536 * 210 / 256
    size += 16 * 192 * 576 * q5_bpv + 14 * 192 * 576 * q8_bpv
    rest = [(n, k) for name, n, k in lin if not ("ffn_down" in name or "attn_v" in name)]
    size += sum(n * k for n, k in rest) * q5_bpv
    assert size == files["downloaded Q4_K_M GGUF"]


def test_row_bytes_rejects_ragged_K(orc):
    """K-quants need K divisible by 256 (the Q4K shape error for 576-wide rows)."""
    with pytest.raises(ValueError):
        orc.row_bytes("q4_k", 576)
    assert orc.row_bytes("q8_0", 576) == 612


# ---------------------------------------------------------------------------
# Q8_0 / Q8K quantization
# ---------------------------------------------------------------------------

def test_q8_0_scale_rule_and_codes(orc):
    """Scale d = max|x|/127 (no freedom); the extreme value gets code +-127;
    every code is the nearest integer to x/d (up to the f32 reciprocal's
    rounding) and lies in [-127, 127]; an all-zero block has codes 0."""
    x = np.concatenate([qmm_synth.weights(64, 576), qmm_synth.special_block_rows(576)])
    q = orc.quantize("q8_0", x)
    for r in range(x.shape[0]):
        d16, codes = py_decode_q8_0(q[r], 576)
        blocks = x[r].reshape(-1, 32).astype(np.float32)
        amax = np.abs(blocks).max(axis=1)
        d = amax / np.float32(127.0)
        assert np.array_equal(d16.astype(np.float16).view(np.uint16), d.astype(np.float16).view(np.uint16))
        assert np.abs(codes).max() <= 127
        nz = amax > 0
        ext = np.abs(codes[nz][np.arange(nz.sum()), np.abs(blocks[nz]).argmax(axis=1)])
        assert (ext == 127).all()
        # blocks whose f32 reciprocal 1/d overflows (amax below ~3.7e-37) leave the
        # nearest-integer property: their codes are pinned by the overflow test below
        with np.errstate(divide="ignore", over="ignore"):
            fin = nz & np.isfinite(np.float32(1.0) / d)
        ratio = blocks[fin].astype(np.float64) / d[fin, None].astype(np.float64)
        assert (np.abs(codes[fin] - ratio) <= 0.5 + 1e-4).all()
        assert (codes[~nz] == 0).all()


def test_q8_0_requantize_is_idempotent(orc):
    """quantize(dequantize(q)) reproduces q byte for byte: the scale rule has
    no freedom, so re-quantizing already-quantized weights is a fixed point
    (the byte-identical own vs downloaded Q8_0 files)."""
    x = qmm_synth.weights(96, 1536)
    q = orc.quantize("q8_0", x)
    w = orc.dequantize("q8_0", q, 1536)
    assert np.array_equal(orc.quantize("q8_0", w), q)


def test_q8_k_fields(orc):
    """Q8K: f32 d = max|x|/127, int8 codes within +-0.5 of x/d, bsums equal
    the sums of 16 consecutive codes."""
    x = np.concatenate([qmm_synth.activations(8, 1536), qmm_synth.special_block_rows(1536)])
    q = orc.quantize("q8_k", x)
    for r in range(x.shape[0]):
        d, codes, bs = py_decode_q8_k(q[r], 1536)
        blocks = x[r].reshape(-1, 256)
        assert np.array_equal(d, np.abs(blocks).max(axis=1) / np.float32(127.0))
        assert np.array_equal(bs, codes.reshape(-1, 16, 16).sum(axis=2))
        ok = d > 0
        # where the f32 reciprocal 1/d overflows, codes leave the nearest-integer
        # property (pinned by the overflow test below)
        with np.errstate(divide="ignore", over="ignore"):
            fin = ok & np.isfinite(np.float32(1.0) / d)
        assert (np.abs(codes[fin] - blocks[fin].astype(np.float64) / d[fin, None]) <= 0.5 + 1e-4).all()
        assert (codes[~ok] == 0).all()


# ---------------------------------------------------------------------------
# Round-trip bounds
# ---------------------------------------------------------------------------

def test_round_trip_bounds(orc):
    """Per element |x - dequant(quant(x))|, with slack 2^-20 amax for the f32
    reciprocal and products:  Q8_0 <= d/2 + 127|d - f16(d)| + 2^-20 amax;
    Q8K <= d/2 + 2^-20 amax;  Q4_K interior points <= e_j/2 + 2^-20 (|x| +
    15 e_j); all Q4_K points <= e_j/2 + 7.97 d + 0.531 dmin + 2^-20 (hi -
    lo + |x|) in the normal f16 range (|sc d - s| <= d/2 and |f(D) - d| <=
    2^-11 d give |e - s| <= 0.531 d; the same for the offset); with the f16
    subnormal spacing the f16 error is max(2^-11 d, 2^-25)."""
    K = 1536
    x = np.concatenate([qmm_synth.weights(64, K), qmm_synth.special_block_rows(K)]).astype(np.float32)
    # Q8_0
    q = orc.quantize("q8_0", x)
    w = orc.dequantize("q8_0", q, K)
    b = x.reshape(-1, 32).astype(np.float64)
    amax = np.abs(b).max(axis=1, keepdims=True)
    d = amax / 127.0
    d16 = np.asarray([py_decode_q8_0(q[r], K)[0] for r in range(x.shape[0])]).reshape(-1, 1).astype(np.float64)
    bound = d / 2 + 127 * np.abs(d - d16) + 2.0 ** -20 * amax
    assert (np.abs(b - w.reshape(-1, 32)) <= bound).all()
    # Q8K
    q = orc.quantize("q8_k", x)
    w = orc.dequantize("q8_k", q, K)
    b = x.reshape(-1, 256).astype(np.float64)
    amax = np.abs(b).max(axis=1, keepdims=True)
    with np.errstate(divide="ignore", over="ignore"):  # blocks whose f32 1/d overflows: the overflow test
        fin = np.isfinite(np.float32(1.0) / (amax.astype(np.float32) / np.float32(127.0)))[:, 0]
    assert (np.abs(b - w.reshape(-1, 256))[fin] <= (amax / 254.0 + 2.0 ** -20 * amax)[fin]).all()
    # Q4_K
    q = orc.quantize("q4_k", x)
    w = orc.dequantize("q4_k", q, K).astype(np.float64)
    for r in range(x.shape[0]):
        D, Dm, sc, mn, codes = py_decode_q4_k(q[r], K)
        xs = x[r].reshape(-1, 8, 32).astype(np.float64)
        ws = w[r].reshape(-1, 8, 32)
        e = (D[:, None].astype(np.float64) * sc)[:, :, None]
        o = (Dm[:, None].astype(np.float64) * mn)[:, :, None]
        lo = np.minimum(0.0, xs.min(axis=2, keepdims=True))
        hi = xs.max(axis=2, keepdims=True)
        err = np.abs(xs - ws)
        interior = (xs + o >= 0) & (xs + o <= 15 * e) & (e > 0)
        ib = e / 2 + 2.0 ** -20 * (np.abs(xs) + 15 * e)
        assert (err[interior] <= ib[interior]).all()
        # super-block scales before f16 rounding; f16 error <= max(2^-11 d, 2^-25)
        d = ((hi - lo) / 15.0).max(axis=1, keepdims=True) / 63.0
        dmin = (-lo).max(axis=1, keepdims=True) / 63.0
        dD = np.maximum(2.0 ** -11 * d, 2.0 ** -25)
        dDm = np.maximum(2.0 ** -11 * dmin, 2.0 ** -25)
        allb = e / 2 + 15 * (d / 2 + 63 * dD) + dmin / 2 + 63 * dDm + 2.0 ** -20 * (hi - lo + np.abs(xs))
        assert (err <= allb).all()
        assert (sc >= 0).all() and (sc <= 63).all() and (mn >= 0).all() and (mn <= 63).all()


def test_q4_k_extreme_subblocks_use_full_scale(orc):
    """Closed form of the min/max reading: the sub-block with the largest step
    gets sc = 63 and the one with the largest offset gets m = 63."""
    x = qmm_synth.weights(32, 2048)
    q = orc.quantize("q4_k", x)
    for r in range(32):
        D, Dm, sc, mn, codes = py_decode_q4_k(q[r], 2048)
        assert (sc.max(axis=1) == 63).all()
        assert (mn.max(axis=1) == 63).all()


def test_q4_k_layout_decode_matches_python_reader(orc):
    """The oracle's Q4_K dequantization equals an independent Python reader
    of the same field layout: w = (f(d) sc) q - f(dmin) m."""
    K = 1024
    x = qmm_synth.weights(16, K)
    q = orc.quantize("q4_k", x)
    w = orc.dequantize("q4_k", q, K)
    for r in range(16):
        D, Dm, sc, mn, codes = py_decode_q4_k(q[r], K)
        e = (D[:, None] * sc.astype(np.float32)).astype(np.float32)
        o = (Dm[:, None] * mn.astype(np.float32)).astype(np.float32)
        ref = (e[:, :, None] * codes.reshape(-1, 8, 32).astype(np.float32)).astype(np.float32) - o[:, :, None]
        assert np.array_equal(ref.astype(np.float32).ravel(), w[r])


# ---------------------------------------------------------------------------
# Integer block sums: brute force on tiny inputs
# ---------------------------------------------------------------------------

def _brute_q8_0(wq, xq, M, N, K):
    out = np.zeros((M, N, K // 32), np.int64)
    for m in range(M):
        _, a = py_decode_q8_0(xq[m], K)
        for n in range(N):
            _, w = py_decode_q8_0(wq[n], K)
            for b in range(K // 32):
                out[m, n, b] = sum(int(w[b, i]) * int(a[b, i]) for i in range(32))
    return out


def _brute_q4_k(wq, xq, M, N, K):
    out = np.zeros((M, N, K // 256, 2), np.int64)
    for m in range(M):
        _, a, _ = py_decode_q8_k(xq[m], K)
        for n in range(N):
            _, _, sc, mn, q = py_decode_q4_k(wq[n], K)
            for s in range(K // 256):
                ssc = sm = 0
                for j in range(8):
                    isum = sum(int(q[s, 32 * j + i]) * int(a[s, 32 * j + i]) for i in range(32))
                    asum = sum(int(a[s, 32 * j + i]) for i in range(32))
                    ssc += int(sc[s, j]) * isum
                    sm += int(mn[s, j]) * asum
                out[m, n, s] = (ssc, sm)
    return out


@pytest.mark.parametrize("K", [256, 512])
def test_block_sums_equal_brute_force(orc, K):
    """Per-block integer sums equal Python-int brute force, including
    adversarial constant (all +-127) rows."""
    M, N = 3, 4
    w = qmm_synth.weights(N, K, seed=11)
    x = qmm_synth.activations(M, K, seed=12)
    w[0] = 1.0
    x[0] = 1.0
    w[1, ::2] = -5.0
    x[1] = -2.0
    wq8, xq8 = orc.quantize("q8_0", w), orc.quantize("q8_0", x)
    assert np.array_equal(orc.block_sums("q8_0", wq8, xq8, M, N, K), _brute_q8_0(wq8, xq8, M, N, K))
    wq4, xqk = orc.quantize("q4_k", w), orc.quantize("q8_k", x)
    assert np.array_equal(orc.block_sums("q4_k", wq4, xqk, M, N, K), _brute_q4_k(wq4, xqk, M, N, K))


def test_block_sums_extremes_stay_exact(orc):
    """All codes +-127 (Q8_0), and a Q4_K ramp whose codes span 0..15: the
    largest per-block sums are still exact integers."""
    K = 256
    w = np.full((2, K), 1.0, np.float32)
    w[1] = np.linspace(0.0, 1.0, K, dtype=np.float32)
    x = np.full((2, K), -1.0, np.float32)
    s = orc.block_sums("q8_0", orc.quantize("q8_0", w), orc.quantize("q8_0", x), 2, 2, K)
    assert (s[:, 0] == -32 * 127 * 127).all()
    wq4, xqk = orc.quantize("q4_k", w), orc.quantize("q8_k", x)
    assert np.array_equal(orc.block_sums("q4_k", wq4, xqk, 2, 2, K), _brute_q4_k(wq4, xqk, 2, 2, K))


# ---------------------------------------------------------------------------
# Matmul forms
# ---------------------------------------------------------------------------

def test_row_permutation_permutes_blocks(orc):
    """Blocks run along a row: permuting output rows (the q/k per-head
    permutation with 9 and 3 heads) permutes the quantized rows byte for byte
    and changes nothing else."""
    for n_head, N in ((9, 576), (3, 192)):
        w = qmm_synth.weights(N, 576, seed=5)
        perm = np.arange(N).reshape(n_head, 2, N // n_head // 2).transpose(0, 2, 1).reshape(N)
        assert np.array_equal(orc.quantize("q8_0", w[perm]), orc.quantize("q8_0", w)[perm])
    w = qmm_synth.weights(576, 1536, seed=5)
    perm = np.random.default_rng(0).permutation(576)
    assert np.array_equal(orc.quantize("q4_k", w[perm]), orc.quantize("q4_k", w)[perm])


@pytest.mark.parametrize("wtype,K", [("q8_0", 576), ("q4_k", 1536), ("q4_0", 576), ("q5_0", 576), ("q6_k", 1536)])
def test_activation_rows_are_independent(orc, wtype, K):
    """Activation quantization is per row: row m's result is the same alone
    and inside a batch of 8 (contrast: per-tensor dynamic quantization)."""
    wq = orc.quantize(wtype, qmm_synth.weights(64, K))
    x = qmm_synth.activations(8, K)
    x[5] *= 50.0
    yb, _ = orc.matmul(wtype, "int8_act", wq, x)
    for m in range(8):
        y1, _ = orc.matmul(wtype, "int8_act", wq, x[m:m + 1])
        assert np.array_equal(y1[0], yb[m])


@pytest.mark.parametrize("wtype,K", [("q8_0", 576), ("q4_k", 1536), ("q4_0", 576), ("q5_0", 576), ("q6_k", 1536)])
def test_one_hot_activation_selects_dequantized_column(orc, wtype, K):
    """f32_act with x = e_k equals column k of the dequantized weights
    exactly (the Metal form multiplies f32 activations by dequantized
    weights)."""
    wq = orc.quantize(wtype, qmm_synth.weights(48, K))
    W = orc.dequantize(wtype, wq, K)
    for k in (0, 31, K // 2 + 3, K - 1):
        x = np.zeros((1, K), np.float32)
        x[0, k] = 1.0
        y, T = orc.matmul(wtype, "f32_act", wq, x)
        assert np.array_equal(y[0], W[:, k].astype(np.float64))
        assert np.array_equal(T[0], np.abs(W[:, k]).astype(np.float64))


def test_f32_act_equals_dequantized_matmul(orc):
    """f32_act = x @ dequant(W)^T (the dequantize-all form), here against
    numpy's float64 matmul of the dequantized weights."""
    for wtype, K in (("q8_0", 576), ("q4_k", 512), ("q4_0", 576), ("q5_0", 576), ("q6_k", 512)):
        wq = orc.quantize(wtype, qmm_synth.weights(40, K))
        x = qmm_synth.activations(3, K)
        y, T = orc.matmul(wtype, "f32_act", wq, x)
        W = orc.dequantize(wtype, wq, K).astype(np.float64)
        ref = x.astype(np.float64) @ W.T
        assert np.allclose(y, ref, rtol=0, atol=1e-12 * np.abs(x).sum() * np.abs(W).max())
        assert np.allclose(T, np.abs(x.astype(np.float64)) @ np.abs(W).T, rtol=1e-12)


def test_exactly_representable_activations_make_the_forms_agree(orc):
    """When every activation block is integers with max |x| = 127, d_a = 1
    and the codes are x itself, so the CPU form equals the Metal form."""
    K = 576
    wq = orc.quantize("q8_0", qmm_synth.weights(64, K))
    r = np.random.default_rng(4)
    x = r.integers(-127, 128, (4, K)).astype(np.float32)
    x[:, ::32] = 127.0
    yi, _ = orc.matmul("q8_0", "int8_act", wq, x)
    yf, _ = orc.matmul("q8_0", "f32_act", wq, x)
    assert np.allclose(yi, yf, rtol=1e-13, atol=0)


def test_constant_row_closed_form(orc):
    """A constant row c: Q8_0 codes are all 127 sign(c), the dequantized
    value is f16(|c|/127) * 127 sign(c)."""
    for c in (0.75, -3.0, 1e-3):
        x = np.full((1, 64), c, np.float32)
        q = orc.quantize("q8_0", x)
        d, codes = py_decode_q8_0(q[0], 64)
        assert (codes == 127 * np.sign(c)).all()
        w = orc.dequantize("q8_0", q, 64)
        ref = np.float32(np.float16(np.float32(abs(c)) / np.float32(127.0))) * np.float32(127.0) * np.sign(c)
        assert (w == ref).all()


@pytest.mark.parametrize("wtype,K", [("q8_0", 576), ("q4_k", 1536), ("q5_0", 576), ("q6_k", 1536)])
def test_activation_quantization_error_has_the_predicted_size(orc, wtype, K):
    """The CPU form differs from the Metal form only by the activation
    rounding: each code moves x by a near-uniform error of width d_a, so the
    gap per output has variance sum_k w_k^2 d_a^2 / 12.  A wrong step (e.g.
    amax/255), a dropped block scale or a wrong block size breaks the ratio."""
    wq = orc.quantize(wtype, qmm_synth.weights(576, K))
    x = qmm_synth.activations(4, K)
    yi, _ = orc.matmul(wtype, "int8_act", wq, x)
    yf, _ = orc.matmul(wtype, "f32_act", wq, x)
    W = orc.dequantize(wtype, wq, K).astype(np.float64)
    bv = 256 if wtype in ("q4_k", "q6_k") else 32
    da = np.abs(x.reshape(4, -1, bv)).max(axis=2) / 127.0
    var = (W ** 2) @ (np.repeat(da, bv, axis=1) ** 2 / 12.0).T        # [N, M]
    z = (yi - yf) / np.sqrt(var.T)
    assert 0.85 < z.std() < 1.15
    assert abs(z.mean()) < 0.1


def test_tolerance_scale_bounds_the_output(orc):
    """T = sum of |scaled terms| >= |y| for both forms and all outputs."""
    for wtype, K in (("q8_0", 576), ("q4_k", 1536), ("q4_0", 576), ("q5_0", 576), ("q6_k", 1536)):
        wq = orc.quantize(wtype, qmm_synth.weights(64, K))
        x = qmm_synth.activations(2, K)
        for mode in ("int8_act", "f32_act"):
            y, T = orc.matmul(wtype, mode, wq, x)
            assert (np.abs(y) <= T * (1 + 1e-12)).all()


# ---------------------------------------------------------------------------
# Q6_K (weights paired with Q8K activations; the pages fix 210 bytes per 256
# values, not the quantizer or the layout: the signed-max reading per group of
# 16 is pinned here by its closed forms and bounds, the layout by the reader)
# ---------------------------------------------------------------------------

def test_q6_k_bytes_close_the_downloaded_file(orc):
    """210 B per 256 values: the size with which the downloaded Q4_K_M closes."""
    assert orc.block_bytes("q6_k") == 210 and orc.block_values("q6_k") == 256
    with pytest.raises(ValueError):
        orc.row_bytes("q6_k", 576)


def test_q6_k_layout_decode_matches_python_reader(orc):
    """The oracle's Q6_K dequantization equals the Python reader of the field
    layout: w = (f(d) sc_j) code, exact in f32."""
    K = 1024
    x = qmm_synth.weights(16, K, seed=21)
    x[3, :16] = np.linspace(-1.0, 1.0, 16, dtype=np.float32)  # one group through zero: codes -32 .. 31
    q = orc.quantize("q6_k", x)
    w = orc.dequantize("q6_k", q, K)
    for r in range(16):
        D, sc, codes = py_decode_q6_k(q[r], K)
        assert (codes >= -32).all() and (codes <= 31).all()
        e = (D[:, None].astype(np.float64) * sc)                      # [nsb, 16]
        ref = np.repeat(e, 16, axis=1) * codes
        assert np.array_equal(ref.ravel().astype(np.float32), w[r])
    _, _, codes = py_decode_q6_k(q[3], K)
    assert codes[0, :16].min() == -32 and codes[0, :16].max() == 31


def test_q6_k_scale_rule_closed_form(orc):
    """Signed-max reading: the group holding the super-block's largest |x|
    gets sc = -127 sign(m) (s_j = m / -32 is the largest step), and that
    element's code is -32; every |sc| <= 127."""
    K = 2048
    x = qmm_synth.weights(24, K, seed=22)
    q = orc.quantize("q6_k", x)
    for r in range(24):
        D, sc, codes = py_decode_q6_k(q[r], K)
        xs = x[r].reshape(-1, 256)
        for s in range(K // 256):
            i = int(np.argmax(np.abs(xs[s])))
            j = i // 16
            assert sc[s, j] == -127 * np.sign(xs[s, i])
            assert codes[s, i] == -32
        assert (np.abs(sc) <= 127).all()


def test_q6_k_round_trip_bound(orc):
    """Per element, with s_j = m_j / -32, d = max|s_j| / 127 and e_j = f(D) sc_j:
    points inside the grid err <= |e_j| / 2 (+ 2^-20 |x|); every point err <=
    32 |s_j - e_j| + |e_j|, and |s_j - e_j| <= d / 2 + 127 |d - f(D)|."""
    K = 1536
    x = qmm_synth.weights(32, K, seed=23)
    q = orc.quantize("q6_k", x)
    w = orc.dequantize("q6_k", q, K).astype(np.float64)
    for r in range(32):
        D, sc, codes = py_decode_q6_k(q[r], K)
        xs = x[r].reshape(-1, 16, 16).astype(np.float64)
        ws = w[r].reshape(-1, 16, 16)
        e = np.abs(D[:, None].astype(np.float64) * sc)[:, :, None]
        err = np.abs(xs - ws)
        inside = (np.abs(xs) <= 31.5 * e) & (e > 0)
        assert (err[inside] <= (e / 2 + 2.0 ** -20 * np.abs(xs))[inside]).all()
        d = np.abs(xs).max(axis=(1, 2), keepdims=True) / 32.0 / 127.0
        dD = np.maximum(2.0 ** -11 * d, 2.0 ** -25)
        allb = 32 * (d / 2 + 127 * dD) + e + 2.0 ** -20 * np.abs(xs).max(axis=2, keepdims=True)
        assert (err <= allb).all()


def _brute_q6_k(wq, xq, M, N, K):
    out = np.zeros((M, N, K // 256), np.int64)
    for m in range(M):
        _, a, _ = py_decode_q8_k(xq[m], K)
        for n in range(N):
            _, sc, q = py_decode_q6_k(wq[n], K)
            for s in range(K // 256):
                out[m, n, s] = sum(int(sc[s, j]) * sum(int(q[s, i]) * int(a[s, i]) for i in range(16 * j, 16 * j + 16))
                                   for j in range(16))
    return out


@pytest.mark.parametrize("K", [256, 512])
def test_q6_k_block_sums_equal_brute_force(orc, K):
    """S = sum_j sc_j sum_{i in group j} code_i a_i equals Python-int brute
    force, with constant and alternating-sign rows among the inputs."""
    M, N = 3, 4
    w = qmm_synth.weights(N, K, seed=24)
    x = qmm_synth.activations(M, K, seed=25)
    w[0] = 1.0
    x[0] = -1.0
    w[1, ::2] = -5.0
    wq, xq = orc.quantize("q6_k", w), orc.quantize("q8_k", x)
    assert np.array_equal(orc.block_sums("q6_k", wq, xq, M, N, K), _brute_q6_k(wq, xq, M, N, K))


def test_q6_k_int8_act_is_the_dequantized_dot(orc):
    """The CPU form equals the float64 dot of the dequantized weights and the
    dequantized Q8K activation rows: a dropped scale, a wrong group index or
    a wrong activation offset in the integer path breaks it."""
    K = 768
    wq = orc.quantize("q6_k", qmm_synth.weights(40, K, seed=26))
    x = qmm_synth.activations(3, K, seed=27)
    y, T = orc.matmul("q6_k", "int8_act", wq, x)
    W = orc.dequantize("q6_k", wq, K).astype(np.float64)  # exact in f32
    xq = orc.quantize("q8_k", x)
    Xq = np.zeros((3, K))
    for m in range(3):  # d_a q_a exactly, in float64 (it need not fit in f32)
        d, q, _ = py_decode_q8_k(xq[m], K)
        Xq[m] = (d[:, None].astype(np.float64) * q).ravel()
    ref = Xq @ W.T
    assert np.allclose(y, ref, rtol=0, atol=1e-12 * (np.abs(Xq) @ np.abs(W).T).max())
    assert (np.abs(y) <= T * (1 + 1e-12)).all()


# ---------------------------------------------------------------------------
# Q4_0 / Q5_0 (weights paired with Q8_0 activations; the pages fix their
# sizes, 18 and 22 bytes per 32 values, not the quantizer: the signed-max
# reading is pinned here by its closed forms and error bounds)
# ---------------------------------------------------------------------------

X0 = [("q4_0", 8), ("q5_0", 16)]


def _x0_scale_codes(orc, t, q, K):
    """f(d) from the block's first two bytes and the signed codes
    dequantized / f(d) (integers when f(d) != 0)."""
    rows = q.shape[0]
    bb = orc.block_bytes(t)
    blk = q.reshape(rows, K // 32, bb)
    fd = py_f16(blk[:, :, 0].astype(np.uint16) | (blk[:, :, 1].astype(np.uint16) << 8)).astype(np.float64)
    w = orc.dequantize(t, q, K).reshape(rows, K // 32, 32).astype(np.float64)
    with np.errstate(divide="ignore", invalid="ignore"):
        c = np.where(fd[:, :, None] != 0, w / fd[:, :, None], 0.0)
    return fd, c, w


@pytest.mark.parametrize("t,off", X0)
def test_x0_scale_rule_and_codes(orc, t, off):
    """The value of largest magnitude m sets d = m / -off and gets code -off;
    every code is an integer in [-off, off - 1] within 1/2 of x/d (the top
    code off - 1 also takes x/d in (off - 1, off]); an all-zero block
    dequantizes to zeros."""
    K = 576
    x = np.concatenate([qmm_synth.weights(64, K), qmm_synth.special_block_rows(K)]).astype(np.float32)
    q = orc.quantize(t, x)
    fd, c, w = _x0_scale_codes(orc, t, q, K)
    b = x.reshape(x.shape[0], -1, 32)
    amax = np.abs(b).max(axis=2)
    m = np.take_along_axis(b, np.abs(b).argmax(axis=2)[:, :, None], axis=2)[:, :, 0]
    d = (m / np.float32(-off)).astype(np.float32)
    assert np.array_equal(fd, py_f16(d.astype(np.float16).view(np.uint16)).astype(np.float64))
    nz = fd != 0
    assert np.array_equal(c[nz], np.round(c[nz]))
    assert (c[nz] >= -off).all() and (c[nz] <= off - 1).all()
    cext = np.take_along_axis(c, np.abs(b).argmax(axis=2)[:, :, None], axis=2)[:, :, 0]
    assert (cext[nz] == -off).all()
    with np.errstate(divide="ignore", invalid="ignore"):
        ratio = b.astype(np.float64) / d[:, :, None].astype(np.float64)
    inner = nz[:, :, None] & (ratio <= off - 1)
    assert (np.abs(c - ratio)[inner] <= 0.5 + 1e-4).all()
    assert (np.abs(c - ratio)[nz[:, :, None] & ~(ratio <= off - 1)] <= 1.0 + 1e-4).all()
    assert (w[amax == 0] == 0).all()


@pytest.mark.parametrize("t,off", X0)
def test_x0_round_trip_bound(orc, t, off):
    """|x - dequant(quant(x))| <= |d| + off |d - f16(d)| + 2^-20 amax per
    element (|d|/2 except for the top code), d = m / -off."""
    K = 1536
    x = np.concatenate([qmm_synth.weights(64, K), qmm_synth.special_block_rows(K)]).astype(np.float32)
    q = orc.quantize(t, x)
    fd, c, w = _x0_scale_codes(orc, t, q, K)
    b = x.reshape(x.shape[0], -1, 32).astype(np.float64)
    amax = np.abs(b).max(axis=2, keepdims=True)
    m = np.take_along_axis(b, np.abs(b).argmax(axis=2)[:, :, None], axis=2)
    d = m / -off
    bound = np.abs(d) + off * np.abs(d - fd[:, :, None]) + 2.0 ** -20 * amax
    assert (np.abs(b - w) <= bound).all()


@pytest.mark.parametrize("t,off", X0)
def test_x0_requantize_is_idempotent(orc, t, off):
    """Re-quantizing dequantized weights reproduces the bytes: the code -off
    element has the unique largest magnitude, so d is recovered exactly when
    f16(d) is a normal number (all blocks here)."""
    x = qmm_synth.weights(96, 1536)
    q = orc.quantize(t, x)
    fd, _, _ = _x0_scale_codes(orc, t, q, 1536)
    assert (np.abs(fd) >= 2.0 ** -14).all()
    assert np.array_equal(orc.quantize(t, orc.dequantize(t, q, 1536)), q)


@pytest.mark.parametrize("t,off", X0)
def test_x0_constant_row_closed_form(orc, t, off):
    """A constant row c: every code is -off and the dequantized value is
    -off f16(c / -off) (= c up to the f16 rounding of d)."""
    for cval in (0.75, -3.0, 1e-3):
        x = np.full((1, 64), cval, np.float32)
        q = orc.quantize(t, x)
        fd, c, w = _x0_scale_codes(orc, t, q, 64)
        assert (c == -off).all()
        ref = np.float32(np.float16(np.float32(cval) / np.float32(-off))) * np.float32(-off)
        assert (w.astype(np.float32) == ref).all()


@pytest.mark.parametrize("t,off", X0)
@pytest.mark.parametrize("K", [64, 576])
def test_x0_block_sums_equal_brute_force(orc, t, off, K):
    """Per-block integer sums with Q8_0 activations equal Python-int brute
    force over the signed weight codes (dequantized / f(d)) and the
    activation codes, including all-(-off) and all-(off - 1) rows."""
    M, N = 3, 4
    w = qmm_synth.weights(N, K, seed=21)
    x = qmm_synth.activations(M, K, seed=22)
    w[0] = 1.0                                 # all codes -off
    w[1, ::2], w[1, 1::2] = -1.0, 1.0          # codes off (clamped to off - 1) and -off
    x[0] = -1.0
    wq, xq = orc.quantize(t, w), orc.quantize("q8_0", x)
    fd, c, _ = _x0_scale_codes(orc, t, wq, K)
    ci = np.round(c).astype(np.int64)
    assert ci.min() == -off and ci.max() == off - 1
    a = np.stack([py_decode_q8_0(xq[m], K)[1] for m in range(M)]).astype(np.int64).reshape(M, K // 32, 32)
    ref = np.einsum("nbi,mbi->mnb", ci, a)
    assert np.array_equal(orc.block_sums(t, wq, xq, M, N, K), ref.astype(np.int32))


# ---------------------------------------------------------------------------
# The CPU form's float combine, pinned exactly: y equals the float64 dot of
# the exactly dequantized weight rows and activation rows, both read from
# the bytes by the Python readers above (not by the oracle's own unpacking)
# ---------------------------------------------------------------------------

def py_decode_x0(row: np.ndarray, K: int, t: str):
    """Q4_0 / Q5_0 block: f16 d, (Q5_0) a little-endian 32-bit word whose bit
    i is bit 4 of code i, then 16 bytes with code j in the low nibble of byte
    j and code j + 16 in the high nibble.  Returns f(d) and the signed codes
    (code - 8 for Q4_0, code - 16 for Q5_0)."""
    bb, off = (18, 8) if t == "q4_0" else (22, 16)
    blocks = row.reshape(K // 32, bb)
    d = py_f16(blocks[:, 0].astype(np.uint16) | (blocks[:, 1].astype(np.uint16) << 8))
    nib = blocks[:, bb - 16:].astype(np.int64)
    q = np.concatenate([nib & 0xF, nib >> 4], axis=1)
    if t == "q5_0":
        qh = (blocks[:, 2].astype(np.int64) | (blocks[:, 3].astype(np.int64) << 8)
              | (blocks[:, 4].astype(np.int64) << 16) | (blocks[:, 5].astype(np.int64) << 24))
        q |= ((qh[:, None] >> np.arange(32)[None, :]) & 1) << 4
    return d, q - off


def _py_dequant_f64(t: str, wq: np.ndarray, K: int) -> np.ndarray:
    """Dequantized weights in float64 from the Python readers: f(d) q for the
    32-value types, f(d) sc_j q - f(dmin) m_j for Q4_K (no f32 rounding
    anywhere: every product is exact in float64)."""
    out = np.zeros((wq.shape[0], K))
    for n in range(wq.shape[0]):
        if t == "q8_0":
            d, q = py_decode_q8_0(wq[n], K)
            out[n] = (d[:, None].astype(np.float64) * q).ravel()
        elif t in ("q4_0", "q5_0"):
            d, q = py_decode_x0(wq[n], K, t)
            out[n] = (d[:, None].astype(np.float64) * q).ravel()
        else:
            D, Dm, sc, mn, q = py_decode_q4_k(wq[n], K)
            e = D[:, None].astype(np.float64) * sc            # [nsb, 8]
            o = Dm[:, None].astype(np.float64) * mn
            out[n] = (np.repeat(e, 32, axis=1) * q - np.repeat(o, 32, axis=1)).ravel()
    return out


def _py_act_f64(atype: str, xq: np.ndarray, K: int) -> np.ndarray:
    """Dequantized activation rows d_a q_a in float64 (Q8_0: f16 d; Q8K: f32 d)."""
    out = np.zeros((xq.shape[0], K))
    for m in range(xq.shape[0]):
        if atype == "q8_0":
            d, q = py_decode_q8_0(xq[m], K)
        else:
            d, q, _ = py_decode_q8_k(xq[m], K)
        out[m] = (d[:, None].astype(np.float64) * q).ravel()
    return out


@pytest.mark.parametrize("wtype,K", [("q8_0", 576), ("q4_0", 576), ("q5_0", 576), ("q4_k", 1536),
                                     ("q8_0", 1536), ("q4_k", 512)])
def test_int8_act_is_the_dequantized_dot(orc, wtype, K):
    """The CPU form's float combine equals, to float64 rounding, the dot of
    the exactly dequantized weights with the exactly dequantized activation
    codes.  A misplaced scale, a dropped min term, a wrong sub-block index,
    or f(d) S rounded through f32 (a relative error near 6e-8) fails the
    1e-12 bound; adversarial rows are in both operands."""
    w = np.concatenate([qmm_synth.weights(40, K, seed=31), qmm_synth.special_block_rows(K)])
    x = np.concatenate([qmm_synth.activations(3, K, seed=32), qmm_synth.special_block_rows(K)[1:6]])
    wq = orc.quantize(wtype, w)
    atype = "q8_k" if wtype == "q4_k" else "q8_0"
    xq = orc.quantize(atype, x)
    y, T = orc.matmul(wtype, "int8_act", wq, x)
    W = _py_dequant_f64(wtype, wq, K)
    X = _py_act_f64(atype, xq, K)
    ref = X @ W.T
    scale = np.abs(X) @ np.abs(W).T
    assert np.all(np.abs(y - ref) <= 1e-12 * scale + 1e-300)
    # T is the sum of |scaled block terms|: at least |y|, and at most the sum of
    # |element products| (for Q4_K with the scale and min parts taken apart)
    assert (np.abs(y) <= T * (1 + 1e-12)).all()
    if wtype == "q4_k":
        parts = np.zeros_like(W)
        for n in range(wq.shape[0]):
            D, Dm, sc, mn, q = py_decode_q4_k(wq[n], K)
            e = np.repeat(D[:, None].astype(np.float64) * sc, 32, axis=1)
            o = np.repeat(Dm[:, None].astype(np.float64) * mn, 32, axis=1)
            parts[n] = (np.abs(e * q) + o).ravel()
        scale = np.abs(X) @ parts.T
    assert (T <= scale * (1 + 1e-12) + 1e-300).all()


@pytest.mark.parametrize("t", ["q4_0", "q5_0"])
def test_x0_layout_decode_matches_python_reader(orc, t):
    """The oracle's dequantization of Q4_0 / Q5_0 bytes equals the Python
    reader's f(d) (code - off): a swapped nibble order or a misread fifth
    bit fails."""
    K = 576
    w = np.concatenate([qmm_synth.weights(32, K, seed=33), qmm_synth.special_block_rows(K)])
    wq = orc.quantize(t, w)
    assert np.array_equal(orc.dequantize(t, wq, K).astype(np.float64), _py_dequant_f64(t, wq, K))


@pytest.mark.parametrize("t", ["q8_0", "q8_k", "q4_0", "q5_0"])
def test_zero_in_a_block_whose_reciprocal_overflows_gets_code_zero(orc, t):
    """Codes are round(x * (1/d)) with the f32 reciprocal.  For a block whose
    largest magnitude is near the bottom of the f32 range, 1/d overflows to
    infinity: nonzero values then take the extreme codes, and a zero value
    takes code 0 (x / d = 0), not the NaN of 0 * inf."""
    K = 256
    x = np.zeros((1, K), np.float32)
    x[0, 3], x[0, 5], x[0, 40] = 1e-38, -5e-39, 2e-39
    q = orc.quantize(t, x)
    if t == "q8_0":
        codes = np.concatenate([py_decode_q8_0(q[0], K)[1][b] for b in range(K // 32)])
        zero, pos, neg = 0, 127, -127
    elif t == "q8_k":
        codes = py_decode_q8_k(q[0], K)[1].ravel()
        zero, pos, neg = 0, 127, -127
    else:
        codes = py_decode_x0(q[0], K, t)[1].ravel()
        off = 8 if t == "q4_0" else 16
        # d = m / -off: the extreme value m = 1e-38 takes code -off, the opposite sign the top code
        zero, pos, neg = 0, -off, off - 1
    assert codes[3] == pos and codes[5] == neg
    nz = np.zeros(K, bool)
    nz[[3, 5, 40]] = True
    blk0 = np.arange(K) < 32
    assert (codes[~nz & blk0] == zero).all()


@pytest.mark.parametrize("wtype", ["q4_k", "q6_k"])
def test_superblock_cancellation_fixture(orc, wtype):
    """The zero-sum super-block operands (tests/superblock_cancel.py) decode as
    built: every weight f(d) sc code, every Q8K activation code one of the
    piece codes; the exact int8_act result is 0 with T = 0 (closed form: the
    piece codes sum to 0 and every weight of a row is the same), while each
    64-value piece's integer sum is not."""
    import superblock_cancel as sc
    N, M, K = 5, 3, 512
    wq = sc.weights(wtype, N, K)
    x = sc.activations(M, K)
    w = orc.dequantize(wtype, wq, K)
    for n in range(N):
        assert np.all(w[n] == np.float32(sc.weight_value(wtype, n)))
    xq = orc.quantize("q8_k", x).reshape(M, K // 256, 292)
    codes = xq[:, :, 4:260].view(np.int8).reshape(M, K).astype(np.int64)
    assert np.array_equal(codes, np.tile(np.repeat(np.array(sc.PIECE_CODES), 64), (M, K // 256)))
    y, T = orc.matmul(wtype, "int8_act", wq, x)
    assert np.all(y == 0.0) and np.all(T == 0.0)
    piece = codes.reshape(M, -1, 4, 64).sum(axis=-1)
    assert np.all(np.abs(piece) >= 100 * 64)
