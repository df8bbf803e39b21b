"""Seeded synthetic inputs for the GGUF block-quantized matmul workloads.

This module is shared by the tests, the benchmark and the oracle's callers.
It holds none of the method's arithmetic (no quantization, no scales, no
products): it only draws f32 weights and activations with the shapes and value
distributions of the workloads, so that both the CUDA path and the CPU oracle
receive the same host buffers.

Distributions (the workloads name only "N(0, 0.02), 1% of columns x8" for
weights and "N(0, 1), 4 outlier channels x20" for prefill activations; this
is the plain reading of those phrases):
  * weights W [N, K] ~ N(0, 0.02^2) drawn in float64 and rounded to float32;
    round(0.01 * K) input columns (k indices), chosen by a seeded permutation,
    are multiplied by 8 ("1% of columns x8 outliers");
  * activations x [M, K] ~ N(0, 1); for prefill-shaped inputs 4 seeded
    channels (k indices) are multiplied by 20 in every row.
Seeds: weights 0, activations 1, outlier picks 2 unless a caller passes others;
the SmolLM2-shaped decode step offsets the weight seed by the matrix index.
"""
from __future__ import annotations

import numpy as np

HIDDEN = 576            # SmolLM2-135M hidden size
INTER = 1536            # SmolLM2-135M MLP size
KV = 192                # 3 KV heads x 64
VOCAB = 49152
LAYERS = 30


def _rng(seed: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(seed))


def outlier_columns(K: int, seed: int = 2, frac: float = 0.01) -> np.ndarray:
    n = int(round(frac * K))
    return np.sort(_rng(seed).permutation(K)[:n])


def weights(N: int, K: int, seed: int = 0, outliers: bool = True, outlier_seed: int = 2) -> np.ndarray:
    w = (_rng(seed).standard_normal((N, K)) * 0.02).astype(np.float32)
    if outliers:
        cols = outlier_columns(K, outlier_seed)
        w[:, cols] *= np.float32(8.0)
    return w


def activations(M: int, K: int, seed: int = 1, outlier_channels: int = 0, outlier_seed: int = 2) -> np.ndarray:
    x = _rng(seed).standard_normal((M, K)).astype(np.float32)
    if outlier_channels:
        ch = np.sort(_rng(outlier_seed + 1000).permutation(K)[:outlier_channels])
        x[:, ch] *= np.float32(20.0)
    return x


def smollm2_linears():
    """(name, N, K) of the 211 linears of one SmolLM2-135M decode step:
    30 layers x {q, k, v, o, gate, up, down} plus the tied lm_head."""
    out = []
    for layer in range(LAYERS):
        out += [(f"blk.{layer}.attn_q", HIDDEN, HIDDEN), (f"blk.{layer}.attn_k", KV, HIDDEN),
                (f"blk.{layer}.attn_v", KV, HIDDEN), (f"blk.{layer}.attn_output", HIDDEN, HIDDEN),
                (f"blk.{layer}.ffn_gate", INTER, HIDDEN), (f"blk.{layer}.ffn_up", INTER, HIDDEN),
                (f"blk.{layer}.ffn_down", HIDDEN, INTER)]
    out.append(("lm_head", VOCAB, HIDDEN))
    return out


def smollm2_q4_k_m_linears():
    """(name, N, K, wtype) of the same 211 linears with the weight types of a
    Q4_K_M file of this model, as the "GGUF 文件" page lists that file's
    tensors: a row of 576 values cannot hold 256-value super-blocks, so those
    matrices are Q5_0, except attn_v in 14 of the 30 layers (Q8_0); ffn_down
    (rows of 1536) is Q6_K in 14 layers and Q4_K in the other 16; the tied
    output head is the Q8_0 token embedding.  The page does not say which 14
    layers: the even layers 0, 2, ..., 26 here (the step's types, shapes and
    bytes do not depend on the choice)."""
    out = []
    for name, N, K in smollm2_linears():
        if name == "lm_head":
            t = "q8_0"
        else:
            layer = int(name.split(".")[1])
            more = layer % 2 == 0 and layer < 28
            t = ("q6_k" if more else "q4_k") if name.endswith("ffn_down") else \
                ("q8_0" if more else "q5_0") if name.endswith("attn_v") else "q5_0"
        out.append((name, N, K, t))
    return out


def special_block_rows(K: int, seed: int = 7) -> np.ndarray:
    """A small set of adversarial rows used by edge-case tests: zeros, constants,
    one-hot values, ties at +-0.5 code steps, all-negative and all-positive
    blocks, tiny and huge magnitudes, +-127 and random integer blocks, and
    values near the bottom of the f32 range (normal and subnormal, where the
    f32 reciprocal of a block scale overflows) mixed with zeros."""
    r = _rng(seed)
    rows = [np.zeros(K), np.full(K, 0.75), np.full(K, -3.0)]
    oh = np.zeros(K); oh[r.integers(K)] = 1.5; rows.append(oh)
    # values (k + 0.5) * amax / 127: rounding ties (up to the reciprocal's rounding)
    t = np.tile(np.arange(-63.5, 64.5, 1.0), K // 128 + 1)[:K] / 127.0
    t[::32] = 1.0
    rows.append(t)
    rows.append(-np.abs(r.standard_normal(K)) - 0.1)
    rows.append(np.abs(r.standard_normal(K)) + 0.1)
    rows.append(r.standard_normal(K) * 1e-6)
    rows.append(r.standard_normal(K) * 1e-9)
    rows.append(r.standard_normal(K) * 3e3)
    rows.append(np.where(r.random(K) < 0.5, -127.0, 127.0))
    ints = r.integers(-127, 128, K).astype(np.float64)
    ints[::32] = 127.0
    rows.append(ints)
    rows.append(r.standard_normal(K) * 1e-30)
    rows.append(np.where(r.random(K) < 0.5, 0.0, r.standard_normal(K) * 1e-38))
    return np.asarray(rows, dtype=np.float32)
