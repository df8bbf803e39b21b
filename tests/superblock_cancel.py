"""Super-blocks whose int8_act sum is exactly zero while its parts are not.

The int8_act bound for Q4_K and Q6_K is 1e-5 * T + 1e-6 with T the sum of
|scaled super-block terms|.  These operands make every super-block's exact
integer sum (Q4_K: S_sc, with dmin = 0; Q6_K: S) zero, so T = 0 and the exact
result is 0, while the sum's four 64-value pieces are large and unequal: a
kernel that scales and converts the pieces to f32 one by one and then adds
them leaves a rounding residue of order 2^-24 * |piece| (about 0.5 here), far
above the 1e-6 the bound allows.  Only whole integer super-block sums pass.

Weights are written as raw GGUF super-blocks (the public layouts the oracle
decodes: Q4_K 144 bytes, Q6_K 210 bytes) with every code at its maximum
(Q4_K 15, Q6_K +31) and every scale at its maximum (Q4_K sc = 63, m = 0;
Q6_K sc = 127), d = f16(0.3 + 0.01 n) for row n.  Activations take, per
64-value piece of each super-block, the integer codes 127, 100, -113, -114
(sum 0) times a per-row factor 0.37 + 0.05 m, so that their Q8K codes are
exactly those integers.
"""
import numpy as np

PIECE_CODES = (127, 100, -113, -114)


def _q4_k_row(nsb: int, d: float) -> bytes:
    blk = bytearray(144)
    blk[0:2] = np.float16(d).tobytes()
    blk[2:4] = np.float16(0.0).tobytes()
    # 6-bit packing: sc_0..3 in bytes 0-3 (low 6 bits), m_0..3 in bytes 4-7;
    # sc_4..7 low 4 bits in bytes 8-11 (low nibble), high 2 bits in bits 6-7 of
    # bytes 0-3; m_4..7 likewise in the high nibbles of 8-11 and bytes 4-7
    blk[4:8] = bytes([63 | (3 << 6)] * 4)
    blk[8:12] = bytes([0] * 4)
    blk[12:16] = bytes([15] * 4)
    blk[16:144] = bytes([0xFF] * 128)
    return bytes(blk) * nsb


def _q6_k_row(nsb: int, d: float) -> bytes:
    blk = bytearray(210)
    blk[0:192] = bytes([0xFF] * 192)  # 6-bit fields 63: code +31
    blk[192:208] = np.array([127] * 16, dtype=np.int8).tobytes()
    blk[208:210] = np.float16(d).tobytes()
    return bytes(blk) * nsb


def weights(wtype: str, N: int, K: int) -> np.ndarray:
    nsb = K // 256
    row = _q4_k_row if wtype == "q4_k" else _q6_k_row
    return np.frombuffer(b"".join(row(nsb, 0.3 + 0.01 * n) for n in range(N)), dtype=np.uint8).reshape(N, -1).copy()


def activations(M: int, K: int) -> np.ndarray:
    codes = np.repeat(np.array(PIECE_CODES, dtype=np.float32), 64)  # one super-block
    codes = np.tile(codes, K // 256)
    return np.stack([codes * np.float32(0.37 + 0.05 * m) for m in range(M)]).astype(np.float32)


def weight_value(wtype: str, n: int) -> float:
    """Every dequantized weight of row n: f(d) * sc * code (- f(dmin) m = 0)."""
    d = float(np.float16(0.3 + 0.01 * n))
    return d * 63 * 15 if wtype == "q4_k" else d * 127 * 31
