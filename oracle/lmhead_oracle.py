"""fp64 CPU oracle of the online-FP8 output projection (LM head) GEMV.

TEST INFRASTRUCTURE ONLY. Only the tests and the benchmark's CPU-baseline leg
may import this module. The CUDA library never calls it, and this module
shares no code with the CUDA path.

What it computes: "Three ways to speed up MoE inference on DGX Spark", section
"Optimization 2": the bf16 output projection (hidden 2,560 -> vocabulary
157,184) is quantized to FP8 when the head is built, which halves the bytes the
per-token GEMV reads. Readings where the page is silent (the plainest reading
of a "dynamic FP8" head that halves the bf16 bytes): FP8 is OCP E4M3 (bias 7, no infinities, 0x7F / 0xFF NaN, largest finite
448); one fp32 scale per output row, s = amax(|row|) / 448 in fp32 (1 for an
all-zero row); codes q = RNE_E4M3(w / s) with the fp32 quotient and saturation
to +-448; activations stay bf16; logits[t, v] = s_v * sum_h e4m3(q[v, h]) * x[t, h].

Steps: decode_e4m3 (the format's definition), encode_e4m3 (nearest code, ties
to the even code, saturating), quantize_rows, forward (fp64, library matmul as
the dot product).
"""
from __future__ import annotations

import numpy as np

E4M3_MAX = 448.0


def decode_e4m3(codes) -> np.ndarray:
    """E4M3 byte -> value (fp64). Exponent field 0 is subnormal: m/8 * 2^-6."""
    c = np.asarray(codes, dtype=np.int64)
    s = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = (c & 0x7).astype(np.float64)
    mag = np.where(e == 0, m / 8.0 * 2.0 ** -6, (1.0 + m / 8.0) * np.exp2(e.astype(np.float64) - 7.0))
    mag = np.where((c & 0x7F) == 0x7F, np.nan, mag)
    return s * mag


def encode_e4m3(v) -> np.ndarray:
    """fp32 values -> E4M3 bytes, round to nearest with ties to the even code,
    magnitudes above 448 saturate to 448 (NaN -> 0x7F)."""
    x = np.asarray(v, dtype=np.float64)
    sign = np.where(np.signbit(x), 0x80, 0).astype(np.int64)
    a = np.abs(x)
    # quantum of the binade that holds a: 2^(e - 3) for normals (e >= -6), 2^-9 below
    with np.errstate(divide="ignore"):
        e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    e = np.maximum(e, -6.0)
    q = np.exp2(e - 3.0)
    n = np.round(a / q)          # numpy rounds halves to even: ties to the even multiple
    r = n * q                    # the rounded magnitude (may step into the next binade)
    r = np.minimum(r, E4M3_MAX)
    # back to a code: exponent and mantissa of r
    out = np.zeros(a.shape, dtype=np.int64)
    nz = r > 0
    er = np.floor(np.log2(np.where(nz, r, 1.0)))
    normal = nz & (er >= -6)
    mant_n = np.round(r / np.exp2(er) * 8.0 - 8.0).astype(np.int64)
    code_n = ((er.astype(np.int64) + 7) << 3) | mant_n
    code_s = np.round(r / 2.0 ** -9).astype(np.int64)      # subnormal: m = r / 2^-9
    out = np.where(normal, code_n, np.where(nz, code_s, 0))
    out = np.where(np.isnan(x), 0x7F, out | sign)
    return out.astype(np.uint8)


def bf16_bits_to_f64(bits) -> np.ndarray:
    return (np.asarray(bits, dtype=np.uint32) << 16).view(np.float32).astype(np.float64)


def quantize_rows(w_bits: np.ndarray):
    """bf16 W [V, H] -> (codes uint8 [V, H], scales float32 [V])."""
    w = (np.asarray(w_bits, dtype=np.uint32) << 16).view(np.float32)   # exact
    amax = np.abs(w).max(axis=1)
    scale = np.where(amax > 0, amax / np.float32(E4M3_MAX), np.float32(1.0)).astype(np.float32)
    quot = (w / scale[:, None]).astype(np.float32)                        # fp32 division
    return encode_e4m3(quot), scale


def forward(codes: np.ndarray, scales: np.ndarray, x_bits: np.ndarray) -> np.ndarray:
    """logits [T, V] (fp64) of the quantized head for bf16 rows x [T, H]."""
    wq = decode_e4m3(codes) * np.asarray(scales, dtype=np.float64)[:, None]
    return bf16_bits_to_f64(x_bits) @ wq.T
