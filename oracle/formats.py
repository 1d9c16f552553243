"""Exact decoding of the expert weight formats to float64 (oracle, test infrastructure).

The pages list the formats FreeToken serves (MXFP4, NVFP4, FP8, BF16: "FreeToken:
a 753B model on one GPU ...", closing section "Why this one matters") but fix no
bit layout; the layouts here are the standard definitions:

  bf16   : the upper 16 bits of an IEEE-754 binary32.
  e4m3   : OCP FP8 E4M3 ("fn"): 1 sign, 4 exponent (bias 7), 3 mantissa bits,
           no infinities, S.1111.111 is NaN, max finite 448, subnormals
           (exponent field 0) are m/8 * 2**-6.
  blockscale: value = e4m3(code) * scale[row // 128, col // 128].

Nothing here rounds: every bf16 / e4m3 value is exactly representable in
float64.
"""
from __future__ import annotations

import numpy as np


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    u = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return u.view(np.float32).astype(np.float64)


def _e4m3_value(code: int) -> float:
    s = -1.0 if code & 0x80 else 1.0
    e = (code >> 3) & 0xF
    m = code & 0x7
    if e == 0xF and m == 0x7:
        return float("nan")
    if e == 0:
        return s * (m / 8.0) * 2.0 ** -6
    return s * (1.0 + m / 8.0) * 2.0 ** (e - 7)


E4M3_TABLE = np.array([_e4m3_value(c) for c in range(256)], dtype=np.float64)


def e4m3_codes_to_f64(codes: np.ndarray) -> np.ndarray:
    return E4M3_TABLE[np.asarray(codes, dtype=np.uint8)]


def blockscale_dequant(codes: np.ndarray, scales: np.ndarray) -> np.ndarray:
    """codes [R, C] e4m3, scales [R/128, C/128] fp32 -> float64 [R, C]."""
    R, C = codes.shape
    assert scales.shape == (R // 128, C // 128)
    v = e4m3_codes_to_f64(codes)
    s = np.asarray(scales, dtype=np.float32).astype(np.float64)
    return v * np.repeat(np.repeat(s, 128, axis=0), 128, axis=1)


def parse_blob(blob: np.ndarray, wdtype: str, H: int, I: int):
    """Split one expert blob (bank layout) into float64 W_gate [I,H], W_up [I,H], W_down [H,I].

    Bank layout: W_gu [2I, H] row-major (gate rows first, then up rows), then
    W_down [H, I] row-major; fp8 blobs append s_gu [2I/128, H/128] and
    s_d [H/128, I/128] fp32 scales.
    """
    blob = np.asarray(blob, dtype=np.uint8)
    if wdtype == "f32":
        w = blob[: 12 * I * H].view(np.float32).astype(np.float64)
        w_gu = w[: 2 * I * H].reshape(2 * I, H)
        w_d = w[2 * I * H: 3 * I * H].reshape(H, I)
    elif wdtype == "bf16":
        w = bf16_bits_to_f64(blob[: 6 * I * H].view(np.uint16))
        w_gu = w[: 2 * I * H].reshape(2 * I, H)
        w_d = w[2 * I * H: 3 * I * H].reshape(H, I)
    elif wdtype == "fp8":
        n_gu = 2 * I * H
        n_d = H * I
        c_gu = blob[:n_gu].reshape(2 * I, H)
        c_d = blob[n_gu:n_gu + n_d].reshape(H, I)
        o = n_gu + n_d
        n_sgu = (2 * I // 128) * (H // 128)
        n_sd = (H // 128) * (I // 128)
        s_gu = blob[o:o + 4 * n_sgu].view(np.float32).reshape(2 * I // 128, H // 128)
        s_d = blob[o + 4 * n_sgu:o + 4 * (n_sgu + n_sd)].view(np.float32).reshape(H // 128, I // 128)
        w_gu = blockscale_dequant(c_gu, s_gu)
        w_d = blockscale_dequant(c_d, s_d)
    else:
        raise ValueError(wdtype)
    return w_gu[:I], w_gu[I:], w_d


def activations_to_f64(x: np.ndarray, adtype: str) -> np.ndarray:
    if adtype == "f32":
        return np.asarray(x, dtype=np.float32).astype(np.float64)
    if adtype == "bf16":
        return bf16_bits_to_f64(x)
    raise ValueError(adtype)
