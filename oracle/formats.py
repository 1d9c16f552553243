"""Exact decoding of the expert weight formats to float64 (oracle, test infrastructure).

The pages list the formats FreeToken serves (MXFP4, NVFP4, FP8, BF16: "FreeToken:
a 753B model on one GPU ...", closing section "Why this one matters") but fix no
bit layout; the layouts here are the standard definitions:

  bf16   : the upper 16 bits of an IEEE-754 binary32.
  e4m3   : OCP FP8 E4M3 ("fn"): 1 sign, 4 exponent (bias 7), 3 mantissa bits,
           no infinities, S.1111.111 is NaN, max finite 448, subnormals
           (exponent field 0) are m/8 * 2**-6.
  blockscale: value = e4m3(code) * scale[row // 128, col // 128].
  e2m1   : FP4 E2M1: 1 sign, 2 exponent (bias 1), 1 mantissa bit, no
           infinities or NaN; exponent field 0 is m/2, otherwise
           (1 + m/2) * 2**(e-1): magnitudes 0, 0.5, 1, 1.5, 2, 3, 4, 6.
  nvfp4  : value = e2m1(code) * e4m3(scale of its 16-element row block) * g of
           the matrix; two codes per byte, the even element in the low nibble.
  e8m0   : OCP Microscaling (MX) shared scale: an unsigned 8-bit biased
           exponent, value 2**(code - 127); code 255 is NaN.
  mxfp4  : OCP MX block of 32: value = e2m1(code) * e8m0(scale of its
           32-element row block); codes packed as in nvfp4, no matrix scale.

Nothing here rounds: every bf16 / e4m3 value is exactly representable in
float64.
"""
from __future__ import annotations

import numpy as np


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns (uint16) -> float64: the upper half of a binary32."""
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
    """OCP e4m3 ("fn") codes -> float64 through the 256-entry table above."""
    return E4M3_TABLE[np.asarray(codes, dtype=np.uint8)]


def _e2m1_value(code: int) -> float:
    s = -1.0 if code & 0x8 else 1.0
    e = (code >> 1) & 0x3
    m = code & 0x1
    if e == 0:
        return s * m / 2.0
    return s * (1.0 + m / 2.0) * 2.0 ** (e - 1)


E2M1_TABLE = np.array([_e2m1_value(c) for c in range(16)], dtype=np.float64)


def nvfp4_dequant(packed: np.ndarray, scales: np.ndarray, g: float) -> np.ndarray:
    """packed [R, C/2] (even element in the low nibble), scales [R, C/16] e4m3 codes,
    g fp32 -> float64 [R, C]."""
    packed = np.asarray(packed, dtype=np.uint8)
    R, C2 = packed.shape
    C = 2 * C2
    codes = np.empty((R, C), np.uint8)
    codes[:, 0::2] = packed & 0xF
    codes[:, 1::2] = packed >> 4
    assert scales.shape == (R, C // 16)
    s = e4m3_codes_to_f64(scales)
    return E2M1_TABLE[codes] * np.repeat(s, 16, axis=1) * float(np.float32(g))


def e8m0_codes_to_f64(codes: np.ndarray) -> np.ndarray:
    """OCP MX E8M0 scale codes -> float64: 2**(code - 127), NaN for code 255."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    return np.where(c == 255, np.nan, np.ldexp(1.0, c - 127))


def mxfp4_dequant(packed: np.ndarray, scales: np.ndarray) -> np.ndarray:
    """packed [R, C/2] (even element in the low nibble), scales [R, C/32] e8m0 codes
    -> float64 [R, C]."""
    packed = np.asarray(packed, dtype=np.uint8)
    R, C2 = packed.shape
    C = 2 * C2
    codes = np.empty((R, C), np.uint8)
    codes[:, 0::2] = packed & 0xF
    codes[:, 1::2] = packed >> 4
    assert scales.shape == (R, C // 32)
    return E2M1_TABLE[codes] * np.repeat(e8m0_codes_to_f64(scales), 32, axis=1)


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
    s_d [H/128, I/128] fp32 scales; nvfp4 blobs hold packed e2m1 codes, then
    per-16-element e4m3 row-block scales s_gu [2I, H/16] and s_d [H, I/16],
    then the two fp32 matrix scales (g_gu, g_d) and 8 bytes of padding; mxfp4
    blobs hold the same packed codes, then per-32-element e8m0 row-block scales
    s_gu [2I, H/32] and s_d [H, I/32].
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
    elif wdtype == "nvfp4":
        o = 0
        p_gu = blob[o:o + I * H].reshape(2 * I, H // 2); o += I * H
        p_d = blob[o:o + H * I // 2].reshape(H, I // 2); o += H * I // 2
        s_gu = blob[o:o + 2 * I * H // 16].reshape(2 * I, H // 16); o += 2 * I * H // 16
        s_d = blob[o:o + H * I // 16].reshape(H, I // 16); o += H * I // 16
        g = blob[o:o + 16].view(np.float32)
        w_gu = nvfp4_dequant(p_gu, s_gu, g[0])
        w_d = nvfp4_dequant(p_d, s_d, g[1])
    elif wdtype == "mxfp4":
        o = 0
        p_gu = blob[o:o + I * H].reshape(2 * I, H // 2); o += I * H
        p_d = blob[o:o + H * I // 2].reshape(H, I // 2); o += H * I // 2
        s_gu = blob[o:o + 2 * I * H // 32].reshape(2 * I, H // 32); o += 2 * I * H // 32
        s_d = blob[o:o + H * I // 32].reshape(H, I // 32)
        w_gu = mxfp4_dequant(p_gu, s_gu)
        w_d = mxfp4_dequant(p_d, s_d)
    else:
        raise ValueError(wdtype)
    return w_gu[:I], w_gu[I:], w_d


def activations_to_f64(x: np.ndarray, adtype: str) -> np.ndarray:
    """Activations as carried (float32, or bf16 bit patterns) -> float64."""
    if adtype == "f32":
        return np.asarray(x, dtype=np.float32).astype(np.float64)
    if adtype == "bf16":
        return bf16_bits_to_f64(x)
    raise ValueError(adtype)
