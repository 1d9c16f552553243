"""Seeded synthetic inputs for the expert-slot-cache MoE layer.

This module only *generates inputs*: problem shapes, expert weight blobs,
routing traces and activations.  It holds none of the method's arithmetic
(no dedup, no residency, no split rule, no FFN).  The oracle under
``oracle/`` and the CUDA library each parse what is generated here with code
of their own.

Expert blob byte layout ("bank layout", one contiguous blob per (layer,
expert), the unit a cache slot holds; FreeToken, "The Architecture, Unpacked",
decision one: a slot holds a whole expert, never a part of one):

  f32 / bf16 weights:
      W_gu  [2I, H] row-major   rows 0..I-1 = gate projection, I..2I-1 = up
      W_d   [H, I]  row-major   down projection
  fp8 e4m3 weights with per-128x128-block fp32 scales:
      W_gu  [2I, H] e4m3 codes, W_d [H, I] e4m3 codes,
      s_gu  [2I/128, H/128] fp32, s_d [H/128, I/128] fp32
      (dequantised value = e4m3(code) * scale of the 128x128 block)
  nvfp4 (e2m1 codes, one e4m3 scale per 16 consecutive elements of a row, one
  fp32 scale per matrix):
      W_gu  [2I, H/2] bytes, W_d [H, I/2] bytes (element 2j in the low nibble
      of byte j, element 2j+1 in the high nibble),
      s_gu  [2I, H/16] e4m3 codes, s_d [H, I/16] e4m3 codes,
      g     [4] fp32 = (g_gu, g_d, 0, 0)
      (dequantised value = e2m1(code) * e4m3(block scale) * g of the matrix)
  mxfp4 (OCP MX: e2m1 codes, one e8m0 scale per 32 consecutive elements of a
  row, no matrix scale):
      W_gu  [2I, H/2] bytes, W_d [H, I/2] bytes (packed as nvfp4),
      s_gu  [2I, H/32] e8m0 codes, s_d [H, I/32] e8m0 codes
      (dequantised value = e2m1(code) * 2**(scale code - 127))

bf16 values are carried as uint16 bit patterns, e4m3 as uint8 codes.

Every generator is seeded (numpy PCG64 through SeedSequence); the same call
gives the same bytes on every machine.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field, replace

import numpy as np

__all__ = [
    "Shape", "Config", "CONFIGS", "config", "blob_bytes", "f32_to_bf16_bits",
    "f32_to_e4m3_codes", "f32_to_e2m1_codes", "make_blob", "make_pool", "make_shared",
    "routing_trace", "prefill_routing", "activations", "default_max_fetch",
]


# ----------------------------------------------------------------------------
# shapes and the five workloads
# ----------------------------------------------------------------------------
@dataclass(frozen=True)
class Shape:
    """MoE layer stack shape.  Flat expert id of (layer l, expert e) is l*E+e."""
    L: int          # MoE layers
    E: int          # routed experts per layer
    k: int          # top-k
    H: int          # hidden size
    I: int          # expert (SwiGLU) intermediate size
    wdtype: str     # 'f32' | 'bf16' | 'fp8' | 'nvfp4' | 'mxfp4'
    adtype: str     # 'f32' | 'bf16'   activation dtype
    n_shared: int = 0   # always-resident shared expert per layer (0 or 1)

    @property
    def n_flat(self) -> int:
        return self.L * self.E

    @property
    def blob_bytes(self) -> int:
        return blob_bytes(self)


@dataclass(frozen=True)
class Config:
    name: str
    shape: Shape
    T: int                      # tokens per decode step (or prefill chunk)
    steps: int                  # decode steps (1 for the prefill chunk)
    capacity: int               # cache slots C
    routing: str                # 'softmax' | 'softmax_bias' | 'zipf'
    seed: int
    zipf_s: float = 0.0
    reuse: float = 0.0
    bias_std: float = 0.0
    bw_mbps: tuple | None = None    # (B_pcie, B_cpu) MB/s; None = measured on the box
    resize_to: int | None = None
    resize_step: int | None = None
    prefill: bool = False
    max_fetch: int | None = None    # K; None = default_max_fetch

    def with_(self, **kw) -> "Config":
        return replace(self, **kw)


def blob_bytes(s: Shape) -> int:
    if s.wdtype == "f32":
        return 3 * s.I * s.H * 4
    if s.wdtype == "bf16":
        return 3 * s.I * s.H * 2
    if s.wdtype == "fp8":
        assert s.H % 128 == 0 and s.I % 128 == 0
        n_scales = (2 * s.I // 128) * (s.H // 128) + (s.H // 128) * (s.I // 128)
        return 3 * s.I * s.H + 4 * n_scales
    if s.wdtype == "nvfp4":
        assert s.H % 32 == 0 and s.I % 32 == 0
        return 3 * s.I * s.H // 2 + 3 * s.I * s.H // 16 + 16
    if s.wdtype == "mxfp4":
        assert s.H % 32 == 0 and s.I % 32 == 0
        return 3 * s.I * s.H // 2 + 3 * s.I * s.H // 32
    raise ValueError(s.wdtype)


def default_max_fetch(shape: Shape, T: int) -> int:
    """K when the fetch cap is not set: every unique routed expert may fill."""
    return min(shape.E, T * shape.k)


QWEN3 = Shape(L=48, E=128, k=8, H=2048, I=768, wdtype="bf16", adtype="bf16")

CONFIGS: dict[str, Config] = {
    # 1. tiny single layer, fp32, exhaustively checkable
    "tiny": Config("tiny", Shape(L=1, E=8, k=2, H=256, I=512, wdtype="f32", adtype="f32"),
                   T=4, steps=32, capacity=4, routing="softmax", seed=1234,
                   bw_mbps=(2000, 1000)),
    # 2. Qwen3-30B-A3B-shaped decode, batch 1, 37% of 6144 slots
    "qwen3_decode_b1": Config("qwen3_decode_b1", QWEN3, T=1, steps=256,
                              capacity=math.floor(0.37 * 6144), routing="zipf",
                              zipf_s=1.1, reuse=0.8, seed=1235),
    # 3. same shape, batch 16, 20% -> 12% resize before step 128, B_p:B_c = 1:1
    "qwen3_decode_b16": Config("qwen3_decode_b16", QWEN3, T=16, steps=256,
                               capacity=math.floor(0.20 * 6144), routing="softmax_bias",
                               bias_std=0.5, seed=1236, bw_mbps=(100000, 100000),
                               resize_to=math.floor(0.12 * 6144), resize_step=128),
    # 4. DeepSeek-V3-shaped slice, fp8 e4m3 + 128x128 fp32 scales, 11% of slots
    "dsv3_decode_slice": Config("dsv3_decode_slice",
                                Shape(L=4, E=256, k=8, H=7168, I=2048, wdtype="fp8",
                                      adtype="bf16", n_shared=1),
                                T=1, steps=128, capacity=math.floor(0.11 * 1024),
                                routing="zipf", zipf_s=1.0, reuse=0.8, seed=1237),
    # 5. prefill chunk, 8192 tokens, all 48 layers double-buffered
    "qwen3_prefill_8k": Config("qwen3_prefill_8k", QWEN3, T=8192, steps=1,
                               capacity=math.floor(0.37 * 6144), routing="softmax",
                               seed=1238, prefill=True),
}


def config(name: str) -> Config:
    return CONFIGS[name]


# ----------------------------------------------------------------------------
# number formats used to *write* inputs
# ----------------------------------------------------------------------------
def _rng(*key: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([int(k) for k in key])))


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round float32 to bfloat16 (nearest, ties to even); finite inputs only."""
    b = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32).astype(np.uint64)
    b = b + 0x7FFF + ((b >> 16) & 1)
    return (b >> 16).astype(np.uint16)


def f32_to_e4m3_codes(a: np.ndarray) -> np.ndarray:
    """Encode float32 as OCP FP8 E4M3 codes: nearest, ties to even, saturating at +-448.

    Normal results: round the binary32 pattern at mantissa bit 20 (carry runs
    into the exponent), then rebias the exponent from 127 to 7.  Subnormal
    results (|a| < 2**-6): rint(|a| * 2**9), which rounds half to even.
    NaN inputs are not expected.
    """
    a = np.ascontiguousarray(a, dtype=np.float32)
    bits = a.view(np.uint32)
    mag = bits & np.uint32(0x7FFFFFFF)
    rnd = (mag >> 20) & np.uint32(1)
    rnd += np.uint32(0x7FFFF)
    rnd += mag
    rnd >>= 20
    code = rnd.astype(np.int32)
    code -= 960
    np.clip(code, 0, 0x7E, out=code)
    sub = mag < np.uint32(0x3C800000)          # |a| < 2**-6
    if sub.any():
        code[sub] = np.rint(mag[sub].view(np.float32) * np.float32(512.0)).astype(np.int32)
    out = code.astype(np.uint8)
    out |= ((bits >> 24) & np.uint32(0x80)).astype(np.uint8)
    return out


_E2M1_MIDPOINTS = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0], np.float32)


def f32_to_e2m1_codes(a: np.ndarray) -> np.ndarray:
    """Encode float32 as FP4 E2M1 codes (bit 3 sign, magnitudes 0, 0.5, 1, 1.5, 2, 3,
    4, 6 for codes 0..7): nearest, ties to the even code, saturating at +-6."""
    a = np.ascontiguousarray(a, dtype=np.float32)
    mag = np.abs(a)
    idx = np.searchsorted(_E2M1_MIDPOINTS, mag, side="left")      # midpoints strictly below |a|
    tie = mag == _E2M1_MIDPOINTS[np.minimum(idx, 6)]
    code = (idx + (tie & (idx % 2 == 1))).astype(np.uint8)
    code |= (np.signbit(a).astype(np.uint8) << 3)
    return code


def _nvfp4(w: np.ndarray):
    """NVFP4 quantisation of one matrix [R, C]: global g = amax / (6 * 448); block
    scale (16 consecutive row elements) = e4m3 code of amax_b / 6 / g; element code =
    e2m1 of w / (decoded block scale * g).  Returns packed codes [R, C/2], scale codes
    [R, C/16] and g."""
    R, C = w.shape
    amax = float(np.abs(w).max())
    g = np.float32(amax / (6.0 * 448.0)) if amax > 0 else np.float32(1.0)
    blk = w.reshape(R, C // 16, 16)
    bmax = np.abs(blk).max(axis=2).astype(np.float32)
    sc = f32_to_e4m3_codes((bmax / np.float32(6.0) / g).astype(np.float32))
    # decoded block scale (e4m3 is exact in float32), times g
    e = ((sc >> 3) & 0xF).astype(np.int32)
    m = (sc & 0x7).astype(np.float32)
    dec = np.where(e == 0, m / np.float32(8.0) * np.float32(2.0 ** -6),
                   (np.float32(1.0) + m / np.float32(8.0)) * np.ldexp(np.float32(1.0), e - 7)).astype(np.float32)
    step = (dec * g).astype(np.float32)
    q = np.where(step[:, :, None] > 0, blk / np.where(step > 0, step, np.float32(1.0))[:, :, None],
                 np.float32(0.0)).astype(np.float32)
    codes = f32_to_e2m1_codes(q).reshape(R, C)
    packed = (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8)
    return packed, sc, g


def _mxfp4(w: np.ndarray):
    """MXFP4 quantisation of one matrix [R, C], the OCP Microscaling conversion of
    each block of 32 consecutive row elements: shared exponent X = floor(log2 amax)
    - 2 (2 = the largest E2M1 exponent), clamped to the E8M0 range [-127, 127];
    scale code X + 127; element code = e2m1 of w / 2**X (nearest, ties to even,
    saturating at +-6).  An all-zero block takes X = 0.  Returns packed codes
    [R, C/2] and scale codes [R, C/32]."""
    R, C = w.shape
    blk = np.ascontiguousarray(w, dtype=np.float32).reshape(R, C // 32, 32)
    amax = np.abs(blk).max(axis=2)
    _, e = np.frexp(amax)                      # amax = m * 2**e, m in [0.5, 1)
    X = np.clip(np.where(amax > 0, e.astype(np.int64) - 1 - 2, 0), -127, 127)
    q = (blk.astype(np.float64) * np.ldexp(1.0, -X)[:, :, None]).astype(np.float32)
    codes = f32_to_e2m1_codes(q).reshape(R, C)
    packed = (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8)
    return packed, (X + 127).astype(np.uint8)


# ----------------------------------------------------------------------------
# expert blobs and the host pool
# ----------------------------------------------------------------------------
WEIGHT_STD = 0.02


def make_blob(shape: Shape, seed: int, index: int, tag: int = 0xB10B) -> np.ndarray:
    """One complete expert in bank layout as a uint8 array of shape.blob_bytes.

    Weights ~ N(0, 0.02) drawn in float32, then stored in the shape's weight
    dtype (bf16: nearest-even; fp8: per-128x128-block scale = amax/448 and
    e4m3 codes of value/scale; nvfp4: see _nvfp4; mxfp4: see _mxfp4).
    """
    H, I = shape.H, shape.I
    g = _rng(seed, tag, index)
    w_gu = g.standard_normal((2 * I, H), dtype=np.float32) * np.float32(WEIGHT_STD)
    w_d = g.standard_normal((H, I), dtype=np.float32) * np.float32(WEIGHT_STD)
    if shape.wdtype == "f32":
        parts = [w_gu.view(np.uint8).ravel(), w_d.view(np.uint8).ravel()]
    elif shape.wdtype == "bf16":
        parts = [f32_to_bf16_bits(w_gu).view(np.uint8).ravel(),
                 f32_to_bf16_bits(w_d).view(np.uint8).ravel()]
    elif shape.wdtype == "fp8":
        codes_gu, s_gu = _blockscale_e4m3(w_gu)
        codes_d, s_d = _blockscale_e4m3(w_d)
        parts = [codes_gu.ravel(), codes_d.ravel(),
                 s_gu.view(np.uint8).ravel(), s_d.view(np.uint8).ravel()]
    elif shape.wdtype == "nvfp4":
        p_gu, s_gu, g_gu = _nvfp4(w_gu)
        p_d, s_d, g_d = _nvfp4(w_d)
        parts = [p_gu.ravel(), p_d.ravel(), s_gu.ravel(), s_d.ravel(),
                 np.array([g_gu, g_d, 0, 0], np.float32).view(np.uint8)]
    elif shape.wdtype == "mxfp4":
        p_gu, s_gu = _mxfp4(w_gu)
        p_d, s_d = _mxfp4(w_d)
        parts = [p_gu.ravel(), p_d.ravel(), s_gu.ravel(), s_d.ravel()]
    else:
        raise ValueError(shape.wdtype)
    blob = np.concatenate(parts)
    assert blob.size == shape.blob_bytes
    return blob


def _blockscale_e4m3(w: np.ndarray):
    R, Cc = w.shape
    blk = w.reshape(R // 128, 128, Cc // 128, 128)
    amax = np.abs(blk).max(axis=(1, 3)).astype(np.float32)
    scale = np.where(amax > 0, amax / np.float32(448.0), np.float32(1.0)).astype(np.float32)
    scaled = (blk / scale[:, None, :, None]).astype(np.float32)
    codes = f32_to_e4m3_codes(scaled).reshape(R, Cc)
    return codes, np.ascontiguousarray(scale)


def make_pool(shape: Shape, seed: int, n_phys: int | None = None, out: np.ndarray | None = None):
    """Host expert pool: an arena of n_phys distinct blobs plus per-expert byte offsets.

    Logical expert f (= l*E+e) lives at byte offset offsets[f] = (f mod n_phys) * S.
    With n_phys = L*E (the default) every expert is distinct; a smaller arena
    stands in for a pool too large to hold, with experts f and f+n_phys sharing
    bytes.  `out` may be a preallocated (e.g. pinned) uint8 buffer of
    n_phys * S bytes.
    """
    S = shape.blob_bytes
    n_phys = shape.n_flat if n_phys is None else int(n_phys)
    assert 1 <= n_phys <= shape.n_flat
    arena = np.empty(n_phys * S, dtype=np.uint8) if out is None else out
    assert arena.size >= n_phys * S
    for p in range(n_phys):
        arena[p * S:(p + 1) * S] = make_blob(shape, seed, p)
    offsets = (np.arange(shape.n_flat, dtype=np.uint64) % np.uint64(n_phys)) * np.uint64(S)
    return arena, offsets


def make_shared(shape: Shape, seed: int) -> np.ndarray:
    """Shared (always resident) expert blobs, one per layer, concatenated."""
    if shape.n_shared == 0:
        return np.zeros(0, dtype=np.uint8)
    return np.concatenate([make_blob(shape, seed, l, tag=0x5AED) for l in range(shape.L)])


# ----------------------------------------------------------------------------
# routing traces and activations
# ----------------------------------------------------------------------------
def _softmax_rows(z: np.ndarray) -> np.ndarray:
    z = z.astype(np.float64)
    z = z - z.max(axis=-1, keepdims=True)
    e = np.exp(z)
    return (e / e.sum(axis=-1, keepdims=True)).astype(np.float32)


def _topk_from_logits(logits: np.ndarray, k: int):
    # ties go to the lower expert index: stable sort of -logits
    idx = np.argsort(-logits, axis=-1, kind="stable")[..., :k]
    chosen = np.take_along_axis(logits, idx, axis=-1)
    return idx.astype(np.int32), _softmax_rows(chosen)


def routing_trace(cfg: Config):
    """Decode routing for every step and layer: ids [steps, L, T, k] int32, gates fp32."""
    s = cfg.shape
    g = _rng(cfg.seed, 0x7A11)
    if cfg.routing in ("softmax", "softmax_bias"):
        bias = (g.standard_normal((s.L, s.E)) * cfg.bias_std) if cfg.routing == "softmax_bias" \
            else np.zeros((s.L, s.E))
        ids = np.empty((cfg.steps, s.L, cfg.T, s.k), np.int32)
        w = np.empty((cfg.steps, s.L, cfg.T, s.k), np.float32)
        for st in range(cfg.steps):
            logits = g.standard_normal((s.L, cfg.T, s.E)) + bias[:, None, :]
            ids[st], w[st] = _topk_from_logits(logits, s.k)
        return ids, w
    if cfg.routing == "zipf":
        return _zipf_trace(cfg, g)
    raise ValueError(cfg.routing)


def _zipf_trace(cfg: Config, g: np.random.Generator):
    """Zipf(s) expert popularity over a fixed per-layer permutation, with step-to-step reuse.

    Pick j of a token reuses the previous step's pick j with probability
    `reuse` (if not already chosen), else draws a fresh Zipf rank; a draw
    that repeats an expert already chosen for this token is redrawn.
    """
    s = cfg.shape
    perm = np.stack([g.permutation(s.E) for _ in range(s.L)])
    ranks = np.arange(1, s.E + 1, dtype=np.float64)
    p = ranks ** (-cfg.zipf_s)
    cdf = np.cumsum(p / p.sum())
    ids = np.empty((cfg.steps, s.L, cfg.T, s.k), np.int32)
    prev = None
    for st in range(cfg.steps):
        u_reuse = g.random((s.L, cfg.T, s.k))
        for l in range(s.L):
            for t in range(cfg.T):
                chosen: list[int] = []
                for j in range(s.k):
                    e = -1
                    if prev is not None and u_reuse[l, t, j] < cfg.reuse:
                        cand = int(prev[l, t, j])
                        if cand not in chosen:
                            e = cand
                    while e < 0 or e in chosen:
                        r = int(np.searchsorted(cdf, g.random(), side="right"))
                        e = int(perm[l, min(r, s.E - 1)])
                    chosen.append(e)
                ids[st, l, t] = chosen
        prev = ids[st]
    w = _softmax_rows(g.standard_normal((cfg.steps, s.L, cfg.T, s.k)))
    return ids, w


def prefill_routing(cfg: Config, layer: int):
    """Prefill routing for one layer: top-k of N(0,1) logits over E, ids [T,k], gates [T,k]."""
    s = cfg.shape
    g = _rng(cfg.seed, 0x9F11, layer)
    logits = g.standard_normal((cfg.T, s.E), dtype=np.float32)
    return _topk_from_logits(logits, s.k)


def activations(cfg: Config, step: int, layer: int) -> np.ndarray:
    """x [T, H] ~ N(0,1) for one (step, layer): float32 array, or uint16 bf16 bits."""
    s = cfg.shape
    g = _rng(cfg.seed, 0xAC7, step, layer)
    x = g.standard_normal((cfg.T, s.H), dtype=np.float32)
    return x if s.adtype == "f32" else f32_to_bf16_bits(x)
