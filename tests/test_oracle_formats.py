"""Pins of the oracle's weight-format decoding against definitions and library conversions."""
import numpy as np
import pytest
import torch

from oracle.formats import bf16_bits_to_f64, blockscale_dequant, e4m3_codes_to_f64, parse_blob
from workloads import Shape, f32_to_bf16_bits, f32_to_e4m3_codes, make_blob


def test_bf16_closed_form_values():
    bits = np.array([0x3F80, 0xC000, 0x0000, 0x8000, 0x7F80, 0x0001, 0x3F81], np.uint16)
    v = bf16_bits_to_f64(bits)
    assert v[0] == 1.0 and v[1] == -2.0 and v[2] == 0.0
    assert np.signbit(v[3]) and v[3] == 0.0
    assert np.isinf(v[4])
    assert v[5] == 2.0 ** -133          # smallest subnormal
    assert v[6] == 1.0 + 2.0 ** -7      # one ulp above 1


def test_bf16_matches_torch_all_finite_codes():
    codes = np.arange(1 << 16, dtype=np.uint16)
    ours = bf16_bits_to_f64(codes)
    t = torch.from_numpy(codes.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    fin = np.isfinite(t)
    assert np.array_equal(ours[fin], t[fin])
    assert np.array_equal(np.isnan(ours), np.isnan(t))


def test_e4m3_closed_form_values():
    v = e4m3_codes_to_f64(np.array([0x38, 0x7E, 0x01, 0x08, 0xB8, 0x7F, 0xFF, 0x00, 0x30], np.uint8))
    assert v[0] == 1.0
    assert v[1] == 448.0                 # max finite
    assert v[2] == 2.0 ** -9             # smallest subnormal
    assert v[3] == 2.0 ** -6             # smallest normal
    assert v[4] == -1.0
    assert np.isnan(v[5]) and np.isnan(v[6])
    assert v[7] == 0.0
    assert v[8] == 0.5


def test_e4m3_matches_torch_all_codes():
    codes = np.arange(256, dtype=np.uint8)
    ours = e4m3_codes_to_f64(codes)
    t = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    assert np.array_equal(np.isnan(ours), np.isnan(t))
    fin = ~np.isnan(t)
    assert np.array_equal(ours[fin], t[fin])


def test_generator_e4m3_encoder_matches_torch_rounding():
    g = np.random.default_rng(5)
    a = np.concatenate([g.standard_normal(200000).astype(np.float32) * 50,
                        g.standard_normal(20000).astype(np.float32) * 0.01,
                        np.array([448, -448, 0.0, 2 ** -10, 3 * 2 ** -10, 1.0625, 1.1875], np.float32)])
    ours = f32_to_e4m3_codes(a)
    t = torch.from_numpy(a).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    inr = np.abs(a) <= 448
    assert np.array_equal(ours[inr], t[inr])


def test_generator_bf16_rounding_matches_torch():
    a = np.random.default_rng(6).standard_normal(100000).astype(np.float32)
    ours = f32_to_bf16_bits(a)
    t = torch.from_numpy(a).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, t)


def test_blockscale_indexing_is_row_block_major():
    # all codes = 1.0; scale of block (rb, cb) = 10*rb + cb + 1 -> dequant shows the grid
    codes = np.full((256, 384), 0x38, np.uint8)
    scales = np.array([[10 * rb + cb + 1 for cb in range(3)] for rb in range(2)], np.float32)
    d = blockscale_dequant(codes, scales)
    assert d[0, 0] == 1 and d[127, 127] == 1
    assert d[0, 128] == 2 and d[0, 383] == 3
    assert d[128, 0] == 11 and d[255, 383] == 13


@pytest.mark.parametrize("wdtype", ["f32", "bf16", "fp8"])
def test_parse_blob_roundtrip(wdtype):
    sh = Shape(L=1, E=1, k=1, H=256, I=128, wdtype=wdtype, adtype="f32")
    blob = make_blob(sh, 7, 0)
    wg, wu, wd = parse_blob(blob, wdtype, sh.H, sh.I)
    assert wg.shape == (128, 256) and wu.shape == (128, 256) and wd.shape == (256, 128)
    # regenerate the float32 draws the generator quantised and compare within the format's step
    from workloads import _rng
    g = _rng(7, 0xB10B, 0)
    gu = g.standard_normal((256, 256), dtype=np.float32) * np.float32(0.02)
    d = g.standard_normal((256, 128), dtype=np.float32) * np.float32(0.02)
    rel = {"f32": 0.0, "bf16": 2 ** -8, "fp8": 2 ** -3}[wdtype]
    assert np.allclose(wg, gu[:128], rtol=rel, atol=1e-3 * (wdtype == "fp8"))
    assert np.allclose(wu, gu[128:], rtol=rel, atol=1e-3 * (wdtype == "fp8"))
    assert np.allclose(wd, d, rtol=rel, atol=1e-3 * (wdtype == "fp8"))


# ---- NVFP4: e2m1 elements, e4m3 scales per 16 row elements, fp32 per matrix ----

def test_e2m1_closed_form_values():
    from oracle.formats import E2M1_TABLE
    # bit 3 sign, bits 2-1 exponent (bias 1), bit 0 mantissa
    assert list(E2M1_TABLE[:8]) == [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
    assert list(E2M1_TABLE[8:]) == [-0.0, -0.5, -1.0, -1.5, -2.0, -3.0, -4.0, -6.0]
    assert np.signbit(E2M1_TABLE[8])


def test_generator_e2m1_encoder_nearest_ties_to_even_saturating():
    from oracle.formats import E2M1_TABLE
    from workloads import f32_to_e2m1_codes
    mags = E2M1_TABLE[:8]
    grid = np.concatenate([np.arange(0, 8.0, 1 / 64.0), mags, (mags[1:] + mags[:-1]) / 2, [6.0, 6.5, 100.0]])
    x = np.concatenate([grid, -grid]).astype(np.float32)
    codes = f32_to_e2m1_codes(x)
    for v, c in zip(x, codes):
        d = np.abs(mags - abs(float(v)))
        best = np.flatnonzero(d == d.min())
        want = best[0] if len(best) == 1 else [b for b in best if b % 2 == 0][0]   # ties: even code
        if abs(v) > 6.0:
            want = 7                                                             # saturate
        assert (c & 7) == want, (v, c, want)
        assert (c >> 3) == (1 if np.signbit(v) else 0)


def test_nvfp4_blob_dequantises_within_one_block_step():
    # each element is within one step (decoded block scale x g) of the float32 draw
    from oracle.formats import E4M3_TABLE, parse_blob
    from workloads import WEIGHT_STD, _rng
    s = Shape(L=1, E=4, k=1, H=128, I=64, wdtype="nvfp4", adtype="bf16")
    for idx in range(3):
        blob = make_blob(s, 77, idx)
        g = _rng(77, 0xB10B, idx)
        w_gu = g.standard_normal((2 * s.I, s.H), dtype=np.float32) * np.float32(WEIGHT_STD)
        w_d = g.standard_normal((s.H, s.I), dtype=np.float32) * np.float32(WEIGHT_STD)
        gate, up, down = parse_blob(blob, "nvfp4", s.H, s.I)
        o = 3 * s.I * s.H // 2
        s_gu = blob[o:o + 2 * s.I * s.H // 16].reshape(2 * s.I, s.H // 16)
        s_d = blob[o + 2 * s.I * s.H // 16:o + 3 * s.I * s.H // 16].reshape(s.H, s.I // 16)
        gg = blob[-16:].view(np.float32)
        for w, deq, sc, gm in ((w_gu, np.vstack([gate, up]), s_gu, gg[0]), (w_d, down, s_d, gg[1])):
            step = np.repeat(E4M3_TABLE[sc], 16, axis=1) * float(gm)
            err = np.abs(deq - w.astype(np.float64))
            assert np.all(err <= step + 1e-12)
            assert np.mean(err) < 0.1 * np.mean(np.abs(w))        # not a constant or a dropped factor
            assert gm == np.float32(np.abs(w).max() / (6.0 * 448.0))


# ---- MXFP4 (OCP Microscaling): e2m1 elements, one e8m0 scale per 32 row elements ----

def test_e8m0_closed_form_values():
    from oracle.formats import e8m0_codes_to_f64
    v = e8m0_codes_to_f64(np.array([127, 128, 126, 0, 254, 255, 121], np.uint8))
    assert v[0] == 1.0 and v[1] == 2.0 and v[2] == 0.5
    assert v[3] == 2.0 ** -127 and v[4] == 2.0 ** 127
    assert np.isnan(v[5])
    assert v[6] == 1.0 / 64


def test_e8m0_matches_torch_all_codes():
    from oracle.formats import e8m0_codes_to_f64
    dt = getattr(torch, "float8_e8m0fnu", None)
    if dt is None:
        pytest.skip("this torch has no float8_e8m0fnu")
    codes = np.arange(256, dtype=np.uint8)
    lib = torch.from_numpy(codes).view(dt).to(torch.float64).numpy()
    ours = e8m0_codes_to_f64(codes)
    assert np.array_equal(np.isnan(lib), np.isnan(ours))
    assert np.array_equal(lib[:255], ours[:255])


def test_mxfp4_hand_built_blob_indexes_scales_by_row_and_32_block():
    # every code fixed by hand: element 2j of a row is code 0x2 (1.0), element
    # 2j+1 code 0xC (-2.0); each (row, 32-element block) has its own scale code,
    # so a scale taken from the wrong row, block width or matrix shows up.
    from oracle.formats import parse_blob
    H, I = 64, 32
    p_gu = np.full((2 * I, H // 2), 0xC2, np.uint8)
    p_d = np.full((H, I // 2), 0xC2, np.uint8)
    s_gu = ((np.arange(2 * I)[:, None] * 3 + np.arange(H // 32)[None, :] * 5) % 40 + 100).astype(np.uint8)
    s_d = ((np.arange(H)[:, None] * 7) % 30 + 110).astype(np.uint8)
    blob = np.concatenate([p_gu.ravel(), p_d.ravel(), s_gu.ravel(), s_d.ravel()])
    assert blob.size == Shape(L=1, E=1, k=1, H=H, I=I, wdtype="mxfp4", adtype="bf16").blob_bytes
    gate, up, down = parse_blob(blob, "mxfp4", H, I)
    for r in range(2 * I):
        for c in range(H):
            want = (1.0 if c % 2 == 0 else -2.0) * 2.0 ** (int(s_gu[r, c // 32]) - 127)
            got = gate[r, c] if r < I else up[r - I, c]
            assert got == want, (r, c)
    for r in range(H):
        for c in range(I):
            assert down[r, c] == (1.0 if c % 2 == 0 else -2.0) * 2.0 ** (int(s_d[r, 0]) - 127)


def test_mxfp4_blob_follows_the_mx_conversion():
    # the generator's blob against the float32 draw: the scale of each 32-element
    # block is 2**(floor(log2 amax) - 2); an element below the saturation point is
    # within half an e2m1 step (at most 2**X) of the draw, one above it decodes to
    # +-6 * 2**X; and the quantisation is not degenerate.
    import math
    from workloads import _rng, WEIGHT_STD
    s = Shape(L=1, E=4, k=1, H=128, I=64, wdtype="mxfp4", adtype="bf16")
    for idx in range(3):
        blob = make_blob(s, 78, idx)
        g = _rng(78, 0xB10B, idx)
        w_gu = g.standard_normal((2 * s.I, s.H), dtype=np.float32) * np.float32(WEIGHT_STD)
        w_d = g.standard_normal((s.H, s.I), dtype=np.float32) * np.float32(WEIGHT_STD)
        gate, up, down = parse_blob(blob, "mxfp4", s.H, s.I)
        for w, deq in ((w_gu, np.vstack([gate, up])), (w_d, down)):
            R, C = w.shape
            for r in range(R):
                for b in range(C // 32):
                    blk = w[r, 32 * b:32 * b + 32].astype(np.float64)
                    X = math.floor(math.log2(np.abs(blk).max())) - 2
                    d = deq[r, 32 * b:32 * b + 32]
                    big = np.abs(blk) > 6.0 * 2.0 ** X
                    assert np.all(d[big] == np.sign(blk[big]) * 6.0 * 2.0 ** X)
                    assert np.all(np.abs(d[~big] - blk[~big]) <= 2.0 ** X)
                    # every decoded value is an e2m1 magnitude times the scale
                    assert np.all(np.isin(np.abs(d) / 2.0 ** X, [0, 0.5, 1, 1.5, 2, 3, 4, 6]))
            err = np.abs(deq - w.astype(np.float64))
            assert np.mean(err) < 0.15 * np.mean(np.abs(w))
