"""Pins of the oracle's SwiGLU expert and combine."""
import math

import numpy as np
import pytest

from oracle.ffn import (ExpertStore, combine, pair_outputs, relative_max_error, silu,
                        swiglu_expert, swiglu_expert_loops)
from oracle.formats import parse_blob
from tests.conftest import read_golden
from workloads import Shape, make_pool


def test_silu_special_values():
    assert silu(np.array(0.0)) == 0.0
    assert abs(float(silu(np.array(1.0))) - 1.0 / (1.0 + math.e ** -1)) < 1e-16
    assert abs(float(silu(np.array(40.0))) - 40.0) < 1e-12          # -> identity
    assert abs(float(silu(np.array(-40.0)))) < 1e-15                 # -> 0
    z = np.linspace(-6, 6, 101)
    assert np.allclose(silu(z) - silu(-z), z)                        # silu(z) - silu(-z) = z


def test_hand_derived_expert():
    gold = {r[0]: float(r[1]) for r in read_golden("swiglu_hand.txt")}
    x = np.array([1.0, 2.0])
    wg = np.array([[1.0, 0.0], [0.0, 1.0]])
    wu = np.array([[1.0, 1.0], [0.0, 0.0]])
    wd = np.array([[1.0, 0.0], [2.0, 0.0]])
    y = swiglu_expert(x, wg, wu, wd)
    assert abs(float(silu(np.array(1.0))) - gold["silu1"]) < 1e-15
    assert abs(y[0] - gold["y0"]) < 1e-13 and abs(y[1] - gold["y1"]) < 1e-13


@pytest.mark.parametrize("seed", range(5))
def test_matrix_form_equals_loops(seed):
    g = np.random.default_rng(seed)
    H, I = 12, 7
    x = g.standard_normal(H)
    wg, wu, wd = g.standard_normal((I, H)), g.standard_normal((I, H)), g.standard_normal((H, I))
    assert np.allclose(swiglu_expert(x, wg, wu, wd), swiglu_expert_loops(x, wg, wu, wd), rtol=1e-12, atol=1e-12)
    # gate and up are not interchangeable (catches swapped operands)
    assert not np.allclose(swiglu_expert(x, wu, wg, wd), swiglu_expert(x, wg, wu, wd))


def test_batched_rows_equal_single_rows():
    g = np.random.default_rng(9)
    H, I = 16, 8
    X = g.standard_normal((5, H))
    w = g.standard_normal((I, H)), g.standard_normal((I, H)), g.standard_normal((H, I))
    Y = swiglu_expert(X, *w)
    for t in range(5):
        assert np.allclose(Y[t], swiglu_expert(X[t], *w), rtol=1e-13, atol=1e-13)


def test_combine_fixed_order_and_exact_split():
    g = np.random.default_rng(1)
    T, k, H = 3, 4, 5
    w = g.random((T, k))
    y = g.standard_normal((T, k, H))
    all_gpu = combine(w, y, np.zeros((T, k), np.int32), None)
    # explicit sum in j order
    for t in range(T):
        acc = np.zeros(H)
        for j in range(k):
            acc = acc + w[t, j] * y[t, j]
        assert np.array_equal(all_gpu[t], acc)
    # split: CPU partial sums are exactly the same per-expert outputs -> bit-identical
    sm = np.array([[0, -1, 2, -1], [-1, -1, -1, -1], [5, 6, 7, 8]], np.int32)
    cpu = np.where(sm[..., None] < 0, y, np.nan)
    gpu = np.where(sm[..., None] >= 0, y, np.nan)
    split = combine(w, gpu, sm, cpu)
    assert np.array_equal(split, all_gpu)
    with pytest.raises(ValueError):
        combine(w, y, sm, None)


def test_combine_adds_shared_expert_last():
    w = np.array([[0.5, 0.5]])
    y = np.array([[[2.0], [4.0]]])
    out = combine(w, y, np.zeros((1, 2), np.int32), None, shared_y=np.array([[10.0]]))
    assert out[0, 0] == 13.0


@pytest.mark.parametrize("wdtype", ["f32", "bf16", "fp8"])
def test_pair_outputs_per_expert(wdtype):
    sh = Shape(L=2, E=3, k=2, H=128, I=128, wdtype=wdtype, adtype="f32")
    arena, offs = make_pool(sh, 11)
    st = ExpertStore(arena, offs, wdtype, sh.H, sh.I, sh.blob_bytes)
    g = np.random.default_rng(0)
    x = g.standard_normal((4, sh.H)).astype(np.float32)
    ids = np.array([[0, 1], [2, 0], [1, 2], [0, 2]], np.int32)
    y = pair_outputs(st, 1, sh.E, x, "f32", ids)
    for t in range(4):
        for j in range(2):
            f = 1 * sh.E + ids[t, j]
            blob = arena[int(offs[f]):int(offs[f]) + sh.blob_bytes]
            ref = swiglu_expert(x[t].astype(np.float64), *parse_blob(blob, wdtype, sh.H, sh.I))
            assert np.allclose(y[t, j], ref, rtol=1e-12, atol=1e-15)


def test_relative_max_error():
    assert relative_max_error(np.array([1.0, 2.0]), np.array([1.0, 2.0])) == 0.0
    assert relative_max_error(np.array([1.1, 2.0]), np.array([1.0, 2.0])) == pytest.approx(0.05)
