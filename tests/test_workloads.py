"""The seeded input generators: determinism, shapes and stated distributions."""
import numpy as np

from workloads import (CONFIGS, activations, blob_bytes, config, make_blob, make_pool,
                       prefill_routing, routing_trace)


def test_config_sizes_match_the_stated_workloads():
    assert config("tiny").shape.blob_bytes == 1572864                 # 1.57 MB fp32 expert
    assert config("qwen3_decode_b1").shape.blob_bytes == 9437184      # 9.44 MB bf16 expert
    assert config("dsv3_decode_slice").shape.blob_bytes == 44050944   # 44.05 MB incl. scales
    assert config("qwen3_decode_b1").capacity == 2273
    assert config("qwen3_decode_b16").capacity == 1228 and config("qwen3_decode_b16").resize_to == 737
    assert config("dsv3_decode_slice").capacity == 112
    assert config("qwen3_prefill_8k").capacity >= 2 * 128
    s = config("qwen3_decode_b1").shape
    assert s.n_flat * s.blob_bytes == 57982058496                     # 58.0 GB pool


def test_generators_are_deterministic():
    c = config("tiny")
    a1, w1 = routing_trace(c)
    a2, w2 = routing_trace(c)
    assert np.array_equal(a1, a2) and np.array_equal(w1, w2)
    assert np.array_equal(activations(c, 3, 0), activations(c, 3, 0))
    assert not np.array_equal(activations(c, 3, 0), activations(c, 4, 0))
    sh = c.shape
    assert np.array_equal(make_blob(sh, 1, 2), make_blob(sh, 1, 2))
    assert not np.array_equal(make_blob(sh, 1, 2), make_blob(sh, 1, 3))


def test_routing_is_valid_topk():
    for name in ["tiny", "qwen3_decode_b16"]:
        c = config(name).with_(steps=8)
        ids, w = routing_trace(c)
        assert ids.shape == (8, c.shape.L, c.T, c.shape.k)
        assert ids.min() >= 0 and ids.max() < c.shape.E
        for row in ids.reshape(-1, c.shape.k):
            assert len(set(row.tolist())) == c.shape.k
        assert np.allclose(w.sum(-1), 1.0, atol=1e-6)


def test_zipf_trace_reuse_and_skew():
    c = config("qwen3_decode_b1").with_(steps=80)
    ids, w = routing_trace(c)
    same = np.mean(ids[1:] == ids[:-1])
    assert 0.7 < same < 0.9                       # 80% step-to-step reuse of each pick
    for row in ids.reshape(-1, c.shape.k):
        assert len(set(row.tolist())) == c.shape.k
    counts = np.bincount(ids[:, 0].ravel(), minlength=c.shape.E)
    assert counts.max() > 5 * np.median(counts)   # heavy head


def test_prefill_routing_covers_nearly_all_experts():
    c = config("qwen3_prefill_8k")
    ids, w = prefill_routing(c, 0)
    assert ids.shape == (8192, 8)
    assert len(np.unique(ids)) == 128


def test_pool_offsets_and_aliasing():
    c = config("tiny")
    arena, offs = make_pool(c.shape, 5)
    assert arena.size == 8 * c.shape.blob_bytes
    assert list(offs) == [i * c.shape.blob_bytes for i in range(8)]
    arena2, offs2 = make_pool(c.shape, 5, n_phys=3)
    assert list(offs2) == [(i % 3) * c.shape.blob_bytes for i in range(8)]
    assert np.array_equal(arena2[: 3 * c.shape.blob_bytes], arena[: 3 * c.shape.blob_bytes])


def test_four_bit_blobs_are_seeded_and_sized():
    # the 4-bit variants of the Qwen3 shape: sizes the bench quotes, seeded bytes,
    # and the host pool's flat-id -> blob mapping unchanged by the format
    base = config("qwen3_decode_b1").shape
    for fmt, size in (("nvfp4", 2654224), ("mxfp4", 2506752)):
        s = base.__class__(**{**base.__dict__, "wdtype": fmt})
        assert blob_bytes(s) == size and size % 16 == 0
        small = base.__class__(L=2, E=4, k=2, H=256, I=128, wdtype=fmt, adtype="bf16")
        assert np.array_equal(make_blob(small, 5, 1), make_blob(small, 5, 1))
        assert not np.array_equal(make_blob(small, 5, 1), make_blob(small, 5, 2))
        arena, offs = make_pool(small, 5, n_phys=3)
        assert offs.shape == (small.L * small.E,)
        for f in range(small.L * small.E):
            o = int(offs[f])
            assert o % 16 == 0
            assert np.array_equal(arena[o:o + small.blob_bytes], make_blob(small, 5, f % 3))
