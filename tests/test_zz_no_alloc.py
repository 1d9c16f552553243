"""The allocation-free entry point, checked against the oracle.

moe_layer_ffn_noalloc serves callers that may not allocate GPU memory (code
inside another framework's memory pool, a process that reserved all device
memory at start-up): it keeps its intermediates in the library's fixed device
scratch array.  These tests call it through the C ABI and compare its layer
output with the oracle's float64 SwiGLU + fixed-order combine, on two calls in
a row (the second reuses the scratch the first one left behind), and once in a
fresh process that never created a cache (so nothing else has set the GEMV
kernels' shared-memory limits).  The argument refusals of the binding run on
the CPU.
"""
import json
import os
import subprocess
import sys

import numpy as np
import pytest

from oracle.ffn import ExpertStore, combine, pair_outputs, relative_max_error
from tests.harness import TOL, torch_act
from workloads import Config, Shape, activations, make_pool, routing_trace

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _oracle_out(store, cfg, ids, w, x):
    s = cfg.shape
    y = pair_outputs(store, 0, s.E, x, s.adtype, ids)
    return combine(w, y, np.zeros(ids.shape, np.int32), None)


def _run_calls(s: Shape, T: int, seed: int, calls: int):
    """(max relative error against the oracle, all outputs finite) over `calls` calls in a row."""
    import torch
    from serving_layer_moe_gb300.binding import ffn_noalloc
    cfg = Config("noalloc", s, T=T, steps=calls, capacity=s.E, routing="softmax", seed=seed)
    arena, offs = make_pool(s, cfg.seed)
    store = ExpertStore(arena, offs, s.wdtype, s.H, s.I, s.blob_bytes)
    dev = torch.device("cuda", 0)
    experts = torch.from_numpy(arena).to(dev)             # the layer's E blobs back to back
    ids, w = routing_trace(cfg)
    worst, finite = 0.0, True
    for call in range(calls):
        x = activations(cfg, call, 0)
        got = torch.full((T, s.H), float("nan"), device=dev)
        ffn_noalloc(experts, torch_act(x, dev), torch.from_numpy(ids[call, 0]).to(dev),
                    torch.from_numpy(w[call, 0]).to(dev), got, E=s.E, H=s.H, I=s.I, top_k=s.k,
                    wdtype=s.wdtype, adtype=s.adtype)
        torch.cuda.synchronize()
        g = got.cpu().numpy()
        finite = finite and bool(np.all(np.isfinite(g)))
        worst = max(worst, relative_max_error(g, _oracle_out(store, cfg, ids[call, 0], w[call, 0], x)))
    return worst, finite


@pytest.mark.gpu
@pytest.mark.parametrize("wdtype,adtype,H,I", [("bf16", "bf16", 512, 256), ("f32", "f32", 512, 256),
                                                ("fp8", "bf16", 512, 256)])
def test_noalloc_matches_oracle_on_two_calls(wdtype, adtype, H, I):
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    err, finite = _run_calls(Shape(L=1, E=16, k=4, H=H, I=I, wdtype=wdtype, adtype=adtype), T=8, seed=77, calls=2)
    assert finite
    assert err <= TOL, err


def _fresh_process_child():
    """Run in a new interpreter: no MoECache is ever created before the call."""
    s = Shape(L=1, E=16, k=4, H=2048, I=256, wdtype="bf16", adtype="bf16")
    err, finite = _run_calls(s, T=16, seed=78, calls=2)   # x (64 KB) + pair lists: above 48 KB of shared memory
    print(json.dumps({"err": err, "finite": finite}))


@pytest.mark.gpu
def test_noalloc_in_a_fresh_process_without_a_cache():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    code = ("import sys; sys.path.insert(0, %r); import tests.test_zz_no_alloc as t; t._fresh_process_child()" % ROOT)
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    d = json.loads([l for l in r.stdout.splitlines() if l.startswith("{")][-1])
    assert d["finite"]
    assert d["err"] <= TOL, d


@pytest.mark.gpu
def test_noalloc_rejects_oversized_calls():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from serving_layer_moe_gb300 import MoEError
    from serving_layer_moe_gb300.binding import ffn_noalloc
    dev = torch.device("cuda", 0)
    for T, k, H, I in ((1024, 8, 2048, 768),      # ~92 MB of scratch needed > 16 MiB
                       (2048, 8, 8, 8)):          # 16384 routed pairs > 9216
        experts = torch.zeros(16 * 6 * H * I, dtype=torch.uint8, device=dev)
        x = torch.zeros(T, H, dtype=torch.int16, device=dev)
        ids = torch.zeros(T, k, dtype=torch.int32, device=dev)
        w = torch.zeros(T, k, device=dev)
        out = torch.zeros(T, H, device=dev)
        with pytest.raises(MoEError) as ei:
            ffn_noalloc(experts, x, ids, w, out, E=16, H=H, I=I, top_k=k, wdtype="bf16", adtype="bf16")
        assert ei.value.status == 4


# ---- argument refusals of the binding (CPU: nothing reaches the library) --------------------
def _cpu_args(T=4, k=2, E=8, H=64, I=32, wdtype="bf16", adtype="bf16"):
    torch = pytest.importorskip("torch")
    from serving_layer_moe_gb300.binding import blob_bytes
    es = 4 if adtype == "f32" else 2
    return dict(experts=torch.zeros(E * blob_bytes(wdtype, H, I), dtype=torch.uint8),
                x=torch.zeros(T, H, dtype=torch.float32 if es == 4 else torch.int16),
                topk_ids=torch.zeros(T, k, dtype=torch.int32), topk_w=torch.zeros(T, k),
                out=torch.zeros(T, H)), dict(E=E, H=H, I=I, top_k=k, wdtype=wdtype, adtype=adtype)


@pytest.mark.parametrize("case", ["short_experts", "ids_dtype", "ids_shape", "w_dtype", "out_shape",
                                  "x_elem", "x_shape", "adtype", "cpu_tensors"])
def test_noalloc_binding_refuses_mismatched_arguments(case):
    torch = pytest.importorskip("torch")
    from serving_layer_moe_gb300.binding import ffn_noalloc
    t, kw = _cpu_args()
    if case == "short_experts":
        t["experts"] = t["experts"][:-16]
    elif case == "ids_dtype":
        t["topk_ids"] = t["topk_ids"].long()
    elif case == "ids_shape":
        t["topk_ids"] = torch.zeros(4, 3, dtype=torch.int32)
    elif case == "w_dtype":
        t["topk_w"] = t["topk_w"].double()
    elif case == "out_shape":
        t["out"] = torch.zeros(4, 32)
    elif case == "x_elem":
        t["x"] = torch.zeros(4, 64, dtype=torch.float32)    # bf16 activations are 2-byte elements
    elif case == "x_shape":
        t["x"] = torch.zeros(3, 64, dtype=torch.int16)
    elif case == "adtype":
        kw["adtype"] = "fp8"
    # cpu_tensors: every argument is right but none is on a CUDA device
    with pytest.raises(ValueError):
        ffn_noalloc(t["experts"], t["x"], t["topk_ids"], t["topk_w"], t["out"], **kw)


def test_binding_blob_bytes_matches_the_workload_generator():
    from serving_layer_moe_gb300.binding import blob_bytes
    for wd, H, I in (("f32", 256, 512), ("bf16", 2048, 768), ("fp8", 7168, 2048), ("nvfp4", 2048, 768),
                     ("mxfp4", 2048, 768)):
        assert blob_bytes(wd, H, I) == Shape(L=1, E=1, k=1, H=H, I=I, wdtype=wd, adtype="bf16").blob_bytes
