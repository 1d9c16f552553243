"""The allocation-free entry point, checked against moe_layer_decode.

moe_layer_ffn_noalloc serves callers that may not allocate GPU memory: it keeps
its intermediates in the library's fixed device scratch array.  With every
routed expert resident, moe_layer_decode computes the same layer output; this
test runs both through the C ABI on the same inputs, twice in a row (the
second call reuses the scratch the first one left behind).
"""
import numpy as np
import pytest

from oracle.ffn import relative_max_error
from tests.harness import TOL, torch_act
from workloads import Config, Shape, activations, make_pool, routing_trace

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("wdtype,adtype", [("bf16", "bf16"), ("f32", "f32")])
def test_noalloc_matches_decode_on_two_calls(wdtype, adtype):
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from serving_layer_moe_gb300 import MoECache
    from serving_layer_moe_gb300.binding import ffn_noalloc
    s = Shape(L=1, E=16, k=4, H=512, I=256, wdtype=wdtype, adtype=adtype)
    cfg = Config("noalloc", s, T=8, steps=2, capacity=16, routing="softmax", seed=77)
    arena, offs = make_pool(s, cfg.seed)
    dev = torch.device("cuda", 0)
    experts = torch.from_numpy(arena).to(dev)             # the layer's 16 blobs back to back
    # reference: a cache that fills every routed expert (offload mode, K = E, C = E)
    cache = MoECache(L=1, E=s.E, H=s.H, I=s.I, top_k=s.k, max_tokens=cfg.T, wdtype=wdtype, adtype=adtype,
                     host_pool=torch.from_numpy(arena).pin_memory(), blob_offsets=offs, n_slots=s.E,
                     max_fetch=s.E, bw_pcie_mbps=1000, bw_cpu_mbps=0, device=0)
    ids, w = routing_trace(cfg)
    for call in range(2):
        x = torch_act(activations(cfg, call, 0), dev)
        i_d = torch.from_numpy(ids[call, 0]).to(dev)
        w_d = torch.from_numpy(w[call, 0]).to(dev)
        ref = torch.empty(cfg.T, s.H, device=dev)
        cache.decode(0, x, i_d, w_d, ref)
        got = torch.full((cfg.T, s.H), float("nan"), device=dev)
        ffn_noalloc(experts, x, i_d, w_d, got, E=s.E, H=s.H, I=s.I, top_k=s.k, wdtype=wdtype, adtype=adtype)
        torch.cuda.synchronize()
        g, r = got.cpu().numpy(), ref.cpu().numpy()
        assert np.all(np.isfinite(g))
        assert relative_max_error(g, r) <= TOL
    cache.close()


def test_noalloc_rejects_oversized_calls():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from serving_layer_moe_gb300 import MoEError
    from serving_layer_moe_gb300.binding import ffn_noalloc
    dev = torch.device("cuda", 0)
    T, k, H, I = 1024, 8, 2048, 768            # ~92 MB of scratch needed > 16 MiB
    experts = torch.zeros(16 * 6 * H * I, dtype=torch.uint8, device=dev)
    x = torch.zeros(T, H, dtype=torch.int16, device=dev)
    ids = torch.zeros(T, k, dtype=torch.int32, device=dev)
    w = torch.zeros(T, k, device=dev)
    out = torch.zeros(T, H, device=dev)
    with pytest.raises(MoEError) as ei:
        ffn_noalloc(experts, x, ids, w, out, E=16, H=H, I=I, top_k=k, wdtype="bf16", adtype="bf16")
    assert ei.value.status == 4
