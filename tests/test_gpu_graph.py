"""The layer inside a CUDA graph: every call of the forward and the backward
only enqueues work on the caller's stream (kernels and memsets, no host
round trip, no allocation), so a captured forward or forward+backward replays
to the same bits as the direct calls.  The first call of each kind runs
before the capture (it sets the kernels' attributes once per process)."""
import pytest
import torch

from combine_top_routing_gb300 import inputs as I
from combine_top_routing_gb300 import mok
from mokhelp import make_layer

pytestmark = pytest.mark.gpu

CASES = {
    # d a multiple of 256: the fused kernel on CTA pairs, gather-first plan
    "mx_pairs": I.Workload("graph_mx", T=1024, d=512, E=16, k=4, F=256, dtype="mxfp8",
                           router="sigmoid", seed=71),
    "bf16": I.Workload("graph_bf16", T=640, d=256, E=8, k=2, F=384, dtype="bf16",
                       router="softmax", seed=72),
    # several sources and a capped ring: the split-gather plan
    "mx_ring": I.Workload("graph_mx_ring", T=2048, d=512, E=32, k=8, F=384, dtype="mxfp8",
                          router="sigmoid", seed=73, n_sources=8, ring_bytes=512 * (512 + 16)),
}


def _grads(layer):
    return [layer.dX.clone(), layer.dgates.clone(), layer.dW_r.clone()] + [g.clone() for g in layer.grads.values()]


@pytest.mark.parametrize("name", list(CASES))
def test_forward_graph_replays_the_same_bits(name):
    w = CASES[name]
    layer, _ = make_layer(w)
    want = layer.forward().clone()
    torch.cuda.synchronize()
    assert layer.status() == 0
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        layer.forward()
    for _ in range(2):
        layer.out.fill_(0)
        g.replay()
        torch.cuda.synchronize()
        assert layer.status() == 0
        assert torch.equal(layer.out.view(torch.int16), want.view(torch.int16))


@pytest.mark.parametrize("name", ["mx_pairs", "bf16"])
def test_forward_backward_graph_replays_the_same_bits(name):
    w = CASES[name]
    layer, inp = make_layer(w, training=True)
    layer.prepare_backward()
    layer.forward()
    layer.backward(inp["dY"])
    torch.cuda.synchronize()
    assert layer.status() == 0 and mok.get_device_status(layer.bws) == 0
    want = _grads(layer)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        layer.forward()
        layer.backward(inp["dY"])
    for t in [layer.dX, layer.dgates, layer.dW_r] + list(layer.grads.values()):
        t.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert layer.status() == 0 and mok.get_device_status(layer.bws) == 0
    for got, ref in zip(_grads(layer), want):
        assert torch.equal(got.view(torch.uint8), ref.view(torch.uint8))
