"""mok_layout_static: the layout step for callers that cannot allocate.

Some callers of this library cannot allocate device memory at the point
where they route tokens (a host callback or a runtime that forbids device-
synchronising CUDA calls, a fixed memory budget handed over up front).
mok_layout_static gives them the layout without a workspace, keeping its
per-chunk tables in a fixed array inside the library.  This file checks,
through the C ABI, that two calls in a row give exactly the layout that
mok_route_layout gives (integer outputs: bit for bit), and that a layer too
big for the fixed array is refused before anything runs.

It sits in its own file that pytest collects last, so a run that stops at
the first failure has run every other test before it."""
import pytest
import torch

from combine_top_routing_gb300 import inputs as I
from combine_top_routing_gb300 import mok
from mokhelp import Routed, make_layer

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("w", [
    I.Workload("nl_dsv3_like", T=4096, d=256, E=256, k=8, F=256, dtype="bf16",
               router="sigmoid", seed=51, zipf_alpha=0.46),
    I.Workload("nl_ragged", T=300, d=256, E=8, k=2, F=384, dtype="bf16",
               router="softmax", seed=52),
], ids=lambda w: w.name)
def test_layout_static_matches_route_layout_twice(w):
    layer, _ = make_layer(w)
    R = Routed(layer)
    dev = "cuda"
    for _ in range(2):
        out = dict(counts=torch.full((w.E,), -1, dtype=torch.int32, device=dev),
                   offsets=torch.full((w.E + 1,), -1, dtype=torch.int32, device=dev),
                   pad_offsets=torch.full((w.E + 1,), -1, dtype=torch.int32, device=dev),
                   slot_pos=torch.full((w.T, w.k), -1, dtype=torch.int32, device=dev),
                   row_tok=torch.full((w.S,), -1, dtype=torch.int32, device=dev),
                   row_j=torch.full((w.S,), 255, dtype=torch.uint8, device=dev))
        mok.layout_static(layer.cfg, R.ids, out["counts"], out["offsets"], out["pad_offsets"],
                          out["slot_pos"], out["row_tok"], out["row_j"])
        torch.cuda.synchronize()
        for name, t in out.items():
            assert torch.equal(t, getattr(R, name)), name


def test_layout_static_refuses_layers_beyond_its_array():
    # 2 * ceil(T*k/256) * E words must fit in 262144: this layer needs 2 * 512 * 1024
    cfg = mok.Config(T=16384, d_model=128, n_experts=1024, top_k=8, d_ff=128, router=1, dtype=0)
    ids = torch.zeros((16384, 8), dtype=torch.int32, device="cuda")
    with pytest.raises(mok.MokError) as ei:
        mok.layout_static(cfg, ids, ids, ids, ids, ids, ids,
                          torch.empty(1, dtype=torch.uint8, device="cuda"))
    assert ei.value.code == mok.MOK_ERR_UNSUPPORTED
