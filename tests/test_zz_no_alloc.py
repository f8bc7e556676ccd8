"""mok_layout_static: the layout step for callers that cannot allocate.

Some callers of this library cannot allocate device memory at the point
where they route tokens (a host callback or a runtime that forbids device-
synchronising CUDA calls, a fixed memory budget handed over up front).
mok_layout_static gives them the layout without a workspace, keeping its
per-chunk tables in a fixed array inside the library.  This file checks,
through the C ABI, that two calls in a row give exactly the layout that
mok_route_layout gives (integer outputs: bit for bit), also for a layer that
fills the array exactly, that a layer one chunk too big for it is refused
before anything runs, and that routing ids outside [0, E) -- this call takes
them from the caller -- are flagged instead of indexing anything.

It sits in its own file that pytest collects last, so a run that stops at
the first failure has run every other test before it."""
import numpy as np
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
    for _ in range(2):
        out = _outputs(w)
        mok.layout_static(layer.cfg, R.ids, out["counts"], out["offsets"], out["pad_offsets"],
                          out["slot_pos"], out["row_tok"], out["row_j"])
        torch.cuda.synchronize()
        for name, t in out.items():
            assert torch.equal(t, getattr(R, name)), name


def test_layout_static_fills_its_array_exactly():
    """2 * ceil(T*k/256) * E = 2 * 128 * 1024 = 262144 words: the whole array,
    still the exact layout of mok_route_layout."""
    w = I.Workload("nl_full_array", T=4096, d=128, E=1024, k=8, F=128, dtype="bf16",
                   router="sigmoid", seed=53)
    layer, _ = make_layer(w)
    R = Routed(layer)
    out = _outputs(w)
    mok.layout_static(layer.cfg, R.ids, out["counts"], out["offsets"], out["pad_offsets"],
                      out["slot_pos"], out["row_tok"], out["row_j"])
    torch.cuda.synchronize()
    for name, t in out.items():
        assert torch.equal(t, getattr(R, name)), name


def test_layout_static_refuses_one_chunk_beyond_its_array():
    # T*k = 32776 slots -> 129 chunks of 256 -> 2 * 129 * 1024 = 264192 words
    cfg = mok.Config(T=4097, d_model=128, n_experts=1024, top_k=8, d_ff=128, router=1, dtype=0)
    ids = torch.zeros((4097, 8), dtype=torch.int32, device="cuda")
    with pytest.raises(mok.MokError) as ei:
        mok.layout_static(cfg, ids, ids, ids, ids, ids, ids,
                          torch.empty(1, dtype=torch.uint8, device="cuda"))
    assert ei.value.code == mok.MOK_ERR_UNSUPPORTED


def test_layout_static_flags_ids_out_of_range():
    """Ids outside [0, E) are checked on the device: such a slot is placed
    nowhere (slot_pos -1), offsets[E] is -1, and the valid slots keep the
    stable layout among themselves."""
    T, k, E = 300, 2, 8
    g = torch.Generator(device="cpu").manual_seed(54)
    ids = torch.randint(0, E, (T, k), generator=g, dtype=torch.int32)
    bad = torch.zeros((T, k), dtype=torch.bool)
    bad[torch.randint(0, T, (12,), generator=g), torch.randint(0, k, (12,), generator=g)] = True
    ids[bad] = torch.tensor([-1, E, 1 << 30, -(1 << 30)], dtype=torch.int32).repeat(12)[:int(bad.sum())]
    cfg = mok.Config(T=T, d_model=128, n_experts=E, top_k=k, d_ff=128, router=0, dtype=0)
    w = I.Workload("nl_bad_ids", T=T, d=128, E=E, k=k, F=128, dtype="bf16", router="softmax", seed=54)
    out = _outputs(w)
    mok.layout_static(cfg, ids.cuda(), out["counts"], out["offsets"], out["pad_offsets"],
                      out["slot_pos"], out["row_tok"], out["row_j"])
    torch.cuda.synchronize()
    flat, badf = ids.reshape(-1).numpy(), bad.reshape(-1).numpy()
    good = ~badf
    counts = np.bincount(flat[good], minlength=E)
    assert np.array_equal(out["counts"].cpu().numpy(), counts)
    offsets = out["offsets"].cpu().numpy()
    assert offsets[E] == -1
    assert np.array_equal(offsets[:E], np.concatenate([[0], np.cumsum(counts)[:-1]]))
    slot_pos = out["slot_pos"].cpu().numpy().reshape(-1)
    assert np.all(slot_pos[badf] == -1)
    # valid slots: stable by slot index within each expert
    order = np.argsort(flat[good], kind="stable")
    want = np.empty(good.sum(), dtype=np.int64)
    want[order] = np.arange(good.sum())
    assert np.array_equal(slot_pos[good], want)
    row_tok = out["row_tok"].cpu().numpy()[:good.sum()]
    assert np.array_equal(row_tok[want], np.nonzero(good)[0] // k)


def _outputs(w):
    dev = "cuda"
    return dict(counts=torch.full((w.E,), -1, dtype=torch.int32, device=dev),
                offsets=torch.full((w.E + 1,), -1, dtype=torch.int32, device=dev),
                pad_offsets=torch.full((w.E + 1,), -1, dtype=torch.int32, device=dev),
                slot_pos=torch.full((w.T, w.k), -1, dtype=torch.int32, device=dev),
                row_tok=torch.full((w.S,), -1, dtype=torch.int32, device=dev),
                row_j=torch.full((w.S,), 255, dtype=torch.uint8, device=dev))


def test_layout_static_refuses_layers_beyond_its_array():
    # 2 * ceil(T*k/256) * E words must fit in 262144: this layer needs 2 * 512 * 1024
    cfg = mok.Config(T=16384, d_model=128, n_experts=1024, top_k=8, d_ff=128, router=1, dtype=0)
    ids = torch.zeros((16384, 8), dtype=torch.int32, device="cuda")
    with pytest.raises(mok.MokError) as ei:
        mok.layout_static(cfg, ids, ids, ids, ids, ids, ids,
                          torch.empty(1, dtype=torch.uint8, device="cuda"))
    assert ei.value.code == mok.MOK_ERR_UNSUPPORTED
