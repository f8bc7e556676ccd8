"""The C ABI without a GPU: the library builds and loads, exports every entry
point include/mok.h declares, and rejects bad configurations on the host."""
import ctypes
import os
import re

import pytest

from combine_top_routing_gb300 import mok

HEADER = os.path.join(os.path.dirname(os.path.dirname(__file__)), "include", "mok.h")


def _declared():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(mok_[a-z_]+)\s*\(", text)))


def test_header_declares_expected_entry_points():
    names = _declared()
    for want in ("mok_route_layout", "mok_dispatch", "mok_expert_ffn", "mok_combine",
                 "mok_moe_forward", "mok_moe_backward", "mok_workspace_size",
                 "mok_status_string", "mok_get_device_status"):
        assert want in names


def test_library_exports_every_declared_symbol():
    L = mok.lib()
    for name in _declared():
        assert hasattr(L, name), name
    assert set(_declared()) <= set(mok.EXPORTS)


def _cfg(**kw):
    base = dict(T=256, d_model=256, n_experts=8, top_k=2, d_ff=256, router=0, dtype=0)
    base.update(kw)
    return mok.Config(**base)


def test_workspace_size_valid_and_monotone():
    small = mok.workspace_size(_cfg())
    big = mok.workspace_size(_cfg(T=4096))
    assert all(s > 0 for s in small)
    assert all(b > s for b, s in zip(big, small))
    assert mok.max_padded_rows(_cfg()) == 512 + 8 * 128


def test_empty_batch_is_a_valid_config():
    """T = 0 (no tokens) is accepted: the workspaces still hold the per-expert
    layout and the status word; T = 0 spread over several sources is not a
    layout of sources (each holds at least one 128-row piece)."""
    assert all(s > 0 for s in mok.workspace_size(_cfg(T=0)))
    assert mok.max_padded_rows(_cfg(T=0)) == 8 * 128
    with pytest.raises(mok.MokError) as ei:
        mok.workspace_size(_cfg(T=0, n_sources=2, source_rows=[128, 128]))
    assert ei.value.code == mok.MOK_ERR_INVALID_ARG


@pytest.mark.parametrize("kw,code", [
    (dict(T=-1), mok.MOK_ERR_INVALID_ARG),
    (dict(top_k=9, n_experts=16), mok.MOK_ERR_UNSUPPORTED),
    (dict(top_k=4, n_experts=2), mok.MOK_ERR_UNSUPPORTED),
    (dict(n_experts=2048), mok.MOK_ERR_UNSUPPORTED),
    (dict(d_model=200), mok.MOK_ERR_UNSUPPORTED),
    (dict(d_ff=100), mok.MOK_ERR_UNSUPPORTED),
    (dict(router=5), mok.MOK_ERR_INVALID_ARG),
    (dict(dtype=7), mok.MOK_ERR_INVALID_ARG),
    (dict(minibatch_rows=100), mok.MOK_ERR_INVALID_ARG),
    (dict(gather_sm_fraction=1.5), mok.MOK_ERR_INVALID_ARG),
    (dict(gather_sm_fraction=-0.5), mok.MOK_ERR_INVALID_ARG),
    (dict(fused_cta_pairs=3), mok.MOK_ERR_INVALID_ARG),
    (dict(gemm_cta_pairs=-1), mok.MOK_ERR_INVALID_ARG),
])
def test_bad_configs_rejected_on_host(kw, code):
    with pytest.raises(mok.MokError) as ei:
        mok.workspace_size(_cfg(**kw))
    assert ei.value.code == code


def test_sources_must_cover_tokens_in_128_row_pieces():
    with pytest.raises(mok.MokError) as ei:
        mok.workspace_size(_cfg(T=512, n_sources=4, source_rows=[128, 128, 128, 256]))
    assert ei.value.code == mok.MOK_ERR_INVALID_ARG
    with pytest.raises(mok.MokError) as ei:
        mok.workspace_size(_cfg(T=400, n_sources=2, source_rows=[200, 200]))
    assert ei.value.code == mok.MOK_ERR_UNSUPPORTED
    assert mok.workspace_size(_cfg(T=512, n_sources=4, source_rows=[128] * 4))[0] > 0


def test_null_pointers_rejected_before_any_launch():
    L = mok.lib()
    cfg = _cfg()
    rc = L.mok_combine(cfg.ref, None, None, None, None)
    assert rc == mok.MOK_ERR_INVALID_ARG
    rc = L.mok_quantize_mx(None, 1, 128, 128, 0, None, None, None)
    assert rc == mok.MOK_ERR_INVALID_ARG
    rc = L.mok_get_device_status(None, None)
    assert rc == mok.MOK_ERR_INVALID_ARG
    rc = L.mok_swiglu_quantize_mx(None, None, 128, 128, None, None, None, None)
    assert rc == mok.MOK_ERR_INVALID_ARG
    dummy = ctypes.c_void_p(16)  # never dereferenced: the shape check fails first
    rc = L.mok_swiglu_quantize_mx(dummy, dummy, 100, 128, None, dummy, dummy, None)
    assert rc == mok.MOK_ERR_UNSUPPORTED


def test_status_strings():
    assert mok.status_string(0) == "MOK_OK"
    assert mok.status_string(4) == "MOK_ERR_TIMEOUT"
    assert mok.status_string(99) == "MOK_ERR_UNKNOWN"


def test_saved_ctx_layout_is_aligned_and_ordered():
    lay = mok.saved_ctx_layout(_cfg())
    fields = [f for f, _ in mok.MokCtxLayout._fields_]
    offs = [getattr(lay, f) for f in fields]
    assert all(o % 256 == 0 for o in offs)
    assert offs == sorted(offs)


def test_bwd_ws_layout_inside_the_backward_workspace():
    for dtype in (0, 1):
        cfg = _cfg(dtype=dtype, T=300)
        lay = mok.bwd_ws_layout(cfg)
        offs = [getattr(lay, f) for f, _ in mok.MokBwdLayout._fields_]
        assert all(o % 256 == 0 for o in offs) and offs == sorted(offs)
        assert lay.total == mok.workspace_size(cfg)[2]
        R = mok.max_padded_rows(cfg)
        assert lay.da - lay.dy >= R * 256 * 2 and lay.dx - lay.db >= R * 256 * 2
        assert lay.total - lay.dl_sel >= 300 * 2 * 4


def _plan(**kw):
    return mok.fused_plan(_cfg(**kw))


def test_fused_plan_honours_explicit_knobs():
    # d = 384: one CTA per tile, gather CTAs = round(fraction x CTAs)
    p = _plan(gather_sm_fraction=0.25, minibatch_rows=64, ring_bytes=1 << 20, T=4096, d_model=384)
    assert p["gather_ctas"] == int(0.25 * p["ctas"] + 0.5)
    assert p["minibatch_rows"] == 64
    # 1 MiB of BF16 rows of 384 elements = 1365 rows -> 1280 (multiple of 256)
    assert p["ring_rows"] == 1280
    # d = 256, BF16: CTA pairs, an even CTA count and gather CTAs rounded up to a pair
    q = _plan(gather_sm_fraction=0.25, ring_bytes=1 << 20, T=4096)
    assert q["cta_pairs"] == 1 and p["cta_pairs"] == 0
    assert q["ctas"] % 2 == 0 and q["gather_ctas"] % 2 == 0
    assert q["gather_ctas"] == (int(0.25 * q["ctas"] + 0.5) + 1) // 2 * 2
    # 1 MiB of BF16 rows of 256 elements = 2048 rows; an uncapped ring holds every padded row
    assert q["ring_rows"] == 2048
    assert _plan()["ring_rows"] == mok.max_padded_rows(_cfg())
    # MXFP8 layers whose experts average under 384 rows and rings below 512 rows
    # run one CTA per tile by default; the config forces either where the shape allows
    assert _plan(dtype=1)["cta_pairs"] == 0
    assert _plan(dtype=1, T=8 * 384 // 2, top_k=2)["cta_pairs"] == 1
    assert _plan(ring_bytes=256 * 256 * 2, T=4096)["cta_pairs"] == 0
    assert _plan(dtype=1, fused_cta_pairs=mok.MOK_PAIRS_ON)["cta_pairs"] == 1
    assert _plan(fused_cta_pairs=mok.MOK_PAIRS_OFF)["cta_pairs"] == 0
    assert _plan(d_model=384, fused_cta_pairs=mok.MOK_PAIRS_ON)["cta_pairs"] == 0


def test_fused_plan_shape_rules():
    # gather share: per-row gather time over per-row FFN1 time grows as F shrinks
    # (a capped ring keeps the split gather)
    cap = dict(ring_bytes=64 << 20)
    wide = _plan(d_model=4096, d_ff=14336, n_experts=8, top_k=2, T=8192, **cap)
    narrow = _plan(d_model=7168, d_ff=2048, n_experts=256, top_k=8, T=16384, dtype=1, **cap)
    for p in (wide, narrow):
        assert p["ctas"] / 16 - 1 <= p["gather_ctas"] <= p["ctas"] / 3 + 1
    assert narrow["gather_ctas"] > wide["gather_ctas"]
    # uncapped ring: every CTA gathers first where the split would give the
    # gather role 1/8 of the CTAs or more (the DeepSeek-V3 shape), not otherwise
    narrow_u = _plan(d_model=7168, d_ff=2048, n_experts=256, top_k=8, T=16384, dtype=1)
    wide_u = _plan(d_model=4096, d_ff=14336, n_experts=8, top_k=2, T=8192)
    assert narrow_u["gather_ctas"] == narrow_u["ctas"] and narrow_u["minibatch_rows"] == 0
    assert 8 * narrow["gather_ctas"] >= narrow["ctas"]
    assert wide_u["gather_ctas"] == wide["gather_ctas"] < wide_u["ctas"] / 8
    # an explicit share of 1 with an uncapped ring
    full = _plan(gather_sm_fraction=1.0)
    assert full["gather_ctas"] == full["ctas"]
    # minibatch: the smallest of 64/128/256 rows for which one gather round
    # (a minibatch per gather CTA) hands over two waves of FFN1 tiles
    for F in (128, 512, 2048, 14336):
        for frac in (0.0625, 0.25):
            p = _plan(d_ff=F, d_model=1024, gather_sm_fraction=frac, ring_bytes=64 << 20)
            g, gemm = p["gather_ctas"], p["ctas"] - p["gather_ctas"]
            want = next((mb for mb in (64, 128) if g * mb * (F // 128) >= 2 * 128 * gemm), 256)
            assert p["minibatch_rows"] == want, (F, frac, p)
