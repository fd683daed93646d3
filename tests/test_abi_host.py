"""Host-side checks of the C-ABI library (no GPU needed): it loads, exports
every symbol include/df_moe.h declares, computes span sizes, and rejects bad
configurations before touching a device."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_symbols():
    text = open(os.path.join(ROOT, "include", "df_moe.h")).read()
    return sorted(set(re.findall(r"DF_MOE_API\s+[\w\s\*]+?\b(df_moe_\w+)\s*\(", text)))


@pytest.fixture(scope="module")
def dfm():
    import __graft_entry__
    __graft_entry__.build()
    import mxfp4_routed_expert_top_gb300 as m
    return m


def test_header_declares_the_boundary():
    syms = declared_symbols()
    for name in ["df_moe_create", "df_moe_load_experts", "df_moe_forward",
                 "df_moe_destroy", "df_moe_expert_span_bytes", "df_moe_last_error"]:
        assert name in syms


def test_library_exports_every_declared_symbol(dfm):
    L = dfm.lib()
    syms = declared_symbols()
    assert syms == sorted(dfm.SYMBOLS)
    for name in syms:
        assert hasattr(L, name), name


def test_span_bytes(dfm):
    assert dfm.span_bytes_for(7168, 1536) == 17547264
    assert dfm.span_bytes_for(256, 64) == 3 * (256 * 64 // 2 + 256 * 64 // 32)
    assert dfm.span_bytes_for(0, 64) == 0


def test_create_rejects_bad_config(dfm):
    base = dict(hidden=256, n_experts=8, top_k=2, inter=64, n_shared=1,
                shared_inter=64, max_tokens=1)
    bad = [dict(hidden=255), dict(inter=48), dict(top_k=9), dict(top_k=0),
           dict(n_experts=2000), dict(max_tokens=0), dict(n_shared=9),
           dict(flags=32),                                   # unknown flag
           dict(flags=dfm.MXFP8_ACT),                        # inter 64: not a multiple of 128
           dict(flags=dfm.MXFP8_ACT | dfm.PREFILL_MMA_SYNC, inter=128),
           dict(flags=dfm.MXFP8_ACT | dfm.PLANES, inter=128),
           dict(flags=dfm.PLANES)]                           # inter 64 again
    for b in bad:
        cfg = dict(base, **b)
        with pytest.raises(dfm.DfMoeError) as ei:
            dfm.MoE(**cfg)
        assert ei.value.code == -1, b


def test_null_handle_calls_are_safe(dfm):
    L = dfm.lib()
    L.df_moe_destroy(None)
    assert L.df_moe_forward(None, None, 1, None, None, None, None, None, None) == -1
    assert L.df_moe_expert_span_bytes(None) == 0
    assert isinstance(L.df_moe_last_error(None), bytes)
