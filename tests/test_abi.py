"""The C-ABI library builds, loads and exports every symbol include/*.h declares.

CPU only: no compute call is made here.
"""

import ctypes
import glob
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_symbols():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(h).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        names |= set(re.findall(r"QWEN_API\s+[\w\s\*]+?\b(qwen_\w+)\s*\(", text))
    return names


@pytest.fixture(scope="module")
def built_lib():
    from transformer_decoder_layer_gb300 import _build
    path = _build.build()
    return path


def test_header_declares_the_boundary():
    names = declared_symbols()
    for must in ("qwen_layer_create", "qwen_layer_prefill", "qwen_layer_decode", "qwen_moe_ffn",
                 "qwen_layer_destroy", "qwen_head_last_token", "qwen_status_string"):
        assert must in names


def test_library_exports_every_declared_symbol(built_lib):
    lib = ctypes.CDLL(built_lib)
    missing = [n for n in sorted(declared_symbols()) if not hasattr(lib, n)]
    assert not missing, f"not exported: {missing}"


def test_binding_signatures_cover_header(built_lib):
    import transformer_decoder_layer_gb300 as q
    assert declared_symbols() == set(q._SIGS), "Python binding and header disagree"
    L = q.lib()
    assert L.qwen_status_string(0) == b"ok"
    assert L.qwen_status_string(6).startswith(b"cache slot")
    assert b"FP16" in L.qwen_status_string(7)
    assert q.STATUS[7] == "QWEN_ERR_OVERFLOW"


def test_config_struct_layout_matches_c(built_lib):
    """Host-only: invalid configs are rejected by the library without a GPU."""
    import transformer_decoder_layer_gb300 as q
    cfg = q.LayerConfig(dict(d=512, n_q_heads=8, n_kv_heads=2, head_dim=64, ffn=1536, qk_norm=1),
                        max_tokens=128, max_batch=1, max_seq=128, max_position=128)
    L = q.lib()
    assert L.qwen_layer_packed_bytes(ctypes.byref(cfg.c)) > 0
    bad = q.LayerConfig(dict(d=512, n_q_heads=8, n_kv_heads=3, head_dim=64, ffn=1536),
                        max_tokens=128, max_batch=1, max_seq=128, max_position=128)
    assert L.qwen_layer_packed_bytes(ctypes.byref(bad.c)) == 0
    dh2 = q.LayerConfig(dict(d=4, n_q_heads=2, n_kv_heads=1, head_dim=2, ffn=6),
                        max_tokens=3, max_batch=1, max_seq=3, max_position=3)
    assert L.qwen_layer_packed_bytes(ctypes.byref(dh2.c)) == 0


def test_shared_expert_config_reaches_the_library(built_lib):
    """Host-only: shared_ffn (the last config field) changes the packed size by
    exactly the shared expert's FP16 weights (its gate row joins the router,
    whose rows are padded to 128 either way), so the field is read where the
    binding writes it."""
    import transformer_decoder_layer_gb300 as q
    L = q.lib()
    d, sf = 512, 512
    moe = dict(d=d, n_q_heads=8, n_kv_heads=2, head_dim=64, ffn=256, n_experts=16, top_k=4)

    def packed(**kw):
        c = q.LayerConfig(dict(moe, **kw), max_tokens=64, max_batch=1, max_seq=64,
                          max_position=64)
        return L.qwen_layer_packed_bytes(ctypes.byref(c.c))

    base = packed()
    assert base > 0
    assert packed(norm_topk_prob=0) == base
    assert packed(shared_ffn=sf, norm_topk_prob=0) - base == 3 * sf * d * 2
    assert packed(shared_ffn=100) == 0            # not a multiple of 64
    assert packed(norm_topk_prob=2) == 0
    dense = q.LayerConfig(dict(d=d, n_q_heads=8, n_kv_heads=2, head_dim=64, ffn=256,
                               shared_ffn=sf), max_tokens=64, max_batch=1, max_seq=64,
                          max_position=64)
    assert L.qwen_layer_packed_bytes(ctypes.byref(dense.c)) == 0  # shared expert needs MoE
