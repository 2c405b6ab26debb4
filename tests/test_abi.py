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
