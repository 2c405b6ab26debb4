"""The layer workspace as the library lays it out, read through the C ABI on
the host (no GPU): every region is 256-byte aligned, no two regions overlap,
all fit in qwen_layer_workspace_bytes, and each buffer the forward pass needs
for a given shape is there with the size its definition gives.

A prefill of one token per sequence once shared offset 0 between the FP16
copies of the call's K and V rows (they were laid out only for T > 1); the
size check on k16 / v16 at T = 1 is the regression test for that."""

import ctypes

import pytest

import synth

q = pytest.importorskip("transformer_decoder_layer_gb300")

SMALL_MOE = synth.LayerConfig(d=512, n_q_heads=8, n_kv_heads=2, head_dim=64, ffn=256, qk_norm=1,
                              n_experts=16, top_k=4, router_bias=1)
SMALL_SHARED = synth.LayerConfig(d=512, n_q_heads=8, n_kv_heads=2, head_dim=64, ffn=128,
                                 qkv_bias=1, n_experts=16, top_k=4, norm_topk_prob=0,
                                 shared_ffn=512)
SHAPES = {"tiny": synth.TINY, "qwen25_7b": synth.QWEN25_7B, "qwen3_8b": synth.QWEN3_8B,
          "small_moe": SMALL_MOE, "small_shared": SMALL_SHARED,
          "qwen3_30b_a3b": synth.QWEN3_30B_A3B, "qwen2_57b_a14b": synth.QWEN2_57B_A14B}
SIZES = [(1, 1), (2, 1), (3, 1), (64, 1), (1, 2), (3, 5), (1, 128), (8, 1024), (1, 4096)]


def _cfg(shape):
    return q.LayerConfig(shape, max_tokens=16384, max_batch=64, max_seq=16384,
                         max_position=16384)


@pytest.mark.parametrize("name", sorted(SHAPES))
@pytest.mark.parametrize("B,T", SIZES)
def test_regions_are_disjoint_aligned_and_complete(name, B, T):
    shape = SHAPES[name]
    cfg = _cfg(shape)
    regs = q.workspace_regions(cfg, B, T)
    total = q.lib().qwen_layer_workspace_bytes(ctypes.byref(cfg.c), B, T)
    names = [r[0] for r in regs]
    assert len(set(names)) == len(names)
    prev_end = 0
    for n, off, size in sorted(regs, key=lambda r: r[1]):
        assert off % 256 == 0, n
        assert size > 0, n
        assert off >= prev_end, f"{n} overlaps the region before it"
        prev_end = off + size
    assert prev_end <= total

    M, d, dh = B * T, shape.d, shape.head_dim
    by = {n: size for n, _, size in regs}
    need = {"xh": M * d * 2, "q": M * shape.n_q_heads * dh * 2,
            "k16": M * shape.n_kv_heads * dh * 2, "v16": M * shape.n_kv_heads * dh * 2,
            "attn": M * shape.n_q_heads * dh * 2, "r32": M * d * 4}
    for n, size in need.items():
        assert by.get(n) == size, f"{n}: {by.get(n)} bytes, expected {size}"
    if shape.n_experts:
        for n in ("logits", "topk_idx", "topk_w", "offsets", "perm", "inv", "zp", "hp", "yp"):
            assert n in by, n
        assert by["z"] == M * d * 2 * 2  # [Z_hi | Z_lo]
        assert by["topk_idx"] == M * shape.top_k * 4
    else:
        assert by["h"] == M * shape.ffn * 2
    if shape.shared_ffn:
        assert by["hs"] == M * shape.shared_ffn * 2 and by["ys32"] == M * d * 4
    for n in ("part", "attn_o", "attn_ml"):  # split-K / split-KV partials
        assert (n in by) == (T == 1), n


def test_region_query_rejects_bad_sizes():
    cfg = _cfg(synth.TINY)
    for B, T in ((0, 1), (1, 0), (-1, 4)):
        with pytest.raises(ValueError):
            q.workspace_regions(cfg, B, T)
    n = q.lib().qwen_layer_workspace_regions(ctypes.byref(cfg.c), 1, 1, None, 0)
    assert n > 0
    assert q.lib().qwen_layer_workspace_regions(ctypes.byref(cfg.c), 1, 1, None, 1) == -1
