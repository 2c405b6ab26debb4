"""The oracle's closed-form counter against the totals the pages print."""

import pytest

from oracle import counts as C

Q7 = dict(L=28, d=3584, n_q=28, n_kv=4, dh=128, f=18944, vocab=152064)


def test_qwen25_7b_totals(golden):
    g = golden["qwen25_7b"]
    total = C.dense_model_params(**Q7)
    assert total == g["total_params"]
    assert total - Q7["vocab"] * Q7["d"] == g["matmul_params_incl_norm_bias"]
    assert total - 2 * Q7["vocab"] * Q7["d"] == g["backbone_params"]
    assert C.attn_params(3584, 28, 4, 128) == g["attn_per_layer"]
    assert C.qkv_bias_params(28, 4, 128) == g["qkv_bias_per_layer"]
    assert C.mlp_params(3584, 18944) == g["mlp_per_layer"]
    assert C.layer_norm_params(3584) == g["norm_per_layer"]
    assert 28 * C.layer_norm_params(3584) == g["layer_norms_total"]
    assert 28 * C.qkv_bias_params(28, 4, 128) == g["qkv_bias_total"]
    # 2 FLOPs per matmul weight per token
    assert round(2 * g["matmul_params_incl_norm_bias"] / 1e9, 2) == g["gflop_per_token"]
    assert round(2 * g["backbone_params"] / 1e9, 2) == g["backbone_gflop_per_token"]
    assert round(2 * g["embed_tokens"] / 1e9, 2) == g["lm_head_gflop_per_token"]
    assert round(C.linear_flops(1, 3584 * 3584) / 1e6, 2) == g["q_proj_mflop_per_token"]
    assert C.kv_bytes_per_token(28, 4, 128) == g["kv_bytes_per_token"]


def test_p4_counter_table(golden):
    """Transformer 的 Infra 视角 §4: the table leaves norms and biases out."""
    g = golden["qwen25_7b_p4_counter"]
    attn_all = 28 * C.attn_params(3584, 28, 4, 128)
    ffn_all = 28 * C.mlp_params(3584, 18944)
    assert attn_all == g["all_attention"] and ffn_all == g["all_ffn"]
    total = C.dense_model_params(**Q7, bias=False, final_norm=False) - 28 * 2 * 3584
    assert total == g["total"]
    assert C.dense_model_params(**Q7) - total == 333312
    assert round(2 * ffn_all / 1e9, 2) == g["ffn_gflop_per_token"]
    assert round(2 * attn_all / 1e9, 2) == g["attn_gflop_per_token"]


def test_attention_constants(golden):
    g = golden["qwen25_7b_attention_constants"]
    assert C.attention_flops_prefill_causal(28, 28, 128, 1) == g["prefill_causal_per_S2"]
    assert C.attention_flops_decode(28, 28, 128, 1) == g["decode_per_T"]
    s = 8192
    summed = sum(C.attention_flops_decode(28, 28, 128, t) for t in range(s))
    assert summed == pytest.approx(g["S8192_sum_decode"], rel=1e-4)
    assert C.attention_flops_prefill_causal(28, 28, 128, s) == pytest.approx(
        g["S8192_prefill_formula"], rel=1e-4)


def test_flop_counter_cross_check(golden):
    """Qwen2.5-7B 结构拆解 §03.9: 1024 in / 256 out."""
    g = golden["qwen25_7b_flop_counter_check"]
    backbone = 2 * golden["qwen25_7b"]["backbone_params"]
    lm = 2 * golden["qwen25_7b"]["embed_tokens"]
    bb = 1280 * backbone / 1e9
    lh = 257 * lm / 1e9
    ap = C.attention_flops_prefill_causal(28, 28, 128, 1024) / 1e9
    ad = sum(C.attention_flops_decode(28, 28, 128, t) for t in range(1024, 1280)) / 1e9
    assert round(bb, 1) == g["backbone_gflop"]
    assert round(lh, 1) == g["lm_head_gflop"]
    assert round(ap, 1) == g["attn_prefill_gflop"]
    assert round(ad, 1) == g["attn_decode_gflop"]
    assert round(bb + lh + ap + ad, 1) == g["total_gflop"]
    assert round((bb + lh + ap + ad) / 256, 2) == g["gflop_per_output_token"]


def test_kv_reuse_savings(golden):
    """§09.1: T=1152 with and without the cache (rounded backbone 13.05 GFLOP)."""
    g = golden["qwen25_7b_kv_reuse"]
    t = 1152
    with_cache = 13.05e9 + C.attention_flops_decode(28, 28, 128, t)
    without = t * 13.05e9 + C.attention_flops_prefill_causal(28, 28, 128, t)
    assert round(with_cache / 1e10, 2) == 1.35 and round(without / 1e13, 2) == 1.53
    assert round(without / with_cache) == g["ratio"]
    for tt, gb in g["kv_read_gb"].items():
        assert round(int(tt) * C.kv_bytes_per_token(28, 4, 128) / 1e9, 3) == gb


def test_qwen3_8b_layer(golden):
    """推理系统 03 §11-§12."""
    g = golden["qwen3_8b_layer"]
    pa = C.attn_params(4096, 32, 8, 128)
    pm = C.mlp_params(4096, 12288)
    assert pa == g["p_attn"] and pm == g["p_mlp"] and pa + pm == g["p_linear"]
    assert C.layer_norm_params(4096, 128, qk_norm=True) == g["norm_params"]
    assert pa + pm + g["norm_params"] == g["p_layer"]
    assert round(pm / (pa + pm), 3) == g["mlp_share"]
    assert round(C.linear_flops(128, pa + pm) / 1e9, 2) == g["linear_gflop_T128"]
    assert round(C.attention_flops_dense(32, 128, 128) / 1e9, 3) == g["dense_attention_gflop_T128"]
    assert C.kv_bytes_per_token(1, 8, 128) == g["kv_bytes_per_layer_position"]
    assert C.kv_bytes_per_token(36, 8, 128) == g["kv_kib_36_layers"] * 1024


def test_qwen2_57b_a14b(golden):
    """Qwen2.5-7B 结构拆解 §10.1, §10.3."""
    g = golden["qwen2_57b_a14b"]
    d, E, k, mf, sf = 3584, 64, 8, 2560, 20480
    assert 3 * d * sf + d == g["shared_expert_per_layer"]
    assert k * 3 * d * mf == g["routed_active_per_layer"]
    assert d * E == g["router_per_layer"]
    assert C.moe_block_active_params(d, E, k, mf, sf) == g["ffn_active_per_layer"]
    kw = dict(L=28, d=d, n_q=28, n_kv=4, dh=128, E=E, k=k, mf=mf, sf=sf, vocab=152064)
    assert C.moe_model_params(**kw) == g["total_params"]
    assert C.moe_model_params(**kw, active=True) == g["active_params"]


def test_qwen3_30b_a3b_layer(golden):
    """MoE 初步 (lecture01), 每层参数量."""
    g = golden["qwen3_30b_a3b_layer"]
    assert C.attn_params(2048, 32, 4, 128) == g["p_attn"]
    assert 2048 * 128 == g["p_router"]
    assert C.moe_block_params(2048, 128, 768) - 2048 * 128 == g["p_experts"]


def test_touched_experts_limits():
    """Qwen2.5-7B 结构拆解 §11.1: B=1 touches k experts; large B touches all E."""
    assert C.touched_experts(128, 8, 1) == pytest.approx(8.0)
    assert C.touched_experts(128, 8, 4096) == pytest.approx(128.0)
