"""Seeded synthetic inputs shared by the oracle tests, the GPU tests and bench.py.

This module holds none of the decoder layer's arithmetic: it only draws seeded
normal numbers on the CPU (torch's CPU generator, float32) and rounds them to
BF16, so both the FP64 oracle and the CUDA library read bit-identical inputs.

Recipe (all seeded, per-tensor seed = crc32("<tag>/<name>") + base):
* activations X ~ N(0, 1);
* projection / expert / router / lm_head weights ~ N(0, 0.02), stored [out, in];
* qkv biases ~ N(0, 0.02); router per-expert bias ~ N(0, 0.5) (skews loads);
* RMSNorm and QK-norm gammas ~ 1 + N(0, 0.1);
* a pre-filled KV cache holds N(0, 1) in its filled slots, zeros elsewhere.
"""

from __future__ import annotations

import dataclasses
import zlib

import torch


@dataclasses.dataclass(frozen=True)
class LayerConfig:
    """Shape of one decoder layer (mirrors the C struct ``qwen_layer_config``)."""
    d: int
    n_q_heads: int
    n_kv_heads: int
    head_dim: int
    ffn: int                 # f (dense) or per-expert width mf (MoE)
    qkv_bias: int = 0
    qk_norm: int = 0
    rope_theta: float = 1.0e6
    rms_eps: float = 1.0e-6
    n_experts: int = 0       # 0 = dense MLP
    top_k: int = 0
    norm_topk_prob: int = 1
    router_bias: int = 0
    shared_ffn: int = 0      # width of the shared expert (Qwen2-MoE); 0 = none

    def as_dict(self):
        return dataclasses.asdict(self)


# The named layer shapes of the workloads (random-init weights, no checkpoints).
TINY = LayerConfig(d=512, n_q_heads=8, n_kv_heads=2, head_dim=64, ffn=1536, qk_norm=1)
TOY = LayerConfig(d=4, n_q_heads=2, n_kv_heads=1, head_dim=2, ffn=6)
QWEN25_7B = LayerConfig(d=3584, n_q_heads=28, n_kv_heads=4, head_dim=128, ffn=18944,
                        qkv_bias=1)
QWEN3_8B = LayerConfig(d=4096, n_q_heads=32, n_kv_heads=8, head_dim=128, ffn=12288,
                       qk_norm=1)
QWEN3_30B_A3B = LayerConfig(d=2048, n_q_heads=32, n_kv_heads=4, head_dim=128, ffn=768,
                            qk_norm=1, n_experts=128, top_k=8, norm_topk_prob=1,
                            router_bias=1)
# Qwen2-57B-A14B MoE layer: 64 experts, top-8, mf=2560, a shared expert of width
# 20480 with a sigmoid gate, weights without renormalisation; attention shapes
# those of Qwen2.5-7B ("Qwen2.5-7B 结构拆解" §10, §10.1).
QWEN2_57B_A14B = LayerConfig(d=3584, n_q_heads=28, n_kv_heads=4, head_dim=128, ffn=2560,
                             qkv_bias=1, n_experts=64, top_k=8, norm_topk_prob=0,
                             shared_ffn=20480)
QWEN25_7B_VOCAB = 152064
QWEN25_7B_LAYERS = 28


def seed_for(tag: str, name: str, base: int = 0) -> int:
    return (zlib.crc32(f"{tag}/{name}".encode()) + base) & 0x7FFFFFFF


def normal_bf16(shape, seed: int, std: float = 1.0, mean: float = 0.0) -> torch.Tensor:
    """N(mean, std^2) drawn in float32 on the CPU generator, rounded to BF16."""
    g = torch.Generator(device="cpu").manual_seed(int(seed))
    t = torch.randn(tuple(shape), generator=g, dtype=torch.float32)
    if std != 1.0:
        t.mul_(std)
    if mean != 0.0:
        t.add_(mean)
    return t.to(torch.bfloat16)


def layer_weights(cfg: LayerConfig, tag: str, base: int = 0) -> dict:
    """All weights of one layer as BF16 CPU tensors ([out, in] layout).

    Names match the fields of the C struct ``qwen_layer_weights``.  The router
    bias, when present, is a float32 tensor holding BF16-representable values.
    """
    d, hq, hkv, dh, f = cfg.d, cfg.n_q_heads, cfg.n_kv_heads, cfg.head_dim, cfg.ffn
    nq, nkv = hq * dh, hkv * dh
    s = lambda name: seed_for(tag, name, base)  # noqa: E731
    w = {
        "gamma_attn": normal_bf16([d], s("gamma_attn"), 0.1, 1.0),
        "gamma_mlp": normal_bf16([d], s("gamma_mlp"), 0.1, 1.0),
        "w_q": normal_bf16([nq, d], s("w_q"), 0.02),
        "w_k": normal_bf16([nkv, d], s("w_k"), 0.02),
        "w_v": normal_bf16([nkv, d], s("w_v"), 0.02),
        "w_o": normal_bf16([d, nq], s("w_o"), 0.02),
    }
    if cfg.qk_norm:
        w["gamma_q"] = normal_bf16([dh], s("gamma_q"), 0.1, 1.0)
        w["gamma_k"] = normal_bf16([dh], s("gamma_k"), 0.1, 1.0)
    if cfg.qkv_bias:
        w["b_q"] = normal_bf16([nq], s("b_q"), 0.02)
        w["b_k"] = normal_bf16([nkv], s("b_k"), 0.02)
        w["b_v"] = normal_bf16([nkv], s("b_v"), 0.02)
    if cfg.n_experts:
        e = cfg.n_experts
        w["w_router"] = normal_bf16([e, d], s("w_router"), 0.02)
        if cfg.router_bias:
            w["b_router"] = normal_bf16([e], s("b_router"), 0.5).float()
        w["w_gate"] = normal_bf16([e, f, d], s("w_gate"), 0.02)
        w["w_up"] = normal_bf16([e, f, d], s("w_up"), 0.02)
        w["w_down"] = normal_bf16([e, d, f], s("w_down"), 0.02)
        if cfg.shared_ffn:
            sf = cfg.shared_ffn
            w["w_shared_gate"] = normal_bf16([sf, d], s("w_shared_gate"), 0.02)
            w["w_shared_up"] = normal_bf16([sf, d], s("w_shared_up"), 0.02)
            w["w_shared_down"] = normal_bf16([d, sf], s("w_shared_down"), 0.02)
            w["w_shared_expert_gate"] = normal_bf16([d], s("w_shared_expert_gate"), 0.02)
    else:
        w["w_gate"] = normal_bf16([f, d], s("w_gate"), 0.02)
        w["w_up"] = normal_bf16([f, d], s("w_up"), 0.02)
        w["w_down"] = normal_bf16([d, f], s("w_down"), 0.02)
    return w


def activations(shape, tag: str, name: str = "x", base: int = 0) -> torch.Tensor:
    """Layer input X ~ N(0, 1), BF16."""
    return normal_bf16(shape, seed_for(tag, name, base))


def kv_cache(batch: int, n_kv: int, max_seq: int, dh: int, filled, tag: str,
             base: int = 0):
    """K and V caches [B, Hkv, max_seq, dh] BF16: N(0,1) in slots < filled[b].

    The filled rows stand for keys that an earlier step already normalised and
    rotated.  ``filled`` is an int or a per-sequence list.
    """
    if isinstance(filled, int):
        filled = [filled] * batch
    k = torch.zeros((batch, n_kv, max_seq, dh), dtype=torch.bfloat16)
    v = torch.zeros((batch, n_kv, max_seq, dh), dtype=torch.bfloat16)
    for b, n in enumerate(filled):
        if n:
            k[b, :, :n] = normal_bf16([n_kv, n, dh], seed_for(tag, f"k_cache{b}", base))
            v[b, :, :n] = normal_bf16([n_kv, n, dh], seed_for(tag, f"v_cache{b}", base))
    return k, v


def to_f64(t: torch.Tensor):
    """Exact widening of a BF16/FP32 CPU tensor to a float64 numpy array."""
    return t.detach().to("cpu", torch.float64).numpy()


def weights_f64(w: dict) -> dict:
    return {k: to_f64(v) for k, v in w.items()}
