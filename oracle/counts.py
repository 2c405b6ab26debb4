"""Closed-form parameter, FLOP and KV-byte counts (test infrastructure).

Written from the formulas the pages state; pinned against the totals they
print (tests/test_oracle_counts.py).  Page key in ``oracle/__init__.py``.
"""

from __future__ import annotations


def attn_params(d, n_q, n_kv, dh):
    """Q, K, V, O projection weights of one layer.

    [P2] "每层参数量" (GQA attention term); [P4] §3; [P5] §1:
    d*(Hq*dh) + 2*d*(Hkv*dh) + (Hq*dh)*d.
    """
    return d * (n_q * dh) + 2 * d * (n_kv * dh) + (n_q * dh) * d


def qkv_bias_params(n_q, n_kv, dh):
    """q/k/v biases: Hq*dh + 2*Hkv*dh ([P1] §11 "qkv bias")."""
    return n_q * dh + 2 * n_kv * dh


def mlp_params(d, f):
    """SwiGLU gate, up, down: 3*d*f ([P1] §11; [P3] §11; [P5] §1)."""
    return 3 * d * f


def layer_norm_params(d, dh=0, qk_norm=False):
    """Two length-d RMSNorm gammas, plus two length-dh QK-norm gammas ([P3] §11)."""
    return 2 * d + (2 * dh if qk_norm else 0)


def dense_model_params(L, d, n_q, n_kv, dh, f, vocab, tied=False, bias=True,
                       final_norm=True):
    """Whole dense model ([P1] §11 total formula; [P5] §2 boxed formula):
    L*(attn + bias + mlp + norm) + (1 or 2)*V*d + d.
    """
    per_layer = attn_params(d, n_q, n_kv, dh) + mlp_params(d, f) + 2 * d
    if bias:
        per_layer += qkv_bias_params(n_q, n_kv, dh)
    return L * per_layer + (1 if tied else 2) * vocab * d + (d if final_norm else 0)


def matmul_params_dense(L, d, n_q, n_kv, dh, f, vocab):
    """Parameters that take part in matrix products: everything except the
    embedding lookup, norms and biases ([P1] §03.8 counts the norms and biases
    in and notes them as a 0.005% error; this is the strict count)."""
    return L * (attn_params(d, n_q, n_kv, dh) + mlp_params(d, f)) + vocab * d


def kv_bytes_per_token(L, n_kv, dh, dtype_bytes=2):
    """KV cache bytes per token: 2 * L * Hkv * dh * b ([P1] §11; [P4] §3)."""
    return 2 * L * n_kv * dh * dtype_bytes


def attention_flops_prefill_causal(L, n_q, dh, S):
    """QK^T and PV of a causal prefill, upper triangle skipped:
    4*dh*S^2 * Hq / 2 * L ([P1] §05.4)."""
    return 4 * dh * S * S * n_q * L // 2


def attention_flops_decode(L, n_q, dh, T):
    """One decode query against T cached keys: 4*dh*T*Hq*L ([P1] §05.5)."""
    return 4 * dh * T * n_q * L


def attention_flops_dense(n_q, dh, T):
    """Dense (no causal skipping) QK^T + AV of one layer: 4*Hq*T^2*dh ([P3] §11)."""
    return 4 * n_q * T * T * dh


def linear_flops(T, params):
    """2 * T * params: two FLOPs per weight per token ([P1] §03.6; [P3] §11)."""
    return 2 * T * params


def moe_block_params(d, E, mf, sf=0, shared_gate=True):
    """MoE block: router d*E + experts E*3*d*mf (+ shared 3*d*sf + d gate).

    [P1] §11.1; [P5] §3.
    """
    p = d * E + E * 3 * d * mf
    if sf:
        p += 3 * d * sf + (d if shared_gate else 0)
    return p


def moe_block_active_params(d, E, k, mf, sf=0, shared_gate=True):
    """Per-token active MoE block parameters: k experts instead of E ([P1] §11.1)."""
    p = d * E + k * 3 * d * mf
    if sf:
        p += 3 * d * sf + (d if shared_gate else 0)
    return p


def moe_model_params(L, d, n_q, n_kv, dh, E, k, mf, sf, vocab, tied=False,
                     bias=True, active=False):
    """Whole MoE model: per layer attention + bias + 2 norms + MoE block, plus
    embeddings / lm_head and the final norm ([P1] §11, §11.1)."""
    per_layer = attn_params(d, n_q, n_kv, dh) + 2 * d
    if bias:
        per_layer += qkv_bias_params(n_q, n_kv, dh)
    if active:
        per_layer += moe_block_active_params(d, E, k, mf, sf)
    else:
        per_layer += moe_block_params(d, E, mf, sf)
    return L * per_layer + (1 if tied else 2) * vocab * d + d


def touched_experts(E, k, B):
    """Expected distinct experts a decode batch of B tokens touches under
    uniform routing: E * (1 - (1 - k/E)^B) ([P1] §11.1)."""
    return E * (1.0 - (1.0 - k / E) ** B)
