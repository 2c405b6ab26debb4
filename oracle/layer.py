"""Plain FP64 definition of a Qwen-style pre-norm decoder layer (test infrastructure).

Every function takes and returns float64 numpy arrays.  Inputs are the
BF16-rounded tensors both sides see, widened exactly to float64; nothing is
rounded in between.  Sources are cited by page title and section; the page key
([P1]..[P5]) is listed in ``oracle/__init__.py``.

Conventions
-----------
* Weights are stored ``[out, in]`` and applied as ``y = x W^T``
  ([P1] §03.1 "权重存的是 [out, in]"; [P3] §4, the Linear convention note).
* One sequence's activations are ``[T, d]``; heads split the projection output
  so head ``h`` owns channels ``[h*dh, (h+1)*dh)`` ([P1] §05.1).
* A KV cache for one sequence is ``[Hkv, max_seq, dh]``.  Cache *slots* decide
  the causal mask and where K/V rows are written; *positions* drive RoPE only.
  A query in slot ``s_q`` sees every slot ``<= s_q`` of its own sequence.

Readings where the pages are silent or disagree (each is also listed in the
design notes):

* RoPE pairs channel ``i`` with ``i + dh/2`` (rotate_half), the pairing [P3] §6
  says the reference implementation uses; [P1] §05.3 prints the interleaved
  pairing (2i, 2i+1), which is the same rotation under a fixed channel
  permutation.
* SwiGLU applies SiLU to the *gate* projection ([P3] §10, [P1] §07.1); the
  lecture notes' expert formula [P2] "Expert 的 FFN 结构" puts SiLU on up and
  contradicts its own prose ("门控分支 ... 与 W_up 的输出逐元素相乘").
* QK-norm uses the layer's ``rms_eps`` (not stated for QK-norm on the pages).
* Router: a per-expert bias, when given, is added to the logits before top-k
  selection and gating.  Top-k ranks by logit, larger first, lower expert
  index first on exact ties.
"""

from __future__ import annotations

import numpy as np


# --------------------------------------------------------------------------
# Elementary steps
# --------------------------------------------------------------------------

def rmsnorm(x, gamma, eps):
    """RMSNorm over the last axis.

    [P3] §3 (RMSNorm equation): y_j = gamma_j * x_j / sqrt(mean_k x_k^2 + eps).
    The mean square is over the feature axis of one position only; no mean is
    subtracted.  epsilon sits inside the square root.
    """
    x = np.asarray(x, dtype=np.float64)
    ms = np.mean(x * x, axis=-1, keepdims=True)
    return np.asarray(gamma, dtype=np.float64) * (x / np.sqrt(ms + eps))


def linear(x, w, b=None):
    """y = x W^T (+ b), W stored [out, in] ([P1] §03.1; [P3] §4)."""
    y = np.asarray(x, dtype=np.float64) @ np.asarray(w, dtype=np.float64).T
    if b is not None:
        y = y + np.asarray(b, dtype=np.float64)
    return y


def silu(z):
    """SiLU(z) = z * sigmoid(z) = z / (1 + e^{-z}) ([P3] §10; [P1] §07.1)."""
    z = np.asarray(z, dtype=np.float64)
    with np.errstate(over="ignore"):
        return z / (1.0 + np.exp(-z))


def matmul_counted(a, b):
    """Matrix product by the dot-product definition, counting operations.

    [P1] §03.4-03.5: each output element is a length-k dot product costing k
    multiplies and k-1 additions, so an [m,k]x[k,n] product costs m*n*(2k-1)
    operations exactly (the 2*m*k*n convention over-counts by m*n).
    Returns (C, exact_ops).  Pure Python loops: for small inputs only.
    """
    a = [[float(v) for v in row] for row in np.asarray(a)]
    b = [[float(v) for v in row] for row in np.asarray(b)]
    m, k, n = len(a), len(b), len(b[0])
    c = [[0.0] * n for _ in range(m)]
    ops = 0
    for i in range(m):
        for j in range(n):
            acc = a[i][0] * b[0][j]
            ops += 1
            for p in range(1, k):
                acc = acc + a[i][p] * b[p][j]
                ops += 2
            c[i][j] = acc
    return np.array(c), ops


def rope_angles(positions, dh, theta):
    """Angles p * omega_r with omega_r = theta^(-2r/dh), r = 0..dh/2-1.

    [P3] §6 (frequency equation); theta = 1e6 and no scaling for the Qwen
    configurations.  Computed in float64.
    """
    r = np.arange(dh // 2, dtype=np.float64)
    omega = np.float64(theta) ** (-2.0 * r / dh)
    return np.outer(np.asarray(positions, dtype=np.float64), omega)


def apply_rope_rotate_half(x, positions, theta):
    """Rotate each head vector by its position, pairing (i, i + dh/2).

    x: [T, H, dh]; positions: [T].  For pair r the 2-D rotation R(p*omega_r)
    of [P3] §6 acts on (x_r, x_{r+dh/2}):
        x'_r        = x_r cos - x_{r+dh/2} sin
        x'_{r+dh/2} = x_{r+dh/2} cos + x_r sin
    """
    x = np.asarray(x, dtype=np.float64)
    dh = x.shape[-1]
    half = dh // 2
    ang = rope_angles(positions, dh, theta)[:, None, :]  # [T, 1, half]
    c, s = np.cos(ang), np.sin(ang)
    lo, hi = x[..., :half], x[..., half:]
    return np.concatenate([lo * c - hi * s, hi * c + lo * s], axis=-1)


def gqa_attention(q, k, v, q_slots, k_slots, causal=True, return_probs=False):
    """Scaled, masked softmax attention with grouped K/V heads.

    q: [Tq, Hq, dh]; k, v: [Tk, Hkv, dh]; q_slots [Tq], k_slots [Tk].
    [P3] §7: query head h reads K/V head g(h) = floor(h / (Hq/Hkv)), score
    S = q.k / sqrt(dh) + M.  [P3] §8: M = 0 where the key slot is <= the query
    slot and -inf otherwise; softmax subtracts the row max and normalises over
    key positions of one head.  [P3] §9: o = sum_s a_s v_s.
    Returns o [Tq, Hq, dh] (and the probabilities [Hq, Tq, Tk] on request).
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    tq, hq, dh = q.shape
    hkv = k.shape[1]
    assert hq % hkv == 0, "Hq must be a multiple of Hkv"
    group = hq // hkv
    q_slots = np.asarray(q_slots)
    k_slots = np.asarray(k_slots)
    visible = k_slots[None, :] <= q_slots[:, None]
    out = np.empty((tq, hq, dh), dtype=np.float64)
    probs = np.empty((hq, tq, k.shape[0]), dtype=np.float64) if return_probs else None
    for h in range(hq):
        g = h // group
        s = (q[:, h, :] @ k[:, g, :].T) / np.sqrt(np.float64(dh))
        if causal:
            s = np.where(visible, s, -np.inf)
        m = np.max(s, axis=1, keepdims=True)
        e = np.exp(s - m)
        a = e / np.sum(e, axis=1, keepdims=True)
        out[:, h, :] = a @ v[:, g, :]
        if return_probs:
            probs[h] = a
    if return_probs:
        return out, probs
    return out


# --------------------------------------------------------------------------
# Blocks
# --------------------------------------------------------------------------

def _qkv(xh, w, cfg, positions):
    """Q/K/V projections, optional bias, QK-norm, then RoPE ([P3] §4-§6).

    [P3] §5: with QK-norm each head vector of Q (and of K) is normalised on
    its own, over its dh channels, with one length-dh gamma shared by all Q
    heads (gamma_q) and one shared by all K heads (gamma_k); V is not
    normalised.  [P3] §6 then rotates the normalised Q and K by position.
    Returns q [T,Hq,dh], k [T,Hkv,dh] (both rotated) and v [T,Hkv,dh].
    """
    t = xh.shape[0]
    hq, hkv, dh = cfg["n_q_heads"], cfg["n_kv_heads"], cfg["head_dim"]
    theta = cfg["rope_theta"]
    bias = bool(cfg.get("qkv_bias", 0))
    q = linear(xh, w["w_q"], w["b_q"] if bias else None).reshape(t, hq, dh)
    k = linear(xh, w["w_k"], w["b_k"] if bias else None).reshape(t, hkv, dh)
    v = linear(xh, w["w_v"], w["b_v"] if bias else None).reshape(t, hkv, dh)
    if cfg.get("qk_norm", 0):
        q = rmsnorm(q, w["gamma_q"], cfg["rms_eps"])
        k = rmsnorm(k, w["gamma_k"], cfg["rms_eps"])
    q = apply_rope_rotate_half(q, positions, theta)
    k = apply_rope_rotate_half(k, positions, theta)
    return q, k, v


def attention_block(x, w, cfg, positions, k_cache, v_cache, slots,
                    causal=True, rows=None):
    """R = X + Attention(RMSNorm_1(X)) for one sequence ([P3] §2, §4-§9).

    x: [T, d]; positions, slots: [T] ints; k_cache, v_cache: [Hkv, S_max, dh]
    float64 arrays updated in place with the new post-QK-norm, post-RoPE K and
    V rows ([P1] §09.1; [P3] §12).  ``rows`` restricts the returned rows (the
    K/V of every row is still computed and written, since later rows read it).
    Returns R for the requested rows.
    """
    x = np.asarray(x, dtype=np.float64)
    slots = np.asarray(slots)
    positions = np.asarray(positions)
    xh = rmsnorm(x, w["gamma_attn"], cfg["rms_eps"])
    q, k, v = _qkv(xh, w, cfg, positions)
    k_cache[:, slots, :] = k.transpose(1, 0, 2)
    v_cache[:, slots, :] = v.transpose(1, 0, 2)
    if rows is None:
        rows = np.arange(x.shape[0])
    rows = np.asarray(rows)
    n_keys = int(slots[rows].max()) + 1 if causal else k_cache.shape[1]
    k_slots = np.arange(n_keys)
    kk = k_cache[:, :n_keys, :].transpose(1, 0, 2)
    vv = v_cache[:, :n_keys, :].transpose(1, 0, 2)
    o = gqa_attention(q[rows], kk, vv, slots[rows], k_slots, causal=causal)
    c = o.reshape(len(rows), -1)  # concat heads along features ([P3] §9)
    return x[rows] + linear(c, w["w_o"])


def mlp_block(r, w, cfg):
    """Y = R + (SiLU(Z W_gate^T) * (Z W_up^T)) W_down^T, Z = RMSNorm_2(R).

    [P3] §10 (gated MLP equations); [P1] §07.1.  No biases.
    """
    r = np.asarray(r, dtype=np.float64)
    z = rmsnorm(r, w["gamma_mlp"], cfg["rms_eps"])
    h = silu(linear(z, w["w_gate"])) * linear(z, w["w_up"])
    return r + linear(h, w["w_down"])


def layer_forward(x, w, cfg, positions, k_cache, v_cache, slots,
                  causal=True, rows=None):
    """Dense layer forward for one sequence: attention block then MLP block.

    [P3] §2: R = X + Attention(RMSNorm_1(X)), Y = R + MLP(RMSNorm_2(R)); the
    first residual adds the raw X and the second norm reads R.  Decode is the
    same call with T = 1 in slot ``cache_len`` ([P1] §09.1).
    """
    r = attention_block(x, w, cfg, positions, k_cache, v_cache, slots,
                        causal=causal, rows=rows)
    return mlp_block(r, w, cfg)


# --------------------------------------------------------------------------
# Mixture of experts
# --------------------------------------------------------------------------

def router_topk(z, w_router, b_router, k, norm_topk_prob=True):
    """Router logits, top-k selection and the gating weights.

    [P1] §10.2 and [P2] "Router 机制": logits = z W_router (+ bias), one score
    per expert for every expert; probs = softmax over all experts; the k
    largest are selected (ranking by probability equals ranking by logit).
    With norm_topk_prob the k weights are the selected probabilities
    renormalised to sum 1, which equals a softmax over the k selected logits;
    without it ([P1] §10.2, Qwen2) they are the selected probabilities as they
    are (their sum is below 1).
    Returns (logits [T,E], idx [T,k] int64, weights [T,k], gap [T]) where gap
    is the k-th minus the (k+1)-th largest logit (inf when k == E).
    """
    logits = linear(z, w_router, b_router)
    # stable sort on -logit: larger logit first, lower index first on ties
    order = np.argsort(-logits, axis=1, kind="stable")
    idx = order[:, :k]
    sel = np.take_along_axis(logits, idx, axis=1)
    if norm_topk_prob:
        m = np.max(sel, axis=1, keepdims=True)
        e = np.exp(sel - m)
        wts = e / np.sum(e, axis=1, keepdims=True)
    else:
        m = np.max(logits, axis=1, keepdims=True)
        wts = np.exp(sel - m) / np.sum(np.exp(logits - m), axis=1, keepdims=True)
    if k < logits.shape[1]:
        kth = sel[:, k - 1]
        nxt = np.take_along_axis(logits, order[:, k:k + 1], axis=1)[:, 0]
        gap = kth - nxt
    else:
        gap = np.full(logits.shape[0], np.inf)
    return logits, idx, wts, gap


def _expert(z, wg, wu, wd):
    """One SwiGLU expert ([P2] "Expert 的 FFN 结构", read with SiLU on gate)."""
    return linear(silu(linear(z, wg)) * linear(z, wu), wd)


def sigmoid(x):
    """The logistic function 1 / (1 + e^-x)."""
    return 1.0 / (1.0 + np.exp(-x))


def moe_block(r, w, cfg, routing=None):
    """Y = R + sum_j w_j * Expert_{idx_j}(Z) [+ g * SharedExpert(Z)],
    Z = RMSNorm_2(R).

    [P1] §10.2 (the weighted sum is a plain element-wise sum, no further
    normalisation) and [P2] "MoE 的最终输出".  With a shared expert ([P1]
    §10.1, Qwen2-MoE): a SwiGLU of width ``shared_ffn`` on the same Z whose
    output is scaled per token by g = sigmoid(Z W_sg), W_sg one column without
    bias, and added to the routed sum.  ``routing`` may supply (idx, weights)
    to evaluate the experts under a given selection.
    Returns (Y, logits, idx, weights, gap, z).
    """
    r = np.asarray(r, dtype=np.float64)
    z = rmsnorm(r, w["gamma_mlp"], cfg["rms_eps"])
    logits, idx, wts, gap = router_topk(z, w["w_router"], w.get("b_router"),
                                        cfg["top_k"], cfg.get("norm_topk_prob", 1))
    if routing is not None:
        idx, wts = routing
    t, kk = idx.shape
    eo = np.zeros((t, kk, r.shape[1]), dtype=np.float64)
    for e in np.unique(idx):
        tok, slot = np.nonzero(idx == e)
        eo[tok, slot] = _expert(z[tok], w["w_gate"][e], w["w_up"][e], w["w_down"][e])
    acc = np.zeros_like(r)
    for j in range(kk):  # summed in slot order
        acc = acc + wts[:, j:j + 1] * eo[:, j, :]
    if cfg.get("shared_ffn", 0):
        g = sigmoid(z @ np.asarray(w["w_shared_expert_gate"], dtype=np.float64))
        acc = acc + g[:, None] * _expert(z, w["w_shared_gate"], w["w_shared_up"],
                                         w["w_shared_down"])
    return r + acc, logits, idx, wts, gap, z


def moe_layer_forward(x, w, cfg, positions, k_cache, v_cache, slots, rows=None):
    """MoE layer: the attention block unchanged, the MLP replaced by MoE.

    [P1] §10 ("MoE 只改 MLP 这一块").  Returns (Y, R, routing tuple).
    """
    r = attention_block(x, w, cfg, positions, k_cache, v_cache, slots, rows=rows)
    y, logits, idx, wts, gap, _ = moe_block(r, w, cfg)
    return y, r, (logits, idx, wts, gap)


def head_last_token(y_last, gamma_final, w_lm, eps):
    """logits = RMSNorm_final(y) W_lm^T for the last position of each sequence.

    [P1] §03.8: the model-level final norm and lm_head; during prefill only the
    last position needs logits.
    """
    return linear(rmsnorm(y_last, gamma_final, eps), w_lm)
