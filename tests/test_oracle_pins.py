"""Pins of the FP64 oracle against what the pages and mathematics fix.

Each test names the page and section it pins.  None of these tests re-types the
oracle's own formula: they use values printed on the pages, textbook values,
special cases with closed forms, invariants the pages state, and brute force on
tiny inputs.
"""

import itertools
import math

import numpy as np
import pytest

import oracle as O
import synth

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


def small_cfg(**kw):
    base = dict(d=16, n_q_heads=4, n_kv_heads=2, head_dim=4, ffn=24, qkv_bias=0,
                qk_norm=1, rope_theta=1.0e6, rms_eps=1.0e-6)
    base.update(kw)
    return base


def rand_weights(cfg, seed=0, bias=False):
    rng = np.random.default_rng(seed)
    d, hq, hkv, dh, f = cfg["d"], cfg["n_q_heads"], cfg["n_kv_heads"], cfg["head_dim"], cfg["ffn"]
    w = {
        "gamma_attn": 1 + 0.1 * rng.standard_normal(d),
        "gamma_mlp": 1 + 0.1 * rng.standard_normal(d),
        "gamma_q": 1 + 0.1 * rng.standard_normal(dh),
        "gamma_k": 1 + 0.1 * rng.standard_normal(dh),
        "w_q": 0.3 * rng.standard_normal((hq * dh, d)),
        "w_k": 0.3 * rng.standard_normal((hkv * dh, d)),
        "w_v": 0.3 * rng.standard_normal((hkv * dh, d)),
        "w_o": 0.3 * rng.standard_normal((d, hq * dh)),
        "w_gate": 0.3 * rng.standard_normal((f, d)),
        "w_up": 0.3 * rng.standard_normal((f, d)),
        "w_down": 0.3 * rng.standard_normal((d, f)),
    }
    if bias:
        w["b_q"] = 0.1 * rng.standard_normal(hq * dh)
        w["b_k"] = 0.1 * rng.standard_normal(hkv * dh)
        w["b_v"] = 0.1 * rng.standard_normal(hkv * dh)
    return w


def run_layer(x, w, cfg, positions=None, causal=True, max_seq=None):
    t = x.shape[0]
    max_seq = max_seq or t
    kc = np.zeros((cfg["n_kv_heads"], max_seq, cfg["head_dim"]))
    vc = np.zeros_like(kc)
    pos = np.arange(t) if positions is None else np.asarray(positions)
    y = O.layer_forward(x, w, cfg, pos, kc, vc, np.arange(t), causal=causal)
    return y, kc, vc


# ---------------------------------------------------------------- matmul


def test_matmul_worked_example(golden):
    """Qwen2.5-7B 结构拆解 §03.5: [[1,2,3],[4,5,6]] @ [[7,8],[9,10],[11,12]]."""
    g = golden["matmul_2x3_3x2"]
    c, ops = O.matmul_counted(g["A"], g["B"])
    assert c.tolist() == g["C"]
    assert ops == g["exact_ops"]
    m, k, n = 2, 3, 2
    assert 2 * m * k * n == g["ops_2mkn"]


def test_linear_uses_out_in_storage(golden):
    """§03.1 of the same page: weights are stored [out, in] and y = x W^T.

    The worked example's B is [in=3, out=2]; stored as [out, in] it is B^T.
    """
    g = golden["matmul_2x3_3x2"]
    a = np.array(g["A"], dtype=np.float64)
    w_stored = np.array(g["B"], dtype=np.float64).T  # [out, in]
    assert O.linear(a, w_stored).tolist() == g["C"]
    # a non-square weight keeps its [out, in] shape: out = 2 rows
    assert O.linear(np.ones((1, 3)), w_stored).shape == (1, 2)


# ---------------------------------------------------------------- RMSNorm


def test_rmsnorm_worked_example(golden):
    """推理系统 03 §3: x=[1,0,-1,0.5] -> about [1.3333, 0, -1.3333, 0.6667]."""
    g = golden["rmsnorm_example"]
    y = O.rmsnorm(np.array(g["x"]), np.ones(4), 1e-6)
    assert np.allclose(np.round(y, g["printed_decimals"]), g["y_approx"], atol=0, rtol=0)
    # exact value with epsilon inside the square root
    assert y[0] == pytest.approx(1.0 / math.sqrt(g["mean_square"] + 1e-6), rel=1e-15)
    assert abs(y[0] - 4.0 / 3.0) < 1e-5


def test_rmsnorm_does_not_subtract_mean():
    """§3: RMSNorm does not subtract the mean, so a constant row stays constant."""
    y = O.rmsnorm(np.full(8, 2.0), np.ones(8), 0.0)
    assert np.array_equal(y, np.ones(8))


def test_rmsnorm_output_rms_with_eps():
    """§3: with gamma=1 the output RMS is sqrt(ms/(ms+eps)), not exactly 1."""
    x = np.array([3.0, 4.0])  # mean square 12.5
    y = O.rmsnorm(x, np.ones(2), 0.5)
    assert math.sqrt(np.mean(y * y)) == pytest.approx(math.sqrt(12.5 / 13.0), rel=1e-14)


def test_rmsnorm_rows_independent():
    """§3: each position is normalised on its own (no averaging over T)."""
    x = np.array([[1.0, 2.0, 3.0], [100.0, -5.0, 0.25]])
    y = O.rmsnorm(x, np.ones(3), 1e-6)
    assert np.array_equal(y[0], O.rmsnorm(x[:1], np.ones(3), 1e-6)[0])


# ---------------------------------------------------------------- RoPE


def test_rope_position_zero_is_identity():
    x = np.random.default_rng(1).standard_normal((1, 3, 8))
    assert np.array_equal(O.apply_rope_rotate_half(x, [0], 1e6), x)


def test_rope_pairs_i_with_i_plus_half():
    """推理系统 03 §6: rotate_half pairs (0,64), (1,65), ...; omega_r = theta^(-2r/dh).

    dh=4, theta=100: omega = [1, 0.1].  At p=2 the unit vector e0 rotates into
    channel 2 (its partner), e1 into channel 3 with the slower frequency.
    Textbook values: cos 2, sin 2, cos 0.2, sin 0.2.
    """
    cos2, sin2 = -0.4161468365471424, 0.9092974268256817
    cos02, sin02 = 0.9800665778412416, 0.19866933079506122
    e = np.eye(4)[:, None, :]  # [4 rows as T, H=1, dh=4]
    y = O.apply_rope_rotate_half(e, [2, 2, 2, 2], 100.0)[:, 0, :]
    assert np.allclose(y[0], [cos2, 0, sin2, 0], atol=1e-15)
    assert np.allclose(y[1], [0, cos02, 0, sin02], atol=1e-15)
    assert np.allclose(y[2], [-sin2, 0, cos2, 0], atol=1e-15)
    assert np.allclose(y[3], [0, -sin02, 0, cos02], atol=1e-15)


def test_rope_preserves_pair_norms():
    x = np.random.default_rng(2).standard_normal((5, 2, 8))
    y = O.apply_rope_rotate_half(x, [0, 3, 17, 1000, 16383], 1e6)
    n = lambda a: a[..., :4] ** 2 + a[..., 4:] ** 2  # noqa: E731
    assert np.allclose(n(x), n(y), rtol=1e-13)


def test_rope_dot_depends_on_position_difference_only():
    """推理系统 03 §6: (R(p w) q)^T (R(s w) k) = q^T R((s-p) w) k."""
    rng = np.random.default_rng(3)
    q = rng.standard_normal((1, 1, 128))
    k = rng.standard_normal((1, 1, 128))
    d1 = np.sum(O.apply_rope_rotate_half(q, [3], 1e6) * O.apply_rope_rotate_half(k, [10], 1e6))
    d2 = np.sum(O.apply_rope_rotate_half(q, [1003], 1e6) * O.apply_rope_rotate_half(k, [1010], 1e6))
    assert d1 == pytest.approx(d2, abs=1e-10)


# ---------------------------------------------------------------- attention


def test_attention_two_key_closed_form():
    """推理系统 03 §7-§9 on a hand example: dh=4 so the scale is 1/2.

    q.k1 = 2 ln 3 and q.k2 = 0 give scaled scores (ln 3, 0), so the softmax is
    (3/4, 1/4) and the output is 3/4 v1 + 1/4 v2.
    """
    q = np.array([[[1.0, 0, 0, 0]]])
    k = np.array([[[2 * math.log(3.0), 0, 0, 0]], [[0.0, 0, 0, 0]]])
    v = np.array([[[1.0, 0, 0, 0]], [[0.0, 1, 0, 0]]])
    o, p = O.gqa_attention(q, k, v, [1], [0, 1], return_probs=True)
    assert np.allclose(p[0, 0], [0.75, 0.25], atol=1e-15)
    assert np.allclose(o[0, 0], [0.75, 0.25, 0, 0], atol=1e-15)


def test_attention_causal_mask_and_row_sums():
    """§8: future keys get probability exactly 0; visible probabilities sum to 1."""
    rng = np.random.default_rng(4)
    q, k, v = (rng.standard_normal((6, 4, 8)), rng.standard_normal((6, 2, 8)),
               rng.standard_normal((6, 2, 8)))
    _, p = O.gqa_attention(q, k, v, np.arange(6), np.arange(6), return_probs=True)
    assert np.all(p[:, np.triu_indices(6, 1)[0], np.triu_indices(6, 1)[1]] == 0.0)
    assert np.allclose(p.sum(axis=-1), 1.0, atol=1e-14)


def test_attention_first_position_returns_its_value():
    """§9: a query that sees one key returns that key's value exactly."""
    rng = np.random.default_rng(5)
    q, k, v = (rng.standard_normal((3, 2, 4)), rng.standard_normal((3, 1, 4)),
               rng.standard_normal((3, 1, 4)))
    o = O.gqa_attention(q, k, v, np.arange(3), np.arange(3))
    assert np.array_equal(o[0, 0], v[0, 0]) and np.array_equal(o[0, 1], v[0, 0])


def test_attention_equal_keys_give_mean_of_visible_values():
    rng = np.random.default_rng(6)
    q = rng.standard_normal((4, 1, 4))
    k = np.tile(rng.standard_normal((1, 1, 4)), (4, 1, 1))
    v = rng.standard_normal((4, 1, 4))
    o = O.gqa_attention(q, k, v, np.arange(4), np.arange(4))
    for t in range(4):
        assert np.allclose(o[t, 0], v[: t + 1, 0].mean(axis=0), atol=1e-14)


def test_gqa_head_mapping_floor_division():
    """推理系统 03 §7: g(h) = floor(h / (Hq/Hkv)); heads 0-1 read KV head 0."""
    q = np.zeros((1, 4, 2))
    k = np.zeros((1, 2, 2))
    v = np.stack([np.ones((1, 2)), np.zeros((1, 2))], axis=1)  # kv head 0 = 1, head 1 = 0
    o = O.gqa_attention(q, k, v, [0], [0])
    assert o[0, :, 0].tolist() == [1.0, 1.0, 0.0, 0.0]


def test_gqa_equals_mha_with_repeated_kv_weights():
    """Qwen2.5-7B 结构拆解 §05.2: GQA is MHA with K/V heads repeat_interleave'd."""
    cfg = small_cfg(n_q_heads=4, n_kv_heads=2)
    w = rand_weights(cfg, 7, bias=True)
    x = np.random.default_rng(8).standard_normal((5, cfg["d"]))
    y_gqa, _, _ = run_layer(x, w, cfg)
    rep = cfg["n_q_heads"] // cfg["n_kv_heads"]
    dh = cfg["head_dim"]
    mha = dict(w)
    for name in ("w_k", "w_v", "b_k", "b_v"):
        a = w[name].reshape(cfg["n_kv_heads"], dh, *w[name].shape[1:])
        mha[name] = np.repeat(a, rep, axis=0).reshape(-1, *w[name].shape[1:])
    y_mha, _, _ = run_layer(x, mha, dict(cfg, n_kv_heads=cfg["n_q_heads"]))
    assert np.allclose(y_gqa, y_mha, rtol=0, atol=1e-13)


# ---------------------------------------------------------------- layer invariants


def toy_inputs():
    """推理系统 03 §1: T=3, d=4, Hq=2, Hkv=1, dh=2, f=6, gamma=1, eps=1e-6.

    The page's hand-set weights are not printed, so the weights are seeded; the
    relational results are what is pinned.  x_2[0] = 1 so that §14's edit to -3
    applies.
    """
    cfg = synth.TOY.as_dict()
    w = synth.weights_f64(synth.layer_weights(synth.TOY, "toy"))
    for gname in ("gamma_attn", "gamma_mlp"):
        w[gname] = np.ones(cfg["d"])
    for name in ("w_q", "w_k", "w_v", "w_o", "w_gate", "w_up", "w_down"):
        w[name] = w[name] * 25.0  # N(0, 0.5): large enough that rows mix visibly
    x = synth.to_f64(synth.activations([3, 4], "toy"))
    x[2, 0] = 1.0
    return cfg, w, x


def test_toy_experiment_1_change_future():
    """推理系统 03 §14 experiment 1: x_2[0] 1 -> -3 leaves rows 0,1 exactly unchanged."""
    cfg, w, x = toy_inputs()
    y0, _, _ = run_layer(x, w, cfg)
    x2 = x.copy()
    x2[2, 0] = -3.0
    y1, _, _ = run_layer(x2, w, cfg)
    assert np.array_equal(y0[:2], y1[:2])
    assert not np.array_equal(y0[2], y1[2])
    # with the mask off the guarantee is gone
    z0, _, _ = run_layer(x, w, cfg, causal=False)
    z1, _, _ = run_layer(x2, w, cfg, causal=False)
    assert np.max(np.abs(z0[:2] - z1[:2])) > 1e-6


def test_toy_experiment_2_shift_positions():
    """§14 experiment 2: positions [0,1,2] -> [7,8,9] give the same output."""
    cfg, w, x = toy_inputs()
    y0, _, _ = run_layer(x, w, cfg, positions=[0, 1, 2])
    y1, _, _ = run_layer(x, w, cfg, positions=[7, 8, 9])
    y2, _, _ = run_layer(x, w, cfg, positions=[1000, 1001, 1002])
    assert np.max(np.abs(y0 - y1)) < 1e-12
    assert np.max(np.abs(y0 - y2)) < 1e-12
    # changing one relative distance does change the output
    y3, _, _ = run_layer(x, w, cfg, positions=[0, 1, 5])
    assert np.max(np.abs(y0 - y3)) > 1e-6


def test_toy_experiment_3_same_kv_different_query():
    """§14 experiment 3: two query heads share K/V but get different probabilities."""
    cfg, w, x = toy_inputs()
    xh = O.rmsnorm(x, w["gamma_attn"], cfg["rms_eps"])
    q = O.linear(xh, w["w_q"]).reshape(3, 2, 2)
    k = O.linear(xh, w["w_k"]).reshape(3, 1, 2)
    v = O.linear(xh, w["w_v"]).reshape(3, 1, 2)
    q = O.apply_rope_rotate_half(q, np.arange(3), 1e6)
    k = O.apply_rope_rotate_half(k, np.arange(3), 1e6)
    _, p = O.gqa_attention(q, k, v, np.arange(3), np.arange(3), return_probs=True)
    assert np.max(np.abs(p[0] - p[1])) > 1e-3


def test_single_token_layer_passes_v_through_residual():
    """T=1: the only visible key is the token itself, so each head outputs its
    V row (§9), untouched by QK-norm and RoPE (§5, §6), and the first residual
    adds the raw X (§2).  With W_o the identity and W_down = 0, Y - X is the
    concatenation of the V heads in g(h) order."""
    cfg = small_cfg(d=16, n_q_heads=4, n_kv_heads=2, head_dim=4)
    w = rand_weights(cfg, 9, bias=True)
    cfg["qkv_bias"] = 1
    w["w_o"] = np.eye(16)
    w["w_down"] = np.zeros_like(w["w_down"])
    x = np.random.default_rng(10).standard_normal((1, 16))
    kc = np.zeros((2, 4, 4))
    vc = np.zeros_like(kc)
    y = O.layer_forward(x, w, cfg, [37], kc, vc, [0])
    xh = x[0] * w["gamma_attn"] / np.sqrt(np.mean(x[0] ** 2) + 1e-6)
    v = w["w_v"] @ xh + w["b_v"]  # [Hkv*dh], plain projection
    expect = np.concatenate([v[0:4], v[0:4], v[4:8], v[4:8]])
    assert np.allclose(y[0] - x[0], expect, atol=1e-13)
    assert np.allclose(vc[:, 0, :].reshape(-1), v, atol=1e-14)


def test_prefill_then_decode_equals_longer_prefill():
    """Qwen2.5-7B 结构拆解 §09.1: K/V of earlier positions never change, so the
    last row of prefill(T) equals prefill(T-1) followed by one decode step."""
    cfg = small_cfg()
    w = rand_weights(cfg, 11, bias=True)
    cfg["qkv_bias"] = 1
    x = np.random.default_rng(12).standard_normal((7, cfg["d"]))
    y_full, kf, vf = run_layer(x, w, cfg, max_seq=8)
    kc = np.zeros((cfg["n_kv_heads"], 8, cfg["head_dim"]))
    vc = np.zeros_like(kc)
    O.layer_forward(x[:6], w, cfg, np.arange(6), kc, vc, np.arange(6))
    y_dec = O.layer_forward(x[6:], w, cfg, [6], kc, vc, [6])
    assert np.max(np.abs(y_dec[0] - y_full[6])) < 1e-12
    assert np.max(np.abs(kc - kf)) < 1e-12 and np.max(np.abs(vc - vf)) < 1e-12


# ---------------------------------------------------------------- SwiGLU


def test_silu_textbook_values():
    assert O.silu(0.0) == 0.0
    assert O.silu(1.0) == pytest.approx(0.7310585786300049, rel=1e-15)
    assert O.silu(40.0) == pytest.approx(40.0, rel=1e-15)
    assert abs(O.silu(-40.0)) < 1e-15


def test_swiglu_applies_silu_to_gate():
    """推理系统 03 §10: F = (SiLU(Z W_gate) * (Z W_up)) W_down.

    d=f=1, R=[3] so Z = 3/sqrt(9+eps) ~ 1; W_gate=10, W_up=2, W_down=1 gives
    F = 2*SiLU(10) (SiLU on up instead would give 10*SiLU(2) = 17.6).
    SiLU(10) = 10/(1+e^-10) = 9.999546021312976.
    """
    cfg = dict(rms_eps=0.0)
    w = {"gamma_mlp": np.ones(1), "w_gate": np.array([[10.0]]),
         "w_up": np.array([[2.0]]), "w_down": np.array([[1.0]])}
    y = O.mlp_block(np.array([[3.0]]), w, cfg)
    assert y[0, 0] - 3.0 == pytest.approx(2 * 9.999546021312976, rel=1e-14)


# ---------------------------------------------------------------- MoE


def test_topk_matches_brute_force_over_subsets():
    """Top-k by logit equals the k-subset with the largest logit sum (E=6, k=2)."""
    rng = np.random.default_rng(13)
    for trial in range(50):
        z = rng.standard_normal((1, 5))
        wr = rng.standard_normal((6, 5))
        logits, idx, wts, gap = O.router_topk(z, wr, None, 2)
        best = max(itertools.combinations(range(6), 2),
                   key=lambda s: sum(logits[0, list(s)]))
        assert sorted(idx[0].tolist()) == sorted(best)
        assert wts[0].sum() == pytest.approx(1.0, abs=1e-15)
        assert gap[0] > 0 or trial  # generic inputs have no ties


def test_topk_tie_break_prefers_lower_index():
    logits_w = np.array([[1.0], [2.0], [2.0], [0.5]])  # experts 1 and 2 tie
    _, idx, _, gap = O.router_topk(np.ones((1, 1)), logits_w, None, 1)
    assert idx[0].tolist() == [1] and gap[0] == 0.0


def test_gating_softmax_over_k_equals_renormalised_full_softmax():
    """Qwen2.5-7B 结构拆解 §10.2 renormalises the top-k of a softmax over all E;
    the lecture notes' router section takes a softmax over the k selected
    logits.  The two agree exactly for norm_topk_prob=True."""
    rng = np.random.default_rng(14)
    z = rng.standard_normal((8, 6))
    wr = rng.standard_normal((16, 6))
    br = rng.standard_normal(16)
    logits, idx, wts, _ = O.router_topk(z, wr, br, 4)
    p = np.exp(logits - logits.max(1, keepdims=True))
    p /= p.sum(1, keepdims=True)
    sel = np.take_along_axis(p, idx, 1)
    assert np.allclose(sel / sel.sum(1, keepdims=True), wts, atol=1e-15)
    # ranking by probability is ranking by logit
    assert np.array_equal(np.argsort(-p, 1, kind="stable")[:, :4], idx)


def test_moe_with_one_expert_is_the_dense_mlp():
    """E = k = 1: the single expert gets weight 1, so MoE equals the dense MLP."""
    cfg = dict(rms_eps=1e-6, top_k=1)
    rng = np.random.default_rng(15)
    d, f = 8, 12
    dense = {"gamma_mlp": 1 + 0.1 * rng.standard_normal(d),
             "w_gate": rng.standard_normal((f, d)), "w_up": rng.standard_normal((f, d)),
             "w_down": rng.standard_normal((d, f))}
    moe = {"gamma_mlp": dense["gamma_mlp"], "w_router": rng.standard_normal((1, d)),
           "w_gate": dense["w_gate"][None], "w_up": dense["w_up"][None],
           "w_down": dense["w_down"][None]}
    r = rng.standard_normal((5, d))
    y_moe = O.moe_block(r, moe, cfg)[0]
    assert np.allclose(y_moe, O.mlp_block(r, dense, cfg), rtol=0, atol=1e-13)


def test_moe_output_is_gated_sum_of_chosen_experts():
    """Qwen2.5-7B 结构拆解 §10.2: y = sum_i w_i E_i(x), a plain element-wise sum.

    E=3, k=2 and expert 2 made identically zero: a token routed to {0, 1}
    gets w0 E0 + w1 E1, each expert evaluated as a one-expert MoE."""
    rng = np.random.default_rng(16)
    d, f = 6, 10
    w = {"gamma_mlp": np.ones(d), "w_router": np.array([[5.0] * d, [4.0] * d, [-9.0] * d]),
         "w_gate": rng.standard_normal((3, f, d)), "w_up": rng.standard_normal((3, f, d)),
         "w_down": rng.standard_normal((3, d, f))}
    w["w_down"][2] = 0.0
    r = np.abs(rng.standard_normal((1, d))) + 0.5  # positive row: logits 5s > 4s > -9s
    y, logits, idx, wts, gap, z = O.moe_block(r, w, dict(rms_eps=1e-6, top_k=2))
    assert idx[0].tolist() == [0, 1]
    s = z[0].sum()
    assert wts[0, 0] == pytest.approx(1 / (1 + math.exp(-s)), rel=1e-13)
    singles = []
    for e in (0, 1):
        one = {"gamma_mlp": w["gamma_mlp"], "w_router": np.zeros((1, d)),
               "w_gate": w["w_gate"][e:e + 1], "w_up": w["w_up"][e:e + 1],
               "w_down": w["w_down"][e:e + 1]}
        singles.append(O.moe_block(r, one, dict(rms_eps=1e-6, top_k=1))[0] - r)
    assert np.allclose(y - r, wts[0, 0] * singles[0] + wts[0, 1] * singles[1], atol=1e-13)


def test_topk_without_renormalisation_is_the_full_softmax_probability():
    """Qwen2.5-7B 结构拆解 §10.2, norm_topk_prob = false: the k weights are the
    selected experts' probabilities under the softmax over all experts.

    E = 2, k = 1: the one weight is the logistic of the logit difference; and
    in general the renormalised weights are these divided by their sum."""
    rng = np.random.default_rng(30)
    z = rng.standard_normal((5, 4))
    w_r = rng.standard_normal((2, 4))
    logits, idx, wts, _ = O.router_topk(z, w_r, None, 1, norm_topk_prob=False)
    other = 1 - idx[:, 0]
    diff = logits[np.arange(5), idx[:, 0]] - logits[np.arange(5), other]
    assert np.allclose(wts[:, 0], 1 / (1 + np.exp(-diff)), rtol=1e-13)
    w_r = rng.standard_normal((6, 4))
    _, idx_n, wts_n, _ = O.router_topk(z, w_r, None, 3, norm_topk_prob=True)
    _, idx_r, wts_r, _ = O.router_topk(z, w_r, None, 3, norm_topk_prob=False)
    assert np.array_equal(idx_n, idx_r)
    assert np.all(wts_r.sum(axis=1) < 1)
    assert np.allclose(wts_r / wts_r.sum(axis=1, keepdims=True), wts_n, rtol=1e-13)


def test_shared_expert_is_a_sigmoid_gated_dense_swiglu():
    """Qwen2.5-7B 结构拆解 §10.1: y_shared = sigmoid(x W_sg) SharedExpert(x),
    added to the routed sum; the shared expert is a plain SwiGLU.

    One routed expert (weight 1) plus a shared expert: with W_sg = 0 the gate is
    exactly 1/2, so y - r = MLP_routed + MLP_shared / 2, each term checked
    against the dense MLP block; a large positive gate logit gives ~1."""
    rng = np.random.default_rng(31)
    d, f, sf = 6, 8, 12
    gam = 1 + 0.1 * rng.standard_normal(d)
    w = {"gamma_mlp": gam, "w_router": np.zeros((1, d)),
         "w_gate": rng.standard_normal((1, f, d)), "w_up": rng.standard_normal((1, f, d)),
         "w_down": rng.standard_normal((1, d, f)),
         "w_shared_gate": rng.standard_normal((sf, d)), "w_shared_up": rng.standard_normal((sf, d)),
         "w_shared_down": rng.standard_normal((d, sf)), "w_shared_expert_gate": np.zeros(d)}
    cfg = dict(rms_eps=1e-6, top_k=1, shared_ffn=sf)
    r = rng.standard_normal((3, d))
    y = O.moe_block(r, w, cfg)[0]
    routed = O.mlp_block(r, {"gamma_mlp": gam, "w_gate": w["w_gate"][0], "w_up": w["w_up"][0],
                             "w_down": w["w_down"][0]}, cfg) - r
    shared = O.mlp_block(r, {"gamma_mlp": gam, "w_gate": w["w_shared_gate"],
                             "w_up": w["w_shared_up"], "w_down": w["w_shared_down"]}, cfg) - r
    assert np.allclose(y - r, routed + 0.5 * shared, atol=1e-12)
    w["w_shared_expert_gate"] = 50.0 * np.sign(O.rmsnorm(r, gam, 1e-6)[0])
    z0 = O.rmsnorm(r, gam, 1e-6)[0]
    g = O.sigmoid(z0 @ w["w_shared_expert_gate"])
    assert g > 1 - 1e-12
    y0 = O.moe_block(r[:1], w, cfg)[0]
    assert np.allclose(y0 - r[:1], routed[:1] + g * shared[:1], atol=1e-10)
    with np.errstate(over="ignore"):
        assert O.sigmoid(0.0) == 0.5 and O.sigmoid(-800.0) == 0.0


# ---------------------------------------------------------------- head


def test_head_last_token_identity_lm_head():
    """Qwen2.5-7B 结构拆解 §03.8: logits = RMSNorm_final(y_last) W_lm^T."""
    y = np.array([[1.0, 0.0, -1.0, 0.5]])
    logits = O.head_last_token(y, np.ones(4), np.eye(4), 0.0)
    assert np.allclose(logits[0], np.array([1.0, 0.0, -1.0, 0.5]) / 0.75, atol=1e-15)
