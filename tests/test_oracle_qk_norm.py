"""Pins of the oracle's QK-norm step ("推理系统 03" §5, with §6 for the order).

The page fixes four facts about QK-norm in a Qwen3 layer:
  * each head vector is normalised on its own, the mean square taken over its
    dh channels and not over all heads together;
  * Q heads share one length-dh gamma (gamma_q) and K heads another (gamma_k);
  * V is not normalised;
  * the order is projection -> QK-norm -> RoPE.

Every pin below uses hand-built weights whose outputs have closed forms
(textbook cos/sin values and rational RMS values), so none of them re-types
the oracle's code.  The last test plants each plausible mistake in the
oracle's Q/K/V step and checks that the matching pin fails.

Construction shared by the pins: d = 16, two Q heads and two K/V heads of
dh = 4, gamma_attn = 1 and eps = 0.  Token t's input is the unit vector e_t,
so RMSNorm_1 gives exactly 4 e_t and each projection of token t is 4 times
column t of its weight.  W_o copies the 8 attention channels into the first 8
outputs and W_down = 0, so Y - X is the concatenated attention output.
RoPE theta = 100, so pair (0, 2) turns by p radians and pair (1, 3) by p/10.
"""

import math

import numpy as np
import pytest

import oracle as O
import oracle.layer as OL

GAMMA_Q = np.array([0.5, 1.0, 2.0, 1.5])   # gamma_q[i] != gamma_q[i + 2]
GAMMA_K = np.array([1.0, 2.0, 0.5, 3.0])   # and gamma_q != gamma_k
CFG = dict(d=16, n_q_heads=2, n_kv_heads=2, head_dim=4, ffn=2, qkv_bias=0,
           qk_norm=1, rope_theta=100.0, rms_eps=0.0)


def weights(q_cols, k_cols, v_cols):
    """q_cols[t] etc. are token t's raw projection [8] (two heads of 4)."""
    w = {
        "gamma_attn": np.ones(16), "gamma_mlp": np.ones(16),
        "gamma_q": GAMMA_Q.copy(), "gamma_k": GAMMA_K.copy(),
        "w_q": np.zeros((8, 16)), "w_k": np.zeros((8, 16)), "w_v": np.zeros((8, 16)),
        "w_o": np.vstack([np.eye(8), np.zeros((8, 8))]),
        "w_gate": np.zeros((2, 16)), "w_up": np.zeros((2, 16)), "w_down": np.zeros((16, 2)),
    }
    for t, (q, k, v) in enumerate(zip(q_cols, k_cols, v_cols)):
        w["w_q"][:, t] = np.asarray(q, dtype=np.float64) / 4.0
        w["w_k"][:, t] = np.asarray(k, dtype=np.float64) / 4.0
        w["w_v"][:, t] = np.asarray(v, dtype=np.float64) / 4.0
    return w


def run(w, positions, slots):
    t = len(positions)
    x = np.eye(16)[:t]
    kc = np.zeros((2, max(slots) + 1, 4))
    vc = np.zeros_like(kc)
    y = O.layer_forward(x, w, CFG, np.asarray(positions), kc, vc, np.asarray(slots))
    return y - x, kc, vc


# ------------------------------------------------------------------ the pins


def pin_per_head_normalisation():
    """Per-head mean square, shared gamma_k: one token at position 0 (no
    rotation) whose K heads are [3,4,0,0] (RMS 2.5) and [100,0,0,0] (RMS 50).
    The cached rows are gamma_k * k / RMS(k) of each head on its own:
    [1.2, 3.2, 0, 0] and [2, 0, 0, 0].

    On the Q side two heads [1,1,0,0] and [100,100,0,0] must give the same
    attention probabilities, since each normalises to sqrt(2) [1,1,0,0].
    Fails if the norm runs over all heads together, if gamma_q and gamma_k
    are swapped, or if QK-norm is skipped."""
    w = weights([[1, 1, 0, 0, 100, 100, 0, 0]], [[3, 4, 0, 0, 100, 0, 0, 0]],
                [[1, 0, 0, 0, 1, 0, 0, 0]])
    _, kc, _ = run(w, [0], [0])
    assert np.allclose(kc[0, 0], [1.2, 3.2, 0.0, 0.0], rtol=0, atol=1e-15)
    assert np.allclose(kc[1, 0], [2.0, 0.0, 0.0, 0.0], rtol=0, atol=1e-15)

    # Q side: two tokens at position 0 (no rotation).  Keys: token 0 has
    # [1,0,0,0] in both heads -> gamma_k * [2,0,0,0] = [2,0,0,0]; token 1 has
    # [0,1,0,0] -> [0,4,0,0].  Query of token 1: head 0 [1,1,0,0], head 1
    # [100,100,0,0], both -> gamma_q * sqrt(2)[1,1,0,0] = sqrt(2)[0.5,1,0,0].
    # Scores / sqrt(4): s0 = sqrt(2)/2, s1 = 2 sqrt(2); V rows e0 and e1, so
    # head output = [p0, p1, 0, 0] with p0 = 1 / (1 + e^{1.5 sqrt(2)}).
    q = [1, 1, 0, 0, 100, 100, 0, 0]
    w = weights([q, q], [[1, 0, 0, 0, 1, 0, 0, 0], [0, 1, 0, 0, 0, 1, 0, 0]],
                [[1, 0, 0, 0, 1, 0, 0, 0], [0, 1, 0, 0, 0, 1, 0, 0]])
    y, _, _ = run(w, [0, 0], [0, 1])
    p0 = 1.0 / (1.0 + math.exp(1.5 * math.sqrt(2.0)))
    expect = [p0, 1 - p0, 0, 0, p0, 1 - p0, 0, 0]
    assert np.allclose(y[1, :8], expect, rtol=0, atol=1e-15)


def pin_gammas_in_rotated_score():
    """gamma_q scales Q and gamma_k scales K, seen in a score across a
    position difference.  Token 0 at position 0: key [0,0,1,0] -> gamma_k *
    [0,0,2,0] = [0,0,1,0].  Token 1 at position 1: query [1,0,0,0] ->
    gamma_q * [2,0,0,0] = [1,0,0,0], turned by 1 rad into [cos 1, 0, sin 1, 0];
    key [1,0,0,0] -> [2,0,0,0] turned into [2 cos 1, 0, 2 sin 1, 0].
    Scores / 2: s0 = sin(1)/2, s1 = 1, so p0 = 1 / (1 + e^{1 - sin(1)/2}).
    With the two gammas swapped s0 = 4 sin 1 and p0 flips above 1/2."""
    w = weights([[1, 0, 0, 0] * 2, [1, 0, 0, 0] * 2],
                [[0, 0, 1, 0] * 2, [1, 0, 0, 0] * 2],
                [[1, 0, 0, 0] * 2, [0, 1, 0, 0] * 2])
    y, _, _ = run(w, [0, 1], [0, 1])
    p0 = 1.0 / (1.0 + math.exp(1.0 - math.sin(1.0) / 2.0))
    expect = [p0, 1 - p0, 0, 0] * 2
    assert np.allclose(y[1, :8], expect, rtol=0, atol=1e-15)


def pin_norm_before_rope():
    """Order projection -> QK-norm -> RoPE, with gamma_k[i] != gamma_k[i+2].
    One token at position 1 (slot 0) with K heads [1,2,3,4] and [4,3,2,1]
    (RMS sqrt(7.5) each).  a = gamma_k * k / sqrt(7.5), then pair (0,2) turns
    by 1 rad and pair (1,3) by 0.1 rad.  Rotating first and scaling after
    gives a different vector because gamma_k is not pair-symmetric."""
    k0, k1 = [1.0, 2.0, 3.0, 4.0], [4.0, 3.0, 2.0, 1.0]
    w = weights([[1, 0, 0, 0] * 2], [k0 + k1], [[1, 0, 0, 0] * 2])
    _, kc, _ = run(w, [1], [0])
    c1, s1, c2, s2 = math.cos(1.0), math.sin(1.0), math.cos(0.1), math.sin(0.1)
    r = math.sqrt(7.5)
    for h, k in enumerate((k0, k1)):
        a = [GAMMA_K[i] * k[i] / r for i in range(4)]
        expect = [a[0] * c1 - a[2] * s1, a[1] * c2 - a[3] * s2,
                  a[2] * c1 + a[0] * s1, a[3] * c2 + a[1] * s2]
        assert np.allclose(kc[h, 0], expect, rtol=0, atol=1e-14)


def pin_v_not_normalised():
    """V is the plain projection: V heads [3,4,0,0] and [0,0,100,0] are cached
    as they are, and with one token the attention output is V itself."""
    v = [3, 4, 0, 0, 0, 0, 100, 0]
    w = weights([[1, 2, 3, 4] * 2], [[4, 3, 2, 1] * 2], [v])
    y, _, vc = run(w, [5], [0])
    assert np.array_equal(vc[:, 0, :].reshape(-1), np.array(v, dtype=np.float64))
    assert np.allclose(y[0, :8], v, rtol=0, atol=1e-13)


@pytest.mark.parametrize("pin", [pin_per_head_normalisation, pin_gammas_in_rotated_score,
                                 pin_norm_before_rope, pin_v_not_normalised])
def test_qk_norm_pin(pin):
    """推理系统 03 §5-§6 (see each pin's docstring)."""
    pin()


def test_shift_invariance_with_qk_norm():
    """推理系统 03 §14 experiment 2 with QK-norm on and gammas that are neither
    uniform nor pair-symmetric: shifting every position leaves the layer
    output unchanged within 1e-12, since QK-norm acts per token before RoPE."""
    cfg = dict(d=16, n_q_heads=4, n_kv_heads=2, head_dim=8, ffn=24, qkv_bias=1,
               qk_norm=1, rope_theta=1.0e6, rms_eps=1.0e-6)
    rng = np.random.default_rng(40)
    w = {
        "gamma_attn": 1 + 0.1 * rng.standard_normal(16),
        "gamma_mlp": 1 + 0.1 * rng.standard_normal(16),
        "gamma_q": 1 + 0.5 * rng.standard_normal(8),
        "gamma_k": 1 + 0.5 * rng.standard_normal(8),
        "w_q": 0.4 * rng.standard_normal((32, 16)), "w_k": 0.4 * rng.standard_normal((16, 16)),
        "w_v": 0.4 * rng.standard_normal((16, 16)), "w_o": 0.4 * rng.standard_normal((16, 32)),
        "b_q": 0.1 * rng.standard_normal(32), "b_k": 0.1 * rng.standard_normal(16),
        "b_v": 0.1 * rng.standard_normal(16),
        "w_gate": 0.3 * rng.standard_normal((24, 16)), "w_up": 0.3 * rng.standard_normal((24, 16)),
        "w_down": 0.3 * rng.standard_normal((16, 24)),
    }
    assert np.min(np.abs(w["gamma_q"][:4] - w["gamma_q"][4:])) > 1e-3
    assert np.min(np.abs(w["gamma_k"][:4] - w["gamma_k"][4:])) > 1e-3
    x = rng.standard_normal((6, 16))

    def fwd(pos):
        kc = np.zeros((2, 6, 8))
        return O.layer_forward(x, w, cfg, np.asarray(pos), kc, np.zeros_like(kc), np.arange(6))

    y0 = fwd(np.arange(6))
    assert np.max(np.abs(fwd(np.arange(6) + 7) - y0)) < 1e-12
    assert np.max(np.abs(fwd(np.arange(6) + 1000) - y0)) < 1e-12
    assert np.max(np.abs(fwd([0, 1, 2, 3, 4, 9]) - y0)) > 1e-6


# ------------------------------------------------ planted mistakes (CPU only)


def _mutant_qkv(kind):
    """The oracle's Q/K/V step with one planted mistake of the given kind."""
    def qkv(xh, w, cfg, positions):
        t = xh.shape[0]
        hq, hkv, dh = cfg["n_q_heads"], cfg["n_kv_heads"], cfg["head_dim"]
        eps, theta = cfg["rms_eps"], cfg["rope_theta"]
        q = O.linear(xh, w["w_q"]).reshape(t, hq, dh)
        k = O.linear(xh, w["w_k"]).reshape(t, hkv, dh)
        v = O.linear(xh, w["w_v"]).reshape(t, hkv, dh)
        gq, gk = w["gamma_q"], w["gamma_k"]
        if kind == "swap_gammas":
            gq, gk = gk, gq
        if kind == "rope_first":
            q = O.apply_rope_rotate_half(q, positions, theta)
            k = O.apply_rope_rotate_half(k, positions, theta)
        if kind == "across_heads":
            q = O.rmsnorm(q.reshape(t, -1), np.tile(gq, hq), eps).reshape(t, hq, dh)
            k = O.rmsnorm(k.reshape(t, -1), np.tile(gk, hkv), eps).reshape(t, hkv, dh)
        elif kind != "no_norm":
            q = O.rmsnorm(q, gq, eps)
            k = O.rmsnorm(k, gk, eps)
        if kind == "norm_v":
            v = O.rmsnorm(v, gk, eps)
        if kind != "rope_first":
            q = O.apply_rope_rotate_half(q, positions, theta)
            k = O.apply_rope_rotate_half(k, positions, theta)
        return q, k, v
    return qkv


@pytest.mark.parametrize("kind,pin", [
    ("across_heads", pin_per_head_normalisation),
    ("no_norm", pin_per_head_normalisation),
    ("swap_gammas", pin_per_head_normalisation),
    ("swap_gammas", pin_gammas_in_rotated_score),
    ("rope_first", pin_norm_before_rope),
    ("norm_v", pin_v_not_normalised),
])
def test_planted_qk_norm_mistake_fails_its_pin(monkeypatch, kind, pin):
    """Each plausible slip in the QK-norm step, planted in the oracle, makes
    the pin aimed at it fail; the unmutated replica passes all four."""
    monkeypatch.setattr(OL, "_qkv", _mutant_qkv("none"))
    for p in (pin_per_head_normalisation, pin_gammas_in_rotated_score,
              pin_norm_before_rope, pin_v_not_normalised):
        p()
    monkeypatch.setattr(OL, "_qkv", _mutant_qkv(kind))
    with np.errstate(all="ignore"), pytest.raises(AssertionError):
        pin()
