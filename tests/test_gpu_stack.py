"""The 28-layer Qwen2.5-7B-shaped stack with the final norm and the lm_head on
the last position ("Qwen2.5-7B 结构拆解" §01, §03.8), through the C ABI.

* decode at the full size the bench runs (B=32, 2048 cached tokens per layer):
  the oracle recomputes two of the 32 independent sequences through all 28
  layers and the head, in FP64;
* prefill of 128 tokens through all layers against the FP64 oracle, element
  by element: prefill attention reads this call's K/V rows from FP16 copies
  (the BF16 cache rows are only read by later calls), so the BF16 storage
  rounding of the cache does not enter the prefill result;
* prefill at T=1024 (the full prefill workload): all 152064 last-token
  logits against the FP64 oracle run through the 28 layers, element by
  element at the stated tolerance;
* also at T=1024: the last-token logits equal prefill(1023) + decode(1);
  both sides are GPU results with independent rounding, so the bound is twice
  the oracle bound.
"""

import numpy as np
import pytest

import oracle
import synth
from layer_harness import f64
from parity import assert_parity

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

L_LAYERS = synth.QWEN25_7B_LAYERS
VOCAB = synth.QWEN25_7B_VOCAB
SHAPE = synth.QWEN25_7B
B_DEC, CACHED = 32, 2048


@pytest.fixture(scope="module")
def stack_setup():
    import transformer_decoder_layer_gb300 as q
    cpu_w = [synth.layer_weights(SHAPE, f"c5L{l}") for l in range(L_LAYERS)]
    gamma_f = synth.normal_bf16([SHAPE.d], synth.seed_for("c5", "gamma_final"), 0.1, 1.0)
    w_lm = synth.normal_bf16([VOCAB, SHAPE.d], synth.seed_for("c5", "w_lm"), 0.02)

    def gpu_weights():
        for w in cpu_w:
            yield {k: t.cuda() for k, t in w.items()}

    st = q.Stack(SHAPE, gpu_weights(), gamma_f.cuda(), w_lm.cuda(), max_batch=B_DEC,
                 max_seq=CACHED + 1, max_tokens=1024)
    return q, st, cpu_w, gamma_f, w_lm


def _cache_rows(l, b, n):
    tag = f"c5L{l}"
    k = synth.normal_bf16([SHAPE.n_kv_heads, n, SHAPE.head_dim], synth.seed_for(tag, f"k_cache{b}"))
    v = synth.normal_bf16([SHAPE.n_kv_heads, n, SHAPE.head_dim], synth.seed_for(tag, f"v_cache{b}"))
    return k, v


def test_stack_decode_full_size_sampled_sequences(stack_setup):
    q, st, cpu_w, gamma_f, w_lm = stack_setup
    for l in range(L_LAYERS):
        kc, vc = synth.kv_cache(B_DEC, SHAPE.n_kv_heads, CACHED + 1, SHAPE.head_dim, CACHED,
                                f"c5L{l}")
        st.k[l].copy_(kc)
        st.v[l].copy_(vc)
    x = synth.activations([B_DEC, SHAPE.d], "c5dec")
    pos = torch.full((B_DEC,), CACHED, dtype=torch.int32, device="cuda")
    logits = st.decode(x.cuda(), pos, pos.clone())
    assert st.poll_error() == 0
    got = logits.cpu().numpy()
    assert np.all(np.isfinite(got))
    cfg = SHAPE.as_dict()
    for b in (0, B_DEC - 1):
        h = f64(x)[b][None]
        for l in range(L_LAYERS):
            w64 = synth.weights_f64(cpu_w[l])
            k, v = _cache_rows(l, b, CACHED)
            kk = np.zeros((SHAPE.n_kv_heads, CACHED + 1, SHAPE.head_dim))
            vv = np.zeros_like(kk)
            kk[:, :CACHED], vv[:, :CACHED] = f64(k), f64(v)
            h = oracle.layer_forward(h, w64, cfg, np.array([CACHED]), kk, vv, np.array([CACHED]))
        ref = oracle.head_last_token(h, f64(gamma_f), f64(w_lm), cfg["rms_eps"])[0]
        assert_parity(got[b], ref, what=f"stack decode logits b={b}")


def test_stack_prefill_128_tokens(stack_setup):
    q, st, cpu_w, gamma_f, w_lm = stack_setup
    T = 128
    x = synth.activations([1, T, SHAPE.d], "c5pf")
    pos = torch.arange(T, dtype=torch.int32, device="cuda")
    start = torch.zeros(1, dtype=torch.int32, device="cuda")
    logits, _ = st.prefill(x.cuda(), pos, start)
    assert st.poll_error() == 0
    cfg = SHAPE.as_dict()
    h = f64(x)[0]
    for l in range(L_LAYERS):
        kk = np.zeros((SHAPE.n_kv_heads, T, SHAPE.head_dim))
        vv = np.zeros_like(kk)
        h = oracle.layer_forward(h, synth.weights_f64(cpu_w[l]), cfg, np.arange(T), kk, vv,
                                 np.arange(T))
    ref = oracle.head_last_token(h[-1:], f64(gamma_f), f64(w_lm), cfg["rms_eps"])[0]
    assert_parity(logits.cpu().numpy()[0], ref, what="stack prefill logits")


def test_stack_prefill_1024_last_token_logits(stack_setup):
    """Qwen2.5-7B 结构拆解 §03.8: a prefill of 1024 tokens computes logits for
    the last position only.  The oracle runs every layer over all 1024 rows
    (later layers read every row's K/V) and only the last row through the
    final layer's attention output and MLP."""
    q, st, cpu_w, gamma_f, w_lm = stack_setup
    T = 1024
    x = synth.activations([1, T, SHAPE.d], "c5pf1024")
    start = torch.zeros(1, dtype=torch.int32, device="cuda")
    logits, _ = st.prefill(x.cuda(), torch.arange(T, dtype=torch.int32, device="cuda"), start)
    assert st.poll_error() == 0
    got = logits.cpu().numpy()[0]
    cfg = SHAPE.as_dict()
    h = f64(x)[0]
    for l in range(L_LAYERS):
        kk = np.zeros((SHAPE.n_kv_heads, T, SHAPE.head_dim))
        vv = np.zeros_like(kk)
        rows = [T - 1] if l == L_LAYERS - 1 else None
        h = oracle.layer_forward(h, synth.weights_f64(cpu_w[l]), cfg, np.arange(T), kk, vv,
                                 np.arange(T), rows=rows)
    ref = oracle.head_last_token(h[-1:], f64(gamma_f), f64(w_lm), cfg["rms_eps"])[0]
    assert_parity(got, ref, what="stack prefill T=1024 logits")


def test_stack_prefill_1024_equals_prefill_then_decode(stack_setup):
    q, st, cpu_w, gamma_f, w_lm = stack_setup
    T = 1024
    x = synth.activations([1, T, SHAPE.d], "c5pf1024").cuda()
    start = torch.zeros(1, dtype=torch.int32, device="cuda")
    full, _ = st.prefill(x, torch.arange(T, dtype=torch.int32, device="cuda"), start)
    full = full.clone()
    st.prefill(x[:, :T - 1].contiguous(), torch.arange(T - 1, dtype=torch.int32, device="cuda"),
               start)
    p = torch.full((1,), T - 1, dtype=torch.int32, device="cuda")
    step = st.decode(x[:, T - 1].contiguous(), p, p.clone())
    assert st.poll_error() == 0
    assert_parity(step.cpu().numpy(), full.cpu().numpy(), atol=4e-2, rtol=4e-2, frob=1e-2,
                  what="prefill(1023)+decode vs prefill(1024)")
