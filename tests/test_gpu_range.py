"""FP16 operand range on the GPU: nothing overflows silently.

The layer's GEMM operands are FP16 (weights packed from BF16, normalised
activations, the attention output C and the SwiGLU product H), while the
pages define the layer in BF16 ("推理系统 03" §3: BF16 storage with an FP32
mean square).  BF16 reaches 3.4e38, FP16 only 65504.  Real checkpoints carry
outlier channels, and H = SiLU(gate) * up is the first place one would pass
65504.  The library therefore checks every FP16 store: a value that FP16
cannot hold is stored as +-65504 and QWEN_ERR_OVERFLOW is recorded in the
status word, and a weight beyond FP16 makes qwen_layer_create fail.  These
tests build such inputs and check that the status says so, that every output
stays finite, and that rows the outlier does not reach still match the FP64
oracle.
"""

import numpy as np
import pytest

import oracle
import synth
from layer_harness import GpuLayer, f64
from parity import assert_parity

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

QWEN_ERR_OVERFLOW = 7
SHAPE = synth.TINY  # d=512, 8 Q heads, 2 KV heads, dh=64, f=1536, QK-norm


def _outlier_weights(tag):
    """One gate row and its up row read channel 0 with weight 100: a token
    whose channel 0 dominates has z_0 ~ sqrt(d) gamma_0 ~ 22, so gate and up
    of feature 7 are ~2e3 and H_7 ~ 5e6, far past FP16.  Every other token
    has channel 0 at zero (_x_with_outlier), so its H stays ordinary."""
    w = synth.layer_weights(SHAPE, tag)
    w["w_gate"][7, 0] = 100.0
    w["w_up"][7, 0] = 100.0
    return w


def _x_with_outlier(shape, tag, rows):
    x = synth.activations(shape, tag).reshape(-1, SHAPE.d)
    x[:, 0] = 0.0
    for r in rows:
        x[r, 0] = 2000.0
    return x.reshape(shape)


def test_prefill_outlier_channel_reports_overflow():
    T = 96
    w = _outlier_weights("range_pf")
    x = _x_with_outlier([1, T, SHAPE.d], "range_pf", [40])
    g = GpuLayer(SHAPE, w, max_tokens=T, max_batch=1, max_seq=T, max_position=T)
    kc = torch.zeros((1, SHAPE.n_kv_heads, T, SHAPE.head_dim), dtype=torch.bfloat16, device="cuda")
    vc = torch.zeros_like(kc)
    pos = torch.arange(T, dtype=torch.int32, device="cuda")
    y = g.layer.prefill(x.cuda(), pos, torch.zeros(1, dtype=torch.int32, device="cuda"), kc, vc,
                        out=torch.empty((1, T, SHAPE.d), dtype=torch.bfloat16, device="cuda"))
    assert g.layer.poll_error() == QWEN_ERR_OVERFLOW
    yg = f64(y.float())[0]
    assert np.isfinite(yg).all(), "an FP16 overflow reached the output as inf/NaN"
    # the oracle's H at the outlier token is indeed beyond FP16
    w64 = synth.weights_f64(w)
    kk = np.zeros((SHAPE.n_kv_heads, T, SHAPE.head_dim))
    vv = np.zeros_like(kk)
    ref = oracle.layer_forward(f64(x)[0], w64, SHAPE.as_dict(), np.arange(T), kk, vv,
                               np.arange(T))
    assert np.abs(ref[40]).max() > 1e4
    # rows whose MLP does not see the outlier still match the oracle
    others = np.r_[0:40, 41:T]
    assert_parity(yg[others], ref[others], what="rows without the outlier")
    # the status word was cleared by the poll: a clean call reports nothing
    x_clean = _x_with_outlier([1, T, SHAPE.d], "range_pf", [])
    g.layer.prefill(x_clean.cuda(), pos, torch.zeros(1, dtype=torch.int32, device="cuda"), kc,
                    vc, out=torch.empty((1, T, SHAPE.d), dtype=torch.bfloat16, device="cuda"))
    assert g.layer.poll_error() == 0


def test_decode_outlier_channel_reports_overflow():
    B, L = 4, 50
    w = _outlier_weights("range_dec")
    x = _x_with_outlier([B, SHAPE.d], "range_dec", [2])
    kc, vc = synth.kv_cache(B, SHAPE.n_kv_heads, L + 1, SHAPE.head_dim, L, "range_dec")
    g = GpuLayer(SHAPE, w, max_tokens=B, max_batch=B, max_seq=L + 1, max_position=L + 1)
    kd, vd = kc.cuda(), vc.cuda()
    lens = torch.full((B,), L, dtype=torch.int32, device="cuda")
    y = g.layer.decode(x.cuda(), lens, lens.clone(), kd, vd,
                       out=torch.empty((B, SHAPE.d), dtype=torch.bfloat16, device="cuda"))
    assert g.layer.poll_error() == QWEN_ERR_OVERFLOW
    yg = f64(y.float())
    assert np.isfinite(yg).all()
    w64 = synth.weights_f64(w)
    for b in (0, 1, 3):
        kk, vv = f64(kc[b]), f64(vc[b])
        ref = oracle.layer_forward(f64(x)[b][None], w64, SHAPE.as_dict(), np.array([L]), kk, vv,
                                   np.array([L]))[0]
        assert_parity(yg[b], ref, what=f"decode row {b} without the outlier")


def test_decode_cache_values_beyond_fp16_report_overflow():
    """The KV cache is BF16 and may hold values FP16 cannot: a sequence whose
    cached V rows are 1e5 gives an attention output C past 65504 (C is the O
    projection's FP16 operand)."""
    B, L = 2, 40
    w = synth.layer_weights(SHAPE, "range_kv")
    x = synth.activations([B, SHAPE.d], "range_kv")
    kc, vc = synth.kv_cache(B, SHAPE.n_kv_heads, L + 1, SHAPE.head_dim, L, "range_kv")
    vc[1, :, :L] = 1.0e5
    g = GpuLayer(SHAPE, w, max_tokens=B, max_batch=B, max_seq=L + 1, max_position=L + 1)
    lens = torch.full((B,), L, dtype=torch.int32, device="cuda")
    kd, vd = kc.cuda(), vc.cuda()
    y = g.layer.decode(x.cuda(), lens, lens.clone(), kd, vd,
                       out=torch.empty((B, SHAPE.d), dtype=torch.bfloat16, device="cuda"))
    assert g.layer.poll_error() == QWEN_ERR_OVERFLOW
    assert torch.isfinite(y.float()).all()
    kk, vv = f64(kc[0]), f64(vc[0])
    ref = oracle.layer_forward(f64(x)[0][None], synth.weights_f64(w), SHAPE.as_dict(),
                               np.array([L]), kk, vv, np.array([L]))[0]
    assert_parity(f64(y.float())[0], ref, what="the sequence with an ordinary cache")


@pytest.mark.parametrize("value,ok", [(65280.0, True), (65536.0, False), (1.0e5, False)])
def test_create_refuses_weights_beyond_fp16(value, ok):
    """65280 is the largest BF16 value below FP16's limit and packs exactly;
    65536 and above would round to infinity in FP16, so create fails with
    QWEN_ERR_OVERFLOW and returns no handle."""
    import transformer_decoder_layer_gb300 as q
    w = synth.layer_weights(SHAPE, "range_w")
    w["w_down"][3, 11] = value
    if ok:
        GpuLayer(SHAPE, w, max_tokens=8, max_batch=1, max_seq=8, max_position=8)
    else:
        with pytest.raises(q.QwenError) as e:
            GpuLayer(SHAPE, w, max_tokens=8, max_batch=1, max_seq=8, max_position=8)
        assert e.value.code == QWEN_ERR_OVERFLOW


def test_chunked_prefill_over_large_cached_values_reports_overflow():
    """Prefill of a chunk onto a filled cache reads the cached BF16 K/V: cached
    V rows of 1e5 give attention outputs past 65504 in the prefill attention
    kernel's read-out.  The first sequence has an ordinary cache and must
    still match the oracle."""
    B, T, L = 2, 64, 100
    w = synth.layer_weights(SHAPE, "range_pfkv")
    x = synth.activations([B, T, SHAPE.d], "range_pfkv")
    kc, vc = synth.kv_cache(B, SHAPE.n_kv_heads, L + T, SHAPE.head_dim, [L, L], "range_pfkv")
    vc[1, :, :L] = 1.0e5
    g = GpuLayer(SHAPE, w, max_tokens=B * T, max_batch=B, max_seq=L + T, max_position=L + T)
    kd, vd = kc.cuda(), vc.cuda()
    pos = torch.arange(L, L + T, dtype=torch.int32, device="cuda").repeat(B)
    start = torch.full((B,), L, dtype=torch.int32, device="cuda")
    y = g.layer.prefill(x.cuda(), pos, start, kd, vd,
                        out=torch.empty((B, T, SHAPE.d), dtype=torch.bfloat16, device="cuda"))
    assert g.layer.poll_error() == QWEN_ERR_OVERFLOW
    assert torch.isfinite(y.float()).all()
    kk, vv = f64(kc[0]), f64(vc[0])
    ref = oracle.layer_forward(f64(x)[0], synth.weights_f64(w), SHAPE.as_dict(),
                               np.arange(L, L + T), kk, vv, np.arange(L, L + T))
    assert_parity(f64(y.float())[0], ref, what="the sequence with an ordinary cache")
