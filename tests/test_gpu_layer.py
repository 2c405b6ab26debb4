"""Layer parity of the CUDA path (through the C ABI) against the FP64 oracle.

Dense prefill (tiny Qwen3 layer, Qwen3-8B-shaped layer), ragged and chunked
prefill, Qwen2.5-7B-shaped decode against a 4096-slot cache, and GPU-side
invariants (causality is bit-exact, prefill/decode agree)."""

import numpy as np
import pytest

import synth
from layer_harness import GpuLayer, f64, oracle_prefill
from parity import assert_parity

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


def _prefill_case(shape, tag, B, T, cache_start=None, max_seq=None, prefilled=0, rows=None,
                  positions=None):
    w_cpu = synth.layer_weights(shape, tag)
    x = synth.activations([B, T, shape.d], tag)
    cache_start = [0] * B if cache_start is None else cache_start
    max_seq = max_seq or (max(cache_start) + T)
    pos = (np.asarray(cache_start)[:, None] + np.arange(T)[None, :]) if positions is None \
        else np.asarray(positions)
    kc, vc = synth.kv_cache(B, shape.n_kv_heads, max_seq, shape.head_dim, prefilled, tag)
    g = GpuLayer(shape, w_cpu, max_tokens=B * T, max_batch=B, max_seq=max_seq,
                 max_position=int(pos.max()) + 1)
    kd, vd = kc.cuda(), vc.cuda()
    y = g.prefill(x, pos, cache_start, kd, vd)
    ref, k_ref, v_ref = oracle_prefill(shape, synth.weights_f64(w_cpu), f64(x), pos,
                                       cache_start, f64(kc), f64(vc), rows=rows)
    yg = f64(y.float())
    if rows is not None:
        yg = yg[:, rows]
    return yg, ref, f64(kd.float()), k_ref, f64(vd.float()), v_ref


def test_tiny_layer_prefill_full():
    """Tiny Qwen3-style layer, B=1, T=128, d=512, dh=64, QK-norm, seed 0."""
    y, ref, k, kr, v, vr = _prefill_case(synth.TINY, "tiny", 1, 128)
    assert_parity(y, ref, what="Y")
    assert_parity(k, kr, what="K cache")
    assert_parity(v, vr, what="V cache")


def test_ragged_batch_prefill():
    """Two sequences, T=200 (a partial 128-row tile), dh=64."""
    y, ref, k, kr, v, vr = _prefill_case(synth.TINY, "ragged", 2, 200)
    assert_parity(y, ref, what="Y")
    assert_parity(k, kr, what="K cache")


def test_chunked_prefill_onto_filled_cache():
    """Tokens appended after 70 and 131 pre-filled slots: queries see the old keys."""
    y, ref, k, kr, v, vr = _prefill_case(synth.TINY, "chunk", 2, 96, cache_start=[70, 131],
                                         max_seq=300, prefilled=[70, 131])
    assert_parity(y, ref, what="Y")
    assert_parity(k, kr, what="K cache")
    assert_parity(v, vr, what="V cache")


QWEN3_SMALL = synth.LayerConfig(d=1024, n_q_heads=16, n_kv_heads=4, head_dim=128, ffn=2816,
                                qk_norm=1)


def test_qwen3_style_dh128_prefill():
    """dh=128, G=4, several query tiles and a ragged tail (T=333)."""
    y, ref, k, kr, v, vr = _prefill_case(QWEN3_SMALL, "q3s", 2, 333)
    assert_parity(y, ref, what="Y")
    assert_parity(k, kr, what="K cache")
    assert_parity(v, vr, what="V cache")


def test_qwen3_style_dh128_chunked_prefill():
    """dh=128 chunk appended to filled caches (slots 45 and 200): keys come from
    the BF16 cache, partly written by this call."""
    y, ref, k, kr, v, vr = _prefill_case(QWEN3_SMALL, "q3chunk", 2, 150, cache_start=[200, 45],
                                         max_seq=400, prefilled=[200, 45])
    assert_parity(y, ref, what="Y")
    assert_parity(k, kr, what="K cache")
    assert_parity(v, vr, what="V cache")


def test_qwen25_style_bias_prefill():
    """qkv bias, no QK-norm, G=7, dh=128."""
    shape = synth.LayerConfig(d=896, n_q_heads=14, n_kv_heads=2, head_dim=128, ffn=1792,
                              qkv_bias=1)
    y, ref, k, kr, v, vr = _prefill_case(shape, "q25s", 1, 257)
    assert_parity(y, ref, what="Y")
    assert_parity(k, kr, what="K cache")


def test_prefill_attention_mixed_work_items():
    """7 query heads per KV group (three two-head items and one one-head item per
    group and query tile), two sequences of 2560 tokens of which the second
    continues a filled cache (BF16 operands): 320 attention work items dealt
    over 152 SMs in alternating directions, so CTAs process one-head and
    two-head items, fresh and cached, one after another."""
    shape = synth.LayerConfig(d=896, n_q_heads=14, n_kv_heads=2, head_dim=128, ffn=1792,
                              qkv_bias=1)
    T = 2560
    rng = np.random.default_rng(7)
    rows = np.unique(np.r_[0, 127, 128, 1279, 1280, T - 129, T - 128, T - 1,
                           rng.integers(0, T, 24)])
    y, ref, k, kr, v, vr = _prefill_case(shape, "mixed_items", 2, T, cache_start=[0, 300],
                                         prefilled=[0, 300], rows=rows)
    assert_parity(y, ref, what="Y")
    assert_parity(k, kr, what="K cache")
    assert_parity(v, vr, what="V cache")


def test_single_token_prefill_over_mixed_cache_offsets():
    """T=1 for three sequences whose chunks start at slots 0, 5 and 17: one
    query row per attention item, fresh and cached items in one call."""
    shape = synth.LayerConfig(d=512, n_q_heads=8, n_kv_heads=2, head_dim=64, ffn=1536,
                              qk_norm=1)
    y, ref, k, kr, v, vr = _prefill_case(shape, "t1_mixed", 3, 1, cache_start=[0, 5, 17],
                                         max_seq=32, prefilled=[0, 5, 17])
    assert_parity(y, ref, what="Y")
    assert_parity(k, kr, what="K cache")
    assert_parity(v, vr, what="V cache")


def test_empty_calls_succeed_without_launches():
    """Zero rows, zero tokens and zero sequences are valid calls: success, no
    kernel launched, nothing written."""
    import transformer_decoder_layer_gb300 as q
    shape = synth.LayerConfig(d=512, n_q_heads=8, n_kv_heads=2, head_dim=64, ffn=256,
                              qk_norm=1, n_experts=16, top_k=4)
    g = GpuLayer(shape, synth.layer_weights(shape, "empty"), max_tokens=8, max_batch=2,
                 max_seq=8, max_position=8)
    bf, i32, dev = torch.bfloat16, torch.int32, "cuda"
    kc = torch.zeros((2, 2, 8, 64), dtype=bf, device=dev)
    vc = torch.zeros_like(kc)
    torch.cuda.synchronize()
    n0 = q.launch_count()
    assert q.linear(torch.empty((0, 512), dtype=bf, device=dev),
                    torch.zeros((256, 512), dtype=bf, device=dev)).shape == (0, 256)
    assert q.rmsnorm(torch.empty((0, 512), dtype=bf, device=dev),
                     torch.ones(512, dtype=bf, device=dev), 1e-6).shape == (0, 512)
    yp = g.layer.prefill(torch.empty((2, 0, 512), dtype=bf, device=dev),
                         torch.empty(0, dtype=i32, device=dev), torch.zeros(2, dtype=i32, device=dev),
                         kc, vc)
    assert yp.shape == (2, 0, 512)
    yd = g.layer.decode(torch.empty((0, 512), dtype=bf, device=dev),
                        torch.empty(0, dtype=i32, device=dev), torch.empty(0, dtype=i32, device=dev),
                        kc, vc)
    assert yd.shape == (0, 512)
    assert g.layer.moe_ffn(torch.empty((0, 512), dtype=bf, device=dev)).shape == (0, 512)
    assert q.launch_count() == n0
    assert g.layer.poll_error() == 0 and q.poll_error() == 0
    assert torch.count_nonzero(kc) == 0 and torch.count_nonzero(vc) == 0


@pytest.mark.parametrize("T", [1024, 4096])
def test_qwen3_8b_layer_prefill_sampled_rows(T):
    """Qwen3-8B-shaped layer at full size, sampled output rows."""
    rng = np.random.default_rng(T)
    rows = np.unique(np.r_[0, 1, 127, 128, T // 2, T - 129, T - 1, rng.integers(0, T, 24)])
    y, ref, k, kr, v, vr = _prefill_case(synth.QWEN3_8B, f"q3_8b_{T}", 1, T, rows=rows)
    assert_parity(y, ref, what="Y")
    assert_parity(k, kr, what="K cache")
    assert_parity(v, vr, what="V cache")


def test_qwen3_8b_layer_prefill_batch8():
    """B=8, T=1024 independent sequences; sampled rows of every sequence."""
    rows = np.array([0, 513, 1023])
    y, ref, _, _, _, _ = _prefill_case(synth.QWEN3_8B, "q3_8b_b8", 8, 1024, rows=rows)
    assert_parity(y, ref, what="Y")


def _decode_case(shape, tag, B, filled, max_seq):
    w_cpu = synth.layer_weights(shape, tag)
    x = synth.activations([B, shape.d], tag)
    kc, vc = synth.kv_cache(B, shape.n_kv_heads, max_seq, shape.head_dim, filled, tag)
    cache_len = [filled] * B if isinstance(filled, int) else list(filled)
    pos = np.asarray(cache_len)
    g = GpuLayer(shape, w_cpu, max_tokens=B, max_batch=B, max_seq=max_seq,
                 max_position=int(pos.max()) + 1)
    kd, vd = kc.cuda(), vc.cuda()
    y = g.decode(x, pos, cache_len, kd, vd)
    ref, k_ref, v_ref = oracle_prefill(shape, synth.weights_f64(w_cpu), f64(x)[:, None, :],
                                       pos[:, None], cache_len, f64(kc), f64(vc))
    return f64(y.float()), ref[:, 0], f64(kd.float()), k_ref, f64(vd.float()), v_ref, cache_len


@pytest.mark.parametrize("B", [1, 8])
def test_qwen25_7b_decode_full_cache(B):
    """Qwen2.5-7B-shaped decode: 4096 cached slots, the new token in slot 4096."""
    y, ref, k, kr, v, vr, cl = _decode_case(synth.QWEN25_7B, f"q25_dec{B}", B, 4096, 4097)
    assert_parity(y, ref, what="Y")
    assert_parity(k[:, :, 4096], kr[:, :, 4096], what="appended K")
    assert_parity(v[:, :, 4096], vr[:, :, 4096], what="appended V")


def test_decode_ragged_cache_lengths():
    """Per-sequence cache lengths (0, 1, 63, 64, 65, 1000), dh=64, G=4."""
    lens = [0, 1, 63, 64, 65, 1000]
    y, ref, k, kr, v, vr, cl = _decode_case(synth.TINY, "dec_ragged", len(lens), lens, 1100)
    assert_parity(y, ref, what="Y")
    for b, L in enumerate(cl):
        assert_parity(k[b, :, L], kr[b, :, L], what=f"K row b={b}")


def test_decode_batch_64_dh128_g8():
    """B=64 with per-sequence lengths around block edges, G=8."""
    shape = synth.LayerConfig(d=1024, n_q_heads=16, n_kv_heads=2, head_dim=128, ffn=2048,
                              qk_norm=1)
    lens = [int(v) for v in np.random.default_rng(3).integers(0, 700, 64)]
    y, ref, *_ = _decode_case(shape, "dec64", 64, lens, 800)
    assert_parity(y, ref, what="Y")


@pytest.mark.parametrize("B", [256, 300], ids=["swap_max", "row_tiled"])
def test_decode_large_batches(B):
    """B=256 is the largest batch of the swap-AB decode GEMMs (tokens on the
    MMA's N = 256); B=300 takes the prefill-shaped GEMMs with their fused QKV,
    residual and SwiGLU epilogues.  Ragged cache lengths; every sequence is
    checked against the oracle, with its appended K/V row."""
    lens = [int(v) for v in np.random.default_rng(B).integers(0, 90, B)]
    y, ref, k, kr, v, vr, cl = _decode_case(synth.TINY, f"dec_big{B}", B, lens, 96)
    assert_parity(y, ref, what="Y")
    for b in range(0, B, 37):
        assert_parity(k[b, :, cl[b]], kr[b, :, cl[b]], what=f"K row b={b}")
        assert_parity(v[b, :, cl[b]], vr[b, :, cl[b]], what=f"V row b={b}")


@pytest.mark.parametrize("bad", ["slot", "position"])
def test_decode_reports_out_of_range(bad):
    """A cache slot at max_seq or a position at max_position is reported as
    QWEN_ERR_RANGE in the status word (nothing is written outside the cache);
    the other sequences of the step are unaffected."""
    shape = synth.TINY
    B, S = 4, 64
    w_cpu = synth.layer_weights(shape, "dec_oor")
    x = synth.activations([B, shape.d], "dec_oor")
    kc, vc = synth.kv_cache(B, shape.n_kv_heads, S, shape.head_dim, 20, "dec_oor")
    g = GpuLayer(shape, w_cpu, max_tokens=B, max_batch=B, max_seq=S, max_position=S)
    lens = [20, 20, 20, 20]
    pos = [20, 20, 20, 20]
    if bad == "slot":
        lens[2] = S  # no slot for the new row
    else:
        pos[2] = S   # beyond the RoPE table
    kd, vd = kc.cuda(), vc.cuda()
    t = torch
    y = g.layer.decode(x.cuda(), t.as_tensor(pos, dtype=t.int32).cuda(),
                       t.as_tensor(lens, dtype=t.int32).cuda(), kd, vd)
    range_code = next(c for c, n in g.q.STATUS.items() if n == "QWEN_ERR_RANGE")
    assert g.layer.poll_error() == range_code
    assert g.layer.poll_error() == 0  # polling clears the word
    # the well-formed sequences match the oracle
    ok = [0, 1, 3]
    ref, _, _ = oracle_prefill(shape, synth.weights_f64(w_cpu), f64(x)[ok][:, None, :],
                               np.array(pos)[ok][:, None], [lens[i] for i in ok],
                               f64(kc)[ok], f64(vc)[ok])
    assert_parity(f64(y.float())[ok], ref[:, 0], what="Y of the other sequences")


def test_prefill_reproducible_bit_for_bit():
    """T=512 of a d=1024 layer (GEMMs of fewer tiles than SMs, split-tail
    tiles, split attention work items): the result matches the oracle and is
    the same, bit for bit, on every run."""
    shape = QWEN3_SMALL
    T = 512
    w_cpu = synth.layer_weights(shape, "repro")
    x = synth.activations([1, T, shape.d], "repro")
    g = GpuLayer(shape, w_cpu, T, 1, T, T)
    pos = np.arange(T)[None]
    outs = []
    for _ in range(3):
        kc, vc = (torch.zeros((1, shape.n_kv_heads, T, shape.head_dim), dtype=torch.bfloat16,
                              device="cuda") for _ in range(2))
        outs.append((g.prefill(x, pos, [0], kc, vc), kc, vc))
    for y, kc, vc in outs[1:]:
        assert torch.equal(y, outs[0][0])
        assert torch.equal(kc, outs[0][1]) and torch.equal(vc, outs[0][2])
    z = np.zeros((1, shape.n_kv_heads, T, shape.head_dim))
    ref, k_ref, _ = oracle_prefill(shape, synth.weights_f64(w_cpu), f64(x), pos, [0], z, z)
    assert_parity(f64(outs[0][0].float()), ref, what="Y")
    assert_parity(f64(outs[0][1].float()), k_ref, what="K cache")


def test_causality_bit_exact_on_gpu():
    """Changing the last position leaves earlier rows bit-identical (推理系统 03 §14)."""
    shape = QWEN3_SMALL
    w_cpu = synth.layer_weights(shape, "caus")
    x = synth.activations([1, 200, shape.d], "caus")
    g = GpuLayer(shape, w_cpu, 200, 1, 200, 200)
    pos = np.arange(200)[None]
    k1, v1 = (torch.zeros((1, 4, 200, 128), dtype=torch.bfloat16, device="cuda") for _ in range(2))
    y1 = g.prefill(x, pos, [0], k1, v1)
    x2 = x.clone()
    x2[0, -1] = -3.0
    k2, v2 = (torch.zeros_like(k1) for _ in range(2))
    y2 = g.prefill(x2, pos, [0], k2, v2)
    assert torch.equal(y1[0, :-1], y2[0, :-1])
    assert not torch.equal(y1[0, -1], y2[0, -1])


def test_prefill_then_decode_matches_longer_prefill():
    """Qwen2.5-7B 结构拆解 §09.1 on the GPU: prefill(T-1) + decode(1) ~ prefill(T)."""
    shape = QWEN3_SMALL
    w_cpu = synth.layer_weights(shape, "pd")
    T = 150
    x = synth.activations([1, T, shape.d], "pd")
    g = GpuLayer(shape, w_cpu, T, 1, T, T)
    kf, vf = (torch.zeros((1, 4, T, 128), dtype=torch.bfloat16, device="cuda") for _ in range(2))
    yf = g.prefill(x, np.arange(T)[None], [0], kf, vf)
    kc, vc = (torch.zeros_like(kf) for _ in range(2))
    g.prefill(x[:, :T - 1].contiguous(), np.arange(T - 1)[None], [0], kc, vc)
    yd = g.decode(x[:, T - 1].contiguous(), np.array([T - 1]), [T - 1], kc, vc)
    assert_parity(f64(yd.float())[0], f64(yf.float())[0, -1], what="decode vs prefill row")
    assert torch.equal(kc[:, :, :T - 1], kf[:, :, :T - 1])


@pytest.mark.parametrize("pinned", [True, False], ids=["mapped", "pageable"])
def test_decode_from_host_buffers_matches_device_call(pinned):
    """qwen_layer_decode_host gives the same bits as the device-buffer call,
    with pinned host buffers (the kernels read and write them directly) and
    with pageable ones (staged copies)."""
    shape = synth.TINY
    B, L = 5, 300
    w_cpu = synth.layer_weights(shape, "dhost")
    x = synth.activations([B, shape.d], "dhost")
    kc, vc = synth.kv_cache(B, shape.n_kv_heads, L + 1, shape.head_dim, L, "dhost")
    g = GpuLayer(shape, w_cpu, max_tokens=B, max_batch=B, max_seq=L + 1, max_position=L + 1)
    lens = np.array([L, 7, 150, L, 1], dtype=np.int32)
    k1, v1 = kc.cuda(), vc.cuda()
    y_dev = g.decode(x, lens, lens, k1, v1)
    k2, v2 = kc.cuda(), vc.cuda()
    xh = x.contiguous().clone()
    lh = torch.from_numpy(lens).clone()
    yh = torch.empty_like(xh)
    if pinned:
        xh, lh, yh = xh.pin_memory(), lh.pin_memory(), yh.pin_memory()
    g.layer.decode_host(xh, lh, lh, k2, v2, yh)
    torch.cuda.synchronize()
    assert g.layer.poll_error() == 0
    assert torch.equal(yh, y_dev.cpu())
    assert torch.equal(k1, k2) and torch.equal(v1, v2)
