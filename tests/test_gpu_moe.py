"""MoE parity of the CUDA path (through the C ABI) against the FP64 oracle.

Top-k indices must match the oracle exactly wherever the oracle's k-th minus
(k+1)-th logit gap exceeds 1e-3; where it does not, both selections are
correct, and the GPU output is compared with the oracle evaluated under the
GPU's selection (weights = softmax of the oracle logits at those experts).

Whole MoE layers are checked teacher-forced: the oracle's MoE block runs on
the residual stream R that the GPU's attention block produced (read from the
workspace), so every sampled row is compared; R itself is compared with the
oracle's attention block."""

import numpy as np
import pytest

import oracle
import synth
from layer_harness import GpuLayer, f64, workspace_region
from parity import assert_parity

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

GAP = 1e-3

SMALL_MOE = synth.LayerConfig(d=512, n_q_heads=8, n_kv_heads=2, head_dim=64, ffn=256, qk_norm=1,
                              n_experts=16, top_k=4, router_bias=1)
# Qwen2-MoE-like: q/k/v bias, weights without renormalisation, shared expert
SMALL_QWEN2_MOE = synth.LayerConfig(d=512, n_q_heads=8, n_kv_heads=2, head_dim=64, ffn=128,
                                    qkv_bias=1, n_experts=16, top_k=4, norm_topk_prob=0,
                                    shared_ffn=512)


def _gate_weights(logits, sel_idx, norm):
    """Gate weights of a given selection from the oracle's logits."""
    sel = np.take_along_axis(logits, sel_idx.astype(np.int64), axis=1)
    if norm:
        p = np.exp(sel - sel.max(1, keepdims=True))
        return p / p.sum(1, keepdims=True)
    m = logits.max(1, keepdims=True)
    return np.exp(sel - m) / np.exp(logits - m).sum(1, keepdims=True)


def _moe_reference(r64, w64, cfg, gpu_idx):
    """Oracle MoE; ambiguous tokens re-evaluated under the GPU's selection."""
    y, logits, idx, wts, gap, z = oracle.moe_block(r64, w64, cfg)
    amb = gap <= GAP
    if amb.any():
        p = _gate_weights(logits, gpu_idx, cfg.get("norm_topk_prob", 1))
        idx2 = np.where(amb[:, None], gpu_idx, idx)
        wts2 = np.where(amb[:, None], p, wts)
        y = oracle.moe_block(r64, w64, cfg, routing=(idx2, wts2))[0]
    return y, logits, idx, wts, gap


def _run_moe_ffn(shape, tag, T, fp32_input=False):
    w_cpu = synth.layer_weights(shape, tag)
    r = synth.activations([T, shape.d], tag, "r")
    g = GpuLayer(shape, w_cpu, max_tokens=T, max_batch=1, max_seq=8, max_position=8)
    k, E = shape.top_k, shape.n_experts
    idx = torch.empty((T, k), dtype=torch.int32, device="cuda")
    wts = torch.empty((T, k), dtype=torch.float32, device="cuda")
    lg = torch.empty((T, E), dtype=torch.float32, device="cuda")
    r_dev = r.cuda()
    r32 = r_dev.float() if fp32_input else None
    y = g.layer.moe_ffn(r_dev, r_fp32=r32, topk_idx=idx, topk_w=wts, logits=lg)
    assert g.layer.poll_error() == 0
    w64 = synth.weights_f64(w_cpu)
    gi = idx.cpu().numpy()
    ref, logits, oidx, owts, gap = _moe_reference(f64(r), w64, shape.as_dict(), gi)
    return f64(y.float()), ref, gi, wts.cpu().numpy(), lg.cpu().numpy(), logits, oidx, owts, gap


def _check_routing(gi, gw, glog, logits, oidx, owts, gap, norm=1):
    clear = gap > GAP
    assert clear.mean() > 0.8, "too few unambiguous tokens for a meaningful check"
    assert np.array_equal(gi[clear], oidx[clear]), (
        f"top-k mismatch on {np.sum(np.any(gi[clear] != oidx[clear], axis=1))} unambiguous tokens")
    assert np.allclose(gw[clear], owts[clear], atol=1e-5)
    # the selection claim needs logit errors well below the 1e-3 gap; the
    # router's FP32 accumulation over K = 2d grows with d (about 3e-5 at d=3584)
    assert np.abs(glog - logits).max() < 1e-4
    # every selection is a valid top-k: distinct experts, and its weights are
    # those of the oracle's logits at the selected experts
    assert all(len(set(row)) == len(row) for row in gi)
    assert np.allclose(gw, _gate_weights(logits, gi, norm), atol=1e-5)
    if norm:
        assert np.allclose(gw.sum(1), 1.0, atol=1e-5)
    else:  # probabilities of a softmax over all E: the k selected sum below 1
        assert np.all(gw.sum(1) < 1.0)


def test_moe_ffn_small_ragged():
    """E=16, k=4, T=300 (ragged tiles per expert), biased router."""
    y, ref, gi, gw, glog, logits, oidx, owts, gap = _run_moe_ffn(SMALL_MOE, "moe_s", 300)
    _check_routing(gi, gw, glog, logits, oidx, owts, gap)
    assert_parity(y, ref, what="MoE Y")


def test_moe_ffn_shared_expert_without_renormalisation():
    """Qwen2-MoE block: full-softmax gate weights and a sigmoid-gated shared
    expert (sf = 512), T=300 ragged over 16 experts."""
    shape = SMALL_QWEN2_MOE
    y, ref, gi, gw, glog, logits, oidx, owts, gap = _run_moe_ffn(shape, "q2moe", 300)
    _check_routing(gi, gw, glog, logits, oidx, owts, gap, norm=0)
    assert_parity(y, ref, what="Qwen2-MoE Y")
    # the shared expert is not lost in the tolerance: the oracle without it fails
    w64 = synth.weights_f64(synth.layer_weights(shape, "q2moe"))
    r = synth.activations([300, shape.d], "q2moe", "r")
    no_shared = oracle.moe_block(f64(r), w64, dict(shape.as_dict(), shared_ffn=0))[0]
    with pytest.raises(AssertionError):
        assert_parity(y, no_shared, what="Qwen2-MoE Y without the shared expert")


def test_moe_ffn_pair_tiles():
    """T=2000 over 16 experts (about 500 routed rows each): the grouped expert
    GEMMs take 256-row tiles on 2-CTA pairs, ragged at every group's end."""
    y, ref, gi, gw, glog, logits, oidx, owts, gap = _run_moe_ffn(SMALL_MOE, "moe_pair", 2000)
    _check_routing(gi, gw, glog, logits, oidx, owts, gap)
    assert_parity(y, ref, what="MoE Y (pair tiles)")


def test_moe_ffn_fp32_residual_input():
    y, ref, gi, gw, glog, logits, oidx, owts, gap = _run_moe_ffn(SMALL_MOE, "moe_s32", 77,
                                                                 fp32_input=True)
    _check_routing(gi, gw, glog, logits, oidx, owts, gap)
    assert_parity(y, ref, what="MoE Y (fp32 R)")


@pytest.fixture(scope="module")
def a3b_weights():
    return synth.layer_weights(synth.QWEN3_30B_A3B, "a3b")


def test_moe_ffn_qwen3_30b_a3b_full(a3b_weights):
    """Qwen3-30B-A3B-shaped MoE block at T=4096, E=128, k=8, mf=768."""
    shape = synth.QWEN3_30B_A3B
    T = 4096
    r = synth.activations([T, shape.d], "a3b", "r")
    g = GpuLayer(shape, a3b_weights, max_tokens=T, max_batch=1, max_seq=8, max_position=8)
    idx = torch.empty((T, 8), dtype=torch.int32, device="cuda")
    wts = torch.empty((T, 8), dtype=torch.float32, device="cuda")
    lg = torch.empty((T, 128), dtype=torch.float32, device="cuda")
    y = g.layer.moe_ffn(r.cuda(), topk_idx=idx, topk_w=wts, logits=lg)
    assert g.layer.poll_error() == 0
    gi = idx.cpu().numpy()
    w64 = synth.weights_f64(a3b_weights)
    ref, logits, oidx, owts, gap = _moe_reference(f64(r), w64, shape.as_dict(), gi)
    _check_routing(gi, wts.cpu().numpy(), lg.cpu().numpy(), logits, oidx, owts, gap)
    assert_parity(f64(y.float()), ref, what="MoE Y")
    # the router bias skews expert loads, as the workload intends
    loads = np.bincount(gi.reshape(-1), minlength=128)
    assert loads.max() > 2 * loads.mean()


class _PerExpertF64:
    """w[e] widened to float64 on demand (the full expert stack in FP64 would
    not fit the test's memory)."""

    def __init__(self, t):
        self.t = t

    def __getitem__(self, e):
        return synth.to_f64(self.t[e])


def test_moe_ffn_qwen2_57b_a14b_full():
    """Qwen2-57B-A14B-shaped MoE block at T=4096 (64 experts, top-8, mf=2560,
    shared expert sf=20480, no renormalisation): routing of every token, Y on
    sampled tokens."""
    shape = synth.QWEN2_57B_A14B
    T, E, k = 4096, shape.n_experts, shape.top_k
    w_cpu = synth.layer_weights(shape, "q2full")
    r = synth.activations([T, shape.d], "q2full", "r")
    g = GpuLayer(shape, w_cpu, max_tokens=T, max_batch=1, max_seq=8, max_position=8)
    idx = torch.empty((T, k), dtype=torch.int32, device="cuda")
    wts = torch.empty((T, k), dtype=torch.float32, device="cuda")
    lg = torch.empty((T, E), dtype=torch.float32, device="cuda")
    y = g.layer.moe_ffn(r.cuda(), topk_idx=idx, topk_w=wts, logits=lg)
    assert g.layer.poll_error() == 0
    del g
    gi, r64 = idx.cpu().numpy(), f64(r)
    w64 = {n: (_PerExpertF64(t) if n in ("w_gate", "w_up", "w_down") else synth.to_f64(t))
           for n, t in w_cpu.items()}
    cfg = shape.as_dict()
    z = oracle.rmsnorm(r64, w64["gamma_mlp"], cfg["rms_eps"])
    logits, oidx, owts, gap = oracle.router_topk(z, w64["w_router"], None, k, 0)
    _check_routing(gi, wts.cpu().numpy(), lg.cpu().numpy(), logits, oidx, owts, gap, norm=0)
    rows = np.unique(np.r_[0, 1, 127, 128, 2048, 4095,
                           np.random.default_rng(2).integers(0, T, 26)])
    ref = _moe_reference(r64[rows], w64, cfg, gi[rows])[0]
    assert_parity(f64(y.float())[rows], ref, what="Qwen2-57B-A14B MoE Y")


def _teacher_forced_check(shape, w64, r_gpu, gi, gw, y_gpu, what):
    """The MoE block checked on the GPU's own residual stream R (FP32).

    The oracle runs its own FP64 RMSNorm_2, router and experts on R as the GPU
    holds it, so the attention block's rounding does not move the routing.
    Every row is compared: the top-k bit-exact where the oracle's gap exceeds
    1e-3, any valid top-k elsewhere (the oracle is then evaluated under the
    GPU's selection with its own gate weights at those experts), and Y within
    the tolerance on every row."""
    cfg = shape.as_dict()
    ref, logits, oidx, owts, gap = _moe_reference(r_gpu, w64, cfg, gi)
    clear = gap > GAP
    assert np.array_equal(gi[clear], oidx[clear]), (
        f"{what}: top-k mismatch on {np.sum(np.any(gi[clear] != oidx[clear], axis=1))} "
        f"rows with gap > {GAP}")
    assert all(len(set(row)) == len(row) for row in gi)
    assert np.allclose(gw, _gate_weights(logits, gi, cfg.get("norm_topk_prob", 1)), atol=1e-5)
    assert_parity(y_gpu, ref, what=what)


def _layer_routing(g, ws, B, T, shape):
    """R (FP32), top-k indices and gate weights of the last layer call, read
    from the workspace regions the C ABI names."""
    M, k = B * T, shape.top_k
    r32 = workspace_region(g.cfg, ws, B, T, "r32", torch.float32, (M, shape.d))
    idx = workspace_region(g.cfg, ws, B, T, "topk_idx", torch.int32, (M, k))
    wts = workspace_region(g.cfg, ws, B, T, "topk_w", torch.float32, (M, k))
    return f64(r32), idx.cpu().numpy(), wts.cpu().numpy()


def _moe_layer_case(shape, w_cpu, tag, B, T, rows):
    """MoE layer prefill.  The attention block's output R is compared with the
    oracle's on every sampled row, and the MoE block teacher-forced on the
    GPU's R (every sampled row).  End to end, rows whose routing agrees with
    the plain oracle's are compared with its Y as well."""
    x = synth.activations([B, T, shape.d], tag)
    g = GpuLayer(shape, w_cpu, max_tokens=B * T, max_batch=B, max_seq=T, max_position=T)
    kc = torch.zeros((B, shape.n_kv_heads, T, shape.head_dim), dtype=torch.bfloat16, device="cuda")
    vc = torch.zeros_like(kc)
    ws = g.layer.workspace(B, T)
    pos = torch.arange(T, dtype=torch.int32, device="cuda").repeat(B)
    y = g.layer.prefill(x.cuda(), pos, torch.zeros(B, dtype=torch.int32, device="cuda"), kc, vc,
                        out=torch.empty((B, T, shape.d), dtype=torch.bfloat16, device="cuda"),
                        workspace=ws)
    assert g.layer.poll_error() == 0
    r_gpu, gi, gw = _layer_routing(g, ws, B, T, shape)
    w64 = synth.weights_f64(w_cpu)
    cfg = shape.as_dict()
    yg = f64(y.float())
    for b in range(B):
        kk = np.zeros((shape.n_kv_heads, T, shape.head_dim))
        vv = np.zeros_like(kk)
        yo, r, (logits, idx, wts, gap) = oracle.moe_layer_forward(
            f64(x)[b], w64, cfg, np.arange(T), kk, vv, np.arange(T), rows=rows)
        sel = b * T + rows
        assert_parity(r_gpu[sel], r, what=f"MoE layer R (b={b})")
        _teacher_forced_check(shape, w64, r_gpu[sel], gi[sel], gw[sel], yg[b, rows],
                              what=f"MoE layer Y on the GPU's R (b={b})")
        agree = np.all(gi[sel] == idx, axis=1)
        assert_parity(yg[b, rows][agree], yo[agree], what=f"MoE layer Y end to end (b={b})")


def test_moe_layer_prefill_small():
    shape = SMALL_MOE
    rows = np.array([0, 1, 63, 64, 65, 127, 128, 200, 255])
    _moe_layer_case(shape, synth.layer_weights(shape, "moel"), "moel", 2, 256, rows)


def test_moe_layer_prefill_qwen3_30b_a3b(a3b_weights):
    """Full Qwen3-30B-A3B-shaped MoE layer, T=4096, sampled rows."""
    T = 4096
    rows = np.unique(np.r_[0, 1, 127, 128, 2048, 4095,
                           np.random.default_rng(1).integers(0, T, 40)])
    _moe_layer_case(synth.QWEN3_30B_A3B, a3b_weights, "a3bl", 1, T, rows)


def test_moe_layer_prefill_shared_expert():
    shape = SMALL_QWEN2_MOE
    rows = np.array([0, 1, 63, 64, 65, 127, 128, 200, 255])
    _moe_layer_case(shape, synth.layer_weights(shape, "q2moel"), "q2moel", 2, 256, rows)


@pytest.mark.parametrize("shape,tag,B", [(SMALL_MOE, "moed", 8), (SMALL_QWEN2_MOE, "q2moed", 8),
                                         (SMALL_MOE, "moed1", 1), (SMALL_QWEN2_MOE, "q2moed2", 2),
                                         (SMALL_MOE, "moed64", 64),
                                         (SMALL_QWEN2_MOE, "q2moed65", 65)],
                         ids=["qwen3", "qwen2_shared", "qwen3_b1", "qwen2_b2", "qwen3_b64",
                              "qwen2_b65"])
def test_moe_layer_decode(shape, tag, B):
    """MoE layer decode against 100 cached slots.  Up to 64 tokens the experts
    run as the grouped swap-AB decode GEMM (B=64 is its largest padding); 65
    tokens take the 128-row grouped GEMM.  The Qwen2-MoE cases run the shared
    expert through the split-K GEMMs.  One or two tokens are routed by the
    CTA-wide expert ranks, more by the per-token warp top-k."""
    L = 100
    w_cpu = synth.layer_weights(shape, tag)
    x = synth.activations([B, shape.d], tag)
    kc, vc = synth.kv_cache(B, shape.n_kv_heads, L + 1, shape.head_dim, L, tag)
    g = GpuLayer(shape, w_cpu, max_tokens=B, max_batch=B, max_seq=L + 1, max_position=L + 1)
    kd, vd = kc.cuda(), vc.cuda()
    ws = g.layer.workspace(B, 1)
    lens = torch.full((B,), L, dtype=torch.int32, device="cuda")
    y = g.layer.decode(x.cuda(), lens, lens.clone(), kd, vd,
                       out=torch.empty((B, shape.d), dtype=torch.bfloat16, device="cuda"),
                       workspace=ws)
    assert g.layer.poll_error() == 0
    r_gpu, gi, gw = _layer_routing(g, ws, B, 1, shape)
    w64 = synth.weights_f64(w_cpu)
    cfg = shape.as_dict()
    yg = f64(y.float())
    r_ref = np.empty_like(r_gpu)
    for b in range(B):
        kk, vv = f64(kc)[b].copy(), f64(vc)[b].copy()
        r_ref[b] = oracle.attention_block(f64(x)[b][None], w64, cfg, np.array([L]), kk, vv,
                                          np.array([L]))[0]
    assert_parity(r_gpu, r_ref, what="decode R")
    _teacher_forced_check(shape, w64, r_gpu, gi, gw, yg, what="decode Y on the GPU's R")


@pytest.mark.parametrize("B", [1, 8])
def test_moe_layer_decode_qwen3_30b_a3b(a3b_weights, B):
    """Full Qwen3-30B-A3B-shaped MoE layer decode against 4096 cached slots
    (the bench's MoE decode workload): R of every sequence against the oracle,
    then the MoE block teacher-forced on the GPU's R (top-k bit-exact where the
    oracle's gap exceeds 1e-3, Y on every sequence), and the appended K/V rows."""
    shape = synth.QWEN3_30B_A3B
    L = 4096
    x = synth.activations([B, shape.d], f"a3bd{B}")
    kc, vc = synth.kv_cache(B, shape.n_kv_heads, L + 1, shape.head_dim, L, f"a3bd{B}")
    g = GpuLayer(shape, a3b_weights, max_tokens=B, max_batch=B, max_seq=L + 1,
                 max_position=L + 1)
    kd, vd = kc.cuda(), vc.cuda()
    ws = g.layer.workspace(B, 1)
    lens = torch.full((B,), L, dtype=torch.int32, device="cuda")
    y = g.layer.decode(x.cuda(), lens, lens.clone(), kd, vd,
                       out=torch.empty((B, shape.d), dtype=torch.bfloat16, device="cuda"),
                       workspace=ws)
    assert g.layer.poll_error() == 0
    r_gpu, gi, gw = _layer_routing(g, ws, B, 1, shape)
    w64 = {n: (_PerExpertF64(t) if n in ("w_gate", "w_up", "w_down") else synth.to_f64(t))
           for n, t in a3b_weights.items()}
    cfg = shape.as_dict()
    r_ref = np.empty_like(r_gpu)
    k_ref = np.empty((B, shape.n_kv_heads, shape.head_dim))
    v_ref = np.empty_like(k_ref)
    for b in range(B):
        kk, vv = f64(kc)[b].copy(), f64(vc)[b].copy()
        r_ref[b] = oracle.attention_block(f64(x)[b][None], w64, cfg, np.array([L]), kk, vv,
                                          np.array([L]))[0]
        k_ref[b], v_ref[b] = kk[:, L], vv[:, L]
    assert_parity(r_gpu, r_ref, what="decode R")
    assert_parity(f64(kd.float())[:, :, L], k_ref, what="appended K")
    assert_parity(f64(vd.float())[:, :, L], v_ref, what="appended V")
    _teacher_forced_check(shape, w64, r_gpu, gi, gw, f64(y.float()),
                          what="decode Y on the GPU's R")
