"""The largest sizes of the workloads against the FP64 oracle, kept in their own
file and collected after the other layer tests (their oracles are the slowest).

* Qwen3-8B-shaped prefill at B=1 x T=16384 on sampled output rows (every K/V
  row is still projected by the oracle, since later rows read it), with the
  whole K/V cache compared;
* Qwen2.5-7B-shaped decode at B=32 and B=64 against 4096 filled cache slots,
  in the layer configuration the benchmark uses (capacity 64 sequences),
  the oracle run on sampled sequences including the first and the last; at
  B=32 the same step replayed from a CUDA graph, as the benchmark times it,
  gives the same bits as the eager call;
* long-context decode: B=8 against 32768 filled slots ("Qwen2.5-7B 结构拆解"
  §09.1: at 32k the KV read is about 13 % of the weight bytes), sampled
  sequences and every appended K/V row.
"""

import numpy as np
import pytest

import oracle
import synth
from layer_harness import GpuLayer, f64
from parity import assert_parity
from test_gpu_layer import _prefill_case

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


def test_qwen3_8b_layer_prefill_t16384_sampled_rows():
    T = 16384
    rng = np.random.default_rng(T)
    rows = np.unique(np.r_[0, 1, 127, 128, T // 2, T - 129, T - 1, rng.integers(0, T, 24)])
    y, ref, k, kr, v, vr = _prefill_case(synth.QWEN3_8B, f"q3_8b_{T}", 1, T, rows=rows)
    assert_parity(y, ref, what="Y")
    assert_parity(k, kr, what="K cache")
    assert_parity(v, vr, what="V cache")


def _decode_sampled(shape, tag, B, filled, sample, capacity, graph_check=False):
    """One decode step of B sequences against `filled` cached slots each (the
    new token at position and slot `filled`); the oracle recomputes the
    sequences in `sample`.  Returns nothing; asserts parity of Y and of the
    appended K/V rows."""
    w_cpu = synth.layer_weights(shape, tag)
    x = synth.activations([B, shape.d], tag)
    max_seq = filled + 1
    kc, vc = synth.kv_cache(B, shape.n_kv_heads, max_seq, shape.head_dim, filled, tag)
    g = GpuLayer(shape, w_cpu, max_tokens=capacity, max_batch=capacity, max_seq=max_seq,
                 max_position=max_seq)
    kd, vd = kc.cuda(), vc.cuda()
    pos = np.full(B, filled)
    y = g.decode(x, pos, pos, kd, vd)
    got = f64(y.float())
    if graph_check:
        xd = x.cuda()
        pd = torch.full((B,), filled, dtype=torch.int32, device="cuda")
        cd = pd.clone()
        yg = torch.empty_like(xd)
        ws = g.layer.workspace(B, 1)
        g.layer.decode(xd, pd, cd, kd, vd, out=yg, workspace=ws)  # warm-up outside capture
        torch.cuda.synchronize()
        cap = torch.cuda.Stream()
        cap.wait_stream(torch.cuda.current_stream())
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=cap):
            g.layer.decode(xd, pd, cd, kd, vd, out=yg, workspace=ws)
        yg.zero_()
        graph.replay()
        torch.cuda.synchronize()
        assert g.layer.poll_error() == 0
        assert torch.equal(yg, y), "graph replay differs from the eager decode step"
        del graph
    kg, vg = f64(kd[:, :, filled].float()), f64(vd[:, :, filled].float())
    cfg = shape.as_dict()
    w64 = synth.weights_f64(w_cpu)
    x64 = f64(x)
    for b in sample:
        kk, vv = f64(kc[b]), f64(vc[b])
        ref = oracle.layer_forward(x64[b][None], w64, cfg, np.array([filled]), kk, vv,
                                   np.array([filled]))[0]
        assert_parity(got[b], ref, what=f"Y b={b}")
        assert_parity(kg[b], kk[:, filled], what=f"appended K b={b}")
        assert_parity(vg[b], vv[:, filled], what=f"appended V b={b}")


@pytest.mark.parametrize("B", [32, 64])
def test_qwen25_7b_decode_full_size(B):
    """Qwen2.5-7B-shaped decode, B sequences against 4096 filled slots."""
    rng = np.random.default_rng(B)
    sample = sorted(set([0, B - 1]) | set(rng.choice(np.arange(1, B - 1), 6, replace=False)))
    _decode_sampled(synth.QWEN25_7B, f"q25_full{B}", B, 4096, sample, capacity=64,
                    graph_check=(B == 32))


def test_qwen25_7b_long_context_decode_32768():
    """B=8 against 32768 filled slots: 513 key blocks of 64 per (sequence,
    KV head) pair for the stream-K split of the decode attention."""
    _decode_sampled(synth.QWEN25_7B, "q25_long", 8, 32768, [0, 2, 5, 7], capacity=8)
