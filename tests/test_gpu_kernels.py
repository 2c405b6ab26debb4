"""GPU parity of the single-step entry points (RMSNorm, tensor-core projection)
against the FP64 oracle, through the C ABI."""

import numpy as np
import pytest

import oracle
import synth
from parity import assert_parity

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def q():
    import transformer_decoder_layer_gb300 as q
    q.lib()
    return q


@pytest.mark.parametrize("rows,d", [(1, 512), (7, 3584), (300, 4096), (33, 8192), (64, 2048),
                                    (1024, 4096), (3000, 3584), (2500, 2048), (4096, 4096),
                                    (1500, 5120)])
def test_rmsnorm_matches_oracle(q, rows, d):
    """Up to 8 rows per SM one CTA per row (1024 rows included); above that a
    warp per row (3000, 2500, 4096 and 1500 rows; d = 3584 and 5120 leave
    lanes with fewer chunks than others)."""
    x = synth.activations([rows, d], "rms", f"x{rows}_{d}")
    g = synth.normal_bf16([d], synth.seed_for("rms", f"g{d}"), 0.1, 1.0)
    y32 = torch.empty((rows, d), dtype=torch.float32, device="cuda")
    y = q.rmsnorm(x.cuda(), g.cuda(), 1e-6, out_fp32=y32)
    assert q.poll_error() == 0
    ref = oracle.rmsnorm(synth.to_f64(x), synth.to_f64(g), 1e-6)
    assert_parity(y.float().cpu().numpy(), ref, what="rmsnorm bf16")
    # the FP32 copy is the same value before rounding: much tighter
    assert_parity(y32.cpu().numpy(), ref, atol=1e-5, rtol=1e-5, frob=1e-6, what="rmsnorm fp32")


@pytest.mark.parametrize("M,N,K", [
    (128, 256, 64),       # one tile, one k-block
    (1, 256, 512),        # single token row
    (300, 520, 1000),     # ragged M, N and K tails
    (1024, 6144, 4096),   # many tiles, grouped raster
    (257, 768, 512),      # tiny-layer QKV width
    (2000, 1800, 1000),   # 2-CTA pair tiles: ragged M, N and K; the last B half lies past N
])
def test_linear_matches_oracle(q, M, N, K):
    x = synth.activations([M, K], "lin", f"x{M}_{K}")
    w = synth.normal_bf16([N, K], synth.seed_for("lin", f"w{N}_{K}"), 0.02)
    y = q.linear(x.cuda(), w.cuda())
    assert q.poll_error() == 0
    ref = oracle.linear(synth.to_f64(x), synth.to_f64(w))
    assert_parity(y.float().cpu().numpy(), ref, what=f"linear {M}x{N}x{K}")


def test_linear_large_sampled_rows(q):
    """A full-size projection (C3 QKV: 16384 x 6144 x 4096) on sampled rows."""
    M, N, K = 16384, 6144, 4096
    x = synth.activations([M, K], "linbig")
    w = synth.normal_bf16([N, K], synth.seed_for("linbig", "w"), 0.02)
    y = q.linear(x.cuda(), w.cuda())
    assert q.poll_error() == 0
    rows = np.unique(np.r_[0, 1, 127, 128, 129, M - 129, M - 1,
                           np.random.default_rng(0).integers(0, M, 64)])
    ref = oracle.linear(synth.to_f64(x[rows]), synth.to_f64(w))
    assert_parity(y[rows].float().cpu().numpy(), ref, what="linear large")


def test_linear_pair_split_tail_sampled_rows(q):
    """4096 x 4096 x 1024: 256 pair tiles on the co-resident clusters leave a
    partial last wave, which runs as 256 x 128 half tiles (each CTA of a pair
    holding 64 rows of W).  Whole rows sampled across every m-block."""
    M, N, K = 4096, 4096, 1024
    x = synth.activations([M, K], "linsplit")
    w = synth.normal_bf16([N, K], synth.seed_for("linsplit", "w"), 0.02)
    y = q.linear(x.cuda(), w.cuda())
    assert q.poll_error() == 0
    rng = np.random.default_rng(1)
    rows = np.unique(np.r_[0, 255, 256, 1023, 1024, 3839, 3840, M - 1,
                           [256 * m + rng.integers(0, 256) for m in range(M // 256)]])
    ref = oracle.linear(synth.to_f64(x[rows]), synth.to_f64(w))
    assert_parity(y[rows].float().cpu().numpy(), ref, what="linear pair split tail")


def test_linear_is_deterministic(q):
    x = synth.activations([512, 1024], "det").cuda()
    w = synth.normal_bf16([768, 1024], 5, 0.02).cuda()
    a = q.linear(x, w)
    b = q.linear(x, w)
    assert torch.equal(a, b)
