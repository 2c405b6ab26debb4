"""The workspace-free last-token head on the GPU, against the workspace one
and against the FP64 oracle.

qwen_head_last_token_noalloc serves callers that cannot allocate device memory
when they call the head (for example a server whose HBM is already committed
to a fixed arena); it keeps its normalised rows in a fixed array inside the
library.  Two calls in a row, with different inputs, must each match
qwen_head_last_token on the same inputs within the parity tolerance, and both
must match the oracle's final RMSNorm + lm_head.  A call that fills the array
exactly (B * d * 2 = 2 MiB) is accepted and correct; sizes beyond it are
refused.  This file is collected last on purpose.
"""

import ctypes

import numpy as np
import pytest

import oracle
import synth
from parity import assert_parity

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


def _inputs(tag, B, T, d, V):
    y = synth.activations([B, T, d], tag, "y")
    g = synth.normal_bf16([d], synth.seed_for(tag, "g"), 0.1, 1.0)
    w = synth.normal_bf16([V, d], synth.seed_for(tag, "w"), 0.02)
    return y, g, w


def _oracle_logits(y, g, w):
    """Qwen2.5-7B 结构拆解 §03.8: logits = RMSNorm_final(y[:, T-1]) W_lm^T."""
    return oracle.head_last_token(synth.to_f64(y[:, -1]), synth.to_f64(g), synth.to_f64(w), 1e-6)


def test_noalloc_head_matches_workspace_head_twice():
    import transformer_decoder_layer_gb300 as q
    first = _inputs("noalloc1", 4, 3, 3584, 32000)
    second = _inputs("noalloc2", 32, 2, 3584, 20000)
    for y, g, w in (first, second):
        yd, gd, wd = y.cuda(), g.cuda(), w.cuda()
        ref = q.head_last_token(yd, gd, wd, 1e-6)
        got = q.head_last_token_noalloc(yd, gd, wd, 1e-6)
        assert q.poll_error() == 0
        got = got.cpu().numpy()
        assert_parity(got, ref.cpu().numpy(), what="no-alloc head vs workspace head")
        assert_parity(got, _oracle_logits(y, g, w), what="no-alloc head vs oracle")


def test_noalloc_head_at_the_array_limit():
    """B = 256 rows of d = 4096: the normalised rows fill the 2 MiB array to
    its last byte, and the decode GEMM runs its widest (256-token) tile."""
    import transformer_decoder_layer_gb300 as q
    y, g, w = _inputs("noalloc_limit", 256, 1, 4096, 512)
    assert 256 * 4096 * 2 == 2 << 20
    got = q.head_last_token_noalloc(y.cuda(), g.cuda(), w.cuda(), 1e-6)
    assert q.poll_error() == 0
    ref = _oracle_logits(y, g, w)
    assert ref.shape == (256, 512)
    assert_parity(got.cpu().numpy(), ref, what="no-alloc head at the array limit")
    assert np.isfinite(got.cpu().numpy()).all()


def test_noalloc_head_rejects_sizes_beyond_its_array():
    import transformer_decoder_layer_gb300 as q
    L = q.lib()
    # B * d * 2 = 128 * 8192 * 2 = 2 MiB fits; one more row does not
    rc = L.qwen_head_last_token_noalloc(ctypes.c_void_p(16), 129, 1, 8192, ctypes.c_void_p(16),
                                        ctypes.c_void_p(16), 1024, ctypes.c_float(1e-6),
                                        ctypes.c_void_p(16), None)
    assert rc == 3  # QWEN_ERR_CAPACITY, refused before any launch
