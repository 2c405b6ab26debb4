"""The workspace-free last-token head against the workspace one, on the GPU.

qwen_head_last_token_noalloc serves callers that cannot allocate device memory
when they call the head (for example a server whose HBM is already committed
to a fixed arena); it keeps its normalised rows in a fixed array inside the
library.  Two calls in a row, with different inputs, must each match
qwen_head_last_token on the same inputs within the parity tolerance, and sizes
beyond the array are refused.  This file is collected last on purpose.
"""

import ctypes

import pytest

import synth
from parity import assert_parity

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


def _inputs(tag, B, T, d, V):
    y = synth.activations([B, T, d], tag, "y").cuda()
    g = synth.normal_bf16([d], synth.seed_for(tag, "g"), 0.1, 1.0).cuda()
    w = synth.normal_bf16([V, d], synth.seed_for(tag, "w"), 0.02).cuda()
    return y, g, w


def test_noalloc_head_matches_workspace_head_twice():
    import transformer_decoder_layer_gb300 as q
    first = _inputs("noalloc1", 4, 3, 3584, 32000)
    second = _inputs("noalloc2", 32, 2, 3584, 20000)
    for y, g, w in (first, second):
        ref = q.head_last_token(y, g, w, 1e-6)
        got = q.head_last_token_noalloc(y, g, w, 1e-6)
        assert q.poll_error() == 0
        assert_parity(got.cpu().numpy(), ref.cpu().numpy(), what="no-alloc head logits")


def test_noalloc_head_rejects_sizes_beyond_its_array():
    import transformer_decoder_layer_gb300 as q
    L = q.lib()
    # B * d * 2 = 128 * 8192 * 2 = 2 MiB fits; one more row does not
    rc = L.qwen_head_last_token_noalloc(ctypes.c_void_p(16), 129, 1, 8192, ctypes.c_void_p(16),
                                        ctypes.c_void_p(16), 1024, ctypes.c_float(1e-6),
                                        ctypes.c_void_p(16), None)
    assert rc == 3  # QWEN_ERR_CAPACITY, refused before any launch
