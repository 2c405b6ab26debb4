"""The largest prefill size of the Qwen3-8B-shaped workload, B=1 x T=16384,
against the FP64 oracle on sampled output rows (every K/V row is still
projected by the oracle, since later rows read it), with the whole K/V cache
compared.  Kept in its own file, collected after the other layer tests: its
oracle projects 16384 rows in FP64."""

import numpy as np
import pytest

import synth
from parity import assert_parity
from test_gpu_layer import _prefill_case

pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


def test_qwen3_8b_layer_prefill_t16384_sampled_rows():
    T = 16384
    rng = np.random.default_rng(T)
    rows = np.unique(np.r_[0, 1, 127, 128, T // 2, T - 129, T - 1, rng.integers(0, T, 24)])
    y, ref, k, kr, v, vr = _prefill_case(synth.QWEN3_8B, f"q3_8b_{T}", 1, T, rows=rows)
    assert_parity(y, ref, what="Y")
    assert_parity(k, kr, what="K cache")
    assert_parity(v, vr, what="V cache")
