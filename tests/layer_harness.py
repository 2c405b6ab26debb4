"""Shared set-up for the layer parity tests: seeded inputs on both sides, the
oracle run per sequence, and the CUDA path through the C ABI."""

from __future__ import annotations

import numpy as np

import oracle
import synth


def oracle_prefill(shape, w64, x, positions, cache_start, k0, v0, rows=None):
    """Run the FP64 oracle per sequence.  x [B,T,d] float64; caches [B,Hkv,S,dh]
    (copied).  Returns (y [B,len(rows),d], k, v)."""
    B, T, _ = x.shape
    cfg = shape.as_dict()
    k = k0.copy()
    v = v0.copy()
    ys = []
    for b in range(B):
        slots = cache_start[b] + np.arange(T)
        pos = positions[b]
        ys.append(oracle.layer_forward(x[b], w64, cfg, pos, k[b], v[b], slots, rows=rows))
    return np.stack(ys), k, v


class GpuLayer:
    """A layer handle plus device copies of its weights."""

    def __init__(self, shape, w_cpu, max_tokens, max_batch, max_seq, max_position):
        import torch
        import transformer_decoder_layer_gb300 as q
        self.q = q
        self.shape = shape
        self.w = {k: t.cuda() for k, t in w_cpu.items()}
        self.cfg = q.LayerConfig(shape, max_tokens=max_tokens, max_batch=max_batch,
                                 max_seq=max_seq, max_position=max_position)
        self.layer = q.Layer(self.cfg, self.w)
        self.torch = torch

    def prefill(self, x, positions, cache_start, kc, vc):
        t = self.torch
        y = self.layer.prefill(x.cuda(), t.as_tensor(positions, dtype=t.int32).cuda().reshape(-1),
                               t.as_tensor(cache_start, dtype=t.int32).cuda(), kc, vc)
        rc = self.layer.poll_error()
        assert rc == 0, f"device status {rc}"
        return y

    def decode(self, x, positions, cache_len, kc, vc):
        t = self.torch
        y = self.layer.decode(x.cuda(), t.as_tensor(positions, dtype=t.int32).cuda(),
                              t.as_tensor(cache_len, dtype=t.int32).cuda(), kc, vc)
        rc = self.layer.poll_error()
        assert rc == 0, f"device status {rc}"
        return y


def f64(t):
    return synth.to_f64(t.cpu() if hasattr(t, "cpu") else t)


def workspace_region(layer_cfg, ws, B, T, name, dtype, shape):
    """View of one named region of a layer workspace (the layout the C ABI
    reports through qwen_layer_workspace_regions) as a tensor."""
    import transformer_decoder_layer_gb300 as q
    for n, off, nbytes in q.workspace_regions(layer_cfg, B, T):
        if n == name:
            view = ws[off:off + nbytes].view(dtype)
            count = 1
            for s in shape:
                count *= s
            return view[:count].reshape(shape)
    raise KeyError(name)
