"""Python binding of libqwenlayer.so: a GB300 (sm_103a) Qwen-style decoder layer.

This module only marshals arguments (torch tensors -> device pointers, the
current CUDA stream) into the C ABI declared in ``include/qwen_layer.h``.
Every step of the layer runs in the library's CUDA kernels; there is no CPU
fallback, and every call raises if the shared library is not built or a call
returns an error.
"""

from __future__ import annotations

import ctypes
import os

from ._build import LIB as _LIB_PATH

__all__ = [
    "QwenError", "lib", "LayerConfig", "Layer", "Stack", "rmsnorm", "linear", "head_last_token",
    "head_last_token_noalloc", "poll_error", "launch_count", "STATUS",
]

STATUS = {
    0: "QWEN_OK", 1: "QWEN_ERR_INVALID_ARG", 2: "QWEN_ERR_UNSUPPORTED",
    3: "QWEN_ERR_CAPACITY", 4: "QWEN_ERR_CUDA", 5: "QWEN_ERR_TIMEOUT", 6: "QWEN_ERR_RANGE",
    7: "QWEN_ERR_OVERFLOW",
}


class QwenError(RuntimeError):
    def __init__(self, code, where=""):
        self.code = int(code)
        super().__init__(f"{where}: {STATUS.get(self.code, self.code)}")


class _Config(ctypes.Structure):
    _fields_ = [
        ("d", ctypes.c_int32), ("n_q_heads", ctypes.c_int32), ("n_kv_heads", ctypes.c_int32),
        ("head_dim", ctypes.c_int32), ("ffn", ctypes.c_int32), ("qkv_bias", ctypes.c_int32),
        ("qk_norm", ctypes.c_int32), ("rope_theta", ctypes.c_double),
        ("rms_eps", ctypes.c_float), ("n_experts", ctypes.c_int32), ("top_k", ctypes.c_int32),
        ("norm_topk_prob", ctypes.c_int32), ("router_bias", ctypes.c_int32),
        ("max_tokens", ctypes.c_int32), ("max_batch", ctypes.c_int32),
        ("max_seq", ctypes.c_int32), ("max_position", ctypes.c_int32),
        ("shared_ffn", ctypes.c_int32),
    ]


_WEIGHT_FIELDS = ["gamma_attn", "gamma_mlp", "gamma_q", "gamma_k", "w_q", "w_k", "w_v", "b_q",
                  "b_k", "b_v", "w_o", "w_gate", "w_up", "w_down", "w_router", "b_router",
                  "w_shared_gate", "w_shared_up", "w_shared_down", "w_shared_expert_gate"]


class _Weights(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in _WEIGHT_FIELDS]


class _Region(ctypes.Structure):
    _fields_ = [("name", ctypes.c_char_p), ("offset", ctypes.c_size_t),
                ("bytes", ctypes.c_size_t)]


_VP, _I32, _SZ, _F32 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_size_t, ctypes.c_float
_SIGS = {
    "qwen_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "qwen_layer_packed_bytes": (_SZ, [ctypes.POINTER(_Config)]),
    "qwen_layer_workspace_bytes": (_SZ, [ctypes.POINTER(_Config), _I32, _I32]),
    "qwen_layer_workspace_regions": (_I32, [ctypes.POINTER(_Config), _I32, _I32,
                                            ctypes.POINTER(_Region), _I32]),
    "qwen_layer_create": (ctypes.c_int, [ctypes.POINTER(_Config), ctypes.POINTER(_Weights), _VP,
                                         _SZ, _VP, ctypes.POINTER(_VP)]),
    "qwen_layer_destroy": (None, [_VP]),
    "qwen_layer_prefill": (ctypes.c_int, [_VP, _VP, _VP, _I32, _I32, _VP, _VP, _VP, _VP, _VP,
                                          _SZ, _VP]),
    "qwen_layer_decode": (ctypes.c_int, [_VP, _VP, _VP, _I32, _VP, _VP, _VP, _VP, _VP, _SZ,
                                         _VP]),
    "qwen_layer_prefill_ex": (ctypes.c_int, [_VP, _VP, _VP, _VP, _VP, _I32, _I32, _VP, _VP, _VP,
                                             _VP, _VP, _SZ, _VP]),
    "qwen_layer_decode_ex": (ctypes.c_int, [_VP, _VP, _VP, _VP, _VP, _I32, _VP, _VP, _VP, _VP,
                                            _VP, _SZ, _VP]),
    "qwen_layer_host_workspace_bytes": (_SZ, [ctypes.POINTER(_Config), _I32]),
    "qwen_layer_decode_host": (ctypes.c_int, [_VP, _VP, _VP, _I32, _VP, _VP, _VP, _VP, _VP,
                                              _SZ, _VP]),
    "qwen_moe_ffn": (ctypes.c_int, [_VP, _VP, _VP, _VP, _I32, _VP, _VP, _VP, _VP, _SZ, _VP]),
    "qwen_head_workspace_bytes": (_SZ, [_I32, _I32, _I32]),
    "qwen_head_last_token": (ctypes.c_int, [_VP, _I32, _I32, _I32, _VP, _VP, _I32, _F32, _VP,
                                            _VP, _SZ, _VP]),
    "qwen_head_last_token_noalloc": (ctypes.c_int, [_VP, _I32, _I32, _I32, _VP, _VP, _I32, _F32,
                                                    _VP, _VP]),
    "qwen_rmsnorm": (ctypes.c_int, [_VP, _VP, _VP, _VP, _I32, _I32, _F32, _VP]),
    "qwen_linear": (ctypes.c_int, [_VP, _VP, _VP, _I32, _I32, _I32, _VP]),
    "qwen_layer_poll_error": (ctypes.c_int, [_VP, _VP]),
    "qwen_poll_error": (ctypes.c_int, [_VP]),
    "qwen_device_sm_count": (_I32, []),
    "qwen_layer_set_trace": (ctypes.c_int, [_VP, _VP]),
    "qwen_launch_count": (ctypes.c_uint64, []),
}

STAGES = ["norm1", "qkv", "qkv_finish", "attn", "attn_merge", "o", "o_finish", "norm2",
          "gate_up", "gate_up_finish", "down", "down_finish", "moe"]

_lib = None


def lib_path() -> str:
    return _LIB_PATH


def lib():
    """Load libqwenlayer.so (built in-tree by ``__graft_entry__.build()``)."""
    global _lib
    if _lib is None:
        if not os.path.exists(_LIB_PATH):
            raise RuntimeError(
                f"{_LIB_PATH} is not built; run `python -c 'import __graft_entry__ as g; g.build()'`")
        L = ctypes.CDLL(_LIB_PATH)
        for name, (res, args) in _SIGS.items():
            if not hasattr(L, name):
                continue  # the ABI test insists every declared symbol exists
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
    return _lib


def _check(rc, where):
    if rc != 0:
        raise QwenError(rc, where)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    import torch
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _need(t, dtype, name):
    import torch
    if t is None:
        raise ValueError(f"{name} is required")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor (there is no CPU path)")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t


# ---------------------------------------------------------------- handle-less calls

def rmsnorm(x, gamma, eps, out=None, out_fp32=None, stream=None):
    """y = gamma * x / sqrt(mean(x^2) + eps) row-wise (BF16 in/out)."""
    import torch
    _need(x, torch.bfloat16, "x")
    _need(gamma, torch.bfloat16, "gamma")
    d = x.shape[-1]
    rows = x.numel() // d
    out = torch.empty_like(x) if out is None else out
    _check(lib().qwen_rmsnorm(_ptr(x), _ptr(gamma), _ptr(out), _ptr(out_fp32), rows, d,
                              float(eps), _stream(stream)), "qwen_rmsnorm")
    return out


def linear(x, w, out=None, stream=None):
    """y = x W^T on the tensor cores: x [M,K], w [N,K] BF16 -> y [M,N] BF16."""
    import torch
    _need(x, torch.bfloat16, "x")
    _need(w, torch.bfloat16, "w")
    K = x.shape[-1]
    M = x.numel() // K
    N = w.shape[0]
    out = torch.empty((*x.shape[:-1], N), dtype=torch.bfloat16, device=x.device) if out is None else out
    _check(lib().qwen_linear(_ptr(x), _ptr(w), _ptr(out), M, N, K, _stream(stream)), "qwen_linear")
    return out


def poll_error(stream=None):
    """Synchronise and return (then clear) the library-wide device status."""
    return lib().qwen_poll_error(_stream(stream))


def head_workspace_bytes(B, d, V):
    return lib().qwen_head_workspace_bytes(B, d, V)


def workspace_regions(cfg, B, T):
    """[(name, offset, bytes)] of the layer workspace for (B, T) under a
    LayerConfig, in layout order (host only)."""
    n = lib().qwen_layer_workspace_regions(ctypes.byref(cfg.c), B, T, None, 0)
    if n < 0:
        raise ValueError(f"invalid config or sizes (B={B}, T={T})")
    arr = (_Region * max(n, 1))()
    lib().qwen_layer_workspace_regions(ctypes.byref(cfg.c), B, T, arr, n)
    return [(r.name.decode(), int(r.offset), int(r.bytes)) for r in arr[:n]]


def head_last_token(y, gamma_final, w_lm, eps, logits=None, workspace=None, stream=None):
    """logits[b] = RMSNorm(y[b, -1]) W_lm^T (FP32 logits)."""
    import torch
    _need(y, torch.bfloat16, "y")
    B, T, d = y.shape
    V = w_lm.shape[0]
    logits = torch.empty((B, V), dtype=torch.float32, device=y.device) if logits is None else logits
    nbytes = head_workspace_bytes(B, d, V)
    if workspace is None:
        workspace = torch.empty(max(nbytes, 256), dtype=torch.uint8, device=y.device)
    _check(lib().qwen_head_last_token(_ptr(y), B, T, d, _ptr(gamma_final), _ptr(w_lm), V,
                                      float(eps), _ptr(logits), _ptr(workspace),
                                      workspace.numel(), _stream(stream)),
           "qwen_head_last_token")
    return logits


def head_last_token_noalloc(y, gamma_final, w_lm, eps, logits=None, stream=None):
    """Same result as head_last_token, with no workspace: for callers that
    cannot allocate device memory at call time (the library keeps the
    normalised rows in its own fixed device array; B * d * 2 <= 2 MiB).
    Calls that overlap on the GPU race on that array."""
    import torch
    _need(y, torch.bfloat16, "y")
    B, T, d = y.shape
    V = w_lm.shape[0]
    logits = torch.empty((B, V), dtype=torch.float32, device=y.device) if logits is None else logits
    _check(lib().qwen_head_last_token_noalloc(_ptr(y), B, T, d, _ptr(gamma_final), _ptr(w_lm), V,
                                              float(eps), _ptr(logits), _stream(stream)),
           "qwen_head_last_token_noalloc")
    return logits


# ---------------------------------------------------------------- layer handle

class LayerConfig:
    """Build the C ``qwen_layer_config`` from a shape object (any object or dict
    with the shape fields) plus capacities."""

    def __init__(self, shape, max_tokens, max_batch, max_seq, max_position):
        get = (lambda k, dflt=0: shape.get(k, dflt)) if isinstance(shape, dict) else \
            (lambda k, dflt=0: getattr(shape, k, dflt))
        self.c = _Config(
            d=get("d"), n_q_heads=get("n_q_heads"), n_kv_heads=get("n_kv_heads"),
            head_dim=get("head_dim"), ffn=get("ffn"), qkv_bias=get("qkv_bias"),
            qk_norm=get("qk_norm"), rope_theta=float(get("rope_theta", 1.0e6)),
            rms_eps=float(get("rms_eps", 1.0e-6)), n_experts=get("n_experts"),
            top_k=get("top_k"), norm_topk_prob=get("norm_topk_prob", 1),
            router_bias=get("router_bias"), max_tokens=int(max_tokens),
            max_batch=int(max_batch), max_seq=int(max_seq), max_position=int(max_position),
            shared_ffn=get("shared_ffn"))

    def __getattr__(self, k):
        return getattr(self.__dict__["c"], k)


class Layer:
    """One decoder layer: packed weights (device) + a library handle."""

    def __init__(self, cfg: LayerConfig, weights: dict, device="cuda", stream=None):
        import torch
        self.cfg = cfg
        L = lib()
        nbytes = L.qwen_layer_packed_bytes(ctypes.byref(cfg.c))
        if nbytes == 0:
            raise QwenError(1, "qwen_layer_packed_bytes (invalid config)")
        self.packed = torch.empty(nbytes, dtype=torch.uint8, device=device)
        w = _Weights()
        for n in _WEIGHT_FIELDS:
            t = weights.get(n)
            if t is not None:
                if not t.is_cuda or not t.is_contiguous():
                    raise ValueError(f"weight {n} must be a contiguous CUDA tensor")
                setattr(w, n, t.data_ptr())
        h = ctypes.c_void_p()
        _check(L.qwen_layer_create(ctypes.byref(cfg.c), ctypes.byref(w), _ptr(self.packed),
                                   nbytes, _stream(stream), ctypes.byref(h)), "qwen_layer_create")
        self.handle = h

    def close(self):
        if getattr(self, "handle", None) is not None and self.handle.value:
            lib().qwen_layer_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def workspace_bytes(self, B, T):
        return lib().qwen_layer_workspace_bytes(ctypes.byref(self.cfg.c), B, T)

    def workspace(self, B, T, device="cuda"):
        import torch
        return torch.empty(max(self.workspace_bytes(B, T), 256), dtype=torch.uint8, device=device)

    @staticmethod
    def _io(x, out, out32):
        """Split x into (bf16, fp32) inputs and default the output: BF16 in ->
        BF16 out; FP32 in -> FP32 out (the residual interface across layers)."""
        import torch
        if not x.is_cuda or not x.is_contiguous():
            raise ValueError("x must be a contiguous CUDA tensor")
        if x.dtype == torch.bfloat16:
            xb, x32 = x, None
        elif x.dtype == torch.float32:
            xb, x32 = None, x
        else:
            raise ValueError(f"x must be bfloat16 or float32, got {x.dtype}")
        if out is None and out32 is None:
            if x32 is None:
                out = torch.empty_like(x)
            else:
                out32 = torch.empty_like(x)
        return xb, x32, out, out32

    def prefill(self, x, positions, cache_start, k_cache, v_cache, out=None, workspace=None,
                stream=None, out32=None):
        """x [B, T, d] BF16 (or FP32: the FP32 residual interface).  Returns the
        BF16 output if `out` is used, else the FP32 one."""
        B, T, _ = x.shape
        xb, x32, out, out32 = self._io(x, out, out32)
        ws = self.workspace(B, T, x.device) if workspace is None else workspace
        _check(lib().qwen_layer_prefill_ex(self.handle, _ptr(xb), _ptr(x32), _ptr(out),
                                           _ptr(out32), B, T, _ptr(positions), _ptr(cache_start),
                                           _ptr(k_cache), _ptr(v_cache), _ptr(ws), ws.numel(),
                                           _stream(stream)), "qwen_layer_prefill")
        return out if out is not None else out32

    def decode(self, x, positions, cache_len, k_cache, v_cache, out=None, workspace=None,
               stream=None, out32=None):
        """x [B, d] BF16 (or FP32).  Returns the BF16 output if `out` is used,
        else the FP32 one."""
        B = x.shape[0]
        xb, x32, out, out32 = self._io(x, out, out32)
        ws = self.workspace(B, 1, x.device) if workspace is None else workspace
        _check(lib().qwen_layer_decode_ex(self.handle, _ptr(xb), _ptr(x32), _ptr(out),
                                          _ptr(out32), B, _ptr(positions), _ptr(cache_len),
                                          _ptr(k_cache), _ptr(v_cache), _ptr(ws), ws.numel(),
                                          _stream(stream)), "qwen_layer_decode")
        return out if out is not None else out32

    def host_workspace(self, B, device="cuda"):
        """Workspace for decode_host (the decode workspace plus host staging)."""
        import torch
        n = lib().qwen_layer_host_workspace_bytes(ctypes.byref(self.cfg.c), B)
        return torch.empty(max(n, 256), dtype=torch.uint8, device=device)

    def decode_host(self, x_host, positions_host, cache_len_host, k_cache, v_cache, y_host,
                    workspace=None, stream=None):
        """One decode step from host buffers: x_host [B, d] BF16, positions_host and
        cache_len_host [B] int32 (CPU tensors, pinned for asynchronous copies);
        the output lands in y_host [B, d] BF16 once the stream is synchronised."""
        import torch
        for n, t in (("x_host", x_host), ("positions_host", positions_host),
                     ("cache_len_host", cache_len_host), ("y_host", y_host)):
            if t.is_cuda or not t.is_contiguous():
                raise ValueError(f"{n} must be a contiguous host tensor")
        if x_host.dtype != torch.bfloat16 or y_host.dtype != torch.bfloat16:
            raise ValueError("x_host and y_host must be bfloat16")
        if positions_host.dtype != torch.int32 or cache_len_host.dtype != torch.int32:
            raise ValueError("positions_host and cache_len_host must be int32")
        B = x_host.shape[0]
        ws = self.host_workspace(B) if workspace is None else workspace
        _check(lib().qwen_layer_decode_host(self.handle, _ptr(x_host), _ptr(y_host), B,
                                            _ptr(positions_host), _ptr(cache_len_host),
                                            _ptr(k_cache), _ptr(v_cache), _ptr(ws), ws.numel(),
                                            _stream(stream)), "qwen_layer_decode_host")
        return y_host

    def moe_ffn(self, r, r_fp32=None, out=None, topk_idx=None, topk_w=None, logits=None,
                workspace=None, stream=None):
        import torch
        _need(r, torch.bfloat16, "r")
        T = r.shape[0]
        out = torch.empty_like(r) if out is None else out
        ws = self.workspace(1, T, r.device) if workspace is None else workspace
        _check(lib().qwen_moe_ffn(self.handle, _ptr(r), _ptr(r_fp32), _ptr(out), T,
                                  _ptr(topk_idx), _ptr(topk_w), _ptr(logits), _ptr(ws),
                                  ws.numel(), _stream(stream)), "qwen_moe_ffn")
        return out

    def poll_error(self, stream=None):
        return lib().qwen_layer_poll_error(self.handle, _stream(stream))

    def set_trace(self, events):
        """events: dict stage-name -> (start, end) torch.cuda.Event (or None to stop).

        Later prefill/decode calls record the given events around those stages."""
        if events is None:
            self._trace = None
            _check(lib().qwen_layer_set_trace(self.handle, None), "qwen_layer_set_trace")
            return
        arr = (ctypes.c_void_p * (2 * len(STAGES)))()
        for name, (ev0, ev1) in events.items():
            i = STAGES.index(name)
            arr[2 * i] = ev0.cuda_event
            arr[2 * i + 1] = ev1.cuda_event
        self._trace = (arr, events)  # keep alive while tracing
        _check(lib().qwen_layer_set_trace(self.handle, arr), "qwen_layer_set_trace")


def launch_count():
    """Kernel launches issued by the library so far in this process."""
    return int(lib().qwen_launch_count())


class Stack:
    """A stack of decoder layers followed by the final RMSNorm and the lm_head
    applied to the last position of each sequence ("Qwen2.5-7B 结构拆解" §01,
    §03.8).  Holds one layer handle and one KV cache pair per layer; every call
    is a sequence of C-ABI calls on the current stream (capturable as a CUDA
    graph: nothing here allocates inside prefill/decode after the first call
    of a given shape).  The hidden state passes between layers in FP32 (the
    FP32 residual interface); only the last layer's output is BF16."""

    def __init__(self, shape, layer_weights, gamma_final, w_lm, max_batch, max_seq,
                 max_tokens=None, device="cuda"):
        import torch
        self.shape = shape
        get = (lambda k: shape[k]) if isinstance(shape, dict) else (lambda k: getattr(shape, k))
        self.d, self.hkv, self.dh = get("d"), get("n_kv_heads"), get("head_dim")
        self.eps = float(get("rms_eps"))
        self.max_batch, self.max_seq = max_batch, max_seq
        self.max_tokens = max_tokens or max_batch * max_seq
        cfg = LayerConfig(shape, max_tokens=self.max_tokens, max_batch=max_batch,
                          max_seq=max_seq, max_position=max_seq)
        self.layers = []
        for w in layer_weights:  # an iterable: weights may be produced one layer at a time
            self.layers.append(Layer(cfg, w))
        self.gamma_final, self.w_lm = gamma_final, w_lm
        self.V = w_lm.shape[0]
        n = len(self.layers)
        shp = (max_batch, self.hkv, max_seq, self.dh)
        self.k = [torch.zeros(shp, dtype=torch.bfloat16, device=device) for _ in range(n)]
        self.v = [torch.zeros(shp, dtype=torch.bfloat16, device=device) for _ in range(n)]
        self._ws = {}
        self._bufs = {}

    def workspace(self, B, T):
        import torch
        key = (B, T)
        if key not in self._ws:
            nbytes = max(self.layers[0].workspace_bytes(B, T), head_workspace_bytes(B, self.d, self.V))
            self._ws[key] = torch.empty(nbytes, dtype=torch.uint8, device=self.k[0].device)
        return self._ws[key]

    def _pingpong(self, shape):
        """Two FP32 buffers for the hidden state between layers plus the BF16
        output of the last layer."""
        import torch
        if shape not in self._bufs:
            dev = self.k[0].device
            self._bufs[shape] = ([torch.empty(shape, dtype=torch.float32, device=dev)
                                  for _ in range(2)],
                                 torch.empty(shape, dtype=torch.bfloat16, device=dev))
        return self._bufs[shape]

    def caches(self, B):
        """Per-layer cache views for the first B sequences."""
        return [(k[:B], v[:B]) for k, v in zip(self.k, self.v)]

    def decode(self, x, positions, cache_len, logits=None):
        """One decode step through every layer, then the head: x [B, d] BF16."""
        B = x.shape[0]
        ws = self.workspace(B, 1)
        f32, last = self._pingpong(tuple(x.shape))
        h = x
        n = len(self.layers)
        for i, layer in enumerate(self.layers):
            if i == n - 1:
                layer.decode(h, positions, cache_len, self.k[i][:B], self.v[i][:B], out=last,
                             workspace=ws)
                h = last
            else:
                h = layer.decode(h, positions, cache_len, self.k[i][:B], self.v[i][:B],
                                 out32=f32[i % 2], workspace=ws)
        return head_last_token(h.view(B, 1, self.d), self.gamma_final, self.w_lm, self.eps,
                               logits=logits, workspace=ws)

    def prefill(self, x, positions, cache_start, logits=None):
        """Prefill of x [B, T, d] through every layer; logits of the last position."""
        B, T, _ = x.shape
        ws = self.workspace(B, T)
        f32, last = self._pingpong(tuple(x.shape))
        h = x
        n = len(self.layers)
        for i, layer in enumerate(self.layers):
            if i == n - 1:
                layer.prefill(h, positions, cache_start, self.k[i][:B], self.v[i][:B], out=last,
                              workspace=ws)
                h = last
            else:
                h = layer.prefill(h, positions, cache_start, self.k[i][:B], self.v[i][:B],
                                  out32=f32[i % 2], workspace=ws)
        return head_last_token(h, self.gamma_final, self.w_lm, self.eps, logits=logits,
                               workspace=ws), h

    def poll_error(self):
        return max(layer.poll_error() for layer in self.layers)
