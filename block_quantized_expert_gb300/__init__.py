"""Python binding of libmoe (include/moe.h): the routed-expert FFN layer of a
DeepSeek-V4-Flash-style MoE on one GB300, MXFP4 experts, MXFP8 activations.

Argument marshalling only: every step runs in libmoe's CUDA kernels.  Tensors
are torch CUDA tensors (device memory and streams come from PyTorch); the
functions check dtype, shape, device and contiguity, pass raw pointers and
the current CUDA stream, and raise MoeError on a non-zero status.  There is no
fallback: if libmoe.so cannot be loaded the import of the functions fails.
"""
from __future__ import annotations

import ctypes as C
from dataclasses import dataclass
from typing import Optional

from . import _build

MOE_OK, MOE_ERR_INVALID_ARG, MOE_ERR_UNSUPPORTED, MOE_ERR_OOM, MOE_ERR_CUDA, MOE_ERR_TIMEOUT = range(6)
_STATUS = {1: "MOE_ERR_INVALID_ARG", 2: "MOE_ERR_UNSUPPORTED", 3: "MOE_ERR_OOM",
           4: "MOE_ERR_CUDA", 5: "MOE_ERR_TIMEOUT"}

# Every symbol include/moe.h declares.
EXPORTS = ("moe_create", "moe_destroy", "moe_route", "moe_route_hash", "moe_permute",
           "moe_quantize", "moe_forward", "moe_forward_host", "moe_hidden", "moe_check",
           "moe_workspace_bytes", "moe_last_error", "moe_set_gemm_path", "moe_set_stage_events",
           "moe_kernel_launches", "moe_permute_noalloc", "moe_set_trace", "moe_route_forward",
           "moe_set_route_prune", "moe_set_wait_limit", "moe_test_stall_next_decode", "moe_test_decode_split",
           "moe_set_decode_kernel", "moe_decode_info")


class MoeError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"{_STATUS.get(status, status)}: {msg}")
        self.status = status


class moe_config(C.Structure):
    _fields_ = [("hidden", C.c_int), ("inter", C.c_int), ("n_experts", C.c_int),
                ("top_k", C.c_int), ("max_tokens", C.c_int), ("has_shared", C.c_int),
                ("w_scale", C.c_float), ("weight_format", C.c_int)]


MOE_WEIGHTS_MXFP4, MOE_WEIGHTS_NVFP4 = 0, 1


_WEIGHT_FIELDS = ("gate_q", "gate_s", "up_q", "up_s", "down_q", "down_s",
                  "sh_gate_q", "sh_gate_s", "sh_up_q", "sh_up_s", "sh_down_q", "sh_down_s")


class moe_weights(C.Structure):
    _fields_ = [(n, C.c_void_p) for n in _WEIGHT_FIELDS + ("gate_g", "up_g", "down_g")]


_lib = None


def load_library(build: bool = True) -> C.CDLL:
    """Load (building first if stale and `build`) the in-tree libmoe.so."""
    global _lib
    if _lib is not None:
        return _lib
    path = _build.build() if build else _build.LIB
    if not path.exists():
        raise ImportError(f"libmoe.so not found at {path}")
    L = C.CDLL(str(path))
    vp, i, f = C.c_void_p, C.c_int, C.c_float
    sigs = {
        "moe_create": ([C.POINTER(moe_config), C.POINTER(moe_weights), vp, C.POINTER(vp)], i),
        "moe_destroy": ([vp], i),
        "moe_route": ([vp, vp, i, vp, vp, vp], i),
        "moe_route_hash": ([vp, vp, vp, i, i, vp, vp, vp], i),
        "moe_permute": ([vp, vp, i, vp, vp, vp, vp], i),
        "moe_quantize": ([vp, vp, i, vp, vp, vp], i),
        "moe_forward": ([vp, vp, i, vp, vp, vp, vp], i),
        "moe_forward_host": ([vp, vp, vp, i, vp, vp], i),
        "moe_hidden": ([vp, i, vp, vp, vp], i),
        "moe_check": ([vp, vp], i),
        "moe_workspace_bytes": ([C.POINTER(moe_config)], C.c_size_t),
        "moe_last_error": ([vp], C.c_char_p),
        "moe_set_gemm_path": ([vp, i], i),
        "moe_set_stage_events": ([vp, C.POINTER(vp), i], i),
        "moe_kernel_launches": ([vp], C.c_ulonglong),
        "moe_permute_noalloc": ([vp, i, i, i, vp, vp, vp, vp], i),
        "moe_set_trace": ([vp, vp, C.c_size_t], i),
        "moe_route_forward": ([vp, vp, vp, i, vp, vp, vp, vp], i),
        "moe_set_route_prune": ([vp, i, f, f], i),
        "moe_set_wait_limit": ([vp, C.c_double], i),
        "moe_test_stall_next_decode": ([vp], i),
        "moe_test_decode_split": ([C.c_int, C.c_int, C.c_int, C.c_int, C.c_int, C.c_int, C.POINTER(C.c_int)], i),
        "moe_set_decode_kernel": ([vp, i], i),
        "moe_decode_info": ([vp, C.POINTER(C.c_int)], i),
    }
    for name, (args, res) in sigs.items():
        fn = getattr(L, name)
        fn.argtypes, fn.restype = args, res
    _lib = L
    return L


def _check(status: int, layer_ptr=None):
    if status != MOE_OK:
        msg = load_library().moe_last_error(layer_ptr)
        raise MoeError(status, msg.decode() if msg else "")


def _stream(stream) -> int:
    import torch
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _ptr(t, dtype, shape=None, name="tensor"):
    import torch
    if t is None:
        raise ValueError(f"{name} is None")
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    return t.data_ptr()


def _hptr(t, dtype, shape, name):
    import torch
    if not isinstance(t, torch.Tensor) or t.is_cuda or t.dtype != dtype or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous host {dtype} tensor")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}")
    return t.data_ptr()


@dataclass
class MoeConfig:
    hidden: int
    inter: int
    n_experts: int
    top_k: int
    max_tokens: int
    has_shared: bool = False
    w_scale: float = 1.5
    weight_format: int = MOE_WEIGHTS_MXFP4

    def c(self) -> moe_config:
        return moe_config(self.hidden, self.inter, self.n_experts, self.top_k, self.max_tokens,
                          int(bool(self.has_shared)), self.w_scale, int(self.weight_format))


class Layer:
    """Owner of a moe_layer*; freed by moe_destroy (or when collected)."""

    def __init__(self, ptr: int, cfg: MoeConfig):
        self.ptr = C.c_void_p(ptr)
        self.cfg = cfg

    def close(self):
        if self.ptr and self.ptr.value:
            moe_destroy(self)

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def moe_workspace_bytes(cfg: MoeConfig) -> int:
    return load_library().moe_workspace_bytes(C.byref(cfg.c()))


def moe_create(cfg: MoeConfig, weights: dict, stream=None) -> Layer:
    """weights: dict of CUDA tensors named as the fields of moe_weights (uint8;
    NVFP4 layers also float32 gate_g, up_g, down_g [E])."""
    import torch
    lib = load_library()
    H, I, E = cfg.hidden, cfg.inter, cfg.n_experts
    nv = cfg.weight_format == MOE_WEIGHTS_NVFP4
    blk = 16 if nv else 32
    shapes = {"gate_q": (E, I, H // 2), "gate_s": (E, I, H // blk), "up_q": (E, I, H // 2),
              "up_s": (E, I, H // blk), "down_q": (E, H, I // 2), "down_s": (E, H, I // blk),
              "sh_gate_q": (I, H), "sh_gate_s": (I // 128, H // 128), "sh_up_q": (I, H),
              "sh_up_s": (I // 128, H // 128), "sh_down_q": (H, I), "sh_down_s": (H // 128, I // 128)}
    wt = moe_weights()
    for n in _WEIGHT_FIELDS:
        if n.startswith("sh_") and not cfg.has_shared:
            setattr(wt, n, None)
            continue
        setattr(wt, n, _ptr(weights.get(n), torch.uint8, shapes[n], n))
    for n in ("gate_g", "up_g", "down_g"):
        setattr(wt, n, _ptr(weights.get(n), torch.float32, (E,), n) if nv else None)
    out = C.c_void_p()
    _check(lib.moe_create(C.byref(cfg.c()), C.byref(wt), _stream(stream), C.byref(out)))
    return Layer(out.value, cfg)


def moe_destroy(layer: Layer):
    lib = load_library()
    st = lib.moe_destroy(layer.ptr)
    layer.ptr = C.c_void_p(None)
    _check(st)


def moe_set_gemm_path(layer: Layer, path: int):
    _check(load_library().moe_set_gemm_path(layer.ptr, int(path)), layer.ptr)


def moe_set_decode_kernel(layer: Layer, kind: int):
    """One-token calls: 0 automatic, 1 the CUDA-core GEMV kernel, 2 the tcgen05 kernel."""
    _check(load_library().moe_set_decode_kernel(layer.ptr, int(kind)), layer.ptr)


def moe_decode_info(layer: Layer) -> int:
    """The whole-layer kernel a one-token call takes: 0 none, 1 CUDA-core GEMV, 2 tcgen05."""
    kind = C.c_int(0)
    _check(load_library().moe_decode_info(layer.ptr, C.byref(kind)), layer.ptr)
    return kind.value


def moe_set_route_prune(layer: Layer, keep: int, min_w: float = 0.0, rho: float = 0.0):
    """Tail pruning of the learned router: keep at most `keep` experts, stop at
    the first weight below `min_w`, rescale the kept weights for correlation
    `rho` (0: L2 quadrature, 1: linear).  keep >= k with min_w <= 0: off."""
    _check(load_library().moe_set_route_prune(layer.ptr, int(keep), float(min_w), float(rho)), layer.ptr)


def moe_set_wait_limit(layer: Layer, seconds: float):
    """Wall-time limit of the layer's device-side waits (default 2 s)."""
    _check(load_library().moe_set_wait_limit(layer.ptr, float(seconds)), layer.ptr)


def moe_test_decode_split(num_sms: int, kept: int, hidden: int, inter: int, nvfp4: bool = False,
                          shared: bool = False) -> list:
    """The CUDA-core decode kernel's down-row cuts (host computation, no GPU)."""
    cut = (C.c_int * (num_sms + 1))()
    _check(load_library().moe_test_decode_split(num_sms, kept, hidden, inter, int(nvfp4), int(shared), cut))
    return list(cut)


def moe_test_stall_next_decode(layer: Layer):
    """Test hook: the next one-token decode-kernel call cannot complete its
    hand-off, runs out its bounded waits and reports MOE_ERR_TIMEOUT."""
    _check(load_library().moe_test_stall_next_decode(layer.ptr), layer.ptr)


def moe_set_stage_events(layer: Layer, events):
    """events: 6 torch.cuda.Event (recorded by the next moe_forward), or None."""
    lib = load_library()
    if events is None:
        _check(lib.moe_set_stage_events(layer.ptr, None, 0), layer.ptr)
        return
    if len(events) != 6:
        raise ValueError("need 6 events")
    for ev in events:  # torch creates the CUDA event lazily
        if ev.cuda_event == 0:
            ev.record()
    arr = (C.c_void_p * 6)(*[ev.cuda_event for ev in events])
    _check(lib.moe_set_stage_events(layer.ptr, arr, 6), layer.ptr)


def moe_route(layer: Layer, logits, ids, w, stream=None):
    import torch
    T = logits.shape[0]
    c = layer.cfg
    st = load_library().moe_route(layer.ptr, _ptr(logits, torch.float32, (T, c.n_experts), "logits"), T,
                                  _ptr(ids, torch.int32, (T, c.top_k), "ids"),
                                  _ptr(w, torch.float32, (T, c.top_k), "w"), _stream(stream))
    _check(st, layer.ptr)


def moe_route_hash(layer: Layer, token_ids, tid2eid, ids, w, stream=None):
    import torch
    T = token_ids.shape[0]
    V = tid2eid.shape[0]
    c = layer.cfg
    st = load_library().moe_route_hash(layer.ptr, _ptr(token_ids, torch.int32, (T,), "token_ids"),
                                       _ptr(tid2eid, torch.int32, (V, c.top_k), "tid2eid"), V, T,
                                       _ptr(ids, torch.int32, (T, c.top_k), "ids"),
                                       _ptr(w, torch.float32, (T, c.top_k), "w"), _stream(stream))
    _check(st, layer.ptr)


def moe_permute(layer: Layer, ids, offsets, row_src, row_dst, stream=None):
    import torch
    T = ids.shape[0]
    c = layer.cfg
    R = T * c.top_k
    st = load_library().moe_permute(layer.ptr, _ptr(ids, torch.int32, (T, c.top_k), "ids"), T,
                                    _ptr(offsets, torch.int32, (c.n_experts + 1,), "offsets"),
                                    _ptr(row_src, torch.int32, (R,), "row_src"),
                                    _ptr(row_dst, torch.int32, (R,), "row_dst"), _stream(stream))
    _check(st, layer.ptr)


def moe_permute_noalloc(ids, n_experts: int, offsets, row_src, row_dst, stream=None):
    """The grouping of moe_permute without a layer and without allocating
    (scratch in a static device array; T * top_k <= 65536)."""
    import torch
    T, k = ids.shape
    R = T * k
    st = load_library().moe_permute_noalloc(
        _ptr(ids, torch.int32, (T, k), "ids"), T, k, n_experts,
        _ptr(offsets, torch.int32, (n_experts + 1,), "offsets"),
        _ptr(row_src, torch.int32, (R,), "row_src"), _ptr(row_dst, torch.int32, (R,), "row_dst"),
        _stream(stream))
    _check(st)


def moe_quantize(layer: Layer, x, q, s, stream=None):
    import torch
    T = x.shape[0]
    H = layer.cfg.hidden
    st = load_library().moe_quantize(layer.ptr, _ptr(x, torch.int16, (T, H), "x"), T,
                                     _ptr(q, torch.uint8, (T, H), "q"),
                                     _ptr(s, torch.uint8, (T, H // 32), "s"), _stream(stream))
    _check(st, layer.ptr)


def moe_forward(layer: Layer, x, ids, w, out, stream=None):
    """x: int16 CUDA tensor [T][H] holding bf16 bits (or a bfloat16 tensor)."""
    import torch
    T = x.shape[0]
    c = layer.cfg
    if x.dtype == torch.bfloat16:
        x = x.view(torch.int16)
    st = load_library().moe_forward(layer.ptr, _ptr(x, torch.int16, (T, c.hidden), "x"), T,
                                    _ptr(ids, torch.int32, (T, c.top_k), "ids"),
                                    _ptr(w, torch.float32, (T, c.top_k), "w"),
                                    _ptr(out, torch.float32, (T, c.hidden), "out"), _stream(stream))
    _check(st, layer.ptr)


def moe_route_forward(layer: Layer, logits, x, ids, w, out, stream=None):
    """Routing and layer in one call (ids, w and out are written)."""
    import torch
    T = x.shape[0]
    c = layer.cfg
    if x.dtype == torch.bfloat16:
        x = x.view(torch.int16)
    st = load_library().moe_route_forward(
        layer.ptr, _ptr(logits, torch.float32, (T, c.n_experts), "logits"),
        _ptr(x, torch.int16, (T, c.hidden), "x"), T, _ptr(ids, torch.int32, (T, c.top_k), "ids"),
        _ptr(w, torch.float32, (T, c.top_k), "w"), _ptr(out, torch.float32, (T, c.hidden), "out"),
        _stream(stream))
    _check(st, layer.ptr)


def moe_forward_host(layer: Layer, x, logits, out, stream=None):
    """Host tensors (pinned for overlap): x int16 [T][H], logits f32 [T][E], out f32 [T][H]."""
    import torch
    T = x.shape[0]
    c = layer.cfg
    st = load_library().moe_forward_host(layer.ptr, _hptr(x, torch.int16, (T, c.hidden), "x"),
                                         _hptr(logits, torch.float32, (T, c.n_experts), "logits"), T,
                                         _hptr(out, torch.float32, (T, c.hidden), "out"),
                                         _stream(stream))
    _check(st, layer.ptr)


def moe_hidden(layer: Layer, T: int, hq, hs, stream=None):
    import torch
    c = layer.cfg
    R = T * c.top_k
    st = load_library().moe_hidden(layer.ptr, T, _ptr(hq, torch.uint8, (R, c.inter), "hq"),
                                   _ptr(hs, torch.uint8, (R, c.inter // 32), "hs"), _stream(stream))
    _check(st, layer.ptr)


def moe_check(layer: Layer, stream=None) -> int:
    """Synchronise the stream; raise MoeError if a device-side check fired."""
    st = load_library().moe_check(layer.ptr, _stream(stream))
    _check(st, layer.ptr)
    return st


def moe_set_trace(layer: Layer, buf):
    """buf: CUDA int64 tensor of >= max(48 * num_sms + 4, 8 * num_sms + 1024) entries, or None."""
    import torch
    if buf is None:
        _check(load_library().moe_set_trace(layer.ptr, None, 0), layer.ptr)
        return
    _check(load_library().moe_set_trace(layer.ptr, _ptr(buf, torch.int64, None, "buf"), buf.numel()),
           layer.ptr)


def moe_kernel_launches(layer: Layer) -> int:
    return int(load_library().moe_kernel_launches(layer.ptr))


def moe_last_error(layer: Optional[Layer] = None) -> str:
    m = load_library().moe_last_error(layer.ptr if layer else None)
    return m.decode() if m else ""
