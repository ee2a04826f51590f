"""ctypes driver of the fp64 CPU oracle (moe_oracle.c).

TEST INFRASTRUCTURE ONLY: imported by the tests, by the smoke check and by
the bench's CPU-baseline leg, never by the library.  The C file is built here
with the host compiler (gcc, C99, -O2, OpenMP) into oracle/_build/.

Every function mirrors one step of the routed-expert FFN layer as the
DeepSeek-V4-Flash guide states it (section 1: router and w_scale; section
3.2: the FFN output equation; section 4: SwiGLU) over the formats colibri's
"DeepSeek V4 target engine" page gives for the checkpoint (fp4 experts,
fp8-e4m3 dense weights with UE8M0 block scales).
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess
import threading
from pathlib import Path

import numpy as np

_HERE = Path(__file__).resolve().parent
_SRC = _HERE / "moe_oracle.c"
_LIB_PATH = _HERE / "_build" / "liboracle.so"
_lock = threading.Lock()
_lib = None

u8p = np.ctypeslib.ndpointer(np.uint8, flags="C_CONTIGUOUS")
u16p = np.ctypeslib.ndpointer(np.uint16, flags="C_CONTIGUOUS")
i32p = np.ctypeslib.ndpointer(np.int32, flags="C_CONTIGUOUS")
f32p = np.ctypeslib.ndpointer(np.float32, flags="C_CONTIGUOUS")
f64p = np.ctypeslib.ndpointer(np.float64, flags="C_CONTIGUOUS")


class OrcLayer(C.Structure):
    _fields_ = [("H", C.c_int), ("I", C.c_int), ("E", C.c_int), ("k", C.c_int)] + [
        (n, C.c_void_p) for n in ("gate_q", "gate_s", "up_q", "up_s", "down_q", "down_s",
                                   "sh_gate_q", "sh_gate_s", "sh_up_q", "sh_up_s",
                                   "sh_down_q", "sh_down_s")] + [
        ("wfmt", C.c_int), ("gate_g", C.c_void_p), ("up_g", C.c_void_p), ("down_g", C.c_void_p)]


def build(force: bool = False) -> Path:
    """Compile moe_oracle.c into oracle/_build/liboracle.so (if stale)."""
    _LIB_PATH.parent.mkdir(parents=True, exist_ok=True)
    if force or not _LIB_PATH.exists() or _LIB_PATH.stat().st_mtime < _SRC.stat().st_mtime:
        tmp = _LIB_PATH.with_suffix(f".{os.getpid()}.tmp")
        subprocess.run(["gcc", "-std=c99", "-O2", "-fopenmp", "-fPIC", "-shared", "-Wall",
                        "-o", str(tmp), str(_SRC), "-lm"], check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def lib():
    global _lib
    with _lock:
        if _lib is None:
            L = C.CDLL(str(build()))
            L.orc_e2m1_value.restype = C.c_double
            L.orc_e2m1_value.argtypes = [C.c_int]
            L.orc_e4m3_value.restype = C.c_double
            L.orc_e4m3_value.argtypes = [C.c_int]
            L.orc_ue8m0_value.restype = C.c_double
            L.orc_ue8m0_value.argtypes = [C.c_int]
            L.orc_nvfp4_value.restype = C.c_double
            L.orc_nvfp4_value.argtypes = [C.c_int, C.c_int, C.c_double]
            L.orc_e4m3_encode.restype = C.c_int
            L.orc_e4m3_encode.argtypes = [C.c_double]
            L.orc_sqrt_softplus.restype = C.c_double
            L.orc_sqrt_softplus.argtypes = [C.c_double]
            L.orc_mxfp8_quantize.restype = None
            L.orc_mxfp8_quantize.argtypes = [f64p, C.c_int, u8p, u8p]
            L.orc_quantize_bf16.argtypes = [u16p, C.c_int, C.c_int, u8p, u8p]
            L.orc_route_learned.argtypes = [f32p, C.c_int, C.c_int, C.c_int, C.c_double, i32p, f64p]
            L.orc_route_prune.argtypes = [i32p, f64p, C.c_int, C.c_int, C.c_int, C.c_double, C.c_double]
            L.orc_route_hash.argtypes = [i32p, C.c_int, i32p, C.c_int, C.c_int, C.c_double, i32p, f64p]
            L.orc_permute.argtypes = [i32p, C.c_int, C.c_int, C.c_int, i32p, i32p, i32p]
            L.orc_layer_forward.argtypes = [C.POINTER(OrcLayer), u16p, i32p, f64p, C.c_int, i32p,
                                            C.c_int, f64p, C.c_void_p, C.c_void_p]
            L.orc_max_threads.restype = C.c_int
            _lib = L
    return _lib


# ---------------------------------------------------------------- formats --
def e2m1_value(code: int) -> float:
    return lib().orc_e2m1_value(int(code))


def e4m3_value(code: int) -> float:
    return lib().orc_e4m3_value(int(code))


def ue8m0_value(code: int) -> float:
    return lib().orc_ue8m0_value(int(code))


def nvfp4_value(code: int, sbyte: int, g: float) -> float:
    """NVFP4-style element: e2m1(code) * e4m3(sbyte) * g (fp64)."""
    return lib().orc_nvfp4_value(int(code), int(sbyte), float(g))


def e4m3_encode(y: float) -> int:
    return lib().orc_e4m3_encode(float(y))


def mxfp8_quantize(v: np.ndarray):
    """MXFP8 of a 1-D fp64 vector (length a multiple of 32) -> (q u8, s u8)."""
    v = np.ascontiguousarray(v, dtype=np.float64)
    q = np.empty(v.size, np.uint8)
    s = np.empty(v.size // 32, np.uint8)
    lib().orc_mxfp8_quantize(v, v.size, q, s)
    return q, s


def quantize_bf16(x_bits: np.ndarray):
    """MXFP8 of bf16 rows [T][H] -> (q [T][H], s [T][H/32])."""
    x = np.ascontiguousarray(x_bits, dtype=np.uint16)
    T, H = x.shape
    q = np.empty((T, H), np.uint8)
    s = np.empty((T, H // 32), np.uint8)
    if lib().orc_quantize_bf16(x, T, H, q, s):
        raise ValueError("orc_quantize_bf16 failed")
    return q, s


def sqrt_softplus(l: float) -> float:
    return lib().orc_sqrt_softplus(float(l))


# ---------------------------------------------------------------- routing --
def route_learned(logits: np.ndarray, k: int, w_scale: float = 1.5):
    lg = np.ascontiguousarray(logits, dtype=np.float32)
    T, E = lg.shape
    ids = np.empty((T, k), np.int32)
    w = np.empty((T, k), np.float64)
    if lib().orc_route_learned(lg, T, E, k, float(w_scale), ids, w):
        raise ValueError("orc_route_learned failed")
    return ids, w


def route_prune(ids: np.ndarray, w: np.ndarray, keep: int, min_w: float = 0.0, rho: float = 0.0):
    """Tail pruning of a learned routing (moe_oracle.c: orc_route_prune) on
    copies of ids [T][k] / w [T][k]: kept prefix rescaled by
    sqrt(((1-rho) S2_all + rho S1_all^2) / ((1-rho) S2_kept + rho S1_kept^2)),
    pruned slots id -1, weight 0."""
    ids = np.array(ids, dtype=np.int32, order="C", copy=True)
    w = np.array(w, dtype=np.float64, order="C", copy=True)
    T, k = ids.shape
    if lib().orc_route_prune(ids, w, T, k, int(keep), float(min_w), float(rho)):
        raise ValueError("orc_route_prune: bad arguments")
    return ids, w


def route_hash(token_ids: np.ndarray, tid2eid: np.ndarray, w_scale: float = 1.5):
    tok = np.ascontiguousarray(token_ids, dtype=np.int32)
    tab = np.ascontiguousarray(tid2eid, dtype=np.int32)
    V, k = tab.shape
    T = tok.size
    ids = np.empty((T, k), np.int32)
    w = np.empty((T, k), np.float64)
    if lib().orc_route_hash(tok, T, tab, V, k, float(w_scale), ids, w):
        raise ValueError("orc_route_hash failed")
    return ids, w


def permute(ids: np.ndarray, E: int):
    ids = np.ascontiguousarray(ids, dtype=np.int32)
    T, k = ids.shape
    off = np.empty(E + 1, np.int32)
    src = np.empty(T * k, np.int32)
    dst = np.empty(T * k, np.int32)
    if lib().orc_permute(ids, T, k, E, off, src, dst):
        raise ValueError("orc_permute failed")
    return off, src, dst


# ------------------------------------------------------------------ layer --
def _layer_struct(w, k: int):
    cfg = w.cfg
    st = OrcLayer(cfg.H, cfg.I, cfg.E, k)
    keep = []
    for n in ("gate_q", "gate_s", "up_q", "up_s", "down_q", "down_s",
              "sh_gate_q", "sh_gate_s", "sh_up_q", "sh_up_s", "sh_down_q", "sh_down_s"):
        a = getattr(w, n)
        if a is None:
            setattr(st, n, None)
        else:
            a = np.ascontiguousarray(a, dtype=np.uint8)
            keep.append(a)
            setattr(st, n, a.ctypes.data)
    st.wfmt = 1 if getattr(cfg, "wfmt", "mxfp4") == "nvfp4" else 0
    for n in ("gate_g", "up_g", "down_g"):
        a = getattr(w, n, None)
        if a is None:
            setattr(st, n, None)
        else:
            a = np.ascontiguousarray(a, dtype=np.float32)
            keep.append(a)
            setattr(st, n, a.ctypes.data)
    return st, keep


def layer_forward(weights, x_bits: np.ndarray, ids: np.ndarray, w: np.ndarray,
                  tokens=None, want_h: bool = False):
    """fp64 layer output for the listed tokens (default: all) of one call.

    weights: a workloads.Weights; x_bits u16 [T][H]; ids i32 [T][k];
    w f64/f32 [T][k].  Returns out [n][H] (and hq [n][k][I], hs [n][k][I/32]
    in the token's own expert order when want_h).
    """
    x = np.ascontiguousarray(x_bits, dtype=np.uint16)
    ids = np.ascontiguousarray(ids, dtype=np.int32)
    wt = np.ascontiguousarray(w, dtype=np.float64)
    T, k = ids.shape
    tok = np.arange(T, dtype=np.int32) if tokens is None else np.ascontiguousarray(tokens, dtype=np.int32)
    n = tok.size
    H, I = weights.cfg.H, weights.cfg.I
    out = np.empty((n, H), np.float64)
    hq = np.empty((n, k, I), np.uint8) if want_h else None
    hs = np.empty((n, k, I // 32), np.uint8) if want_h else None
    st, keep = _layer_struct(weights, k)
    rc = lib().orc_layer_forward(C.byref(st), x, ids, wt, T, tok, n, out,
                                 hq.ctypes.data if want_h else None,
                                 hs.ctypes.data if want_h else None)
    del keep
    if rc:
        raise ValueError(f"orc_layer_forward failed ({rc})")
    return (out, hq, hs) if want_h else out


def max_threads() -> int:
    return lib().orc_max_threads()
