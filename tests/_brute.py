"""Independent dense numpy evaluation of the layer, used only to pin the oracle.

It evaluates EVERY expert on EVERY token (no routing-driven grouping, no
permutation), masks the result with the top-k selection, and uses numpy's
matmul, torch's e4m3 decoder and the input generator's round-to-nearest-even
grid search -- none of the oracle's code.
"""
from __future__ import annotations

import os

import numpy as np
import torch

from workloads.generate import _E4M3_MID, _rne_index

_GOLD = os.path.join(os.path.dirname(__file__), "golden")


def e2m1_table() -> np.ndarray:
    vals = []
    with open(os.path.join(_GOLD, "e2m1_codes.txt")) as f:
        for line in f:
            if line.strip() and not line.startswith("#"):
                vals.append(float(line.split()[1]))
    return np.array(vals, np.float64)


def e4m3_table() -> np.ndarray:
    t = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float64)
    return t.numpy()


def dq_mxfp4(q: np.ndarray, s: np.ndarray) -> np.ndarray:
    """[..., rows, K/2] codes + [..., rows, K/32] scales -> fp64 [..., rows, K]."""
    lo, hi = q & 15, q >> 4
    codes = np.stack([lo, hi], axis=-1).reshape(*q.shape[:-1], q.shape[-1] * 2)
    scale = np.ldexp(1.0, s.astype(np.int64) - 127)
    return e2m1_table()[codes] * np.repeat(scale, 32, axis=-1)


def dq_nvfp4(q: np.ndarray, s: np.ndarray, g: float) -> np.ndarray:
    """[rows, K/2] codes + [rows, K/16] e4m3 scales + matrix scale -> fp64 [rows, K]."""
    lo, hi = q & 15, q >> 4
    codes = np.stack([lo, hi], axis=-1).reshape(*q.shape[:-1], q.shape[-1] * 2)
    return e2m1_table()[codes] * np.repeat(e4m3_table()[s], 16, axis=-1) * float(g)


def dq_routed(weights, name: str, e: int) -> np.ndarray:
    """Expert e's gate / up / down matrix, dequantised in the layer's format."""
    q, s = getattr(weights, name + "_q")[e], getattr(weights, name + "_s")[e]
    if getattr(weights.cfg, "wfmt", "mxfp4") == "nvfp4":
        return dq_nvfp4(q, s, getattr(weights, name + "_g")[e])
    return dq_mxfp4(q, s)


def dq_fp8_tiles(q: np.ndarray, s: np.ndarray) -> np.ndarray:
    vals = e4m3_table()[q]
    scale = np.ldexp(1.0, s.astype(np.int64) - 127)
    return vals * np.kron(scale, np.ones((128, 128)))


def mxfp8(v: np.ndarray):
    """MXFP8 along the last axis (32-blocks): returns (codes u8, scale bytes u8)."""
    sh = v.shape
    b = v.reshape(*sh[:-1], sh[-1] // 32, 32)
    amax = np.abs(b).max(axis=-1)
    _, e = np.frexp(amax)
    ex = np.where(amax > 0, e.astype(np.int64) - 1 - 8, -127)
    ex = np.clip(ex, -127, 127)
    y = np.ldexp(b, -ex[..., None])
    code = _rne_index(np.abs(y), _E4M3_MID) | (np.signbit(y).astype(np.uint8) << 7)
    return code.reshape(sh).astype(np.uint8), (ex + 127).astype(np.uint8)


def dq_mxfp8(q: np.ndarray, s: np.ndarray) -> np.ndarray:
    scale = np.ldexp(1.0, s.astype(np.int64) - 127)
    return e4m3_table()[q] * np.repeat(scale, 32, axis=-1)


def swiglu_expert(xd: np.ndarray, wg: np.ndarray, wu: np.ndarray, wd: np.ndarray):
    """xd [T][H] fp64; wg/wu [I][H]; wd [H][I] -> (y [T][H], hq, hs)."""
    g = xd @ wg.T
    u = xd @ wu.T
    h = g / (1.0 + np.exp(-g)) * u
    hq, hs = mxfp8(h)
    return dq_mxfp8(hq, hs) @ wd.T, hq, hs


def dense_layer(weights, x_bits: np.ndarray, ids: np.ndarray, w: np.ndarray):
    """out [T][H] fp64 by evaluating all experts on all tokens, then masking."""
    cfg = weights.cfg
    x = (np.asarray(x_bits, np.uint32) << 16).view(np.float32).astype(np.float64)
    xq, xs = mxfp8(x)
    xd = dq_mxfp8(xq, xs)
    T = x.shape[0]
    out = np.zeros((T, cfg.H))
    for e in range(cfg.E):
        y, _, _ = swiglu_expert(xd, dq_routed(weights, "gate", e), dq_routed(weights, "up", e),
                                dq_routed(weights, "down", e))
        wt = np.where(ids == e, w, 0.0).sum(axis=1)       # routing weight of e per token
        out += wt[:, None] * y
    if weights.sh_gate_q is not None:
        y, _, _ = swiglu_expert(xd, dq_fp8_tiles(weights.sh_gate_q, weights.sh_gate_s),
                                dq_fp8_tiles(weights.sh_up_q, weights.sh_up_s),
                                dq_fp8_tiles(weights.sh_down_q, weights.sh_down_s))
        out += y
    return out
