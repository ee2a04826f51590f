"""Helpers of the GPU tests: upload a workload, build a layer through the C
ABI, and compare the CUDA path with the oracle."""
from __future__ import annotations

import functools

import numpy as np
import torch

import block_quantized_expert_gb300 as bqe
from oracle import oracle as orc
from workloads import CONFIGS, make_tokens, make_weights

DEV = "cuda:0"

# Output tolerance of the layer against the fp64 oracle (normwise relative L2
# error and per-element error relative to rms(out)).
NORM_TOL = 2e-3
ELEM_TOL = 5e-2
# Requantised-h codes may differ from the oracle's where fp32 h sits at an
# e4m3 rounding boundary that fp64 h does not cross: the fp32 h is within
# ~1e-6 relative of the fp64 one, and a code step is 1/8 to 1/16 of the
# value, so a flip needs h within ~1e-5 of a rounding boundary, a chance of
# order 1e-5 per code (the expectation of "far below 1e-4" of the codes).
HQ_FLIP_TOL = 1e-4


def report(kind: str, rec: dict):
    """Append one record to the parity report (JSON lines) named by
    BQE_PARITY_REPORT, if set (observed flip counts and errors)."""
    import json
    import os
    path = os.environ.get("BQE_PARITY_REPORT")
    if path:
        with open(path, "a") as f:
            f.write(json.dumps({"kind": kind, **rec}) + "\n")


def to_dev(a, dtype=None):
    a = np.array(a)
    if a.dtype == np.uint16:
        a = a.view(np.int16)
    t = torch.from_numpy(a)
    if dtype is not None:
        t = t.view(dtype)
    return t.to(DEV)


@functools.lru_cache(maxsize=2)
def weights_np(cfg_id: int):
    return make_weights(CONFIGS[cfg_id])


def upload(w) -> dict:
    d = {}
    for n in ("gate_q", "gate_s", "up_q", "up_s", "down_q", "down_s",
              "sh_gate_q", "sh_gate_s", "sh_up_q", "sh_up_s", "sh_down_q", "sh_down_s",
              "gate_g", "up_g", "down_g"):
        a = getattr(w, n, None)
        if a is not None:
            d[n] = to_dev(a)
    return d


def make_layer(cfg, w, max_tokens: int) -> bqe.Layer:
    mc = bqe.MoeConfig(cfg.H, cfg.I, cfg.E, cfg.k, max_tokens, cfg.shared, cfg.w_scale,
                       bqe.MOE_WEIGHTS_NVFP4 if cfg.wfmt == "nvfp4" else bqe.MOE_WEIGHTS_MXFP4)
    dw = upload(w)
    layer = bqe.moe_create(mc, dw)
    torch.cuda.synchronize()
    del dw
    return layer


def compare_out(got: np.ndarray, ref: np.ndarray):
    """Return (normwise rel L2 error, max |err| / rms(ref))."""
    err = got.astype(np.float64) - ref
    rms = np.sqrt(np.mean(ref ** 2))
    return float(np.linalg.norm(err) / np.linalg.norm(ref)), float(np.abs(err).max() / rms)


def route_dev(layer, logits_np, k):
    T = logits_np.shape[0]
    lg = to_dev(logits_np.astype(np.float32))
    ids = torch.empty((T, k), dtype=torch.int32, device=DEV)
    w = torch.empty((T, k), dtype=torch.float32, device=DEV)
    bqe.moe_route(layer, lg, ids, w)
    return ids, w


def forward_dev(layer, x_bits_np, ids, w):
    T = x_bits_np.shape[0]
    x = to_dev(x_bits_np.astype(np.uint16), torch.int16)
    out = torch.empty((T, layer.cfg.hidden), dtype=torch.float32, device=DEV)
    bqe.moe_forward(layer, x, ids, w, out)
    return out


def tokens(cfg_id: int, n=None):
    return make_tokens(CONFIGS[cfg_id], n=n)
