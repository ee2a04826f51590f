"""GPU parity of the NVFP4-style expert weights (CISM VALIDATION, "4-bit
quantization scheme study", row "E2M1 + E4M3 b16": e2m1 codes, an e4m3 scale
per 16 elements, an fp32 scale per matrix) through the C ABI, against the
fp64 oracle run end to end on its own routing: the tiny layer, one-token
decode calls (grouped path and the whole-layer CUDA-core decode kernel) and
pp512 at full size.  The layer's GEMMs run on the CUDA cores (the
block-scaled tensor-core MMAs take UE8M0 scales per 32 elements only);
routing, sort, quantisation and combine are the MXFP4 layer's kernels.  Same
tolerances as the MXFP4 parity tests."""
import numpy as np
import pytest
import torch

import block_quantized_expert_gb300 as bqe
from oracle import oracle as orc
from tests import _gpu as G
from workloads import CONFIGS

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def tiny():
    cfg = CONFIGS[5]
    w = G.weights_np(5)
    return cfg, w, G.make_layer(cfg, w, max_tokens=64)


@pytest.fixture(scope="module")
def full():
    cfg = CONFIGS[7]
    w = G.weights_np(6)
    return w, G.make_layer(cfg, w, max_tokens=512)


def _run(layer, cfg, tk, n):
    """Route + layer of the first n tokens through the one-call entry point;
    returns the device ids, weights and the output."""
    ids = torch.empty((n, cfg.k), dtype=torch.int32, device=G.DEV)
    w = torch.empty((n, cfg.k), dtype=torch.float32, device=G.DEV)
    out = torch.empty((n, cfg.H), dtype=torch.float32, device=G.DEV)
    bqe.moe_route_forward(layer, G.to_dev(tk.logits[:n].astype(np.float32)),
                          G.to_dev(tk.x_bits[:n].astype(np.uint16), torch.int16), ids, w, out)
    bqe.moe_check(layer)
    return ids, w, out


def _check(cfg, wts, layer, tk, n, sample, name):
    ids, w, out = _run(layer, cfg, tk, n)
    rid, rw = orc.route_learned(tk.logits[:n], cfg.k, cfg.w_scale)
    assert np.array_equal(ids.cpu().numpy(), rid)
    ref, rq, _ = orc.layer_forward(wts, tk.x_bits[:n], rid, rw, tokens=sample, want_h=True)
    norm, elem = G.compare_out(out.cpu().numpy()[sample], ref)
    assert norm <= G.NORM_TOL and elem <= G.ELEM_TOL, (name, norm, elem)
    I = cfg.I
    hq = torch.empty((n * cfg.k, I), dtype=torch.uint8, device=G.DEV)
    hs = torch.empty((n * cfg.k, I // 32), dtype=torch.uint8, device=G.DEV)
    bqe.moe_hidden(layer, n, hq, hs)
    bqe.moe_check(layer)
    hq = hq.cpu().numpy().reshape(n, cfg.k, I)[sample]
    flips = int((hq != rq).sum())
    G.report("hq_flips", {"case": name, "path": 1, "tokens": int(len(sample)), "codes": int(hq.size),
                          "flips": flips, "fraction": flips / hq.size, "norm_err": norm, "elem_err": elem})
    assert flips <= G.HQ_FLIP_TOL * hq.size
    return out


def test_nvfp4_layer_runs_on_cuda_cores(tiny):
    cfg, w, layer = tiny
    with pytest.raises(bqe.MoeError) as ei:
        bqe.moe_set_gemm_path(layer, 2)
    assert ei.value.status == bqe.MOE_ERR_UNSUPPORTED
    with pytest.raises(bqe.MoeError):
        bqe.moe_test_stall_next_decode(layer)  # no whole-layer decode kernel
    bqe.moe_set_gemm_path(layer, 0)


@pytest.mark.parametrize("n", [1, 4, 37])
def test_nvfp4_tiny(tiny, n):
    cfg, w, layer = tiny
    tk = G.tokens(5, n=max(n, cfg.T))
    _check(cfg, w, layer, tk, n, np.arange(n, dtype=np.int32), f"tiny_nvfp4_T{n}")


def test_nvfp4_decode_calls(full):
    """One-token calls on the grouped CUDA-core path (moe_set_gemm_path 1),
    with the requantised h checked too."""
    w, layer = full
    cfg = CONFIGS[6]
    tk = G.tokens(6, n=6)
    bqe.moe_set_gemm_path(layer, 1)
    try:
        for t in range(6):
            one = type(tk)(x_bits=tk.x_bits[t:t + 1], logits=tk.logits[t:t + 1], token_ids=None)
            _check(cfg, w, layer, one, 1, np.array([0], np.int32), "decode_nvfp4")
    finally:
        bqe.moe_set_gemm_path(layer, 0)


def test_nvfp4_decode_kernel(full):
    """One-token calls on the automatic path: the CUDA-core whole-layer decode
    kernel (one launch), the NVFP4 block dot product taking an e4m3 scale per
    16-element half and the matrix scales on the finished dot products;
    routing bit for bit and the output against the oracle end to end, and
    within the oracle tolerance of the grouped path's output."""
    w, layer = full
    cfg = CONFIGS[6]
    assert bqe.moe_decode_info(layer) == 1
    tk = G.tokens(6, n=8)
    for t in range(8):
        one = type(tk)(x_bits=tk.x_bits[t:t + 1], logits=tk.logits[t:t + 1], token_ids=None)
        n0 = bqe.moe_kernel_launches(layer)
        ids, wt, out = _run(layer, cfg, one, 1)
        assert bqe.moe_kernel_launches(layer) - n0 == 1
        rid, rw = orc.route_learned(one.logits, cfg.k, cfg.w_scale)
        assert np.array_equal(ids.cpu().numpy(), rid)
        ref = orc.layer_forward(w, one.x_bits, rid, rw)
        norm, elem = G.compare_out(out.cpu().numpy(), ref)
        assert norm <= G.NORM_TOL and elem <= G.ELEM_TOL, (t, norm, elem)
        bqe.moe_set_gemm_path(layer, 1)
        try:
            _, _, out2 = _run(layer, cfg, one, 1)
        finally:
            bqe.moe_set_gemm_path(layer, 0)
        a, b = out.cpu().numpy().astype(np.float64), out2.cpu().numpy().astype(np.float64)
        assert np.linalg.norm(a - b) <= G.NORM_TOL * np.linalg.norm(b)


def test_nvfp4_prefill_pp512(full):
    w, layer = full
    cfg = CONFIGS[7]
    tk = G.tokens(7)
    out = _check(cfg, w, layer, tk, cfg.T, np.arange(cfg.T, dtype=np.int32), "pp512_nvfp4")
    # deterministic: a second call gives the same bytes
    _, _, out2 = _run(layer, cfg, tk, cfg.T)
    assert out2.cpu().numpy().tobytes() == out.cpu().numpy().tobytes()
