"""The CUDA-core whole-layer decode kernel on the other layer shapes its rules
admit, against the fp64 oracle end to end: hidden sizes of 2048 .. 8192
(2 .. 8 K segments of 1024 per gate/up row, so 32 .. 8 rows per gate/up
stage), intermediate sizes of 1024 and 2048 (one or two K segments per down
row), top-k from 1 to 8 over 8 .. 64 experts, MXFP4 and NVFP4-style weights,
with and without the always-on shared expert (fp8 e4m3 rows with a UE8M0
scale per 128 x 128 tile, added to the routed output unweighted, last).
Each shape also runs on the grouped CUDA-core path, whose output it must
match within the oracle tolerance."""
import dataclasses

import numpy as np
import pytest
import torch

import block_quantized_expert_gb300 as bqe
from oracle import oracle as orc
from tests import _gpu as G
from workloads import CONFIGS, make_tokens, make_weights

pytestmark = pytest.mark.gpu

# (H, I, E, k, weight format, shared expert)
SHAPES = [
    (2048, 1024, 64, 8, "mxfp4", False),
    (4096, 1024, 32, 8, "mxfp4", False),
    (8192, 2048, 8, 6, "mxfp4", False),
    (8192, 1024, 8, 2, "mxfp4", False),
    (2048, 1024, 16, 1, "mxfp4", False),
    (2048, 2048, 16, 4, "nvfp4", False),
    (4096, 2048, 32, 6, "mxfp4", True),
    (8192, 1024, 8, 8, "mxfp4", True),
    (2048, 1024, 16, 3, "nvfp4", True),
]


def _cfg(i, H, I, E, k, wfmt, shared):
    return dataclasses.replace(CONFIGS[1], index=60 + i, name=f"decode_shape_{H}x{I}x{E}k{k}_{wfmt}_{shared}",
                               H=H, I=I, E=E, k=k, T=1, steps=4, wfmt=wfmt, shared=shared)


def _call(layer, cfg, lg, xb):
    ids = torch.empty((1, cfg.k), dtype=torch.int32, device=G.DEV)
    w = torch.empty((1, cfg.k), dtype=torch.float32, device=G.DEV)
    out = torch.full((1, cfg.H), 7.0, dtype=torch.float32, device=G.DEV)
    n0 = bqe.moe_kernel_launches(layer)
    bqe.moe_route_forward(layer, G.to_dev(lg.astype(np.float32)), G.to_dev(xb.astype(np.uint16), torch.int16),
                          ids, w, out)
    bqe.moe_check(layer)
    return ids, w, out, bqe.moe_kernel_launches(layer) - n0


@pytest.mark.parametrize("i", range(len(SHAPES)),
                         ids=[f"{h}x{i}_E{e}_k{k}_{f}{'_shared' if sh else ''}" for h, i, e, k, f, sh in SHAPES])
def test_decode_kernel_shape(i):
    cfg = _cfg(i, *SHAPES[i])
    w = make_weights(cfg, seed=2000 + i, cache=False)
    layer = G.make_layer(cfg, w, max_tokens=1)
    try:
        assert bqe.moe_decode_info(layer) == 1, "the shape should take the CUDA-core decode kernel"
        tk = make_tokens(cfg, n=4)
        for t in range(4):
            lg, xb = tk.logits[t:t + 1], tk.x_bits[t:t + 1]
            ids, wt, out, n = _call(layer, cfg, lg, xb)
            assert n == 1  # one kernel for the whole layer
            rid, rw = orc.route_learned(lg, cfg.k, cfg.w_scale)
            assert np.array_equal(ids.cpu().numpy(), rid)
            assert np.abs(wt.cpu().numpy() - rw).max() <= 8 * 2.0 ** -24 * cfg.w_scale
            ref = orc.layer_forward(w, xb, rid, rw)
            norm, elem = G.compare_out(out.cpu().numpy(), ref)
            assert norm <= G.NORM_TOL and elem <= G.ELEM_TOL, (t, norm, elem)
            bqe.moe_set_gemm_path(layer, 1)  # the grouped CUDA-core kernels
            try:
                ids2, _, out2, n2 = _call(layer, cfg, lg, xb)
            finally:
                bqe.moe_set_gemm_path(layer, 0)
            assert n2 > 1 and torch.equal(ids, ids2)
            a, b = out.cpu().numpy().astype(np.float64), out2.cpu().numpy().astype(np.float64)
            assert np.linalg.norm(a - b) <= G.NORM_TOL * np.linalg.norm(b)
    finally:
        layer.close()
        torch.cuda.empty_cache()


def test_decode_kernel_declines_shapes_it_cannot_hold():
    """I = 4096 with six kept experts needs more shared memory than a CTA has:
    the automatic choice falls back (here to the grouped kernels, the tcgen05
    decode kernel taking I <= 2048 only), and asking for the CUDA-core kernel
    is refused."""
    cfg = dataclasses.replace(CONFIGS[1], index=70, name="decode_shape_2048x4096", H=2048, I=4096, E=8, k=6,
                              T=1, steps=1)
    w = make_weights(cfg, seed=2100, cache=False)
    layer = G.make_layer(cfg, w, max_tokens=1)
    try:
        assert bqe.moe_decode_info(layer) != 1
        with pytest.raises(bqe.MoeError) as ei:
            bqe.moe_set_decode_kernel(layer, 1)
        assert ei.value.status == bqe.MOE_ERR_UNSUPPORTED
    finally:
        layer.close()
        torch.cuda.empty_cache()


@pytest.mark.parametrize("setting", [(4, 0.0, 0.0), (6, 0.245, 0.3), (1, 0.0, 0.0)])
def test_decode_kernel_shared_expert_with_pruning(setting):
    """Tail pruning with the shared expert: the kept count m varies per
    token, so the shared expert's position (m) and the down split move; the
    output against the oracle on its own pruned routing (tokens whose keep
    decision sits within fp32 reach of the threshold are skipped)."""
    cfg = _cfg(20, 4096, 2048, 32, 6, "mxfp4", True)
    w = make_weights(cfg, seed=2200, cache=False)
    layer = G.make_layer(cfg, w, max_tokens=1)
    try:
        bqe.moe_set_route_prune(layer, *setting)
        assert bqe.moe_decode_info(layer) == 1
        tk = make_tokens(cfg, n=6)
        keep, min_w, rho = setting
        checked = 0
        for t in range(6):
            lg, xb = tk.logits[t:t + 1], tk.x_bits[t:t + 1]
            rid, rw = orc.route_learned(lg, cfg.k, cfg.w_scale)
            if min_w > 0 and not (np.abs(rw - min_w) > 1e-5).all():
                continue
            pid, pw = orc.route_prune(rid, rw, keep, min_w, rho)
            ids, _, out, n = _call(layer, cfg, lg, xb)
            assert n == 1
            assert np.array_equal(ids.cpu().numpy(), pid)
            ref = orc.layer_forward(w, xb, pid, pw)
            norm, elem = G.compare_out(out.cpu().numpy(), ref)
            assert norm <= G.NORM_TOL and elem <= G.ELEM_TOL, (t, norm, elem)
            checked += 1
        assert checked >= 4
    finally:
        bqe.moe_set_route_prune(layer, cfg.k)
        layer.close()
        torch.cuda.empty_cache()
