"""The whole-layer decode kernels (one token through moe_route_forward on the
automatic path: route, quantise, gate/up, down and combine in one
cooperative launch) against the fp64 oracle and against the grouped
tensor-core kernels, eagerly and replayed from a CUDA graph.  The decode
shape runs every test on both kernels: the CUDA-core split-K GEMV (kind 1,
the automatic choice) and the tcgen05 kernel (kind 2); the tiny shape has
only the tcgen05 one."""
import numpy as np
import pytest
import torch

import block_quantized_expert_gb300 as bqe
from oracle import oracle as orc
from tests import _gpu as G
from workloads import CONFIGS

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def decode_layer_base():
    cfg = CONFIGS[1]
    w = G.weights_np(1)
    return cfg, w, G.make_layer(cfg, w, max_tokens=64)


@pytest.fixture(params=[1, 2], ids=["gemv", "tcgen05"])
def decode_layer(request, decode_layer_base):
    cfg, w, layer = decode_layer_base
    bqe.moe_set_gemm_path(layer, 0)
    bqe.moe_set_decode_kernel(layer, request.param)
    assert bqe.moe_decode_info(layer) == request.param
    yield cfg, w, layer
    bqe.moe_set_decode_kernel(layer, 0)


@pytest.fixture(scope="module")
def tiny_layer():
    cfg = CONFIGS[0]
    w = G.weights_np(0)
    return cfg, w, G.make_layer(cfg, w, max_tokens=64)


def _route_forward(layer, logits_np, x_bits_np, path):
    bqe.moe_set_gemm_path(layer, path)
    H, k = layer.cfg.hidden, layer.cfg.top_k
    ids = torch.empty((1, k), dtype=torch.int32, device=G.DEV)
    w = torch.empty((1, k), dtype=torch.float32, device=G.DEV)
    out = torch.full((1, H), 7.0, dtype=torch.float32, device=G.DEV)
    n0 = bqe.moe_kernel_launches(layer)
    bqe.moe_route_forward(layer, G.to_dev(logits_np.astype(np.float32)),
                          G.to_dev(x_bits_np.astype(np.uint16), torch.int16), ids, w, out)
    bqe.moe_check(layer)
    return ids, w, out, bqe.moe_kernel_launches(layer) - n0


def _check_token(cfg, wts, layer, tk, t):
    lg, xb = tk.logits[t:t + 1], tk.x_bits[t:t + 1]
    ids, w, out, n = _route_forward(layer, lg, xb, 0)
    assert n == 1  # one kernel for the whole layer
    rid, rw = orc.route_learned(lg, cfg.k, cfg.w_scale)
    assert np.array_equal(ids.cpu().numpy(), rid)
    assert np.abs(w.cpu().numpy() - rw).max() <= 8 * 2.0 ** -24 * cfg.w_scale
    ref = orc.layer_forward(wts, xb, rid, rw)  # the oracle end to end, on its own routing
    norm, elem = G.compare_out(out.cpu().numpy(), ref)
    assert norm <= G.NORM_TOL and elem <= G.ELEM_TOL, (norm, elem)
    # the grouped tcgen05 kernels: the same routing bit for bit; the output
    # within the oracle tolerance of theirs (the decode kernel multiplies
    # with the operands swapped, so fp32 sums may round differently)
    ids2, w2, out2, n2 = _route_forward(layer, lg, xb, 2)
    assert n2 > 1
    assert torch.equal(ids, ids2) and torch.equal(w, w2)
    o1, o2 = out.cpu().numpy().astype(np.float64), out2.cpu().numpy().astype(np.float64)
    assert np.linalg.norm(o1 - o2) <= G.NORM_TOL * np.linalg.norm(o2)


def test_decode_kernel_decode_shape(decode_layer):
    cfg, wts, layer = decode_layer
    tk = G.tokens(1, n=10)
    for t in range(10):
        _check_token(cfg, wts, layer, tk, t)


def test_decode_kernel_tiny_shape(tiny_layer):
    """H = 256, I = 128: two gate/up tiles of two K-steps, no stream-K split,
    most CTAs without weight work (they only route, and write no output)."""
    cfg, wts, layer = tiny_layer
    tk = G.tokens(0, n=6)
    for t in range(6):
        _check_token(cfg, wts, layer, tk, t)


def test_decode_kernel_graph_replay(decode_layer):
    cfg, wts, layer = decode_layer
    bqe.moe_set_gemm_path(layer, 0)
    tk = G.tokens(1, n=4)
    lg = torch.zeros((1, cfg.E), dtype=torch.float32, device=G.DEV)
    xb = torch.zeros((1, cfg.H), dtype=torch.int16, device=G.DEV)
    ids = torch.empty((1, cfg.k), dtype=torch.int32, device=G.DEV)
    w = torch.empty((1, cfg.k), dtype=torch.float32, device=G.DEV)
    out = torch.empty((1, cfg.H), dtype=torch.float32, device=G.DEV)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        bqe.moe_route_forward(layer, lg, xb, ids, w, out)
        s.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            bqe.moe_route_forward(layer, lg, xb, ids, w, out)
    for t in range(4):
        lg.copy_(G.to_dev(tk.logits[t:t + 1].astype(np.float32)))
        xb.copy_(G.to_dev(tk.x_bits[t:t + 1].astype(np.uint16), torch.int16))
        g.replay()
        torch.cuda.synchronize()
        bqe.moe_check(layer)
        ids_e, w_e, out_e, _ = _route_forward(layer, tk.logits[t:t + 1], tk.x_bits[t:t + 1], 0)
        assert torch.equal(ids, ids_e) and torch.equal(w, w_e)
        assert out.cpu().numpy().tobytes() == out_e.cpu().numpy().tobytes()


def test_decode_kernel_unroutable_token(tiny_layer):
    """All logits NaN: no expert can be selected; the ids are -1, the output
    is zero (every row dropped) and moe_check reports the bad routing."""
    cfg, wts, layer = tiny_layer
    bqe.moe_set_gemm_path(layer, 0)
    lg = torch.full((1, cfg.E), float("nan"), dtype=torch.float32, device=G.DEV)
    xb = G.to_dev(G.tokens(0, n=1).x_bits.astype(np.uint16), torch.int16)
    ids = torch.empty((1, cfg.k), dtype=torch.int32, device=G.DEV)
    w = torch.empty((1, cfg.k), dtype=torch.float32, device=G.DEV)
    out = torch.full((1, cfg.H), 7.0, dtype=torch.float32, device=G.DEV)
    bqe.moe_route_forward(layer, lg, xb, ids, w, out)
    with pytest.raises(bqe.MoeError) as ei:
        bqe.moe_check(layer)
    assert ei.value.status == bqe.MOE_ERR_INVALID_ARG
    assert (ids.cpu().numpy() == -1).all()
    assert (out.cpu().numpy() == 0).all()
    # the layer stays usable
    tk = G.tokens(0, n=1)
    _check_token(cfg, wts, layer, tk, 0)


def test_decode_host_entry_zero_copy_and_staged(decode_layer):
    """moe_forward_host for one token: page-locked buffers are read and
    written in place by the decode kernel (one launch, no copies), pageable
    buffers go through the staging copies; both give the device entry's
    bytes, eagerly and replayed from a CUDA graph."""
    cfg, wts, layer = decode_layer
    bqe.moe_set_gemm_path(layer, 0)
    tk = G.tokens(1, n=3)
    for t in range(3):
        lg, xb = tk.logits[t:t + 1].astype(np.float32), tk.x_bits[t:t + 1]
        _, _, out_d, _ = _route_forward(layer, lg, xb, 0)
        ref = out_d.cpu().numpy().tobytes()
        for pinned in (True, False):
            xh = torch.from_numpy(xb.view(np.int16).copy())
            lh = torch.from_numpy(lg.copy())
            oh = torch.full((1, cfg.H), 7.0, dtype=torch.float32)
            if pinned:
                xh, lh, oh = xh.pin_memory(), lh.pin_memory(), oh.pin_memory()
            n0 = bqe.moe_kernel_launches(layer)
            bqe.moe_forward_host(layer, xh, lh, oh)
            torch.cuda.synchronize()
            bqe.moe_check(layer)
            assert bqe.moe_kernel_launches(layer) - n0 == 1
            assert oh.numpy().tobytes() == ref, pinned
    # graph of the zero-copy call: new host inputs written between replays
    xh = torch.zeros((1, cfg.H), dtype=torch.int16).pin_memory()
    lh = torch.zeros((1, cfg.E), dtype=torch.float32).pin_memory()
    oh = torch.zeros((1, cfg.H), dtype=torch.float32).pin_memory()
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        bqe.moe_forward_host(layer, xh, lh, oh)
        s.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            bqe.moe_forward_host(layer, xh, lh, oh)
    for t in range(3):
        lg, xb = tk.logits[t:t + 1].astype(np.float32), tk.x_bits[t:t + 1]
        xh.copy_(torch.from_numpy(xb.view(np.int16).copy()))
        lh.copy_(torch.from_numpy(lg.copy()))
        oh.fill_(7.0)
        g.replay()
        torch.cuda.synchronize()
        bqe.moe_check(layer)
        _, _, out_d, _ = _route_forward(layer, lg, xb, 0)
        assert oh.numpy().tobytes() == out_d.cpu().numpy().tobytes()


def test_two_layers_interleaved_in_one_graph(decode_layer, tiny_layer):
    """Decode calls of two layers alternating on one stream (each kernel
    launched while the previous layer's still runs, as consecutive layers
    of a model are): every call gives the bytes of the same call made alone."""
    cfg_a, _, la = decode_layer
    cfg_b, _, lb = tiny_layer
    bqe.moe_set_gemm_path(la, 0)
    bqe.moe_set_gemm_path(lb, 0)
    ta, tb = G.tokens(1, n=3), G.tokens(0, n=3)

    def bufs(cfg, tk, t):
        return (G.to_dev(tk.logits[t:t + 1].astype(np.float32)), G.to_dev(tk.x_bits[t:t + 1].astype(np.uint16), torch.int16),
                torch.empty((1, cfg.k), dtype=torch.int32, device=G.DEV),
                torch.empty((1, cfg.k), dtype=torch.float32, device=G.DEV),
                torch.empty((1, cfg.H), dtype=torch.float32, device=G.DEV))

    calls = []
    for t in range(3):
        calls.append((la, bufs(cfg_a, ta, t)))
        calls.append((lb, bufs(cfg_b, tb, t)))
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        for L, (lg, xb, ids, w, out) in calls:  # warm-up, eager
            bqe.moe_route_forward(L, lg, xb, ids, w, out)
        s.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            for L, (lg, xb, ids, w, out) in calls:
                bqe.moe_route_forward(L, lg, xb, ids, w, out)
    g.replay()
    torch.cuda.synchronize()
    bqe.moe_check(la)
    bqe.moe_check(lb)
    for L, (lg, xb, ids, w, out) in calls:
        ids1, w1, out1 = torch.empty_like(ids), torch.empty_like(w), torch.empty_like(out)
        bqe.moe_route_forward(L, lg, xb, ids1, w1, out1)
        torch.cuda.synchronize()
        assert torch.equal(ids, ids1) and torch.equal(w, w1)
        assert out.cpu().numpy().tobytes() == out1.cpu().numpy().tobytes()


def test_decode_kernel_choice(decode_layer_base, tiny_layer):
    """The automatic choice: the CUDA-core kernel where its shape rules allow
    (H, I multiples of 1024), else the tcgen05 kernel; an explicit choice the
    shape does not allow is refused and leaves the setting unchanged."""
    _, _, layer = decode_layer_base
    _, _, tiny = tiny_layer
    bqe.moe_set_gemm_path(layer, 0)
    bqe.moe_set_gemm_path(tiny, 0)
    assert bqe.moe_decode_info(layer) == 1
    assert bqe.moe_decode_info(tiny) == 2
    with pytest.raises(bqe.MoeError) as ei:
        bqe.moe_set_decode_kernel(tiny, 1)
    assert ei.value.status == bqe.MOE_ERR_UNSUPPORTED
    assert bqe.moe_decode_info(tiny) == 2
    for bad in (-1, 3):
        with pytest.raises(bqe.MoeError) as ei:
            bqe.moe_set_decode_kernel(layer, bad)
        assert ei.value.status == bqe.MOE_ERR_INVALID_ARG
    bqe.moe_set_gemm_path(layer, 2)   # the tcgen05-only GEMM path has no decode kernel
    assert bqe.moe_decode_info(layer) == 0
    bqe.moe_set_gemm_path(layer, 0)


def test_decode_kernels_agree(decode_layer_base):
    """The two decode kernels on the same tokens: the same routing bit for bit,
    outputs within the oracle tolerance of each other, and the CUDA-core
    kernel's output repeatable bit for bit (fixed reduction order)."""
    cfg, _, layer = decode_layer_base
    bqe.moe_set_gemm_path(layer, 0)
    tk = G.tokens(1, n=6)
    for t in range(6):
        res = {}
        for kind in (1, 2):
            bqe.moe_set_decode_kernel(layer, kind)
            res[kind] = _route_forward(layer, tk.logits[t:t + 1], tk.x_bits[t:t + 1], 0)
        bqe.moe_set_decode_kernel(layer, 1)
        again = _route_forward(layer, tk.logits[t:t + 1], tk.x_bits[t:t + 1], 0)
        bqe.moe_set_decode_kernel(layer, 0)
        (i1, w1, o1, _), (i2, w2, o2, _) = res[1], res[2]
        assert torch.equal(i1, i2) and torch.equal(w1, w2)
        a, b = o1.cpu().numpy().astype(np.float64), o2.cpu().numpy().astype(np.float64)
        assert np.linalg.norm(a - b) <= G.NORM_TOL * np.linalg.norm(b)
        assert o1.cpu().numpy().tobytes() == again[2].cpu().numpy().tobytes()
