"""The combine of batches above 4 tokens (a separate fixed-order kernel after
the down GEMM), with and without a shared expert, against the oracle on every
token of batches that hold tokens without a routed row (all logits NaN: their
output is the shared expert's, or zero), and against the CUDA-core path."""
import numpy as np
import pytest
import torch

import block_quantized_expert_gb300 as bqe
from oracle import oracle as orc
from tests import _gpu as G
from workloads import make_tokens, make_weights
from workloads.generate import LayerConfig

pytestmark = pytest.mark.gpu


def _cfg(shared):
    return LayerConfig(index=0, name="tiny_cmb" + ("_sh" if shared else ""), H=256, I=128, E=16, k=4, T=40,
                       shared=shared)


@pytest.fixture(scope="module", params=[False, True], ids=["routed", "shared"])
def layer(request):
    cfg = _cfg(request.param)
    w = make_weights(cfg)
    L = G.make_layer(cfg, w, max_tokens=64)
    yield cfg, w, L
    L.close()


@pytest.mark.parametrize("T", [5, 33, 64])
def test_combine_matches_oracle(layer, T):
    cfg, w, L = layer
    bqe.moe_set_gemm_path(L, 0)
    tk = make_tokens(cfg, n=T)
    lg = tk.logits.astype(np.float32).copy()
    dead = [1, T - 1]  # tokens no expert can take
    lg[dead] = np.nan
    ids = torch.empty((T, cfg.k), dtype=torch.int32, device=G.DEV)
    wd = torch.empty((T, cfg.k), dtype=torch.float32, device=G.DEV)
    out = torch.full((T, cfg.H), 7.0, dtype=torch.float32, device=G.DEV)
    bqe.moe_route_forward(L, G.to_dev(lg), G.to_dev(tk.x_bits.astype(np.uint16), torch.int16), ids, wd, out)
    with pytest.raises(bqe.MoeError):
        bqe.moe_check(L)  # the NaN tokens raise the routing flag
    gi = ids.cpu().numpy()
    assert (gi[dead] == -1).all()
    # the oracle's own routing; a token with only NaN logits routes nowhere
    rid, rw = orc.route_learned(np.where(np.isnan(lg), 0.0, lg).astype(np.float32), cfg.k, cfg.w_scale)
    rid[dead], rw[dead] = -1, 0.0
    assert np.array_equal(gi, rid)
    ref = orc.layer_forward(w, tk.x_bits, rid, rw)
    got = out.cpu().numpy()
    norm, elem = G.compare_out(got, ref)
    assert norm <= G.NORM_TOL and elem <= G.ELEM_TOL, (norm, elem)
    if not cfg.shared:
        assert (got[dead] == 0).all()
    # the CUDA-core path: the same routing, the same combine order
    bqe.moe_set_gemm_path(L, 1)
    out1 = torch.full((T, cfg.H), 7.0, dtype=torch.float32, device=G.DEV)
    bqe.moe_forward(L, G.to_dev(tk.x_bits.astype(np.uint16), torch.int16), ids, wd, out1)
    bqe.moe_check(L)
    o1 = out1.cpu().numpy().astype(np.float64)
    assert np.linalg.norm(got - o1) <= G.NORM_TOL * np.linalg.norm(o1)
    bqe.moe_set_gemm_path(L, 0)


def test_repeated_calls_of_changing_size(layer):
    """Calls in a row of different sizes on the tensor-core path each give
    the oracle's output (no state carried from one call to the next)."""
    cfg, w, L = layer
    bqe.moe_set_gemm_path(L, 2)
    for T in (40, 40, 17):
        tk = make_tokens(cfg, n=T)
        ids, wd = G.route_dev(L, tk.logits, cfg.k)
        out = G.forward_dev(L, tk.x_bits, ids, wd).cpu().numpy()
        bqe.moe_check(L)
        rid, rw = orc.route_learned(tk.logits, cfg.k, cfg.w_scale)
        assert np.array_equal(ids.cpu().numpy(), rid)
        ref = orc.layer_forward(w, tk.x_bits, rid, rw)
        norm, elem = G.compare_out(out, ref)
        assert norm <= G.NORM_TOL and elem <= G.ELEM_TOL
    bqe.moe_set_gemm_path(L, 0)
