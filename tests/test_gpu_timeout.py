"""The bounded-wait error path on the GPU, made to run out on purpose in a
permitted way: a test hook makes the next decode call wait for a flag value
that no CTA ever writes (plain global-memory flags; no hardware barrier is
given a wrong count), with the wait limit set to a few milliseconds.  Every
CTA's wait then runs out, the kernel frees its tensor memory and exits, the
call reports MOE_ERR_TIMEOUT through moe_check, and the next calls on the
same layer and context are correct again.  Both whole-layer decode kernels
(the CUDA-core GEMV and the tcgen05 one) take the hook."""
import time

import numpy as np
import pytest
import torch

import block_quantized_expert_gb300 as bqe
from oracle import oracle as orc
from tests import _gpu as G
from workloads import CONFIGS

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def decode_layer():
    cfg = CONFIGS[1]
    w = G.weights_np(1)
    return cfg, w, G.make_layer(cfg, w, max_tokens=4)


def _call(layer, tk, t):
    H, k = layer.cfg.hidden, layer.cfg.top_k
    ids = torch.empty((1, k), dtype=torch.int32, device=G.DEV)
    w = torch.empty((1, k), dtype=torch.float32, device=G.DEV)
    out = torch.full((1, H), 7.0, dtype=torch.float32, device=G.DEV)
    bqe.moe_route_forward(layer, G.to_dev(tk.logits[t:t + 1].astype(np.float32)),
                          G.to_dev(tk.x_bits[t:t + 1].astype(np.uint16), torch.int16), ids, w, out)
    return ids, w, out


def _check_oracle(cfg, wts, tk, t, ids, out):
    rid, rw = orc.route_learned(tk.logits[t:t + 1], cfg.k, cfg.w_scale)
    assert np.array_equal(ids.cpu().numpy(), rid)
    ref = orc.layer_forward(wts, tk.x_bits[t:t + 1], rid, rw)
    norm, elem = G.compare_out(out.cpu().numpy(), ref)
    assert norm <= G.NORM_TOL and elem <= G.ELEM_TOL, (norm, elem)


def test_wait_limit_arguments(decode_layer):
    _, _, layer = decode_layer
    for bad in (0.0, -1.0, 1e-6, 100.0, float("nan")):
        with pytest.raises(bqe.MoeError) as ei:
            bqe.moe_set_wait_limit(layer, bad)
        assert ei.value.status == bqe.MOE_ERR_INVALID_ARG
    bqe.moe_set_wait_limit(layer, 2.0)


@pytest.mark.parametrize("kind", [1, 2], ids=["gemv", "tcgen05"])
def test_stalled_decode_times_out_and_layer_recovers(decode_layer, kind):
    cfg, wts, layer = decode_layer
    bqe.moe_set_gemm_path(layer, 0)
    bqe.moe_set_decode_kernel(layer, kind)
    tk = G.tokens(1, n=4)
    ids, _, out = _call(layer, tk, 0)       # a normal call first
    bqe.moe_check(layer)
    _check_oracle(cfg, wts, tk, 0, ids, out)

    bqe.moe_set_wait_limit(layer, 0.005)    # 5 ms per wait
    bqe.moe_test_stall_next_decode(layer)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    _call(layer, tk, 1)
    with pytest.raises(bqe.MoeError) as ei:
        bqe.moe_check(layer)                # synchronises, then reads the flag
    elapsed = time.perf_counter() - t0
    assert ei.value.status == bqe.MOE_ERR_TIMEOUT
    assert "wait" in bqe.moe_last_error(layer)
    # every wait gave up within a few limits, not after the default 2 s
    assert elapsed < 1.0, elapsed
    bqe.moe_check(layer)                    # the flag was cleared

    # the hook is one-shot and the context stays usable: the next calls on
    # the decode kernel (which allocates the same tensor memory the stalled
    # launch freed) and on the grouped kernels match the oracle
    bqe.moe_set_wait_limit(layer, 2.0)
    for t in (2, 3):
        ids, _, out = _call(layer, tk, t)
        bqe.moe_check(layer)
        _check_oracle(cfg, wts, tk, t, ids, out)
    bqe.moe_set_gemm_path(layer, 2)
    ids, _, out = _call(layer, tk, 1)
    bqe.moe_check(layer)
    _check_oracle(cfg, wts, tk, 1, ids, out)
    bqe.moe_set_gemm_path(layer, 0)
    bqe.moe_set_decode_kernel(layer, 0)
