"""Pins of the oracle's layer forward: a dense all-experts evaluation in numpy
(masked to the top-k), the single-expert textbook SwiGLU MLP, linearity in
w_scale, token-permutation equivariance.  CPU only, tiny shapes."""
import dataclasses

import numpy as np
import pytest

from oracle import oracle as orc
from tests import _brute
from workloads import CONFIGS, make_tokens, make_weights
from workloads.generate import LayerConfig


def _tiny(**kw):
    base = dict(index=0, name="tiny", H=256, I=128, E=16, k=2, T=4)
    base.update(kw)
    return LayerConfig(**base)


@pytest.mark.parametrize("cfg", [CONFIGS[0],
                                 _tiny(name="tiny_shared", T=6, shared=True),
                                 _tiny(name="tiny_k4", E=8, k=4, T=5, bias="normal0.5")])
def test_layer_matches_dense_bruteforce(cfg):
    w = make_weights(cfg)
    tk = make_tokens(cfg)
    ids, wt = orc.route_learned(tk.logits, cfg.k, cfg.w_scale)
    out, hq, hs = orc.layer_forward(w, tk.x_bits, ids, wt, want_h=True)
    ref = _brute.dense_layer(w, tk.x_bits, ids, wt)
    assert np.abs(out - ref).max() <= 1e-12 * np.abs(ref).max()
    # the requantised h of every (token, expert) equals the dense evaluation's
    x = (tk.x_bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    xd = _brute.dq_mxfp8(*_brute.mxfp8(x))
    for t in range(cfg.T):
        for j in range(cfg.k):
            e = ids[t, j]
            _, rq, rs = _brute.swiglu_expert(xd[t:t + 1], _brute.dq_mxfp4(w.gate_q[e], w.gate_s[e]),
                                             _brute.dq_mxfp4(w.up_q[e], w.up_s[e]),
                                             _brute.dq_mxfp4(w.down_q[e], w.down_s[e]))
            assert np.array_equal(hq[t, j], rq[0]) and np.array_equal(hs[t, j], rs[0])


def test_single_expert_is_textbook_swiglu():
    cfg = _tiny(name="one_expert", E=1, k=1, T=3, w_scale=1.0)
    w = make_weights(cfg)
    tk = make_tokens(cfg)
    ids = np.zeros((cfg.T, 1), np.int32)
    out = orc.layer_forward(w, tk.x_bits, ids, np.ones((cfg.T, 1)))
    x = (tk.x_bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    xd = _brute.dq_mxfp8(*_brute.mxfp8(x))
    Wg = _brute.dq_mxfp4(w.gate_q[0], w.gate_s[0])
    Wu = _brute.dq_mxfp4(w.up_q[0], w.up_s[0])
    Wd = _brute.dq_mxfp4(w.down_q[0], w.down_s[0])
    g, u = xd @ Wg.T, xd @ Wu.T
    h = g * (1.0 / (1.0 + np.exp(-g))) * u
    ref = _brute.dq_mxfp8(*_brute.mxfp8(h)) @ Wd.T
    assert np.allclose(out, ref, rtol=1e-12, atol=1e-12)


def test_output_is_linear_in_w_scale():
    cfg = CONFIGS[0]
    w = make_weights(cfg)
    tk = make_tokens(cfg)
    ids, w15 = orc.route_learned(tk.logits, cfg.k, 1.5)
    ids3, w30 = orc.route_learned(tk.logits, cfg.k, 3.0)
    assert np.array_equal(ids, ids3) and np.array_equal(w30, 2 * w15)
    a = orc.layer_forward(w, tk.x_bits, ids, w15)
    b = orc.layer_forward(w, tk.x_bits, ids, w30)
    assert np.array_equal(b, 2 * a)


def test_token_permutation_permutes_output():
    cfg = dataclasses.replace(CONFIGS[0], T=7)
    w = make_weights(cfg)
    tk = make_tokens(cfg)
    ids, wt = orc.route_learned(tk.logits, cfg.k)
    out = orc.layer_forward(w, tk.x_bits, ids, wt)
    p = np.random.default_rng(0).permutation(cfg.T)
    out_p = orc.layer_forward(w, tk.x_bits[p], ids[p], wt[p])
    assert np.array_equal(out_p, out[p])
    # a subset of tokens gives the same rows as the full call
    sub = orc.layer_forward(w, tk.x_bits, ids, wt, tokens=np.array([5, 1], np.int32))
    assert np.array_equal(sub, out[[5, 1]])


def test_expert_order_is_ascending_and_hash_weights_flat():
    cfg = CONFIGS[0]
    w = make_weights(cfg)
    tk = make_tokens(cfg)
    ids, wt = orc.route_learned(tk.logits, cfg.k)
    out = orc.layer_forward(w, tk.x_bits, ids, wt)
    # swapping the two (id, w) pairs of every token changes nothing: the sum
    # runs in ascending expert order whatever the selection order
    out2 = orc.layer_forward(w, tk.x_bits, ids[:, ::-1].copy(), wt[:, ::-1].copy())
    assert np.array_equal(out, out2)
