"""Pins of the oracle's router (learned sqrt-softplus top-k, hash-routed) and
of its token -> expert permutation, against closed forms, printed values and
library routines (numpy's stable argsort, logaddexp).  CPU only."""
import os

import numpy as np
import pytest

from oracle import oracle as orc
from workloads import CONFIGS, make_hash_table, make_tokens

_GOLD = os.path.join(os.path.dirname(__file__), "golden", "router_closed_forms.txt")


def _gold():
    d = {}
    with open(_GOLD) as f:
        for line in f:
            if line.strip() and not line.startswith("#"):
                key, *vals = line.split()
                d[key] = [float(v) for v in vals]
    return d


def _scores(logits):
    return np.sqrt(np.logaddexp(0.0, logits.astype(np.float64)))


def test_sqrt_softplus_closed_forms():
    g = _gold()
    assert orc.sqrt_softplus(0.0) == pytest.approx(g["sqrt_softplus_0"][0], abs=1e-15)
    assert orc.sqrt_softplus(50.0) == pytest.approx(np.sqrt(50.0), rel=1e-15)
    assert orc.sqrt_softplus(-50.0) == pytest.approx(np.exp(-25.0), rel=1e-12)
    grid = np.linspace(-30, 30, 601)
    got = np.array([orc.sqrt_softplus(v) for v in grid])
    assert np.allclose(got, _scores(grid), rtol=1e-14, atol=0)


@pytest.mark.parametrize("cfg_id", [0, 3])
def test_learned_route_matches_stable_argsort(cfg_id):
    cfg = CONFIGS[cfg_id]
    tk = make_tokens(cfg, n=min(cfg.T, 256))
    ids, w = orc.route_learned(tk.logits, cfg.k, cfg.w_scale)
    s = _scores(tk.logits)
    ref = np.argsort(-s, axis=1, kind="stable")[:, : cfg.k]
    assert np.array_equal(ids, ref)
    sel = np.take_along_axis(s, ids, axis=1)
    assert np.allclose(w, cfg.w_scale * sel / sel.sum(1, keepdims=True), rtol=1e-15, atol=0)
    assert np.allclose(w.sum(1), _gold()["w_scale"][0], rtol=0, atol=1e-12)
    assert (np.diff(w, axis=1) <= 0).all()          # descending-score order


def test_learned_route_ties_go_to_lower_index():
    logits = np.zeros((3, 16), np.float32)
    logits[1, [3, 9]] = 2.0                         # two equal maxima
    ids, w = orc.route_learned(logits, 2)
    assert ids[0].tolist() == [0, 1] and ids[2].tolist() == [0, 1]
    assert ids[1].tolist() == [3, 9]
    assert np.allclose(w[0], 0.75) and np.allclose(w[1], 0.75)
    ids6, w6 = orc.route_learned(np.zeros((1, 256), np.float32), 6)
    assert ids6[0].tolist() == list(range(6)) and np.allclose(w6, 0.25, atol=0, rtol=1e-15)


def test_generator_score_gap():
    """The k-th and (k+1)-th scores (and every adjacent pair above) differ by >= 1e-4."""
    for cid in (0, 1, 2, 3, 4):
        cfg = CONFIGS[cid]
        tk = make_tokens(cfg, n=min(cfg.T * cfg.steps, 8192))
        s = np.sort(_scores(tk.logits), axis=1)[:, ::-1][:, : cfg.k + 1]
        assert (s[:, :-1] - s[:, 1:]).min() >= 1e-4, cid


def test_hash_route_flat_weights():
    g = _gold()
    cfg = CONFIGS[2]
    tab = make_hash_table(cfg)
    assert tab.shape == (129280, 6)
    assert all(len(set(r)) == 6 for r in tab[:5000].tolist())
    tk = make_tokens(cfg)
    ids, w = orc.route_hash(tk.token_ids, tab, cfg.w_scale)
    assert np.array_equal(ids, tab[tk.token_ids])
    assert (w == g["hash_weight_each"][0]).all() and w.mean() == 0.25
    # the guide's printed flat weights of a hash-routed token also sum to w_scale
    assert sum(g["printed_hash_weights"]) == pytest.approx(g["w_scale"][0], abs=1e-12)
    assert w.sum(1) == pytest.approx(g["w_scale"][0])


def _check_perm(ids, E):
    off, src, dst = orc.permute(ids, E)
    flat = ids.ravel()
    assert np.array_equal(src, np.argsort(flat, kind="stable"))
    assert np.array_equal(off, np.concatenate([[0], np.cumsum(np.bincount(flat, minlength=E))]))
    assert np.array_equal(dst[src], np.arange(flat.size))
    assert np.array_equal(src[dst], np.arange(flat.size))
    for e in range(E):
        seg = src[off[e]:off[e + 1]]
        assert (flat[seg] == e).all() and (np.diff(seg) > 0).all()


def test_permute_matches_stable_argsort():
    rng = np.random.default_rng(1)
    _check_perm(rng.integers(0, 256, size=(512, 6)).astype(np.int32), 256)
    _check_perm(np.zeros((7, 3), np.int32), 5)                      # everything to expert 0
    _check_perm(np.full((1, 2), 4, np.int32), 5)                    # T = 1, last expert
    _check_perm(np.array([[2, 2], [2, 2]], np.int32), 3)            # duplicate ids in a row


def test_permute_rejects_bad_ids():
    with pytest.raises(ValueError):
        orc.permute(np.array([[0, 16]], np.int32), 16)
