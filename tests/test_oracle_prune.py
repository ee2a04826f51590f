"""Pins of the oracle's routed-expert tail pruning (orc_route_prune) and of
the empty-slot reading of ids (-1) in its permutation and layer forward.

DeepSeek-V4-Flash guide, section 3.2 item 3: pruning the tail of a learned
routing and rescaling the kept weights so that the expected squared norm of
the routed sum is unchanged -- in quadrature (L2) for mutually orthogonal
expert outputs, by alpha_gen(rho) for outputs with pairwise correlation rho,
linearly (L1) in the collinear limit.  CPU only."""
from pathlib import Path

import numpy as np
import pytest

from oracle import oracle as orc
from tests import _brute
from workloads import CONFIGS, make_tokens, make_weights
from workloads.generate import LayerConfig

GOLD = Path(__file__).parent / "golden" / "route_prune.txt"


def _gold(tag):
    rows = []
    for line in GOLD.read_text().splitlines():
        if line.startswith(tag + " "):
            rows.append(line.split()[1:])
    return rows


def _one(w, keep, min_w=0.0, rho=0.0):
    w = np.asarray(w, np.float64)[None, :]
    ids = np.arange(w.shape[1], dtype=np.int32)[None, :] + 10
    i2, w2 = orc.route_prune(ids, w, keep, min_w, rho)
    return i2[0], w2[0]


def test_kept_count_hand_cases():
    for r in _gold("case"):
        w = [float(v) for v in r[:6]]
        keep, min_w, m = int(r[6]), float(r[7]), int(r[8])
        ids, w2 = _one(w, keep, min_w)
        assert (ids[:m] == np.arange(10, 10 + m)).all() and (ids[m:] == -1).all(), r
        assert (w2[m:] == 0.0).all() and (w2[:m] > 0).all(), r


def test_factor_hand_cases():
    for r in _gold("factor"):
        keep, rho = int(r[0]), float(r[1])
        alpha = float(r[5])
        w = [0.45, 0.30, 0.25, 0.20, 0.18, 0.12]
        _, w2 = _one(w, keep, 0.0, rho)
        assert w2[:keep] / np.array(w[:keep]) == pytest.approx(alpha, rel=1e-7)


def test_printed_l1_factor():
    # top-4 carrying 81.2 % of w_scale = 1.5, the rest split over experts 5, 6
    r = _gold("printed_l1")[0]
    share, printed = float(r[1]), float(r[3])
    top = 1.5 * share
    w = [0.4 * top, 0.25 * top, 0.2 * top, 0.15 * top, 0.6 * (1.5 - top), 0.4 * (1.5 - top)]
    _, w2 = _one(w, 4, 0.0, 1.0)
    assert round(w2[0] / w[0], 2) == printed


def test_two_experts_closed_forms():
    # k = 2, keep 1: L2 -> sqrt(w0^2 + w1^2); L1 -> w0 + w1
    for w0, w1 in ((0.9, 0.6), (0.75, 0.75), (1.4, 0.1)):
        _, a = _one([w0, w1], 1, 0.0, 0.0)
        _, b = _one([w0, w1], 1, 0.0, 1.0)
        assert a[0] == pytest.approx(np.hypot(w0, w1), rel=1e-14) and a[1] == 0.0
        assert b[0] == pytest.approx(w0 + w1, rel=1e-14) and b[1] == 0.0


@pytest.mark.parametrize("rho", [0.0, 0.3, 1.0])
@pytest.mark.parametrize("keep,min_w", [(5, 0.0), (4, 0.0), (6, 0.11), (3, 0.2)])
def test_variance_preserved_monte_carlo(rho, keep, min_w):
    """The stated purpose, checked by simulation: expert outputs e_i with unit
    variance per feature and pairwise correlation rho; the mean squared norm
    of sum_i w_i e_i over the kept experts (rescaled) matches the unpruned
    one.  A wrong factor (L1 for L2, a dropped term) misses by percents."""
    rng = np.random.default_rng(5)
    lg = make_tokens(CONFIGS[1], n=64).logits
    ids, w = orc.route_learned(lg, 6)
    i2, w2 = orc.route_prune(ids, w, keep, min_w, rho)
    d = 400_000
    z0 = rng.standard_normal(d)
    e = np.sqrt(rho) * z0[None, :] + np.sqrt(1.0 - rho) * rng.standard_normal((6, d))
    for t in range(0, 64, 8):
        full = np.mean((w[t] @ e) ** 2)
        kept = np.mean((np.where(i2[t] >= 0, w2[t], 0.0) @ e) ** 2)
        assert kept == pytest.approx(full, rel=0.02), (t, full, kept)


def test_sum_and_square_sum_limits():
    lg = make_tokens(CONFIGS[3], n=256).logits
    ids, w = orc.route_learned(lg, 6)
    _, a = orc.route_prune(ids, w, 4, 0.0, 0.0)
    _, b = orc.route_prune(ids, w, 4, 0.0, 1.0)
    assert np.allclose((a ** 2).sum(1), (w ** 2).sum(1), rtol=1e-13)
    assert np.allclose(b.sum(1), 1.5, rtol=1e-13)
    # no pruning: the routing is returned unchanged, bit for bit
    i0, w0 = orc.route_prune(ids, w, 6, 0.0, 0.3)
    assert np.array_equal(i0, ids) and w0.tobytes() == w.tobytes()
    with pytest.raises(ValueError):
        orc.route_prune(ids, w, 0)
    with pytest.raises(ValueError):
        orc.route_prune(ids, w, 3, 0.0, 1.5)


def test_permute_skips_empty_slots():
    # worked by hand: rows 0..3 -> experts 3, -, 1, 3
    off, src, dst = orc.permute(np.array([[3, -1], [1, 3]], np.int32), 4)
    assert off.tolist() == [0, 0, 1, 1, 3]
    assert src[:3].tolist() == [2, 0, 3]
    assert dst.tolist() == [1, -1, 0, 2]
    with pytest.raises(ValueError):
        orc.permute(np.array([[3, -2]], np.int32), 4)


def test_forward_with_pruned_slots_matches_dense_bruteforce():
    cfg = LayerConfig(index=0, name="tiny_k4", H=256, I=128, E=8, k=4, T=5)
    wts = make_weights(cfg)
    tk = make_tokens(cfg)
    ids, w = orc.route_learned(tk.logits, cfg.k, cfg.w_scale)
    i2, w2 = orc.route_prune(ids, w, 2, 0.0, 0.0)
    out, hq, hs = orc.layer_forward(wts, tk.x_bits, i2, w2, want_h=True)
    ref = _brute.dense_layer(wts, tk.x_bits, i2, w2)
    assert np.abs(out - ref).max() <= 1e-12 * np.abs(ref).max()
    assert (hq[:, 2:] == 0).all() and (hs[:, 2:] == 0).all()
    # an empty slot adds exactly what a weight-0 expert adds: nothing
    i3 = np.where(i2 < 0, 0, i2).astype(np.int32)
    out3 = orc.layer_forward(wts, tk.x_bits, i3, w2)
    assert out3.tobytes() == out.tobytes()
