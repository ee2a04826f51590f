"""Pins of the NVFP4-style weight variant (CISM VALIDATION, "4-bit
quantization scheme study", row "E2M1 + E4M3 b16 (NVFP4 granularity)": e2m1
elements, one e4m3 scale per 16 elements, plus one fp32 scale per matrix).

- the oracle's element value against the golden e2m1 table times torch's
  e4m3 decoder times the matrix scale, for every code and every finite
  positive scale byte;
- the input generator's encoding: every block's codes are the
  round-to-nearest-even e2m1 grid point of w / (scale * g) (saturating at 6),
  and the block scale the round-to-nearest-even e4m3 value of
  amax / (6 g): checked in fp64 against the fp32 draws;
- the oracle's layer with NVFP4 experts against the dense all-experts numpy
  evaluation (independent dequantisation), and a single expert against the
  textbook SwiGLU MLP;
- NVFP4 reconstructs the fp32 weights more closely than MXFP4 on the same
  draws (the study's finding that scale precision dominates).
"""
import numpy as np
import pytest

from oracle import oracle as orc
from tests import _brute
from workloads import CONFIGS, make_tokens, make_weights
from workloads.generate import LayerConfig, _draw, _streams


def test_nvfp4_element_values():
    e2m1 = _brute.e2m1_table()
    e4m3 = _brute.e4m3_table()
    for g in (1.0, 2.0 ** -20, 3.7e-6):
        for code in range(16):
            for sb in range(0, 127, 5):  # positive finite scale bytes (0x7f is NaN)
                want = e2m1[code] * e4m3[sb] * g
                assert orc.nvfp4_value(code, sb, g) == want, (code, sb, g)
    # closed forms: code 7 (6.0) x byte 0x7e (448) x 1 = 2688; code 9 (-0.5) x byte 1 (2^-9)
    assert orc.nvfp4_value(7, 0x7E, 1.0) == 2688.0
    assert orc.nvfp4_value(9, 1, 1.0) == -(2.0 ** -10)


def _encoding_check(w32, q, s, g):
    rows, K = w32.shape
    assert s.shape == (rows, K // 16) and q.shape == (rows, K // 2)
    assert (s <= 126).all()  # positive finite e4m3 bytes
    e4 = _brute.e4m3_table()
    e2 = _brute.e2m1_table()
    lo, hi = q & 15, q >> 4
    codes = np.stack([lo, hi], -1).reshape(rows, K)
    b = w32.astype(np.float64).reshape(rows, K // 16, 16)
    # the block scale: the e4m3 grid point nearest amax / (6 g) (ties to even code)
    target = (np.abs(w32).reshape(rows, K // 16, 16).max(-1) / np.float32(6.0) / np.float32(g)).astype(np.float64)
    grid = e4[:127]
    best = np.abs(target[..., None] - grid).min(-1)
    assert np.all(np.abs(target - e4[s]) <= best + 1e-12 * np.abs(target))
    # the codes: the e2m1 grid point nearest w / (scale g), or +-6 beyond it
    denom = (e4[s].astype(np.float32) * np.float32(g)).astype(np.float64)
    y = b / np.where(denom > 0, denom, 1.0)[..., None]
    mag = np.abs(e2[codes.reshape(rows, K // 16, 16)])
    grid2 = e2[:8]
    err = np.abs(np.abs(y) - mag)
    nearest = np.abs(np.abs(y)[..., None] - grid2).min(-1)
    assert np.all((err <= nearest + 1e-6 * np.abs(y)) | (np.abs(y) > 6.0))
    # a nonzero code carries the sign of w
    v = e2[codes.reshape(rows, K // 16, 16)]
    assert np.all((v == 0) | (np.signbit(v) == np.signbit(y)))


def test_generator_encoding_is_nearest_grid_point():
    from workloads.generate import encode_nvfp4_rows
    rng = np.random.default_rng(5)
    for K, scale in ((256, 1 / 16), (128, 3.0), (512, 1e-3)):
        w = (rng.standard_normal((24, K)) * scale).astype(np.float32)
        w[0, :16] = 0.0          # an all-zero block
        q, s, g = encode_nvfp4_rows(w)
        assert s[0, 0] == 0 and (q[0, :8] & 0x77).max() == 0
        _encoding_check(w, q, s, g)
        # the matrix scale maps the largest block onto the top of the e4m3 range
        assert abs(float(g) * 6 * 448 - np.abs(w).max()) <= 1e-6 * np.abs(w).max()


def test_nvfp4_layer_matches_dense_bruteforce():
    cfg = CONFIGS[5]
    w = make_weights(cfg)
    assert w.gate_s.shape == (cfg.E, cfg.I, cfg.H // 16) and w.gate_g.shape == (cfg.E,)
    tk = make_tokens(cfg)
    ids, wt = orc.route_learned(tk.logits, cfg.k, cfg.w_scale)
    out, hq, hs = orc.layer_forward(w, tk.x_bits, ids, wt, want_h=True)
    ref = _brute.dense_layer(w, tk.x_bits, ids, wt)
    assert np.abs(out - ref).max() <= 1e-12 * np.abs(ref).max()


def test_nvfp4_single_expert_is_textbook_swiglu():
    cfg = LayerConfig(index=5, name="one_expert_nvfp4", H=256, I=128, E=1, k=1, T=3, w_scale=1.0, wfmt="nvfp4")
    w = make_weights(cfg)
    tk = make_tokens(cfg)
    out = orc.layer_forward(w, tk.x_bits, np.zeros((cfg.T, 1), np.int32), np.ones((cfg.T, 1)))
    x = (tk.x_bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    xd = _brute.dq_mxfp8(*_brute.mxfp8(x))
    Wg = _brute.dq_nvfp4(w.gate_q[0], w.gate_s[0], w.gate_g[0])
    Wu = _brute.dq_nvfp4(w.up_q[0], w.up_s[0], w.up_g[0])
    Wd = _brute.dq_nvfp4(w.down_q[0], w.down_s[0], w.down_g[0])
    g, u = xd @ Wg.T, xd @ Wu.T
    h = g * (1.0 / (1.0 + np.exp(-g))) * u
    ref = _brute.dq_mxfp8(*_brute.mxfp8(h)) @ Wd.T
    assert np.allclose(out, ref, rtol=1e-12, atol=1e-12)


def test_nvfp4_is_closer_to_the_fp32_weights_than_mxfp4():
    # the same fp32 draws (same seed and stream) in both formats
    nv, mx = make_weights(CONFIGS[5]), make_weights(CONFIGS[0])
    kids = _streams(CONFIGS[0].weight_seed)["weights"].spawn(3 * CONFIGS[0].E)
    w32 = _draw(kids[0], CONFIGS[0].I, CONFIGS[0].H).astype(np.float64)  # expert 0's gate
    e_nv = np.linalg.norm(_brute.dq_nvfp4(nv.gate_q[0], nv.gate_s[0], nv.gate_g[0]) - w32)
    e_mx = np.linalg.norm(_brute.dq_mxfp4(mx.gate_q[0], mx.gate_s[0]) - w32)
    assert e_nv < 0.9 * e_mx, (e_nv, e_mx)  # 0.82 on this draw
    _encoding_check(w32.astype(np.float32), nv.gate_q[0], nv.gate_s[0], nv.gate_g[0])
