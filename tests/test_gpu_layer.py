"""GPU parity of the CUDA path (through the C ABI) with the fp64 CPU oracle,
on every workload configuration, for each GEMM kernel path.

Integer work (routing ids, permutation, MXFP8 activation bytes) must match
bit for bit; routing weights within fp32 rounding of the fp64 value; the
layer output within NORM_TOL (normwise relative L2) and ELEM_TOL * rms(out)
per element; requantised-h codes may flip at e4m3 rounding boundaries on at
most HQ_FLIP_TOL of the codes.
"""
import ctypes as C

import numpy as np
import pytest
import torch

import block_quantized_expert_gb300 as bqe
from oracle import oracle as orc
from tests import _gpu as G
from workloads import CONFIGS, make_hash_table

pytestmark = pytest.mark.gpu

PATHS = [1, 2]  # GEMM kernel paths under test (1 = CUDA cores, 2 = tcgen05)


@pytest.fixture(scope="module")
def tiny():
    cfg = CONFIGS[0]
    w = G.weights_np(0)
    return cfg, w, G.make_layer(cfg, w, max_tokens=512)


@pytest.fixture(scope="module")
def full():
    cfg = CONFIGS[3]
    w = G.weights_np(1)
    return w, G.make_layer(cfg, w, max_tokens=512)


@pytest.fixture(scope="module")
def full_shared():
    cfg = CONFIGS[4]
    w = G.weights_np(4)
    return w, G.make_layer(cfg, w, max_tokens=8192)


def _route_check(layer, logits, k, w_scale=1.5):
    ids, w = G.route_dev(layer, logits, k)
    rid, rw = orc.route_learned(logits, k, w_scale)
    assert np.array_equal(ids.cpu().numpy(), rid)
    # fp32 evaluation of exp, log1p, sqrt, a k-term sum and one division:
    # each routing weight (<= w_scale) is within 8 fp32 roundings of the value
    assert np.abs(w.cpu().numpy() - rw).max() <= 8 * 2.0 ** -24 * w_scale
    return ids, w, rid, rw


def _perm_check(layer, ids_dev, E):
    T, k = ids_dev.shape
    off = torch.empty(E + 1, dtype=torch.int32, device=G.DEV)
    src = torch.empty(T * k, dtype=torch.int32, device=G.DEV)
    dst = torch.empty(T * k, dtype=torch.int32, device=G.DEV)
    bqe.moe_permute(layer, ids_dev, off, src, dst)
    ro, rs, rd = orc.permute(ids_dev.cpu().numpy(), E)
    assert np.array_equal(off.cpu().numpy(), ro)
    assert np.array_equal(src.cpu().numpy(), rs)
    assert np.array_equal(dst.cpu().numpy(), rd)


def _quant_check(layer, x_bits):
    T, H = x_bits.shape
    q = torch.empty((T, H), dtype=torch.uint8, device=G.DEV)
    s = torch.empty((T, H // 32), dtype=torch.uint8, device=G.DEV)
    bqe.moe_quantize(layer, G.to_dev(x_bits, torch.int16), q, s)
    rq, rs = orc.quantize_bf16(x_bits)
    assert np.array_equal(s.cpu().numpy(), rs)
    assert np.array_equal(q.cpu().numpy(), rq)


def _forward_check(layer, weights, x_bits, ids_dev, w_dev, sample, path, rid=None, rw=None, name=""):
    """The layer output of `sample` tokens (and their requantised h codes)
    against the oracle.  The oracle runs end to end on its own routing
    (rid, rw from orc.route_*) where the test routed through the router;
    tests that give the layer hand-made routing pass it to both."""
    bqe.moe_set_gemm_path(layer, path)
    out = G.forward_dev(layer, x_bits, ids_dev, w_dev).cpu().numpy()
    T, k = ids_dev.shape
    I = layer.cfg.inter
    hq = torch.empty((T * k, I), dtype=torch.uint8, device=G.DEV)
    hs = torch.empty((T * k, I // 32), dtype=torch.uint8, device=G.DEV)
    bqe.moe_hidden(layer, T, hq, hs)
    bqe.moe_check(layer)
    if rid is None:
        rid, rw = ids_dev.cpu().numpy(), w_dev.cpu().numpy().astype(np.float64)
    assert np.array_equal(ids_dev.cpu().numpy(), rid)
    ref, rq, rsc = orc.layer_forward(weights, x_bits, rid, rw, tokens=sample, want_h=True)
    norm, elem = G.compare_out(out[sample], ref)
    assert norm <= G.NORM_TOL and elem <= G.ELEM_TOL, (norm, elem)
    hq = hq.cpu().numpy().reshape(T, k, I)[sample]
    live = rid[sample] >= 0  # h rows of routed slots
    n_codes = int(live.sum()) * I
    n_flips = int((hq != rq)[live].sum())
    flips = n_flips / max(1, n_codes)
    G.report("hq_flips", {"case": name, "path": path, "tokens": int(len(sample)), "codes": n_codes,
                          "flips": n_flips, "fraction": flips, "norm_err": norm, "elem_err": elem})
    assert flips <= G.HQ_FLIP_TOL, flips
    return out, norm, elem, flips


def tile_covering_sample(rid, E, extra=0, seed=0):
    """Tokens such that every 128-row tile of every non-empty expert segment
    (the row tiles the grouped GEMMs take, including each ragged last tile)
    holds at least two compared rows: a random row of the tile and its last
    row.  Segments are the oracle's stable counting sort of the rows t*k+j."""
    off, src, _ = orc.permute(rid, E)
    k = rid.shape[1]
    rng = np.random.default_rng(seed)
    toks = set()
    for e in range(E):
        n = int(off[e + 1] - off[e])
        for u in range(0, n, 128):
            m = min(128, n - u)
            for r in (int(rng.integers(0, m)), m - 1):
                toks.add(int(src[off[e] + u + r]) // k)
    if extra:
        toks.update(int(t) for t in rng.choice(rid.shape[0], extra, replace=False))
    return np.array(sorted(toks), dtype=np.int32)


@pytest.mark.parametrize("path", PATHS)
def test_tiny_config_all_steps(tiny, path):
    cfg, w, layer = tiny
    tk = G.tokens(0)
    ids, wd, rid, rw = _route_check(layer, tk.logits, cfg.k)
    _perm_check(layer, ids, cfg.E)
    _quant_check(layer, tk.x_bits)
    _forward_check(layer, w, tk.x_bits, ids, wd, np.arange(cfg.T), path, rid, rw, "tiny")


@pytest.mark.parametrize("path", PATHS)
def test_tiny_ragged_segments_and_one_hot_expert(tiny, path):
    """Segments longer than a 128-row tile with ragged tails, empty experts."""
    cfg, w, layer = tiny
    T = 300
    tk = G.tokens(0, n=T)
    ids = np.tile(np.array([[3, 7]], np.int32), (T, 1))
    ids[::5] = [[7, 3]]
    ids[1::7] = [[15, 0]]
    wt = np.tile(np.array([[0.9, 0.6]], np.float32), (T, 1))
    ids_d, w_d = G.to_dev(ids), G.to_dev(wt)
    _perm_check(layer, ids_d, cfg.E)
    _forward_check(layer, w, tk.x_bits, ids_d, w_d, np.arange(T), path, ids, wt.astype(np.float64), "ragged")


def test_route_ties_and_hash(tiny):
    cfg, w, layer = tiny
    ids, wd = G.route_dev(layer, np.zeros((3, cfg.E), np.float32), cfg.k)
    assert ids.cpu().tolist() == [[0, 1]] * 3
    assert np.allclose(wd.cpu().numpy(), 0.75)


@pytest.mark.parametrize("path", PATHS)
def test_decode_t1_calls(full, path):
    """The decode workload: independent T = 1 calls, fresh logits each."""
    w, layer = full
    cfg = CONFIGS[1]
    tk = G.tokens(1, n=12)
    for t in range(12):
        ids, wd, rid, rw = _route_check(layer, tk.logits[t:t + 1], cfg.k)
        _forward_check(layer, w, tk.x_bits[t:t + 1], ids, wd, np.array([0]), path, rid, rw, "decode_t1")


@pytest.mark.parametrize("path", PATHS)
def test_batched_decode_hash_then_learned(full, path):
    w, layer = full
    cfg = CONFIGS[2]
    tk = G.tokens(2)
    tab = make_hash_table(cfg)
    ids = torch.empty((cfg.T, cfg.k), dtype=torch.int32, device=G.DEV)
    wd = torch.empty((cfg.T, cfg.k), dtype=torch.float32, device=G.DEV)
    bqe.moe_route_hash(layer, G.to_dev(tk.token_ids), G.to_dev(tab), ids, wd)
    rid, rw = orc.route_hash(tk.token_ids, tab, cfg.w_scale)
    assert np.array_equal(ids.cpu().numpy(), rid) and (wd.cpu().numpy() == 0.25).all()
    _perm_check(layer, ids, cfg.E)
    _forward_check(layer, w, tk.x_bits, ids, wd, np.arange(cfg.T), path, rid, rw, "batched_hash")
    ids2, wd2, rid2, rw2 = _route_check(layer, tk.logits, cfg.k)
    _forward_check(layer, w, tk.x_bits, ids2, wd2, np.arange(cfg.T), path, rid2, rw2, "batched_learned")


@pytest.mark.parametrize("path", PATHS)
def test_prefill_pp512(full, path):
    w, layer = full
    cfg = CONFIGS[3]
    tk = G.tokens(3)
    ids, wd, rid, rw = _route_check(layer, tk.logits, cfg.k)
    _perm_check(layer, ids, cfg.E)
    _quant_check(layer, tk.x_bits)
    # every token: all 128-row tiles of all segments are compared
    _forward_check(layer, w, tk.x_bits, ids, wd, np.arange(cfg.T, dtype=np.int32), path, rid, rw, "pp512")


@pytest.mark.parametrize("path", PATHS)
def test_prefill_8192_zipf_shared(full_shared, path):
    w, layer = full_shared
    cfg = CONFIGS[4]
    tk = G.tokens(4)
    ids, wd, rid, rw = _route_check(layer, tk.logits, cfg.k)
    _perm_check(layer, ids, cfg.E)
    # two rows of every 128-row tile of every segment (the Zipf head
    # expert's ~60 tiles, the ragged tails, the one-row segments) plus 64
    # random tokens; their shared-expert rows span every token tile too
    sample = tile_covering_sample(rid, cfg.E, extra=64, seed=1)
    # and one token of every 128-token tile of the shared expert's rows
    sample = np.union1d(sample, np.arange(0, cfg.T, 128) + 77).astype(np.int32)
    _forward_check(layer, w, tk.x_bits, ids, wd, sample, path, rid, rw, "prefill8192")


def test_forward_is_deterministic_and_host_entry_matches(tiny):
    cfg, w, layer = tiny
    tk = G.tokens(0, n=64)
    ids, wd = G.route_dev(layer, tk.logits, cfg.k)
    a = G.forward_dev(layer, tk.x_bits, ids, wd).cpu().numpy()
    b = G.forward_dev(layer, tk.x_bits, ids, wd).cpu().numpy()
    assert a.tobytes() == b.tobytes()
    xh = torch.from_numpy(tk.x_bits.view(np.int16).copy()).pin_memory()
    lh = torch.from_numpy(tk.logits.copy()).pin_memory()
    oh = torch.empty((64, cfg.H), dtype=torch.float32).pin_memory()
    bqe.moe_forward_host(layer, xh, lh, oh)
    torch.cuda.synchronize()
    assert oh.numpy().tobytes() == a.tobytes()


@pytest.mark.parametrize("path", PATHS)
@pytest.mark.parametrize("T", [1, 4, 32, 64])
def test_route_forward_equals_route_then_forward(tiny, path, T):
    """The one-call entry point (fused routing/sort/quantisation for small
    batches) gives the same bytes as the two calls."""
    cfg, w, layer = tiny
    bqe.moe_set_gemm_path(layer, path)
    tk = G.tokens(0, n=T)
    ids, wd = G.route_dev(layer, tk.logits, cfg.k)
    a = G.forward_dev(layer, tk.x_bits, ids, wd).cpu().numpy()
    ids2 = torch.empty_like(ids)
    w2 = torch.empty_like(wd)
    out2 = torch.empty((T, cfg.H), dtype=torch.float32, device=G.DEV)
    bqe.moe_route_forward(layer, G.to_dev(tk.logits), G.to_dev(tk.x_bits, torch.int16), ids2, w2, out2)
    bqe.moe_check(layer)
    assert torch.equal(ids, ids2) and torch.equal(wd, w2)
    assert out2.cpu().numpy().tobytes() == a.tobytes()


def test_argument_errors(tiny):
    cfg, w, layer = tiny
    lib = bqe.load_library()
    s = torch.cuda.current_stream().cuda_stream
    ids = torch.zeros((4, cfg.k), dtype=torch.int32, device=G.DEV)
    wd = torch.zeros((4, cfg.k), dtype=torch.float32, device=G.DEV)
    assert lib.moe_route(layer.ptr, None, 4, ids.data_ptr(), wd.data_ptr(), s) == bqe.MOE_ERR_INVALID_ARG
    lg = torch.zeros((600, cfg.E), dtype=torch.float32, device=G.DEV)
    i6 = torch.zeros((600, cfg.k), dtype=torch.int32, device=G.DEV)
    w6 = torch.zeros((600, cfg.k), dtype=torch.float32, device=G.DEV)
    with pytest.raises(bqe.MoeError):
        bqe.moe_route(layer, lg, i6, w6)              # T > max_tokens
    assert lib.moe_forward(layer.ptr, None, 0, None, None, None, s) == bqe.MOE_ERR_INVALID_ARG
    assert "NULL" in bqe.moe_last_error(layer) or "outside" in bqe.moe_last_error(layer)
    # ids out of range are skipped on the device and reported by moe_check
    bad = torch.tensor([[0, 99]], dtype=torch.int32, device=G.DEV)
    off = torch.empty(cfg.E + 1, dtype=torch.int32, device=G.DEV)
    src = torch.empty(2, dtype=torch.int32, device=G.DEV)
    dst = torch.empty(2, dtype=torch.int32, device=G.DEV)
    bqe.moe_permute(layer, bad, off, src, dst)
    with pytest.raises(bqe.MoeError) as ei:
        bqe.moe_check(layer)
    assert ei.value.status == bqe.MOE_ERR_INVALID_ARG
    assert dst.cpu().tolist()[1] == -1
    bqe.moe_check(layer)                              # flag was cleared
    cfgp = bqe.moe_config(100, 128, 16, 2, 4, 0, 1.5)
    out = C.c_void_p()
    assert lib.moe_create(C.byref(cfgp), None, None, C.byref(out)) == bqe.MOE_ERR_INVALID_ARG
