"""The diagnostic entry points of the C ABI: stage events
(moe_set_stage_events) and the kernel trace (moe_set_trace).

- Stage events: a count other than 6 is refused by the library; with 6
  events the next moe_forward records all of them on its stream, in stage
  order (every interval non-negative).
- Trace: a buffer below the documented size (the larger of the GEMMs' and
  front kernel's counters and the CUDA-core decode kernel's stamps and event
  times) is refused; the decode kernel stamps every CTA's entry, first copy
  and final barrier in that order; a batch writes the front kernel's
  [entry, wait end, exit] and the tensor-core GEMMs' per-CTA entry and exit.
  The setting is one-shot: the call after it writes nothing.

The outputs of the traced calls are checked against untraced ones: tracing
changes no result."""
import ctypes as C
import dataclasses

import numpy as np
import pytest
import torch

import block_quantized_expert_gb300 as bqe
from tests import _gpu as G
from workloads import CONFIGS, make_tokens, make_weights

pytestmark = pytest.mark.gpu

T_BATCH = 8  # front kernel + tensor-core GEMMs + the combine kernel


@pytest.fixture(scope="module")
def diag():
    cfg = dataclasses.replace(CONFIGS[1], index=90, name="diag_2048x1024x16k4", H=2048, I=1024, E=16, k=4,
                              T=T_BATCH, steps=1)
    w = make_weights(cfg, seed=2300, cache=False)
    layer = G.make_layer(cfg, w, max_tokens=T_BATCH)
    tk = make_tokens(cfg, n=T_BATCH)
    yield cfg, layer, tk
    layer.close()
    torch.cuda.empty_cache()


def _need(sms):
    return max(48 * sms + 4, 8 * sms + 1024)


def _route_forward(cfg, layer, tk, T):
    lg = G.to_dev(tk.logits[:T].astype(np.float32))
    x = G.to_dev(tk.x_bits[:T].astype(np.uint16), torch.int16)
    ids = torch.empty((T, cfg.k), dtype=torch.int32, device=G.DEV)
    w = torch.empty((T, cfg.k), dtype=torch.float32, device=G.DEV)
    out = torch.empty((T, cfg.H), dtype=torch.float32, device=G.DEV)
    bqe.moe_route_forward(layer, lg, x, ids, w, out)
    bqe.moe_check(layer)
    return ids, w, out


def test_stage_events_recorded_in_order(diag):
    cfg, layer, tk = diag
    lib = bqe.load_library()
    arr = (C.c_void_p * 6)()
    assert lib.moe_set_stage_events(layer.ptr, arr, 5) == bqe.MOE_ERR_INVALID_ARG
    ids, w, _ = _route_forward(cfg, layer, tk, T_BATCH)
    x = G.to_dev(tk.x_bits[:T_BATCH].astype(np.uint16), torch.int16)
    ref = G.forward_dev(layer, tk.x_bits[:T_BATCH], ids, w)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(6)]
    bqe.moe_set_stage_events(layer, ev)
    out = torch.empty((T_BATCH, cfg.H), dtype=torch.float32, device=G.DEV)
    bqe.moe_forward(layer, x, ids, w, out)
    bqe.moe_check(layer)
    torch.cuda.synchronize()
    gaps = [ev[i].elapsed_time(ev[i + 1]) for i in range(5)]
    assert all(g >= 0.0 for g in gaps), gaps
    assert ev[0].elapsed_time(ev[5]) > 0.0
    assert torch.equal(out, ref)


def test_trace_refuses_a_short_buffer(diag):
    _, layer, _ = diag
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    short = torch.zeros(_need(sms) - 1, dtype=torch.int64, device=G.DEV)
    with pytest.raises(bqe.MoeError) as ei:
        bqe.moe_set_trace(layer, short)
    assert ei.value.status == bqe.MOE_ERR_INVALID_ARG


def test_trace_of_the_decode_kernel(diag):
    cfg, layer, tk = diag
    assert bqe.moe_decode_info(layer) == 1
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    _, _, ref = _route_forward(cfg, layer, tk, 1)
    buf = torch.zeros(_need(sms), dtype=torch.int64, device=G.DEV)
    bqe.moe_set_trace(layer, buf)
    _, _, out = _route_forward(cfg, layer, tk, 1)
    assert torch.equal(out, ref)
    st = buf.cpu().numpy()[: 8 * sms].reshape(sms, 8).astype(np.uint64)
    entry, first_copy, done = st[:, 0], st[:, 4], st[:, 5]
    assert (entry > 0).all()
    assert (first_copy >= entry).all() and (done >= first_copy).all()
    # one-shot: the next call writes nothing
    buf.zero_()
    _route_forward(cfg, layer, tk, 1)
    torch.cuda.synchronize()
    assert int(buf.count_nonzero()) == 0


def test_trace_of_a_batch(diag):
    cfg, layer, tk = diag
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    _, _, ref = _route_forward(cfg, layer, tk, T_BATCH)
    buf = torch.zeros(_need(sms), dtype=torch.int64, device=G.DEV)
    bqe.moe_set_trace(layer, buf)
    _, _, out = _route_forward(cfg, layer, tk, T_BATCH)
    assert torch.equal(out, ref)
    tr = buf.cpu().numpy().astype(np.uint64)
    front = tr[4 * sms * 12: 4 * sms * 12 + 3]
    assert front[0] > 0 and front[1] >= front[0] and front[2] >= front[1]
    for j in (0, 1):  # gate/up, down
        ctr = tr[j * sms * 12: (j + 1) * sms * 12].reshape(sms, 12)
        ran = ctr[:, 0] > 0
        assert ran.any(), j
        assert (ctr[ran, 1] >= ctr[ran, 0]).all(), j
