"""The allocation-free grouping entry point (moe_permute_noalloc), called
through the C ABI, gives the same permutation as moe_permute on a layer.

moe_permute_noalloc serves callers that cannot call cudaMalloc (a framework
arena that forbids foreign allocations, a serving loop with frozen device
memory, an engine that only wants the grouping): its scratch is a static
device array, so it needs neither a layer nor an allocation.  This file is
collected last on purpose; it builds its own small layer and runs the same in
a fresh process or after the other tests.
"""
import ctypes as C

import numpy as np
import pytest
import torch

import block_quantized_expert_gb300 as bqe
from oracle import oracle as orc
from workloads import CONFIGS, make_tokens

pytestmark = pytest.mark.gpu


def _small_layer(E, k, max_tokens):
    H, I = 256, 128
    dev = "cuda:0"
    w = {"gate_q": torch.zeros((E, I, H // 2), dtype=torch.uint8, device=dev),
         "gate_s": torch.full((E, I, H // 32), 127, dtype=torch.uint8, device=dev),
         "up_q": torch.zeros((E, I, H // 2), dtype=torch.uint8, device=dev),
         "up_s": torch.full((E, I, H // 32), 127, dtype=torch.uint8, device=dev),
         "down_q": torch.zeros((E, H, I // 2), dtype=torch.uint8, device=dev),
         "down_s": torch.full((E, H, I // 32), 127, dtype=torch.uint8, device=dev)}
    return bqe.moe_create(bqe.MoeConfig(H, I, E, k, max_tokens), w)


def _run_both(lib, layer, ids, E):
    T, k = ids.shape
    R = T * k
    outs = []
    for use_static in (False, True):
        off = torch.full((E + 1,), -7, dtype=torch.int32, device="cuda")
        src = torch.full((R,), -7, dtype=torch.int32, device="cuda")
        dst = torch.full((R,), -7, dtype=torch.int32, device="cuda")
        s = torch.cuda.current_stream().cuda_stream
        if use_static:
            st = lib.moe_permute_noalloc(ids.data_ptr(), T, k, E, off.data_ptr(), src.data_ptr(),
                                         dst.data_ptr(), s)
        else:
            st = lib.moe_permute(layer.ptr, ids.data_ptr(), T, off.data_ptr(), src.data_ptr(),
                                 dst.data_ptr(), s)
        assert st == bqe.MOE_OK, bqe.moe_last_error(None if use_static else layer)
        torch.cuda.synchronize()
        outs.append((off.cpu().numpy(), src.cpu().numpy(), dst.cpu().numpy()))
    return outs


def test_noalloc_permute_matches_layer_permute_twice():
    lib = bqe.load_library()
    E, k = 256, 6
    layer = _small_layer(E, k, 8192)
    # two calls in a row with different routings: the prefill-8192 (Zipf
    # skewed: many empty experts, one huge segment) and pp512 rows
    for cid, n in ((4, 8192), (3, 512)):
        logits = make_tokens(CONFIGS[cid], n=n).logits
        ids_np, _ = orc.route_learned(logits, k)
        ids = torch.from_numpy(ids_np).cuda()
        (o1, s1, d1), (o2, s2, d2) = _run_both(lib, layer, ids, E)
        assert np.array_equal(o1, o2) and np.array_equal(s1, s2) and np.array_equal(d1, d2)
        ro, rs, rd = orc.permute(ids_np, E)
        assert np.array_equal(o2, ro) and np.array_equal(s2, rs) and np.array_equal(d2, rd)
    layer.close()


def test_noalloc_permute_rejects_sizes_beyond_its_scratch():
    lib = bqe.load_library()
    ids = torch.zeros((10923, 6), dtype=torch.int32, device="cuda")   # 65538 rows > 65536
    off = torch.empty(257, dtype=torch.int32, device="cuda")
    src = torch.empty(10923 * 6, dtype=torch.int32, device="cuda")
    st = lib.moe_permute_noalloc(ids.data_ptr(), 10923, 6, 256, off.data_ptr(), src.data_ptr(),
                                 src.data_ptr(), None)
    assert st == bqe.MOE_ERR_INVALID_ARG
    assert "65536" in bqe.moe_last_error(None)
    st = lib.moe_permute_noalloc(None, 1, 6, 256, off.data_ptr(), src.data_ptr(), src.data_ptr(), None)
    assert st == bqe.MOE_ERR_INVALID_ARG
