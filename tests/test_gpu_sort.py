"""The token -> expert counting sort at the sizes where it runs over one CTA
per 1024-row chunk (more than 8192 rows), against the oracle: ragged last
chunks, empty experts, empty slots (id -1) and an out-of-range id."""
import numpy as np
import pytest
import torch

import block_quantized_expert_gb300 as bqe
from oracle import oracle as orc

pytestmark = pytest.mark.gpu

E, K = 256, 6


@pytest.fixture(scope="module")
def layer():
    H, I = 256, 128
    dev = "cuda:0"
    w = {"gate_q": torch.zeros((E, I, H // 2), dtype=torch.uint8, device=dev),
         "gate_s": torch.full((E, I, H // 32), 127, dtype=torch.uint8, device=dev),
         "up_q": torch.zeros((E, I, H // 2), dtype=torch.uint8, device=dev),
         "up_s": torch.full((E, I, H // 32), 127, dtype=torch.uint8, device=dev),
         "down_q": torch.zeros((E, H, I // 2), dtype=torch.uint8, device=dev),
         "down_s": torch.full((E, H, I // 32), 127, dtype=torch.uint8, device=dev)}
    L = bqe.moe_create(bqe.MoeConfig(H, I, E, K, 4096), w)
    yield L
    L.close()


def _sort(layer, ids_np):
    T = ids_np.shape[0]
    ids = torch.from_numpy(ids_np).cuda()
    off = torch.full((E + 1,), -7, dtype=torch.int32, device="cuda")
    src = torch.full((T * K,), -7, dtype=torch.int32, device="cuda")
    dst = torch.full((T * K,), -7, dtype=torch.int32, device="cuda")
    bqe.moe_permute(layer, ids, off, src, dst)
    return off.cpu().numpy(), src.cpu().numpy(), dst.cpu().numpy()


@pytest.mark.parametrize("T,seed", [(1366, 0), (1400, 1), (2731, 2), (4096, 3)])
def test_grid_sort_matches_oracle(layer, T, seed):
    rng = np.random.default_rng(seed)
    # a skewed expert distribution (many empty experts, one large segment)
    # with some empty slots
    ids = np.minimum(rng.zipf(1.3, size=(T, K)) - 1, E - 1).astype(np.int32)
    ids[rng.random((T, K)) < 0.05] = -1
    off, src, dst = _sort(layer, ids)
    bqe.moe_check(layer)
    ro, rs, rd = orc.permute(ids, E)
    n = int(ro[-1])
    assert np.array_equal(off, ro)
    assert np.array_equal(src[:n], rs[:n])
    assert np.array_equal(dst, rd)


def test_grid_sort_flags_out_of_range_id(layer):
    T = 1400
    ids = np.random.default_rng(4).integers(0, E, size=(T, K)).astype(np.int32)
    ids[700, 3] = E  # out of range: left out and reported
    off, src, dst = _sort(layer, ids)
    with pytest.raises(bqe.MoeError) as ei:
        bqe.moe_check(layer)
    assert ei.value.status == bqe.MOE_ERR_INVALID_ARG
    assert dst[700 * K + 3] == -1
    ok = ids.copy()
    ok[700, 3] = -1  # the same sort with the row as an empty slot
    ro, rs, rd = orc.permute(ok, E)
    assert np.array_equal(off, ro) and np.array_equal(dst, rd)
    bqe.moe_check(layer)
