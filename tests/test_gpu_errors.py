"""Failure paths through the C ABI that need a device but fault nothing: a
workspace larger than the GPU's memory fails cleanly (MOE_ERR_OOM, every
partial allocation released, the device still usable)."""
import pytest
import torch

import block_quantized_expert_gb300 as bqe

pytestmark = pytest.mark.gpu


def _weights(H, I, E):
    dev = "cuda:0"
    return {"gate_q": torch.zeros((E, I, H // 2), dtype=torch.uint8, device=dev),
            "gate_s": torch.full((E, I, H // 32), 127, dtype=torch.uint8, device=dev),
            "up_q": torch.zeros((E, I, H // 2), dtype=torch.uint8, device=dev),
            "up_s": torch.full((E, I, H // 32), 127, dtype=torch.uint8, device=dev),
            "down_q": torch.zeros((E, H, I // 2), dtype=torch.uint8, device=dev),
            "down_s": torch.full((E, H, I // 32), 127, dtype=torch.uint8, device=dev)}


def test_workspace_larger_than_the_device_fails_cleanly():
    H, I, E, k = 4096, 128, 16, 2
    w = _weights(H, I, E)
    torch.cuda.synchronize()
    free0, total = torch.cuda.mem_get_info()
    # y alone would be max_tokens * k * H * 4 bytes = 2^24 * 2 * 4096 * 4 > the device
    max_tokens = 1 << 24
    assert max_tokens * k * H * 4 > total
    with pytest.raises(bqe.MoeError) as ei:
        bqe.moe_create(bqe.MoeConfig(H, I, E, k, max_tokens), w)
    assert ei.value.status == bqe.MOE_ERR_OOM
    assert "allocation" in str(ei.value)
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert free1 >= free0 - (64 << 20)  # what was allocated before the failure is released
    layer = bqe.moe_create(bqe.MoeConfig(H, I, E, k, 64), w)  # the device is still usable
    layer.close()
