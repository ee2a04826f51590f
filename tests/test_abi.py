"""CPU checks of the C ABI boundary: libmoe.so builds, loads without a GPU and
exports every entry point include/moe.h declares; host-side validation and
workspace sizing need no device."""
import ctypes as C
import os
import re

import block_quantized_expert_gb300 as bqe

HEADER = os.path.join(os.path.dirname(os.path.dirname(__file__)), "include", "moe.h")


def declared_symbols():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_[a-z_]+)\s*\(", text)))


def test_library_exports_every_declared_symbol():
    lib = bqe.load_library()
    names = declared_symbols()
    assert len(names) >= 13
    for n in names:
        assert hasattr(lib, n), n
    assert sorted(bqe.EXPORTS) == names


def test_workspace_and_config_validation_on_host():
    lib = bqe.load_library()
    good = bqe.MoeConfig(4096, 2048, 256, 6, 8192, True)
    n = bqe.moe_workspace_bytes(good)
    # dominated by the fp32 down outputs of every routed row: T*k*H*4
    assert n > 8192 * 6 * 4096 * 4
    for bad in (bqe.MoeConfig(4000, 2048, 256, 6, 1), bqe.MoeConfig(4096, 2048, 256, 9, 1),
                bqe.MoeConfig(4096, 2048, 0, 1, 1), bqe.MoeConfig(4096, 2048, 4, 6, 1),
                bqe.MoeConfig(4096, 2048, 256, 6, 0), bqe.MoeConfig(16384, 2048, 256, 6, 1)):
        assert bqe.moe_workspace_bytes(bad) == 0
        out = C.c_void_p()
        st = lib.moe_create(C.byref(bad.c()), None, None, C.byref(out))
        assert st == bqe.MOE_ERR_INVALID_ARG and out.value is None
        assert bqe.moe_last_error(None)
    # NULL layer is rejected before any CUDA call
    assert lib.moe_route(None, None, 1, None, None, None) == bqe.MOE_ERR_INVALID_ARG
    assert lib.moe_destroy(None) == bqe.MOE_OK


def test_peaks_library_exports_its_header():
    """libmoe_peaks.so (the roofline denominators) builds and exports what
    include/moe_peaks.h declares."""
    from block_quantized_expert_gb300 import peaks

    text = open(os.path.join(os.path.dirname(HEADER), "moe_peaks.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = sorted(set(re.findall(r"\b(peak_[a-z_]+)\s*\(", text)))
    assert names == ["peak_mma_mx", "peak_read_stream"]
    lib = peaks.load()
    for n in names:
        assert hasattr(lib, n), n
