"""Single-tile GPU checks of the tcgen05 building blocks (tests/csrc/tc_probe.cu):
the 4-bit TMA unpacking (transaction size, shared-memory image) and one
block-scaled MMA against exact numpy arithmetic.  A failure here localises
a fault of the grouped GEMM kernels to a descriptor or a layout."""
import ctypes as C
import os
import subprocess

import numpy as np
import pytest
import torch

from tests import _brute

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
SRC = os.path.join(HERE, "csrc", "tc_probe.cu")
LIB = os.path.join(HERE, "_build", "libtcprobe.so")


@pytest.fixture(scope="module")
def probe():
    os.makedirs(os.path.dirname(LIB), exist_ok=True)
    subprocess.run(["/usr/local/cuda/bin/nvcc", "-gencode", "arch=compute_103a,code=sm_103a", "-O2",
                    "-std=c++17", "-Xcompiler", "-fPIC", "-shared",
                    "-I", os.path.join(ROOT, "block_quantized_expert_gb300", "csrc"), "-o", LIB, SRC],
                   check=True)
    lib = C.CDLL(LIB)
    vp = C.c_void_p
    lib.probe_tma4.argtypes = [vp, vp, vp]
    lib.probe_mma.argtypes = [vp, vp, vp, vp, C.c_int, C.c_uint32, C.c_uint32, vp, vp, vp]
    return lib


def _unswizzle(img: np.ndarray) -> np.ndarray:
    """[rows][128] image written with the 128-byte swizzle -> logical rows."""
    out = np.empty_like(img)
    for r in range(img.shape[0]):
        for c in range(8):
            out[r, 16 * c:16 * c + 16] = img[r, 16 * (c ^ (r % 8)):16 * (c ^ (r % 8)) + 16]
    return out


def test_tma_fp4_unpack(probe):
    rng = np.random.default_rng(0)
    a = rng.integers(0, 256, size=(128, 64), dtype=np.uint8)
    da = torch.from_numpy(a).cuda()
    dump = torch.zeros(16384, dtype=torch.uint8, device="cuda")
    flags = torch.zeros(2, dtype=torch.int32, device="cuda")
    rc = probe.probe_tma4(da.data_ptr(), dump.data_ptr(), flags.data_ptr())
    assert rc == 0
    img = _unswizzle(dump.cpu().numpy().reshape(128, 128))
    data = img.reshape(128, 8, 16)[:, :, :8].reshape(128, 64)
    # the copy completes a barrier armed with the 8192 packed bytes of the
    # tile and writes each 8-byte group of codes into the low half of a
    # 16-byte slot, leaving the other half as it was
    assert flags.cpu().tolist()[0] == 1, "a 128x128 fp4 tile should count 8192 transaction bytes"
    assert np.array_equal(data, a)
    assert (img.reshape(128, 8, 16)[:, :, 8:] == 0xEE).all()


def _atom(exps: np.ndarray) -> np.ndarray:
    """exps [rows<=128][4] -> 512-byte atom (row r, block kb at (r%32)*16+(r//32)*4+kb)."""
    at = np.full(512, 127, np.uint8)
    for r in range(exps.shape[0]):
        for kb in range(4):
            at[(r % 32) * 16 + (r // 32) * 4 + kb] = exps[r, kb]
    return at


@pytest.mark.parametrize("a_fmt", [5, 0])
def test_block_scaled_mma_tile(probe, a_fmt):
    rng = np.random.default_rng(1 + a_fmt)
    e4 = _brute.e4m3_table()
    finite = np.array([c for c in range(256) if c not in (0x7F, 0xFF) and abs(e4[c]) <= 16], np.uint8)
    if a_fmt == 5:
        codes = rng.integers(0, 16, size=(128, 128), dtype=np.uint8)
        a_bytes = (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8)
        a_val = _brute.e2m1_table()[codes]
        a_tx = 8192
    else:
        codes = rng.choice(finite, size=(128, 128))
        a_bytes = codes
        a_val = e4[codes]
        a_tx = 16384
    b_codes = rng.choice(finite, size=(32, 128))
    b_val = e4[b_codes]
    sa = rng.integers(120, 134, size=(128, 4)).astype(np.uint8)
    sb = rng.integers(120, 134, size=(32, 4)).astype(np.uint8)
    A = a_val * np.ldexp(1.0, sa.astype(int) - 127).repeat(32, 1)
    Bm = b_val * np.ldexp(1.0, sb.astype(int) - 127).repeat(32, 1)
    want = A @ Bm.T
    d_a = torch.from_numpy(np.ascontiguousarray(a_bytes)).cuda()
    d_b = torch.from_numpy(np.ascontiguousarray(b_codes)).cuda()
    d_sa = torch.from_numpy(_atom(sa)).cuda()
    d_sb = torch.from_numpy(_atom(sb)).cuda()
    d = torch.zeros((128, 32), dtype=torch.float32, device="cuda")
    sf = torch.zeros((128, 8), dtype=torch.int32, device="cuda")
    flags = torch.zeros(2, dtype=torch.int32, device="cuda")
    rc = probe.probe_mma(d_a.data_ptr(), d_b.data_ptr(), d_sa.data_ptr(), d_sb.data_ptr(), 0, a_tx, a_fmt,
                         d.data_ptr(), sf.data_ptr(), flags.data_ptr())
    assert rc == 0
    assert flags.cpu().tolist() == [1, 1]
    got = d.cpu().numpy().astype(np.float64)
    err = np.abs(got - want).max() / np.abs(want).max()
    print("a_fmt", a_fmt, "max rel err", err)
    if err >= 1e-5:  # diagnostics: per-row-quarter error, ratios, the copied scale columns
        rows = np.abs(got - want).max(1) / np.abs(want).max()
        print("row-quarter max err:", [float(rows[32 * q:32 * q + 32].max()) for q in range(4)])
        print("got/want row 0:", np.round(got[0, :8] / want[0, :8], 4))
        print("got/want row 40:", np.round(got[40, :8] / want[40, :8], 4))
        sfd = sf.cpu().numpy().view(np.uint8).reshape(128, 8, 4)
        print("tmem sf cols 128..135, lanes 0,1,33:", sfd[0].tolist(), sfd[1].tolist(), sfd[33].tolist())
        print("sa rows 0,1,32,33:", sa[[0, 1, 32, 33]].tolist(), " sb rows 0,1:", sb[[0, 1]].tolist())
    assert err < 1e-5
