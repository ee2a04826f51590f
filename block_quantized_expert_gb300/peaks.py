"""Measured roofline denominators of the layer's kernels (libmoe_peaks.so).

* hbm_read_gbs(): a plain 16-byte-load read stream over a buffer larger
  than L2 -- the bound of the weight-streaming kernels (decode, pp512).
* mma_mx_tflops(): block-scaled tcgen05 MMAs of the shape the grouped GEMMs
  issue (kind::mxf8f6f4, M 128, N 256, K 32, e4m3 x e2m1, UE8M0 / 32), one
  issuing thread per SM on resident operands -- the bound of prefill.
* dot_e2m1_el_per_clk(): the CUDA-core decode kernel's block dot products
  (e2m1 codes -> f16 by the hardware converter, times f16 operands, fp32
  sums) in elements per SM clock -- its arithmetic ceiling.

Both run on the current CUDA device and return figures from CUDA events.
``python -m block_quantized_expert_gb300.peaks [--out FILE]`` prints (and
writes) one JSON record with the SM clocks sampled while they ran.
"""
from __future__ import annotations

import ctypes as C
import json

from . import _build

_lib = None


def load(build: bool = True):
    global _lib
    if _lib is None:
        path = _build.build_peaks() if build else _build.PEAKS_LIB
        L = C.CDLL(str(path))
        L.peak_read_stream.argtypes = [C.c_void_p, C.c_longlong, C.c_int, C.c_void_p, C.POINTER(C.c_float)]
        L.peak_mma_mx.argtypes = [C.c_int, C.c_int, C.c_void_p, C.POINTER(C.c_float)]
        L.peak_dot_e2m1.argtypes = [C.c_int, C.c_int, C.c_void_p, C.c_void_p, C.c_void_p, C.POINTER(C.c_float)]
        _lib = L
    return _lib


def hbm_read_gbs(nbytes: int = 4 << 30, reps: int = 5) -> float:
    """Best of `reps` reads of an `nbytes` device buffer, in GB/s (1e9 B/s)."""
    import torch

    sms = torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count
    buf = torch.empty(nbytes // 16 * 16, dtype=torch.uint8, device="cuda")
    buf.fill_(1)
    sink = torch.zeros(1, dtype=torch.int32, device="cuda")
    torch.cuda.synchronize()
    best = 0.0
    for _ in range(reps + 1):  # the first is a warm-up
        ms = C.c_float(0.0)
        rc = load().peak_read_stream(buf.data_ptr(), buf.numel(), 4 * sms, sink.data_ptr(), C.byref(ms))
        if rc:
            raise RuntimeError(f"peak_read_stream failed ({rc})")
        best = max(best, buf.numel() / (ms.value * 1e-3) / 1e9)
    del buf
    return best


def mma_mx_tflops(iters: int = 200000, reps: int = 3) -> float:
    """Best of `reps` runs of the block-scaled MMA loop on every SM, in TFLOP/s."""
    import torch

    sms = torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count
    ok = torch.ones(1, dtype=torch.int32, device="cuda")
    best = 0.0
    load().peak_mma_mx(sms, 1000, ok.data_ptr(), C.byref(C.c_float(0.0)))  # warm-up
    for _ in range(reps):
        ms = C.c_float(0.0)
        rc = load().peak_mma_mx(sms, iters, ok.data_ptr(), C.byref(ms))
        if rc or int(ok.item()) != 1:
            raise RuntimeError(f"peak_mma_mx failed ({rc}, ok={int(ok.item())})")
        flops = sms * iters * 4 * 2.0 * 128 * 256 * 32
        best = max(best, flops / (ms.value * 1e-3) / 1e12)
    return best


def dot_e2m1_el_per_clk(iters: int = 4096, reps: int = 3) -> float:
    """Elements per SM clock of the decode kernel's e2m1 x f16 -> fp32 block
    dot products on the CUDA cores (one CTA of 16 warps per SM, operands in
    shared memory), the median CTA of the best of `reps` runs."""
    import torch

    sms = torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count
    g = torch.Generator().manual_seed(12345)
    seed = torch.randint(0, 2 ** 31 - 1, (1024,), generator=g, dtype=torch.int64).to(torch.int32).cuda()
    out = torch.empty(sms * 512, dtype=torch.float32, device="cuda")
    cyc = torch.zeros(sms, dtype=torch.int64, device="cuda")
    best = 0.0
    for r in range(reps + 1):  # the first is a warm-up
        ms = C.c_float(0.0)
        rc = load().peak_dot_e2m1(sms, iters if r else 64, seed.data_ptr(), out.data_ptr(), cyc.data_ptr(),
                                  C.byref(ms))
        if rc:
            raise RuntimeError(f"peak_dot_e2m1 failed ({rc})")
        if r:
            c = float(cyc.cpu().median().item())
            best = max(best, iters * 16 * 4 * 1024 / c)
    return best


def main():
    import argparse
    import subprocess
    import tempfile

    import torch

    ap = argparse.ArgumentParser()
    ap.add_argument("--out", default=None)
    args = ap.parse_args()
    dev = torch.cuda.current_device()
    props = torch.cuda.get_device_properties(dev)
    f = tempfile.NamedTemporaryFile("w+", suffix=".csv")
    smi = subprocess.Popen(["nvidia-smi", "-i", str(dev), "--query-gpu=clocks.sm,clocks.max.sm,power.draw",
                            "--format=csv,noheader,nounits", "-lms", "100"], stdout=f,
                           stderr=subprocess.DEVNULL)
    rec = {"gpu": props.name, "sms": props.multi_processor_count,
           "hbm_read_gbs": round(hbm_read_gbs(), 1),
           "mma_mxf8f6f4_tflops": round(mma_mx_tflops(), 1),
           "mma_shape": "kind::mxf8f6f4 block_scale scale_vec::1X, M128 N256 K32, e4m3 x e2m1",
           "dot_e2m1_el_per_clk_per_sm": round(dot_e2m1_el_per_clk(), 1),
           "dot_e2m1": "cvt.rn.f16x2.e2m1x2 + fma.rn.f32.f16, 16 warps x 4 32-blocks per iteration, operands in shared memory",
           "read_stream": "16-byte evict-first loads, 4 GiB, grid 4 x SMs x 512 threads, best of 5"}
    smi.terminate()
    smi.wait()
    f.seek(0)
    sm = []
    for line in f.read().splitlines():
        parts = [p.strip() for p in line.split(",")]
        if len(parts) == 3 and parts[0].replace(".", "").isdigit():
            sm.append(float(parts[0]))
    rec["sm_mhz_samples"] = sm
    rec["sm_mhz_max_seen"] = max(sm) if sm else None
    print(json.dumps(rec))
    if args.out:
        with open(args.out, "w") as fo:
            json.dump(rec, fo, indent=1)


if __name__ == "__main__":
    main()
