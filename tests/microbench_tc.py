#!/usr/bin/env python
"""Microbenchmarks of the sm_103a building blocks (tests/csrc/tc_probe.cu):
a plain HBM read stream, the block-scaled MMA issue rate, and TMA weight
streaming with and without MMAs.  Prints one line per case and writes all
results as JSON (default tests/_build/microbench_tc.json).  Timing only.

    python tests/microbench_tc.py [--out PATH]
"""
import argparse
import ctypes as C
import json
import os
import subprocess

import torch

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)


def load():
    lib_path = os.path.join(HERE, "_build", "libtcprobe.so")
    os.makedirs(os.path.dirname(lib_path), exist_ok=True)
    subprocess.run(["/usr/local/cuda/bin/nvcc", "-gencode", "arch=compute_103a,code=sm_103a", "-O2",
                    "-std=c++17", "-Xcompiler", "-fPIC", "-shared",
                    "-I", os.path.join(ROOT, "block_quantized_expert_gb300", "csrc"),
                    "-o", lib_path, os.path.join(HERE, "csrc", "tc_probe.cu")], check=True)
    lib = C.CDLL(lib_path)
    vp = C.c_void_p
    lib.probe_read.argtypes = [vp, C.c_longlong, C.c_int, C.c_int, vp, vp]
    lib.probe_stream.argtypes = [vp, C.c_longlong, C.c_int, C.c_int, C.c_int, C.c_int, C.c_int, vp, vp,
                                 vp, C.c_int]
    lib.probe_stream_lsu.argtypes = [vp, C.c_longlong, C.c_int, C.c_int, C.c_int, vp, vp, vp]
    lib.probe_mma_peak.argtypes = [C.c_int, C.c_int, C.c_int, C.c_uint32, vp, vp]
    lib.probe_contend.argtypes = [C.c_int, C.c_int, C.c_int, vp, vp, vp]
    lib.probe_stream_ldg.argtypes = [vp, C.c_longlong, vp, C.c_longlong, C.c_int, C.c_int, C.c_int, C.c_int, vp, vp]
    lib.probe_stream_indep.argtypes = [vp, C.c_longlong, C.c_int, C.c_int, C.c_int, C.c_int, vp, vp, vp]
    lib.probe_prim.argtypes = [C.c_int, C.c_int, C.c_int, vp]
    lib.probe_mma_mix.argtypes = [C.c_int, C.c_int, C.c_int, C.c_int, C.c_int, C.c_int, C.c_uint32, C.c_int,
                                  vp, vp]
    return lib


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--out", default=os.path.join(HERE, "_build", "microbench_tc.json"))
    ap.add_argument("--only-mix", action="store_true", help="only the per-stage MMA group issue costs")
    ap.add_argument("--only-stream", action="store_true", help="only the 256-row weight-box TMA streams")
    ap.add_argument("--only-ldg", action="store_true",
                    help="weight stream copied by the load/store units instead of the TMA, with / without MMAs")
    ap.add_argument("--only-pf", action="store_true",
                    help="the 256-row weight-box stream with MMAs and an L2 prefetch running ahead of the ring")
    ap.add_argument("--only-prim", action="store_true",
                    help="cycles per mbarrier wait on a completed phase and per %%globaltimer read")
    ap.add_argument("--only-indep", action="store_true",
                    help="TMA stream and an independent MMA loop, alone and side by side")
    ap.add_argument("--only-contend", action="store_true",
                    help="MMA loop time with shared-memory stores / loads by other warps")
    args = ap.parse_args()
    lib = load()
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    ms = C.c_float()
    ok = torch.ones(1, dtype=torch.int32, device="cuda")
    out = {"sms": sms}
    if args.only_ldg:
        tiles = 8
        W = torch.zeros(sms * tiles * 256 * 2048, dtype=torch.uint8, device="cuda")
        SF = torch.full((sms * tiles * 32 * 1024,), 127, dtype=torch.uint8, device="cuda")
        for stages, mode in ((6, 0), (4, 1), (6, 2), (6, 3), (4, 3), (4, 2)):
            for _ in range(2):
                ok.fill_(1)
                rc = lib.probe_stream_ldg(W.data_ptr(), W.numel(), SF.data_ptr(), SF.numel(), sms, tiles, stages,
                                          mode, ok.data_ptr(), C.byref(ms))
            key = f"ldg_stages{stages}_mode{mode}"
            out[key] = {"GBs": round(sms * tiles * 32 * (16384 + 1024) / ms.value / 1e6, 1),
                        "us_per_stage": round(ms.value * 1e3 / (tiles * 32), 3), "rc": rc, "ok": int(ok.item())}
            print(key, out[key], flush=True)
        os.makedirs(os.path.dirname(args.out), exist_ok=True)
        json.dump(out, open(args.out, "w"), indent=1)
        return
    if args.only_prim:
        iters = 4096
        res = torch.zeros(4 * sms, dtype=torch.int64, device="cuda")
        for park in (0, 2, 4, 3, 1):
            for _ in range(2):
                res.zero_()
                rc = lib.probe_prim(sms, iters, park, res.data_ptr())
            r = res.view(sms, 4).double().median(dim=0).values / iters
            key = f"prim_cycles_park{park}"
            out[key] = {"try_wait_completed": round(r[0].item(), 1), "test_wait_completed": round(r[1].item(), 1),
                        "globaltimer_read": round(r[2].item(), 1), "arrive_then_try_wait": round(r[3].item(), 1),
                        "rc": rc}
            print(key, out[key], flush=True)
        os.makedirs(os.path.dirname(args.out), exist_ok=True)
        json.dump(out, open(args.out, "w"), indent=1)
        return
    if args.only_indep:
        tiles, groups = 8, 224
        W = torch.zeros(sms * tiles * 256 * 2048, dtype=torch.uint8, device="cuda")
        times = torch.zeros(4 * sms, dtype=torch.int64, device="cuda")
        for which in (1, 2, 3, 1, 2, 3, 6, 7):
            times.zero_()
            ok.fill_(1)
            rc = lib.probe_stream_indep(W.data_ptr(), W.numel() // 2048, sms, tiles, groups, which,
                                        times.data_ptr(), ok.data_ptr(), C.byref(ms))
            t = times.view(sms, 4).cpu().double()
            rec = {"rc": rc, "ok": int(ok.item()), "kernel_ms": round(ms.value, 4)}
            if which & 1:
                d = (t[:, 1] - t[:, 0]) / 1e3
                rec["stream_us_per_stage_median"] = round(d.median().item() / (tiles * 32), 4)
                rec["stream_us_per_stage_max"] = round(d.max().item() / (tiles * 32), 4)
                rec["stream_TBs"] = round(sms * tiles * 32 * 16384 / (d.max().item() * 1e-6) / 1e12, 3)
            if which & 2:
                d = (t[:, 3] - t[:, 2]) / 1e3
                rec["mma_ns_per_group_median"] = round(d.median().item() * 1e3 / groups, 1)
            key = f"indep_which{which}"
            out[key] = rec
            print(key, rec, flush=True)
        os.makedirs(os.path.dirname(args.out), exist_ok=True)
        json.dump(out, open(args.out, "w"), indent=1)
        return
    if args.only_contend:
        stamps = torch.zeros(2 * sms, dtype=torch.int64, device="cuda")
        iters = 4000
        for busy in (0, 1, 2, 0):
            ok.fill_(1)
            rc = lib.probe_contend(sms, iters, busy, stamps.data_ptr(), ok.data_ptr(), C.byref(ms))
            ns = stamps[:sms].float().mean().item() / iters
            key = f"contend_load{busy}"
            out[key] = {"ns_per_mma_group": round(ns, 1), "rc": rc, "ok": int(ok.item())}
            print(key, out[key], flush=True)
        os.makedirs(os.path.dirname(args.out), exist_ok=True)
        json.dump(out, open(args.out, "w"), indent=1)
        return
    if args.only_mix:
        mma_mix(lib, sms, ok, ms, out)
        os.makedirs(os.path.dirname(args.out), exist_ok=True)
        json.dump(out, open(args.out, "w"), indent=1)
        return

    buf = torch.zeros(4 << 30, dtype=torch.uint8, device="cuda")
    sink = torch.zeros(1, dtype=torch.int32, device="cuda")
    for grid, block in ((sms * 4, 512), (sms * 8, 512), (sms * 16, 256)):
        for _ in range(3):
            rc = lib.probe_read(buf.data_ptr(), buf.numel(), grid, block, sink.data_ptr(), C.byref(ms))
        out[f"read_{grid}x{block}_GBs"] = round(buf.numel() / ms.value / 1e6, 1)
        print("read", grid, block, rc, out[f"read_{grid}x{block}_GBs"], flush=True)
    del buf

    rows = sms * 128 * 16
    A = torch.zeros(rows * 2048, dtype=torch.uint8, device="cuda")
    stamps = torch.zeros(1280, dtype=torch.int64, device="cuda")

    def stage_stats():
        st = stamps.cpu().tolist()
        lat = sorted((st[2 * i + 1] - st[2 * i]) / 1000 for i in range(64, 200))
        per = sorted((st[2 * i + 3] - st[2 * i + 1]) / 1000 for i in range(64, 200))
        return lat[len(lat) // 2], per[len(per) // 2]

    if args.only_pf:
        for layout, stages, mode, pf in ((5, 6, 1 | 64 | 262144, 1), (5, 6, 1 | 64 | 262144, 2),
                                         (5, 6, 1 | 64 | 262144, 3), (5, 5, 1 | 64 | 262144, 2),
                                         (5, 6, 1 | 64 | 128 | 262144, 2),
                                         (5, 5, 1 | 64, 0), (5, 5, 1 | 64 | 2048, 0), (5, 5, 1 | 64 | 2048 | 4096, 0),
                                         (5, 6, 1 | 64, 0), (5, 6, 1 | 64 | 2, 6), (5, 6, 1 | 64 | 2, 12),
                                         (5, 6, 1 | 64 | 2, 24), (5, 6, 1 | 64 | 2, 48), (5, 6, 1 | 64 | 128 | 2, 12),
                                         (5, 6, 2, 12), (5, 6, 0, 0),
                                         (5, 6, 1 | 64 | 4, 0), (5, 6, 1 | 64 | 8192, 0),
                                         (5, 6, 16384, 150), (5, 6, 16384, 290), (5, 6, 16384, 450),
                                         (5, 6, 16384 | 32768, 290), (5, 6, 16384 | 32768 | 131072, 290),
                                         (5, 6, 16384 | 32768 | 65536, 290), (5, 6, 1 | 64 | 32768, 0)):
            for _ in range(2):
                ok.fill_(1)
                rc = lib.probe_stream(A.data_ptr(), rows, sms, 8, stages, mode, pf, stamps.data_ptr(),
                                      ok.data_ptr(), C.byref(ms), layout)
            lat, per = stage_stats()
            st = stamps.cpu().tolist()
            iss = sorted((st[512 + i] - st[2 * i + 1]) / 1000 for i in range(64, 200)) if mode & (1 | 16384) else [0]
            obs = {}
            if mode & 32768:
                land = [st[768 + i] for i in range(256)]
                rel = [st[512 + i] for i in range(256)]
                med = lambda v: sorted(v)[len(v) // 2] if v else None
                obs = {"land_gap_us": med([(land[i + 1] - land[i]) / 1000 for i in range(64, 200)]),
                       "seen_after_land_us": med([(st[2 * i + 1] - land[i]) / 1000 for i in range(64, 200)]),
                       "next_land_after_release_us": med([(land[i + 1] - rel[i]) / 1000 for i in range(64, 200)])
                       if mode & (1 | 16384) else None,
                       "true_issue_to_land_us": med([(land[i] - st[2 * i]) / 1000 for i in range(64, 200)])}
                if mode & 16384:
                    obs["arrive_us"] = med([(st[1024 + i] - st[512 + i]) / 1000 for i in range(64, 200)])
                    obs["wait_done_after_arrive_us"] = med([(st[2 * i + 3] - st[1024 + i]) / 1000 for i in range(64, 200)])
            key = f"tma_layout{layout}_stages{stages}_mode{mode}_pf{pf}"
            out[key] = {"GBs": round(sms * 8 * 32 * 16384 / ms.value / 1e6, 1), "issue_to_land_us": lat,
                        "us_per_stage_cta0_median": per, "us_per_stage_mean": round(ms.value * 1e3 / (8 * 32), 3),
                        "mma_issue_us_median": iss[len(iss) // 2], "mma_issue_us_max": iss[-1], **obs,
                        "ok": int(ok.item()), "rc": rc}
            print(key, out[key], flush=True)
        os.makedirs(os.path.dirname(args.out), exist_ok=True)
        json.dump(out, open(args.out, "w"), indent=1)
        return

    if args.only_stream:
        for layout, stages, mode in ((5, 6, 0), (5, 6, 128), (5, 6, 1 | 64), (5, 6, 1 | 64 | 128),
                                     (6, 6, 128), (6, 6, 1 | 64 | 128), (7, 6, 0), (7, 6, 1 | 64 | 256),
                                     (5, 6, 1 | 64 | 512), (5, 6, 1 | 64 | 128 | 512), (5, 6, 1 | 64 | 1024),
                                     (5, 6, 1 | 64 | 128 | 1024)):
            for _ in range(2):
                ok.fill_(1)
                rc = lib.probe_stream(A.data_ptr(), rows, sms, 8, stages, mode, 0, stamps.data_ptr(),
                                      ok.data_ptr(), C.byref(ms), layout)
            lat, per = stage_stats()
            key = f"tma_layout{layout}_stages{stages}_mode{mode}"
            out[key] = {"GBs": round(sms * 8 * 32 * 16384 / ms.value / 1e6, 1), "issue_to_land_us": lat,
                        "us_per_stage": per, "ok": int(ok.item()), "rc": rc}
            print(key, out[key], flush=True)
        os.makedirs(os.path.dirname(args.out), exist_ok=True)
        json.dump(out, open(args.out, "w"), indent=1)
        return
    # layout: 0 fp4 128-row box, 1 fp4 contiguous tiles, 2 uint8 128-row box, 3 fp4 256-row box
    # mode: 1 = MMAs (N=32), |8 = 16 MMAs per stage, |16 = N=128, |32 = unscaled kind
    cases = [(0, 8192, 4, 0), (0, 8192, 8, 0), (1, 8192, 4, 0), (2, 16384, 4, 0), (2, 16384, 8, 0),
             (3, 16384, 4, 0), (0, 8192, 4, 1), (3, 16384, 4, 1), (0, 8192, 4, 1 | 16),
             (0, 8192, 4, 1 | 8), (0, 8192, 4, 1 | 32)]
    for layout, box, stages, mode in cases:
        for _ in range(2):
            ok.fill_(1)
            rc = lib.probe_stream(A.data_ptr(), rows, sms, 8, stages, mode, 0, stamps.data_ptr(),
                                  ok.data_ptr(), C.byref(ms), layout)
        lat, per = stage_stats()
        key = f"tma_layout{layout}_stages{stages}_mode{mode}"
        out[key] = {"GBs": round(sms * 8 * 32 * box / ms.value / 1e6, 1), "issue_to_land_us": lat,
                    "us_per_stage": per, "ok": int(ok.item()), "rc": rc}
        print(key, out[key], flush=True)
    for stages in (4, 8):
        ok.fill_(1)
        for _ in range(2):
            rc = lib.probe_stream_lsu(A.data_ptr(), rows, sms, 8, stages, stamps.data_ptr(), ok.data_ptr(),
                                      C.byref(ms))
        lat, per = stage_stats()
        out[f"cpasync_stages{stages}"] = {"GBs": round(sms * 8 * 32 * 8192 / ms.value / 1e6, 1),
                                          "us_per_stage": per, "ok": int(ok.item()), "rc": rc}
        print(f"cpasync_stages{stages}", out[f"cpasync_stages{stages}"], flush=True)
    del A

    mma_mix(lib, sms, ok, ms, out)
    for fmt in (5, 0):
        for n in (32, 128, 256):
            iters = 20000 if n >= 128 else 40000
            ok.fill_(1)
            lib.probe_mma_peak(sms, 100, n, fmt, ok.data_ptr(), C.byref(ms))
            rc = lib.probe_mma_peak(sms, iters, n, fmt, ok.data_ptr(), C.byref(ms))
            tf = sms * iters * 4 * 2 * 128 * n * 32 / ms.value / 1e9
            out[f"mma_afmt{fmt}_n{n}_TFs"] = round(tf, 1)
            print("mma", fmt, n, rc, int(ok.item()), round(tf, 1), flush=True)
    os.makedirs(os.path.dirname(args.out), exist_ok=True)
    json.dump(out, open(args.out, "w"), indent=1)


def mma_mix(lib, sms, ok, ms, out):
    """ns per iteration of [ncp scale copies + 4 (or 8) MMAs (+ commit)] on every SM."""
    iters = 20000
    cases = [(16, 0, 0, 0, 0), (16, 0, 0, 1, 0), (16, 3, 1, 1, 0), (16, 1, 1, 1, 0), (128, 3, 1, 1, 0),
             (16, 0, 0, 2, 0), (16, 0, 0, 1, 1), (16, 0, 0, 1, 2), (16, 0, 0, 0, 1), (16, 3, 1, 1, 1),
             (16, 0, 0, 1, 3), (16, 3, 1, 1, 3), (16, 0, 0, 0, 4), (16, 2, 1, 0, 4), (16, 3, 1, 0, 4),
             (16, 0, 1, 0, 5), (16, 0, 1, 0, 6), (16, 0, 0, 0, 5), (16, 0, 0, 0, 6), (16, 0, 0, 0, 7),
             (16, 0, 0, 0, 8), (16, 0, 0, 0, 9)]
    for fmt in (5,):
        for n, ncp, commit, acc2, mode in cases:
                ok.fill_(1)
                lib.probe_mma_mix(sms, 100, n, ncp, commit, acc2, fmt, mode, ok.data_ptr(), C.byref(ms))
                rc = lib.probe_mma_mix(sms, iters, n, ncp, commit, acc2, fmt, mode, ok.data_ptr(), C.byref(ms))
                key = (f"mix_f{fmt}_n{n}_cp{ncp}_commit{commit}_" + ("acc1", "acc2", "acc8split")[acc2] +
                       ("", "_samesfid", "_sameaddr", "_nswzB", "_swapN256", "_swapN256_sfres_cpnow",
                        "_swapN256_sfres_cpahead", "_swapN256_nswzB", "_swapN256_realA",
                        "_swapN256_tmemA")[mode])
                out[key] = {"ns_per_iter": round(ms.value * 1e6 / iters, 2), "rc": rc, "ok": int(ok.item())}
                print(key, out[key], flush=True)


if __name__ == "__main__":
    main()
