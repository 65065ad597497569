"""Configuration sweep: time every kernel configuration the library can run
for given GEMM shapes and report the fastest (the tuning harness of the
pages: block sizes, pipeline depth and rasterisation screened per shape).

Configurations, two axes at a time as the pages tune them: the CTA-pair
kernel (256 x 256 tiles, k-block 128) with grouped tile orders of 2..32
tile rows at its default three stages, and with 2 or 3 stages at its
default group; the one-CTA kernel with 128 x 64 / 128 x 128 / 128 x 256
tiles (at most 4 / 3 / 4 stages, k-blocks of 128 / 128 / 64 fp16
elements) with group heights 4..32 at
the most stages, with every depth from 2 stages up at the default group,
and unsplit or split over K by clusters of 2, 4 or 8 CTAs; the skinny
kernel when M <= 64.  Each configuration is forced through
tg_gemm_force_path / tg_gemm_force_tiling / tg_gemm_force_stages /
tg_gemm_force_split_k, launched `reps` times from one CUDA graph over
operand sets rotated past L2, and timed with CUDA events.

    python -m tiled_gemm_tg_gb300.sweep --shapes 1024x1024x1024,8192x8192x8192

A shape of four numbers, BxMxNxK, is a strided batch of B packed products
(tg_gemm_batched).
"""
from __future__ import annotations

import argparse
import json

import tiled_gemm_tg_gb300 as tg

PAIR, MAIN, SKINNY = 6, 3, 5
L2_BYTES = 129 * 2**20


MAX_STAGES = {(PAIR, 0): 3, (MAIN, 64): 4, (MAIN, 128): 3, (MAIN, 256): 4}


def candidates(M: int, N: int, K: int):
    """(path, tile width, group height, stages, split over K); 0 = the
    kernel's default (for the split: its own choice; 1 = unsplit)."""
    out = [(PAIR, 0, g, 0, 0) for g in (2, 4, 8, 16, 32)]
    out += [(PAIR, 0, 0, st, 0) for st in range(2, MAX_STAGES[(PAIR, 0)])]
    for bn in (64, 128, 256):
        out += [(MAIN, bn, g, 0, 1) for g in (4, 8, 16, 32)]
        out += [(MAIN, bn, 0, st, 1) for st in range(2, MAX_STAGES[(MAIN, bn)])]
        out += [(MAIN, bn, 0, 0, sp) for sp in (1, 2, 4, 8)]
    if M <= 64:
        out.append((SKINNY, 0, 0, 0, 0))
    return out


def time_config(M, N, K, path, bn, group, reps=50, sets=None, batch=1, stages=0, split=0):
    """Microseconds per launch (CUDA-graph replay), or None if not served."""
    import torch

    if sets is None:
        sets = make_sets(M, N, K, batch)
    a0, b0, c0 = sets[0]
    sa, sb, sc = M * K, K * N, M * N
    tg.tg_gemm_force_path(path)
    if (tg.tg_gemm_force_tiling(bn, group) != tg.TG_OK or tg.tg_gemm_force_stages(stages) != tg.TG_OK
            or tg.tg_gemm_force_split_k(split) != tg.TG_OK):
        tg.tg_gemm_force_path(0)
        tg.tg_gemm_force_tiling(0, 0)
        tg.tg_gemm_force_stages(0)
        tg.tg_gemm_force_split_k(0)
        return None
    try:
        if tg.tg_gemm_batched_path(batch, M, N, K, a0.data_ptr(), K, sa, b0.data_ptr(), N, sb,
                                   c0.data_ptr(), N, sc, tg.F16, tg.F16) != path:
            return None

        def launch(i, h):
            a, b, c = sets[i % len(sets)]
            st = tg.tg_gemm_batched(batch, M, N, K, a.data_ptr(), K, sa, b.data_ptr(), N, sb,
                                    c.data_ptr(), N, sc, tg.F16, tg.F16, h)
            if st != tg.TG_OK:
                raise tg.TgError(st)

        h = torch.cuda.current_stream().cuda_stream
        for i in range(3):
            launch(i, h)
        tg.check()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            hc = torch.cuda.current_stream().cuda_stream
            for i in range(reps):
                launch(i, hc)
        g.replay()
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record()
        g.replay()
        e1.record()
        torch.cuda.synchronize()
        tg.check()
        return e0.elapsed_time(e1) * 1e3 / reps
    finally:
        tg.tg_gemm_force_path(0)
        tg.tg_gemm_force_tiling(0, 0)
        tg.tg_gemm_force_stages(0)
        tg.tg_gemm_force_split_k(0)


def make_sets(M, N, K, batch=1):
    import torch

    dev = torch.device("cuda")
    set_bytes = batch * (M * K + K * N + M * N) * 2
    n = max(2, min(64, -(-3 * L2_BYTES // set_bytes)))
    g = torch.Generator(device=dev).manual_seed(7)
    return [((torch.rand(batch, M, K, device=dev, generator=g) * 2 - 1).half(),
             (torch.rand(batch, K, N, device=dev, generator=g) * 2 - 1).half(),
             torch.empty(batch, M, N, dtype=torch.half, device=dev)) for _ in range(n)]


def sweep(shapes, reps=50):
    import torch

    torch.cuda.set_device(0)
    results = []
    for shape in shapes:
        batch, (M, N, K) = (shape[0], shape[1:]) if len(shape) == 4 else (1, shape)
        sets = make_sets(M, N, K, batch)
        a0, b0, c0 = sets[0]
        auto_path = tg.tg_gemm_batched_path(batch, M, N, K, a0.data_ptr(), K, M * K,
                                            b0.data_ptr(), N, K * N, c0.data_ptr(), N, M * N,
                                            tg.F16, tg.F16)
        auto_us = time_config(M, N, K, auto_path, 0, 0, reps, sets, batch)
        rows = []
        for path, bn, group, stages, split in candidates(M, N, K):
            us = time_config(M, N, K, path, bn, group, reps, sets, batch, stages, split)
            if us is not None:
                rows.append({"path": path, "bn": bn, "group_m": group, "stages": stages,
                             "split": split, "us": us,
                             "tflops": 2.0 * batch * M * N * K / (us * 1e-6) / 1e12})
        best = min(rows, key=lambda r: r["us"])
        results.append({"shape": list(shape), "auto_path": auto_path, "auto_us": auto_us,
                        "best": best, "configs": rows})
        del sets
        torch.cuda.empty_cache()
    return results


def parse_shapes(text: str):
    return [tuple(int(v) for v in s.lower().split("x")) for s in text.split(",") if s]


def main():
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--shapes", default="1024x1024x1024,1024x2048x512,4096x4096x4096,"
                                        "8192x8192x8192,4096x16384x4096")
    ap.add_argument("--reps", type=int, default=50)
    ap.add_argument("--json", default="")
    args = ap.parse_args()
    res = sweep(parse_shapes(args.shapes), args.reps)
    names = {PAIR: "pair 256x256", MAIN: "one-CTA 128x{bn}", SKINNY: "skinny"}
    for r in res:
        print(f"\n{'x'.join(str(v) for v in r['shape'])}: automatic path {r['auto_path']} {r['auto_us']:.1f} us; "
              f"best {names[r['best']['path']].format(bn=r['best']['bn'])} "
              f"group {r['best']['group_m']} stages {r['best']['stages']} "
              f"split {r['best']['split'] or 'auto'} {r['best']['us']:.1f} us")
        print("| config | group_m | stages | split over K | us | TFLOP/s |")
        print("|---|---|---|---|---|---|")
        for c in sorted(r["configs"], key=lambda c: c["us"]):
            st = c["stages"] or MAX_STAGES.get((c["path"], c["bn"]), "-")
            sp = c["split"] or ("auto" if c["path"] == MAIN else "-")
            print(f"| {names[c['path']].format(bn=c['bn'])} | {c['group_m'] or 'default'} | "
                  f"{st} | {sp} | {c['us']:.1f} | {c['tflops']:.0f} |")
    if args.json:
        with open(args.json, "w") as f:
            json.dump(res, f, indent=1)


if __name__ == "__main__":
    main()
