"""Concurrent calls through the C ABI: several host threads, each with its
own CUDA stream, call tg_gemm at once on shapes that take every GEMM path
(the tensor-map cache, the per-device state and the kernel attributes are
shared between them; ctypes releases the GIL for each call).

A kernel's order of fp32 additions is fixed by the shape, the path and the
tiling, so every concurrent result must equal, bit for bit, the same call
made alone; each lone call is checked against the oracle on every element.
"""
import threading

import numpy as np
import pytest
import torch

import oracle
import tiled_gemm_tg_gb300 as tg
from tiled_gemm_tg_gb300 import inputs

from gpu_util import bits, code, compare

pytestmark = pytest.mark.gpu

MAIN, BOUNDARY, SIMT, PAIR, SKINNY = 3, 4, 2, 6, 5

# (M, N, K, input dtype, output dtype, path the library takes)
SHAPES = [
    (16, 4096, 4096, torch.float16, torch.float16, SKINNY),
    (1024, 2048, 512, torch.float16, torch.float16, MAIN),
    (2048, 4608, 1024, torch.float16, torch.float16, PAIR),
    (127, 255, 512, torch.float16, torch.float16, BOUNDARY),  # 510-byte rows of B
    (128, 128, 128, torch.float32, torch.float32, SIMT),
    (300, 520, 1000, torch.float16, torch.float32, MAIN),
    (256, 256, 8192, torch.float16, torch.float16, MAIN),  # split over K in clusters
]
THREADS = 4
ROUNDS = 3


def _operands(i, M, N, K, dt):
    name = "f16" if dt == torch.float16 else "f32"
    a = inputs.draw((M, K), "normal", 7100 + 2 * i, name)
    b = inputs.draw((K, N), "normal", 7101 + 2 * i, name)
    return a, b


def _call(dev_a, dev_b, c, M, N, K, in_dt, out_dt, stream_handle):
    return tg.tg_gemm(M, N, K, dev_a.data_ptr(), K, dev_b.data_ptr(), N, c.data_ptr(), N,
                      code(in_dt), code(out_dt), stream_handle)


@pytest.fixture(scope="module")
def lone_results():
    """Every shape called alone on the current stream: operands on the
    device, the result, and its check against the oracle."""
    tg.tg_gemm_force_path(0)
    dev = torch.device("cuda")
    out = []
    for i, (M, N, K, in_dt, out_dt, want_path) in enumerate(SHAPES):
        a, b = _operands(i, M, N, K, in_dt)
        da, db = a.to(dev), b.to(dev)
        c = torch.empty((M, N), dtype=out_dt, device=dev)
        assert tg.tg_gemm_path(M, N, K, da.data_ptr(), K, db.data_ptr(), N, c.data_ptr(), N,
                               code(in_dt), code(out_dt)) == want_path
        h = torch.cuda.current_stream().cuda_stream
        assert _call(da, db, c, M, N, K, in_dt, out_dt, h) == tg.TG_OK
        assert tg.tg_gemm_check(h) == tg.TG_OK
        C_ref, S = oracle.gemm(a.numpy(), b.numpy())
        compare(c.double().cpu().numpy(), C_ref, S, out_dt == torch.float16,
                f"{M}x{N}x{K} alone")
        out.append((da, db, c.clone()))
    return out


def test_concurrent_calls_match_lone_calls(lone_results):
    dev = torch.device("cuda")
    # each thread: its own stream and its own outputs, the shapes in its own
    # rotation so that different paths run side by side
    streams = [torch.cuda.Stream(device=dev) for _ in range(THREADS)]
    outs = [[[torch.full_like(lone_results[s][2], float("nan")) for s in range(len(SHAPES))]
             for _ in range(ROUNDS)] for _ in range(THREADS)]
    torch.cuda.synchronize()
    start = threading.Barrier(THREADS)
    errors = []

    def worker(t):
        try:
            h = streams[t].cuda_stream
            start.wait()
            for r in range(ROUNDS):
                for j in range(len(SHAPES)):
                    s = (j + t + r) % len(SHAPES)
                    M, N, K, in_dt, out_dt, _ = SHAPES[s]
                    da, db, _ = lone_results[s]
                    st = _call(da, db, outs[t][r][s], M, N, K, in_dt, out_dt, h)
                    if st != tg.TG_OK:
                        errors.append((t, r, s, tg.tg_status_string(st)))
                        return
            st = tg.tg_gemm_check(h)
            if st != tg.TG_OK:
                errors.append((t, "check", tg.tg_status_string(st)))
        except Exception as e:  # reported below, on the main thread
            errors.append((t, repr(e)))

    threads = [threading.Thread(target=worker, args=(t,)) for t in range(THREADS)]
    for th in threads:
        th.start()
    for th in threads:
        th.join(timeout=300)
    assert not any(th.is_alive() for th in threads), "a calling thread did not finish"
    torch.cuda.synchronize()
    assert not errors, errors
    for t in range(THREADS):
        for r in range(ROUNDS):
            for s, (M, N, K, _, _, _) in enumerate(SHAPES):
                want = bits(lone_results[s][2])
                got = bits(outs[t][r][s])
                same = torch.equal(got, want)
                assert same, (f"thread {t} round {r} shape {M}x{N}x{K}: "
                              f"{int((got != want).sum())} elements differ from the lone call")


def test_concurrent_error_word_stays_clean(lone_results):
    """After the concurrent calls, a check on a fresh stream reports no
    expired wait or other device error."""
    s = torch.cuda.Stream()
    assert tg.tg_gemm_check(s.cuda_stream) == tg.TG_OK
    assert np.isfinite(lone_results[0][2].float().cpu().numpy()).all()
