"""GPU parity of the 8-bit GEMM: FP8 E4M3 inputs, fp32 accumulation on
tcgen05 (kind::f8f6f4), fp16 or fp32 output, against the oracle's exact
E4M3 decode and fp64 product.

Integer-valued E4M3 operands (0, +-1, +-2, +-3) make every fp32 partial sum
exact and the result unique: those cases must match bit for bit.  Random
operands are held to the same bound as fp16 inputs, 2e-3 S + 1e-5
(+ 1e-2 |C| for an fp16 output), since the products of two E4M3 values are
exact in fp32 like those of two fp16 values.
"""
import os

import numpy as np
import pytest
import torch

import oracle
import tiled_gemm_tg_gb300 as tg
from tiled_gemm_tg_gb300 import inputs

from gpu_util import GUARD, bits, compare, f16_bits_of

pytestmark = pytest.mark.gpu

MAIN, PAIR = 3, 6


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(0)
    tg.tg_gemm_force_path(0)
    yield
    tg.tg_gemm_force_path(0)
    tg.tg_gemm_force_tiling(0, 0)


def int_e4m3(shape, seed):
    """E4M3 operands whose values are the integers -3..3 (all exact)."""
    g = torch.Generator().manual_seed(seed)
    return torch.randint(-3, 4, shape, generator=g).to(torch.float32).to(torch.float8_e4m3fn)


def u8(x):
    return x.view(torch.uint8).numpy()


def run_e4m3(a, b, out_dtype, lda=None, ldb=None, ldc=None):
    """tg_gemm on E4M3 operands placed with row strides lda/ldb (multiples of
    16); C guarded by canaries.  Returns (C float64, canaries intact, path)."""
    M, K = a.shape
    N = b.shape[1]
    lda = K if lda is None else lda
    ldb = N if ldb is None else ldb
    ldc = N if ldc is None else ldc
    A = torch.zeros(max(M, 1) * lda + 64, dtype=torch.uint8)
    A[:M * lda].view(M, lda)[:, :K] = a.view(torch.uint8)
    B = torch.zeros(max(K, 1) * ldb + 64, dtype=torch.uint8)
    B[:K * ldb].view(K, ldb)[:, :N] = b.view(torch.uint8)
    A, B = A.cuda(), B.cuda()
    n = GUARD + M * ldc + GUARD
    Cbuf = torch.empty(n, dtype=out_dtype, device="cuda")
    bits(Cbuf).fill_(0x7E5A if out_dtype == torch.float16 else 0x7FC0A5A5)
    canary = bits(Cbuf[:1].clone()).item()
    oc = tg.F16 if out_dtype == torch.float16 else tg.F32
    C = Cbuf.data_ptr() + GUARD * Cbuf.element_size()
    s = torch.cuda.current_stream().cuda_stream
    path = tg.tg_gemm_path(M, N, K, A.data_ptr(), lda, B.data_ptr(), ldb, C, ldc, tg.E4M3, oc)
    st = tg.tg_gemm(M, N, K, A.data_ptr(), lda, B.data_ptr(), ldb, C, ldc, tg.E4M3, oc, s)
    assert st == tg.TG_OK, tg.tg_status_string(st)
    assert tg.tg_gemm_check(s) == tg.TG_OK
    h = Cbuf.cpu()
    hb = bits(h)
    body = h[GUARD:GUARD + M * ldc].view(M, ldc)
    intact = bool((hb[:GUARD] == canary).all()) and bool((hb[GUARD + M * ldc:] == canary).all())
    if ldc > N:
        intact = intact and bool((bits(body)[:, N:] == canary).all())
    return body[:, :N].double().numpy(), intact, path


def _exact(got, C, out):
    if out == torch.float16:
        assert np.array_equal(f16_bits_of(got), f16_bits_of(C))
    else:
        assert np.array_equal(got, C)


@pytest.mark.parametrize("M,N,K", [(128, 128, 128), (300, 520, 448), (129, 384, 1000),
                                   (1, 256, 32), (64, 128, 2048)])
@pytest.mark.parametrize("force,bn", [(MAIN, 128), (MAIN, 256), (PAIR, 0)])
@pytest.mark.parametrize("out", [torch.float16, torch.float32])
def test_e4m3_integer_bitwise(M, N, K, force, bn, out):
    a, b = int_e4m3((M, K), 12000 + M), int_e4m3((K, N), 12100 + N)
    pad16 = lambda x: (x + 15) // 16 * 16  # noqa: E731
    tg.tg_gemm_force_path(force)
    tg.tg_gemm_force_tiling(bn, 0)
    try:
        got, intact, p = run_e4m3(a, b, out, lda=pad16(K), ldb=pad16(N), ldc=N + 3)
    finally:
        tg.tg_gemm_force_path(0)
        tg.tg_gemm_force_tiling(0, 0)
    assert p == force and intact
    C, _ = oracle.gemm(u8(a), u8(b))
    _exact(got, C, out)


@pytest.mark.parametrize("M,N,K,want", [(300, 520, 448, MAIN), (2048, 2048, 4096, PAIR),
                                        (1792, 2816, 4096, PAIR), (2048, 2048, 2048, MAIN)])
@pytest.mark.parametrize("out", [torch.float16, torch.float32])
def test_e4m3_random(M, N, K, want, out):
    a = inputs.draw((M, K), "normal", 12200 + M, "e4m3")
    b = inputs.draw((K, N), "normal", 12300 + N, "e4m3")
    pad16 = lambda x: (x + 15) // 16 * 16  # noqa: E731
    got, intact, p = run_e4m3(a, b, out, lda=pad16(K), ldb=pad16(N))
    assert p == want and intact
    if M * N * K <= 2 ** 31:
        C, S = oracle.gemm(u8(a), u8(b))
        compare(got, C, S, out == torch.float16, f"e4m3 {M}x{N}x{K}")
    else:
        rng = np.random.default_rng(12400)
        r, c = rng.integers(0, M, 2000), rng.integers(0, N, 2000)
        Cs, Ss = oracle.gemm_at(u8(a), u8(b), r, c)
        compare(got[r, c], Cs, Ss, out == torch.float16, f"e4m3 {M}x{N}x{K} sampled")


def test_e4m3_square_8192_full():
    """The 8-bit square workload on every one of its 67 M outputs against the
    oracle's full fp64 product of the exactly decoded E4M3 inputs."""
    w = inputs.WORKLOADS["square_8192_e4m3"]
    a, b = inputs.operands(w)
    got, intact, p = run_e4m3(a, b, torch.float16)
    assert p == PAIR and intact
    C_ref, S = oracle.gemm(u8(a), u8(b), nthreads=os.cpu_count() or 0)
    compare(got, C_ref, S, True, "e4m3 8192^3, all elements")


def test_e4m3_batched_and_epilogue():
    """E4M3 through tg_gemm_batched (3 products, broadcast B) and tg_gemm_ex."""
    M, N, K, batch = 256, 384, 512, 3
    a = torch.stack([int_e4m3((M, K), 12600 + i) for i in range(batch)])
    b = int_e4m3((K, N), 12700)
    A, B = a.view(torch.uint8).cuda(), b.view(torch.uint8).cuda()
    C = torch.empty(batch, M, N, dtype=torch.float32, device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    st = tg.tg_gemm_batched(batch, M, N, K, A.data_ptr(), K, M * K, B.data_ptr(), N, 0,
                            C.data_ptr(), N, M * N, tg.E4M3, tg.F32, s)
    assert st == tg.TG_OK and tg.tg_gemm_check(s) == tg.TG_OK
    for i in range(batch):
        Ci, _ = oracle.gemm(u8(a[i]), u8(b))
        assert np.array_equal(C[i].double().cpu().numpy(), Ci)
    bias = torch.arange(N, dtype=torch.float32) - 100
    bd = bias.cuda()
    D = torch.empty(M, N, dtype=torch.float16, device="cuda")
    st = tg.tg_gemm_ex(M, N, K, A.data_ptr(), K, B.data_ptr(), N, D.data_ptr(), N, tg.E4M3,
                       tg.F16, 2.0, 0.0, 0, N, bd.data_ptr(), tg.ACT_RELU, s)
    assert st == tg.TG_OK and tg.tg_gemm_check(s) == tg.TG_OK
    C0, _ = oracle.gemm(u8(a[0]), u8(b))
    ref = oracle.epilogue(C0, 2.0, 0.0, None, bias.numpy(), tg.ACT_RELU)
    assert np.array_equal(f16_bits_of(D.double().cpu().numpy()), f16_bits_of(ref))


@pytest.mark.parametrize("split", [0, 1, 2, 8])
@pytest.mark.parametrize("out", [torch.float16, torch.float32])
def test_e4m3_split_k_bitwise(split, out):
    """E4M3 through the one-CTA kernel with its tiles shared over K by a
    cluster (0: the automatic choice, which splits this few-tile, deep-K
    shape): integer-valued operands, exact whatever the split."""
    M, N, K = 200, 272, 8192
    a = int_e4m3((M, K), 12900)
    b = int_e4m3((K, N), 12901)
    assert tg.tg_gemm_force_split_k(split) == tg.TG_OK
    try:
        got, intact, p = run_e4m3(a, b, out, ldc=N + 8)
    finally:
        tg.tg_gemm_force_split_k(0)
    assert p == MAIN and intact
    C, _ = oracle.gemm(u8(a), u8(b))
    _exact(got, C, out)
