"""GPU parity of the strided batch, C_b = A_b x B_b, through tg_gemm_batched.

Each product is exactly the one tg_gemm computes, so every matrix of the
batch is compared with the oracle's product of its own operands, under the
same acceptance bound (bit for bit on integer inputs).  C lives in one
buffer whose gaps (between rows beyond N, and between matrices beyond the
last row) are filled with a canary the kernels never write; every test
checks that the gaps and the guard bands are intact.
"""
import numpy as np
import pytest
import torch

import oracle
import tiled_gemm_tg_gb300 as tg
from tiled_gemm_tg_gb300 import inputs

from gpu_util import GUARD, bits, code, compare, esize, f16_bits_of

pytestmark = pytest.mark.gpu

SIMT, MAIN, BOUNDARY, SKINNY, PAIR = 2, 3, 4, 5, 6


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


def _place(mats, ld, stride, off, dtype):
    """Matrices of one shape at `off + b*stride` with row stride ld, in one
    device buffer (a stride of 0 places the single given matrix)."""
    rows, cols = mats[0].shape
    count = len(mats)
    n = off + max(count - 1, 0) * stride + rows * ld + 64
    buf = torch.zeros(n, dtype=dtype)
    for b, x in enumerate(mats):
        s = off + b * stride
        buf[s:s + rows * ld].view(rows, ld)[:, :cols] = x
    dev = buf.cuda()
    return dev, dev.data_ptr() + off * esize(dtype)


def run_batched(a_list, b_list, out_dtype, lda, sA, ldb, sB, ldc, sC, batch=None):
    """a_list/b_list: CPU matrices (one matrix for a broadcast operand)."""
    batch = batch if batch is not None else max(len(a_list), len(b_list))
    M, K = a_list[0].shape
    N = b_list[0].shape[1]
    dt = a_list[0].dtype
    Abuf, A = _place(a_list, lda, sA, 0, dt)
    Bbuf, B = _place(b_list, ldb, sB, 0, dt)
    n = GUARD + (batch - 1) * sC + M * ldc + GUARD
    Cbuf = torch.empty(n, dtype=out_dtype, device="cuda")
    bits(Cbuf).fill_(0x7E5A if out_dtype == torch.float16 else 0x7FC0A5A5)
    canary = bits(Cbuf[:1].clone()).item()
    C = Cbuf.data_ptr() + GUARD * esize(out_dtype)
    s = torch.cuda.current_stream().cuda_stream
    path = tg.tg_gemm_batched_path(batch, M, N, K, A, lda, sA, B, ldb, sB, C, ldc, sC,
                                   code(dt), code(out_dtype))
    st = tg.tg_gemm_batched(batch, M, N, K, A, lda, sA, B, ldb, sB, C, ldc, sC, code(dt),
                            code(out_dtype), s)
    assert st == tg.TG_OK, tg.tg_status_string(st)
    assert tg.tg_gemm_check(s) == tg.TG_OK
    h = Cbuf.cpu()
    hb = bits(h)
    written = torch.zeros(n, dtype=torch.bool)
    outs = []
    for b in range(batch):
        start = GUARD + b * sC
        body = h[start:start + M * ldc].view(M, ldc)
        outs.append(body[:, :N].double().numpy())
        written[start:start + M * ldc].view(M, ldc)[:, :N] = True
    intact = bool((hb[~written] == canary).all())
    return outs, intact, path


def _mats(count, shape, dist, seed, dt, k):
    return [inputs.draw(shape, dist, seed + i, dt, k=k) for i in range(count)]


def _check(a_list, b_list, outs, out_dtype, exact=False):
    for b, got in enumerate(outs):
        a = a_list[b if len(a_list) > 1 else 0]
        bb = b_list[b if len(b_list) > 1 else 0]
        C, S = oracle.gemm(a.numpy(), bb.numpy())
        if exact:
            if out_dtype == torch.float16:
                assert np.array_equal(f16_bits_of(got), f16_bits_of(C)), f"matrix {b}"
            else:
                assert np.array_equal(got, C), f"matrix {b}"
        else:
            compare(got, C, S, out_dtype == torch.float16, f"matrix {b}")


# path -> (M, N, K, in dtype); N is not a multiple of the tile width
SHAPES = {
    MAIN: (200, 300, 272, "f16"),
    PAIR: (200, 300, 272, "f16"),
    BOUNDARY: (127, 255, 130, "f16"),
    SKINNY: (37, 300, 520, "f16"),
    SIMT: (77, 130, 45, "f32"),
}


def _layout(path, M, N, K, kind):
    """(lda, sA, ldb, sB, ldc, sC) for a layout kind: packed, padded strides,
    broadcast A or broadcast B."""
    al = 8 if path != BOUNDARY else 1
    lda = (K + al - 1) // al * al
    ldb = (N + al - 1) // al * al
    if path == BOUNDARY:
        lda, ldb = K + 1, N + 3
    ldc = N + 5
    sA, sB = M * lda, K * ldb
    sC = M * ldc + 7
    if kind == "padded":
        sA += 64
        sB += 8 * 13
        sC += 100
    elif kind == "bcast_a":
        sA = 0
    elif kind == "bcast_b":
        sB = 0
    return lda, sA, ldb, sB, ldc, sC


@pytest.mark.parametrize("kind", ["packed", "padded", "bcast_a", "bcast_b"])
@pytest.mark.parametrize("path", [MAIN, PAIR, BOUNDARY, SKINNY, SIMT])
@pytest.mark.parametrize("out", [torch.float16, torch.float32])
def test_batched_every_path(kind, path, out):
    M, N, K, dt = SHAPES[path]
    if dt == "f32" and out == torch.float16:
        pytest.skip("the fp32 path writes fp32")
    batch = 3
    a_list = _mats(1 if kind == "bcast_a" else batch, (M, K), "normal_rsqrtk", 11000 + path, dt, K)
    b_list = _mats(1 if kind == "bcast_b" else batch, (K, N), "normal_rsqrtk", 11100 + path, dt, K)
    lda, sA, ldb, sB, ldc, sC = _layout(path, M, N, K, kind)
    tg.tg_gemm_force_path(path)
    try:
        outs, intact, p = run_batched(a_list, b_list, out, lda, sA, ldb, sB, ldc, sC, batch)
    finally:
        tg.tg_gemm_force_path(0)
    assert p == path and intact
    _check(a_list, b_list, outs, out)


@pytest.mark.parametrize("path", [MAIN, PAIR, BOUNDARY, SKINNY, SIMT])
def test_batched_integer_bitwise(path):
    M, N, K, dt = SHAPES[path]
    out = torch.float32 if dt == "f32" else torch.float16
    batch = 5
    a_list = _mats(batch, (M, K), "int2", 11200 + path, dt, K)
    b_list = _mats(batch, (K, N), "int2", 11300 + path, dt, K)
    lda, sA, ldb, sB, ldc, sC = _layout(path, M, N, K, "packed")
    tg.tg_gemm_force_path(path)
    try:
        outs, intact, p = run_batched(a_list, b_list, out, lda, sA, ldb, sB, ldc, sC)
    finally:
        tg.tg_gemm_force_path(0)
    assert p == path and intact
    _check(a_list, b_list, outs, out, exact=True)


@pytest.mark.parametrize("kind", ["packed", "bcast_b"])
@pytest.mark.parametrize("split", [0, 2, 8])
def test_batched_split_k_integer_bitwise(kind, split):
    """A strided batch through the one-CTA kernel split over K (0: the
    automatic choice, which splits these few deep-K tiles): each cluster
    reduces one tile of one product, exactly."""
    M, N, K, batch = 200, 136, 3000, 3
    a_list = _mats(batch, (M, K), "int2", 11600, "f16", K)
    b_list = _mats(1 if kind == "bcast_b" else batch, (K, N), "int2", 11700, "f16", K)
    lda, sA, ldb, sB, ldc, sC = _layout(MAIN, M, N, K, kind)
    tg.tg_gemm_force_path(MAIN)
    assert tg.tg_gemm_force_split_k(split) == tg.TG_OK
    try:
        outs, intact, p = run_batched(a_list, b_list, torch.float16, lda, sA, ldb, sB, ldc, sC,
                                      batch)
    finally:
        tg.tg_gemm_force_split_k(0)
        tg.tg_gemm_force_path(0)
    assert p == MAIN and intact
    _check(a_list, b_list, outs, torch.float16, exact=True)


@pytest.mark.parametrize("batch,M,N,K,want", [
    (16, 512, 512, 4096, PAIR),     # 64 pair tiles over the batch, K = 4096
    (16, 512, 512, 1024, MAIN),     # 64 pair tiles with K < 4096
    (6, 300, 200, 128, MAIN),
    (12, 16, 1024, 2048, SKINNY),
    (2, 1, 8, 8, SKINNY),
])
def test_batched_natural_paths(batch, M, N, K, want):
    a_list = _mats(batch, (M, K), "int2", 11400 + M, "f16", K)
    b_list = _mats(batch, (K, N), "int2", 11500 + N, "f16", K)
    outs, intact, p = run_batched(a_list, b_list, torch.float16, K, M * K, N, K * N, N, M * N)
    assert p == want and intact
    _check(a_list, b_list, outs, torch.float16, exact=True)


@pytest.mark.parametrize("M,N,K,dt,want", [
    (4, 4, 4, "f32", SIMT),
    (4, 4, 4, "f16", BOUNDARY),    # 8-byte rows: not TMA-addressable
    (16, 128, 64, "f16", SKINNY),
    (72, 64, 64, "f16", MAIN),
])
def test_batched_largest_batch(M, N, K, dt, want):
    """The largest batch the ABI accepts, 65535 packed products, on every
    kernel that indexes the batch (the grid's z extent, or the tile order and
    the tensor maps' third dimension): integer inputs, so each product is
    unique and compared bit for bit with the oracle's, on every product for
    the tiny shapes and on 300 of them (the first, the last and random ones)
    for the others; the guard bands around C keep their canary."""
    batch = 65535
    a_list = _mats(batch, (M, K), "int2", 11900, dt, K)
    b_list = _mats(batch, (K, N), "int2", 11950, dt, K)
    out_dtype = torch.float32 if dt == "f32" else torch.float16
    A = torch.stack(a_list).cuda()
    B = torch.stack(b_list).cuda()
    Cbuf = torch.empty(GUARD + batch * M * N + GUARD, dtype=out_dtype, device="cuda")
    bits(Cbuf).fill_(0x7E5A if out_dtype == torch.float16 else 0x7FC0A5A5)
    canary = bits(Cbuf[:1].clone()).item()
    C = Cbuf.data_ptr() + GUARD * esize(out_dtype)
    s = torch.cuda.current_stream().cuda_stream
    args = (batch, M, N, K, A.data_ptr(), K, M * K, B.data_ptr(), N, K * N, C, N, M * N,
            code(A.dtype), code(out_dtype))
    assert tg.tg_gemm_batched_path(*args) == want
    st = tg.tg_gemm_batched(*args, s)
    assert st == tg.TG_OK, tg.tg_status_string(st)
    assert tg.tg_gemm_check(s) == tg.TG_OK
    h = Cbuf.cpu()
    hb = bits(h)
    assert bool((hb[:GUARD] == canary).all()) and bool((hb[-GUARD:] == canary).all())
    body = h[GUARD:GUARD + batch * M * N].view(batch, M, N)
    if M * N * K <= 64:
        pick = list(range(batch))
    else:
        rng = np.random.default_rng(11999)
        pick = sorted({0, 1, batch - 2, batch - 1, *rng.integers(0, batch, 296).tolist()})
    _check([a_list[i] for i in pick], [b_list[i] for i in pick],
           [body[i].double().numpy() for i in pick], out_dtype, exact=True)


@pytest.mark.parametrize("out", [torch.float16, torch.float32])
def test_batched_k_zero(out):
    M, N, batch = 40, 70, 4
    a = [torch.zeros((M, 0), dtype=torch.float16)]
    b = [torch.zeros((0, N), dtype=torch.float16)]
    outs, intact, p = run_batched(a, b, out, 1, 0, N, 0, N + 2, M * (N + 2) + 3, batch)
    assert p == 1 and intact
    for got in outs:
        assert np.all(got == 0)


def test_bmm_binding_and_sampled_large():
    """tg.bmm on 3-D torch tensors: 8 products of 1024^3 on the pair kernel,
    every matrix checked on sampled outputs, plus an expand()ed broadcast B."""
    batch, M, N, K = 8, 1024, 1024, 1024
    a = torch.stack(_mats(batch, (M, K), "uniform", 11600, "f16", K)).cuda()
    b = torch.stack(_mats(batch, (K, N), "uniform", 11700, "f16", K)).cuda()
    c = tg.bmm(a, b)
    tg.check()
    rng = np.random.default_rng(11800)
    r = rng.integers(0, M, 300)
    col = rng.integers(0, N, 300)
    for i in range(batch):
        Cs, Ss = oracle.gemm_at(a[i].cpu().numpy(), b[i].cpu().numpy(), r, col)
        compare(c[i].double().cpu().numpy()[r, col], Cs, Ss, True, f"bmm matrix {i}")
    bb = b[0:1].expand(batch, K, N)
    c2 = tg.bmm(a, bb)
    tg.check()
    for i in (0, batch - 1):
        Cs, Ss = oracle.gemm_at(a[i].cpu().numpy(), b[0].cpu().numpy(), r, col)
        compare(c2[i].double().cpu().numpy()[r, col], Cs, Ss, True, f"broadcast B, matrix {i}")
