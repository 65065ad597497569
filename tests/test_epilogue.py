"""GPU parity of the fused epilogue  C = act(alpha * AB + beta * D + bias).

Every path runs the epilogue in its own kernel, on the fp32 accumulator,
before the output conversion.  The oracle computes the product and the
epilogue in fp64 (act(alpha*C + beta*D + bias[j]), GELU in its erf form) and
the acceptance bound is oracle.epilogue_tolerance: the product's bound
scaled by |alpha|, fp32 rounding of the other terms, an activation slope of
at most 1.13, and the 1e-2 relative term for an fp16 output.  With small
integer operands, power-of-two alpha and integer D and bias, every step is
exact in fp32 and the result must match the oracle bit for bit (ReLU and no
activation; GELU is transcendental and is held to the bound).
"""
import numpy as np
import pytest
import torch

import oracle
import tiled_gemm_tg_gb300 as tg
from tiled_gemm_tg_gb300 import inputs

from gpu_util import compare_ex, f16_bits_of, run, run_ex

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


def forced(path):
    class _Ctx:
        def __enter__(self):
            tg.tg_gemm_force_path(path)

        def __exit__(self, *exc):
            tg.tg_gemm_force_path(0)
    return _Ctx()


EPILOGUES = {
    "scale_bias_relu": dict(alpha=0.5, beta=0.0, use_d=False, use_bias=True, act=tg.ACT_RELU),
    "axpby_bias_gelu": dict(alpha=-1.25, beta=0.75, use_d=True, use_bias=True, act=tg.ACT_GELU),
    "beta_only": dict(alpha=1.0, beta=-1.0, use_d=True, use_bias=False, act=tg.ACT_NONE),
    "gelu_only": dict(alpha=2.0, beta=0.0, use_d=False, use_bias=False, act=tg.ACT_GELU),
}

# path -> (M, N, K, input dtype); N is not a multiple of 32, so every path
# runs its ragged column chunk as well as full ones.
SHAPES = {
    MAIN: (300, 520, 320, "f16"),
    PAIR: (300, 520, 320, "f16"),
    BOUNDARY: (127, 255, 200, "f16"),
    SKINNY: (37, 1000, 700, "f16"),
    SIMT: (77, 130, 45, "f32"),
}


def _operands(M, N, K, dt, dist, seed):
    a = inputs.draw((M, K), dist, seed, dt, k=K)
    b = inputs.draw((K, N), dist, seed + 1, dt, k=K)
    return a, b


def _extras(M, N, out, epi, seed, integer=False):
    rng = np.random.default_rng(seed)
    d = bias = None
    if epi["use_d"]:
        x = rng.integers(-4, 5, (M, N)) if integer else rng.standard_normal((M, N))
        d = torch.from_numpy(x.astype(np.float32)).to(out)
    if epi["use_bias"]:
        bias = (rng.integers(-8, 9, N) if integer else rng.standard_normal(N)).astype(np.float32)
    return d, bias


def _ld(path, n):
    # the boundary path gets row strides that the TMA engine cannot address
    return n + 1 if path == BOUNDARY else (n + 7) // 8 * 8


def _reference(a, b, epi, d, bias):
    C, S = oracle.gemm(a.numpy(), b.numpy())
    cin = None if d is None else d.numpy()
    ref = oracle.epilogue(C, epi["alpha"], epi["beta"], cin, bias, epi["act"])
    return ref, S


@pytest.mark.parametrize("name", sorted(EPILOGUES))
@pytest.mark.parametrize("path", [MAIN, PAIR, BOUNDARY, SKINNY, SIMT])
@pytest.mark.parametrize("out", [torch.float16, torch.float32])
def test_epilogue_every_path(name, path, out):
    M, N, K, dt = SHAPES[path]
    if dt == "f32" and out == torch.float16:
        pytest.skip("the fp32 path writes fp32")
    epi = EPILOGUES[name]
    a, b = _operands(M, N, K, dt, "normal_rsqrtk", 9100 + path)
    d, bias = _extras(M, N, out, epi, 9200 + path)
    with forced(path):
        got, intact, p = run_ex(a, b, out, epi["alpha"], epi["beta"], d, bias, epi["act"],
                                lda=_ld(path, K), ldb=_ld(path, N), ldc=N + 3,
                                ldd=N + 5 if d is not None else None)
    assert p == path and intact
    ref, S = _reference(a, b, epi, d, bias)
    compare_ex(got, ref, S, epi["alpha"], epi["beta"], d, bias, out == torch.float16,
               f"{name} path {path}")


@pytest.mark.parametrize("path", [MAIN, PAIR, BOUNDARY, SKINNY, SIMT])
@pytest.mark.parametrize("out", [torch.float16, torch.float32])
def test_epilogue_integer_bitwise(path, out):
    M, N, K, dt = SHAPES[path]
    if dt == "f32" and out == torch.float16:
        pytest.skip("the fp32 path writes fp32")
    epi = dict(alpha=2.0, beta=-1.0, use_d=True, use_bias=True, act=tg.ACT_RELU)
    a, b = _operands(M, N, K, dt, "int2", 9300 + path)
    d, bias = _extras(M, N, out, epi, 9400 + path, integer=True)
    with forced(path):
        got, intact, p = run_ex(a, b, out, epi["alpha"], epi["beta"], d, bias, epi["act"],
                                lda=_ld(path, K), ldb=_ld(path, N))
    assert p == path and intact
    ref, _ = _reference(a, b, epi, d, bias)
    if out == torch.float16:
        want = f16_bits_of(ref)
        have = f16_bits_of(got)  # got holds fp16 values exactly, so this recovers its bits
        assert np.array_equal(have, want)
    else:
        assert np.array_equal(got, ref)


@pytest.mark.parametrize("path", [MAIN, PAIR, BOUNDARY, SKINNY, SIMT])
def test_epilogue_in_place_accumulate(path):
    """D == C: C = alpha*AB + beta*C, each element read before it is written."""
    M, N, K, dt = SHAPES[path]
    out = torch.float32
    a, b = _operands(M, N, K, dt, "int2", 9500 + path)
    rng = np.random.default_rng(9600 + path)
    c0 = torch.from_numpy(rng.integers(-100, 101, (M, N)).astype(np.float32))
    with forced(path):
        got, intact, p = run_ex(a, b, out, 1.0, 1.0, c0, None, tg.ACT_NONE,
                                lda=_ld(path, K), ldb=_ld(path, N), in_place=True)
    assert p == path and intact
    C, _ = oracle.gemm(a.numpy(), b.numpy())
    assert np.array_equal(got, C + c0.double().numpy())


@pytest.mark.parametrize("out", [torch.float16, torch.float32])
def test_epilogue_unaligned_d_and_bias(out):
    """D and bias that are not 16-byte aligned take the scalar loads."""
    M, N, K = 256, 384, 256
    epi = EPILOGUES["axpby_bias_gelu"]
    a, b = _operands(M, N, K, "f16", "normal_rsqrtk", 9700)
    d, bias = _extras(M, N, out, epi, 9701)
    got, intact, p = run_ex(a, b, out, epi["alpha"], epi["beta"], d, bias, epi["act"],
                            ldd=N + 1, d_off=1, bias_off=1)
    assert p == MAIN and intact
    ref, S = _reference(a, b, epi, d, bias)
    compare_ex(got, ref, S, epi["alpha"], epi["beta"], d, bias, out == torch.float16, "unaligned")


@pytest.mark.parametrize("out", [torch.float16, torch.float32])
def test_epilogue_k_zero(out):
    """K == 0: the product is the empty sum, so C = act(beta*D + bias)."""
    M, N = 70, 300
    epi = dict(alpha=3.0, beta=0.5, use_d=True, use_bias=True, act=tg.ACT_GELU)
    a = torch.zeros((M, 0), dtype=torch.float16)
    b = torch.zeros((0, N), dtype=torch.float16)
    d, bias = _extras(M, N, out, epi, 9800)
    got, intact, p = run_ex(a, b, out, epi["alpha"], epi["beta"], d, bias, epi["act"])
    assert p == 1 and intact
    ref = oracle.epilogue(np.zeros((M, N)), epi["alpha"], epi["beta"], d.numpy(), bias, epi["act"])
    compare_ex(got, ref, np.zeros((M, N)), epi["alpha"], epi["beta"], d, bias,
               out == torch.float16, "K=0")


def test_identity_epilogue_is_tg_gemm_bitwise():
    """alpha 1, beta 0, no bias, no activation is the plain call, bit for bit."""
    a, b = _operands(520, 776, 448, "f16", "normal_rsqrtk", 9900)
    for path in (MAIN, PAIR):
        with forced(path):
            g1, _, p1 = run(a, b, torch.float16)
            g2, _, p2 = run_ex(a, b, torch.float16, 1.0, 0.0, None, None, tg.ACT_NONE)
        assert p1 == p2 == path
        assert np.array_equal(g1, g2)


def test_epilogue_square_8192_sampled():
    """The full-size fp16 workload with bias, beta*D and GELU in the pair kernel;
    whole rows of the output checked against the oracle."""
    w = inputs.WORKLOADS["square_8192"]
    a, b = inputs.operands(w)
    M, N = w.M, w.N
    epi = EPILOGUES["axpby_bias_gelu"]
    d, bias = _extras(M, N, torch.float16, epi, 9950)
    got, intact, p = run_ex(a, b, torch.float16, epi["alpha"], epi["beta"], d, bias, epi["act"])
    assert p == PAIR and intact
    assert np.isfinite(got).all()
    rows = np.array([0, 255, 256, 4097, 8191])
    cols = np.arange(N)
    rr, cc = np.repeat(rows, N), np.tile(cols, len(rows))
    C, S = oracle.gemm_at(a.numpy(), b.numpy(), rr, cc)
    C = C.reshape(len(rows), N)
    S = S.reshape(len(rows), N)
    dsub = d[torch.from_numpy(rows)]
    ref = oracle.epilogue(C, epi["alpha"], epi["beta"], dsub.numpy(), bias, epi["act"])
    compare_ex(got[rows], ref, S, epi["alpha"], epi["beta"], dsub, bias, True, "8192^3 sampled")


@pytest.mark.parametrize("split", [2, 4])
@pytest.mark.parametrize("name", sorted(EPILOGUES))
@pytest.mark.parametrize("out", [torch.float16, torch.float32])
def test_epilogue_split_k(split, name, out):
    """The one-CTA kernel split over K (forced) applies the fused epilogue in
    its cluster reduction, once per element after the partials are added."""
    M, N, K, dt = 300, 520, 1000, "f16"
    epi = EPILOGUES[name]
    a, b = _operands(M, N, K, dt, "normal_rsqrtk", 9800 + split)
    d, bias = _extras(M, N, out, epi, 9810 + split)
    assert tg.tg_gemm_force_split_k(split) == tg.TG_OK
    try:
        with forced(MAIN):
            got, intact, p = run_ex(a, b, out, epi["alpha"], epi["beta"], d, bias, epi["act"],
                                    lda=_ld(MAIN, K), ldb=_ld(MAIN, N), ldc=N + 3,
                                    ldd=N + 5 if d is not None else None)
    finally:
        tg.tg_gemm_force_split_k(0)
    assert p == MAIN and intact
    ref, S = _reference(a, b, epi, d, bias)
    compare_ex(got, ref, S, epi["alpha"], epi["beta"], d, bias, out == torch.float16,
               f"{name} split {split}")


def test_epilogue_split_k_in_place_integer():
    """Split over K with D == C (C = AB + C), integer values: exact."""
    M, N, K = 256, 264, 2048
    a, b = _operands(M, N, K, "f16", "int2", 9820)
    rng = np.random.default_rng(9821)
    c0 = torch.from_numpy(rng.integers(-100, 101, (M, N)).astype(np.float32))
    assert tg.tg_gemm_force_split_k(8) == tg.TG_OK
    try:
        with forced(MAIN):
            got, intact, p = run_ex(a, b, torch.float32, 1.0, 1.0, c0, None, tg.ACT_NONE,
                                    lda=_ld(MAIN, K), ldb=_ld(MAIN, N), in_place=True)
    finally:
        tg.tg_gemm_force_split_k(0)
    assert p == MAIN and intact
    C, _ = oracle.gemm(a.numpy(), b.numpy())
    assert np.array_equal(got, C + c0.double().numpy())
