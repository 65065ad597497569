"""Pins for the CPU oracle, checked against facts that do not come from it.

Each pin would fail for a plausible mistake in the oracle: a wrong exponent
bias or subnormal scale in the binary16 decoder, round-half-away instead of
ties-to-even or an fp32 detour in the encoder, a dropped term, a wrong sign,
a transposed operand or an ignored leading dimension in the product, or a
missing absolute value in S.  test_planted_mistakes_are_caught builds such
mutants of the oracle's C source and checks that the pins reject each one.
"""
import os
import re
import subprocess

import numpy as np
import pytest

import oracle
from oracle import Oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _read_blocks(path):
    blocks, cur = {}, None
    with open(path) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            if re.fullmatch(r"[A-Za-z]+", line):
                cur = line
                blocks[cur] = []
            else:
                blocks[cur].append([float(v) for v in line.split()])
    return {k: np.array(v) for k, v in blocks.items()}


def _read_ties():
    rows = []
    with open(os.path.join(GOLDEN, "f16_ties.txt")) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            tok = line.split()
            x = float.fromhex(tok[0]) if "0x" in tok[0] else float(tok[0])
            rows.append((x, int(tok[1], 16)))
    return rows


# ---------------------------------------------------------------- pins, as
# functions of an Oracle so the mutation test can run them on mutants.

def pin_decode_exhaustive(o: Oracle):
    bits = np.arange(65536, dtype=np.uint16)
    got = o.f16_bits_to_f64(bits)
    ref = bits.view(np.float16).astype(np.float64)  # NumPy's own binary16 conversion
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])
    # sign of zero
    assert np.signbit(got[0x8000]) and not np.signbit(got[0x0000])


def pin_decode_by_hand(o: Oracle):
    cases = {0x3c00: 1.0, 0x0001: 2.0 ** -24, 0x0400: 2.0 ** -14, 0x03ff: 1023 * 2.0 ** -24,
             0x7bff: 65504.0, 0xc000: -2.0, 0x3555: 0x555 * 2.0 ** -12,
             0x7c00: np.inf, 0xfc00: -np.inf}
    got = o.f16_bits_to_f64(np.array(list(cases), dtype=np.uint16))
    assert np.array_equal(got, np.array(list(cases.values())))


def pin_encode_ties(o: Oracle):
    ties = _read_ties()
    got = o.f64_to_f16_bits(np.array([x for x, _ in ties]))
    want = np.array([h for _, h in ties], dtype=np.uint16)
    bad = [(ties[i][0].hex(), hex(got[i]), hex(want[i])) for i in np.flatnonzero(got != want)]
    assert not bad, bad


def pin_encode_vs_numpy(o: Oracle):
    rng = np.random.default_rng(7)
    parts = [rng.standard_normal(20000) * s for s in (1e-7, 1e-5, 1e-3, 1.0, 1e2, 1e4, 6e4)]
    parts.append(rng.uniform(-70000, 70000, 20000))
    x = np.concatenate(parts)
    got = o.f64_to_f16_bits(x)
    with np.errstate(over="ignore"):
        ref = x.astype(np.float16).view(np.uint16)
    assert np.array_equal(got, ref)


def pin_roundtrip(o: Oracle):
    bits = np.arange(65536, dtype=np.uint16)
    vals = o.f16_bits_to_f64(bits)
    keep = ~np.isnan(vals)
    assert np.array_equal(o.f64_to_f16_bits(vals[keep]), bits[keep])


def pin_gemm_4x4(o: Oracle):
    g = _read_blocks(os.path.join(GOLDEN, "gemm_4x4_int.txt"))
    for dt in (np.float16, np.float32):
        C, S = o.gemm(g["A"].astype(dt), g["B"].astype(dt))
        assert np.array_equal(C, g["C"])
        assert np.array_equal(S, g["S"])


def pin_gemm_8x8_ones(o: Oracle):
    spec = {}
    with open(os.path.join(GOLDEN, "gemm_8x8_ones.txt")) as f:
        for line in f:
            line = line.split("#", 1)[0].split()
            if line:
                spec[line[0]] = int(line[1])
    a = np.ones((spec["M"], spec["K"]), np.float16)
    b = np.ones((spec["K"], spec["N"]), np.float16)
    C, S = o.gemm(a, b)
    assert np.all(C == spec["value"]) and np.all(S == spec["value"])


def pin_closed_forms(o: Oracle):
    rng = np.random.default_rng(1)
    # identity B: C = A exactly (each row sums one exact product and zeros)
    a = rng.standard_normal((37, 29)).astype(np.float16)
    C, _ = o.gemm(a, np.eye(29, dtype=np.float16))
    assert np.array_equal(C, a.astype(np.float64))
    # all-ones: C = K
    C, S = o.gemm(np.ones((5, 300), np.float16), np.ones((300, 7), np.float16))
    assert np.all(C == 300) and np.all(S == 300)
    # diagonal A scales the rows of B
    d = rng.standard_normal(23).astype(np.float16)
    b = rng.standard_normal((23, 19)).astype(np.float16)
    C, _ = o.gemm(np.diag(d), b)
    assert np.array_equal(C, d.astype(np.float64)[:, None] * b.astype(np.float64))
    # a single nonzero A entry picks one row of B at one output row
    a = np.zeros((6, 11), np.float16)
    a[4, 9] = -3
    b = rng.standard_normal((11, 13)).astype(np.float16)
    C, _ = o.gemm(a, b)
    want = np.zeros((6, 13))
    want[4] = -3 * b[9].astype(np.float64)
    assert np.array_equal(C, want)


def pin_transpose(o: Oracle):
    rng = np.random.default_rng(2)
    a = rng.standard_normal((21, 34)).astype(np.float16)
    b = rng.standard_normal((34, 13)).astype(np.float16)
    C, S = o.gemm(a, b)
    Ct, St = o.gemm(np.ascontiguousarray(b.T), np.ascontiguousarray(a.T))
    assert np.array_equal(C, Ct.T) and np.array_equal(S, St.T)


def pin_vs_numpy_exact(o: Oracle):
    rng = np.random.default_rng(3)
    a = rng.integers(-3, 4, (45, 70)).astype(np.float16)
    b = rng.integers(-3, 4, (70, 33)).astype(np.float16)
    C, S = o.gemm(a, b)
    A, B = a.astype(np.float64), b.astype(np.float64)
    assert np.array_equal(C, A @ B)
    assert np.array_equal(S, np.abs(A) @ np.abs(B))


def pin_vs_numpy_random(o: Oracle):
    rng = np.random.default_rng(4)
    for dt in (np.float16, np.float32):
        a = rng.standard_normal((50, 130)).astype(dt)
        b = rng.standard_normal((130, 41)).astype(dt)
        C, S = o.gemm(a, b)
        ref = a.astype(np.float64) @ b.astype(np.float64)
        assert np.all(np.abs(C - ref) <= 1e-13 * S)
        assert np.allclose(S, np.abs(a.astype(np.float64)) @ np.abs(b.astype(np.float64)),
                           rtol=1e-13, atol=0)


def pin_leading_dims(o: Oracle):
    rng = np.random.default_rng(5)
    big_a = rng.standard_normal((40, 64)).astype(np.float16)
    big_b = rng.standard_normal((60, 72)).astype(np.float16)
    a, b = big_a[:31, 3:50], big_b[7:54, 5:66]  # row strides exceed row lengths
    C, S = o.gemm(a, b)
    ref = a.astype(np.float64) @ b.astype(np.float64)
    assert np.all(np.abs(C - ref) <= 1e-13 * S)
    C2, S2 = o.gemm(np.ascontiguousarray(a), np.ascontiguousarray(b))
    assert np.array_equal(C, C2) and np.array_equal(S, S2)


def pin_sampled(o: Oracle):
    rng = np.random.default_rng(6)
    a = rng.standard_normal((33, 57)).astype(np.float16)
    b = rng.standard_normal((57, 29)).astype(np.float16)
    C, S = o.gemm(a, b)
    r = rng.integers(0, 33, 200)
    c = rng.integers(0, 29, 200)
    Cs, Ss = o.gemm_at(a, b, r, c)
    assert np.array_equal(Cs, C[r, c]) and np.array_equal(Ss, S[r, c])
    ref = np.einsum("tk,kt->t", a[r].astype(np.float64), b[:, c].astype(np.float64))
    assert np.all(np.abs(Cs - ref) <= 1e-13 * Ss)


def pin_degenerate(o: Oracle):
    C, S = o.gemm(np.zeros((3, 0), np.float16), np.zeros((0, 5), np.float16))
    assert C.shape == (3, 5) and np.all(C == 0) and np.all(S == 0)
    C, S = o.gemm(np.zeros((0, 4), np.float16), np.zeros((4, 5), np.float16))
    assert C.shape == (0, 5)


# ------------------------------------------------------------- FP8 E4M3 pins

def pin_e4m3_decode_exhaustive(o: Oracle):
    # all 256 patterns against PyTorch's own float8_e4m3fn conversion
    torch = pytest.importorskip("torch")
    bits = np.arange(256, dtype=np.uint8)
    got = o.e4m3_bits_to_f64(bits)
    ref = torch.from_numpy(bits).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan) and nan.sum() == 2
    assert np.array_equal(got[~nan], ref[~nan])


def pin_e4m3_decode_by_hand(o: Oracle):
    # the format's defining values: 1.0, the largest finite 448 = 1.75 * 2^8,
    # the smallest normal 2^-6, the smallest subnormal 2^-9, signed zero
    cases = {0x38: 1.0, 0x7E: 448.0, 0x08: 2.0 ** -6, 0x01: 2.0 ** -9, 0x07: 7 * 2.0 ** -9,
             0xC0: -2.0, 0x3C: 1.5, 0x00: 0.0}
    got = o.e4m3_bits_to_f64(np.array(list(cases), dtype=np.uint8))
    assert np.array_equal(got, np.array(list(cases.values())))
    assert np.signbit(o.e4m3_bits_to_f64(np.array([0x80], np.uint8))[0])
    assert np.isnan(o.e4m3_bits_to_f64(np.array([0x7F, 0xFF], np.uint8))).all()
    assert o.e4m3_bits_to_f64(np.array([0x7C], np.uint8))[0] == 384.0  # no infinities


def pin_e4m3_gemm_exact(o: Oracle):
    # E4M3 operands with small-integer values: the product equals NumPy's on
    # the decoded values exactly, and the same matrices in fp16 give the same C
    rng = np.random.default_rng(12)
    vals = np.array([0x00, 0x38, 0x40, 0xB8, 0xC0, 0x44, 0xC4], np.uint8)  # 0, 1, 2, -1, -2, 3, -3
    a = vals[rng.integers(0, len(vals), (19, 37))]
    b = vals[rng.integers(0, len(vals), (37, 23))]
    C, S = o.gemm(a, b)
    A, B = o.e4m3_bits_to_f64(a), o.e4m3_bits_to_f64(b)
    assert set(np.unique(A)) <= {0.0, 1.0, 2.0, -1.0, -2.0, 3.0, -3.0}
    assert np.array_equal(C, A @ B) and np.array_equal(S, np.abs(A) @ np.abs(B))
    C16, _ = o.gemm(A.astype(np.float16), B.astype(np.float16))
    assert np.array_equal(C, C16)


# ------------------------------------------------------------ attention pins

def _softmax_rows(x):
    x = x - x.max(axis=1, keepdims=True)
    e = np.exp(x)
    return e / e.sum(axis=1, keepdims=True)


def pin_attention_vs_scipy(o: Oracle):
    # SciPy's softmax of NumPy's logits, times V: an independent formulation
    special = pytest.importorskip("scipy.special")
    rng = np.random.default_rng(20)
    for (Nq, Nk, d, dv, scale) in [(9, 13, 16, 5, 0.25), (4, 70, 40, 24, 1.0)]:
        q = rng.standard_normal((Nq, d)).astype(np.float16)
        k = rng.standard_normal((Nk, d)).astype(np.float16)
        v = rng.standard_normal((Nk, dv)).astype(np.float16)
        O, E, G = o.attention(q, k, v, scale)
        S = scale * (q.astype(np.float64) @ k.astype(np.float64).T)
        W = special.softmax(S, axis=1)
        assert np.allclose(O, W @ v.astype(np.float64), rtol=0, atol=1e-13)
        assert np.allclose(E, W @ np.abs(v.astype(np.float64)), rtol=0, atol=1e-13)
        assert np.allclose(G, np.abs(scale) * (np.abs(q.astype(np.float64)) @
                                               np.abs(k.astype(np.float64)).T).max(axis=1))


def pin_attention_closed_forms(o: Oracle):
    rng = np.random.default_rng(21)
    # all keys equal: uniform weights, O = mean of the V rows (exact: 8 keys)
    q = rng.standard_normal((6, 32)).astype(np.float16)
    k = np.tile(rng.standard_normal((1, 32)), (8, 1)).astype(np.float16)
    v = rng.integers(-4, 5, (8, 5)).astype(np.float16)
    O, E, _ = o.attention(q, k, v)
    assert np.array_equal(O, np.tile(v.astype(np.float64).mean(axis=0), (6, 1)))
    # one key dominates by a gap of ~1000 in the logit: O is that key's V row
    k = np.zeros((9, 4), np.float16)
    k[5] = [10, 10, 10, 10]
    q = np.full((3, 4), 25, np.float16)
    v = rng.standard_normal((9, 6)).astype(np.float16)
    O, _, _ = o.attention(q, k, v)
    assert np.array_equal(O, np.tile(v[5].astype(np.float64), (3, 1)))
    # V of ones: the weights sum to one
    q = rng.standard_normal((5, 8)).astype(np.float16)
    k = rng.standard_normal((11, 8)).astype(np.float16)
    O, E, _ = o.attention(q, k, np.ones((11, 3), np.float16), 2.0)
    assert np.allclose(O, 1.0, atol=1e-14) and np.allclose(E, 1.0, atol=1e-14)


def pin_attention_invariants(o: Oracle):
    rng = np.random.default_rng(22)
    q = rng.standard_normal((7, 12)).astype(np.float16)
    k = rng.standard_normal((10, 12)).astype(np.float16)
    v = rng.standard_normal((10, 4)).astype(np.float16)
    O, _, _ = o.attention(q, k, v, 0.5)
    # permuting the keys together with their values changes nothing
    perm = rng.permutation(10)
    Op, _, _ = o.attention(q, k[perm], v[perm], 0.5)
    assert np.allclose(Op, O, atol=1e-14)
    # a shift shared by every key moves each row's logits by a constant
    # (integer keys and shift, so the shifted keys are exact in fp16)
    ki = rng.integers(-3, 4, (10, 12)).astype(np.float16)
    shift = np.array([1, -1, 2, 0, 0, 2, 0, 0, -3, 0, 1, 0], np.float16)
    Oa, _, _ = o.attention(q, ki, v, 0.5)
    Ob, _, _ = o.attention(q, ki + shift, v, 0.5)
    assert np.allclose(Ob, Oa, atol=1e-13)
    # rows are independent: one query row alone gives the same output row
    O1, _, _ = o.attention(q[3:4], k, v, 0.5)
    assert np.array_equal(O1[0], O[3])
    # row strides larger than the rows (sub-matrix views) read the same values
    big_q = rng.standard_normal((9, 20)).astype(np.float16)
    big_k = rng.standard_normal((14, 17)).astype(np.float16)
    big_v = rng.standard_normal((12, 9)).astype(np.float16)
    qs, ks, vs = big_q[1:8, 2:14], big_k[2:12, 3:15], big_v[1:11, 4:8]
    Os, _, _ = o.attention(qs, ks, vs, 0.5)
    Oc, _, _ = o.attention(np.ascontiguousarray(qs), np.ascontiguousarray(ks),
                           np.ascontiguousarray(vs), 0.5)
    assert np.array_equal(Os, Oc)


def pin_attention_page_recurrence(o: Oracle):
    # The blockwise recurrence of the TileLang page (running maximum M and
    # normaliser L, blocks of keys), carried out in fp64 in Python on the
    # page's 1024-key shape reduced to 96 keys: it reaches the definition.
    rng = np.random.default_rng(23)
    Nq, Nk, d, blk = 5, 96, 24, 32
    q = rng.standard_normal((Nq, d)).astype(np.float16)
    k = rng.standard_normal((Nk, d)).astype(np.float16)
    v = rng.standard_normal((Nk, 7)).astype(np.float16)
    Q, K, V = (x.astype(np.float64) for x in (q, k, v))
    Ob = np.zeros((Nq, 7))
    L = np.zeros(Nq)
    M = np.full(Nq, -1e9)
    for b0 in range(0, Nk, blk):
        S = Q @ K[b0:b0 + blk].T
        m_new = np.maximum(M, S.max(axis=1))
        l_new = L * np.exp(M - m_new) + np.exp(S - m_new[:, None]).sum(axis=1)
        Ob = (Ob * (L * np.exp(M - m_new))[:, None] +
              np.exp(S - m_new[:, None]) @ V[b0:b0 + blk]) / l_new[:, None]
        L, M = l_new, m_new
    O, _, _ = o.attention(q, k, v, 1.0)
    assert np.allclose(O, Ob, rtol=0, atol=1e-12)


# ----------------------------------------------------- fused epilogue pins

def pin_epilogue_plain(o: Oracle):
    # alpha 1, beta 0, no bias, no activation: the product itself, bit for bit
    rng = np.random.default_rng(8)
    C = rng.standard_normal((9, 14))
    assert np.array_equal(o.epilogue(C), C)


def pin_epilogue_block_identity(o: Oracle):
    # alpha*A@B + beta*D + 1 bias^T is the product of the block matrices
    # [alpha*A | beta*I_M | 1] and [B; D; bias^T]; with small integers and
    # power-of-two scales every term is exact in fp64.  M != N, so a bias
    # indexed by row or a transposed D cannot pass; D is a strided view.
    rng = np.random.default_rng(9)
    M, N, K = 11, 17, 23
    a = rng.integers(-3, 4, (M, K)).astype(np.float16)
    b = rng.integers(-3, 4, (K, N)).astype(np.float16)
    big = rng.integers(-4, 5, (M + 2, N + 9)).astype(np.float16)
    d = big[1:M + 1, 4:N + 4]
    bias = rng.integers(-5, 6, N).astype(np.float32)
    alpha, beta = 0.75, -1.5
    C, _ = o.gemm(a, b)
    got = o.epilogue(C, alpha, beta, d, bias, act=0)
    left = np.hstack([alpha * a.astype(np.float64), beta * np.eye(M), np.ones((M, 1))])
    right = np.vstack([b.astype(np.float64), d.astype(np.float64), bias[None, :].astype(np.float64)])
    assert np.array_equal(got, left @ right)
    # the same with an fp32 D and no bias: the bias row drops out
    d32 = rng.integers(-4, 5, (M, N)).astype(np.float32)
    got = o.epilogue(C, alpha, beta, d32, None, act=0)
    assert np.array_equal(got, np.hstack([alpha * a.astype(np.float64), beta * np.eye(M)]) @
                          np.vstack([b.astype(np.float64), d32.astype(np.float64)]))


def pin_gelu_normal_cdf(o: Oracle):
    # GELU(x) = x * Phi(x); Phi from SciPy's ndtr (an independent routine).
    # Phi(0) = 1/2 exactly, so GELU(0) = 0; Phi(1) = 0.8413447460685429...
    special = pytest.importorskip("scipy.special")
    x = np.concatenate([np.linspace(-8, 8, 161), [-1.0, 0.0, 1.0, 1.959963984540054]])
    got = o.epilogue(x[None, :], act=2)[0]
    want = x * special.ndtr(x)
    assert np.all(np.abs(got - want) <= 1e-15 * np.abs(x) + 1e-300)
    assert got[-3] == 0.0
    assert abs(got[-2] - 0.8413447460685429) < 1e-15


def pin_activation_odd_parts(o: Oracle):
    # Phi(x) + Phi(-x) = 1 gives GELU(x) - GELU(-x) = x; ReLU(x) - ReLU(-x) = x
    # and ReLU(x) >= 0.  A flipped sign or a wrong erf scale breaks these.
    rng = np.random.default_rng(10)
    x = rng.standard_normal(500) * 3
    for act in (1, 2):
        p = o.epilogue(x[None, :], act=act)[0]
        n = o.epilogue(-x[None, :], act=act)[0]
        assert np.allclose(p - n, x, rtol=0, atol=1e-14 * (1 + np.abs(x)).max())
    r = o.epilogue(x[None, :], act=1)[0]
    assert np.all(r >= 0) and np.array_equal(r[x > 0], x[x > 0])
    # GELU lies between min(x, 0) and max(x, 0)
    g = o.epilogue(x[None, :], act=2)[0]
    assert np.all(g <= np.maximum(x, 0) + 1e-15) and np.all(g >= np.minimum(x, 0) - 1e-15)


PINS = [pin_decode_exhaustive, pin_decode_by_hand, pin_encode_ties, pin_encode_vs_numpy,
        pin_roundtrip, pin_gemm_4x4, pin_gemm_8x8_ones, pin_closed_forms, pin_transpose,
        pin_vs_numpy_exact, pin_vs_numpy_random, pin_leading_dims, pin_sampled,
        pin_degenerate, pin_e4m3_decode_exhaustive, pin_e4m3_decode_by_hand,
        pin_e4m3_gemm_exact, pin_attention_vs_scipy, pin_attention_closed_forms,
        pin_attention_invariants, pin_attention_page_recurrence, pin_epilogue_plain, pin_epilogue_block_identity, pin_gelu_normal_cdf,
        pin_activation_odd_parts]


@pytest.fixture(scope="module")
def o():
    return oracle._default()


@pytest.mark.parametrize("pin", PINS, ids=lambda p: p.__name__)
def test_pin(o, pin):
    pin(o)


def test_tolerance_formula():
    C = np.array([1.0, -2.0, 0.0])
    S = np.array([3.0, 4.0, 5.0])
    assert np.allclose(oracle.tolerance(C, S, False), 2e-3 * S + 1e-5)
    assert np.allclose(oracle.tolerance(C, S, True), 2e-3 * S + 1e-5 + 1e-2 * np.abs(C))


def test_epilogue_tolerance_terms():
    out = np.array([[2.0, -1.0]])
    S = np.array([[4.0, 8.0]])
    plain = oracle.epilogue_tolerance(out, S, 1.0, 0.0, None, None, False)
    assert np.allclose(plain, 1.13 * (2e-3 * S + 1e-5) + 1e-6)
    scaled = oracle.epilogue_tolerance(out, S, -2.0, 0.5, np.array([[4.0, 0.0]]),
                                       np.array([1.0, 3.0]), True)
    want = 1.13 * (2.0 * (2e-3 * S + 1e-5) + 1e-6 * np.array([[2.0, 0.0]]) +
                   1e-6 * np.array([[1.0, 3.0]])) + 1e-6 + 1e-2 * np.abs(out)
    assert np.allclose(scaled, want)


def test_threads_reported(o):
    assert o.num_threads() >= 1


# ------------------------------------------------------------ planted mistakes

MUTANTS = {
    "decode_bias": ("(double)(1024 + f), e - 25)", "(double)(1024 + f), e - 24)"),
    "decode_subnormal": ("v = ldexp((double)f, -24);", "v = ldexp((double)f, -25);"),
    "encode_half_away": ("double q = nearbyint(ldexp(a, 10 - E));",
                         "double q = round(ldexp(a, 10 - E));"),
    "encode_fp32_detour": ("double a = fabs(x);", "double a = (double)(float)fabs(x);"),
    "product_sign": ("c[j] += p;", "c[j] -= p;"),
    "dropped_term": ("for (int64_t k = 0; k < K; ++k) {\n            double a =",
                     "for (int64_t k = 1; k < K; ++k) {\n            double a ="),
    "ignored_lda": ("double a = load_elem(A, i * lda + k, in_dtype);",
                    "double a = load_elem(A, i * K + k, in_dtype);"),
    "missing_abs": ("s[j] += fabs(p);", "s[j] += p;"),
    "e4m3_bias": ("(double)(8 + f), e - 10)", "(double)(8 + f), e - 11)"),
    "e4m3_subnormal": ("v = ldexp((double)f, -9);", "v = ldexp((double)f, -10);"),
    "e4m3_no_nan": ("if (e == 0xf && f == 0x7) {", "if (e == 0xf && f == 0x8) {"),
    "attention_no_scale": ("s[j] = scale * acc;", "s[j] = acc;"),
    "attention_v_transposed": ("o += s[j] * Vd[j * dv + c];", "o += s[j] * Vd[(c % Nk) * dv + (j % dv)];"),
    "attention_no_normalise": ("O[i * dv + c] = o / l;", "O[i * dv + c] = o;"),
    "attention_max_not_subtracted": ("s[j] = exp(s[j] - m);", "s[j] = exp(s[j]);"),
    "attention_k_row_stride": ("Kd[j * d + c] = load_elem(K, j * ldk + c, in_dtype);",
                               "Kd[j * d + c] = load_elem(K, j * d + c, in_dtype);"),
    "epilogue_alpha_dropped": ("double y = alpha * C[i * N + j];", "double y = C[i * N + j];"),
    "epilogue_beta_sign": ("y += beta * load_elem(", "y -= beta * load_elem("),
    "epilogue_ignored_ldcin": ("load_elem(Cin, i * ldcin + j, cin_dtype)",
                               "load_elem(Cin, i * N + j, cin_dtype)"),
    "epilogue_bias_by_row": ("y += (double)bias[j];", "y += (double)bias[i % N];"),
    "epilogue_relu_min": ("y = y > 0.0 ? y : 0.0;", "y = y < 0.0 ? y : 0.0;"),
    "epilogue_gelu_scale": ("erf(y / sqrt(2.0))", "erf(y * sqrt(2.0))"),
    "epilogue_gelu_tanh": ("0.5 * y * (1.0 + erf(y / sqrt(2.0)))",
                           "0.5 * y * (1.0 + tanh(0.7978845608 * (y + 0.044715 * y * y * y)))"),
    "transposed_b": ("Bd[k * N + j] = load_elem(B, k * ldb + j, in_dtype);",
                     "Bd[k * N + j] = load_elem(B, (j % K) * ldb + (k % N), in_dtype);"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistakes_are_caught(name, tmp_path):
    src = open(os.path.join(os.path.dirname(oracle.__file__), "tg_oracle.c")).read()
    old, new = MUTANTS[name]
    assert src.count(old) == 1, f"mutation anchor for {name} not found"
    path = tmp_path / "mutant.c"
    path.write_text(src.replace(old, new))
    lib = tmp_path / "libmutant.so"
    subprocess.run(["gcc", "-O1", "-std=c11", "-shared", "-fPIC", "-ffp-contract=off",
                    str(path), "-o", str(lib), "-lm"], check=True)
    mutant = Oracle(str(lib))
    caught = []
    for pin in PINS:
        try:
            pin(mutant)
        except AssertionError:
            caught.append(pin.__name__)
    assert caught, f"no pin caught the planted mistake {name}"
