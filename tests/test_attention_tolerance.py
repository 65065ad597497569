"""Pins for the attention acceptance bound (CPU only).

``oracle.attention_tolerance`` is the per-element bound every attention
parity test applies between a tensor-core forward pass and the oracle's fp64
definition of softmax(scale Q K^T) V (the FlashAttention section, §4.1-4.2,
of "TileLang实战：用Python DSL自动生成高性能GPU计算内核", gsyq.cn).  The
blockwise recurrence of that section reaches the definition only up to
rounding, so the bound is derived from the arithmetic, not printed on the
page.  These tests pin it from both sides:

* an emulation of the kernels' arithmetic in NumPy (below) stays inside the
  bound on adversarial inputs: long key sequences, logits near +-80, a
  maximum that keeps growing, logits that cancel from large partial sums,
  probabilities held up to 2^8 by a stale maximum, and a split of the keys
  into ranges merged afterwards;
* the bound is not loose where it matters: with its logit term or its
  per-key summation term removed, some case violates it, and a variant of
  the emulation that forgets to rescale the output when the maximum grows
  is rejected.

The emulation models the kernels' operations one by one, each in the
precision the hardware uses:
  logits     fp16 x fp16 products (exact in fp32) summed in fp32, one key at
             a time (any summation order is covered by the same bound);
  maximum    running maximum m of the base-2 scaled logits, raised only when
             a 128-key block's maximum exceeds it by more than 8;
  weights    p = fp16(2^(fma(s, scale log2 e, -m))), the power of two with a
             relative error of up to 2^-22 (the approximate exp2 unit);
  rescale    O and L multiplied by 2^(m_old - m_new) in fp32 when m rises;
  sums       O += p v and L += p in fp32 (p v exact in fp32), key by key;
  output     O * (1 / L) in fp32, then fp16 round-to-nearest-even;
  key split  each key range keeps its own (O, m, L); the merge takes
             w_r = 2^(m_r - max m), L = sum w_r L_r and O = sum w_r O_r
             with fused multiply-adds in range order.
"""
from __future__ import annotations

import numpy as np
import pytest

import oracle

F32 = np.float32
LOG2E = F32(1.4426950408889634)
BLOCK = 128
EX2_REL_ERR = 2.0 ** -22


def _f32(x):
    return np.asarray(x, dtype=np.float64).astype(F32)


def _ex2(x, rng):
    """2^x rounded to fp32 with a relative error of up to EX2_REL_ERR in a
    random direction per element (2^-inf = 0)."""
    x = np.asarray(x, dtype=np.float64)
    with np.errstate(over="ignore"):  # only the planted mistake overflows
        y = np.exp2(x)
    sign = rng.choice([-1.0, 1.0], size=y.shape)
    return _f32(y * (1.0 + EX2_REL_ERR * sign))


def _fma(a, b, c):
    """fp32 fused multiply-add: a*b exact in fp64 for fp32 operands, one rounding."""
    return _f32(np.asarray(a, np.float64) * np.asarray(b, np.float64) + np.asarray(c, np.float64))


def _seq_sum(start, terms):
    """start + terms[:, 0] + terms[:, 1] + ... in fp32, one rounding per add.
    start: (rows, ...) fp32; terms: (rows, n, ...) fp32."""
    seq = np.concatenate([start[:, None], terms], axis=1).astype(F32)
    return np.add.accumulate(seq, axis=1, dtype=F32)[:, -1]


def _logits_fp32(q16, k16):
    """Raw scores Q K^T: exact fp16 products summed in fp32, one d at a time."""
    qf = q16.astype(np.float64)
    kf = k16.astype(np.float64)
    s = np.zeros((q16.shape[0], k16.shape[0]), dtype=F32)
    for t in range(q16.shape[1]):
        s = (s + _f32(qf[:, t, None] * kf[None, :, t])).astype(F32)
    return s


def _range_pass(raw, v16, sl2, rng, drop_rescale):
    """One key range: the blockwise recurrence with the deferred maximum.
    Returns the unnormalised O (rows x dv), m and L, all fp32."""
    rows = raw.shape[0]
    dv = v16.shape[1]
    m = np.full(rows, -np.inf, dtype=F32)
    O = np.zeros((rows, dv), dtype=F32)
    L = np.zeros(rows, dtype=F32)
    vf = v16.astype(np.float64)
    pos = sl2 >= 0
    for j0 in range(0, raw.shape[1], BLOCK):
        blk = raw[:, j0:j0 + BLOCK]
        ext = blk.max(axis=1) if pos else blk.min(axis=1)
        mx = _f32(ext.astype(np.float64) * float(sl2))
        rise = mx > _f32(m.astype(np.float64) + 8.0)
        alpha = np.where(rise, _ex2(m.astype(np.float64) - mx, rng), F32(1.0)).astype(F32)
        m = np.where(rise, mx, m).astype(F32)
        a = _fma(blk, sl2, -m[:, None])
        p16 = _ex2(a, rng).astype(np.float16)
        if not drop_rescale:
            O = (O * alpha[:, None]).astype(F32)
            L = (L * alpha).astype(F32)
        pf = p16.astype(np.float64)
        terms = _f32(pf[:, :, None] * vf[None, j0:j0 + BLOCK, :])  # exact products
        O = _seq_sum(O, terms)
        L = _seq_sum(L, pf.astype(F32))
    return O, m, L


def emulate(q16, k16, v16, scale, out_f16, ranges=1, drop_rescale=False, seed=0):
    """The kernels' arithmetic for one head (see the module docstring)."""
    rng = np.random.default_rng(seed)
    sl2 = F32(F32(scale) * LOG2E)
    raw = _logits_fp32(q16, k16)
    nk = k16.shape[0]
    nblk = -(-nk // BLOCK)
    edges = [BLOCK * (nblk * r // ranges) for r in range(ranges + 1)]
    parts = [_range_pass(raw[:, a:min(b, nk)], v16[a:min(b, nk)], sl2, rng, drop_rescale)
             for a, b in zip(edges[:-1], edges[1:]) if a < nk]
    if len(parts) == 1:
        O, _, L = parts[0]
    else:
        mm = np.max(np.stack([p[1] for p in parts]), axis=0)
        L = np.zeros_like(parts[0][2])
        O = np.zeros_like(parts[0][0])
        for Op, mp, Lp in parts:
            w = _ex2(mp.astype(np.float64) - mm, rng)
            L = _fma(w, Lp, L)
            O = _fma(w[:, None], Op, O)
    inv = _f32(1.0 / L.astype(np.float64))  # IEEE division: correctly rounded
    out = (O * inv[:, None]).astype(F32)
    return out.astype(np.float16).astype(np.float64) if out_f16 else out.astype(np.float64)


def _bound(O, E, G, d, nk, out_f16, drop=None):
    """oracle.attention_tolerance, or a version of it with one term removed
    (restated here only for the removal; the full form is the oracle's)."""
    if drop is None:
        return oracle.attention_tolerance(O, E, G, d, nk, out_f16)
    dS = (d + 8) * 2.0 ** -23 * np.asarray(G, dtype=np.float64)[:, None]
    terms = {"dS": 2.5 * dS, "fp16_p": 2.0 ** -10, "nk": nk * 2.0 ** -23}
    terms[drop] = 0.0
    t = E * (terms["dS"] + terms["fp16_p"] + terms["nk"]) + 1e-5
    if out_f16:
        t = t + 1e-2 * np.abs(O)
    return t


# ----------------------------------------------------------------- the cases

def _normal(shape, seed, std=1.0):
    return (np.random.default_rng(seed).standard_normal(shape) * std).astype(np.float16)


def case_page_head():
    """The page's own test head, a slice of its query rows: 1024 keys,
    d_model 768, N(0,1), no 1/sqrt(d) factor (logits of magnitude ~28)."""
    q = _normal((16, 768), 1)
    k = _normal((1024, 768), 2)
    v = _normal((1024, 768), 3)
    return q, k, v, 1.0


def case_logits_near_80():
    """Logits spread over about +-80 (each row's maximum near 80)."""
    rng = np.random.default_rng(4)
    q = np.full((8, 64), 1.25, dtype=np.float16)
    k = (rng.uniform(-1.0, 1.0, (640, 64))).astype(np.float16)
    v = _normal((640, 96), 5)
    return q, k, v, 1.0


def case_growing_maximum():
    """The maximum rises block after block (by 5 to 40 in base 2), so the
    stale maximum is kept through some blocks and replaced in others."""
    rng = np.random.default_rng(6)
    nk = 12 * BLOCK
    q = np.ones((6, 16), dtype=np.float16)
    base = np.repeat(np.cumsum(rng.uniform(3.5, 28.0, 12)), BLOCK)
    jitter = rng.uniform(-2.0, 2.0, nk)
    logit = (base + jitter) / np.float64(LOG2E)  # natural-log units
    k = np.zeros((nk, 16), dtype=np.float16)
    k[:, 0] = (logit / 1.0).astype(np.float16)
    v = _normal((nk, 64), 7)
    return q, k, v, 1.0


def case_stale_max_weights_up_to_256():
    """Every later block sits 7.9 (base 2) above the first: the maximum is
    never raised and the fp16 weights run up to 2^7.9."""
    nk = 8 * BLOCK
    rng = np.random.default_rng(8)
    q = np.ones((4, 8), dtype=np.float16)
    k = np.zeros((nk, 8), dtype=np.float16)
    lg = np.where(np.arange(nk) < BLOCK, 0.0, 7.9) + rng.uniform(-0.5, 0.0, nk)
    k[:, 0] = (lg / np.float64(LOG2E)).astype(np.float16)
    v = _normal((nk, 48), 9)
    return q, k, v, 1.0


def case_cancelling_logits():
    """Large products that cancel: partial sums reach ~6e4 while the logits
    themselves stay O(1), so fp32 accumulation error in the logits (the
    bound's dS term) dominates every other error."""
    rng = np.random.default_rng(10)
    d, nk = 128, 256
    h = d // 2
    q = np.empty((8, d), dtype=np.float16)
    q[:, :h] = rng.uniform(29.0, 31.0, (8, h)).astype(np.float16)
    q[:, h:] = q[:, :h]
    big = rng.uniform(29.0, 31.0, (nk, h)).astype(np.float16)
    k = np.empty((nk, d), dtype=np.float16)
    k[:, :h] = big
    # the second half cancels the first up to a small remainder per element
    k[:, h:] = (-big.astype(np.float64) + rng.uniform(-0.05, 0.05, (nk, h))).astype(np.float16)
    v = _normal((nk, 32), 11)
    return q, k, v, 1.0


def case_long_keys_stale_weights():
    """131072 keys whose weights sit just above 1 under a stale maximum
    (fp16 1 + 3/1024).  While L lies in [2^16, 2^17) every fp32 add drops 3/8
    of an ulp; a column of O that sums only every second (or fourth, or third)
    weight sits one binade lower at that point and rounds the other way, so
    the error of O / L grows with the number of keys (the bound's Nk 2^-23
    term)."""
    nk = 1024 * BLOCK
    q = np.ones((2, 8), dtype=np.float16)
    k = np.zeros((nk, 8), dtype=np.float16)
    # block 0 sets the maximum at 0; every other key's weight is 2^0.00422 = 1 + 3/1024 after fp16
    k[BLOCK:, 0] = np.float16(np.log2(1.0 + 3.0 / 1024.0) / float(LOG2E))
    v = np.zeros((nk, 8), dtype=np.float16)
    v[:, 0] = 3.0
    v[:, 1] = 1.0
    v[::2, 2] = 1.0
    v[::4, 3] = 1.0
    v[::2, 4] = 3.0
    v[::2, 5] = 1.0
    v[1::2, 5] = -1.0
    v[:, 6] = 0.75
    v[::3, 7] = 1.0
    return q, k, v, 1.0


CASES = {
    "page_head": case_page_head,
    "logits_near_80": case_logits_near_80,
    "growing_maximum": case_growing_maximum,
    "stale_max_weights": case_stale_max_weights_up_to_256,
    "cancelling_logits": case_cancelling_logits,
    "long_keys": case_long_keys_stale_weights,
}


def _run(name, out_f16, ranges=1, drop_rescale=False, seed=0):
    q, k, v, scale = CASES[name]()
    O, E, G = oracle.attention(q, k, v, scale)
    got = emulate(q, k, v, scale, out_f16, ranges=ranges, drop_rescale=drop_rescale, seed=seed)
    return got, O, E, G, q.shape[1], k.shape[0]


_cache = {}


def _cached(name, out_f16, ranges=1):
    key = (name, out_f16, ranges)
    if key not in _cache:
        _cache[key] = _run(name, out_f16, ranges)
    return _cache[key]


@pytest.mark.parametrize("name", sorted(CASES))
@pytest.mark.parametrize("out_f16", [False, True])
def test_emulation_inside_bound(name, out_f16):
    got, O, E, G, d, nk = _cached(name, out_f16)
    tol = oracle.attention_tolerance(O, E, G, d, nk, out_f16)
    err = np.abs(got - O)
    assert np.all(err <= tol), (name, float(np.max(err / tol)))


@pytest.mark.parametrize("name,ranges", [("page_head", 3), ("growing_maximum", 4),
                                         ("long_keys", 2), ("logits_near_80", 2)])
def test_emulation_with_key_ranges_inside_bound(name, ranges):
    """The key split and the last-wave split: ranges merged after the pass."""
    got, O, E, G, d, nk = _cached(name, False, ranges)
    tol = oracle.attention_tolerance(O, E, G, d, nk, False)
    assert np.all(np.abs(got - O) <= tol)


def test_bound_without_logit_term_is_violated():
    """Drop 2.5 dS E: fp32 accumulation of cancelling logits breaks it."""
    got, O, E, G, d, nk = _cached("cancelling_logits", False)
    assert np.any(np.abs(got - O) > _bound(O, E, G, d, nk, False, drop="dS"))
    assert np.all(np.abs(got - O) <= _bound(O, E, G, d, nk, False))


def test_bound_without_key_count_term_is_violated():
    """Drop Nk 2^-23 E: 131072 fp32 additions of stale-maximum weights break it."""
    got, O, E, G, d, nk = _cached("long_keys", False)
    assert np.any(np.abs(got - O) > _bound(O, E, G, d, nk, False, drop="nk"))
    assert np.all(np.abs(got - O) <= _bound(O, E, G, d, nk, False))


def test_page_head_error_well_inside_bound():
    """On the page's own head the bound is not vacuous: the emulated error
    uses a visible share of it, but not all of it."""
    got, O, E, G, d, nk = _cached("page_head", False)
    r = np.abs(got - O) / oracle.attention_tolerance(O, E, G, d, nk, False)
    assert 1e-4 < float(np.max(r)) < 1.0


@pytest.mark.parametrize("out_f16", [False, True])
def test_dropped_rescale_is_caught(out_f16):
    """A forward pass that keeps the old O and L unscaled when the maximum
    grows (a dropped 2^(m_old - m_new)) fails the bound, fp16 output too."""
    got, O, E, G, d, nk = _run("growing_maximum", out_f16, drop_rescale=True)
    tol = oracle.attention_tolerance(O, E, G, d, nk, out_f16)
    assert np.any(np.abs(got - O) > tol)


def test_exact_cases_of_the_emulation():
    """Sanity of the emulation itself: identical keys give the plain mean of
    V's rows; a key 1000 ahead gives its own V row; both as the oracle."""
    v = _normal((300, 16), 12)
    q = np.ones((3, 4), dtype=np.float16)
    k = np.zeros((300, 4), dtype=np.float16)
    got = emulate(q, k, v, 1.0, False)
    O, _, _ = oracle.attention(q, k, v, 1.0)
    assert np.allclose(got, O, rtol=0, atol=1e-6)
    k2 = np.zeros((300, 4), dtype=np.float16)
    k2[123, 0] = 1000.0
    got2 = emulate(q, k2, v, 1.0, False)
    assert np.array_equal(got2, np.broadcast_to(v[123].astype(np.float64), got2.shape))
