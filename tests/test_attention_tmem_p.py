"""GPU parity of the attention forward that keeps P in tensor memory (two
score buffers, d <= 128, dv <= 128) against the oracle's fp64 definition,
through tg_attention with the kernel forced (tg_attention_force_kernel(3)),
and the automatic choice between the forward kernels.

The bound per element is oracle.attention_tolerance, as for the one-tile
kernel; structured inputs whose softmax is exact must match bit for bit.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import tiled_gemm_tg_gb300 as tg

from gpu_util import f16_bits_of
from test_attention import _check, _qkv, run_attn

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(0)
    yield


@pytest.fixture
def tmem_p():
    assert tg.tg_attention_force_kernel(3) == tg.TG_OK
    try:
        yield
    finally:
        tg.tg_attention_force_kernel(0)


@pytest.mark.parametrize("Nq,Nk,d,dv,scale", [
    (128, 128, 64, 64, 0.125),       # one CTA, one key block
    (200, 300, 64, 64, 0.125),       # ragged in both
    (1, 1, 64, 64, 1.0),
    (130, 257, 128, 128, 1 / math.sqrt(128)),
    (300, 500, 96, 80, 0.1),         # d not a multiple of 64, dv not of 32
    (256, 384, 128, 128, 0.09),      # two CTAs, three key blocks
    (513, 1000, 32, 128, 0.2),       # one Q chunk, five CTAs, last one row
    (257, 129, 128, 40, 0.3),
    (260, 700, 16, 8, 0.5),
])
@pytest.mark.parametrize("out", [torch.float16, torch.float32])
def test_tmem_p_shapes(tmem_p, Nq, Nk, d, dv, scale, out):
    assert tg.tg_attention_kernel(1, Nq, Nk, d, dv) == 3
    q, k, v = _qkv(1, Nq, Nk, d, dv, 14000 + Nq + Nk + d)
    got, intact = run_attn(q, k, v, scale, out)
    assert intact
    _check(q, k, v, scale, got, out, f"tmem-p {Nq}x{Nk} d{d} dv{dv}")


def test_tmem_p_batched_and_shared_kv(tmem_p):
    q, k, v = _qkv(3, 400, 260, 128, 128, 14100)
    got, intact = run_attn(q, k, v, 0.09)
    assert intact
    _check(q, k, v, 0.09, got, torch.float16, "tmem-p batched")
    got, intact = run_attn(q, k[:1], v[:1], 0.09, share_kv=True)
    assert intact
    _check(q, k[:1], v[:1], 0.09, got, torch.float16, "tmem-p shared K/V")


def test_tmem_p_padded_rows(tmem_p):
    """Row strides past the head sizes (ldq, ldk, ldv, ldo all padded)."""
    q, k, v = _qkv(2, 300, 333, 64, 96, 14150)
    got, intact = run_attn(q, k, v, 0.125, torch.float32, ldq=72, ldk=80, ldv=104, ldo=101)
    assert intact
    _check(q, k, v, 0.125, got, torch.float32, "tmem-p padded rows")


@pytest.mark.parametrize("scale", [-0.1, 0.0])
def test_tmem_p_negative_and_zero_scale(tmem_p, scale):
    """A negative scale turns the row maximum into the minimum raw score; a
    zero scale gives uniform weights over the valid keys (the masked keys
    of the ragged last block must still get none)."""
    q, k, v = _qkv(1, 300, 390, 64, 64, 14200)
    got, intact = run_attn(q, k, v, scale, torch.float32)
    assert intact
    _check(q, k, v, scale, got, torch.float32, f"tmem-p scale {scale}")


def test_tmem_p_growing_logits_rescale(tmem_p):
    """Logits that grow key by key in both CTAs: O in tensor memory is
    rescaled in every block."""
    Nq, Nk, d, dv = 256, 1024, 64, 64
    g = torch.Generator().manual_seed(14300)
    u = torch.randn(d, generator=g)
    u = u / u.norm()
    q = (u * 4).expand(Nq, d).clone() + 0.01 * torch.randn(Nq, d, generator=g)
    t = torch.linspace(-4, 4, Nk)
    k = t[:, None] * u[None, :] + 0.01 * torch.randn(Nk, d, generator=g)
    v = torch.randn(Nk, dv, generator=g)
    q, k, v = q.half()[None], k.half()[None], v.half()[None]
    got, intact = run_attn(q, k, v, 1.0, torch.float32)
    assert intact
    _check(q, k, v, 1.0, got, torch.float32, "tmem-p growing logits")


def test_tmem_p_rescale_in_some_rows_only(tmem_p):
    """The first CTA's rows see growing logits (rescaled every block), the
    second's see flat ones (never rescaled after the first block)."""
    Nq, Nk, d, dv = 256, 896, 64, 128
    g = torch.Generator().manual_seed(14350)
    u = torch.randn(d, generator=g)
    u = u / u.norm()
    q = 0.3 * torch.randn(Nq, d, generator=g)
    q[:128] = (u * 4).expand(128, d) + 0.01 * torch.randn(128, d, generator=g)
    t = torch.linspace(-4, 4, Nk)
    k = t[:, None] * u[None, :] + 0.3 * torch.randn(Nk, d, generator=g)
    v = torch.randn(Nk, dv, generator=g)
    q, k, v = q.half()[None], k.half()[None], v.half()[None]
    got, intact = run_attn(q, k, v, 1.0, torch.float16)
    assert intact
    _check(q, k, v, 1.0, got, torch.float16, "tmem-p one-sided rescale")


@pytest.mark.parametrize("out", [torch.float16, torch.float32])
def test_tmem_p_uniform_weights_exact(tmem_p, out):
    """Identical keys: every probability is 1 and O is the mean of V's rows,
    exact for integer V and 256 keys."""
    Nq, Nk, d, dv = 300, 256, 128, 96
    g = torch.Generator().manual_seed(14400)
    q = torch.randn(1, Nq, d, generator=g).half()
    k = torch.randn(1, 1, d, generator=g).half().expand(1, Nk, d).contiguous()
    v = torch.randint(-8, 9, (1, Nk, dv), generator=g).half()
    got, intact = run_attn(q, k, v, 0.125, out)
    assert intact
    want = np.broadcast_to(v[0].double().numpy().mean(axis=0), (Nq, dv))
    if out == torch.float16:
        assert np.array_equal(f16_bits_of(got[0]), f16_bits_of(want))
    else:
        assert np.array_equal(got[0], want)


def test_tmem_p_one_hot_exact(tmem_p):
    """Each query has one key whose logit exceeds all others by 369 in base
    2: O is exactly that key's V row, in both CTAs."""
    Nq, Nk, d, dv = 256, 640, 128, 128
    g = torch.Generator().manual_seed(14500)
    hot = torch.randint(0, Nk, (Nq,), generator=g)
    q = torch.zeros(Nq, d)
    k = torch.zeros(Nk, d)
    for i in range(Nq):
        axis = i % d
        q[i, axis] = 16.0
    # queries i and i + 128 share an axis: give them the same hot key
    hot[128:] = hot[:128]
    for i in range(128):
        k[hot[i], i] = 16.0
    v = torch.randn(Nk, dv, generator=g).half()
    got, intact = run_attn(q.half()[None], k.half()[None], v[None], 1.0, torch.float32)
    assert intact
    want = v[hot].double().numpy()
    assert np.array_equal(got[0], want)


def test_tmem_p_matches_general():
    """The general kernel and this one on the same call: both within the
    oracle's bound, and within a few fp16 units of each other."""
    q, k, v = _qkv(4, 1000, 1000, 128, 128, 14600)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    outs = {}
    try:
        for kern in (1, 3):
            assert tg.tg_attention_force_kernel(kern) == tg.TG_OK
            assert tg.tg_attention_kernel(4, 1000, 1000, 128, 128) == kern
            outs[kern] = tg.attention(qd, kd, vd, 1 / math.sqrt(128)).double().cpu().numpy()
            tg.check()
    finally:
        tg.tg_attention_force_kernel(0)
    _check(q, k, v, 1 / math.sqrt(128), outs[3], torch.float16, "tmem-p vs oracle")
    assert np.allclose(outs[1], outs[3], rtol=2e-2, atol=2e-3)


def test_automatic_choice():
    """Heads with d, dv <= 128: P in tensor memory, unless a call with few
    query tiles is given a workspace (then the key split); larger heads: the
    general kernel."""
    assert tg.tg_attention_kernel(16, 4096, 4096, 128, 128) == 3
    assert tg.tg_attention_kernel(16, 2048, 2048, 128, 128) == 3
    assert tg.tg_attention_kernel(1, 128, 128, 64, 64) == 3
    assert tg.tg_attention_kernel(1, 200, 1000, 64, 64, split_allowed=True) == 2
    assert tg.tg_attention_kernel(1, 1024, 1024, 768, 768) == 1
    assert tg.tg_attention_kernel(1, 1024, 1024, 768, 768, split_allowed=True) == 2
    assert tg.tg_attention_kernel(16, 4096, 4096, 256, 128) == 1
    assert tg.tg_attention_kernel(0, 4096, 4096, 128, 128) == 0
    try:
        assert tg.tg_attention_force_kernel(1) == tg.TG_OK
        assert tg.tg_attention_kernel(16, 4096, 4096, 128, 128) == 1
        assert tg.tg_attention_force_kernel(3) == tg.TG_OK
        assert tg.tg_attention_kernel(1, 128, 128, 64, 64) == 3
        assert tg.tg_attention_kernel(1, 200, 1000, 64, 64, split_allowed=True) == 3
        assert tg.tg_attention_kernel(1, 1024, 1024, 768, 768, split_allowed=True) == 2
    finally:
        tg.tg_attention_force_kernel(0)


def test_tmem_p_binding_sampled_large():
    """16 heads x 4096 positions x d 128 (the automatic choice is this
    kernel): sampled query rows of several CTAs."""
    batch, N, d = 16, 4096, 128
    assert tg.tg_attention_kernel(batch, N, N, d, d) == 3
    q, k, v = _qkv(batch, N, N, d, d, 14700)
    o = tg.attention(q.cuda(), k.cuda(), v.cuda(), 1 / math.sqrt(d))
    tg.check()
    rows = np.array([0, 1, 127, 128, 255, 256, 2049, 4095])
    for b in (0, 7, batch - 1):
        O, E, G = oracle.attention(q[b].numpy()[rows], k[b].numpy(), v[b].numpy(),
                                   1 / math.sqrt(d))
        tol = oracle.attention_tolerance(O, E, G, d, N, True)
        got = o[b].double().cpu().numpy()[rows]
        assert np.all(np.abs(got - O) <= tol), f"head {b}"


def _num_sms():
    return torch.cuda.get_device_properties(0).multi_processor_count


def _tail_case(Nq, extra):
    """A batch count whose query tiles fill the SMs once and leave `extra`
    tiles (up to one tile row more) in a last, short wave."""
    q_blocks = (Nq + 127) // 128
    batch = (_num_sms() + extra + q_blocks - 1) // q_blocks
    tiles = batch * q_blocks
    assert _num_sms() < tiles <= _num_sms() * 3 // 2
    return batch


def _attn_ws(qd, kd, vd, scale, out, ws):
    o = tg.attention(qd, kd, vd, scale, out_dtype=out, workspace=ws)
    tg.check()
    return o.double().cpu().numpy()


@pytest.mark.parametrize("Nq,Nk,d,dv,scale,fill", [
    (128, 1000, 128, 128, 0.09, 0.05),  # eight blocks, the last one ragged: 2 pieces of 4
    (200, 1100, 64, 64, 0.125, 0.05),   # ragged queries; nine blocks: pieces of 4 and 5
    (256, 1500, 96, 80, 0.1, 0.05),     # twelve blocks: 3 pieces; d, dv not multiples of 64
    (130, 2100, 64, 48, 0.125, 0.05),   # seventeen blocks: 4 pieces of 4, 4, 4, 5
    (128, 2100, 128, 128, 0.09, 0.3),   # a third of a wave left: 2 pieces of 8 and 9
])
@pytest.mark.parametrize("out", [torch.float16, torch.float32])
def test_tmem_p_wave_tail_split(Nq, Nk, d, dv, scale, fill, out):
    """A short last wave: its tiles are cut into pieces along the keys,
    merged in the kernel through the workspace.  Every row against the
    oracle, the same call without a workspace close by, and a second call on
    the same workspace bit for bit equal (the merge order is fixed)."""
    batch = _tail_case(Nq, int(fill * _num_sms()))
    assert tg.tg_attention_kernel(batch, Nq, Nk, d, dv) == 3
    need = tg.tg_attention_workspace_size(batch, Nq, Nk, d, dv)
    assert need > 0, "a short last wave should ask for the tail workspace"
    q, k, v = _qkv(batch, Nq, Nk, d, dv, 14800 + Nq + Nk + d)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    ws = torch.full((need,), 0xA5, dtype=torch.uint8, device="cuda")  # contents do not matter
    got = _attn_ws(qd, kd, vd, scale, out, ws)
    _check(q, k, v, scale, got, out, f"tail split {batch}x{Nq}x{Nk} d{d} dv{dv}")
    plain = tg.attention(qd, kd, vd, scale, out_dtype=out).double().cpu().numpy()
    tg.check()
    assert np.allclose(got, plain, rtol=2e-2, atol=2e-3)
    again = _attn_ws(qd, kd, vd, scale, out, ws)
    assert np.array_equal(got, again)


@pytest.mark.parametrize("peak_piece", [0, 2, 3])
def test_tmem_p_wave_tail_split_far_apart_maxima(peak_piece):
    """The pieces' row maxima differ by far more than the rescale threshold:
    one key per row dominates (score 60 against |score| < 1), in the first,
    a middle or the last of four pieces of the keys, so the other pieces'
    merge weights are 2^-86 and every other probability rounds to zero in
    fp16.  The output is that key's value row exactly (fp32 output)."""
    Nq, Nk, d, dv = 128, 2048, 64, 64    # sixteen key blocks: four pieces of 512 keys
    batch = _tail_case(Nq, 6)
    g = torch.Generator().manual_seed(14900 + peak_piece)
    # row r points along axis r % d; each axis has one hot key per batch entry
    hot = torch.randint(0, Nk // 4, (batch, d), generator=g) + peak_piece * (Nk // 4)
    q = torch.zeros(batch, Nq, d)
    q[:, torch.arange(Nq), torch.arange(Nq) % d] = 8.0
    k = torch.randn(batch, Nk, d, generator=g) * 0.01
    for b in range(batch):
        k[b, hot[b], torch.arange(d)] = 7.5
    v = torch.randn(batch, Nk, dv, generator=g)
    q, k, v = q.half(), k.half(), v.half()
    need = tg.tg_attention_workspace_size(batch, Nq, Nk, d, dv)
    assert need > 0
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    got = _attn_ws(q.cuda(), k.cuda(), v.cuda(), 1.0, torch.float32, ws)
    _check(q, k, v, 1.0, got, torch.float32, f"tail split, peak in piece {peak_piece}")
    rows = torch.arange(Nq) % d
    want = np.stack([v[b, hot[b][rows]].double().numpy() for b in range(batch)])
    assert np.array_equal(got, want)
