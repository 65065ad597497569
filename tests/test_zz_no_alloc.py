"""tg_attention_noalloc: the key split and the split of a short last wave
with their partials in the library's static device scratch, against
tg_attention_ws with a caller workspace.

Two calls in a row through the no-alloc entry point (the second reuses
scratch the first left behind, including the last-wave split's per-tile
counters) must give the same output as the caller-workspace entry point,
bit for bit: the same kernels run on the same inputs, only the scratch
address differs.  One call is also checked against the oracle directly.
"""
import numpy as np
import pytest
import torch

import oracle
import tiled_gemm_tg_gb300 as tg

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(0)
    yield


def _call(fn, q, k, v, o, scale, extra=()):
    B, Nq, d = q.shape
    Nk, dv = v.shape[1], v.shape[2]
    s = torch.cuda.current_stream().cuda_stream
    st = fn(B, Nq, Nk, d, dv, q.data_ptr(), d, Nq * d, k.data_ptr(), d, Nk * d, v.data_ptr(), dv,
            Nk * dv, o.data_ptr(), dv, Nq * dv, scale, tg.F16, tg.F16, *extra, s)
    assert st == tg.TG_OK, tg.tg_status_string(st)
    assert tg.tg_gemm_check(s) == tg.TG_OK


@pytest.mark.parametrize("B,N,d", [(1, 1024, 768), (1, 1024, 128), (2, 700, 64)])
def test_noalloc_matches_workspace_entry_point_twice(B, N, d):
    g = torch.Generator().manual_seed(14000 + N + d)
    q = torch.randn(B, N, d, generator=g).half().cuda()
    k = torch.randn(B, N, d, generator=g).half().cuda()
    v = torch.randn(B, N, d, generator=g).half().cuda()
    scale = 1.0 if d == 768 else d ** -0.5
    need = tg.tg_attention_workspace_size(B, N, N, d, d)
    assert 0 < need <= 16 << 20, need
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    want = torch.empty(B, N, d, dtype=torch.half, device="cuda")
    _call(tg.tg_attention_ws, q, k, v, want, scale, (ws.data_ptr(), need))
    for _ in range(2):
        got = torch.full((B, N, d), float("nan"), dtype=torch.half, device="cuda")
        _call(tg.tg_attention_noalloc, q, k, v, got, scale)
        assert torch.equal(got.view(torch.int16), want.view(torch.int16))


def test_noalloc_rejects_a_split_larger_than_its_scratch():
    # one head of 2048 queries with d = dv = 1024 gives 16 x 8 = 128 CTAs of
    # 128 rows by 128 output columns, too few for the SMs: the keys are split
    # in two, and the partials (2 x 2048 x 1024 fp32, about 16.8 MB) exceed
    # the 16 MB scratch; the workspace query says how much
    B, N, d = 1, 2048, 1024
    need = tg.tg_attention_workspace_size(B, N, N, d, d)
    if need <= 16 << 20:
        pytest.skip("this device would not split this call beyond the scratch")
    q = torch.zeros(B, N, d, dtype=torch.half, device="cuda")
    o = torch.empty(B, N, d, dtype=torch.half, device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    st = tg.tg_attention_noalloc(B, N, N, d, d, q.data_ptr(), d, N * d, q.data_ptr(), d, N * d,
                                 q.data_ptr(), d, N * d, o.data_ptr(), d, N * d, 1.0, tg.F16,
                                 tg.F16, s)
    assert st == tg.TG_ERR_UNSUPPORTED


def _heads(B, N, d, seed):
    g = torch.Generator().manual_seed(seed)
    return [torch.randn(B, N, d, generator=g).half() for _ in range(3)]


@pytest.mark.parametrize("B,N,d", [(16, 4096, 128), (4, 5504, 128)])
def test_noalloc_last_wave_split_twice(B, N, d):
    """The P-in-TMEM kernel with its short last wave cut along the keys: the
    scratch holds partial outputs and one counter per cut tile."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    assert tg.tg_attention_kernel(B, N, N, d, d, 1) == 3
    tail, pieces = tg.tg_attention_tail_plan(B, N, N, d, d, sms)
    if tail == 0:
        pytest.skip(f"no last-wave split of this shape on {sms} SMs")
    q, k, v = (x.cuda() for x in _heads(B, N, d, 15000 + B))
    need = tg.tg_attention_workspace_size(B, N, N, d, d)
    assert 0 < need <= 16 << 20, need
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    want = torch.empty(B, N, d, dtype=torch.half, device="cuda")
    scale = d ** -0.5
    _call(tg.tg_attention_ws, q, k, v, want, scale, (ws.data_ptr(), need))
    for _ in range(2):
        got = torch.full((B, N, d), float("nan"), dtype=torch.half, device="cuda")
        _call(tg.tg_attention_noalloc, q, k, v, got, scale)
        assert torch.equal(got.view(torch.int16), want.view(torch.int16))


def test_noalloc_without_a_split_is_the_plain_call():
    """A call that needs no scratch (a last wave of 104 of 152 tiles is not
    cut) runs the single pass, equal to tg_attention bit for bit."""
    B, N, d = 16, 2048, 128
    if tg.tg_attention_workspace_size(B, N, N, d, d) != 0:
        pytest.skip("this device would split this call")
    q, k, v = (x.cuda() for x in _heads(B, N, d, 15100))
    want = torch.empty(B, N, d, dtype=torch.half, device="cuda")
    got = torch.full((B, N, d), float("nan"), dtype=torch.half, device="cuda")
    _call(tg.tg_attention, q, k, v, want, d ** -0.5)
    _call(tg.tg_attention_noalloc, q, k, v, got, d ** -0.5)
    assert torch.equal(got.view(torch.int16), want.view(torch.int16))


@pytest.mark.parametrize("B,N,d,scale", [(1, 1024, 768, 1.0), (4, 5504, 128, 128 ** -0.5)])
def test_noalloc_against_the_oracle(B, N, d, scale):
    """The no-alloc call on its own, every row of the first and last head
    against the oracle's fp64 definition of softmax(scale Q K^T) V, within the
    acceptance bound the other attention tests use."""
    qh, kh, vh = _heads(B, N, d, 15200 + d)
    q, k, v = qh.cuda(), kh.cuda(), vh.cuda()
    o = torch.full((B, N, d), float("nan"), dtype=torch.half, device="cuda")
    _call(tg.tg_attention_noalloc, q, k, v, o, scale)
    got = o.double().cpu().numpy()
    for h in sorted({0, B - 1}):
        O, E, G = oracle.attention(qh[h].numpy(), kh[h].numpy(), vh[h].numpy(), scale)
        tol = oracle.attention_tolerance(O, E, G, d, N, True)
        bad = ~(np.abs(got[h] - O) <= tol)
        assert not bad.any(), f"head {h}: {int(bad.sum())} elements outside tolerance"
