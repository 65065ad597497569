"""tg_attention_noalloc: the key split with its partials in the library's
static device scratch, against tg_attention_ws with a caller workspace.

Two calls in a row through the no-alloc entry point (the second reuses
scratch the first left behind) must give the same output as the caller-
workspace entry point, bit for bit: the same kernels run on the same
inputs, only the scratch address differs.
"""
import pytest
import torch

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
    # 2 heads x 8192 queries x dv 1024 would need far more than 16 MB of
    # partials if split; the workspace query says how much
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
