"""Failure detection without a GPU fault.

The test hook (tg_gemm_test_hook) makes a tensor-core kernel wait on a
barrier that nothing signals.  The bounded wait must run out in about a
second, the kernel must record it in the device error word and return, and
tg_gemm_check must report TG_ERR_TIMEOUT; the CUDA context must stay usable,
so the same path run again without the hook matches the oracle.
"""
import time

import pytest
import torch

import tiled_gemm_tg_gb300 as tg
from tiled_gemm_tg_gb300 import inputs

from gpu_util import DevMatrix, DevOutput, check_full

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(0)
    yield
    tg.tg_gemm_test_hook(0)
    tg.tg_gemm_force_path(0)


# (path, M, N, K, pad_ld): K spans several k-blocks so every kernel waits on
# the unfilled stage (or uncommitted group) before finishing.
CASES = [(3, 300, 520, 1024, True), (6, 512, 768, 1024, True), (5, 16, 1024, 2048, True),
         (4, 127, 255, 512, False),
         # 77 pair tiles: one cluster stalls while the others run two tiles
         (6, 1792, 2816, 1024, True)]


@pytest.mark.parametrize("path,M,N,K,pad", CASES, ids=lambda v: str(v))
def test_bounded_wait_expiry_is_reported(path, M, N, K, pad):
    a = inputs.draw((M, K), "normal", 9100 + path, "f16")
    b = inputs.draw((K, N), "normal", 9200 + path, "f16")
    lda = (K + 7) // 8 * 8 if pad else K
    ldb = (N + 7) // 8 * 8 if pad else N
    A = DevMatrix(a, lda, 0, "cuda")
    B = DevMatrix(b, ldb, 0, "cuda")
    C = DevOutput(M, N, N, 0, torch.float16, "cuda")
    s = torch.cuda.current_stream().cuda_stream
    assert tg.tg_gemm_check(s) == tg.TG_OK
    tg.tg_gemm_force_path(path)
    tg.tg_gemm_test_hook(1)
    try:
        assert tg.tg_gemm_path(M, N, K, A.ptr, lda, B.ptr, ldb, C.ptr, N, tg.F16, tg.F16) == path
        t0 = time.time()
        st = tg.tg_gemm(M, N, K, A.ptr, lda, B.ptr, ldb, C.ptr, N, tg.F16, tg.F16, s)
        assert st == tg.TG_OK
        assert tg.tg_gemm_check(s) == tg.TG_ERR_TIMEOUT
        elapsed = time.time() - t0
    finally:
        tg.tg_gemm_test_hook(0)
    try:
        assert 0.5 < elapsed < 30.0, elapsed
        # the word was cleared and the context still works: same path, no hook
        assert tg.tg_gemm_check(s) == tg.TG_OK
        check_full(a, b, torch.float16, lda=lda, ldb=ldb)
    finally:
        tg.tg_gemm_force_path(0)


def test_simt_path_ignores_the_hook():
    a = inputs.draw((64, 64), "normal", 9301, "f32")
    b = inputs.draw((64, 64), "normal", 9302, "f32")
    tg.tg_gemm_test_hook(1)
    try:
        check_full(a, b, torch.float32)
    finally:
        tg.tg_gemm_test_hook(0)


@pytest.mark.parametrize("kernel", [1, 3])
def test_attention_bounded_wait_expiry_is_reported(kernel):
    """Each attention kernel under the hook (1: the general kernel, 3: the
    one keeping P in tensor memory): its first K stage stays empty, the MMA
    issuer's wait runs out, every role winds down, and the next call without
    the hook is correct."""
    import numpy as np

    import oracle

    g = torch.Generator().manual_seed(9400)
    q = torch.randn(200, 64, generator=g).half()
    k = torch.randn(300, 64, generator=g).half()
    v = torch.randn(300, 64, generator=g).half()
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    s = torch.cuda.current_stream().cuda_stream
    assert tg.tg_gemm_check(s) == tg.TG_OK
    assert tg.tg_attention_force_kernel(kernel) == tg.TG_OK
    try:
        assert tg.tg_attention_kernel(1, 200, 300, 64, 64) == kernel
        tg.tg_gemm_test_hook(1)
        try:
            t0 = time.time()
            tg.attention(qd, kd, vd, 0.125)
            assert tg.tg_gemm_check(s) == tg.TG_ERR_TIMEOUT
            elapsed = time.time() - t0
        finally:
            tg.tg_gemm_test_hook(0)
        assert 0.5 < elapsed < 30.0, elapsed
        assert tg.tg_gemm_check(s) == tg.TG_OK
        o = tg.attention(qd, kd, vd, 0.125)
        tg.check()
    finally:
        tg.tg_attention_force_kernel(0)
    O, E, G = oracle.attention(q.numpy(), k.numpy(), v.numpy(), 0.125)
    tol = oracle.attention_tolerance(O, E, G, 64, 300, True)
    assert np.all(np.abs(o.double().cpu().numpy() - O) <= tol)


def test_attention_tail_split_expiry_then_clean_call():
    """The P-in-TMEM kernel with its last wave split through a workspace:
    under the hook every CTA's wait runs out, no range merges and the tile
    counters are left as the aborted ranges left them; the next call on the
    same workspace (its zeroing kernel resets them) matches the oracle on
    every head, and a third call matches the second bit for bit."""
    import numpy as np

    import oracle

    sms = torch.cuda.get_device_properties(0).multi_processor_count
    batch, Nq, Nk, d = sms + 6, 128, 1024, 64   # six tiles left over: two ranges of 4 blocks
    assert tg.tg_attention_kernel(batch, Nq, Nk, d, d, split_allowed=True) == 3
    assert tg.tg_attention_tail_plan(batch, Nq, Nk, d, d, sms) == (6, 2)
    need = tg.tg_attention_workspace_size(batch, Nq, Nk, d, d)
    assert need > 0
    g = torch.Generator().manual_seed(9500)
    q = torch.randn(batch, Nq, d, generator=g).half()
    k = torch.randn(batch, Nk, d, generator=g).half()
    v = torch.randn(batch, Nk, d, generator=g).half()
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    assert tg.tg_gemm_check(s) == tg.TG_OK
    tg.tg_gemm_test_hook(1)
    try:
        t0 = time.time()
        tg.attention(qd, kd, vd, 0.125, workspace=ws)
        assert tg.tg_gemm_check(s) == tg.TG_ERR_TIMEOUT
        elapsed = time.time() - t0
    finally:
        tg.tg_gemm_test_hook(0)
    assert 0.5 < elapsed < 60.0, elapsed
    assert tg.tg_gemm_check(s) == tg.TG_OK
    o = tg.attention(qd, kd, vd, 0.125, workspace=ws)
    tg.check()
    got = o.double().cpu().numpy()
    for b in range(batch):
        O, E, G = oracle.attention(q[b].numpy(), k[b].numpy(), v[b].numpy(), 0.125)
        tol = oracle.attention_tolerance(O, E, G, d, Nk, True)
        assert np.all(np.abs(got[b] - O) <= tol), f"head {b}"
    again = tg.attention(qd, kd, vd, 0.125, workspace=ws)
    tg.check()
    assert torch.equal(again.view(torch.int16), o.view(torch.int16))
