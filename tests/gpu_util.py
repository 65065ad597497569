"""Helpers for the GPU parity tests: place seeded CPU operands in device
buffers with chosen row strides and base offsets, guard the output with
canaries, call the C ABI, and compare against the oracle element by element.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
import tiled_gemm_tg_gb300 as tg

GUARD = 256  # canary elements before and after C


def code(dt) -> int:
    return tg.F16 if dt == torch.float16 else tg.F32


def esize(dt) -> int:
    return 2 if dt == torch.float16 else 4


def bits(t: torch.Tensor) -> torch.Tensor:
    return t.view(torch.int16) if t.dtype == torch.float16 else t.view(torch.int32)


class DevMatrix:
    """A rows x cols matrix at element offset `off` of a device buffer, with
    row stride `ld` (elements).  Keeps the buffer alive."""

    def __init__(self, x: torch.Tensor, ld: int, off: int, device):
        rows, cols = x.shape
        self.rows, self.cols, self.ld, self.off = rows, cols, ld, off
        buf = torch.zeros(off + max(rows, 1) * ld + 64, dtype=x.dtype)
        if rows and cols:
            buf[off:off + rows * ld].view(rows, ld)[:, :cols] = x
        self.buf = buf.to(device)
        self.ptr = self.buf.data_ptr() + off * esize(x.dtype)


class DevOutput:
    """C with canaries: GUARD elements on either side and the row gaps
    (columns N..ldc-1) hold a NaN bit pattern the kernels never produce."""

    def __init__(self, M, N, ldc, off, dtype, device):
        self.M, self.N, self.ldc, self.off, self.dtype = M, N, ldc, off, dtype
        n = off + GUARD + max(M, 1) * ldc + GUARD
        self.buf = torch.empty(n, dtype=dtype, device=device)
        bits(self.buf).fill_(0x7E5A if dtype == torch.float16 else 0x7FC0A5A5)
        self.canary = bits(self.buf[:1].clone()).item()
        self.ptr = self.buf.data_ptr() + (off + GUARD) * esize(dtype)

    def result(self):
        """(C as float64 numpy array, whether every canary is intact)."""
        h = self.buf.cpu()
        hb = bits(h)
        start = self.off + GUARD
        end = start + self.M * self.ldc
        intact = bool((hb[:start] == self.canary).all()) and bool((hb[end:] == self.canary).all())
        if self.M:
            body = h[start:end].view(self.M, self.ldc)
            C = body[:, :self.N].double().numpy()
            if self.ldc > self.N:
                intact = intact and bool((bits(body)[:, self.N:] == self.canary).all())
        else:
            C = np.zeros((0, self.N))
        return C, intact


def run(a: torch.Tensor, b: torch.Tensor, out_dtype=torch.float16, lda=None, ldb=None,
        ldc=None, offs=(0, 0, 0), device="cuda", stream=None):
    """Run tg_gemm through the C ABI; return (C float64, canaries intact, path)."""
    M, K = a.shape
    N = b.shape[1]
    lda = K if lda is None else lda
    ldb = N if ldb is None else ldb
    ldc = N if ldc is None else ldc
    A = DevMatrix(a, max(lda, 1), offs[0], device)
    B = DevMatrix(b, max(ldb, 1), offs[1], device)
    C = DevOutput(M, N, max(ldc, 1), offs[2], out_dtype, device)
    s = torch.cuda.current_stream() if stream is None else stream
    path = tg.tg_gemm_path(M, N, K, A.ptr, lda, B.ptr, ldb, C.ptr, ldc, code(a.dtype),
                           code(out_dtype))
    st = tg.tg_gemm(M, N, K, A.ptr, lda, B.ptr, ldb, C.ptr, ldc, code(a.dtype),
                    code(out_dtype), s.cuda_stream)
    assert st == tg.TG_OK, tg.tg_status_string(st)
    assert tg.tg_gemm_check(s.cuda_stream) == tg.TG_OK
    got, intact = C.result()
    return got, intact, path


def compare(got: np.ndarray, C_ref: np.ndarray, S: np.ndarray, out_f16: bool, what=""):
    """Element-by-element acceptance: |got - C| <= 2e-3 S + 1e-5 (+ 1e-2 |C|)."""
    tol = oracle.tolerance(C_ref, S, out_f16)
    err = np.abs(got - C_ref)
    bad = ~(err <= tol)  # NaN counts as bad
    if bad.any():
        i = np.argwhere(bad)[0]
        raise AssertionError(
            f"{what}: {int(bad.sum())}/{bad.size} elements outside tolerance; first at "
            f"{tuple(int(v) for v in i)}: got {got[tuple(i)]!r} want {C_ref[tuple(i)]!r} "
            f"tol {tol[tuple(i)]!r}")
    return float(np.max(err)) if err.size else 0.0


def check_full(a, b, out_dtype=torch.float16, **kw):
    got, intact, path = run(a, b, out_dtype, **kw)
    assert intact, "a canary outside C (guard band or row gap) was overwritten"
    C_ref, S = oracle.gemm(a.numpy(), b.numpy())
    compare(got, C_ref, S, out_dtype == torch.float16, f"{tuple(a.shape)}x{tuple(b.shape)}")
    return got, C_ref, path


def f16_bits_of(x: np.ndarray) -> np.ndarray:
    return oracle.f64_to_f16_bits(x)


class DevVector:
    """n fp32 values at element offset `off` of a device buffer."""

    def __init__(self, x: np.ndarray, off: int, device):
        buf = torch.zeros(off + max(len(x), 1) + 16, dtype=torch.float32)
        buf[off:off + len(x)] = torch.from_numpy(np.asarray(x, dtype=np.float32))
        self.buf = buf.to(device)
        self.ptr = self.buf.data_ptr() + off * 4


def run_ex(a: torch.Tensor, b: torch.Tensor, out_dtype, alpha=1.0, beta=0.0, d=None,
           bias=None, act=0, lda=None, ldb=None, ldc=None, ldd=None, offs=(0, 0, 0),
           d_off=0, bias_off=0, in_place=False, device="cuda"):
    """Run tg_gemm_ex through the C ABI: C = act(alpha*AB + beta*D + bias).

    d: an M x N CPU tensor of the output dtype (or None); with in_place the
    output buffer is first filled with d and passed as both C and D.
    Returns (C float64, canaries intact, path)."""
    M, K = a.shape
    N = b.shape[1]
    lda = K if lda is None else lda
    ldb = N if ldb is None else ldb
    ldc = N if ldc is None else ldc
    A = DevMatrix(a, max(lda, 1), offs[0], device)
    B = DevMatrix(b, max(ldb, 1), offs[1], device)
    C = DevOutput(M, N, max(ldc, 1), offs[2], out_dtype, device)
    d_ptr, ldd_v, keep = 0, max(N, 1), []
    if d is not None:
        if in_place:
            body = C.buf[C.off + GUARD:C.off + GUARD + M * ldc].view(M, ldc)
            body[:, :N] = d.to(device)
            d_ptr, ldd_v = C.ptr, ldc
        else:
            ldd_v = N if ldd is None else ldd
            D = DevMatrix(d, max(ldd_v, 1), d_off, device)
            keep.append(D)
            d_ptr = D.ptr
    b_ptr = 0
    if bias is not None:
        bv = DevVector(bias, bias_off, device)
        keep.append(bv)
        b_ptr = bv.ptr
    s = torch.cuda.current_stream()
    path = tg.tg_gemm_path(M, N, K, A.ptr, lda, B.ptr, ldb, C.ptr, ldc, code(a.dtype),
                           code(out_dtype))
    st = tg.tg_gemm_ex(M, N, K, A.ptr, lda, B.ptr, ldb, C.ptr, ldc, code(a.dtype),
                       code(out_dtype), alpha, beta, d_ptr, ldd_v, b_ptr, act, s.cuda_stream)
    assert st == tg.TG_OK, tg.tg_status_string(st)
    assert tg.tg_gemm_check(s.cuda_stream) == tg.TG_OK
    got, intact = C.result()
    return got, intact, path


def compare_ex(got, out_ref, S, alpha, beta, d, bias, out_f16, what=""):
    """Fused-epilogue acceptance (oracle.epilogue_tolerance)."""
    tol = oracle.epilogue_tolerance(out_ref, S, alpha, beta,
                                    None if d is None else d.double().numpy(), bias, out_f16)
    err = np.abs(got - out_ref)
    bad = ~(err <= tol)
    if bad.any():
        i = tuple(int(v) for v in np.argwhere(bad)[0])
        raise AssertionError(f"{what}: {int(bad.sum())}/{bad.size} elements outside tolerance; "
                             f"first at {i}: got {got[i]!r} want {out_ref[i]!r} tol {tol[i]!r}")
    return float(np.max(err)) if err.size else 0.0
