"""tiled_gemm_tg_gb300 -- thin Python binding over libtg_gemm.so.

The library computes C[M,N] = A[M,K] x B[K,N] (row-major; fp16 or fp32
inputs, fp32 accumulation, fp16 or fp32 output) with hand-written CUDA
kernels for sm_103a, optionally with a fused epilogue
C = act(alpha*AB + beta*D + bias) (``tg_gemm_ex``).  This module only marshals arguments: the entry points
carry the names of the C ABI in include/tg_gemm.h, and ``gemm`` is a
convenience that takes torch tensors, allocates the output with torch and
calls ``tg_gemm``.  There is no fallback: if the compiled library is missing
every call raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

__all__ = [
    "F16", "F32", "E4M3", "TG_OK", "TG_ERR_INVALID_ARG", "TG_ERR_UNSUPPORTED", "TG_ERR_CUDA",
    "TG_ERR_TIMEOUT", "PATHS", "TgError", "lib", "library_path", "tg_gemm", "tg_gemm_check",
    "tg_status_string", "tg_gemm_path", "tg_gemm_force_path", "tg_gemm_force_tiling",
    "tg_gemm_force_split_tail", "tg_gemm_pair_split_tail", "tg_gemm_force_stages",
    "tg_gemm_boundary_split", "tg_gemm_force_split_k", "tg_gemm_main_plan",
    "tg_gemm_test_hook", "tg_gemm_ex", "tg_gemm_batched", "tg_gemm_batched_path",
    "tg_attention", "tg_attention_ws", "tg_attention_workspace_size", "tg_attention_noalloc",
    "tg_attention_kernel", "tg_attention_force_kernel", "tg_attention_tail_plan",
    "attention", "ACT_NONE", "ACT_RELU", "ACT_GELU",
    "tg_gemm_version", "gemm", "bmm",
    "check",
]

F16 = 1
F32 = 2
E4M3 = 3
TG_OK = 0
TG_ERR_INVALID_ARG = 1
TG_ERR_UNSUPPORTED = 2
TG_ERR_CUDA = 3
TG_ERR_TIMEOUT = 4
ACT_NONE = 0
ACT_RELU = 1
ACT_GELU = 2
PATHS = {0: "none", 1: "zero", 2: "simt_f32", 3: "tc_main", 4: "tc_boundary", 5: "tc_skinny",
         6: "tc_pair"}

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "libtg_gemm.so")
_lock = threading.Lock()
_lib = None


class TgError(RuntimeError):
    def __init__(self, status: int, what: str = "tg_gemm"):
        self.status = status
        super().__init__(f"{what} failed: {tg_status_string(status)} ({status})")


def library_path() -> str:
    return _LIB_PATH


def lib() -> ctypes.CDLL:
    """The loaded libtg_gemm.so; raises if it has not been built."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(_LIB_PATH):
            raise RuntimeError(
                f"{_LIB_PATH} is missing: build it with "
                "`python -c 'import __graft_entry__ as g; g.build()'`")
        L = ctypes.CDLL(_LIB_PATH)
        i64, vp, i32 = ctypes.c_int64, ctypes.c_void_p, ctypes.c_int
        L.tg_gemm.restype = i32
        L.tg_gemm.argtypes = [i64, i64, i64, vp, i64, vp, i64, vp, i64, i32, i32, vp]
        L.tg_gemm_ex.restype = i32
        L.tg_gemm_ex.argtypes = [i64, i64, i64, vp, i64, vp, i64, vp, i64, i32, i32,
                                 ctypes.c_float, ctypes.c_float, vp, i64, vp, i32, vp]
        L.tg_gemm_batched.restype = i32
        L.tg_gemm_batched.argtypes = [i64, i64, i64, i64, vp, i64, i64, vp, i64, i64, vp, i64, i64,
                                      i32, i32, vp]
        L.tg_gemm_batched_path.restype = i32
        L.tg_gemm_batched_path.argtypes = [i64, i64, i64, i64, vp, i64, i64, vp, i64, i64, vp,
                                           i64, i64, i32, i32]
        L.tg_attention.restype = i32
        L.tg_attention.argtypes = [i64, i64, i64, i64, i64, vp, i64, i64, vp, i64, i64, vp, i64,
                                   i64, vp, i64, i64, ctypes.c_float, i32, i32, vp]
        L.tg_attention_ws.restype = i32
        L.tg_attention_ws.argtypes = [i64, i64, i64, i64, i64, vp, i64, i64, vp, i64, i64, vp,
                                      i64, i64, vp, i64, i64, ctypes.c_float, i32, i32, vp,
                                      ctypes.c_size_t, vp]
        L.tg_attention_noalloc.restype = i32
        L.tg_attention_noalloc.argtypes = [i64, i64, i64, i64, i64, vp, i64, i64, vp, i64, i64,
                                           vp, i64, i64, vp, i64, i64, ctypes.c_float, i32, i32,
                                           vp]
        L.tg_attention_workspace_size.restype = ctypes.c_size_t
        L.tg_attention_workspace_size.argtypes = [i64, i64, i64, i64, i64]
        L.tg_attention_kernel.restype = i32
        L.tg_attention_kernel.argtypes = [i64, i64, i64, i64, i64, i32]
        L.tg_attention_tail_plan.restype = i32
        L.tg_attention_tail_plan.argtypes = [i64, i64, i64, i64, i64, i32,
                                             ctypes.POINTER(ctypes.c_int)]
        L.tg_attention_force_kernel.restype = i32
        L.tg_attention_force_kernel.argtypes = [i32]
        L.tg_gemm_check.restype = i32
        L.tg_gemm_check.argtypes = [vp]
        L.tg_status_string.restype = ctypes.c_char_p
        L.tg_status_string.argtypes = [i32]
        L.tg_gemm_path.restype = i32
        L.tg_gemm_path.argtypes = [i64, i64, i64, vp, i64, vp, i64, vp, i64, i32, i32]
        L.tg_gemm_force_path.restype = None
        L.tg_gemm_force_path.argtypes = [i32]
        L.tg_gemm_force_tiling.restype = i32
        L.tg_gemm_force_tiling.argtypes = [i32, i32]
        L.tg_gemm_force_split_tail.restype = i32
        L.tg_gemm_force_split_tail.argtypes = [i32]
        L.tg_gemm_pair_split_tail.restype = i32
        L.tg_gemm_pair_split_tail.argtypes = [i64, i32]
        L.tg_gemm_force_split_k.restype = i32
        L.tg_gemm_force_split_k.argtypes = [i32]
        L.tg_gemm_main_plan.restype = i32
        L.tg_gemm_main_plan.argtypes = [i64, i64, i64, i64, i32, i32, ctypes.POINTER(i32)]
        L.tg_gemm_boundary_split.restype = i32
        L.tg_gemm_boundary_split.argtypes = [i64, i32, i32]
        L.tg_gemm_force_stages.restype = i32
        L.tg_gemm_force_stages.argtypes = [i32]
        L.tg_gemm_test_hook.restype = None
        L.tg_gemm_test_hook.argtypes = [i32]
        L.tg_gemm_version.restype = i32
        L.tg_gemm_version.argtypes = []
        _lib = L
        return L


# ------------------------------------------------------------ raw C entry points

def tg_gemm(M, N, K, A, lda, B, ldb, C, ldc, in_dtype, out_dtype, stream=0) -> int:
    """Enqueue C = A x B on `stream`; pointers are integers (device addresses)."""
    return int(lib().tg_gemm(M, N, K, A, lda, B, ldb, C, ldc, in_dtype, out_dtype, stream))


def tg_gemm_ex(M, N, K, A, lda, B, ldb, C, ldc, in_dtype, out_dtype, alpha, beta, D, ldd,
               bias, act, stream=0) -> int:
    """Enqueue C = act(alpha * A x B + beta * D + bias) on `stream` (D and bias
    are device addresses or 0/None)."""
    return int(lib().tg_gemm_ex(M, N, K, A, lda, B, ldb, C, ldc, in_dtype, out_dtype,
                                float(alpha), float(beta), D or None, ldd, bias or None,
                                int(act), stream))


def tg_gemm_batched(batch, M, N, K, A, lda, sA, B, ldb, sB, C, ldc, sC, in_dtype, out_dtype,
                    stream=0) -> int:
    """Enqueue C_b = A_b x B_b, X_b = X + b*sX elements, for b < batch."""
    return int(lib().tg_gemm_batched(batch, M, N, K, A, lda, sA, B, ldb, sB, C, ldc, sC,
                                     in_dtype, out_dtype, stream))


def tg_gemm_batched_path(batch, M, N, K, A, lda, sA, B, ldb, sB, C, ldc, sC, in_dtype,
                         out_dtype) -> int:
    return int(lib().tg_gemm_batched_path(batch, M, N, K, A, lda, sA, B, ldb, sB, C, ldc, sC,
                                          in_dtype, out_dtype))


def tg_attention(batch, Nq, Nk, d, dv, Q, ldq, sQ, K, ldk, sK, V, ldv, sV, O, ldo, sO, scale,
                 in_dtype, out_dtype, stream=0) -> int:
    """Enqueue O_b = softmax(scale * Q_b K_b^T) V_b for b < batch."""
    return int(lib().tg_attention(batch, Nq, Nk, d, dv, Q, ldq, sQ, K, ldk, sK, V, ldv, sV, O,
                                  ldo, sO, float(scale), in_dtype, out_dtype, stream))


def tg_attention_ws(batch, Nq, Nk, d, dv, Q, ldq, sQ, K, ldk, sK, V, ldv, sV, O, ldo, sO, scale,
                    in_dtype, out_dtype, workspace, workspace_bytes, stream=0) -> int:
    return int(lib().tg_attention_ws(batch, Nq, Nk, d, dv, Q, ldq, sQ, K, ldk, sK, V, ldv, sV, O,
                                     ldo, sO, float(scale), in_dtype, out_dtype, workspace or None,
                                     workspace_bytes, stream))


def tg_attention_noalloc(batch, Nq, Nk, d, dv, Q, ldq, sQ, K, ldk, sK, V, ldv, sV, O, ldo, sO,
                         scale, in_dtype, out_dtype, stream=0) -> int:
    """tg_attention with the key split's partials in the library's static
    scratch (no allocation; overlapping calls race on it)."""
    return int(lib().tg_attention_noalloc(batch, Nq, Nk, d, dv, Q, ldq, sQ, K, ldk, sK, V, ldv,
                                          sV, O, ldo, sO, float(scale), in_dtype, out_dtype,
                                          stream))


def tg_attention_workspace_size(batch, Nq, Nk, d, dv) -> int:
    return int(lib().tg_attention_workspace_size(batch, Nq, Nk, d, dv))


def tg_gemm_check(stream=0) -> int:
    """Synchronize `stream` and read/clear the device error word."""
    return int(lib().tg_gemm_check(stream))


def tg_status_string(status: int) -> str:
    return lib().tg_status_string(int(status)).decode()


def tg_gemm_path(M, N, K, A, lda, B, ldb, C, ldc, in_dtype, out_dtype) -> int:
    return int(lib().tg_gemm_path(M, N, K, A, lda, B, ldb, C, ldc, in_dtype, out_dtype))


def tg_attention_kernel(batch, Nq, Nk, d, dv, split_allowed: bool = False) -> int:
    return int(lib().tg_attention_kernel(batch, Nq, Nk, d, dv, 1 if split_allowed else 0))


def tg_attention_tail_plan(batch, Nq, Nk, d, dv, num_sms):
    """(tiles of the last wave that are split, key ranges per tile)."""
    p = ctypes.c_int(-1)
    tail = int(lib().tg_attention_tail_plan(batch, Nq, Nk, d, dv, num_sms, ctypes.byref(p)))
    return tail, int(p.value)


def tg_attention_force_kernel(kernel: int) -> int:
    return int(lib().tg_attention_force_kernel(int(kernel)))


def tg_gemm_force_path(path: int) -> None:
    lib().tg_gemm_force_path(int(path))


def tg_gemm_force_tiling(bn: int, group_m: int) -> int:
    return int(lib().tg_gemm_force_tiling(int(bn), int(group_m)))


def tg_gemm_force_split_tail(tiles: int) -> int:
    return int(lib().tg_gemm_force_split_tail(int(tiles)))


def tg_gemm_force_stages(stages: int) -> int:
    return int(lib().tg_gemm_force_stages(int(stages)))


def tg_gemm_pair_split_tail(tiles: int, max_pairs: int) -> int:
    return int(lib().tg_gemm_pair_split_tail(int(tiles), int(max_pairs)))


def tg_gemm_force_split_k(split: int) -> int:
    return int(lib().tg_gemm_force_split_k(int(split)))


def tg_gemm_main_plan(M: int, N: int, K: int, batch: int, in_dtype: int, num_sms: int):
    """(tile width, split over K) the one-CTA kernel would choose, host only."""
    bn = ctypes.c_int(0)
    split = int(lib().tg_gemm_main_plan(int(M), int(N), int(K), int(batch), int(in_dtype),
                                        int(num_sms), ctypes.byref(bn)))
    return bn.value, split


def tg_gemm_boundary_split(tiles: int, kblocks: int, num_sms: int) -> int:
    return int(lib().tg_gemm_boundary_split(int(tiles), int(kblocks), int(num_sms)))


def tg_gemm_test_hook(hook: int) -> None:
    lib().tg_gemm_test_hook(int(hook))


def tg_gemm_version() -> int:
    return int(lib().tg_gemm_version())


# ------------------------------------------------------------- torch marshalling

def _code(dtype) -> int:
    import torch
    if dtype == torch.float16:
        return F16
    if dtype == torch.float32:
        return F32
    if dtype == torch.float8_e4m3fn:
        return E4M3
    raise TypeError(f"unsupported dtype {dtype}")


def _ld(t) -> int:
    if t.dim() != 2:
        raise ValueError("operands must be 2-D")
    if t.size(1) > 1 and t.stride(1) != 1:
        raise ValueError("rows must be contiguous (row-major)")
    return int(t.stride(0)) if t.size(0) > 1 else max(int(t.size(1)), 1)


def _stream_handle(stream) -> int:
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return int(stream.cuda_stream) if hasattr(stream, "cuda_stream") else int(stream)


def gemm(a, b, out=None, out_dtype=None, stream=None, alpha=1.0, beta=0.0, d=None, bias=None,
         act=ACT_NONE):
    """C = act(alpha * A x B + beta * D + bias) for 2-D CUDA tensors (row-major
    rows; row strides may exceed the row length); the defaults give C = A x B.
    `d` has the output's dtype and may be `out` itself; `bias` is N fp32
    values.  Allocates C with torch unless `out` is given."""
    import torch
    if not (a.is_cuda and b.is_cuda):
        raise ValueError("operands must be CUDA tensors")
    M, K = a.shape
    K2, N = b.shape
    if K != K2:
        raise ValueError("inner dimensions differ")
    if out is None:
        od = out_dtype if out_dtype is not None else a.dtype
        out = torch.empty((M, N), dtype=od, device=a.device)
    fused = alpha != 1.0 or beta != 0.0 or bias is not None or act != ACT_NONE
    if not fused:
        st = tg_gemm(M, N, K, a.data_ptr(), _ld(a), b.data_ptr(), _ld(b), out.data_ptr(),
                     _ld(out), _code(a.dtype), _code(out.dtype), _stream_handle(stream))
    else:
        d_ptr, ldd = 0, N
        if beta != 0.0:
            if d is None or d.dtype != out.dtype or tuple(d.shape) != (M, N) or not d.is_cuda:
                raise ValueError("beta != 0 needs d: an M x N CUDA tensor of the output dtype")
            d_ptr, ldd = d.data_ptr(), _ld(d)
        b_ptr = 0
        if bias is not None:
            if bias.dtype != torch.float32 or bias.numel() != N or not bias.is_cuda or \
                    not bias.is_contiguous():
                raise ValueError("bias must be N contiguous fp32 CUDA values")
            b_ptr = bias.data_ptr()
        st = tg_gemm_ex(M, N, K, a.data_ptr(), _ld(a), b.data_ptr(), _ld(b), out.data_ptr(),
                        _ld(out), _code(a.dtype), _code(out.dtype), alpha, beta, d_ptr, ldd,
                        b_ptr, act, _stream_handle(stream))
    if st != TG_OK:
        raise TgError(st)
    return out


def bmm(a, b, out=None, out_dtype=None, stream=None):
    """C[i] = A[i] x B[i] for 3-D CUDA tensors (rows contiguous; a batch
    stride of 0, as from expand(), broadcasts one matrix).  Allocates C with
    torch unless `out` is given."""
    import torch
    if a.dim() != 3 or b.dim() != 3 or not (a.is_cuda and b.is_cuda):
        raise ValueError("operands must be 3-D CUDA tensors")
    batch, M, K = a.shape
    b2, K2, N = b.shape
    if K != K2 or batch != b2:
        raise ValueError("batch or inner dimensions differ")
    if out is None:
        od = out_dtype if out_dtype is not None else a.dtype
        out = torch.empty((batch, M, N), dtype=od, device=a.device)

    def ld3(t):
        if t.size(2) > 1 and t.stride(2) != 1:
            raise ValueError("rows must be contiguous (row-major)")
        ld = int(t.stride(1)) if t.size(1) > 1 else max(int(t.size(2)), 1)
        sb = int(t.stride(0)) if t.size(0) > 1 else 0
        return ld, sb

    (lda, sa), (ldb, sb), (ldc, sc) = ld3(a), ld3(b), ld3(out)
    st = tg_gemm_batched(batch, M, N, K, a.data_ptr(), lda, sa, b.data_ptr(), ldb, sb,
                         out.data_ptr(), ldc, sc, _code(a.dtype), _code(out.dtype),
                         _stream_handle(stream))
    if st != TG_OK:
        raise TgError(st, "tg_gemm_batched")
    return out


def attention(q, k, v, scale=1.0, out=None, out_dtype=None, stream=None, workspace=None):
    """softmax(scale * Q K^T) V for 2-D (Nq x d, Nk x d, Nk x dv) or 3-D
    (batch first) fp16 CUDA tensors with contiguous rows; a batch stride of 0,
    as from expand(), shares one matrix.  Allocates O with torch unless `out`
    is given.  `workspace` (a CUDA tensor of tg_attention_workspace_size
    bytes) lets small calls split the keys over more CTAs."""
    import torch
    squeeze = q.dim() == 2
    if squeeze:
        q, k, v = q.unsqueeze(0), k.unsqueeze(0), v.unsqueeze(0)
        if out is not None:
            out = out.unsqueeze(0)
    if q.dim() != 3 or k.dim() != 3 or v.dim() != 3 or not (q.is_cuda and k.is_cuda and v.is_cuda):
        raise ValueError("q, k, v must be 2-D or 3-D CUDA tensors")
    batch, Nq, d = q.shape
    bk, Nk, dk = k.shape
    bv, Nv, dv = v.shape
    if dk != d or Nv != Nk or not (bk == bv == batch):
        raise ValueError("shapes do not match: q (b, Nq, d), k (b, Nk, d), v (b, Nk, dv)")
    if out is None:
        od = out_dtype if out_dtype is not None else q.dtype
        out = torch.empty((batch, Nq, dv), dtype=od, device=q.device)

    def ld3(t):
        if t.size(2) > 1 and t.stride(2) != 1:
            raise ValueError("rows must be contiguous (row-major)")
        ld = int(t.stride(1)) if t.size(1) > 1 else max(int(t.size(2)), 1)
        return ld, (int(t.stride(0)) if t.size(0) > 1 else 0)

    (ldq, sq), (ldk, sk), (ldv, sv), (ldo, so) = ld3(q), ld3(k), ld3(v), ld3(out)
    ws_ptr, ws_bytes = 0, 0
    if workspace is not None:
        ws_ptr, ws_bytes = workspace.data_ptr(), workspace.numel() * workspace.element_size()
    st = tg_attention_ws(batch, Nq, Nk, d, dv, q.data_ptr(), ldq, sq, k.data_ptr(), ldk, sk,
                         v.data_ptr(), ldv, sv, out.data_ptr(), ldo, so, scale, _code(q.dtype),
                         _code(out.dtype), ws_ptr, ws_bytes, _stream_handle(stream))
    if st != TG_OK:
        raise TgError(st, "tg_attention")
    return out[0] if squeeze else out


def check(stream=None) -> None:
    """Raise TgError if a kernel on `stream` abandoned a bounded wait."""
    st = tg_gemm_check(_stream_handle(stream))
    if st != TG_OK:
        raise TgError(st, "tg_gemm_check")
