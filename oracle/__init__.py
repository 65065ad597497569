"""CPU oracle for the tiled GEMM C = A x B (test infrastructure only).

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The CUDA library in
``tiled_gemm_tg_gb300`` never imports it, and it never imports that library.

The arithmetic lives in ``tg_oracle.c`` (plain C, fp64, exact binary16
decode); this module only compiles it with gcc and marshals NumPy arrays.
Every function states the passage it follows in the C source's header.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "tg_oracle.c")
_LIB_PATH = os.path.join(_HERE, "libtg_oracle.so")
_lock = threading.Lock()
_lib = None

F16 = 1
F32 = 2
E4M3 = 3


def build(force: bool = False) -> str:
    """Compile tg_oracle.c into libtg_oracle.so (gcc, OpenMP when available)."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    base = ["gcc", "-O2", "-std=c11", "-shared", "-fPIC", "-fno-fast-math",
            "-ffp-contract=off", _SRC, "-o", tmp, "-lm"]
    try:
        subprocess.run(base[:5] + ["-fopenmp"] + base[5:], check=True,
                       capture_output=True, text=True)
    except subprocess.CalledProcessError:
        # No OpenMP runtime: the oracle still works, single-threaded.
        subprocess.run(base, check=True, capture_output=True, text=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _bind(path: str):
    lib = ctypes.CDLL(path)
    i64, vp = ctypes.c_int64, ctypes.c_void_p
    lib.tgo_f16_to_f64.restype = ctypes.c_double
    lib.tgo_f16_to_f64.argtypes = [ctypes.c_uint16]
    lib.tgo_f64_to_f16.restype = ctypes.c_uint16
    lib.tgo_f64_to_f16.argtypes = [ctypes.c_double]
    lib.tgo_f16_to_f64_n.argtypes = [vp, vp, i64]
    lib.tgo_f64_to_f16_n.argtypes = [vp, vp, i64]
    lib.tgo_e4m3_to_f64_n.argtypes = [vp, vp, i64]
    lib.tgo_num_threads.restype = ctypes.c_int
    lib.tgo_gemm.restype = ctypes.c_int
    lib.tgo_gemm.argtypes = [i64, i64, i64, vp, i64, vp, i64, ctypes.c_int,
                             vp, vp, ctypes.c_int]
    lib.tgo_attention.restype = ctypes.c_int
    lib.tgo_attention.argtypes = [i64, i64, i64, i64, vp, i64, vp, i64, vp, i64, ctypes.c_int,
                                  ctypes.c_double, vp, vp, vp, ctypes.c_int]
    lib.tgo_epilogue.restype = ctypes.c_int
    lib.tgo_epilogue.argtypes = [i64, i64, vp, ctypes.c_double, ctypes.c_double, vp, i64,
                                 ctypes.c_int, vp, ctypes.c_int, vp]
    lib.tgo_gemm_at.restype = ctypes.c_int
    lib.tgo_gemm_at.argtypes = [i64, i64, i64, vp, i64, vp, i64, ctypes.c_int,
                                i64, vp, vp, vp, vp, ctypes.c_int]
    return lib


def _operand(x: np.ndarray):
    """Return (array, dtype code, row stride in elements) for a 2-D operand.

    fp16 operands may be given as float16 or as uint16 bit patterns, FP8
    E4M3 operands as uint8 bit patterns.  Rows
    must be unit-stride; the row stride (leading dimension) may exceed the
    row length, as with a sub-matrix view.
    """
    if x.ndim != 2:
        raise ValueError("operands must be 2-D")
    if x.dtype == np.float16:
        x = x.view(np.uint16)
    if x.dtype == np.uint16:
        code = F16
    elif x.dtype == np.uint8:
        code = E4M3  # FP8 E4M3 bit patterns
    elif x.dtype == np.float32:
        code = F32
    else:
        raise TypeError(f"unsupported operand dtype {x.dtype}")
    if x.size == 0:
        return x, code, max(x.shape[1], 1)
    if x.shape[1] > 1 and x.strides[1] != x.itemsize:
        raise ValueError("rows must be contiguous")
    ld = x.strides[0] // x.itemsize if x.shape[0] > 1 else max(x.shape[1], 1)
    return x, code, int(ld)


def _pair(a, b):
    a, ca, lda = _operand(a)
    b, cb, ldb = _operand(b)
    if ca != cb:
        raise TypeError("A and B must have the same dtype")
    if a.shape[1] != b.shape[0]:
        raise ValueError("inner dimensions differ")
    return a, b, ca, lda, ldb


class Oracle:
    """The oracle bound to one compiled copy of tg_oracle.c."""

    def __init__(self, lib_path: str):
        self.lib = _bind(lib_path)

    def num_threads(self) -> int:
        """Threads the oracle's OpenMP loops use by default."""
        return int(self.lib.tgo_num_threads())

    def f16_bits_to_f64(self, bits: np.ndarray) -> np.ndarray:
        """Exact binary16 -> binary64 decode of uint16 bit patterns."""
        src = np.ascontiguousarray(bits, dtype=np.uint16)
        out = np.empty(src.shape, dtype=np.float64)
        self.lib.tgo_f16_to_f64_n(src.ctypes.data, out.ctypes.data, src.size)
        return out

    def e4m3_bits_to_f64(self, bits: np.ndarray) -> np.ndarray:
        """Exact FP8 E4M3 -> binary64 decode of uint8 bit patterns."""
        src = np.ascontiguousarray(bits, dtype=np.uint8)
        out = np.empty(src.shape, dtype=np.float64)
        self.lib.tgo_e4m3_to_f64_n(src.ctypes.data, out.ctypes.data, src.size)
        return out

    def f64_to_f16_bits(self, x: np.ndarray) -> np.ndarray:
        """binary64 -> binary16 bit patterns, round to nearest, ties to even."""
        src = np.ascontiguousarray(x, dtype=np.float64)
        out = np.empty(src.shape, dtype=np.uint16)
        self.lib.tgo_f64_to_f16_n(src.ctypes.data, out.ctypes.data, src.size)
        return out

    def gemm(self, a: np.ndarray, b: np.ndarray, nthreads: int = 0):
        """C = A x B and S = sum_k |A_ik B_kj|, both fp64 M x N arrays."""
        a, b, code, lda, ldb = _pair(a, b)
        M, K = a.shape
        N = b.shape[1]
        C = np.empty((M, N), dtype=np.float64)
        S = np.empty((M, N), dtype=np.float64)
        rc = self.lib.tgo_gemm(M, N, K, a.ctypes.data, lda, b.ctypes.data, ldb,
                               code, C.ctypes.data, S.ctypes.data, int(nthreads))
        if rc != 0:
            raise RuntimeError("oracle rejected its arguments")
        return C, S

    def gemm_at(self, a: np.ndarray, b: np.ndarray, rows, cols, nthreads: int = 0):
        """C and S at the listed output positions only (same definition)."""
        a, b, code, lda, ldb = _pair(a, b)
        M, K = a.shape
        N = b.shape[1]
        r = np.ascontiguousarray(rows, dtype=np.int64)
        c = np.ascontiguousarray(cols, dtype=np.int64)
        if r.shape != c.shape:
            raise ValueError("rows and cols differ in length")
        C = np.empty(r.shape, dtype=np.float64)
        S = np.empty(r.shape, dtype=np.float64)
        rc = self.lib.tgo_gemm_at(M, N, K, a.ctypes.data, lda, b.ctypes.data, ldb,
                                  code, r.size, r.ctypes.data, c.ctypes.data,
                                  C.ctypes.data, S.ctypes.data, int(nthreads))
        if rc != 0:
            raise RuntimeError("oracle rejected its arguments")
        return C, S


    def epilogue(self, C: np.ndarray, alpha=1.0, beta=0.0, cin=None, bias=None, act=0):
        """act(alpha * C + beta * Cin + bias[j]) in fp64 (C: the oracle's M x N
        product; cin: M x N fp16/fp32 array or None; bias: N values or None)."""
        C = np.ascontiguousarray(C, dtype=np.float64)
        M, N = C.shape
        out = np.empty((M, N), dtype=np.float64)
        cin_ptr, ldcin, code = None, max(N, 1), F32
        if cin is not None:
            cin, code, ldcin = _operand(cin)
            cin_ptr = cin.ctypes.data
        b = None if bias is None else np.ascontiguousarray(bias, dtype=np.float32)
        rc = self.lib.tgo_epilogue(M, N, C.ctypes.data, float(alpha), float(beta), cin_ptr,
                                   ldcin, code, None if b is None else b.ctypes.data, int(act),
                                   out.ctypes.data)
        if rc != 0:
            raise RuntimeError("oracle rejected its arguments")
        return out


    def attention(self, q: np.ndarray, k: np.ndarray, v: np.ndarray, scale: float = 1.0,
                  nthreads: int = 0):
        """softmax(scale * Q K^T) V by its definition in fp64.  Returns (O, E, G):
        O and E are Nq x dv, E[i,c] = sum_j w_ij |V[j,c]|; G[i] is the largest
        |scale| * sum_d |Q[i,d] K[j,d]| over j."""
        q, code, ldq = _operand(q)
        k, code_k, ldk = _operand(k)
        v, code_v, ldv = _operand(v)
        if not (code == code_k == code_v):
            raise TypeError("Q, K and V must share a dtype")
        Nq, d = q.shape
        Nk, dv = v.shape
        if k.shape != (Nk, d):
            raise ValueError("K must be Nk x d")
        O = np.empty((Nq, dv), dtype=np.float64)
        E = np.empty((Nq, dv), dtype=np.float64)
        G = np.empty(Nq, dtype=np.float64)
        rc = self.lib.tgo_attention(Nq, Nk, d, dv, q.ctypes.data, ldq, k.ctypes.data, ldk,
                                    v.ctypes.data, ldv, code, float(scale), O.ctypes.data,
                                    E.ctypes.data, G.ctypes.data, int(nthreads))
        if rc != 0:
            raise RuntimeError("oracle rejected its arguments")
        return O, E, G


def _default() -> Oracle:
    global _lib
    with _lock:
        if _lib is None:
            _lib = Oracle(build())
        return _lib


def num_threads() -> int:
    return _default().num_threads()


def f16_bits_to_f64(bits):
    return _default().f16_bits_to_f64(bits)


def f64_to_f16_bits(x):
    return _default().f64_to_f16_bits(x)


def e4m3_bits_to_f64(bits):
    return _default().e4m3_bits_to_f64(bits)


def gemm(a, b, nthreads: int = 0):
    return _default().gemm(a, b, nthreads)


def gemm_at(a, b, rows, cols, nthreads: int = 0):
    return _default().gemm_at(a, b, rows, cols, nthreads)


def epilogue(C, alpha=1.0, beta=0.0, cin=None, bias=None, act=0):
    return _default().epilogue(C, alpha, beta, cin, bias, act)


def attention(q, k, v, scale=1.0, nthreads: int = 0):
    return _default().attention(q, k, v, scale, nthreads)


def attention_tolerance(O, E, G, d: int, nk: int, out_f16: bool):
    """Bound for a tensor-core attention forward against the fp64 definition:
    logits from fp16 products summed in fp32 are off by at most about
    (d + 8) * 2^-23 * G (G bounds every |logit| and its magnitude sum), which
    moves each softmax weight by a factor within exp(+-2 * that), so O by
    2.5 * dS * E; the probabilities rounded to fp16 for the P.V product and
    summed in fp32 over nk keys add (2^-10 + nk * 2^-23) * E; plus 1e-5 and
    the 1e-2 relative term for an fp16 output."""
    dS = (d + 8) * 2.0 ** -23 * np.asarray(G, dtype=np.float64)[:, None]
    t = E * (2.5 * dS + 2.0 ** -10 + nk * 2.0 ** -23) + 1e-5
    if out_f16:
        t = t + 1e-2 * np.abs(O)
    return t


def tolerance(C_ref: np.ndarray, S: np.ndarray, out_f16: bool) -> np.ndarray:
    """Per-element acceptance bound for a kernel result against the oracle.

    2e-3 * S + 1e-5 for fp32 accumulation, plus 1e-2 * |C_ref| when the
    output is fp16 (the relative threshold of §3.3 第四步 of the
    gsyq.cn/news/429607 article).
    """
    tol = 2e-3 * S + 1e-5
    if out_f16:
        tol = tol + 1e-2 * np.abs(C_ref)
    return tol


def epilogue_tolerance(out_ref, S, alpha, beta, cin, bias, out_f16: bool):
    """Bound for a fused result act(alpha*AB + beta*Cin + bias): the product's
    bound scaled by |alpha|, fp32 rounding of the other terms, all carried
    through an activation whose slope is at most 1.13 (ReLU 1, GELU
    max d/dx x*Phi(x) = 1.129), plus 1e-2 relative for an fp16 output."""
    t = abs(alpha) * (2e-3 * S + 1e-5)
    if cin is not None and beta != 0.0:
        t = t + 1e-6 * np.abs(beta * np.asarray(cin, dtype=np.float64))
    if bias is not None:
        t = t + 1e-6 * np.abs(np.asarray(bias, dtype=np.float64))[None, :]
    t = 1.13 * t + 1e-6
    if out_f16:
        t = t + 1e-2 * np.abs(out_ref)
    return t
