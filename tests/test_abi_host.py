"""Host-side checks of the C ABI that need no GPU.

The library must build, load, and export every function declared in
include/tg_gemm.h.  Argument validation and path selection run entirely on
the host before any CUDA call, so they are exercised here with fake device
addresses (nothing is ever dereferenced or launched).
"""
import os
import re

import numpy as np
import pytest

import tiled_gemm_tg_gb300 as tg
from tiled_gemm_tg_gb300 import build as tgbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "tg_gemm.h")

# fake, 256-byte aligned device addresses far apart from one another
PA, PB, PC = 0x7F0000000000, 0x7F1000000000, 0x7F2000000000


@pytest.fixture(scope="module", autouse=True)
def built():
    tgbuild.build()
    tg.lib()
    yield
    tg.tg_gemm_force_path(0)


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"\b(tg_[a-z_]+)\s*\(", text)
    return sorted(set(names))


def test_header_declares_the_abi():
    names = declared_functions()
    for must in ["tg_gemm", "tg_gemm_ex", "tg_gemm_check", "tg_status_string", "tg_gemm_path",
                 "tg_gemm_force_path", "tg_gemm_force_tiling", "tg_gemm_test_hook",
                 "tg_gemm_version"]:
        assert must in names


def test_every_declared_symbol_is_exported():
    L = tg.lib()
    for name in declared_functions():
        assert hasattr(L, name), f"{name} declared in tg_gemm.h but not exported"


def test_status_strings():
    assert tg.tg_status_string(0) == "TG_OK"
    assert tg.tg_status_string(1) == "TG_ERR_INVALID_ARG"
    assert tg.tg_status_string(2) == "TG_ERR_UNSUPPORTED"
    assert tg.tg_status_string(3) == "TG_ERR_CUDA"
    assert tg.tg_status_string(4) == "TG_ERR_TIMEOUT"
    assert tg.tg_status_string(99) == "TG_ERR_UNKNOWN"


def test_version():
    assert tg.tg_gemm_version() >= 100


def call(M, N, K, A=PA, lda=None, B=PB, ldb=None, C=PC, ldc=None, i=tg.F16, o=tg.F16):
    lda = K if lda is None else lda
    ldb = N if ldb is None else ldb
    ldc = N if ldc is None else ldc
    return tg.tg_gemm(M, N, K, A, lda, B, ldb, C, ldc, i, o, 0)


def path(M, N, K, A=PA, lda=None, B=PB, ldb=None, C=PC, ldc=None, i=tg.F16, o=tg.F16):
    lda = K if lda is None else lda
    ldb = N if ldb is None else ldb
    ldc = N if ldc is None else ldc
    return tg.tg_gemm_path(M, N, K, A, lda, B, ldb, C, ldc, i, o)


@pytest.mark.parametrize("args,status", [
    (dict(M=-1, N=4, K=4), tg.TG_ERR_INVALID_ARG),
    (dict(M=4, N=-1, K=4), tg.TG_ERR_INVALID_ARG),
    (dict(M=4, N=4, K=-1), tg.TG_ERR_INVALID_ARG),
    (dict(M=4, N=4, K=4, C=0), tg.TG_ERR_INVALID_ARG),
    (dict(M=4, N=4, K=4, A=0), tg.TG_ERR_INVALID_ARG),
    (dict(M=4, N=4, K=4, B=0), tg.TG_ERR_INVALID_ARG),
    (dict(M=4, N=4, K=8, lda=7), tg.TG_ERR_INVALID_ARG),
    (dict(M=4, N=8, K=4, ldb=7), tg.TG_ERR_INVALID_ARG),
    (dict(M=4, N=8, K=4, ldc=7), tg.TG_ERR_INVALID_ARG),
    (dict(M=4, N=4, K=4, i=tg.F32, o=tg.F16), tg.TG_ERR_UNSUPPORTED),
    (dict(M=4, N=4, K=4, i=3, o=3), tg.TG_ERR_UNSUPPORTED),
    (dict(M=4, N=4, K=4, i=0, o=tg.F16), tg.TG_ERR_UNSUPPORTED),
    (dict(M=2 ** 31, N=4, K=4), tg.TG_ERR_UNSUPPORTED),
    (dict(M=4, N=4, K=2 ** 31), tg.TG_ERR_UNSUPPORTED),
    (dict(M=2 ** 31 - 1023, N=8, K=8), tg.TG_ERR_UNSUPPORTED),
    # C overlapping A or B
    (dict(M=64, N=64, K=64, C=PA + 64), tg.TG_ERR_INVALID_ARG),
    (dict(M=64, N=64, K=64, C=PB - 100), tg.TG_ERR_INVALID_ARG),
    # a span that would wrap past the end of the address space
    (dict(M=2 ** 30, N=8, K=8, ldc=2 ** 40), tg.TG_ERR_INVALID_ARG),
    # pointers that are not a multiple of their element size
    (dict(M=64, N=64, K=64, A=PA + 1), tg.TG_ERR_INVALID_ARG),
    (dict(M=64, N=64, K=64, B=PB + 3), tg.TG_ERR_INVALID_ARG),
    (dict(M=64, N=64, K=64, C=PC + 1), tg.TG_ERR_INVALID_ARG),
    (dict(M=64, N=64, K=64, C=PC + 2, o=tg.F32), tg.TG_ERR_INVALID_ARG),
    (dict(M=64, N=64, K=64, A=PA + 2, i=tg.F32, o=tg.F32), tg.TG_ERR_INVALID_ARG),
    (dict(M=64, N=64, K=0, C=PC + 1), tg.TG_ERR_INVALID_ARG),
])
def test_invalid_arguments_rejected_on_host(args, status):
    assert call(**args) == status
    assert path(**args) == 0


PD, PBIAS = 0x7F3000000000, 0x7F4000000000


def call_ex(M, N, K, A=PA, B=PB, C=PC, ldc=None, i=tg.F16, o=tg.F16, alpha=1.0, beta=0.0, D=0,
            ldd=None, bias=0, act=tg.ACT_NONE):
    ldc = N if ldc is None else ldc
    ldd = N if ldd is None else ldd
    return tg.tg_gemm_ex(M, N, K, A, K, B, N, C, ldc, i, o, alpha, beta, D, ldd, bias, act, 0)


@pytest.mark.parametrize("args,status", [
    (dict(M=4, N=4, K=4, act=3), tg.TG_ERR_INVALID_ARG),
    (dict(M=4, N=4, K=4, act=-1), tg.TG_ERR_INVALID_ARG),
    (dict(M=0, N=4, K=4, act=7), tg.TG_ERR_INVALID_ARG),
    (dict(M=4, N=4, K=4, beta=1.0, D=0), tg.TG_ERR_INVALID_ARG),
    (dict(M=4, N=8, K=4, beta=1.0, D=PD, ldd=7), tg.TG_ERR_INVALID_ARG),
    (dict(M=4, N=4, K=4, beta=1.0, D=PD + 1), tg.TG_ERR_INVALID_ARG),
    (dict(M=4, N=4, K=4, beta=1.0, D=PD + 2, o=tg.F32), tg.TG_ERR_INVALID_ARG),
    # D overlapping C other than exactly in place
    (dict(M=64, N=64, K=64, beta=1.0, D=PC + 128), tg.TG_ERR_INVALID_ARG),
    (dict(M=64, N=64, K=64, beta=1.0, D=PC, ldd=72, ldc=64), tg.TG_ERR_INVALID_ARG),
    (dict(M=64, N=64, K=0, beta=1.0, D=PC - 2), tg.TG_ERR_INVALID_ARG),
    # bias misaligned or inside C
    (dict(M=4, N=4, K=4, bias=PBIAS + 2), tg.TG_ERR_INVALID_ARG),
    (dict(M=64, N=64, K=64, bias=PC + 64), tg.TG_ERR_INVALID_ARG),
    # the plain call's own checks come first
    (dict(M=4, N=4, K=4, i=tg.F32, o=tg.F16, beta=1.0, D=PD), tg.TG_ERR_UNSUPPORTED),
    (dict(M=64, N=64, K=64, C=PA + 64, beta=1.0, D=PD), tg.TG_ERR_INVALID_ARG),
])
def test_epilogue_arguments_rejected_on_host(args, status):
    assert call_ex(**args) == status


def test_epilogue_degenerate_sizes_are_noops():
    # M == 0 or N == 0 returns before any CUDA call, even with NULL pointers
    assert call_ex(0, 5, 7, A=0, B=0, C=0, beta=2.0, D=0, act=tg.ACT_GELU) == tg.TG_OK
    assert call_ex(5, 0, 7, A=0, B=0, C=0, alpha=3.0, act=tg.ACT_RELU) == tg.TG_OK


def test_degenerate_sizes_are_noops():
    # M == 0 or N == 0 returns before any CUDA call, even with NULL pointers
    assert call(0, 5, 7, A=0, B=0, C=0) == tg.TG_OK
    assert call(5, 0, 7, A=0, B=0, C=0) == tg.TG_OK
    assert path(0, 5, 7) == 0
    # K == 0 is the empty sum: C is zero-filled; A and B may be NULL
    assert path(3, 5, 0, A=0, B=0) == 1


def test_adjacent_operands_are_not_overlap():
    # C starts exactly where A's span ends: legal
    M, N, K = 128, 8, 8
    end_a = PA + ((M - 1) * K + K) * 2
    assert path(M, N, K, C=end_a) == 3
    assert path(M, N, K, C=end_a - 2) == 0       # one element of overlap


def test_path_selection():
    assert path(128, 128, 128, i=tg.F32, o=tg.F32) == 2
    assert path(1024, 2048, 512) == 3
    assert path(1024, 2048, 512, o=tg.F32) == 3
    assert path(8192, 8192, 8192) == 6           # 1024 tiles of 256x256: CTA pairs
    assert path(4096, 16384, 4096) == 6
    assert path(2048, 2048, 1024) == 3           # 64 pair tiles, K < 4096: one CTA per tile
    assert path(2048, 2048, 4096) == 6           # 64 pair tiles, K = 4096: CTA pairs
    assert path(2048, 1792, 4096) == 3           # 56 pair tiles: one CTA per tile
    assert path(4096, 2048, 2048) == 3           # 128 pair tiles, K < 4096
    assert path(3072, 3072, 1024) == 6           # 144 pair tiles
    assert path(2048, 2048, 512) == 3            # K < 1024: the one-CTA kernel
    assert path(8192, 8192, 512) == 3
    assert path(4096, 4096, 1024) == 6
    # row stride not a multiple of 16 bytes -> boundary kernel
    assert path(127, 255, 512) == 4
    assert path(4, 4, 4) == 4
    assert path(1, 255, 17) == 4
    # small M with TMA-addressable operands -> skinny split-K kernel
    assert path(16, 4096, 4096) == 5
    assert path(64, 4096, 4096) == 5
    assert path(65, 4096, 4096) == 3
    assert path(1, 8, 8) == 5
    # base pointer not 16-byte aligned -> boundary kernel
    assert path(128, 256, 512, A=PA + 2) == 4
    assert path(128, 256, 512, B=PB + 8) == 4
    # C alignment does not matter for the path (stores are predicated)
    assert path(128, 256, 512, C=PC + 2) == 3


def test_forced_paths():
    try:
        tg.tg_gemm_force_path(4)
        assert path(1024, 2048, 512) == 4            # boundary can serve an aligned case
        assert path(128, 128, 128, i=tg.F32, o=tg.F32) == 0  # but not fp32 inputs
        tg.tg_gemm_force_path(3)
        assert path(8192, 8192, 8192) == 3
        assert path(127, 255, 512) == 0              # main cannot serve misaligned operands
        tg.tg_gemm_force_path(6)
        assert path(16, 16, 16) == 6
        tg.tg_gemm_force_path(5)
        assert path(64, 512, 512) == 5
        assert path(65, 512, 512) == 0              # skinny serves M <= 64 only
        assert path(127, 255, 512) == 0
        assert call(127, 255, 512) == tg.TG_ERR_UNSUPPORTED
        tg.tg_gemm_force_path(2)
        assert path(64, 64, 64) == 0                 # SIMT is fp32 only
        assert path(3, 5, 0) == 1                    # K == 0 is never forced
    finally:
        tg.tg_gemm_force_path(0)
    assert path(1024, 2048, 512) == 3


def test_force_tiling_validates():
    try:
        for bn, g in [(0, 0), (64, 1), (128, 8), (256, 64)]:
            assert tg.tg_gemm_force_tiling(bn, g) == tg.TG_OK
        for bn, g in [(96, 0), (512, 0), (-1, 0), (0, -1), (0, 65)]:
            assert tg.tg_gemm_force_tiling(bn, g) == tg.TG_ERR_INVALID_ARG
    finally:
        assert tg.tg_gemm_force_tiling(0, 0) == tg.TG_OK


C_CLIENT = r"""
#include <stdio.h>
#include "tg_gemm.h"
int main(void) {
    int bn = 0;
    int split = tg_gemm_main_plan(256, 256, 8192, 1, TG_F16, 152, &bn);
    int path = tg_gemm_path(8192, 8192, 8192, (const void*)0x7F0000000000, 8192,
                            (const void*)0x7F1000000000, 8192, (void*)0x7F2000000000, 8192,
                            TG_F16, TG_F16);
    tg_status bad = tg_gemm(-1, 8, 8, 0, 8, 0, 8, 0, 8, TG_F16, TG_F16, 0);
    printf("%d %s %d %d %d %d\n", tg_gemm_version(), tg_status_string(bad), path, bn, split,
           (int)bad);
    return 0;
}
"""


def test_plain_c_client(tmp_path):
    """The header is plain C: a C99 program (-pedantic, warnings as errors)
    includes it, links libtg_gemm.so and calls host-only entry points."""
    import shutil
    import subprocess
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    src = tmp_path / "client.c"
    src.write_text(C_CLIENT)
    exe = tmp_path / "client"
    libdir = os.path.dirname(tg.library_path())
    r = subprocess.run([cc, "-std=c99", "-Wall", "-Wextra", "-pedantic", "-Werror",
                        f"-I{os.path.dirname(HEADER)}", str(src), f"-L{libdir}", "-ltg_gemm",
                        f"-Wl,-rpath,{libdir}", "-o", str(exe)],
                       capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=60)
    assert r.returncode == 0, r.stderr
    version, status, path, bn, split, code = r.stdout.split()
    assert int(version) == tg.tg_gemm_version()
    assert status == tg.tg_status_string(tg.TG_ERR_INVALID_ARG)
    assert int(code) == tg.TG_ERR_INVALID_ARG
    assert int(path) == 6  # the CTA-pair kernel for 8192^3
    assert (int(bn), int(split)) == (64, 8)


def test_missing_library_fails_loudly():
    """Without the built library every entry point raises: there is no CPU
    or library fallback to run instead (checked in a child process whose
    binding points at a path that does not exist)."""
    import subprocess
    import sys
    code = (
        "import tiled_gemm_tg_gb300 as tg\n"
        "tg._LIB_PATH = '/nonexistent/libtg_gemm.so'\n"
        "tg._lib = None\n"
        "for f in (tg.tg_gemm_version, lambda: tg.tg_gemm(8, 8, 8, 0, 8, 0, 8, 0, 8, tg.F16, tg.F16),\n"
        "          lambda: tg.tg_gemm_path(8, 8, 8, 0, 8, 0, 8, 0, 8, tg.F16, tg.F16)):\n"
        "    try:\n"
        "        f()\n"
        "    except RuntimeError as e:\n"
        "        assert 'is missing' in str(e), e\n"
        "    else:\n"
        "        raise SystemExit('an entry point ran without the library')\n"
        "print('ok')\n")
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    r = subprocess.run([sys.executable, "-c", code], cwd=root, capture_output=True, text=True,
                       timeout=120)
    assert r.returncode == 0 and r.stdout.strip() == "ok", r.stdout + r.stderr


def test_product_path_never_imports_oracle():
    """The CUDA package must not import, load or call the CPU oracle."""
    pkg = os.path.dirname(tg.__file__)
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h", ".cpp")):
                text = open(os.path.join(dirpath, f), encoding="utf-8").read()
                for needle in ("import oracle", "from oracle", "tg_oracle", "tgo_"):
                    assert needle not in text, f"{f} mentions {needle}"


# ------------------------------------------------------------ strided batch

def bpath(batch, M, N, K, sA=None, sB=None, sC=None, A=PA, B=PB, C=PC, lda=None, ldb=None,
          ldc=None, i=tg.F16, o=tg.F16):
    lda = K if lda is None else lda
    ldb = N if ldb is None else ldb
    ldc = N if ldc is None else ldc
    sA = M * lda if sA is None else sA
    sB = K * ldb if sB is None else sB
    sC = M * ldc if sC is None else sC
    return tg.tg_gemm_batched_path(batch, M, N, K, A, lda, sA, B, ldb, sB, C, ldc, sC, i, o)


def bcall(batch, M, N, K, sA=None, sB=None, sC=None, A=PA, B=PB, C=PC, i=tg.F16, o=tg.F16):
    sA = M * K if sA is None else sA
    sB = K * N if sB is None else sB
    sC = M * N if sC is None else sC
    return tg.tg_gemm_batched(batch, M, N, K, A, K, sA, B, N, sB, C, N, sC, i, o, 0)


@pytest.mark.parametrize("args,status", [
    (dict(batch=-1, M=4, N=4, K=4), tg.TG_ERR_INVALID_ARG),
    (dict(batch=2, M=4, N=4, K=4, sA=-16), tg.TG_ERR_INVALID_ARG),
    (dict(batch=2, M=4, N=4, K=4, sC=-16), tg.TG_ERR_INVALID_ARG),
    (dict(batch=65536, M=4, N=4, K=4), tg.TG_ERR_UNSUPPORTED),
    # C matrices overlapping one another
    (dict(batch=2, M=4, N=8, K=4, sC=3 * 8 + 7), tg.TG_ERR_INVALID_ARG),
    (dict(batch=3, M=4, N=8, K=4, sC=0), tg.TG_ERR_INVALID_ARG),
    # C's span over the batch reaching into A's (fake A after C: C=PA - 8 KB)
    (dict(batch=64, M=16, N=16, K=16, C=PA - 8192), tg.TG_ERR_INVALID_ARG),
    # more than 2^31 tiles in the whole batch
    (dict(batch=65535, M=2 ** 20, N=2 ** 20, K=8), tg.TG_ERR_UNSUPPORTED),
])
def test_batched_arguments_rejected_on_host(args, status):
    assert bcall(**args) == status
    b = dict(args)
    assert bpath(b.pop("batch"), b.pop("M"), b.pop("N"), b.pop("K"), **b) == 0


def test_batched_degenerate_sizes_are_noops():
    assert bcall(0, 4, 4, 4, A=0, B=0, C=0) == tg.TG_OK
    assert bcall(3, 0, 4, 4, A=0, B=0, C=0) == tg.TG_OK
    assert bpath(3, 5, 7, 0, A=0, B=0) == 1        # K == 0: zeros in every C_b


def test_batched_path_selection():
    assert bpath(1, 8192, 8192, 8192) == 6
    assert bpath(16, 512, 512, 4096) == 6           # 4 pair tiles x 16 = 64, K = 4096
    assert bpath(16, 512, 512, 1024) == 3           # 64 pair tiles, K < 4096
    assert bpath(36, 512, 512, 1024) == 6           # 144 pair tiles
    assert bpath(15, 512, 512, 4096) == 3           # 60 pair tiles
    assert bpath(16, 512, 512, 512) == 3            # K < 1024
    assert bpath(256, 256, 256, 4096) == 3          # products smaller than 512 x 512
    assert bpath(8, 16, 4096, 4096) == 5            # skinny, one cluster row per matrix
    assert bpath(4, 128, 128, 128, i=tg.F32, o=tg.F32) == 2
    assert bpath(4, 256, 256, 256, sA=0) == 3       # broadcast A: TMA map of one matrix
    assert bpath(4, 256, 256, 256, sB=0) == 3
    assert bpath(4, 256, 256, 256, sA=256 * 256 + 8) == 3   # padded stride
    # strides the TMA engine cannot walk: odd, or overlapping operand matrices
    assert bpath(4, 256, 256, 256, sA=256 * 256 + 4) == 4
    assert bpath(4, 256, 256, 256, sB=128 * 256) == 4
    # a single matrix ignores the strides
    assert bpath(1, 256, 256, 256, sA=5, sB=3, sC=1) == 3


# ------------------------------------------------------------ FP8 E4M3 inputs

def test_e4m3_path_selection():
    E = tg.E4M3
    assert path(8192, 8192, 8192, i=E) == 6
    assert path(8192, 8192, 8192, i=E, o=tg.F32) == 6
    assert path(256, 256, 256, i=E) == 3
    assert path(16, 4096, 4096, i=E) == 3          # no skinny kernel for E4M3
    assert bpath(8, 512, 512, 1024, i=E) == 3
    # the TMA engine must address E4M3 operands: row strides of 16 bytes
    assert path(256, 256, 100, i=E) == 0
    assert call(256, 256, 100, i=E) == tg.TG_ERR_UNSUPPORTED
    assert path(256, 256, 256, i=E, A=PA + 8) == 0
    assert path(256, 256, 112, i=E) == 3
    # E4M3 is an input type only
    assert call(64, 64, 64, i=E, o=E) == tg.TG_ERR_UNSUPPORTED
    assert call(64, 64, 64, i=tg.F16, o=E) == tg.TG_ERR_UNSUPPORTED
    try:
        tg.tg_gemm_force_path(4)
        assert path(256, 256, 256, i=E) == 0        # no boundary kernel for E4M3
        tg.tg_gemm_force_path(5)
        assert path(16, 256, 256, i=E) == 0
        tg.tg_gemm_force_path(6)
        assert path(256, 256, 256, i=E) == 6
    finally:
        tg.tg_gemm_force_path(0)


# ------------------------------------------------------------------ attention

PQ, PK, PV, PO = 0x7F5000000000, 0x7F6000000000, 0x7F7000000000, 0x7F8000000000


def acall(batch=1, Nq=128, Nk=128, d=64, dv=64, Q=PQ, K=PK, V=PV, O=PO, ldq=None, ldk=None,
          ldv=None, ldo=None, sQ=None, sK=None, sV=None, sO=None, i=tg.F16, o=tg.F16):
    ldq = d if ldq is None else ldq
    ldk = d if ldk is None else ldk
    ldv = dv if ldv is None else ldv
    ldo = dv if ldo is None else ldo
    sQ = Nq * ldq if sQ is None else sQ
    sK = Nk * ldk if sK is None else sK
    sV = Nk * ldv if sV is None else sV
    sO = Nq * ldo if sO is None else sO
    return tg.tg_attention(batch, Nq, Nk, d, dv, Q, ldq, sQ, K, ldk, sK, V, ldv, sV, O, ldo, sO,
                           1.0, i, o, 0)


@pytest.mark.parametrize("args,status", [
    (dict(Nq=-1), tg.TG_ERR_INVALID_ARG),
    (dict(batch=-1), tg.TG_ERR_INVALID_ARG),
    (dict(Nk=0), tg.TG_ERR_INVALID_ARG),
    (dict(d=0), tg.TG_ERR_INVALID_ARG),
    (dict(Q=0), tg.TG_ERR_INVALID_ARG),
    (dict(O=0), tg.TG_ERR_INVALID_ARG),
    (dict(ldq=32), tg.TG_ERR_INVALID_ARG),
    (dict(ldo=32), tg.TG_ERR_INVALID_ARG),
    (dict(O=PO + 1), tg.TG_ERR_INVALID_ARG),
    (dict(O=PQ + 64), tg.TG_ERR_INVALID_ARG),            # O inside Q
    (dict(batch=2, sO=100), tg.TG_ERR_INVALID_ARG),       # overlapping O matrices
    (dict(sQ=-8), tg.TG_ERR_INVALID_ARG),
    (dict(i=tg.F32, o=tg.F32), tg.TG_ERR_UNSUPPORTED),
    (dict(i=tg.E4M3), tg.TG_ERR_UNSUPPORTED),
    (dict(o=tg.E4M3), tg.TG_ERR_UNSUPPORTED),
    (dict(Q=PQ + 8), tg.TG_ERR_UNSUPPORTED),              # not TMA-addressable
    (dict(ldk=68), tg.TG_ERR_UNSUPPORTED),
    (dict(batch=2, sV=64 * 64 - 8), tg.TG_ERR_UNSUPPORTED),  # overlapping V matrices
    (dict(batch=65536), tg.TG_ERR_UNSUPPORTED),
])
def test_attention_arguments_rejected_on_host(args, status):
    assert acall(**args) == status


def test_attention_degenerate_sizes_are_noops():
    assert acall(batch=0, Q=0, K=0, V=0, O=0) == tg.TG_OK
    assert acall(Nq=0, Q=0, K=0, V=0, O=0) == tg.TG_OK
    assert acall(dv=0, Q=0, K=0, V=0, O=0) == tg.TG_OK


def test_attention_workspace_checks_on_host():
    # a workspace that is not 256-byte aligned is rejected before any CUDA call
    st = tg.tg_attention_ws(1, 128, 128, 64, 64, PQ, 64, 0, PK, 64, 0, PV, 64, 0, PO, 64, 0, 1.0,
                            tg.F16, tg.F16, 0x7F9000000010, 1 << 20, 0)
    assert st == tg.TG_ERR_INVALID_ARG
    # sizes with no work, or invalid ones, need no workspace
    assert tg.tg_attention_workspace_size(0, 128, 128, 64, 64) == 0
    assert tg.tg_attention_workspace_size(1, 128, -1, 64, 64) == 0


def test_attention_kernel_selection_on_host():
    """The kernel override accepts 0, 1 and 3 only; the kernel query reports
    0 for sizes with no work or out of range, before touching a device."""
    try:
        for bad in (-1, 2, 4, 99):
            assert tg.tg_attention_force_kernel(bad) == tg.TG_ERR_INVALID_ARG
        for ok in (1, 3, 0):
            assert tg.tg_attention_force_kernel(ok) == tg.TG_OK
    finally:
        tg.tg_attention_force_kernel(0)
    assert tg.tg_attention_kernel(0, 128, 128, 64, 64) == 0
    assert tg.tg_attention_kernel(1, 128, 0, 64, 64) == 0
    assert tg.tg_attention_kernel(1, -5, 128, 64, 64) == 0
    assert tg.tg_attention_kernel(65536, 128, 128, 64, 64) == 0


def test_attention_tail_plan_on_host():
    """The last-wave split of kernel 3 is host logic: tiles of 128 query
    rows per head, waves of num_sms, a split only of a last wave holding at
    most 45 % of num_sms tiles (4 key ranges up to 20 %), every range at
    least four 128-key blocks."""
    plan = tg.tg_attention_tail_plan
    # 16 heads x 4096: 512 tiles, 56 in the fourth wave on 152 SMs (37 %)
    assert plan(16, 4096, 4096, 128, 128, 152) == (56, 2)
    # on 148 SMs the fourth wave holds 68 tiles (46 %): no split
    assert plan(16, 4096, 4096, 128, 128, 148) == (0, 0)
    # 4 x 5504 queries: 172 tiles, 20 in the second wave (13 %)
    assert plan(4, 5504, 5504, 128, 128, 152) == (20, 4)
    # fewer key blocks, fewer ranges: 8 -> 2, 12 or 13 -> 3, 16 -> 4, 7 -> none
    assert plan(4, 5504, 1024, 128, 128, 152) == (20, 2)
    assert plan(4, 5504, 1536, 128, 128, 152) == (20, 3)
    assert plan(4, 5504, 1537, 128, 128, 152) == (20, 3)
    assert plan(4, 5504, 2048, 64, 32, 152) == (20, 4)
    assert plan(4, 5504, 800, 128, 128, 152) == (0, 0)
    # a last wave 68 % full, an exact number of waves, one wave or less
    assert plan(16, 2048, 2048, 128, 128, 152) == (0, 0)
    assert plan(19, 4096, 4096, 128, 128, 152) == (0, 0)
    assert plan(1, 128 * 152, 4096, 64, 64, 152) == (0, 0)
    assert plan(1, 128 * 152 + 1, 4096, 64, 64, 152) == (1, 4)
    # the thresholds on 100 SMs: 20 and 45 tiles left are in, 21 and 46 not
    assert plan(120, 100, 4096, 64, 64, 100) == (20, 4)
    assert plan(121, 100, 4096, 64, 64, 100) == (21, 2)
    assert plan(145, 100, 4096, 64, 64, 100) == (45, 2)
    assert plan(146, 100, 4096, 64, 64, 100) == (0, 0)
    # heads kernel 3 does not serve, and sizes with no work
    assert plan(4, 5504, 5504, 160, 128, 152) == (0, 0)
    assert plan(4, 5504, 5504, 128, 256, 152) == (0, 0)
    for args in [(0, 4096, 4096, 128, 128, 152), (16, -1, 4096, 128, 128, 152),
                 (16, 4096, 0, 128, 128, 152), (16, 4096, 4096, 128, 128, 0)]:
        assert plan(*args) == (0, 0), args


def test_attention_tail_plan_invariants():
    """Over a grid of shapes and SM counts: a split takes exactly the tiles
    of the last wave, into 2 to 4 ranges of at least four key blocks, and
    leaves a last wave of at most 45 % of the SMs."""
    for sms in (100, 132, 148, 152, 160):
        for batch in (1, 3, 16, 40):
            for Nq in (1, 128, 1000, 4096, 5504):
                for Nk in (1, 512, 1023, 1024, 3000, 8192):
                    tail, pieces = tg.tg_attention_tail_plan(batch, Nq, Nk, 128, 128, sms)
                    tiles = batch * ((Nq + 127) // 128)
                    n_kv = (Nk + 127) // 128
                    if tail == 0:
                        assert pieces == 0
                        continue
                    waves = (tiles + sms - 1) // sms
                    assert waves >= 2
                    assert tail == tiles - (waves - 1) * sms
                    assert 100 * tail <= 45 * sms
                    assert 2 <= pieces <= 4 and 4 * pieces <= n_kv
                    assert pieces < 4 or 100 * tail <= 20 * sms


@pytest.mark.parametrize("tiles,pairs,want", [
    (1024, 76, 36),    # 8192^3: 13 whole waves and 36 tiles, cut into 72 halves
    (1024, 74, 0),     # 13 waves and 62 tiles: more than half a wave, none cut
    (77, 76, 1), (152, 76, 0), (153, 76, 1), (100, 76, 24), (114, 76, 38), (115, 76, 0),
    (64, 76, 0),       # one wave, 128 halves would not fit
    (38, 76, 38), (39, 76, 0), (1, 76, 1), (1, 1, 0), (5, 2, 1),
    (0, 76, 0), (10, 0, 0), (-3, 76, 0),
])
def test_pair_split_tail_rule(tiles, pairs, want):
    """The short-last-wave rule of the pair kernel, on the host."""
    got = tg.tg_gemm_pair_split_tail(tiles, pairs)
    assert got == want
    if got:
        last = tiles - pairs * ((tiles - 1) // pairs)
        assert got == last and 2 * last <= pairs


@pytest.mark.parametrize("tiles,kblocks,sms,want", [
    (2, 8, 152, 8),        # 127 x 255 x 512: two tiles, one k-block per CTA
    (15, 8, 152, 8), (19, 8, 152, 8), (20, 8, 152, 4), (38, 8, 152, 4), (39, 8, 152, 2),
    (76, 8, 152, 2), (77, 8, 152, 1), (128, 16, 152, 1),
    (1, 1, 152, 1), (1, 2, 152, 2), (1, 3, 152, 2), (1, 7, 152, 4), (1, 100, 152, 8),
    (3, 8, 4, 1), (2, 8, 4, 2),
    (0, 8, 152, 1), (5, 0, 152, 1), (5, 8, 0, 1), (-1, 8, 152, 1),
])
def test_boundary_split_rule(tiles, kblocks, sms, want):
    """The boundary kernel's split over K, on the host: the largest cluster
    of 2, 4 or 8 CTAs per output tile that keeps every CTA on its own SM and
    gives each at least one k-block."""
    got = tg.tg_gemm_boundary_split(tiles, kblocks, sms)
    assert got == want
    if got > 1:
        assert tiles * got <= sms and got <= kblocks
        assert got == 8 or tiles * 2 * got > sms or 2 * got > kblocks


@pytest.mark.parametrize("M,N,K,batch,want", [
    # measured best on GB300 (tile width / split): the estimate picks them
    ((256, 256, 8192, 1, (64, 8))),
    # 16 clusters of 8: more than GB300 holds at once, so on the device
    # the library falls back to 64 / 4, the measured best
    ((512, 512, 8192, 1, (128, 8))),
    ((1024, 1024, 4096, 1, (128, 2))),
    ((304, 520, 1024, 1, (64, 4))),
    ((512, 1024, 2048, 1, (128, 4))),
    ((256, 4096, 4096, 1, (128, 2))),
    # unsplit, but wider tiles in fewer waves than the default width
    ((2048, 2048, 1024, 1, (256, 1))),
    ((4096, 1024, 2048, 1, (256, 1))),
    ((1536, 1536, 1024, 1, (128, 1))),
    # no split: the tiles fill the GPU, or K is too short to pay for it
    ((128, 256, 512, 1, (64, 1))),
    ((1024, 2048, 512, 1, (128, 1))),
    ((1024, 1024, 1024, 1, (64, 1))),
    ((2048, 1024, 512, 1, (128, 1))),
    ((8192, 8192, 8192, 1, (256, 1))),
    ((256, 256, 256, 256, (256, 1))),
    # many tiles, but no wider than N needs
    ((72, 64, 64, 65535, (64, 1))),
    ((4096, 100, 1024, 8, (128, 1))),
])
def test_main_plan(M, N, K, batch, want):
    """The one-CTA kernel's tile width and split over K, on the host."""
    assert tg.tg_gemm_main_plan(M, N, K, batch, tg.F16, 152) == want


def test_main_plan_rules():
    """Whatever the estimate picks, a split keeps every CTA on its own SM,
    at least one k-block each, and only for tiles that leave half the SMs
    idle; E4M3 never gets 64-column tiles; bad arguments give (0, 0)."""
    rng = np.random.default_rng(5)
    for _ in range(400):
        M, N = (int(v) for v in rng.integers(65, 4097, 2))
        K = int(rng.integers(1, 20000))
        batch = int(rng.integers(1, 4))
        for dt, bk in ((tg.F16, 64), (tg.E4M3, 128)):
            bn, split = tg.tg_gemm_main_plan(M, N, K, batch, dt, 152)
            assert bn in ((128, 256) if dt == tg.E4M3 else (64, 128, 256))
            assert split in (1, 2, 4, 8)
            if split > 1:
                tiles = -(-M // 128) * -(-N // bn) * batch
                assert 2 * tiles <= 152 and tiles * split <= 152 and split <= -(-K // bk)
    assert tg.tg_gemm_main_plan(0, 8, 8, 1, tg.F16, 152) == (0, 0)
    assert tg.tg_gemm_main_plan(8, 8, 8, 1, tg.F32, 152) == (0, 0)


def test_main_plan_width_never_wider_than_n():
    """Narrow products, alone or in batches up to 65535: the tile width is
    at most N rounded up to 64 or 128 columns (128 at least for E4M3, whose
    B copies are 128 elements wide), since wider tiles only multiply zeros."""
    rng = np.random.default_rng(6)
    for _ in range(300):
        M = int(rng.integers(65, 5000))
        N = int(rng.integers(1, 129))
        K = int(rng.integers(1, 5000))
        batch = int(rng.integers(1, 65536))
        cap = 64 if N <= 64 else 128
        bn, split = tg.tg_gemm_main_plan(M, N, K, batch, tg.F16, 152)
        assert bn <= cap, (M, N, K, batch, bn)
        bn8, _ = tg.tg_gemm_main_plan(M, N, K, batch, tg.E4M3, 152)
        assert bn8 == 128, (M, N, K, batch, bn8)


def test_force_split_k_arguments():
    for bad in (-1, 3, 5, 6, 16):
        assert tg.tg_gemm_force_split_k(bad) == tg.TG_ERR_INVALID_ARG
    for ok in (1, 2, 4, 8, 0):
        assert tg.tg_gemm_force_split_k(ok) == tg.TG_OK


def test_force_split_tail_arguments():
    assert tg.tg_gemm_force_split_tail(-2) == tg.TG_ERR_INVALID_ARG
    for v in (0, 5, -1):
        assert tg.tg_gemm_force_split_tail(v) == tg.TG_OK


def test_force_stages_arguments():
    for bad in (-1, 1, 9, 100):
        assert tg.tg_gemm_force_stages(bad) == tg.TG_ERR_INVALID_ARG
    for ok in (2, 3, 8, 0):
        assert tg.tg_gemm_force_stages(ok) == tg.TG_OK
