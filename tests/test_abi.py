"""Host-side checks of the C ABI that need no GPU.

The shared library must load, export every function that include/tcm.h
declares, and reject bad arguments synchronously (before any CUDA call), so
these run on a build host without a device.  Pointers passed here are never
dereferenced: every call is rejected by validation first.
"""
import ctypes
import os
import re

import pytest

import tensor_core_matrix_gb300 as tcm
from tensor_core_matrix_gb300 import build as tcm_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "tcm.h")


@pytest.fixture(scope="module")
def lib():
    tcm_build.build()
    return tcm.load_library()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(tcm_[a-z_0-9]+)\s*\(", text)))


def test_header_declares_the_binding_exports():
    assert set(declared_functions()) == set(tcm.EXPORTS)


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_status_strings_and_version(lib):
    for code, name in tcm.STATUS_NAMES.items():
        assert tcm.tcm_status_string(code) == name
    assert tcm.tcm_version() >= 100


ALIGNED = 0x10000
BF16, F16, F32, E4M3, E5M2 = 0, 1, 2, 3, 4


def gemm_ex(lib, **kw):
    a = dict(M=64, N=64, K=64, a_dtype=BF16, A=ALIGNED, lda=64, b_dtype=BF16, B=ALIGNED, ldb=64,
             C=None, ldc=0, D=ALIGNED, ldd=64, out_dtype=BF16, alpha=1.0, beta=0.0,
             a_scale=None, b_scale=None, bias=None, stream=None)
    a.update(kw)
    return lib.tcm_gemm_ex(a["M"], a["N"], a["K"], a["a_dtype"], a["A"], a["lda"], a["b_dtype"], a["B"],
                           a["ldb"], a["C"], a["ldc"], a["D"], a["ldd"], a["out_dtype"], a["alpha"],
                           a["beta"], a["a_scale"], a["b_scale"], a["bias"], a["stream"])


@pytest.mark.parametrize("kw,status", [
    (dict(M=0), 1), (dict(N=-1), 1), (dict(K=-5), 1), (dict(D=None), 1), (dict(A=None), 1),
    (dict(beta=1.0, C=None), 1), (dict(lda=32), 1), (dict(ldd=32), 1),
    (dict(A=ALIGNED + 2), 3), (dict(D=ALIGNED + 8), 3), (dict(lda=68), 3), (dict(ldd=66), 3),
    (dict(a_dtype=BF16, b_dtype=F16), 2), (dict(a_dtype=F32, b_dtype=F32), 2),
    (dict(a_dtype=E4M3, b_dtype=BF16), 2), (dict(out_dtype=E4M3), 2),
    (dict(a_dtype=E4M3, b_dtype=E5M2, K=24, lda=24, ldb=24), 3),
])
def test_gemm_ex_rejects_bad_arguments(lib, kw, status):
    assert gemm_ex(lib, **kw) == status


def test_gemm_rejects_fp8_without_scales(lib):
    assert lib.tcm_gemm(64, 64, 64, E4M3, ALIGNED, ALIGNED, None, ALIGNED, 1.0, 0.0, BF16, None) == 2


@pytest.mark.parametrize("M,K,dtype,lda,status", [
    (64, 48, BF16, 48, 1), (64, 64, F32, 64, 2), (-1, 64, BF16, 64, 1), (64, 64, BF16, 32, 1),
    (64, 64, BF16, 68, 3),
])
def test_sparse_rejects_bad_arguments(lib, M, K, dtype, lda, status):
    assert lib.tcm_sp_compress(M, K, dtype, ALIGNED, lda, ALIGNED, ALIGNED, None) == status
    assert lib.tcm_sp_decompress(M, K, dtype, ALIGNED, ALIGNED, ALIGNED, lda, None) == status


def test_library_is_built_for_sm_103a_only():
    src = open(os.path.join(ROOT, "tensor_core_matrix_gb300", "build.py")).read()
    assert "arch=compute_103a,code=sm_103a" in src


@pytest.mark.parametrize("a,b,K,status", [(E4M3, BF16, 64, 2), (BF16, BF16, 64, 2), (E4M3, E5M2, 48, 1),
                                          (E4M3, E4M3, -32, 1)])
def test_gemm_mx_rejects_bad_arguments(lib, a, b, K, status):
    assert lib.tcm_gemm_mx(64, 64, K, a, ALIGNED, ALIGNED, b, ALIGNED, ALIGNED, None, ALIGNED, 1.0, 0.0, None,
                           BF16, None) == status


def fused(lib, **kw):
    a = dict(M=64, N=64, K=64, a_dtype=BF16, A=ALIGNED, lda=64, b_dtype=BF16, B=ALIGNED, ldb=64,
             C=None, ldc=0, D=ALIGNED, ldd=64, out_dtype=BF16, alpha=1.0, beta=0.0,
             a_scale=None, b_scale=None, bias=None, act=0, d_scale=None, amax=None, stream=None)
    a.update(kw)
    return lib.tcm_gemm_fused(a["M"], a["N"], a["K"], a["a_dtype"], a["A"], a["lda"], a["b_dtype"], a["B"],
                              a["ldb"], a["C"], a["ldc"], a["D"], a["ldd"], a["out_dtype"], a["alpha"],
                              a["beta"], a["a_scale"], a["b_scale"], a["bias"], a["act"], a["d_scale"],
                              a["amax"], a["stream"])


@pytest.mark.parametrize("kw,status", [
    (dict(act=3), 1), (dict(act=-1), 1), (dict(M=0), 1),
    (dict(out_dtype=E4M3, beta=1.0, C=ALIGNED, ldc=64), 2),   # no FP8 C
    (dict(out_dtype=E4M3, ldd=72), 3),                        # 72 bytes: not a multiple of 16
    (dict(amax=ALIGNED + 2), 3), (dict(d_scale=ALIGNED + 1), 3),
    (dict(a_dtype=E4M3, b_dtype=BF16), 2),
])
def test_gemm_fused_rejects_bad_arguments(lib, kw, status):
    assert fused(lib, **kw) == status


def test_gemm_ex_still_rejects_fp8_output(lib):
    assert gemm_ex(lib, out_dtype=E5M2) == 2


E2M1 = 5


@pytest.mark.parametrize("kw,status", [
    (dict(a_dtype=E2M1, b_dtype=E4M3, K=64, lda=64, ldb=64), 2),                # K not a multiple of 128
    (dict(a_dtype=E2M1, b_dtype=E4M3, K=128, lda=160, ldb=128), 3),             # 80-byte FP4 rows
    (dict(a_dtype=E4M3, b_dtype=E2M1, K=128, lda=128, ldb=128, B=ALIGNED + 16), 3),  # FP4 base not 32-aligned
    (dict(a_dtype=E2M1, b_dtype=BF16, K=128, lda=128, ldb=128), 2),
])
def test_gemm_ex_fp4_argument_rules(lib, kw, status):
    assert gemm_ex(lib, **kw) == status


@pytest.mark.parametrize("K,out,D,status", [(128, BF16, ALIGNED, 1), (256, E4M3, ALIGNED, 2),
                                            (256, BF16, ALIGNED + 8, 3), (-256, BF16, ALIGNED, 1)])
def test_gemm_nvfp4_rejects_bad_arguments(lib, K, out, D, status):
    assert lib.tcm_gemm_nvfp4(64, 64, K, ALIGNED, ALIGNED, ALIGNED, ALIGNED, None, D, 1.0, 0.0, None, out,
                              None) == status


def test_nvfp4_scales_bytes(lib):
    assert lib.tcm_nvfp4_scales_bytes(130, 256) == 2 * 4 * 512
    assert lib.tcm_nvfp4_scales_bytes(1, 64) == 512
    assert lib.tcm_nvfp4_scales_bytes(1, 24) == -1


def test_sp_meta_tc_bytes_and_rejections(lib):
    assert lib.tcm_sp_meta_tc_bytes(130, 160) == 2 * 2 * 2048
    assert lib.tcm_sp_meta_tc_bytes(1, 48) == -1
    assert lib.tcm_sp_meta_pack(64, 48, ALIGNED, ALIGNED, None) == 1
    assert lib.tcm_sp_meta_pack(64, 64, ALIGNED, ALIGNED + 4, None) == 3
    assert lib.tcm_gemm_sp_tc(64, 64, 48, BF16, ALIGNED, ALIGNED, ALIGNED, None, ALIGNED, 1.0, 0.0, BF16, None) == 1
    assert lib.tcm_gemm_sp_tc(64, 64, 64, E4M3, ALIGNED, ALIGNED, ALIGNED, None, ALIGNED, 1.0, 0.0, BF16, None) == 2
