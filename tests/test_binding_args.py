"""The Python binding rejects tensors the C ABI cannot use, before any library call.

The C ABI receives raw pointers and row pitches; a host tensor, a wrong shape, a
strided layout or an undersized buffer would otherwise reach the kernels as a device
address.  These run without a GPU: every call here fails validation (shapes, dtypes
and layouts are checked first, device placement last), so nothing is launched.
"""
import pytest
import torch

import tensor_core_matrix_gb300 as tcm
from tensor_core_matrix_gb300 import build as tcm_build

BF, F32, E4 = torch.bfloat16, torch.float32, torch.float8_e4m3fn


@pytest.fixture(scope="module", autouse=True)
def lib():
    tcm_build.build()  # the size queries (tcm_mx_scales_bytes, ...) are host-only library calls
    return tcm.load_library()


def z(*shape, dtype=BF):
    return torch.zeros(shape, dtype=dtype)


def raises(fn, text):
    with pytest.raises(ValueError, match=text):
        fn()


def test_gemm_ex_checks_shapes_dtypes_and_device():
    A, B, D = z(64, 32), z(48, 32), z(64, 48)
    raises(lambda: tcm.tcm_gemm_ex(A, z(48, 16), D), "K")
    raises(lambda: tcm.tcm_gemm_ex(A, B, z(64, 40)), "D must be 64 x 48")
    raises(lambda: tcm.tcm_gemm_ex(A, B, D, C=z(48, 64), beta=1.0), "C must be 64 x 48")
    raises(lambda: tcm.tcm_gemm_ex(A, B, D, C=z(64, 48, dtype=F32), beta=1.0), "C: dtype")
    raises(lambda: tcm.tcm_gemm_ex(A, B, D, bias=z(47)), "bias must be")
    raises(lambda: tcm.tcm_gemm_ex(A, B, D, bias=z(48, dtype=F32)), "bias: dtype")
    raises(lambda: tcm.tcm_gemm_ex(z(32, 64).t(), B, D), "unit column stride")
    raises(lambda: tcm.tcm_gemm_ex(A, B, D, a_scale=torch.ones(1, dtype=torch.float64)), "a_scale")
    raises(lambda: tcm.tcm_gemm_ex(A, B, z(64, 48, dtype=E4)), "D: dtype")
    raises(lambda: tcm.tcm_gemm_ex(A, B, D), "CUDA tensor")
    raises(lambda: tcm.tcm_gemm_ex(z(64, 16, dtype=torch.uint8), z(48, 16, dtype=torch.uint8), D,
                                   a_fmt="e2m1", b_fmt="e2m1", bias=z(48, dtype=F32)), "bias: dtype")


def test_gemm_fused_bias_of_fp8_output_is_bf16():
    A, B = z(64, 32, dtype=E4), z(48, 32, dtype=E4)
    D8 = z(64, 48, dtype=E4)
    raises(lambda: tcm.tcm_gemm_fused(A, B, D8, bias=z(48, dtype=torch.float16)), "bias: dtype")
    raises(lambda: tcm.tcm_gemm_fused(A, B, D8, amax=z(1, dtype=BF)), "amax")
    raises(lambda: tcm.tcm_gemm_fused(A, B, D8, act="tanh"), "activation")
    raises(lambda: tcm.tcm_gemm_fused(A, B, D8, bias=z(48)), "CUDA tensor")


def test_gemm_requires_dense_matching_operands():
    A, B, D = z(64, 32), z(48, 32), z(64, 48)
    raises(lambda: tcm.tcm_gemm(A, z(48, 32, dtype=torch.float16), D), "B: dtype")
    raises(lambda: tcm.tcm_gemm(A, B, z(128, 48)[::2]), "contiguous")
    raises(lambda: tcm.tcm_gemm(A, B, D, C=z(64, 48, dtype=F32), beta=1.0), "C: dtype")
    raises(lambda: tcm.tcm_gemm(A, B, D), "CUDA tensor")


def test_sparse_entry_points_check_compressed_shapes():
    Ac, meta, B, D = z(64, 64), z(64, 4, dtype=torch.int32), z(48, 128), z(64, 48)
    raises(lambda: tcm.tcm_gemm_sp(Ac, z(64, 3, dtype=torch.int32), B, D), "meta must be 64 x 4")
    raises(lambda: tcm.tcm_gemm_sp(Ac, meta.to(torch.int64), B, D), "meta: dtype")
    raises(lambda: tcm.tcm_gemm_sp(Ac, meta, z(48, 96), D), "B must be")
    raises(lambda: tcm.tcm_gemm_sp(z(64, 128)[:, :64], meta, B, D), "contiguous")
    raises(lambda: tcm.tcm_gemm_sp(Ac, meta, B, D), "CUDA tensor")
    raises(lambda: tcm.tcm_sp_compress(z(64, 48)), "multiple of 32")
    raises(lambda: tcm.tcm_sp_compress(z(64, 128), A_comp=z(64, 32)), "A_comp must be 64 x 64")
    raises(lambda: tcm.tcm_sp_compress(z(64, 128)), "CUDA tensor")
    raises(lambda: tcm.tcm_sp_decompress(Ac, z(64, 2, dtype=torch.int32)), "meta must be")
    raises(lambda: tcm.tcm_gemm_sp_tc(Ac, z(16, dtype=torch.uint8), B, D), "meta_tc holds")
    raises(lambda: tcm.tcm_sp_meta_pack(z(64, 4, dtype=torch.int32), 96), "meta must be")


def test_block_scaled_entry_points_check_scale_sizes():
    A, B, D = z(128, 64, dtype=E4), z(128, 64, dtype=E4), z(128, 128)
    S = z(tcm.tcm_mx_scales_bytes(128, 64), dtype=torch.uint8)
    raises(lambda: tcm.tcm_gemm_mx(A, S[:-1], B, S, D), "a_scales holds")
    raises(lambda: tcm.tcm_gemm_mx(A, S, z(128, 32, dtype=E4), S, D), "B must be")
    raises(lambda: tcm.tcm_gemm_mx(A, S, B, S, D, bias=z(128, dtype=F32)), "bias: dtype")
    raises(lambda: tcm.tcm_gemm_mx(A, S, B, S, D), "CUDA tensor")
    raises(lambda: tcm.tcm_mx_pack_scales(z(128, 3, dtype=torch.uint8), 64), "scales must be")
    A4, B4 = z(128, 128, dtype=torch.uint8), z(128, 128, dtype=torch.uint8)
    S4 = z(tcm.tcm_nvfp4_scales_bytes(128, 256), dtype=torch.uint8)
    raises(lambda: tcm.tcm_gemm_nvfp4(A4, S4, z(128, 64, dtype=torch.uint8), S4, D), "B must be")
    raises(lambda: tcm.tcm_gemm_nvfp4(A4, S4[:100], B4, S4, D), "a_scales holds")
    raises(lambda: tcm.tcm_gemm_nvfp4(A4, S4, B4, S4, D), "CUDA tensor")
    raises(lambda: tcm.tcm_nvfp4_pack_scales(z(128, 3, dtype=torch.uint8), 64), "scales must be")
