"""K == 0 through every GEMM entry point that accepts it: no MMA runs, the accumulator
is never read, and D = beta * C + bias exactly as the oracle computes it ("NVIDIA MMA",
section "从 FMA 到 MMA，再到 GEMM": D = A B + C with an empty sum).  D is pre-filled with
NaN, so an output the epilogue skipped fails."""
import numpy as np
import pytest
import torch

import oracle
import synth_inputs as si
from parity import FMT_OF, dev, ratio

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _build():
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(0)
    import tensor_core_matrix_gb300 as tcm
    tcm.tcm_clear_device_status()


@pytest.fixture
def tcm():
    import tensor_core_matrix_gb300 as t
    yield t
    t.tcm_set_config_override(0, 0, 0, 0, 0)


def expected(C, beta, bias=None):
    M, N = C.shape
    ref, S = oracle.gemm(np.zeros((M, 0), np.uint16), np.zeros((N, 0), np.uint16), "bf16", "bf16",
                         C=si.codes(C), c_fmt=FMT_OF[C.dtype], bias=None if bias is None else si.codes(bias),
                         bias_fmt=FMT_OF[bias.dtype] if bias is not None else "bf16", alpha=1.0, beta=beta)
    return ref, S


def check(tcm, D, C, beta, bias=None):
    code, site = tcm.tcm_get_device_status()
    assert code == 0, (code, site)
    ref, S = expected(C, beta, bias)
    assert ratio(D.cpu(), ref, S) <= 1.0


@pytest.mark.parametrize("cg,bn", [(0, 0), (2, 256), (1, 128), (1, 32)])
@pytest.mark.parametrize("in_dtype,out_dtype", [(torch.bfloat16, torch.float32), (torch.float8_e4m3fn, torch.bfloat16)])
def test_dense_k0(tcm, cg, bn, in_dtype, out_dtype):
    tcm.tcm_set_config_override(cg, bn, 0, 0, 0)
    d = dev()
    M, N = 384, 544
    g = si.generator(40 + bn)
    C = si.normal((M, N), g, dtype=FMT_OF[out_dtype])
    bias = si.normal((N,), g, dtype=FMT_OF[out_dtype])
    A = torch.empty((M, 0), dtype=in_dtype, device=d)
    B = torch.empty((N, 0), dtype=in_dtype, device=d)
    D = torch.full((M, N), float("nan"), dtype=out_dtype, device=d)
    tcm.tcm_gemm_ex(A, B, D, C=C.to(d), beta=0.5, bias=bias.to(d))
    check(tcm, D, C, 0.5, bias)


def test_mx_k0(tcm):
    d = dev()
    M, N = 300, 512
    C = si.normal((M, N), si.generator(41), dtype="bf16")
    A = torch.empty((M, 0), dtype=torch.float8_e4m3fn, device=d)
    B = torch.empty((N, 0), dtype=torch.float8_e4m3fn, device=d)
    S0 = torch.empty(0, dtype=torch.uint8, device=d)
    D = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device=d)
    tcm.tcm_gemm_mx(A, S0, B, S0, D, C=C.to(d), beta=2.0)
    check(tcm, D, C, 2.0)


def test_nvfp4_k0(tcm):
    d = dev()
    M, N = 256, 384
    C = si.normal((M, N), si.generator(42), dtype="f32")
    A = torch.empty((M, 0), dtype=torch.uint8, device=d)
    B = torch.empty((N, 0), dtype=torch.uint8, device=d)
    S0 = torch.empty(0, dtype=torch.uint8, device=d)
    D = torch.full((M, N), float("nan"), dtype=torch.float32, device=d)
    tcm.tcm_gemm_nvfp4(A, S0, B, S0, D, C=C.to(d), beta=-1.0)
    check(tcm, D, C, -1.0)


@pytest.mark.parametrize("tc", [False, True])
@pytest.mark.parametrize("cg,bn", [(2, 256), (1, 128)])
def test_sparse_k0(tcm, tc, cg, bn):
    tcm.tcm_set_config_override(cg, bn, 0, 0, 0)
    d = dev()
    M, N = 512, 256
    C = si.normal((M, N), si.generator(43), dtype="bf16")
    Ac = torch.empty((M, 0), dtype=torch.bfloat16, device=d)
    meta = torch.empty((M, 0), dtype=torch.int32, device=d)
    B = torch.empty((N, 0), dtype=torch.bfloat16, device=d)
    D = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device=d)
    if tc:
        tcm.tcm_gemm_sp_tc(Ac, torch.empty(0, dtype=torch.uint8, device=d), B, D, C=C.to(d), beta=0.25)
    else:
        tcm.tcm_gemm_sp(Ac, meta, B, D, C=C.to(d), beta=0.25)
    check(tcm, D, C, 0.25)
