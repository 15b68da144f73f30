"""GPU parity of the MXFP4 GEMM (tcm_gemm_mx with E2M1 operands: kind::mxf4nvf4.block_scale
.scale_vec::2X, UE8M0 scales per 32 in the MX blocked layout) against the oracle."""
import numpy as np
import pytest
import torch

import oracle
import synth_inputs as si
from parity import dev, ratio, sample_indices

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
    t.tcm_set_config_override()


def run_mxfp4(tcm, A, SA, B, SB, out=torch.bfloat16, C=None, beta=0.0, alpha=1.0, bias=None):
    """Row-major E8M0 codes are packed on the device by the library, then the GEMM runs."""
    d = dev()
    M, K = A.shape[0], 2 * A.shape[1]
    N = B.shape[0]
    D = torch.full((M, N), float("nan"), dtype=out, device=d)
    pa = tcm.tcm_mx_pack_scales(SA.to(d), K)
    pb = tcm.tcm_mx_pack_scales(SB.to(d), K)
    tcm.tcm_gemm_mx(A.to(d), pa, B.to(d), pb, D, C=None if C is None else C.to(d), alpha=alpha, beta=beta,
                    bias=None if bias is None else bias.to(d), fmt="e2m1")
    code, site = tcm.tcm_get_device_status()
    assert code == 0, (code, site)
    return D.cpu()


def oracle_mxfp4(A, SA, B, SB, **kw):
    return oracle.gemm_mx(A.numpy(), SA.numpy(), B.numpy(), SB.numpy(), "e2m1", "e2m1", block=32, sf_fmt="e8m0", **kw)


VARIANTS = [(0, 0), (1, 128), (1, 256), (2, 256)]


@pytest.mark.parametrize("cg,bn", VARIANTS)
@pytest.mark.parametrize("M,N,K", [(128, 128, 256), (256, 512, 1024), (300, 520, 768), (1000, 136, 256)])
def test_mxfp4_integer_exact(tcm, cg, bn, M, N, K):
    """E2M1 values times power-of-two block scales 0.5, 1, 2 (E8M0 126..128): every partial sum is exact
    in fp32; a wrong scale byte (scale-factor id) or a wrong atom would change the result."""
    tcm.tcm_set_config_override(cg, bn)
    g = si.generator(M + N + K + cg + bn + 1)
    A = si.pack_fp4(torch.randint(0, 16, (M, K), generator=g).to(torch.uint8))
    B = si.pack_fp4(torch.randint(0, 16, (N, K), generator=g).to(torch.uint8))
    SA = torch.randint(126, 129, (M, K // 32), generator=g).to(torch.uint8)
    SB = torch.randint(126, 129, (N, K // 32), generator=g).to(torch.uint8)
    D = run_mxfp4(tcm, A, SA, B, SB, out=torch.float32)
    ref, _ = oracle_mxfp4(A, SA, B, SB)
    assert np.array_equal(D.double().numpy(), ref)


@pytest.mark.parametrize("cg,bn", VARIANTS[1:])
def test_mxfp4_normal_data_bound(tcm, cg, bn):
    tcm.tcm_set_config_override(cg, bn)
    c = si.mxfp4_case(640, 768, 1024, seed=9)
    g = si.generator(10)
    C = si.normal((640, 768), g)
    bias = si.normal((768,), g)
    D = run_mxfp4(tcm, c["A"], c["SA"], c["B"], c["SB"], C=C, beta=0.5, alpha=0.75, bias=bias)
    ref, S = oracle_mxfp4(c["A"], c["SA"], c["B"], c["SB"], C=si.codes(C), c_fmt="bf16", beta=0.5, alpha=0.75,
                          bias=si.codes(bias))
    assert ratio(D, ref, S, scale=0.75) <= 1.0


def test_mxfp4_8192_sampled(tcm):
    c = si.mxfp4_case()
    D = run_mxfp4(tcm, c["A"], c["SA"], c["B"], c["SB"])
    rows, cols = sample_indices(8192, 8192)
    ref, S = oracle_mxfp4(c["A"], c["SA"], c["B"], c["SB"], rows=rows, cols=cols)
    assert ratio(D, ref, S, rows=rows, cols=cols) <= 1.0
    assert not torch.isnan(D).any()


def test_mxfp4_rejects_mixed_and_ragged_k(tcm):
    d = dev()
    A = torch.zeros((128, 64), dtype=torch.uint8, device=d)
    S = torch.zeros(tcm.tcm_mx_scales_bytes(128, 128), dtype=torch.uint8, device=d)
    D = torch.empty((128, 128), dtype=torch.bfloat16, device=d)
    with pytest.raises(tcm.TcmError, match="INVALID_ARG"):  # K = 128: not a whole 256-value stage
        tcm.tcm_gemm_mx(A, S, A, S, D, fmt="e2m1")
