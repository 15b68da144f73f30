"""GPU parity of the NVFP4 GEMM (kind::mxf4nvf4.block_scale.scale_vec::4X) against the oracle."""
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
    t.tcm_set_config_override(0, 0, 0, 0, 0)


def run_nv(tcm, A, SA, B, SB, out=torch.bfloat16, C=None, beta=0.0, alpha=1.0, bias=None):
    """Row-major UE4M3 codes are packed on the device by the library, then the GEMM runs."""
    d = dev()
    M, K = A.shape[0], 2 * A.shape[1]
    N = B.shape[0]
    D = torch.full((M, N), float("nan"), dtype=out, device=d)
    pa = tcm.tcm_nvfp4_pack_scales(SA.to(d), K)
    pb = tcm.tcm_nvfp4_pack_scales(SB.to(d), K)
    tcm.tcm_gemm_nvfp4(A.to(d), pa, B.to(d), pb, D, C=None if C is None else C.to(d), alpha=alpha, beta=beta,
                       bias=None if bias is None else bias.to(d))
    code, site = tcm.tcm_get_device_status()
    assert code == 0, (code, site)
    return D.cpu()


def oracle_nv(A, SA, B, SB, **kw):
    return oracle.gemm_mx(A.numpy(), SA.numpy(), B.numpy(), SB.numpy(), "e2m1", "e2m1", block=16, sf_fmt="ue4m3",
                          **kw)


@pytest.mark.parametrize("rows,K", [(1, 256), (130, 512), (300, 1024), (8192, 8192)])
def test_nvfp4_pack_scales_bit_exact(tcm, rows, K):
    g = si.generator(rows + K)
    SC = torch.randint(0, 127, (rows, K // 16), generator=g).to(torch.uint8)
    got = tcm.tcm_nvfp4_pack_scales(SC.to(dev()), K).cpu().numpy()
    assert np.array_equal(got, oracle.mx_pack_scales(SC.numpy(), K, block=16, pad=0x38))


VARIANTS = [(0, 0), (1, 128), (1, 256), (2, 256)]


@pytest.mark.parametrize("cg,bn", VARIANTS)
@pytest.mark.parametrize("M,N,K", [(128, 128, 256), (256, 512, 1024), (300, 520, 768), (1000, 136, 256)])
def test_nvfp4_integer_exact(tcm, cg, bn, M, N, K):
    """E2M1 values times power-of-two scales 0.5, 1, 2: every partial sum is exact in fp32."""
    tcm.tcm_set_config_override(cg, bn)
    g = si.generator(M + N + K + cg + bn)
    A = si.pack_fp4(torch.randint(0, 16, (M, K), generator=g).to(torch.uint8))
    B = si.pack_fp4(torch.randint(0, 16, (N, K), generator=g).to(torch.uint8))
    pick = torch.tensor([0x30, 0x38, 0x40], dtype=torch.uint8)
    SA = pick[torch.randint(0, 3, (M, K // 16), generator=g)]
    SB = pick[torch.randint(0, 3, (N, K // 16), generator=g)]
    D = run_nv(tcm, A, SA, B, SB, out=torch.float32)
    ref, _ = oracle_nv(A, SA, B, SB)
    assert np.array_equal(D.double().numpy(), ref)


@pytest.mark.parametrize("cg,bn", VARIANTS[1:])
def test_nvfp4_normal_data_bound(tcm, cg, bn):
    tcm.tcm_set_config_override(cg, bn)
    c = si.nvfp4_case(640, 768, 1024, seed=9)
    g = si.generator(10)
    C = si.normal((640, 768), g)
    bias = si.normal((768,), g)
    D = run_nv(tcm, c["A"], c["SA"], c["B"], c["SB"], C=C, beta=0.5, alpha=c["alpha"], bias=bias)
    ref, S = oracle_nv(c["A"], c["SA"], c["B"], c["SB"], C=si.codes(C), c_fmt="bf16", beta=0.5, alpha=c["alpha"],
                       bias=si.codes(bias))
    assert ratio(D, ref, S, scale=c["alpha"]) <= 1.0


def test_nvfp4_8192_sampled(tcm):
    c = si.nvfp4_case()
    D = run_nv(tcm, c["A"], c["SA"], c["B"], c["SB"], alpha=c["alpha"])
    rows, cols = sample_indices(8192, 8192)
    ref, S = oracle_nv(c["A"], c["SA"], c["B"], c["SB"], alpha=c["alpha"], rows=rows, cols=cols)
    assert ratio(D, ref, S, scale=c["alpha"], rows=rows, cols=cols) <= 1.0
    assert not torch.isnan(D).any()
