"""GPU parity of the block-scaled (MXFP8) GEMM against the oracle's block-scaled reference."""
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


def run_mx(tcm, A, SA, B, SB, out=torch.bfloat16, C=None, beta=0.0, alpha=1.0, bias=None):
    """Row-major scales are packed on the device by the library, then the GEMM runs."""
    d = dev()
    M, K = A.shape
    N = B.shape[0]
    D = torch.full((M, N), float("nan"), dtype=out, device=d)
    pa = tcm.tcm_mx_pack_scales(SA.to(d), K)
    pb = tcm.tcm_mx_pack_scales(SB.to(d), K)
    tcm.tcm_gemm_mx(A.to(d), pa, B.to(d), pb, D, C=None if C is None else C.to(d), alpha=alpha,
                    beta=beta, bias=None if bias is None else bias.to(d))
    code, site = tcm.tcm_get_device_status()
    assert code == 0, (code, site)
    return D.cpu()


def oracle_mx(A, SA, B, SB, fa, fb, **kw):
    return oracle.gemm_mx(si.codes(A), SA.numpy(), si.codes(B), SB.numpy(), fa, fb, **kw)


@pytest.mark.parametrize("rows,K", [(1, 32), (127, 96), (128, 128), (130, 160), (300, 1024), (8192, 8192)])
def test_mx_pack_scales_bit_exact(tcm, rows, K):
    g = si.generator(rows + K)
    SC = torch.randint(0, 255, (rows, K // 32), generator=g).to(torch.uint8)
    got = tcm.tcm_mx_pack_scales(SC.to(dev()), K).cpu().numpy()
    assert np.array_equal(got, oracle.mx_pack_scales(SC.numpy(), K))


# (cta_group, tile_n): 0 = the library's choice; (2, 256) = the CTA-pair 256 x 256 tile
VARIANTS = [(0, 0), (1, 128), (1, 256), (2, 256)]


@pytest.mark.parametrize("cg,bn", VARIANTS)
@pytest.mark.parametrize("M,N,K", [(128, 128, 128), (256, 512, 1024), (300, 520, 416), (1000, 136, 96)])
def test_mx_integer_exact(tcm, cg, bn, M, N, K):
    tcm.tcm_set_config_override(cg, bn)
    g = si.generator(M + N + K)
    A = si.integers((M, K), g, dtype="e4m3")
    B = si.integers((N, K), g, dtype="e4m3")
    SA = torch.randint(126, 129, (M, K // 32), generator=g).to(torch.uint8)
    SB = torch.randint(126, 129, (N, K // 32), generator=g).to(torch.uint8)
    D = run_mx(tcm, A, SA, B, SB, out=torch.float32)
    ref, _ = oracle_mx(A, SA, B, SB, "e4m3", "e4m3")
    assert np.array_equal(D.double().numpy(), ref)


@pytest.mark.parametrize("fa,fb", [("e4m3", "e4m3"), ("e4m3", "e5m2"), ("e5m2", "e4m3")])
@pytest.mark.parametrize("cg,bn", VARIANTS[1:])
def test_mx_normal_data_bound(tcm, fa, fb, cg, bn):
    tcm.tcm_set_config_override(cg, bn)
    c = si.mx_case(640, 768, 1024, a_fmt=fa, b_fmt=fb, seed=7)
    g = si.generator(8)
    C = si.normal((640, 768), g)
    bias = si.normal((768,), g)
    D = run_mx(tcm, c["A"], c["SA"], c["B"], c["SB"], C=C, beta=0.5, alpha=2.0, bias=bias)
    ref, S = oracle_mx(c["A"], c["SA"], c["B"], c["SB"], fa, fb, C=si.codes(C), c_fmt="bf16", beta=0.5,
                       alpha=2.0, bias=si.codes(bias))
    assert ratio(D, ref, S, scale=2.0) <= 1.0


@pytest.mark.parametrize("cg,bn", VARIANTS)
@pytest.mark.parametrize("out,fmt", [(torch.bfloat16, "bf16"), (torch.float16, "f16")])
def test_mx_bias_without_c_bound(tcm, cg, bn, out, fmt):
    """16-bit output, beta = 0, bias: full-width tiles take the drain-and-convert epilogue,
    the ragged last tile (N = 520) the general one."""
    tcm.tcm_set_config_override(cg, bn)
    c = si.mx_case(300, 520, 416, seed=11)
    bias = si.normal((520,), si.generator(12), dtype=fmt)
    D = run_mx(tcm, c["A"], c["SA"], c["B"], c["SB"], out=out, alpha=0.75, bias=bias)
    ref, S = oracle_mx(c["A"], c["SA"], c["B"], c["SB"], "e4m3", "e4m3", alpha=0.75, bias=si.codes(bias),
                       bias_fmt=fmt)
    assert ratio(D, ref, S, scale=0.75) <= 1.0


def test_mx_wide_scale_range_bound(tcm):
    """Block scales spread over many binades (2^-20 .. 2^20) still meet the bound."""
    M, N, K = 256, 256, 512
    g = si.generator(9)
    A = si.normal((M, K), g, dtype="e4m3")
    B = si.normal((N, K), g, dtype="e4m3")
    SA = torch.randint(107, 148, (M, K // 32), generator=g).to(torch.uint8)
    SB = torch.randint(107, 148, (N, K // 32), generator=g).to(torch.uint8)
    D = run_mx(tcm, A, SA, B, SB, out=torch.float32)
    ref, S = oracle_mx(A, SA, B, SB, "e4m3", "e4m3")
    assert ratio(D, ref, S) <= 1.0


@pytest.mark.parametrize("cg", [0, 1])
def test_mx_8192_sampled(tcm, cg):
    tcm.tcm_set_config_override(cg, 0)
    c = si.mx_case()
    D = run_mx(tcm, c["A"], c["SA"], c["B"], c["SB"])
    rows, cols = sample_indices(8192, 8192)
    ref, S = oracle_mx(c["A"], c["SA"], c["B"], c["SB"], "e4m3", "e4m3", rows=rows, cols=cols)
    assert ratio(D, ref, S, rows=rows, cols=cols) <= 1.0
    assert not torch.isnan(D).any()
