"""Failure path of the block-scaled and sparse kernels (MXFP8, NVFP4, 2:4 sparse with
hardware-ordered or canonical metadata): a stage whose loads are never issued makes its waits run out,
the status names a pipeline wait, the kernel winds down, and the next launch computes the
same result as an unstarved one."""
import pytest
import torch

import synth_inputs as si
from parity import dev

pytestmark = pytest.mark.gpu

# 2: the MMA issuer or a side-data thread waiting for data; 4: the epilogue waiting for the
# tile; 6: the MMA issuer waiting for the stage's scales or metadata in tensor memory;
# 7: a metadata writer waiting for a stage's previous MMAs (canonical sparse path, K % 128 != 0)
SITES = (2, 4, 6, 7)


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
    t.tcm_set_timeout_ns(0)
    t.tcm_clear_device_status()


def starve_then_recover(tcm, launch, D):
    """Reference launch, starved launch (timeout reported), recovery launch equal to the reference."""
    launch()
    assert tcm.tcm_get_device_status() == (0, 0)
    ref = D.clone()
    tcm.tcm_set_timeout_ns(50_000_000)
    try:
        tcm.tcm_debug_fail_next_launch(1)
        launch()
        code, site = tcm.tcm_get_device_status()
        assert code == 5 and site in SITES, (code, site)
    finally:
        tcm.tcm_set_timeout_ns(0)
        tcm.tcm_clear_device_status()
    D.fill_(float("nan"))
    launch()
    assert tcm.tcm_get_device_status() == (0, 0)
    assert torch.equal(D, ref)


@pytest.mark.parametrize("cg,bn", [(2, 256), (1, 256), (1, 128)])
def test_mxfp8_starved_stage(tcm, cg, bn):
    tcm.tcm_set_config_override(cg, bn, 0, 0, 0)
    d = dev()
    g = si.generator(90 + cg + bn)
    M, N, K = 512, 512, 512
    A = si.integers((M, K), g, -8, 8, dtype="e4m3").to(d)
    B = si.integers((N, K), g, -8, 8, dtype="e4m3").to(d)
    codes = torch.full((M, K // 32), 127, dtype=torch.uint8)  # 2^0
    SA = tcm.tcm_mx_pack_scales(codes.to(d), K)
    SB = tcm.tcm_mx_pack_scales(codes[:N].to(d), K)
    D = torch.empty((M, N), dtype=torch.float32, device=d)
    starve_then_recover(tcm, lambda: tcm.tcm_gemm_mx(A, SA, B, SB, D), D)


@pytest.mark.parametrize("cg,bn", [(2, 256), (1, 256)])
def test_nvfp4_starved_stage(tcm, cg, bn):
    tcm.tcm_set_config_override(cg, bn, 0, 0, 0)
    d = dev()
    c = si.nvfp4_case(512, 512, 1024, seed=91)
    A, B = c["A"].to(d), c["B"].to(d)
    SA = tcm.tcm_nvfp4_pack_scales(c["SA"].to(d), 1024)
    SB = tcm.tcm_nvfp4_pack_scales(c["SB"].to(d), 1024)
    D = torch.empty((512, 512), dtype=torch.bfloat16, device=d)
    starve_then_recover(tcm, lambda: tcm.tcm_gemm_nvfp4(A, SA, B, SB, D, alpha=c["alpha"]), D)


@pytest.mark.parametrize("cg,bn", [(2, 256), (1, 128)])
def test_sparse_tc_starved_stage(tcm, cg, bn):
    tcm.tcm_set_config_override(cg, bn, 0, 0, 0)
    d = dev()
    s = si.sparse_case(512, 512, 512, seed=92)
    Ac, meta = tcm.tcm_sp_compress(s["A_logical"].to(d))
    meta_tc = tcm.tcm_sp_meta_pack(meta, 512)
    B = s["B"].to(d)
    D = torch.empty((512, 512), dtype=torch.bfloat16, device=d)
    starve_then_recover(tcm, lambda: tcm.tcm_gemm_sp_tc(Ac, meta_tc, B, D), D)


@pytest.mark.parametrize("K", [512, 160])  # metadata staged by TMA; loaded by the writer warps
@pytest.mark.parametrize("cg,bn", [(2, 256), (1, 128)])
def test_sparse_canonical_starved_stage(tcm, cg, bn, K):
    tcm.tcm_set_config_override(cg, bn, 0, 0, 0)
    d = dev()
    s = si.sparse_case(512, 512, K, seed=93)
    Ac, meta = tcm.tcm_sp_compress(s["A_logical"].to(d))
    B = s["B"].to(d)
    D = torch.empty((512, 512), dtype=torch.bfloat16, device=d)
    starve_then_recover(tcm, lambda: tcm.tcm_gemm_sp(Ac, meta, B, D), D)


@pytest.mark.parametrize("cg,bn", [(2, 256), (1, 128)])
def test_mxfp4_starved_stage(tcm, cg, bn):
    tcm.tcm_set_config_override(cg, bn, 0, 0, 0)
    d = dev()
    c = si.mxfp4_case(512, 512, 1024, seed=94)
    A, B = c["A"].to(d), c["B"].to(d)
    SA = tcm.tcm_mx_pack_scales(c["SA"].to(d), 1024)
    SB = tcm.tcm_mx_pack_scales(c["SB"].to(d), 1024)
    D = torch.empty((512, 512), dtype=torch.bfloat16, device=d)
    starve_then_recover(tcm, lambda: tcm.tcm_gemm_mx(A, SA, B, SB, D, fmt="e2m1"), D)
