"""FP8 accumulation precision against K.

"NVIDIA MMA", section "Hopper：wgmma.mma_async" warns that FP8 MMAs there accumulate
with less than full fp32 precision; the pages say nothing about tcgen05.  The plain
reading is that the library's bound, 1e-5 * |scale| * sum_k |a b| plus one output
rounding, holds at every K.  This sweep measures max err / bound of E4M3 x E4M3,
E4M3 x E5M2 and E5M2 x E5M2 GEMMs with fp32 output (so that the output cast does not
hide the accumulation error) for K from 256 to 65536 and requires <= 1 at each K,
i.e. that the margin does not run out as the K loop grows.  The measured values are
printed (pytest -s) for the record.
"""
import numpy as np
import pytest
import torch

import oracle
import synth_inputs as si
from parity import dev

pytestmark = pytest.mark.gpu

KS = (256, 1024, 4096, 16384, 32768, 65536)


@pytest.fixture(scope="module", autouse=True)
def _build():
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(0)
    import tensor_core_matrix_gb300 as tcm
    tcm.tcm_clear_device_status()


@pytest.mark.parametrize("fa,fb", [("e4m3", "e4m3"), ("e4m3", "e5m2"), ("e5m2", "e5m2")])
def test_fp8_error_does_not_outgrow_bound_with_k(fa, fb):
    import tensor_core_matrix_gb300 as tcm
    d = dev()
    M, N = 128, 256
    rows = []
    for K in KS:
        g = si.generator(500 + K)
        A, sa = si.fp8_per_tensor(torch.randn((M, K), generator=g), fa)
        B, sb = si.fp8_per_tensor(torch.randn((N, K), generator=g), fb)
        D = torch.full((M, N), float("nan"), dtype=torch.float32, device=d)
        tcm.tcm_gemm_ex(A.to(d), B.to(d), D, a_scale=torch.tensor([sa], device=d), b_scale=torch.tensor([sb], device=d))
        code, site = tcm.tcm_get_device_status()
        assert code == 0, (code, site)
        ref, S = oracle.gemm(si.codes(A), si.codes(B), fa, fb, sa=sa, sb=sb)
        got = D.cpu().double().numpy()
        r = oracle.err_over_bound(si.codes(D.cpu()), "f32", ref, S, scale=sa * sb)
        rel = float(np.max(np.abs(got - ref) / (abs(sa * sb) * S)))  # error in units of sum |a b|
        rows.append((K, r, rel))
        assert r <= 1.0, f"{fa} x {fb}, K = {K}: err/bound {r}"
    print(f"\n{fa} x {fb}: " + "; ".join(f"K={K} err/bound {r:.3g} (|err|/sum|ab| {e:.2e})" for K, r, e in rows))
