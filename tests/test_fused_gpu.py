"""GPU parity of the fused epilogue (tcm_gemm_fused): activation, FP8 output, amax.

Expected values come from the oracle: ``oracle.gemm`` for the scaled, biased
sum and ``oracle.fused_reference`` for the activation, the FP8 target
(y / d_scale, saturated) and the propagated bound.
"""
import numpy as np
import pytest
import torch

import oracle
import synth_inputs as si
from parity import FMT_OF, dev, oracle_ref, padded, sample_indices

pytestmark = pytest.mark.gpu

OUT = {"bf16": torch.bfloat16, "f16": torch.float16, "f32": torch.float32, "e4m3": torch.float8_e4m3fn,
       "e5m2": torch.float8_e5m2}


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


def run_fused(tcm, A, B, out, *, act=None, d_scale=None, C=None, beta=0.0, alpha=1.0, sa=None, sb=None, bias=None):
    """Run tcm_gemm_fused on CPU tensors moved to the GPU; returns (D on the CPU, amax)."""
    d = dev()
    M, N = A.shape[0], B.shape[0]
    D = padded(torch.zeros((M, N), dtype=OUT[out]), d)
    amax = torch.full((1,), -1.0, dtype=torch.float32, device=d)  # the call must reset it
    one = lambda v: None if v is None else torch.tensor([v], dtype=torch.float32, device=d)
    tcm.tcm_gemm_fused(padded(A, d), padded(B, d), D, C=None if C is None else padded(C, d), alpha=alpha, beta=beta,
                       a_scale=one(sa), b_scale=one(sb), bias=None if bias is None else bias.to(d), act=act,
                       d_scale=one(d_scale), amax=amax)
    code, site = tcm.tcm_get_device_status()
    assert code == 0, (code, site)
    return D.cpu(), float(amax.item())


def check(D, out, target, bound, rows=None, cols=None):
    d = oracle.decode(si.codes(D), out)
    if rows is not None:
        d = d[rows, cols]
    e = np.abs(d - target) / bound
    assert not np.isnan(e).any()
    assert float(e.max()) <= 1.0, float(e.max())


def check_amax(amax, y, e_y):
    lo = float(np.max(np.abs(y) - e_y))
    hi = float(np.max(np.abs(y) + e_y))
    assert lo <= amax <= hi, (lo, amax, hi)


def pm1_inputs(M, N, K, nnz, seed, fmt):
    """+-1 in the first `nnz` K positions, zeros elsewhere: every sum is an integer in [-nnz, nnz]."""
    g = si.generator(seed)
    A = torch.zeros((M, K))
    B = torch.zeros((N, K))
    A[:, :nnz] = torch.randint(0, 2, (M, nnz), generator=g).float() * 2 - 1
    B[:, :nnz] = torch.randint(0, 2, (N, nnz), generator=g).float() * 2 - 1
    return A.to(si.TORCH_DTYPE[fmt]), B.to(si.TORCH_DTYPE[fmt])


@pytest.mark.parametrize("out,nnz", [("e4m3", 16), ("e5m2", 8)])
@pytest.mark.parametrize("in_fmt", ["bf16", "e4m3"])
@pytest.mark.parametrize("act", [None, "relu"])
@pytest.mark.parametrize("d_scale", [1.0, 2.0])
@pytest.mark.parametrize("M,N,K", [(256, 512, 128), (300, 520, 256)])
def test_fp8_output_integer_exact(tcm, out, nnz, in_fmt, act, d_scale, M, N, K):
    """Integer sums up to nnz (and their halves) are exact in the FP8 output: stored values and amax exact."""
    A, B = pm1_inputs(M, N, K, nnz, M + N + nnz, in_fmt)
    D, amax = run_fused(tcm, A, B, out, act=act, d_scale=d_scale, sa=1.0 if in_fmt != "bf16" else None,
                        sb=1.0 if in_fmt != "bf16" else None)
    ref, _ = oracle_ref(A, B)
    y = oracle.activate(ref, act)
    assert np.array_equal(oracle.decode(si.codes(D), out), y / d_scale)
    assert amax == float(np.abs(y).max())


@pytest.mark.parametrize("act", [None, "relu", "gelu"])
@pytest.mark.parametrize("out", ["bf16", "f32", "e4m3", "e5m2"])
def test_fused_fp8_inputs_bound(tcm, act, out):
    c = si.fp8_case(300, 520, 416, seed=13)
    bias = c["bias"] if out in ("bf16", "e4m3", "e5m2") else c["bias"].to(torch.float32)
    ref, S = oracle_ref(c["A"], c["B"], sa=c["sa"], sb=c["sb"], bias=bias, alpha=1.5)
    y_max = float(np.abs(oracle.activate(ref, act)).max())
    d_scale = y_max / 300.0 if out in ("e4m3", "e5m2") else None  # most of the FP8 range used
    D, amax = run_fused(tcm, c["A"], c["B"], out, act=act, d_scale=d_scale, sa=c["sa"], sb=c["sb"], bias=bias,
                        alpha=1.5)
    target, bound, y, e_y = oracle.fused_reference(ref, S, act, out, scale=1.5 * c["sa"] * c["sb"],
                                                   d_scale=d_scale or 1.0)
    check(D, out, target, bound)
    check_amax(amax, y, e_y)


@pytest.mark.parametrize("act", ["relu", "gelu"])
def test_fused_bf16_inputs_with_c(tcm, act):
    """beta * C enters before the activation (16-bit output)."""
    case = si.llm_case(264, 392, 520, seed=21)
    g = si.generator(22)
    C = si.normal((264, 392), g)
    bias = si.normal((392,), g)
    D, amax = run_fused(tcm, case["A"], case["B"], "bf16", act=act, C=C, beta=-0.5, bias=bias)
    ref, S = oracle_ref(case["A"], case["B"], C=C, beta=-0.5, bias=bias)
    target, bound, y, e_y = oracle.fused_reference(ref, S, act, "bf16")
    check(D, "bf16", target, bound)
    check_amax(amax, y, e_y)


@pytest.mark.parametrize("cg,bn,ks", [(1, 256, 0), (1, 128, 0), (1, 64, 0), (1, 32, 0), (2, 256, 0)])
def test_fused_each_variant(tcm, cg, bn, ks):
    tcm.tcm_set_config_override(cg, bn, 0, 0, ks)
    c = si.fp8_case(520, 640, 768, b_fmt="e5m2", seed=17)
    ref, S = oracle_ref(c["A"], c["B"], sa=c["sa"], sb=c["sb"], bias=c["bias"])
    d_scale = float(np.abs(oracle.activate(ref, "gelu")).max()) / 400.0
    D, amax = run_fused(tcm, c["A"], c["B"], "e4m3", act="gelu", d_scale=d_scale, sa=c["sa"], sb=c["sb"],
                        bias=c["bias"])
    target, bound, y, e_y = oracle.fused_reference(ref, S, "gelu", "e4m3", scale=c["sa"] * c["sb"], d_scale=d_scale)
    check(D, "e4m3", target, bound)
    check_amax(amax, y, e_y)


@pytest.mark.parametrize("ks", [0, 2, 4])
@pytest.mark.parametrize("M", [1, 16, 40])
def test_fused_skinny_swapped_and_k_split(tcm, ks, M):
    """Skinny M runs with A and B swapped (bias per kernel row), optionally K-split over a cluster."""
    tcm.tcm_set_config_override(0, 0, 0, 0, ks)
    c = si.fp8_case(M, 1024, 2048, seed=19)
    ref, S = oracle_ref(c["A"], c["B"], sa=c["sa"], sb=c["sb"], bias=c["bias"])
    d_scale = float(np.abs(oracle.activate(ref, "gelu")).max()) / 400.0
    D, amax = run_fused(tcm, c["A"], c["B"], "e4m3", act="gelu", d_scale=d_scale, sa=c["sa"], sb=c["sb"],
                        bias=c["bias"])
    target, bound, y, e_y = oracle.fused_reference(ref, S, "gelu", "e4m3", scale=c["sa"] * c["sb"], d_scale=d_scale)
    check(D, "e4m3", target, bound)
    check_amax(amax, y, e_y)


def test_fused_saturates_and_amax_sees_the_unsaturated_value(tcm):
    """d_scale small enough that many outputs exceed 448: they store +-448, amax keeps the true max |y|."""
    c = si.fp8_case(256, 256, 256, seed=23)
    ref, S = oracle_ref(c["A"], c["B"], sa=c["sa"], sb=c["sb"])
    d_scale = float(np.abs(ref).max()) / 2000.0
    D, amax = run_fused(tcm, c["A"], c["B"], "e4m3", d_scale=d_scale, sa=c["sa"], sb=c["sb"])
    target, bound, y, e_y = oracle.fused_reference(ref, S, None, "e4m3", scale=c["sa"] * c["sb"], d_scale=d_scale)
    assert (np.abs(target) == 448.0).sum() > 100
    check(D, "e4m3", target, bound)
    check_amax(amax, y, e_y)


def test_fused_8192_fp8_gelu_e4m3_sampled(tcm):
    """The fused workload at full size: E4M3 x E4M3 + scales + bias, GELU, E4M3 output, amax."""
    c = si.fp8_case()
    rows, cols = sample_indices(8192, 8192)
    ref, S = oracle_ref(c["A"], c["B"], sa=c["sa"], sb=c["sb"], bias=c["bias"], rows=rows, cols=cols)
    d_scale = 2.0  # the largest |y| (about 5.6 sigma of N(0, 8192) plus bias) stays below 448 * 2
    D, amax = run_fused(tcm, c["A"], c["B"], "e4m3", act="gelu", d_scale=d_scale, sa=c["sa"], sb=c["sb"],
                        bias=c["bias"])
    target, bound, y, e_y = oracle.fused_reference(ref, S, "gelu", "e4m3", scale=c["sa"] * c["sb"], d_scale=d_scale)
    check(D, "e4m3", target, bound, rows=rows, cols=cols)
    # amax covers every sampled output, and matches the largest stored output within one FP8 rounding
    assert amax >= float(np.max(np.abs(y) - e_y))
    stored = oracle.decode(si.codes(D), "e4m3")
    assert not np.isnan(stored).any()
    top = float(np.abs(stored).max()) * d_scale
    assert abs(top - min(amax, 448.0 * d_scale)) <= 2.0 ** -4 * top + 2.0 ** -9 * d_scale
