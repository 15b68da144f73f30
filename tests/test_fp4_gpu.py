"""GPU parity of FP4 (E2M1, packed two per byte) operands in kind::f8f6f4: FP4 x FP8, FP8 x FP4, FP4 x FP4."""
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


def fmt_of(t, fmt):
    return fmt if fmt is not None else {torch.float8_e4m3fn: "e4m3", torch.float8_e5m2: "e5m2"}[t.dtype]


def run(tcm, A, B, out=torch.float32, a_fmt=None, b_fmt=None, sa=None, sb=None, bias=None):
    d = dev()
    M, N = A.shape[0], B.shape[0]
    D = torch.full((M, N), float("nan"), dtype=out, device=d)
    one = lambda v: None if v is None else torch.tensor([v], dtype=torch.float32, device=d)
    tcm.tcm_gemm_ex(A.to(d), B.to(d), D, a_scale=one(sa), b_scale=one(sb), bias=None if bias is None else bias.to(d),
                    a_fmt=a_fmt, b_fmt=b_fmt)
    code, site = tcm.tcm_get_device_status()
    assert code == 0, (code, site)
    return D.cpu()


def fp4_random(rows, K, g):
    """Random packed E2M1 codes: every value 0, +-0.5 .. +-6."""
    return si.pack_fp4(torch.randint(0, 16, (rows, K), generator=g).to(torch.uint8))


def ref_of(A, B, a_fmt, b_fmt, **kw):
    return oracle.gemm(si.codes(A), si.codes(B), a_fmt, b_fmt, **kw)


ORDERS = [("e2m1", "e4m3"), ("e4m3", "e2m1"), ("e2m1", "e5m2"), ("e2m1", "e2m1")]


def operands(order, M, N, K, g):
    fa, fb = order
    A = fp4_random(M, K, g) if fa == "e2m1" else si.integers((M, K), g, -8, 8, dtype=fa)
    B = fp4_random(N, K, g) if fb == "e2m1" else si.integers((N, K), g, -8, 8, dtype=fb)
    return A, B


@pytest.mark.parametrize("order", ORDERS)
@pytest.mark.parametrize("M,N,K", [(128, 128, 128), (256, 512, 1024), (300, 520, 384), (1000, 136, 256)])
def test_fp4_integer_sums_exact(tcm, order, M, N, K):
    """Products of E2M1 values (multiples of 1/2 up to 6) and small integers sum exactly in fp32."""
    g = si.generator(M + N + K + len(order[1]))
    A, B = operands(order, M, N, K, g)
    fa, fb = order
    D = run(tcm, A, B, a_fmt="e2m1" if fa == "e2m1" else None, b_fmt="e2m1" if fb == "e2m1" else None)
    ref, _ = ref_of(A, B, fa, fb)
    assert np.array_equal(D.double().numpy(), ref)


@pytest.mark.parametrize("cg,bn,ks", [(1, 256, 0), (1, 128, 0), (1, 64, 0), (1, 32, 0), (2, 256, 0)])
@pytest.mark.parametrize("order", [("e4m3", "e2m1"), ("e2m1", "e4m3")])
def test_fp4_each_variant_exact(tcm, cg, bn, ks, order):
    tcm.tcm_set_config_override(cg, bn, 0, 0, ks)
    g = si.generator(cg * 1000 + bn)
    A, B = operands(order, 520, 640, 768, g)
    fa, fb = order
    D = run(tcm, A, B, a_fmt="e2m1" if fa == "e2m1" else None, b_fmt="e2m1" if fb == "e2m1" else None)
    ref, _ = ref_of(A, B, fa, fb)
    assert np.array_equal(D.double().numpy(), ref)


@pytest.mark.parametrize("K", [128, 384, 640])
@pytest.mark.parametrize("order", [("e4m3", "e2m1"), ("e2m1", "e2m1")])
def test_fp4_pair_tiles_with_a_half_filled_last_stage(tcm, order, K):
    """CTA-pair tiles of 8-bit kinds take two 128-value K atoms per stage: with K an odd number
    of atoms the last stage's second atom lies past K (zero-filled by TMA, still counted on
    the stage's barrier)."""
    tcm.tcm_set_config_override(2, 256, 0, 0, 0)
    g = si.generator(K + 7)
    A, B = operands(order, 512, 768, K, g)
    fa, fb = order
    D = run(tcm, A, B, a_fmt="e2m1" if fa == "e2m1" else None, b_fmt="e2m1" if fb == "e2m1" else None)
    ref, _ = ref_of(A, B, fa, fb)
    assert np.array_equal(D.double().numpy(), ref)


@pytest.mark.parametrize("ks", [0, 2, 4])
@pytest.mark.parametrize("M", [1, 16, 48])
def test_fp4_skinny_swapped_and_k_split_exact(tcm, ks, M):
    """Skinny M: the FP4 weight becomes the kernel's 128-row operand; optionally K-split."""
    tcm.tcm_set_config_override(0, 0, 0, 0, ks)
    g = si.generator(M + ks)
    A, B = operands(("e4m3", "e2m1"), M, 1024, 2048, g)
    D = run(tcm, A, B, b_fmt="e2m1")
    ref, _ = ref_of(A, B, "e4m3", "e2m1")
    assert np.array_equal(D.double().numpy(), ref)


def test_w4a8_normal_data_bound_with_scales_and_bias(tcm):
    c = si.w4a8_case(300, 520, 1024, seed=7)
    bias = si.normal((520,), si.generator(8))
    D = run(tcm, c["A"], c["B"], out=torch.bfloat16, b_fmt="e2m1", sa=c["sa"], sb=c["sb"], bias=bias)
    ref, S = ref_of(c["A"], c["B"], "e4m3", "e2m1", sa=c["sa"], sb=c["sb"], bias=si.codes(bias))
    assert ratio(D, ref, S, scale=c["sa"] * c["sb"]) <= 1.0


def test_w4a8_8192_sampled(tcm):
    c = si.w4a8_case()
    D = run(tcm, c["A"], c["B"], out=torch.bfloat16, b_fmt="e2m1", sa=c["sa"], sb=c["sb"])
    rows, cols = sample_indices(8192, 8192)
    ref, S = ref_of(c["A"], c["B"], "e4m3", "e2m1", sa=c["sa"], sb=c["sb"], rows=rows, cols=cols)
    assert ratio(D, ref, S, scale=c["sa"] * c["sb"], rows=rows, cols=cols) <= 1.0
    assert not torch.isnan(D).any()
