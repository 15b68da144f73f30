"""GPU parity of the 2:4 path: compress / decompress bit-exact against the oracle,
and the tcgen05.mma.sp GEMM against the oracle's dense GEMM of the decompressed A.
"""
import json
import os

import numpy as np
import pytest
import torch

import oracle
import synth_inputs as si
from parity import dev, ratio, sample_indices

pytestmark = pytest.mark.gpu

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


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


def gpu_compress(tcm, A):
    Ac, meta = tcm.tcm_sp_compress(A.to(dev()))
    torch.cuda.synchronize()
    return Ac.cpu(), meta.cpu()


def meta_codes(meta):
    return meta.numpy().view(np.uint32)


@pytest.mark.parametrize("fmt", ["bf16", "f16"])
@pytest.mark.parametrize("M,K,kind", [(64, 256, "normal"), (333, 96, "int"), (8, 2048, "int"), (1, 32, "normal")])
def test_compress_bit_exact(tcm, fmt, M, K, kind):
    g = si.generator(M * K)
    A = si.normal((M, K), g, dtype=fmt) if kind == "normal" else si.integers((M, K), g, lo=-2, hi=2, dtype=fmt)
    Ac, meta = gpu_compress(tcm, A)
    rAc, rmeta = oracle.sp_compress(si.codes(A), fmt)
    assert np.array_equal(si.codes(Ac), rAc)
    assert np.array_equal(meta_codes(meta), rmeta)
    back = tcm.tcm_sp_decompress(Ac.to(dev()), meta.to(dev()))
    assert np.array_equal(si.codes(back.cpu()), oracle.sp_decompress(rAc, rmeta, fmt))


def test_compress_worked_example_from_page(tcm):
    spec = json.load(open(os.path.join(GOLDEN, "sp24_worked_example.json")))
    for case in spec["cases"]:
        A = torch.tensor([case["logical"] * 8], dtype=torch.bfloat16)
        Ac, meta = gpu_compress(tcm, A)
        assert Ac[0, :2].float().tolist() == case["values"]
        i0, i1 = case["positions"]
        assert int(meta_codes(meta)[0, 0]) == sum((i0 | (i1 << 2)) << (4 * g) for g in range(8))


def test_compress_with_pitch(tcm):
    M, K, lda = 40, 64, 96
    g = si.generator(3)
    full = si.normal((M, lda), g)
    A = full.to(dev())[:, :K]
    Ac, meta = tcm.tcm_sp_compress(A)
    rAc, rmeta = oracle.sp_compress(si.codes(full[:, :K].contiguous()), "bf16")
    assert np.array_equal(si.codes(Ac.cpu()), rAc) and np.array_equal(meta_codes(meta.cpu()), rmeta)


def run_sparse(tcm, A_logical, B, out_dtype, C=None, alpha=1.0, beta=0.0, tc=False):
    """Compress on the GPU, then tcm_gemm_sp (canonical metadata) or, with tc, tcm_sp_meta_pack +
    tcm_gemm_sp_tc (hardware-ordered metadata copied into tensor memory by tcgen05.cp)."""
    d = dev()
    Ac, meta = tcm.tcm_sp_compress(A_logical.to(d))
    D = torch.full((A_logical.shape[0], B.shape[0]), float("nan"), dtype=out_dtype, device=d)
    Cd = None if C is None else C.to(d)
    if tc:
        meta_tc = tcm.tcm_sp_meta_pack(meta, A_logical.shape[1])
        tcm.tcm_gemm_sp_tc(Ac, meta_tc, B.to(d), D, C=Cd, alpha=alpha, beta=beta)
    else:
        tcm.tcm_gemm_sp(Ac, meta, B.to(d), D, C=Cd, alpha=alpha, beta=beta)
    code, site = tcm.tcm_get_device_status()
    assert code == 0, (code, site)
    return D.cpu(), Ac.cpu(), meta.cpu()


def oracle_sparse(A_logical, B, fmt, C=None, alpha=1.0, beta=0.0, rows=None, cols=None):
    Ac, meta = oracle.sp_compress(si.codes(A_logical), fmt)
    Ap = oracle.sp_decompress(Ac, meta, fmt)
    return oracle.gemm(Ap, si.codes(B), fmt, fmt, C=None if C is None else si.codes(C),
                       c_fmt="f32" if C is None else {torch.float32: "f32", torch.bfloat16: "bf16",
                                                       torch.float16: "f16"}[C.dtype],
                       alpha=alpha, beta=beta, rows=rows, cols=cols)


@pytest.mark.parametrize("tc", [False, True])
@pytest.mark.parametrize("cg,bn", [(0, 0), (1, 128), (2, 256), (2, 128)])
@pytest.mark.parametrize("M,N,K", [(128, 128, 32), (256, 224, 128), (300, 520, 160), (512, 672, 1024),
                                   (1000, 448, 2048)])
def test_sparse_gemm_integer_exact(tcm, cg, bn, M, N, K, tc):
    tcm.tcm_set_config_override(cg, bn, 0, 2)
    g = si.generator(M + N + K)
    A = si.integers((M, K), g)
    B = si.integers((N, K), g)
    D, _, _ = run_sparse(tcm, A, B, torch.float32, tc=tc)
    ref, _ = oracle_sparse(A, B, "bf16")
    assert np.array_equal(D.double().numpy(), ref)


@pytest.mark.parametrize("tc", [False, True])
@pytest.mark.parametrize("fmt,out", [("bf16", torch.bfloat16), ("f16", torch.float32)])
def test_sparse_gemm_bound_with_beta(tcm, fmt, out, tc):
    M, N, K = 640, 800, 1536
    g = si.generator(11)
    A = si.normal((M, K), g, dtype=fmt)
    B = si.normal((N, K), g, dtype=fmt)
    C = si.normal((M, N), g, dtype={torch.bfloat16: "bf16", torch.float32: "f32"}[out])
    D, _, _ = run_sparse(tcm, A, B, out, C=C, alpha=0.75, beta=0.5, tc=tc)
    ref, S = oracle_sparse(A, B, fmt, C=C, alpha=0.75, beta=0.5)
    assert ratio(D, ref, S, scale=0.75) <= 1.0


def test_sparse_matches_dense_on_decompressed(tcm):
    """The sparse GEMM and the dense GEMM of the decompressed A agree within the bound."""
    M, N, K = 512, 448, 1024
    g = si.generator(12)
    A = si.normal((M, K), g)
    B = si.normal((N, K), g)
    d = dev()
    Ds, Ac, meta = run_sparse(tcm, A, B, torch.float32)
    Ap = tcm.tcm_sp_decompress(Ac.to(d), meta.to(d))
    Dd = torch.empty((M, N), dtype=torch.float32, device=d)
    tcm.tcm_gemm_ex(Ap, B.to(d), Dd)
    ref, S = oracle_sparse(A, B, "bf16")
    assert ratio(Ds, ref, S) <= 1.0 and ratio(Dd.cpu(), ref, S) <= 1.0
    diff = (Ds - Dd.cpu()).abs().max().item()
    assert diff <= 2e-5 * float(np.max(S))


@pytest.mark.parametrize("tc", [False, True])
def test_sparse_8192_sampled(tcm, tc):
    case = si.sparse_case()
    D, _, _ = run_sparse(tcm, case["A_logical"], case["B"], torch.bfloat16, tc=tc)
    rows, cols = sample_indices(8192, 8192)
    ref, S = oracle_sparse(case["A_logical"], case["B"], "bf16", rows=rows, cols=cols)
    assert ratio(D, ref, S, rows=rows, cols=cols) <= 1.0
    assert not torch.isnan(D).any()


@pytest.mark.parametrize("M,K", [(1, 32), (130, 96), (300, 512), (8192, 8192)])
def test_meta_pack_bit_exact(tcm, M, K):
    g = si.generator(M + K)
    meta = torch.randint(-2 ** 31, 2 ** 31 - 1, (M, K // 32), generator=g, dtype=torch.int64).to(torch.int32)
    got = tcm.tcm_sp_meta_pack(meta.to(dev()), K).cpu().numpy()
    assert np.array_equal(got, oracle.sp_meta_pack(meta.numpy().view(np.uint32), K))


@pytest.mark.parametrize("M,N,K", [(1024, 768, 2048), (520, 384, 1184)])
def test_sparse_tc_identical_to_canonical_path(tcm, M, N, K):
    """Same MMAs in the same order: the two metadata paths give bit-identical D, with the
    canonical words staged by TMA (K % 128 == 0) and loaded by the writer warps (otherwise)."""
    case = si.sparse_case(M, N, K, seed=13)
    D1, _, _ = run_sparse(tcm, case["A_logical"], case["B"], torch.float32, tc=False)
    D2, _, _ = run_sparse(tcm, case["A_logical"], case["B"], torch.float32, tc=True)
    assert torch.equal(D1, D2)
