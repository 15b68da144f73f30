"""GPU parity of the dense tcgen05 GEMM against the CPU oracle, through the C ABI.

Bars: integer-valued inputs (exact in fp32 as long as |partial sums| < 2^24)
must match bit for bit; everything else must satisfy
|D - ref| <= 1e-5 * |alpha sA sB| * sum_k |a b| + 2^-p |ref| + min_subnormal
element by element (oracle.bound).  D is pre-filled with NaN so an unwritten
output fails.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import synth_inputs as si
from parity import dev, oracle_ref, ratio, run_gemm_ex, sample_indices

pytestmark = pytest.mark.gpu

F8 = {"e4m3": torch.float8_e4m3fn, "e5m2": torch.float8_e5m2}


@pytest.fixture(scope="module", autouse=True)
def _build():
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(0)
    import tensor_core_matrix_gb300 as tcm
    tcm.tcm_clear_device_status()


# ------------------------------------------------------------------ exact cases

@pytest.mark.parametrize("M,N,K", [
    (128, 32, 16), (128, 64, 64), (128, 128, 64), (128, 256, 64), (256, 512, 256),
    (300, 520, 136), (1000, 260, 1024), (129, 257, 72),
])
@pytest.mark.parametrize("fmt", ["bf16", "f16"])
def test_integer_inputs_bit_exact(M, N, K, fmt):
    g = si.generator(100 + M + N + K)
    A = si.integers((M, K), g, dtype=fmt)
    B = si.integers((N, K), g, dtype=fmt)
    D = run_gemm_ex(A, B, torch.float32)
    ref, _ = oracle_ref(A, B)
    assert np.array_equal(D.double().numpy(), ref)


@pytest.mark.parametrize("fa,fb", [("e4m3", "e4m3"), ("e4m3", "e5m2"), ("e5m2", "e4m3"), ("e5m2", "e5m2")])
@pytest.mark.parametrize("M,N,K", [(128, 256, 128), (200, 136, 400)])
def test_fp8_integer_inputs_bit_exact(fa, fb, M, N, K):
    g = si.generator(7 + M)
    A = si.integers((M, K), g, dtype=fa)
    B = si.integers((N, K), g, dtype=fb)
    D = run_gemm_ex(A, B, torch.float32)
    ref, _ = oracle_ref(A, B)
    assert np.array_equal(D.double().numpy(), ref)


def test_identity_gives_b_transposed():
    K, N = 256, 384
    A = torch.eye(K, dtype=torch.bfloat16)
    B = si.normal((N, K), si.generator(5))
    D = run_gemm_ex(A, B, torch.float32)
    assert torch.equal(D, B.float().t())


def test_permutation_permutes_rows():
    K, N = 192, 160
    perm = torch.randperm(K, generator=si.generator(6))
    P = torch.zeros((K, K), dtype=torch.bfloat16)
    P[torch.arange(K), perm] = 1.0
    B = si.normal((N, K), si.generator(7))
    D = run_gemm_ex(P, B, torch.float32)
    assert torch.equal(D, B.float().t()[perm])


def test_rank1_closed_form():
    M, N, K = 256, 256, 512
    u = 2.0 ** torch.randint(-3, 3, (M,), generator=si.generator(8)).float()
    v = -(2.0 ** torch.randint(-3, 3, (N,), generator=si.generator(9)).float())
    A = u[:, None].expand(M, K).to(torch.bfloat16).contiguous()
    B = v[:, None].expand(N, K).to(torch.bfloat16).contiguous()
    D = run_gemm_ex(A, B, torch.float32, alpha=0.5)
    assert torch.equal(D, 0.5 * K * torch.outer(u, v))


# ------------------------------------------------------------------ every kernel variant

@pytest.fixture
def override():
    import tensor_core_matrix_gb300 as tcm
    yield tcm
    tcm.tcm_set_config_override(0, 0, 0, 0, 0)


@pytest.mark.parametrize("cg,bn,stages", [(1, 256, 0), (1, 128, 0), (1, 64, 0), (1, 32, 0), (2, 256, 0)])
@pytest.mark.parametrize("M,N,K", [(256, 256, 64), (512, 768, 320), (300, 520, 136), (1000, 1030, 1024)])
def test_each_variant_integer_exact(override, cg, bn, stages, M, N, K):
    override.tcm_set_config_override(cg, bn, stages, 3)
    g = si.generator(M + N + K + cg + bn)
    A = si.integers((M, K), g)
    B = si.integers((N, K), g)
    D = run_gemm_ex(A, B, torch.float32)
    ref, _ = oracle_ref(A, B)
    assert np.array_equal(D.double().numpy(), ref)


@pytest.mark.parametrize("cg,bn,stages", [(1, 256, 0), (2, 256, 0), (1, 128, 0), (1, 64, 0), (1, 32, 0)])
@pytest.mark.parametrize("fb", ["e4m3", "e5m2"])
def test_each_variant_fp8_bound(override, cg, bn, stages, fb):
    override.tcm_set_config_override(cg, bn, stages)
    case = si.fp8_case(640, 768, 1024, b_fmt=fb, seed=3)
    D = run_gemm_ex(case["A"], case["B"], torch.bfloat16, sa=case["sa"], sb=case["sb"], bias=case["bias"])
    ref, S = oracle_ref(case["A"], case["B"], sa=case["sa"], sb=case["sb"], bias=case["bias"])
    assert ratio(D, ref, S, scale=case["sa"] * case["sb"]) <= 1.0


@pytest.mark.parametrize("K", [128, 384, 1152])
def test_fp8_pair_tiles_with_a_half_filled_last_stage(override, K):
    """E4M3 CTA-pair tiles take two 128-value K atoms per stage: with K an odd number of atoms
    the last stage's second atom lies past K (zero-filled by TMA, counted on the barrier)."""
    override.tcm_set_config_override(2, 256, 0, 0, 0)
    g = si.generator(K + 3)
    A = si.integers((512, K), g, -8, 8, dtype="e4m3")
    B = si.integers((768, K), g, -8, 8, dtype="e4m3")
    D = run_gemm_ex(A, B, torch.float32)
    ref, _ = oracle_ref(A, B)
    assert np.array_equal(D.double().numpy(), ref)


@pytest.mark.parametrize("split", [1, 2])
@pytest.mark.parametrize("M,N,K", [(512, 768, 320), (300, 520, 136), (4096, 2560, 256), (4000, 2600, 200),
                                   (1024, 1024, 1000)])
def test_pair_tail_k_split_integer_exact(override, split, M, N, K):
    """tcm_gemm_ex_ws: the tiles of the last, partly filled round of CTA pairs split into two K
    halves (split 2: whenever each pair gets at most one half) or not (1); 4096 x 2560 has two full
    rounds of 76 pairs plus 8 tiles.  Integer sums are exact whatever the order."""
    override.tcm_set_config_override(2, 256, 0, 0, 0, split)
    g = si.generator(M + 2 * N + K + split)
    A = si.integers((M, K), g)
    B = si.integers((N, K), g)
    D = run_gemm_ex(A, B, torch.float32, workspace=True)
    ref, _ = oracle_ref(A, B)
    assert np.array_equal(D.double().numpy(), ref)


@pytest.mark.parametrize("in_fmt", ["bf16", "e4m3"])
def test_pair_tail_k_split_with_epilogue(override, in_fmt):
    """Split tail tiles with the whole epilogue (alpha, scales, beta * C, bias): within the bound of the
    oracle on sampled outputs of every tile, and within it of the unsplit launch (3 rounds + 28 tiles)."""
    M = N = 4096
    K = 512
    g = si.generator(31)
    if in_fmt == "e4m3":
        c = si.fp8_case(M, N, K, seed=32)
        A, B, kw = c["A"], c["B"], dict(sa=c["sa"], sb=c["sb"], bias=c["bias"])
    else:
        A, B = si.normal((M, K), g), si.normal((N, K), g)
        kw = dict(bias=si.normal((N,), g))
    C = si.normal((M, N), g)
    override.tcm_set_config_override(2, 256, 0, 0, 0, 2)  # 256-column pair tiles, 28 tail tiles split
    out = [run_gemm_ex(A, B, torch.bfloat16, C=C, alpha=0.5, beta=0.25, workspace=ws, **kw) for ws in (False, True)]
    rows, cols = sample_indices(M, N, per_tile=2)
    ref, S = oracle_ref(A, B, C=C, alpha=0.5, beta=0.25, rows=rows, cols=cols, **kw)
    scale = 0.5 * kw.get("sa", 1.0) * kw.get("sb", 1.0)
    for D in out:
        assert ratio(D, ref, S, scale=scale, rows=rows, cols=cols) <= 1.0


def test_workspace_size_and_rejection(override):
    """The workspace query matches the plan (36 split tiles at 8192^3 on 76 pairs: flags plus one
    128 x 256 fp32 slot per CTA per helper part); a smaller workspace is rejected before launch."""
    import tensor_core_matrix_gb300 as tcm
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    pairs = sms // 2
    rem = 1024 % pairs
    n = tcm.tcm_gemm_workspace_bytes(8192, 8192, 8192, torch.bfloat16, torch.bfloat16)
    if rem == 0:
        assert n == 0
        return
    assert 2 * rem <= pairs  # 36 leftover tiles on 76 pairs: split in two K halves
    assert n == -(-(rem * 2 * 4) // 256) * 256 + rem * 2 * 128 * 256 * 4
    assert tcm.tcm_gemm_workspace_bytes(16, 28672, 8192, torch.bfloat16, torch.bfloat16) == 0  # no pair tiles
    d = dev()
    A = torch.zeros((8192, 8192), dtype=torch.bfloat16, device=d)
    D = torch.empty((8192, 8192), dtype=torch.bfloat16, device=d)
    small = torch.empty(n - 256, dtype=torch.uint8, device=d)
    with pytest.raises(tcm.TcmError, match="INVALID_ARG"):
        tcm.tcm_gemm_ex(A, A, D, workspace=small)


def test_tail_k_split_wait_times_out_and_context_stays_usable(override):
    """Helper parts that never announce their partial sums: each owner's bounded wait runs out
    (site 10), the kernel returns, and the next launch is correct."""
    tcm = override
    d = dev()
    M, N, K = 4096, 2560, 512
    g = si.generator(78)
    A = si.integers((M, K), g)
    B = si.integers((N, K), g)
    Ad, Bd = A.to(d), B.to(d)
    tcm.tcm_set_config_override(2, 256, 0, 0, 0, 2)  # 256-column pair tiles, 8 tail tiles split
    ws = torch.empty(tcm.tcm_gemm_workspace_bytes(M, N, K, torch.bfloat16), dtype=torch.uint8, device=d)
    assert ws.numel() > 0
    D = torch.zeros((M, N), dtype=torch.float32, device=d)
    tcm.tcm_clear_device_status()
    tcm.tcm_set_timeout_ns(50_000_000)
    try:
        tcm.tcm_debug_fail_next_launch(2)
        tcm.tcm_gemm_ex(Ad, Bd, D, workspace=ws)
        code, site = tcm.tcm_get_device_status()
        assert (code, site) == (5, 10)
    finally:
        tcm.tcm_set_timeout_ns(0)
        tcm.tcm_clear_device_status()
    D.fill_(float("nan"))
    tcm.tcm_gemm_ex(Ad, Bd, D, workspace=ws)
    assert tcm.tcm_get_device_status() == (0, 0)
    ref, _ = oracle_ref(A, B)
    assert np.array_equal(D.cpu().double().numpy(), ref)


def test_4096_cubed_with_workspace_skewed_split_exact():
    """4096^3 through tcm_gemm_ex_ws as the bench times it: the 28 tiles of the last round split
    automatically, the owner part 41 of the 64 K blocks and the helper 23 (skewed).  Integer inputs,
    so every sampled output of every 128 x 128 block must equal the oracle exactly."""
    import tensor_core_matrix_gb300 as tcm
    M = N = K = 4096
    g = si.generator(4096)
    A = si.integers((M, K), g)
    B = si.integers((N, K), g)
    if torch.cuda.get_device_properties(0).multi_processor_count == 152:
        assert tcm.tcm_gemm_workspace_bytes(M, N, K, torch.bfloat16) > 0  # the split is used
    D = run_gemm_ex(A, B, torch.float32, workspace=True)
    rows, cols = sample_indices(M, N)
    ref, _ = oracle_ref(A, B, rows=rows, cols=cols)
    assert np.array_equal(D.double().numpy()[rows, cols], ref)


@pytest.mark.parametrize("in_fmt", ["bf16", "e4m3"])
def test_8192_cubed_with_workspace_sampled(in_fmt):
    """The bench's two dense GEMMs through tcm_gemm_ex_ws at full size (tail tiles split over K),
    sampled outputs of every 128 x 128 block against the oracle."""
    if in_fmt == "bf16":
        c = si.llm_case(8192, 8192, 8192, seed=2)
        kw = {}
    else:
        c = si.fp8_case(seed=3)
        kw = dict(sa=c["sa"], sb=c["sb"], bias=c["bias"])
    D = run_gemm_ex(c["A"], c["B"], torch.bfloat16, workspace=True, **kw)
    rows, cols = sample_indices(8192, 8192)
    ref, S = oracle_ref(c["A"], c["B"], rows=rows, cols=cols, **kw)
    assert ratio(D, ref, S, scale=kw.get("sa", 1.0) * kw.get("sb", 1.0), rows=rows, cols=cols) <= 1.0
    assert not torch.isnan(D).any()


@pytest.mark.parametrize("ks", [2, 4])
@pytest.mark.parametrize("M,N,K", [(16, 1024, 2048), (64, 384, 1000), (1, 256, 512), (16, 512, 64), (40, 300, 4096)])
def test_k_split_cluster_integer_exact(override, ks, M, N, K):
    """Skinny M (operands swapped) with each tile's K split over a cluster and reduced through DSMEM;
    K = 64 leaves some CTAs of a 4-way split with no K blocks."""
    override.tcm_set_config_override(0, 0, 0, 0, ks)
    g = si.generator(M * 3 + N + K + ks)
    A = si.integers((M, K), g)
    B = si.integers((N, K), g)
    D = run_gemm_ex(A, B, torch.float32)
    ref, _ = oracle_ref(A, B)
    assert np.array_equal(D.double().numpy(), ref)


@pytest.mark.parametrize("ks", [2, 4])
def test_k_split_cluster_fp8_with_epilogue(override, ks):
    override.tcm_set_config_override(0, 0, 0, 0, ks)
    case = si.fp8_case(16, 2048, 4096, b_fmt="e5m2", seed=5)
    g = si.generator(9)
    C = si.normal((16, 2048), g)
    D = run_gemm_ex(case["A"], case["B"], torch.bfloat16, C=C, beta=0.5, sa=case["sa"], sb=case["sb"],
                    bias=case["bias"])
    ref, S = oracle_ref(case["A"], case["B"], C=C, beta=0.5, sa=case["sa"], sb=case["sb"], bias=case["bias"])
    assert ratio(D, ref, S, scale=case["sa"] * case["sb"]) <= 1.0


@pytest.mark.parametrize("cg", [1, 2])
def test_pipeline_timeout_is_reported_and_context_stays_usable(override, cg):
    """A wait that nothing will satisfy runs out, is reported, and the next launch is correct."""
    tcm = override
    override.tcm_set_config_override(cg, 256)
    d = dev()
    g = si.generator(77)
    A = si.integers((512, 256), g)
    B = si.integers((512, 256), g)
    Ad, Bd = A.to(d), B.to(d)
    D = torch.zeros((512, 512), dtype=torch.float32, device=d)
    tcm.tcm_clear_device_status()
    tcm.tcm_set_timeout_ns(50_000_000)
    try:
        tcm.tcm_debug_fail_next_launch(1)
        tcm.tcm_gemm_ex(Ad, Bd, D)
        code, site = tcm.tcm_get_device_status()
        # whichever wait on the starved stage gives up first: the issuer's (2)
        # or the epilogue's, which waits for the same tile (4)
        assert code == 5 and site in (2, 4)
    finally:
        tcm.tcm_set_timeout_ns(0)
        tcm.tcm_clear_device_status()
    tcm.tcm_gemm_ex(Ad, Bd, D)
    assert tcm.tcm_get_device_status() == (0, 0)
    ref, _ = oracle_ref(A, B)
    assert np.array_equal(D.cpu().double().numpy(), ref)


# ------------------------------------------------------------------ configured workloads

def test_small_config_512_bf16_with_c_and_16x8x16_tile():
    case = si.small_case()
    D = run_gemm_ex(case["A"], case["B"], torch.float32, C=case["C"], alpha=1.0, beta=1.0)
    ref, S = oracle_ref(case["A"], case["B"], C=case["C"], alpha=1.0, beta=1.0)
    assert ratio(D, ref, S) <= 1.0
    # the single m16n8k16 tile: A 16x16, B 16x8 (stored 8 x 16), C/D 16x8
    A, B, C = case["A"][:16, :16].contiguous(), case["B"][:8, :16].contiguous(), case["C"][:16, :8].contiguous()
    D1 = run_gemm_ex(A, B, torch.float32, C=C, alpha=1.0, beta=1.0)
    ref1, S1 = oracle_ref(A, B, C=C, alpha=1.0, beta=1.0)
    assert ratio(D1, ref1, S1) <= 1.0


@pytest.mark.parametrize("M,N,K,fmt,out", [
    (777, 1000, 520, "bf16", torch.bfloat16), (130, 300, 8, "f16", torch.float16),
    (64, 96, 4096, "bf16", torch.float32), (1536, 1280, 320, "f16", torch.bfloat16),
    (96, 40, 200, "bf16", torch.bfloat16),
])
def test_ragged_shapes_with_beta(M, N, K, fmt, out):
    g = si.generator(M * 7 + N)
    A = si.normal((M, K), g, dtype=fmt)
    B = si.normal((N, K), g, dtype=fmt)
    C = si.normal((M, N), g, dtype={torch.bfloat16: "bf16", torch.float16: "f16", torch.float32: "f32"}[out])
    D = run_gemm_ex(A, B, out, C=C, alpha=1.25, beta=-0.5)
    ref, S = oracle_ref(A, B, C=C, alpha=1.25, beta=-0.5)
    assert ratio(D, ref, S, scale=1.25) <= 1.0


@pytest.mark.parametrize("fb", ["e4m3", "e5m2"])
@pytest.mark.parametrize("M,N,K", [(512, 512, 512), (333, 700, 1040)])
def test_fp8_scales_and_bias(fb, M, N, K):
    case = si.fp8_case(M, N, K, b_fmt=fb, seed=3)
    D = run_gemm_ex(case["A"], case["B"], torch.bfloat16, sa=case["sa"], sb=case["sb"], bias=case["bias"])
    ref, S = oracle_ref(case["A"], case["B"], sa=case["sa"], sb=case["sb"], bias=case["bias"])
    assert ratio(D, ref, S, scale=case["sa"] * case["sb"]) <= 1.0


@pytest.mark.parametrize("M,N,K", [(1, 256, 512), (16, 1024, 1024), (64, 384, 256), (16, 200, 64)])
def test_skinny_m_swaps_operands(M, N, K):
    g = si.generator(M + 3 * N)
    A = si.normal((M, K), g)
    B = si.normal((N, K), g, std=0.02)
    C = si.normal((M, N), g)
    bias = si.normal((N,), g)
    D = run_gemm_ex(A, B, torch.bfloat16, C=C, beta=1.0, bias=bias)
    ref, S = oracle_ref(A, B, C=C, beta=1.0, bias=bias)
    assert ratio(D, ref, S) <= 1.0


def test_k_zero_gives_beta_c():
    M, N = 100, 72
    C = si.normal((M, N), si.generator(1), dtype="f32")
    A = torch.zeros((M, 8), dtype=torch.bfloat16)[:, :0]
    B = torch.zeros((N, 8), dtype=torch.bfloat16)[:, :0]
    d = dev()
    D = torch.full((M, N), float("nan"), dtype=torch.float32, device=d)
    import tensor_core_matrix_gb300 as tcm
    Ad = torch.zeros((M, 8), dtype=torch.bfloat16, device=d)
    Bd = torch.zeros((N, 8), dtype=torch.bfloat16, device=d)
    tcm.tcm_gemm_ex(Ad[:, :0], Bd[:, :0], D, C=C.to(d), beta=2.0)
    assert torch.equal(D.cpu(), 2.0 * C)
    del A, B


def test_tcm_gemm_packed_entry_point():
    import tensor_core_matrix_gb300 as tcm
    d = dev()
    g = si.generator(12)
    A = si.normal((256, 384), g)
    B = si.normal((320, 384), g)
    C = si.normal((256, 320), g)
    D = torch.empty((256, 320), dtype=torch.bfloat16, device=d)
    tcm.tcm_gemm(A.to(d), B.to(d), D, C=C.to(d), alpha=2.0, beta=1.0)
    ref, S = oracle_ref(A, B, C=C, alpha=2.0, beta=1.0)
    assert ratio(D.cpu(), ref, S, scale=2.0) <= 1.0


def test_c_aliasing_d_in_place():
    import tensor_core_matrix_gb300 as tcm
    d = dev()
    g = si.generator(13)
    A = si.normal((384, 256), g)
    B = si.normal((512, 256), g)
    C = si.normal((384, 512), g, dtype="f32")
    Dd = C.to(d).clone()
    tcm.tcm_gemm_ex(A.to(d), B.to(d), Dd, C=Dd, beta=1.0)
    ref, S = oracle_ref(A, B, C=C, beta=1.0)
    assert ratio(Dd.cpu(), ref, S) <= 1.0


# ------------------------------------------------------------------ full-size workloads

@pytest.mark.parametrize("fmt", ["f16", "bf16"])
def test_square_4096_full_oracle(fmt):
    case = si.square_case(4096, fmt=fmt)
    D = run_gemm_ex(case["A"], case["B"], torch.bfloat16)
    ref, S = oracle_ref(case["A"], case["B"])
    assert ratio(D, ref, S) <= 1.0


@pytest.mark.parametrize("M,N,K", [(8192, 28672, 8192), (8192, 8192, 28672), (8192, 24576, 8192),
                                   (16, 28672, 8192)])
def test_llm_shapes_sampled(M, N, K):
    case = si.llm_case(M, N, K)
    D = run_gemm_ex(case["A"], case["B"], torch.bfloat16)
    rows, cols = sample_indices(M, N)
    ref, S = oracle_ref(case["A"], case["B"], rows=rows, cols=cols)
    assert ratio(D, ref, S, rows=rows, cols=cols) <= 1.0
    assert not torch.isnan(D).any()


@pytest.mark.parametrize("fb", ["e4m3", "e5m2"])
def test_fp8_8192_sampled(fb):
    case = si.fp8_case(b_fmt=fb)
    D = run_gemm_ex(case["A"], case["B"], torch.bfloat16, sa=case["sa"], sb=case["sb"], bias=case["bias"])
    rows, cols = sample_indices(8192, 8192)
    ref, S = oracle_ref(case["A"], case["B"], sa=case["sa"], sb=case["sb"], bias=case["bias"], rows=rows, cols=cols)
    assert ratio(D, ref, S, scale=case["sa"] * case["sb"], rows=rows, cols=cols) <= 1.0
    assert not torch.isnan(D).any()
