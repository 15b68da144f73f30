"""tcm_gemm_ex_builtin_ws: the dense GEMM whose workspace lives inside the library.

It serves callers that cannot allocate device memory (for example code running under
another framework's memory manager, or a latency-critical path that must not call
cudaMalloc) and so cannot hand tcm_gemm_ex_ws a workspace.  Called through the C ABI
(ctypes), twice in a row on problems whose last round of CTA-pair tiles is split over
K -- so the built-in workspace is used, and the second call starts from the first
call's leftovers -- its output must equal that of tcm_gemm_ex_ws with a caller
workspace (same kernel, same order of accumulation), and stay within the oracle's bound
on sampled outputs.  This file is collected last.
"""
import ctypes

import numpy as np
import pytest
import torch

import synth_inputs as si
from parity import dev, oracle_ref, ratio, sample_indices

pytestmark = pytest.mark.gpu

BF16, E4M3 = 0, 3


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(0)
    import tensor_core_matrix_gb300 as tcm
    tcm.tcm_clear_device_status()
    yield tcm.load_library()
    tcm.tcm_set_config_override()


def builtin_gemm(lib, A, B, D, code, sa=None, sb=None, bias=None):
    """tcm_gemm_ex_builtin_ws through the C ABI (device pointers of contiguous tensors)."""
    vp = ctypes.c_void_p
    M, K = A.shape
    N = B.shape[0]
    st = lib.tcm_gemm_ex_builtin_ws(M, N, K, code, vp(A.data_ptr()), K, code, vp(B.data_ptr()), K, None, 0,
                                    vp(D.data_ptr()), N, BF16, 1.0, 0.0,
                                    vp(sa.data_ptr()) if sa is not None else None,
                                    vp(sb.data_ptr()) if sb is not None else None,
                                    vp(bias.data_ptr()) if bias is not None else None,
                                    vp(torch.cuda.current_stream().cuda_stream))
    assert st == 0, f"tcm_gemm_ex_builtin_ws returned status {st}"


@pytest.mark.parametrize("fmt", ["bf16", "e4m3"])
def test_builtin_workspace_matches_caller_workspace_twice(lib, fmt):
    import tensor_core_matrix_gb300 as tcm
    d = dev()
    M = N = K = 8192  # 1024 pair tiles on 76 pairs: 36 split over K, ~9 MiB of workspace
    if fmt == "bf16":
        c = si.llm_case(M, N, K, seed=2)
        code, kw, scale = BF16, {}, 1.0
    else:
        c = si.fp8_case(M, N, K, seed=3)
        code, scale = E4M3, c["sa"] * c["sb"]
        kw = dict(sa=torch.tensor([c["sa"]], device=d), sb=torch.tensor([c["sb"]], device=d), bias=c["bias"].to(d))
    A, B = c["A"].to(d), c["B"].to(d)
    need = tcm.tcm_gemm_workspace_bytes(M, N, K, A.dtype)
    assert 0 < need <= 10 << 20
    ref = torch.empty((M, N), dtype=torch.bfloat16, device=d)
    ws = torch.empty(need, dtype=torch.uint8, device=d)
    tcm.tcm_gemm_ex(A, B, ref, a_scale=kw.get("sa"), b_scale=kw.get("sb"), bias=kw.get("bias"), workspace=ws)
    rows, cols = sample_indices(M, N, per_tile=1)
    want, S = oracle_ref(c["A"], c["B"], rows=rows, cols=cols,
                         **({} if fmt == "bf16" else dict(sa=c["sa"], sb=c["sb"], bias=c["bias"])))
    for call in range(2):
        D = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device=d)
        builtin_gemm(lib, A, B, D, code, kw.get("sa"), kw.get("sb"), kw.get("bias"))
        assert tcm.tcm_get_device_status() == (0, 0)
        assert torch.equal(D, ref), f"call {call}: differs from tcm_gemm_ex_ws"
        assert ratio(D.cpu(), want, S, scale=scale, rows=rows, cols=cols) <= 1.0


def test_builtin_workspace_integer_exact_twice(lib):
    """Integer inputs (exact sums) on a shape with 8 split tiles, forced split: bit-exact with the
    oracle on every output, twice in a row."""
    import tensor_core_matrix_gb300 as tcm
    tcm.tcm_set_config_override(2, 256, 0, 0, 0, 2)  # 256-column pair tiles: 8 tail tiles split
    try:
        d = dev()
        M, N, K = 4096, 2560, 512
        g = si.generator(501)
        A, B = si.integers((M, K), g), si.integers((N, K), g)
        Ad, Bd = A.to(d), B.to(d)
        assert tcm.tcm_gemm_workspace_bytes(M, N, K, torch.bfloat16) > 0
        ref, _ = oracle_ref(A, B)
        for _ in range(2):
            D = torch.full((M, N), float("nan"), dtype=torch.float32, device=d)
            vp = ctypes.c_void_p
            st = lib.tcm_gemm_ex_builtin_ws(M, N, K, BF16, vp(Ad.data_ptr()), K, BF16, vp(Bd.data_ptr()), K, None, 0,
                                            vp(D.data_ptr()), N, 2, 1.0, 0.0, None, None, None,
                                            vp(torch.cuda.current_stream().cuda_stream))
            assert st == 0
            assert tcm.tcm_get_device_status() == (0, 0)
            assert np.array_equal(D.cpu().double().numpy(), ref)
    finally:
        tcm.tcm_set_config_override()
