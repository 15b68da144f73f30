"""GPU parity of the exact INT8 x INT8 -> INT32 GEMM (.satfinite) on the bf16 tensor path
against the oracle: integer results, so every output must match bit for bit."""
import numpy as np
import pytest
import torch

import oracle
import synth_inputs as si
from parity import dev, padded, sample_indices

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


def run_i8(tcm, A, B, C=None):
    """D (and C) with row pitches rounded up to 16 bytes, as the entry point requires; A and B
    with their natural (any) pitch."""
    d = dev()
    M, N = A.shape[0], B.shape[0]
    D = padded(torch.full((M, N), -7, dtype=torch.int32), d)
    tcm.tcm_gemm_i8(A.to(d), B.to(d), D, C=None if C is None else padded(C, d))
    code, site = tcm.tcm_get_device_status()
    assert code == 0, (code, site)
    return D.cpu().numpy()


@pytest.mark.parametrize("with_c", [False, True])
@pytest.mark.parametrize("M,N,K", [(128, 128, 64), (256, 512, 1024), (300, 520, 136), (1000, 1030, 2000),
                                   (1, 256, 4096), (513, 257, 3000)])
def test_int8_full_range_exact(tcm, M, N, K, with_c):
    g = si.generator(M * 7 + N + K + with_c)
    A = torch.randint(-128, 128, (M, K), generator=g, dtype=torch.int8)
    B = torch.randint(-128, 128, (N, K), generator=g, dtype=torch.int8)
    C = torch.randint(-2 ** 31, 2 ** 31 - 1, (M, N), generator=g, dtype=torch.int64).to(torch.int32) if with_c else None
    D = run_i8(tcm, A, B, C)
    ref = oracle.gemm_i8(A.numpy(), B.numpy(), None if C is None else C.numpy())
    assert np.array_equal(D, ref)


def test_int8_chunks_at_two_to_the_24(tcm):
    """a = b = -128 everywhere: every 1024-long chunk sums to exactly 2^24 (the largest partial sum
    the fp32 accumulator must hold), four chunks per output."""
    A = torch.full((256, 4096), -128, dtype=torch.int8)
    D = run_i8(tcm, A, A[:256])
    assert np.all(D == 16384 * 4096)


def test_int8_saturation_both_ways(tcm):
    """K = 131071 (the limit): 16384 K = 2^31 - 16384; + C = 2^31 - 1 clamps to INT32_MAX, and the
    negative case (-128 * 127 * K + INT32_MIN) clamps to INT32_MIN."""
    K = 131071
    A = torch.full((2, K), -128, dtype=torch.int8)
    B = torch.stack([torch.full((K,), -128, dtype=torch.int8), torch.full((K,), 127, dtype=torch.int8)])
    C = torch.tensor([[2 ** 31 - 1, -2 ** 31], [0, 0]], dtype=torch.int32)
    D = run_i8(tcm, A, B, C)
    assert D[0, 0] == 2 ** 31 - 1 and D[0, 1] == -2 ** 31
    assert D[1, 0] == 16384 * K and D[1, 1] == -16256 * K
    assert np.array_equal(D, oracle.gemm_i8(A.numpy(), B.numpy(), C.numpy()))


def test_int8_8192_sampled(tcm):
    c = si.int8_case()
    D = run_i8(tcm, c["A"], c["B"])
    rows, cols = sample_indices(8192, 8192)
    assert np.array_equal(D[rows, cols], oracle.gemm_i8(c["A"].numpy(), c["B"].numpy(), rows=rows, cols=cols))


def test_int8_k0_gives_c_and_limits(tcm):
    d = dev()
    C = torch.randint(-1000, 1000, (300, 260), dtype=torch.int32)
    D = run_i8(tcm, torch.empty((300, 0), dtype=torch.int8), torch.empty((260, 0), dtype=torch.int8), C)
    assert np.array_equal(D, C.numpy())
    A = torch.zeros((128, 131072), dtype=torch.int8, device=d)
    with pytest.raises(ValueError, match="unsupported sizes"):
        tcm.tcm_gemm_i8(A, A, torch.empty((128, 128), dtype=torch.int32, device=d))
    A = torch.zeros((128, 256), dtype=torch.int8, device=d)
    with pytest.raises(ValueError, match="workspace holds"):
        tcm.tcm_gemm_i8(A, A, torch.empty((128, 128), dtype=torch.int32, device=d),
                        workspace=torch.empty(1024, dtype=torch.uint8, device=d))


def test_int8_odd_pitches_and_unaligned_bases(tcm):
    """A and B may have any row pitch and start at any byte (the conversion reads single bytes):
    A at a 3-byte offset with pitch K + 13, B at a 1-byte offset with pitch K + 5, K = 777
    (not a multiple of 8 or 64), ragged M and N; C and D padded to 16-byte pitches."""
    d = dev()
    M, N, K = 300, 260, 777
    g = si.generator(12)
    A = torch.randint(-128, 128, (M, K), generator=g, dtype=torch.int8)
    B = torch.randint(-128, 128, (N, K), generator=g, dtype=torch.int8)
    C = torch.randint(-2 ** 31, 2 ** 31 - 1, (M, N), generator=g, dtype=torch.int64).to(torch.int32)
    buf_a = torch.zeros((M, K + 13), dtype=torch.int8, device=d)
    buf_a[:, 3:3 + K] = A.to(d)
    buf_b = torch.zeros((N, K + 5), dtype=torch.int8, device=d)
    buf_b[:, 1:1 + K] = B.to(d)
    D = padded(torch.full((M, N), -7, dtype=torch.int32), d)
    tcm.tcm_gemm_i8(buf_a[:, 3:3 + K], buf_b[:, 1:1 + K], D, C=padded(C, d))
    code, site = tcm.tcm_get_device_status()
    assert code == 0, (code, site)
    assert np.array_equal(D.cpu().numpy(), oracle.gemm_i8(A.numpy(), B.numpy(), C.numpy()))


def test_int8_starved_stage_times_out_and_context_stays_usable(tcm):
    """The first stage is never loaded (test hook): a bounded wait gives up (MMA issuer, site 2, or
    epilogue, site 4), the status says so, the kernel returns, and the next launch is exact."""
    d = dev()
    M, N, K = 512, 512, 2048
    g = si.generator(13)
    A = torch.randint(-128, 128, (M, K), generator=g, dtype=torch.int8)
    B = torch.randint(-128, 128, (N, K), generator=g, dtype=torch.int8)
    Ad, Bd = A.to(d), B.to(d)
    D = torch.zeros((M, N), dtype=torch.int32, device=d)
    tcm.tcm_clear_device_status()
    tcm.tcm_set_timeout_ns(50_000_000)
    try:
        tcm.tcm_debug_fail_next_launch(1)
        tcm.tcm_gemm_i8(Ad, Bd, D)
        code, site = tcm.tcm_get_device_status()
        assert code == 5 and site in (2, 4)
    finally:
        tcm.tcm_set_timeout_ns(0)
        tcm.tcm_clear_device_status()
    tcm.tcm_gemm_i8(Ad, Bd, D)
    assert tcm.tcm_get_device_status() == (0, 0)
    assert np.array_equal(D.cpu().numpy(), oracle.gemm_i8(A.numpy(), B.numpy()))
