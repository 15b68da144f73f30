"""Shared helpers of the GPU parity tests: run the library, compare with the oracle."""
import numpy as np
import torch

import oracle
import synth_inputs as si
import tensor_core_matrix_gb300 as tcm

FMT_OF = {torch.bfloat16: "bf16", torch.float16: "f16", torch.float32: "f32",
          torch.float8_e4m3fn: "e4m3", torch.float8_e5m2: "e5m2"}


def dev():
    return torch.device("cuda:0")


def padded(t, device):
    """Copy of 2-D ``t`` on ``device`` whose row pitch is rounded up to 16 bytes (a view of a wider buffer)."""
    rows, cols = t.shape
    per = max(1, 16 // t.element_size())
    pitch = max(per, -(-cols // per) * per)
    if pitch == cols:
        return t.to(device).contiguous()
    buf = torch.zeros((rows, pitch), dtype=t.dtype, device=device)
    buf[:, :cols] = t.to(device)
    return buf[:, :cols]


def workspace_for(M, N, K, a_dtype, b_dtype, device):
    """A workspace of the size tcm_gemm_ex_ws asks for (at least 16 bytes)."""
    n = tcm.tcm_gemm_workspace_bytes(M, N, K, a_dtype, b_dtype)
    return torch.empty(max(n, 16), dtype=torch.uint8, device=device)


def run_gemm_ex(A, B, out_dtype, *, C=None, alpha=1.0, beta=0.0, sa=None, sb=None, bias=None,
                fill=float("nan"), workspace=False):
    """Run tcm_gemm_ex (tcm_gemm_ex_ws with a workspace of the queried size if `workspace`) on
    CPU tensors moved to the GPU; D is pre-filled with NaN."""
    d = dev()
    Ad, Bd = padded(A, d), padded(B, d)
    M, N = A.shape[0], B.shape[0]
    D = padded(torch.full((M, N), fill, dtype=out_dtype), d)
    Cd = None if C is None else padded(C, d)
    sad = None if sa is None else torch.tensor([sa], dtype=torch.float32, device=d)
    sbd = None if sb is None else torch.tensor([sb], dtype=torch.float32, device=d)
    biasd = None if bias is None else bias.to(d)
    ws = workspace_for(M, N, A.shape[1], A.dtype, B.dtype, d) if workspace else None
    tcm.tcm_gemm_ex(Ad, Bd, D, C=Cd, alpha=alpha, beta=beta, a_scale=sad, b_scale=sbd, bias=biasd, workspace=ws)
    code, site = tcm.tcm_get_device_status()
    assert code == 0, f"device status {code} at site {site}"
    return D.cpu()


def oracle_ref(A, B, *, C=None, alpha=1.0, beta=0.0, sa=1.0, sb=1.0, bias=None, rows=None, cols=None,
               K=None):
    return oracle.gemm(si.codes(A), si.codes(B), FMT_OF[A.dtype], FMT_OF[B.dtype],
                       C=None if C is None else si.codes(C), c_fmt=FMT_OF[C.dtype] if C is not None else "f32",
                       bias=None if bias is None else si.codes(bias),
                       bias_fmt=FMT_OF[bias.dtype] if bias is not None else "bf16",
                       alpha=alpha, beta=beta, sa=sa, sb=sb, rows=rows, cols=cols, K=K)


def ratio(D, ref, S, scale=1.0, rows=None, cols=None):
    """max |D - ref| / bound over the (sampled) outputs."""
    codes = si.codes(D)
    if rows is not None:
        codes = codes[rows, cols]
    return oracle.err_over_bound(codes, FMT_OF[D.dtype], ref, S, scale)


def sample_indices(M, N, per_tile=4, tile=128, seed=0):
    """>= per_tile random outputs in every tile x tile block, plus rows 0 and M-1 and columns 0 and N-1."""
    g = np.random.default_rng(seed)
    rows, cols = [], []
    for m0 in range(0, M, tile):
        for n0 in range(0, N, tile):
            mh, nh = min(tile, M - m0), min(tile, N - n0)
            rows.append(m0 + g.integers(0, mh, per_tile))
            cols.append(n0 + g.integers(0, nh, per_tile))
    rows.append(np.zeros(N, dtype=np.int64)); cols.append(np.arange(N))
    rows.append(np.full(N, M - 1, dtype=np.int64)); cols.append(np.arange(N))
    rows.append(np.arange(M)); cols.append(np.zeros(M, dtype=np.int64))
    rows.append(np.arange(M)); cols.append(np.full(M, N - 1, dtype=np.int64))
    return np.concatenate(rows).astype(np.int64), np.concatenate(cols).astype(np.int64)
