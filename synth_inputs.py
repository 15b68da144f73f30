"""Seeded synthetic inputs for the GEMM workloads.

This module is shared by the CUDA path's tests/bench and by the CPU oracle,
and therefore holds none of the GEMM's arithmetic: it only draws random
numbers with a seeded ``torch.Generator`` on the CPU and stores them in the
input formats with torch's own round-to-nearest-even casts.  Everything is
returned as CPU tensors; callers move them to the device.

Workloads (shapes, value distributions, seeds):

* ``small``       512^3 bf16, A/B ~ U[-1,1], C fp32 ~ U[-1,1], alpha=beta=1, seed 0
* ``square``      4096^3 fp16 (or bf16), A/B ~ N(0,1)/sqrt(K), beta=0, seed 1
* ``llm``         bf16 activations ~ N(0,1) (M x K), weights ~ N(0,0.02) (N x K), seed 2
* ``fp8``         8192^3 E4M3 (x E4M3 or E5M2), N(0,1) scaled so amax lands
                  on the format's largest finite value, bias bf16 ~ N(0,1), seed 3
* ``sparse``      logical A ~ N(0,1) bf16 (pruned by the method), B ~ N(0,1), seed 4
* ``mx``          MXFP8: N(0,1) in blocks of 32 along K with E8M0 scales (OCP MX
                  conversion), E4M3 elements, seed 5
* ``nvfp4``       8192^3 NVFP4 x NVFP4: N(0,1), per-tensor fp32 scale, UE4M3 scales per
                  16 along K, E2M1 elements (packed), seed 7; alpha = product of the
                  two per-tensor scales
* ``w4a8``        8192^3 A E4M3 activations x B E2M1 weights (FP4, two per byte),
                  N(0,1) each scaled per tensor so amax lands on the format max
                  (448, 6), seed 6

torch has no cast to FP4 E2M1, so :func:`fp4_e2m1` rounds to the E2M1 grid
itself: nearest value, ties to the even code, saturating at +-6 (OCP FP4).
"""
from __future__ import annotations

import math

import torch

FP8_MAX = {"e4m3": 448.0, "e5m2": 57344.0}
TORCH_DTYPE = {
    "bf16": torch.bfloat16,
    "f16": torch.float16,
    "f32": torch.float32,
    "e4m3": torch.float8_e4m3fn,
    "e5m2": torch.float8_e5m2,
}


def generator(seed: int) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    return g


def uniform(shape, g, lo=-1.0, hi=1.0, dtype="bf16"):
    x = torch.rand(shape, generator=g, dtype=torch.float32) * (hi - lo) + lo
    return x.to(TORCH_DTYPE[dtype])


def normal(shape, g, std=1.0, dtype="bf16"):
    x = torch.randn(shape, generator=g, dtype=torch.float32) * std
    return x.to(TORCH_DTYPE[dtype])


def integers(shape, g, lo=-8, hi=8, dtype="bf16"):
    """Integer-valued inputs in [lo, hi]; exactly representable in every format here."""
    x = torch.randint(lo, hi + 1, shape, generator=g, dtype=torch.int32).to(torch.float32)
    return x.to(TORCH_DTYPE[dtype])


FP4_GRID = (0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0)  # E2M1 magnitudes of codes 0..7


def fp4_e2m1(x: torch.Tensor) -> torch.Tensor:
    """E2M1 codes (uint8, one per element) of fp32 ``x``: nearest grid value, ties to
    the even code, |x| > 6 saturating to 6; the sign is bit 3."""
    x = x.to(torch.float32)
    grid = torch.tensor(FP4_GRID, dtype=torch.float32)
    a = x.abs().clamp(max=6.0)
    d = (a[..., None] - grid).abs()
    best = d == d.min(dim=-1, keepdim=True).values
    idx = torch.arange(8)
    score = best.to(torch.int64) * (2 - (idx & 1))  # of two nearest codes the even one wins
    code = score.argmax(dim=-1).to(torch.uint8)
    return code | ((x < 0).to(torch.uint8) << 3)


def pack_fp4(codes: torch.Tensor) -> torch.Tensor:
    """Two E2M1 codes per byte along the last dimension: element 2i in the low nibble."""
    return (codes[..., 0::2] | (codes[..., 1::2] << 4)).contiguous()


def fp4_per_tensor(x: torch.Tensor):
    """Packed E2M1 of fp32 ``x`` scaled so its amax lands on 6; returns (packed, dequant scale)."""
    amax = float(x.abs().max())
    s_quant = 6.0 / amax if amax > 0 else 1.0
    return pack_fp4(fp4_e2m1(x * s_quant)), float(torch.tensor(1.0 / s_quant, dtype=torch.float32))


def fp8_per_tensor(x: torch.Tensor, fmt: str):
    """Store fp32 ``x`` in ``fmt`` with one per-tensor factor chosen so that the
    largest |x| lands on the format's largest finite value.

    Returns ``(q, scale)``: the fp8 tensor and the fp32 dequantisation factor
    (real value ~= q * scale).
    """
    amax = float(x.abs().max())
    s_quant = FP8_MAX[fmt] / amax if amax > 0 else 1.0
    q = (x * s_quant).clamp(-FP8_MAX[fmt], FP8_MAX[fmt]).to(TORCH_DTYPE[fmt])
    return q, float(torch.tensor(1.0 / s_quant, dtype=torch.float32))


FP8_EMAX = {"e4m3": 8, "e5m2": 15}  # exponent of the largest finite value


def mx_quantize(x: torch.Tensor, fmt: str, block: int = 32):
    """Store fp32 ``x`` (rows x K) as MX blocks: per ``block`` consecutive K
    elements one E8M0 scale 2^e with e = floor(log2(amax)) - emax(fmt) (the OCP
    MX conversion; an all-zero block gets e = -127), elements stored in ``fmt``
    with torch's round-to-nearest-even cast of x / 2^e, clamped to the format's
    finite range.  Returns ``(q, scale_codes)``: q in ``fmt``, scale codes uint8
    (rows x K/block, code = e + 127)."""
    rows, K = x.shape
    xb = x.reshape(rows, K // block, block).to(torch.float32)
    amax = xb.abs().amax(dim=2)
    e = torch.floor(torch.log2(torch.where(amax > 0, amax, torch.ones_like(amax)))) - FP8_EMAX[fmt]
    e = torch.where(amax > 0, e, torch.full_like(e, -127.0)).clamp(-127, 127)
    q = (xb / torch.exp2(e)[..., None]).clamp(-FP8_MAX[fmt], FP8_MAX[fmt]).reshape(rows, K)
    return q.to(TORCH_DTYPE[fmt]), (e + 127).to(torch.uint8)


def mx_case(M=8192, N=8192, K=8192, a_fmt="e4m3", b_fmt="e4m3", seed=5):
    g = generator(seed)
    xa = torch.randn((M, K), generator=g, dtype=torch.float32)
    xb = torch.randn((N, K), generator=g, dtype=torch.float32)
    A, SA = mx_quantize(xa, a_fmt)
    B, SB = mx_quantize(xb, b_fmt)
    return dict(A=A, SA=SA, B=B, SB=SB, a_fmt=a_fmt, b_fmt=b_fmt, out_fmt="bf16")


def nvfp4_quantize(x: torch.Tensor, block: int = 16):
    """NVFP4 storage of fp32 ``x`` (rows x K): a per-tensor fp32 scale g = amax / (448 * 6),
    per ``block`` K elements a UE4M3 scale s = RNE_e4m3(block_amax / 6 / g) (torch's cast of
    a non-negative value; its code is the UE4M3 code), and E2M1 elements RNE(x / (s g)).
    Real value ~= element * s * g.  Returns (packed E2M1, scale codes uint8 rows x K/block, g)."""
    rows, K = x.shape
    x = x.to(torch.float32)
    amax = float(x.abs().max())
    g = float(torch.tensor(amax / (448.0 * 6.0) if amax > 0 else 1.0, dtype=torch.float32))
    xb = x.reshape(rows, K // block, block)
    s = (xb.abs().amax(dim=2) / 6.0 / g).clamp(max=448.0).to(torch.float8_e4m3fn)
    s_val = s.to(torch.float32)
    denom = torch.where(s_val > 0, s_val * g, torch.ones_like(s_val))
    q = fp4_e2m1((xb / denom[..., None]).reshape(rows, K))
    return pack_fp4(q), s.view(torch.uint8), g


def nvfp4_case(M=8192, N=8192, K=8192, seed=7):
    g = generator(seed)
    xa = torch.randn((M, K), generator=g, dtype=torch.float32)
    xb = torch.randn((N, K), generator=g, dtype=torch.float32)
    A, SA, ga = nvfp4_quantize(xa)
    B, SB, gb = nvfp4_quantize(xb)
    return dict(A=A, SA=SA, B=B, SB=SB, alpha=float(torch.tensor(ga * gb, dtype=torch.float32)), out_fmt="bf16")


FP4_EMAX = 2  # exponent of E2M1's largest finite value (6 = 1.5 * 2^2)


def mxfp4_quantize(x: torch.Tensor, block: int = 32):
    """MXFP4 storage of fp32 ``x`` (rows x K): per ``block`` consecutive K elements one
    E8M0 scale 2^e with e = floor(log2(amax)) - emax(E2M1) (the OCP MX conversion; an
    all-zero block gets e = -127), elements E2M1 rounded to nearest (ties to the even
    code) of x / 2^e, saturated at +-6.  Returns (packed E2M1 rows x K/2, scale codes
    uint8 rows x K/block)."""
    rows, K = x.shape
    xb = x.reshape(rows, K // block, block).to(torch.float32)
    amax = xb.abs().amax(dim=2)
    e = torch.floor(torch.log2(torch.where(amax > 0, amax, torch.ones_like(amax)))) - FP4_EMAX
    e = torch.where(amax > 0, e, torch.full_like(e, -127.0)).clamp(-127, 127)
    q = fp4_e2m1((xb / torch.exp2(e)[..., None]).reshape(rows, K))
    return pack_fp4(q), (e + 127).to(torch.uint8)


def mxfp4_case(M=8192, N=8192, K=8192, seed=8):
    g = generator(seed)
    xa = torch.randn((M, K), generator=g, dtype=torch.float32)
    xb = torch.randn((N, K), generator=g, dtype=torch.float32)
    A, SA = mxfp4_quantize(xa)
    B, SB = mxfp4_quantize(xb)
    return dict(A=A, SA=SA, B=B, SB=SB, a_fmt="e2m1", b_fmt="e2m1", out_fmt="bf16")


def w4a8_case(M=8192, N=8192, K=8192, a_fmt="e4m3", seed=6):
    """FP8 activations A (M x K) times FP4 E2M1 weights B (N x K, packed: N x K/2 bytes)."""
    g = generator(seed)
    xa = torch.randn((M, K), generator=g, dtype=torch.float32)
    xb = torch.randn((N, K), generator=g, dtype=torch.float32)
    A, sa = fp8_per_tensor(xa, a_fmt)
    B, sb = fp4_per_tensor(xb)
    return dict(A=A, B=B, sa=sa, sb=sb, a_fmt=a_fmt, b_fmt="e2m1", out_fmt="bf16")


def int8_case(M=8192, N=8192, K=8192, seed=10):
    """Signed 8-bit A (M x K) and B (N x K), uniform over the full range -128 .. 127."""
    g = generator(seed)
    A = torch.randint(-128, 128, (M, K), generator=g, dtype=torch.int8)
    B = torch.randint(-128, 128, (N, K), generator=g, dtype=torch.int8)
    return dict(A=A, B=B, i8=True, out_fmt="i32")


def small_case(M=512, N=512, K=512, seed=0):
    g = generator(seed)
    A = uniform((M, K), g)
    B = uniform((N, K), g)
    C = uniform((M, N), g, dtype="f32")
    return dict(A=A, B=B, C=C, alpha=1.0, beta=1.0, in_fmt="bf16", out_fmt="f32")


def square_case(n=4096, fmt="f16", seed=1):
    g = generator(seed)
    A = normal((n, n), g, std=1.0 / math.sqrt(n), dtype=fmt)
    B = normal((n, n), g, std=1.0 / math.sqrt(n), dtype=fmt)
    return dict(A=A, B=B, C=None, alpha=1.0, beta=0.0, in_fmt=fmt, out_fmt="bf16")


def llm_case(M, N, K, seed=2):
    g = generator(seed)
    A = normal((M, K), g, std=1.0)
    B = normal((N, K), g, std=0.02)
    return dict(A=A, B=B, C=None, alpha=1.0, beta=0.0, in_fmt="bf16", out_fmt="bf16")


def fp8_case(M=8192, N=8192, K=8192, b_fmt="e4m3", seed=3):
    g = generator(seed)
    xa = torch.randn((M, K), generator=g, dtype=torch.float32)
    xb = torch.randn((N, K), generator=g, dtype=torch.float32)
    bias = normal((N,), g, std=1.0)
    A, sa = fp8_per_tensor(xa, "e4m3")
    B, sb = fp8_per_tensor(xb, b_fmt)
    return dict(A=A, B=B, C=None, bias=bias, sa=sa, sb=sb, alpha=1.0, beta=0.0,
                a_fmt="e4m3", b_fmt=b_fmt, out_fmt="bf16")


def sparse_case(M=8192, N=8192, K=8192, seed=4):
    g = generator(seed)
    A = normal((M, K), g, std=1.0)
    B = normal((N, K), g, std=1.0)
    return dict(A_logical=A, B=B, C=None, alpha=1.0, beta=0.0, in_fmt="bf16", out_fmt="bf16")


def codes(t: torch.Tensor):
    """Stored bit patterns of a CPU tensor as a numpy unsigned-integer array."""
    import numpy as np
    size = t.element_size()
    view = {1: torch.uint8, 2: torch.int16, 4: torch.int32}[size]
    arr = t.contiguous().view(view).numpy()
    return arr.view({1: np.uint8, 2: np.uint16, 4: np.uint32}[size])


def from_codes(arr, fmt: str) -> torch.Tensor:
    """CPU tensor of format ``fmt`` holding the given stored bit patterns."""
    import numpy as np
    size = {"bf16": 2, "f16": 2, "f32": 4, "e4m3": 1, "e5m2": 1}[fmt]
    signed = {1: np.uint8, 2: np.int16, 4: np.int32}[size]
    t = torch.from_numpy(np.ascontiguousarray(arr).view(signed).copy())
    return t.view(TORCH_DTYPE[fmt])
