"""CPU oracle for the tensor-core GEMM -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product library never loads it and
shares no code with it; the two meet only on the stored bit patterns of the
seeded inputs.

The arithmetic lives in ``oracle.c`` (plain C, binary64, natural k order).
This wrapper only marshals numpy arrays of stored codes into it, plus the
acceptance bound that compares a tensor-core result with the fp64 reference.

Sources of the definitions (page titles and sections):

* GEMM ``D = A B + C``: "NVIDIA MMA", section "从 FMA 到 MMA，再到 GEMM".
* A row-major / B column-major: "CUDA 014 - MMA 指令的用法详解", section
  "MMA 指令的格式" (the ``.row.col`` modifier).
* Input / accumulator / output stages and the epilogue
  (scale / bias / cast): "NVIDIA MMA", section "输入/累加/输出".
* 2:4 sparse A with ordered position metadata: "NVIDIA MMA", sections
  "稠密乘法与 2:4 结构化稀疏乘法" and "Ampere：FP16/BF16 与整数 MMA 基线".
* Block-scaled MMA (per-K-block scales applied before accumulation) and the
  MXFP8 block size of 32 with E8M0 scales: "NVIDIA MMA", sections
  "SM100：tcgen05.mma" and "MXFP4 与 NVFP4".
* Blocked scale layout (:func:`mx_pack_scales`): the pages require a scale
  layout contract without stating one ("MXFP4 与 NVFP4"); the layout checked
  here is the library's documented one, a pure index permutation.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

# The oracle's own format codes (mirrors the enum in oracle.c only).
FMT = {"bf16": 0, "f16": 1, "f32": 2, "e4m3": 3, "e5m2": 4, "e8m0": 5, "e2m1": 6, "ue4m3": 7}
# bytes of one stored unit; an E2M1 byte holds two elements (element 2i in the low nibble)
ELEM_BYTES = {"bf16": 2, "f16": 2, "f32": 4, "e4m3": 1, "e5m2": 1, "e8m0": 1, "e2m1": 1, "ue4m3": 1}
PER_UNIT = {"e2m1": 2}
CODE_DTYPE = {1: np.uint8, 2: np.uint16, 4: np.uint32}
# significand precision p (bits incl. the implicit one) and the smallest
# positive subnormal of each output format; an RNE cast to the format is
# within 2^-p relative (half an ulp) of its argument, plus the subnormal step.
PRECISION = {"bf16": 8, "f16": 11, "f32": 24, "e4m3": 4, "e5m2": 3}
MIN_SUBNORMAL = {"bf16": 2.0 ** -133, "f16": 2.0 ** -24, "f32": 2.0 ** -149, "e4m3": 2.0 ** -9, "e5m2": 2.0 ** -16}
ACT = {None: 0, "none": 0, "relu": 1, "gelu": 2}
# max |d/dx x Phi(x)| = 1.1289 (at x = +-sqrt 2): how far GELU can stretch an input error
GELU_LIPSCHITZ = 1.13
# Accumulation allowance relative to sum_k |a*b|, the tolerance the GEMM is
# held to for fp32 accumulation of any K.
ACC_REL = 1e-5


def build(force: bool = False) -> str:
    """Compile ``oracle.c`` into ``liboracle.so`` beside it (gcc, OpenMP).

    ``-ffp-contract=off`` keeps gcc from fusing a*b+c into fma on any host
    architecture, so the oracle does the same roundings on x86 and Arm.
    """
    with _lock:
        stale = (not os.path.exists(_LIB)) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC)
        if force or stale:
            tmp = _LIB + f".tmp{os.getpid()}"
            cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp",
                   "-ffp-contract=off", "-Wall", "-o", tmp, _SRC, "-lm"]
            subprocess.run(cmd, check=True)
            os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is not None:
        return _lib
    build()
    lib = ctypes.CDLL(_LIB)
    i64, i32, dbl, vp = ctypes.c_int64, ctypes.c_int, ctypes.c_double, ctypes.c_void_p
    lib.orc_decode.restype = dbl
    lib.orc_decode.argtypes = [ctypes.c_uint32, i32]
    lib.orc_decode_array.restype = i32
    lib.orc_decode_array.argtypes = [vp, i32, i64, vp]
    lib.orc_gemm.restype = i32
    lib.orc_gemm.argtypes = [i64, i64, i64, i32, vp, i64, i32, vp, i64, i32, vp, i64,
                             i32, vp, dbl, dbl, dbl, dbl, i64, vp, vp, vp, vp]
    lib.orc_gemm_mx.restype = i32
    lib.orc_gemm_mx.argtypes = [i64, i64, i64, i64, i32, i32, vp, i64, vp, i64, i32, vp, i64, vp, i64,
                                i32, vp, i64, i32, vp, dbl, dbl, i64, vp, vp, vp, vp]
    lib.orc_sp_compress.restype = i32
    lib.orc_activate.restype = i32
    lib.orc_activate.argtypes = [i64, vp, i32, vp]
    lib.orc_fp8_target.restype = i32
    lib.orc_fp8_target.argtypes = [i64, vp, ctypes.c_double, i32, vp]
    lib.orc_sp_compress.argtypes = [i64, i64, i32, vp, i64, vp, vp]
    lib.orc_sp_decompress.restype = i32
    lib.orc_sp_decompress.argtypes = [i64, i64, i32, vp, vp, vp, i64]
    lib.orc_gemm_i8.restype = i32
    lib.orc_gemm_i8.argtypes = [i64, i64, i64, vp, i64, vp, i64, vp, i64, i64, vp, vp, vp]
    _lib = lib
    return lib


def _codes(x: np.ndarray, fmt: str) -> np.ndarray:
    want = CODE_DTYPE[ELEM_BYTES[fmt]]
    x = np.ascontiguousarray(x)
    if x.dtype.itemsize != ELEM_BYTES[fmt]:
        raise ValueError(f"{fmt} codes need {ELEM_BYTES[fmt]}-byte elements, got {x.dtype}")
    return x.view(want)


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def decode(codes: np.ndarray, fmt: str) -> np.ndarray:
    """Exact real values (float64) of an array of stored codes of ``fmt``."""
    c = _codes(codes, fmt)
    per = PER_UNIT.get(fmt, 1)
    out = np.empty(c.shape[:-1] + (c.shape[-1] * per,) if c.ndim else (per,), dtype=np.float64)
    if _load().orc_decode_array(_ptr(c), FMT[fmt], c.size * per, _ptr(out)) != 0:
        raise ValueError("bad format")
    return out


def gemm(A, B, a_fmt, b_fmt, *, C=None, c_fmt="f32", bias=None, bias_fmt="bf16",
         alpha=1.0, beta=0.0, sa=1.0, sb=1.0, rows=None, cols=None, K=None):
    """fp64 reference ``alpha*sa*sb*sum_k a[m,k] b[n,k] + beta*C[m,n] + bias[n]``.

    ``A`` is M x lda codes (row-major, the first K columns used), ``B`` is
    N x ldb codes (B stored K-major), ``C`` M x ldc codes or None, ``bias``
    N codes or None.  With ``rows``/``cols`` (equal-length index arrays) only
    those outputs are computed.  Returns ``(ref, S)`` with
    ``S = sum_k |a b|``: shaped M x N, or like ``rows`` when sampling.
    """
    A = _codes(A, a_fmt)
    B = _codes(B, b_fmt)
    M, lda = A.shape
    N, ldb = B.shape
    lda *= PER_UNIT.get(a_fmt, 1)  # leading dimensions in elements
    ldb *= PER_UNIT.get(b_fmt, 1)
    K = lda if K is None else K
    if K > lda or K > ldb:
        raise ValueError("K exceeds a leading dimension")
    Cc = None if C is None else _codes(C, c_fmt)
    ldc = 0 if Cc is None else Cc.shape[1]
    bc = None if bias is None else _codes(bias, bias_fmt)
    if rows is None:
        nsamp = -1
        r = c = None
        ref = np.empty((M, N), dtype=np.float64)
    else:
        r = np.ascontiguousarray(rows, dtype=np.int64)
        c = np.ascontiguousarray(cols, dtype=np.int64)
        if r.shape != c.shape:
            raise ValueError("rows and cols differ in shape")
        nsamp = r.size
        ref = np.empty(r.shape, dtype=np.float64)
    S = np.empty_like(ref)
    rc = _load().orc_gemm(M, N, K, FMT[a_fmt], _ptr(A), lda, FMT[b_fmt], _ptr(B), ldb,
                          FMT[c_fmt], _ptr(Cc), ldc, FMT[bias_fmt], _ptr(bc),
                          float(alpha), float(beta), float(sa), float(sb),
                          nsamp, _ptr(r), _ptr(c), _ptr(ref), _ptr(S))
    if rc != 0:
        raise ValueError("orc_gemm rejected its arguments")
    return ref, S


def gemm_mx(A, SA, B, SB, a_fmt, b_fmt, *, block=32, sf_fmt="e8m0", C=None, c_fmt="f32", bias=None,
            bias_fmt="bf16", alpha=1.0, beta=0.0, rows=None, cols=None):
    """fp64 block-scaled reference: alpha * sum_g sa[m,g] sb[n,g] sum_{k in g} a[m,k] b[n,k] + beta C + bias.

    ``A`` M x K and ``B`` N x K element codes (packed for E2M1), ``SA`` M x K/block
    and ``SB`` N x K/block scale codes (uint8) of ``sf_fmt``: "e8m0" (MX, block 32:
    2^(code-127)) or "ue4m3" (NVFP4, block 16); other arguments as :func:`gemm`.
    Returns ``(ref, S)`` with S = sum_g sa sb sum_k |a b|.
    """
    A = _codes(A, a_fmt)
    B = _codes(B, b_fmt)
    SA = np.ascontiguousarray(SA, dtype=np.uint8)
    SB = np.ascontiguousarray(SB, dtype=np.uint8)
    M, lda = A.shape
    N, ldb = B.shape
    lda *= PER_UNIT.get(a_fmt, 1)
    ldb *= PER_UNIT.get(b_fmt, 1)
    K = lda
    if SA.shape != (M, K // block) or SB.shape != (N, K // block):
        raise ValueError("scale arrays must be M x K/block and N x K/block")
    Cc = None if C is None else _codes(C, c_fmt)
    ldc = 0 if Cc is None else Cc.shape[1]
    bc = None if bias is None else _codes(bias, bias_fmt)
    if rows is None:
        nsamp, r, c = -1, None, None
        ref = np.empty((M, N), dtype=np.float64)
    else:
        r = np.ascontiguousarray(rows, dtype=np.int64)
        c = np.ascontiguousarray(cols, dtype=np.int64)
        nsamp = r.size
        ref = np.empty(r.shape, dtype=np.float64)
    S = np.empty_like(ref)
    rc = _load().orc_gemm_mx(M, N, K, block, FMT[sf_fmt], FMT[a_fmt], _ptr(A), lda, _ptr(SA), SA.shape[1],
                             FMT[b_fmt], _ptr(B), ldb, _ptr(SB), SB.shape[1], FMT[c_fmt], _ptr(Cc), ldc,
                             FMT[bias_fmt], _ptr(bc), float(alpha), float(beta), nsamp, _ptr(r), _ptr(c),
                             _ptr(ref), _ptr(S))
    if rc != 0:
        raise ValueError("orc_gemm_mx rejected its arguments")
    return ref, S


def mx_pack_scales(SC, K, block=32, pad=127, reps=1):
    """Blocked layout of row-major scale codes ``SC`` (rows x K/block uint8).

    Code (r, j) goes to byte ``(r//128 * KT + j//4) * 512 + (r%32)*16 + ((r//32)%4)*4 + j%4``
    with ``KT = ceil(K / (4 block))``; every other byte of the ``ceil(rows/128) * KT * 512``
    bytes holds ``pad`` (1.0: 127 for E8M0, 0x38 for UE4M3).  With ``reps`` > 1 every
    512-byte atom is stored ``reps`` times in a row (NVFP4: 4).  Written as plain loops."""
    SC = np.ascontiguousarray(SC, dtype=np.uint8)
    rows, nblk = SC.shape
    assert K % block == 0 and nblk == K // block
    kt = (nblk + 3) // 4
    out = np.full(((rows + 127) // 128) * kt * 512 * reps, pad, dtype=np.uint8)
    for r in range(rows):
        for j in range(nblk):
            atom = (r // 128) * kt + j // 4
            for c in range(reps):
                out[(atom * reps + c) * 512 + (r % 32) * 16 + ((r // 32) % 4) * 4 + j % 4] = SC[r, j]
    return out

def sp_meta_pack(meta, K):
    """Hardware-ordered 2:4 metadata (the layout of ``tcm_sp_meta_pack`` in include/tcm.h) of
    canonical words ``meta`` (M x K/32 uint32), as bytes.  Plain loops over the definition:
    stage (t, kb) holds 128 lanes of 16 bytes; word k of lane L = 16a + 8s + r is the word the
    sparse MMA k of that stage reads for lane L: bits 16s..16s+15 of row 128t+16a+r's word
    q = 4kb+k in its low half and those of row 128t+16a+8+r in its high half."""
    meta = np.ascontiguousarray(meta).view(np.uint32)
    M, qn = meta.shape
    assert K % 32 == 0 and qn == K // 32
    kbs = (K + 127) // 128
    tiles = (M + 127) // 128
    out = np.zeros(tiles * kbs * 128 * 4, dtype=np.uint32)  # per stage: 128 lanes x 4 words
    fill = 0x44444444

    def word(row, q):
        return int(meta[row, q]) if row < M and q < qn else fill

    for t in range(tiles):
        for kb in range(kbs):
            for L in range(128):
                a, s, r = L // 16, (L // 8) % 2, L % 8
                for k in range(4):
                    q = 4 * kb + k
                    lo = (word(128 * t + 16 * a + r, q) >> (16 * s)) & 0xFFFF
                    hi = (word(128 * t + 16 * a + 8 + r, q) >> (16 * s)) & 0xFFFF
                    out[((t * kbs + kb) * 128 + L) * 4 + k] = lo | (hi << 16)
    return out.view(np.uint8)


def sp_compress(A, fmt):
    """2:4 prune+compress of logical A (M x K codes) -> (Ac M x K/2, meta M x K/32 uint32)."""
    A = _codes(A, fmt)
    M, K = A.shape
    Ac = np.zeros((M, K // 2), dtype=A.dtype)
    meta = np.zeros((M, K // 32), dtype=np.uint32)
    if _load().orc_sp_compress(M, K, FMT[fmt], _ptr(A), K, _ptr(Ac), _ptr(meta)) != 0:
        raise ValueError("orc_sp_compress rejected its arguments (K % 32 != 0?)")
    return Ac, meta


def sp_decompress(Ac, meta, fmt):
    """Inverse of :func:`sp_compress`: logical M x K codes with zeros restored."""
    Ac = _codes(Ac, fmt)
    meta = np.ascontiguousarray(meta, dtype=np.uint32)
    M, Kh = Ac.shape
    K = 2 * Kh
    A = np.zeros((M, K), dtype=Ac.dtype)
    if _load().orc_sp_decompress(M, K, FMT[fmt], _ptr(Ac), _ptr(meta), _ptr(A), K) != 0:
        raise ValueError("orc_sp_decompress rejected its arguments")
    return A


def gemm_i8(A, B, C=None, rows=None, cols=None):
    """Exact integer GEMM with .satfinite (``oracle.c``): int8 A (M x K), int8 B (N x K),
    optional int32 C (M x N); returns int32 outputs, clamped to the 32-bit range, of every
    (row, col) -- M x N -- or of the sampled (rows[t], cols[t])."""
    A = np.ascontiguousarray(A, dtype=np.int8)
    B = np.ascontiguousarray(B, dtype=np.int8)
    M, K = A.shape
    N = B.shape[0]
    assert B.shape[1] == K
    Cc = None if C is None else np.ascontiguousarray(C, dtype=np.int32)
    if rows is None:
        n, r, c = M * N, None, None
    else:
        r = np.ascontiguousarray(rows, dtype=np.int64)
        c = np.ascontiguousarray(cols, dtype=np.int64)
        n = r.size
    out = np.empty(n, dtype=np.int32)
    if _load().orc_gemm_i8(M, N, K, _ptr(A), K, _ptr(B), K, _ptr(Cc), N if Cc is not None else 0, n,
                           _ptr(r), _ptr(c), _ptr(out)) != 0:
        raise ValueError("orc_gemm_i8 rejected its arguments")
    return out.reshape(M, N) if rows is None else out


def activate(x, act):
    """act(x) in fp64 (``oracle.c``: RELU, GELU = x Phi(x)); x any float array."""
    x = np.ascontiguousarray(x, dtype=np.float64)
    y = np.empty_like(x)
    if _load().orc_activate(x.size, _ptr(x), ACT[act], _ptr(y)) != 0:
        raise ValueError(f"unknown activation {act!r}")
    return y


def fp32_reciprocal(d):
    """1 / d rounded to the nearest fp32 value, ties to even, decided exactly: the float
    candidates around fp32(1 / d) are compared with the rational 1 / d."""
    from fractions import Fraction
    exact = 1 / Fraction(float(d))
    c = np.float32(1.0 / float(d))
    cands = [np.nextafter(c, np.float32(-np.inf)), c, np.nextafter(c, np.float32(np.inf))]
    best = min(cands, key=lambda v: (abs(Fraction(float(v)) - exact), int(np.float32(v).view(np.uint32)) & 1))
    return float(best)


def fused_reference(ref, S, act, out_fmt, scale=1.0, d_scale=1.0):
    """Expected outputs of the fused epilogue and their bounds.

    ``ref``/``S`` come from :func:`gemm` (alpha, scales, C and bias applied).
    Returns ``(target, bound, y, bound_y)``: ``y = act(ref)`` with the bound
    ``bound_y`` on |y_gpu - y| (accumulation allowance and the fp32 epilogue
    arithmetic, stretched by the activation's Lipschitz constant, plus the
    device GELU's own evaluation error), and the stored value's target -- y,
    or y * RN32(1 / d_scale) saturated for FP8 outputs (the library's documented
    rule) -- with the bound on the decoded output (bound_y carried through the
    multiplier, the fp32 rounding of the device's product, then one RNE cast)."""
    ref = np.asarray(ref, dtype=np.float64)
    y = activate(ref, act)
    lip = GELU_LIPSCHITZ if ACT[act] == 2 else 1.0
    e_pre = ACC_REL * abs(scale) * np.asarray(S) + 2.0 ** -23 * np.abs(ref)
    e_y = lip * e_pre + (2.0 ** -20 * np.abs(ref) if ACT[act] == 2 else 0.0)
    if out_fmt in ("e4m3", "e5m2"):
        target = np.empty_like(y)
        mult = fp32_reciprocal(d_scale)
        _load().orc_fp8_target(y.size, _ptr(np.ascontiguousarray(y)), mult, FMT[out_fmt], _ptr(target))
        e_t = e_y * abs(mult) + 2.0 ** -23 * np.abs(target)
    else:
        target, e_t = y, e_y
    return target, e_t + 2.0 ** -PRECISION[out_fmt] * np.abs(target) + MIN_SUBNORMAL[out_fmt], y, e_y


def bound(ref, S, out_fmt, scale=1.0):
    """Per-element acceptance bound for a result cast to ``out_fmt``.

    ``ACC_REL * |scale| * S`` allows for fp32 accumulation over K in any order;
    ``2^-p |ref|`` is the round-to-nearest cast of the output;
    the smallest subnormal covers results that underflow.
    """
    p = PRECISION[out_fmt]
    return ACC_REL * abs(scale) * np.asarray(S) + 2.0 ** -p * np.abs(ref) + MIN_SUBNORMAL[out_fmt]


def err_over_bound(D_codes, out_fmt, ref, S, scale=1.0):
    """max over elements of |D - ref| / bound (must be <= 1); NaN in D gives inf."""
    d = decode(D_codes, out_fmt)
    e = np.abs(d - ref) / bound(ref, S, out_fmt, scale)
    e = np.where(np.isnan(e), np.inf, e)
    return float(e.max()) if e.size else 0.0
