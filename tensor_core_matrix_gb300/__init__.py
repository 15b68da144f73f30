"""Python binding of libtcm.so, the GB300 (sm_103a) tensor-core GEMM library.

Argument marshalling only: every step of the computation runs in the
library's CUDA kernels.  Functions carry the C ABI's names (``tcm_gemm``,
``tcm_gemm_ex``, ``tcm_sp_compress``, ...) and take torch CUDA tensors, whose
device pointers, shapes and row pitches are passed straight through; torch
supplies device memory and the current stream, nothing else.

There is no fallback: if ``libtcm.so`` is missing or cannot be loaded, every
call raises.  Build it with ``python -m tensor_core_matrix_gb300.build`` (or
``__graft_entry__.build()``).
"""
from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libtcm.so")

TCM_OK = 0
STATUS_NAMES = {0: "TCM_OK", 1: "TCM_ERR_INVALID_ARG", 2: "TCM_ERR_UNSUPPORTED",
                3: "TCM_ERR_MISALIGNED", 4: "TCM_ERR_CUDA", 5: "TCM_ERR_TIMEOUT"}
DTYPE_CODE = {torch.bfloat16: 0, torch.float16: 1, torch.float32: 2,
              torch.float8_e4m3fn: 3, torch.float8_e5m2: 4}
# tcm_activation codes of the fused epilogue
ACT_CODE = {None: 0, "none": 0, "relu": 1, "gelu": 2}
# Symbols the C ABI (include/tcm.h) exports.
EXPORTS = ("tcm_gemm", "tcm_gemm_ex", "tcm_gemm_fused", "tcm_sp_compress", "tcm_sp_meta_tc_bytes",
           "tcm_sp_meta_pack", "tcm_gemm_sp_tc", "tcm_sp_decompress", "tcm_gemm_sp", "tcm_gemm_mx",
           "tcm_mx_scales_bytes", "tcm_mx_pack_scales", "tcm_gemm_nvfp4", "tcm_nvfp4_scales_bytes",
           "tcm_nvfp4_pack_scales",
           "tcm_get_device_status", "tcm_clear_device_status", "tcm_set_timeout_ns",
           "tcm_status_string", "tcm_version", "tcm_set_config_override", "tcm_debug_fail_next_launch",
           "tcm_set_clock_probe", "tcm_gemm_ex_ws", "tcm_gemm_workspace_bytes", "tcm_gemm_ex_builtin_ws",
           "tcm_gemm_i8", "tcm_gemm_i8_workspace_bytes")


class TcmError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {STATUS_NAMES.get(status, status)}")


_lib = None


def load_library(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load libtcm.so and declare its signatures (raises if it is absent)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise ImportError(f"{path} is missing: build the CUDA library first "
                          "(python -m tensor_core_matrix_gb300.build)")
    lib = ctypes.CDLL(path)
    i64, i32, f32, vp = ctypes.c_int64, ctypes.c_int, ctypes.c_float, ctypes.c_void_p
    lib.tcm_gemm.restype = i32
    lib.tcm_gemm.argtypes = [i64, i64, i64, i32, vp, vp, vp, vp, f32, f32, i32, vp]
    lib.tcm_gemm_ex.restype = i32
    lib.tcm_gemm_ex.argtypes = [i64, i64, i64, i32, vp, i64, i32, vp, i64, vp, i64, vp, i64,
                                i32, f32, f32, vp, vp, vp, vp]
    lib.tcm_gemm_ex_ws.restype = i32
    lib.tcm_gemm_ex_ws.argtypes = [i64, i64, i64, i32, vp, i64, i32, vp, i64, vp, i64, vp, i64,
                                   i32, f32, f32, vp, vp, vp, vp, i64, vp]
    lib.tcm_gemm_ex_builtin_ws.restype = i32
    lib.tcm_gemm_ex_builtin_ws.argtypes = [i64, i64, i64, i32, vp, i64, i32, vp, i64, vp, i64, vp, i64,
                                           i32, f32, f32, vp, vp, vp, vp]
    lib.tcm_gemm_i8.restype = i32
    lib.tcm_gemm_i8.argtypes = [i64, i64, i64, vp, i64, vp, i64, vp, i64, vp, i64, vp, i64, vp]
    lib.tcm_gemm_i8_workspace_bytes.restype = i64
    lib.tcm_gemm_i8_workspace_bytes.argtypes = [i64, i64, i64]
    lib.tcm_gemm_workspace_bytes.restype = i64
    lib.tcm_gemm_workspace_bytes.argtypes = [i64, i64, i64, i32, i32]
    lib.tcm_gemm_fused.restype = i32
    lib.tcm_gemm_fused.argtypes = [i64, i64, i64, i32, vp, i64, i32, vp, i64, vp, i64, vp, i64,
                                   i32, f32, f32, vp, vp, vp, i32, vp, vp, vp]
    lib.tcm_sp_compress.restype = i32
    lib.tcm_sp_compress.argtypes = [i64, i64, i32, vp, i64, vp, vp, vp]
    lib.tcm_sp_decompress.restype = i32
    lib.tcm_sp_decompress.argtypes = [i64, i64, i32, vp, vp, vp, i64, vp]
    lib.tcm_gemm_sp.restype = i32
    lib.tcm_gemm_sp.argtypes = [i64, i64, i64, i32, vp, vp, vp, vp, vp, f32, f32, i32, vp]
    lib.tcm_gemm_mx.restype = i32
    lib.tcm_gemm_mx.argtypes = [i64, i64, i64, i32, vp, vp, i32, vp, vp, vp, vp, f32, f32, vp, i32, vp]
    lib.tcm_mx_scales_bytes.restype = i64
    lib.tcm_mx_scales_bytes.argtypes = [i64, i64]
    lib.tcm_mx_pack_scales.restype = i32
    lib.tcm_mx_pack_scales.argtypes = [i64, i64, vp, vp, vp]
    lib.tcm_sp_meta_tc_bytes.restype = i64
    lib.tcm_sp_meta_tc_bytes.argtypes = [i64, i64]
    lib.tcm_sp_meta_pack.restype = i32
    lib.tcm_sp_meta_pack.argtypes = [i64, i64, vp, vp, vp]
    lib.tcm_gemm_sp_tc.restype = i32
    lib.tcm_gemm_sp_tc.argtypes = [i64, i64, i64, i32, vp, vp, vp, vp, vp, f32, f32, i32, vp]
    lib.tcm_gemm_nvfp4.restype = i32
    lib.tcm_gemm_nvfp4.argtypes = [i64, i64, i64, vp, vp, vp, vp, vp, vp, f32, f32, vp, i32, vp]
    lib.tcm_nvfp4_scales_bytes.restype = i64
    lib.tcm_nvfp4_scales_bytes.argtypes = [i64, i64]
    lib.tcm_nvfp4_pack_scales.restype = i32
    lib.tcm_nvfp4_pack_scales.argtypes = [i64, i64, vp, vp, vp]
    lib.tcm_get_device_status.restype = i32
    lib.tcm_get_device_status.argtypes = [vp, ctypes.POINTER(ctypes.c_int32), ctypes.POINTER(ctypes.c_int32)]
    lib.tcm_clear_device_status.restype = i32
    lib.tcm_clear_device_status.argtypes = []
    lib.tcm_set_timeout_ns.restype = None
    lib.tcm_set_timeout_ns.argtypes = [ctypes.c_uint64]
    lib.tcm_set_config_override.restype = None
    lib.tcm_set_config_override.argtypes = [i32, i32, i32, i32, i32, i32]
    lib.tcm_set_clock_probe.restype = None
    lib.tcm_set_clock_probe.argtypes = [vp]
    lib.tcm_debug_fail_next_launch.restype = None
    lib.tcm_debug_fail_next_launch.argtypes = [i32]
    lib.tcm_status_string.restype = ctypes.c_char_p
    lib.tcm_status_string.argtypes = [i32]
    lib.tcm_version.restype = i32
    lib.tcm_version.argtypes = []
    _lib = lib
    return lib


def _check(status: int, what: str):
    if status != TCM_OK:
        raise TcmError(status, what)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


# ------------------------------------------------------------------ argument checks
# Every wrapper checks shapes, dtypes and layouts first and device placement last,
# before anything reaches the library: the C ABI receives raw pointers and pitches
# and cannot tell a host pointer or an undersized buffer from a valid one.

F16_TYPES = (torch.bfloat16, torch.float16)
F8_TYPES = (torch.float8_e4m3fn, torch.float8_e5m2)
OUT_TYPES = (torch.bfloat16, torch.float16, torch.float32)
INDEX_TYPES = tuple(t for t in (torch.int32, getattr(torch, "uint32", None)) if t is not None)


def _mat(t, name, rows=None, cols=None, dtypes=None, contiguous=False):
    """``t`` must be a 2-D tensor of shape (rows, cols) (None: any) with unit column
    stride and a row pitch >= its row length, densely packed if ``contiguous``."""
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch tensor")
    if t.dim() != 2:
        raise ValueError(f"{name} must be 2-D, got shape {tuple(t.shape)}")
    if (rows is not None and t.shape[0] != rows) or (cols is not None and t.shape[1] != cols):
        want = f"{'any' if rows is None else rows} x {'any' if cols is None else cols}"
        raise ValueError(f"{name} must be {want}, got {t.shape[0]} x {t.shape[1]}")
    if dtypes is not None and t.dtype not in dtypes:
        raise ValueError(f"{name}: dtype {t.dtype} not accepted here (expected one of {list(dtypes)})")
    if contiguous:
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous (rows densely packed)")
    elif t.stride(1) != 1 or t.stride(0) < t.shape[1]:
        raise ValueError(f"{name} must have unit column stride and a row pitch >= its row length")
    return t


def _vec(t, name, n, dtypes):
    """``t`` must hold exactly ``n`` contiguous elements of one of ``dtypes``."""
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch tensor")
    if t.numel() != n or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous tensor of {n} elements, got shape {tuple(t.shape)}")
    if t.dtype not in dtypes:
        raise ValueError(f"{name}: dtype {t.dtype} not accepted here (expected one of {list(dtypes)})")
    return t


def _scalar(t, name):
    """``t``: None or a tensor whose first element is the fp32 value the kernel reads."""
    if t is None:
        return None
    if not isinstance(t, torch.Tensor) or t.dtype != torch.float32 or t.numel() < 1 or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous fp32 tensor of at least one element")
    return t


def _bytes(t, name, nbytes):
    """``t`` must be a contiguous uint8 tensor of at least ``nbytes`` bytes."""
    if not isinstance(t, torch.Tensor) or t.dtype != torch.uint8 or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous uint8 tensor")
    if t.numel() < nbytes:
        raise ValueError(f"{name} holds {t.numel()} bytes, {nbytes} needed")
    return t


def _on_device(**named):
    """Every given tensor must live in device memory of the current CUDA device."""
    cur = None
    for name, t in named.items():
        if t is None:
            continue
        if not t.is_cuda:
            raise ValueError(f"{name} must be a CUDA tensor (device memory), got device {t.device}")
        if cur is None:
            cur = torch.cuda.current_device()
        if t.device.index != cur:
            raise ValueError(f"{name} is on {t.device} but the current device is cuda:{cur}")


def _code(t, name):
    try:
        return DTYPE_CODE[t.dtype]
    except KeyError:
        raise ValueError(f"{name}: unsupported dtype {t.dtype}") from None


TCM_E2M1 = 5


def _operand(t, fmt, name):
    """(dtype code, element columns, pitch in elements) of a GEMM operand; fmt="e2m1"
    marks a uint8 tensor of packed FP4 (two elements per byte)."""
    _mat(t, name)
    if fmt == "e2m1":
        if t.dtype != torch.uint8:
            raise ValueError(f"{name}: packed E2M1 operands are uint8 tensors")
        return TCM_E2M1, 2 * t.shape[1], 2 * t.stride(0)
    if fmt is not None:
        raise ValueError(f"{name}: unknown format {fmt!r}")
    if t.dtype not in F16_TYPES + F8_TYPES:
        raise ValueError(f"{name}: unsupported operand dtype {t.dtype}")
    return _code(t, name), t.shape[1], t.stride(0)


def _epilogue_args(D, C, bias, M, N, out_types, bias_types):
    _mat(D, "D", M, N, out_types)
    if C is not None:
        _mat(C, "C", M, N, (D.dtype,))
    if bias is not None:
        _vec(bias, "bias", N, bias_types)


def tcm_gemm_workspace_bytes(M: int, N: int, K: int, a_dtype, b_dtype=None) -> int:
    """Workspace bytes tcm_gemm_ex needs to balance its last round for this problem on the
    current device (0: none); dtypes as torch dtypes or "e2m1"."""
    def code(d):
        return TCM_E2M1 if d == "e2m1" else DTYPE_CODE[d]
    n = int(load_library().tcm_gemm_workspace_bytes(int(M), int(N), int(K), code(a_dtype),
                                                    code(a_dtype if b_dtype is None else b_dtype)))
    if n < 0:
        raise ValueError("unsupported problem")
    return n


def tcm_gemm_ex(A, B, D, *, C=None, alpha=1.0, beta=0.0, a_scale=None, b_scale=None, bias=None, stream=None,
                a_fmt=None, b_fmt=None, workspace=None):
    """D = alpha * a_scale * b_scale * (A @ B_stored.T) + beta * C + bias.

    A: M x K (row-major, pitch = A.stride(0)); B: N x K (K-major storage of
    the K x N operand); C, D: M x N (C of D's dtype); bias: N elements of D's
    dtype; a_scale, b_scale: one-element fp32 CUDA tensors or None.
    a_fmt / b_fmt = "e2m1": that operand is a uint8 tensor of packed FP4
    (M x K/2 or N x K/2 bytes).  workspace: a contiguous uint8 CUDA tensor of at
    least tcm_gemm_workspace_bytes(...) bytes, or None (then the C ABI's
    tcm_gemm_ex; with it, tcm_gemm_ex_ws).
    """
    ca, K, lda = _operand(A, a_fmt, "A")
    cb, Kb, ldb = _operand(B, b_fmt, "B")
    M, N = A.shape[0], B.shape[0]
    if Kb != K:
        raise ValueError(f"A has K = {K}, B has K = {Kb}")
    _epilogue_args(D, C, bias, M, N, OUT_TYPES, (D.dtype,))
    _scalar(a_scale, "a_scale"), _scalar(b_scale, "b_scale")
    if workspace is not None:
        _bytes(workspace, "workspace", 0)
    _on_device(A=A, B=B, D=D, C=C, bias=bias, a_scale=a_scale, b_scale=b_scale, workspace=workspace)
    lib = load_library()
    args = (M, N, K, ca, _ptr(A), lda, cb, _ptr(B), ldb, _ptr(C), C.stride(0) if C is not None else 0,
            _ptr(D), D.stride(0), _code(D, "D"), float(alpha), float(beta),
            _ptr(a_scale), _ptr(b_scale), _ptr(bias))
    if workspace is None:
        _check(lib.tcm_gemm_ex(*args, _stream(stream)), "tcm_gemm_ex")
    else:
        _check(lib.tcm_gemm_ex_ws(*args, _ptr(workspace), workspace.numel(), _stream(stream)), "tcm_gemm_ex_ws")
    return D


def tcm_gemm_fused(A, B, D, *, C=None, alpha=1.0, beta=0.0, a_scale=None, b_scale=None, bias=None,
                   act=None, d_scale=None, amax=None, stream=None, a_fmt=None, b_fmt=None):
    """y = act(alpha * a_scale * b_scale * (A @ B_stored.T) + beta * C + bias); D = y / d_scale in D's
    dtype (FP8 outputs saturate); amax (one-element fp32 CUDA tensor or None) receives max |y|.

    act: None/"none", "relu" or "gelu"; d_scale: one-element fp32 CUDA tensor or None (FP8 D only);
    bias: N elements, bf16 for an FP8 D, else D's dtype.
    """
    ca, K, lda = _operand(A, a_fmt, "A")
    cb, Kb, ldb = _operand(B, b_fmt, "B")
    M, N = A.shape[0], B.shape[0]
    if Kb != K:
        raise ValueError(f"A has K = {K}, B has K = {Kb}")
    if act not in ACT_CODE:
        raise ValueError(f"unknown activation {act!r}")
    out8 = D.dtype in F8_TYPES
    _epilogue_args(D, C, bias, M, N, OUT_TYPES + F8_TYPES, (torch.bfloat16,) if out8 else (D.dtype,))
    for name, t in (("a_scale", a_scale), ("b_scale", b_scale), ("d_scale", d_scale), ("amax", amax)):
        _scalar(t, name)
    _on_device(A=A, B=B, D=D, C=C, bias=bias, a_scale=a_scale, b_scale=b_scale, d_scale=d_scale, amax=amax)
    lib = load_library()
    st = lib.tcm_gemm_fused(M, N, K, ca, _ptr(A), lda, cb, _ptr(B),
                            ldb, _ptr(C), C.stride(0) if C is not None else 0,
                            _ptr(D), D.stride(0), _code(D, "D"), float(alpha), float(beta),
                            _ptr(a_scale), _ptr(b_scale), _ptr(bias), ACT_CODE[act], _ptr(d_scale), _ptr(amax),
                            _stream(stream))
    _check(st, "tcm_gemm_fused")
    return D


def tcm_gemm(A, B, D, *, C=None, alpha=1.0, beta=0.0, stream=None):
    """D = alpha * (A @ B_stored.T) + beta * C for bf16/fp16 A, B; all densely packed."""
    _mat(A, "A", dtypes=F16_TYPES, contiguous=True)
    M, K = A.shape
    N = B.shape[0] if isinstance(B, torch.Tensor) and B.dim() == 2 else None
    _mat(B, "B", N, K, (A.dtype,), contiguous=True)
    _mat(D, "D", M, N, OUT_TYPES, contiguous=True)
    if C is not None:
        _mat(C, "C", M, N, (D.dtype,), contiguous=True)
    _on_device(A=A, B=B, D=D, C=C)
    lib = load_library()
    st = lib.tcm_gemm(M, N, K, _code(A, "A"), _ptr(A), _ptr(B), _ptr(C), _ptr(D), float(alpha),
                      float(beta), _code(D, "D"), _stream(stream))
    _check(st, "tcm_gemm")
    return D


def tcm_gemm_i8_workspace_bytes(M: int, N: int, K: int) -> int:
    """Workspace bytes of tcm_gemm_i8 (the bf16 copies of A and B); -1 if the sizes are rejected."""
    return int(load_library().tcm_gemm_i8_workspace_bytes(int(M), int(N), int(K)))


def tcm_gemm_i8(A, B, D, *, C=None, workspace=None, stream=None):
    """D = satfinite_int32(A @ B_stored.T + C), exact: A int8 (M x K), B int8 (N x K), C and D
    int32 (M x N).  workspace: a contiguous uint8 CUDA tensor of tcm_gemm_i8_workspace_bytes
    bytes, allocated here if None."""
    _mat(A, "A", dtypes=(torch.int8,))
    M, K = A.shape
    _mat(B, "B", None, K, (torch.int8,))
    N = B.shape[0]
    _mat(D, "D", M, N, (torch.int32,))
    if C is not None:
        _mat(C, "C", M, N, (torch.int32,))
    nbytes = tcm_gemm_i8_workspace_bytes(M, N, K)
    if nbytes < 0:
        raise ValueError(f"unsupported sizes {M} x {N} x {K}")
    if workspace is not None:
        _bytes(workspace, "workspace", nbytes)
    _on_device(A=A, B=B, D=D, C=C, workspace=workspace)
    if workspace is None:
        workspace = torch.empty(max(nbytes, 16), dtype=torch.uint8, device=A.device)
    lib = load_library()
    st = lib.tcm_gemm_i8(M, N, K, _ptr(A), A.stride(0), _ptr(B), B.stride(0), _ptr(C),
                         C.stride(0) if C is not None else 0, _ptr(D), D.stride(0), _ptr(workspace),
                         workspace.numel(), _stream(stream))
    _check(st, "tcm_gemm_i8")
    return D


def tcm_sp_compress(A, A_comp=None, meta=None, *, stream=None):
    """2:4 prune + compress of logical A (M x K, K % 32 == 0) -> (A_comp M x K/2, meta M x K/32 int32)."""
    _mat(A, "A", dtypes=F16_TYPES)
    M, K = A.shape
    if K % 32:
        raise ValueError(f"K = {K} must be a multiple of 32")
    if A_comp is not None:
        _mat(A_comp, "A_comp", M, K // 2, (A.dtype,), contiguous=True)
    if meta is not None:
        _mat(meta, "meta", M, K // 32, INDEX_TYPES, contiguous=True)
    _on_device(A=A, A_comp=A_comp, meta=meta)
    if A_comp is None:
        A_comp = torch.empty((M, K // 2), dtype=A.dtype, device=A.device)
    if meta is None:
        meta = torch.empty((M, K // 32), dtype=torch.int32, device=A.device)
    lib = load_library()
    st = lib.tcm_sp_compress(M, K, _code(A, "A"), _ptr(A), A.stride(0), _ptr(A_comp), _ptr(meta),
                             _stream(stream))
    _check(st, "tcm_sp_compress")
    return A_comp, meta


def tcm_sp_decompress(A_comp, meta, A=None, *, stream=None):
    """Logical M x K matrix from (A_comp, meta) with zeros at the dropped positions."""
    _mat(A_comp, "A_comp", dtypes=F16_TYPES, contiguous=True)
    M, Kh = A_comp.shape
    K = 2 * Kh
    if K % 32:
        raise ValueError(f"K = {K} must be a multiple of 32")
    _mat(meta, "meta", M, K // 32, INDEX_TYPES, contiguous=True)
    if A is not None:
        _mat(A, "A", M, K, (A_comp.dtype,))
    _on_device(A_comp=A_comp, meta=meta, A=A)
    if A is None:
        A = torch.empty((M, K), dtype=A_comp.dtype, device=A_comp.device)
    lib = load_library()
    st = lib.tcm_sp_decompress(M, K, _code(A_comp, "A_comp"), _ptr(A_comp), _ptr(meta), _ptr(A),
                               A.stride(0), _stream(stream))
    _check(st, "tcm_sp_decompress")
    return A


def tcm_gemm_sp(A_comp, meta, B, D, *, C=None, alpha=1.0, beta=0.0, stream=None):
    """D = alpha * (A' @ B_stored.T) + beta * C, A' the 2:4 matrix held by (A_comp, meta)
    (A_comp M x K/2, meta M x K/32 int32, B N x K, C and D M x N; all densely packed)."""
    _mat(A_comp, "A_comp", dtypes=F16_TYPES, contiguous=True)
    M, Kh = A_comp.shape
    K = 2 * Kh
    if K % 32:
        raise ValueError(f"K = {K} must be a multiple of 32")
    _mat(meta, "meta", M, K // 32, INDEX_TYPES, contiguous=True)
    _mat(B, "B", None, K, (A_comp.dtype,), contiguous=True)
    N = B.shape[0]
    _mat(D, "D", M, N, OUT_TYPES, contiguous=True)
    if C is not None:
        _mat(C, "C", M, N, (D.dtype,), contiguous=True)
    _on_device(A_comp=A_comp, meta=meta, B=B, D=D, C=C)
    lib = load_library()
    st = lib.tcm_gemm_sp(M, N, K, _code(A_comp, "A_comp"), _ptr(A_comp), _ptr(meta), _ptr(B), _ptr(C),
                         _ptr(D), float(alpha), float(beta), _code(D, "D"), _stream(stream))
    _check(st, "tcm_gemm_sp")
    return D


def tcm_mx_scales_bytes(rows: int, K: int) -> int:
    """Bytes of the blocked scale array of `rows` rows of K elements (-1 if K % 32 != 0)."""
    return int(load_library().tcm_mx_scales_bytes(int(rows), int(K)))


def tcm_mx_pack_scales(scales, K: int, packed=None, stream=None):
    """Blocked layout of row-major E8M0 codes `scales` (rows x K/32 uint8, CUDA);
    allocates `packed` (uint8, tcm_mx_scales_bytes(rows, K) bytes) if not given."""
    if K % 32:
        raise ValueError(f"K = {K} must be a multiple of 32")
    _mat(scales, "scales", None, K // 32, (torch.uint8,), contiguous=True)
    rows = scales.shape[0]
    nbytes = max(tcm_mx_scales_bytes(rows, K), 0)
    if packed is not None:
        _bytes(packed, "packed", nbytes)
    _on_device(scales=scales, packed=packed)
    if packed is None:
        packed = torch.empty(nbytes, dtype=torch.uint8, device=scales.device)
    lib = load_library()
    _check(lib.tcm_mx_pack_scales(rows, K, _ptr(scales), _ptr(packed), _stream(stream)), "tcm_mx_pack_scales")
    return packed


def tcm_gemm_mx(A, a_scales, B, b_scales, D, *, C=None, alpha=1.0, beta=0.0, bias=None, stream=None, fmt=None):
    """Block-scaled MX GEMM: A (M x K) and B (N x K) in E4M3/E5M2 (MXFP8), or, with
    fmt="e2m1", packed E2M1 uint8 tensors of K/2 bytes per row (MXFP4); a_scales and
    b_scales the blocked E8M0 arrays of tcm_mx_pack_scales; D (M x N), C of D's
    dtype, bias N elements of D's dtype; all contiguous CUDA tensors."""
    if fmt not in (None, "e2m1"):
        raise ValueError(f"unknown format {fmt!r}")
    el = (torch.uint8,) if fmt == "e2m1" else F8_TYPES
    _mat(A, "A", dtypes=el, contiguous=True)
    M, K = A.shape[0], A.shape[1] * (2 if fmt == "e2m1" else 1)
    _mat(B, "B", None, A.shape[1], el, contiguous=True)
    N = B.shape[0]
    _bytes(a_scales, "a_scales", tcm_mx_scales_bytes(M, K))
    _bytes(b_scales, "b_scales", tcm_mx_scales_bytes(N, K))
    _epilogue_args(D, C, bias, M, N, OUT_TYPES, (D.dtype,))
    if not D.is_contiguous() or (C is not None and not C.is_contiguous()):
        raise ValueError("C and D must be contiguous")
    _on_device(A=A, a_scales=a_scales, B=B, b_scales=b_scales, D=D, C=C, bias=bias)
    lib = load_library()
    ca, cb = (TCM_E2M1, TCM_E2M1) if fmt == "e2m1" else (_code(A, "A"), _code(B, "B"))
    st = lib.tcm_gemm_mx(M, N, K, ca, _ptr(A), _ptr(a_scales), cb, _ptr(B), _ptr(b_scales),
                         _ptr(C), _ptr(D), float(alpha), float(beta), _ptr(bias), _code(D, "D"), _stream(stream))
    _check(st, "tcm_gemm_mx")
    return D


def tcm_sp_meta_tc_bytes(M: int, K: int) -> int:
    """Bytes of the hardware-ordered 2:4 metadata of an M x K (logical) matrix."""
    return int(load_library().tcm_sp_meta_tc_bytes(int(M), int(K)))


def tcm_sp_meta_pack(meta, K: int, meta_tc=None, stream=None):
    """Hardware-ordered copy of canonical metadata `meta` (M x K/32 int32/uint32, CUDA)."""
    if K % 32:
        raise ValueError(f"K = {K} must be a multiple of 32")
    _mat(meta, "meta", None, K // 32, INDEX_TYPES, contiguous=True)
    M = meta.shape[0]
    nbytes = max(tcm_sp_meta_tc_bytes(M, K), 0)
    if meta_tc is not None:
        _bytes(meta_tc, "meta_tc", nbytes)
    _on_device(meta=meta, meta_tc=meta_tc)
    if meta_tc is None:
        meta_tc = torch.empty(nbytes, dtype=torch.uint8, device=meta.device)
    lib = load_library()
    _check(lib.tcm_sp_meta_pack(M, K, _ptr(meta), _ptr(meta_tc), _stream(stream)), "tcm_sp_meta_pack")
    return meta_tc


def tcm_gemm_sp_tc(A_comp, meta_tc, B, D, *, C=None, alpha=1.0, beta=0.0, stream=None):
    """tcm_gemm_sp with hardware-ordered metadata (tcm_sp_meta_pack); A_comp M x K/2, B N x K."""
    _mat(A_comp, "A_comp", dtypes=F16_TYPES, contiguous=True)
    _mat(B, "B", dtypes=(A_comp.dtype,), contiguous=True)
    M, K, N = A_comp.shape[0], B.shape[1], B.shape[0]
    if A_comp.shape[1] * 2 != K or K % 32:
        raise ValueError(f"A_comp holds K/2 = {A_comp.shape[1]} columns but B has K = {K} (a multiple of 32)")
    _bytes(meta_tc, "meta_tc", tcm_sp_meta_tc_bytes(M, K))
    _mat(D, "D", M, N, OUT_TYPES, contiguous=True)
    if C is not None:
        _mat(C, "C", M, N, (D.dtype,), contiguous=True)
    _on_device(A_comp=A_comp, meta_tc=meta_tc, B=B, D=D, C=C)
    lib = load_library()
    st = lib.tcm_gemm_sp_tc(M, N, K, _code(A_comp, "A_comp"), _ptr(A_comp), _ptr(meta_tc), _ptr(B), _ptr(C), _ptr(D),
                            float(alpha), float(beta), _code(D, "D"), _stream(stream))
    _check(st, "tcm_gemm_sp_tc")
    return D


def tcm_nvfp4_scales_bytes(rows: int, K: int) -> int:
    """Bytes of the blocked NVFP4 scale array of `rows` rows of K elements (-1 if K % 16 != 0)."""
    return int(load_library().tcm_nvfp4_scales_bytes(int(rows), int(K)))


def tcm_nvfp4_pack_scales(scales, K: int, packed=None, stream=None):
    """Blocked layout of row-major UE4M3 codes `scales` (rows x K/16 uint8, CUDA)."""
    if K % 16:
        raise ValueError(f"K = {K} must be a multiple of 16")
    _mat(scales, "scales", None, K // 16, (torch.uint8,), contiguous=True)
    rows = scales.shape[0]
    nbytes = max(tcm_nvfp4_scales_bytes(rows, K), 0)
    if packed is not None:
        _bytes(packed, "packed", nbytes)
    _on_device(scales=scales, packed=packed)
    if packed is None:
        packed = torch.empty(nbytes, dtype=torch.uint8, device=scales.device)
    lib = load_library()
    _check(lib.tcm_nvfp4_pack_scales(rows, K, _ptr(scales), _ptr(packed), _stream(stream)), "tcm_nvfp4_pack_scales")
    return packed


def tcm_gemm_nvfp4(A, a_scales, B, b_scales, D, *, C=None, alpha=1.0, beta=0.0, bias=None, stream=None):
    """NVFP4 GEMM: A (M x K/2 bytes) and B (N x K/2 bytes) packed E2M1, a_scales / b_scales the
    blocked UE4M3 arrays of tcm_nvfp4_pack_scales, D (M x N), C of D's dtype, bias N elements of
    D's dtype; alpha = product of the per-tensor scales.  All contiguous CUDA tensors."""
    _mat(A, "A", dtypes=(torch.uint8,), contiguous=True)
    M, K = A.shape[0], 2 * A.shape[1]
    _mat(B, "B", None, K // 2, (torch.uint8,), contiguous=True)
    N = B.shape[0]
    _bytes(a_scales, "a_scales", tcm_nvfp4_scales_bytes(M, K))
    _bytes(b_scales, "b_scales", tcm_nvfp4_scales_bytes(N, K))
    _epilogue_args(D, C, bias, M, N, OUT_TYPES, (D.dtype,))
    if not D.is_contiguous() or (C is not None and not C.is_contiguous()):
        raise ValueError("C and D must be contiguous")
    _on_device(A=A, a_scales=a_scales, B=B, b_scales=b_scales, D=D, C=C, bias=bias)
    lib = load_library()
    st = lib.tcm_gemm_nvfp4(M, N, K, _ptr(A), _ptr(a_scales), _ptr(B), _ptr(b_scales), _ptr(C), _ptr(D),
                            float(alpha), float(beta), _ptr(bias), _code(D, "D"), _stream(stream))
    _check(st, "tcm_gemm_nvfp4")
    return D


def tcm_get_device_status(stream=None):
    """Synchronise the stream and return (code, site) of the first recorded device failure."""
    lib = load_library()
    code, site = ctypes.c_int32(0), ctypes.c_int32(0)
    _check(lib.tcm_get_device_status(_stream(stream), ctypes.byref(code), ctypes.byref(site)),
           "tcm_get_device_status")
    return code.value, site.value


def tcm_clear_device_status():
    _check(load_library().tcm_clear_device_status(), "tcm_clear_device_status")


def tcm_set_timeout_ns(ns: int):
    load_library().tcm_set_timeout_ns(int(ns))


def tcm_set_config_override(cta_group: int = 0, tile_n: int = 0, stages: int = 0, group_m: int = 0,
                            ksplit: int = 0, tail_split: int = 0):
    """Force kernel-variant fields of later GEMMs (see include/tcm.h); zeros restore the automatic choice."""
    load_library().tcm_set_config_override(int(cta_group), int(tile_n), int(stages), int(group_m), int(ksplit),
                                           int(tail_split))


def tcm_set_clock_probe(counters=None):
    """Measurement hook: later GEMM launches add their first CTA's SM cycles, global-timer ns and 1
    to ``counters`` (a CUDA int64 tensor of >= 3 elements); None turns it off."""
    if counters is not None:
        if counters.dtype != torch.int64 or counters.numel() < 3 or not counters.is_contiguous():
            raise ValueError("counters must be a contiguous int64 tensor of at least 3 elements")
        _on_device(counters=counters)
    load_library().tcm_set_clock_probe(_ptr(counters))


def tcm_debug_fail_next_launch(mask: int = 1):
    """Test hook: bit 1 -- the next GEMM launch skips its first load and times out; bit 2 -- the
    next split tcm_gemm_ex_ws launch's helper parts never announce their partials (see include/tcm.h)."""
    load_library().tcm_debug_fail_next_launch(int(mask))


def tcm_status_string(status: int) -> str:
    return load_library().tcm_status_string(int(status)).decode()


def tcm_version() -> int:
    return load_library().tcm_version()
