"""Pins of the CPU oracle against facts that do not come from the oracle itself.

Each test checks the oracle against one of: the published format definitions
(closed-form special values), an independent decoder (numpy / torch casts),
an exact rational brute force, numpy's fp64 matmul, closed forms (identity,
permutation, rank-1, beta-only, bias-only), integer-exact products, and the
pages' worked 2:4 example.  A dropped term, a wrong sign, a transposed B or a
wrong tie rule in the oracle fails at least one of them.
"""
import itertools
import json
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
import synth_inputs as si

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ---------------------------------------------------------------- decoders

def _all_codes(bits):
    return np.arange(1 << bits, dtype={8: np.uint8, 16: np.uint16}[bits])


def _same(a, b):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    return np.array_equal(np.isnan(a), np.isnan(b)) and np.array_equal(
        np.nan_to_num(a, nan=0.0), np.nan_to_num(b, nan=0.0)) and np.array_equal(
        np.signbit(a[~np.isnan(a)]), np.signbit(b[~np.isnan(b)]))


def test_decode_bf16_exhaustive_matches_torch():
    c = _all_codes(16)
    ours = oracle.decode(c, "bf16")
    theirs = torch.from_numpy(c.view(np.int16).copy()).view(torch.bfloat16).to(torch.float64).numpy()
    assert _same(ours, theirs)


def test_decode_f16_exhaustive_matches_numpy():
    c = _all_codes(16)
    ours = oracle.decode(c, "f16")
    theirs = c.view(np.float16).astype(np.float64)
    assert _same(ours, theirs)


@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
def test_decode_fp8_exhaustive_matches_torch(fmt):
    c = _all_codes(8)
    ours = oracle.decode(c, fmt)
    theirs = torch.from_numpy(c.copy()).view(si.TORCH_DTYPE[fmt]).to(torch.float64).numpy()
    assert _same(ours, theirs)


def test_decode_f32_roundtrip():
    g = np.random.default_rng(5)
    v = g.standard_normal(1000).astype(np.float32)
    assert np.array_equal(oracle.decode(v.view(np.uint32), "f32"), v.astype(np.float64))


@pytest.mark.parametrize("fmt,code,value", [
    # closed forms from the format definitions
    ("bf16", 0x3F80, 1.0), ("bf16", 0xC000, -2.0), ("bf16", 0x0001, 2.0 ** -133),
    ("bf16", 0x7F7F, (2 - 2.0 ** -7) * 2.0 ** 127), ("bf16", 0x7F80, np.inf),
    ("f16", 0x3C00, 1.0), ("f16", 0x0001, 2.0 ** -24), ("f16", 0x7BFF, 65504.0),
    ("f16", 0x0400, 2.0 ** -14), ("f16", 0xFC00, -np.inf),
    ("e4m3", 0x7E, 448.0), ("e4m3", 0x01, 2.0 ** -9), ("e4m3", 0x08, 2.0 ** -6),
    ("e4m3", 0x78, 256.0), ("e4m3", 0x38, 1.0), ("e4m3", 0xB8, -1.0), ("e4m3", 0x7F, np.nan),
    ("e5m2", 0x7B, 57344.0), ("e5m2", 0x7C, np.inf), ("e5m2", 0x01, 2.0 ** -16),
    ("e5m2", 0x3C, 1.0), ("e5m2", 0x7D, np.nan), ("e5m2", 0x04, 2.0 ** -14),
])
def test_decode_closed_forms(fmt, code, value):
    width = np.uint8 if fmt in ("e4m3", "e5m2") else np.uint16
    got = oracle.decode(np.array([code], dtype=width), fmt)[0]
    if np.isnan(value):
        assert np.isnan(got)
    else:
        assert got == value


# ---------------------------------------------------------------- GEMM

def _rand_codes(shape, fmt, seed, kind="normal"):
    g = si.generator(seed)
    if kind == "normal":
        t = si.normal(shape, g, dtype=fmt)
    elif kind == "int":
        t = si.integers(shape, g, dtype=fmt)
    else:
        t = si.uniform(shape, g, dtype=fmt)
    return si.codes(t)


def test_single_tile_m16n8k16_exact_bruteforce():
    """One 16x8x16 tile (the m16n8k16 MMA shape) against exact rationals."""
    spec = json.load(open(os.path.join(GOLDEN, "m16n8k16_tile.json")))
    M, N, K = spec["M"], spec["N"], spec["K"]
    A = _rand_codes((M, K), "bf16", 11)
    B = _rand_codes((N, K), "bf16", 12)
    C = _rand_codes((M, N), "f32", 13, kind="uniform")
    ref, S = oracle.gemm(A, B, "bf16", "bf16", C=C, c_fmt="f32", alpha=1.0, beta=1.0)
    a = torch.from_numpy(A.view(np.int16).copy()).view(torch.bfloat16).float().tolist()
    b = torch.from_numpy(B.view(np.int16).copy()).view(torch.bfloat16).float().tolist()
    c = C.view(np.float32).tolist()
    positions = 0
    for m in range(M):
        for n in range(N):
            exact = sum(Fraction(a[m][k]) * Fraction(b[n][k]) for k in range(K)) + Fraction(c[m][n])
            sabs = sum(abs(Fraction(a[m][k]) * Fraction(b[n][k])) for k in range(K))
            positions += K
            assert abs(Fraction(ref[m, n]) - exact) <= Fraction(2.0 ** -50) * (sabs + abs(Fraction(c[m][n])))
            assert abs(Fraction(S[m, n]) - sabs) <= Fraction(2.0 ** -50) * sabs
    assert positions == spec["multiply_add_positions"]
    # all-ones tile: every output counts exactly K multiply-adds
    ones_a = si.codes(torch.ones((M, K), dtype=torch.bfloat16))
    ones_b = si.codes(torch.ones((N, K), dtype=torch.bfloat16))
    r1, _ = oracle.gemm(ones_a, ones_b, "bf16", "bf16")
    assert r1.sum() == spec["multiply_add_positions"]


@pytest.mark.parametrize("M,N,K,fa,fb", [
    (37, 53, 71, "bf16", "bf16"), (128, 96, 256, "f16", "f16"), (256, 256, 256, "bf16", "bf16"),
    (64, 40, 96, "e4m3", "e5m2"), (33, 17, 128, "e5m2", "e4m3"),
])
def test_gemm_matches_numpy_fp64(M, N, K, fa, fb):
    A = _rand_codes((M, K), fa, 21) if fa in ("bf16", "f16") else si.codes(
        si.fp8_per_tensor(torch.randn((M, K), generator=si.generator(21)), fa)[0])
    B = _rand_codes((N, K), fb, 22) if fb in ("bf16", "f16") else si.codes(
        si.fp8_per_tensor(torch.randn((N, K), generator=si.generator(22)), fb)[0])
    ref, S = oracle.gemm(A, B, fa, fb)
    Ad = oracle.decode(A, fa)
    Bd = oracle.decode(B, fb)
    np_ref = Ad @ Bd.T
    assert np.all(np.abs(ref - np_ref) <= 1e-12 * S + 1e-300)
    assert np.allclose(S, np.abs(Ad) @ np.abs(Bd).T, rtol=1e-12, atol=0)


def test_identity_pins_k_major_b():
    """A = I gives D[m, n] = B_stored[n, m]: pins B stored as N rows of K."""
    K = 48
    N = 40
    A = si.codes(torch.eye(K, dtype=torch.bfloat16))
    B = _rand_codes((N, K), "bf16", 31)
    ref, _ = oracle.gemm(A, B, "bf16", "bf16")
    Bd = oracle.decode(B, "bf16")
    assert np.array_equal(ref, Bd.T)
    assert not np.array_equal(ref[:N, :N], Bd[:, :N]) or np.array_equal(Bd[:, :N], Bd[:, :N].T)


def test_permutation_rows():
    K, N = 32, 24
    perm = np.random.default_rng(7).permutation(K)
    P = torch.zeros((K, K), dtype=torch.bfloat16)
    P[torch.arange(K), torch.from_numpy(perm)] = 1.0
    B = _rand_codes((N, K), "bf16", 32)
    ref, _ = oracle.gemm(si.codes(P), B, "bf16", "bf16")
    Bd = oracle.decode(B, "bf16")
    assert np.array_equal(ref, Bd.T[perm, :])


def test_rank1_closed_form_with_scales():
    """a[m,k] = u_m, b[n,k] = v_n (powers of two): D = alpha*sa*sb*K*u_m*v_n exactly."""
    M, N, K = 12, 10, 96
    g = np.random.default_rng(3)
    u = 2.0 ** g.integers(-4, 4, M) * g.choice([-1, 1], M)
    v = 2.0 ** g.integers(-4, 4, N) * g.choice([-1, 1], N)
    A = si.codes(torch.tensor(np.repeat(u[:, None], K, 1), dtype=torch.bfloat16))
    B = si.codes(torch.tensor(np.repeat(v[:, None], K, 1), dtype=torch.bfloat16))
    ref, S = oracle.gemm(A, B, "bf16", "bf16", alpha=0.5, sa=4.0, sb=0.125)
    expect = 0.5 * 4.0 * 0.125 * K * np.outer(u, v)
    assert np.array_equal(ref, expect)
    assert np.array_equal(S, K * np.abs(np.outer(u, v)))


def test_beta_only_and_bias_only():
    M, N, K = 9, 14, 16
    zA = si.codes(torch.zeros((M, K), dtype=torch.bfloat16))
    B = _rand_codes((N, K), "bf16", 41)
    C = _rand_codes((M, N), "f32", 42, kind="uniform")
    ref, S = oracle.gemm(zA, B, "bf16", "bf16", C=C, c_fmt="f32", alpha=3.0, beta=-0.75)
    assert np.array_equal(ref, -0.75 * C.view(np.float32).astype(np.float64))
    assert np.all(S == 0)
    bias = _rand_codes((N,), "bf16", 43)
    ref2, _ = oracle.gemm(zA, B, "bf16", "bf16", bias=bias, bias_fmt="bf16")
    assert np.array_equal(ref2, np.broadcast_to(oracle.decode(bias, "bf16"), (M, N)))
    # the sign of beta and the C term must enter, and the bias must add (not replace)
    ref3, _ = oracle.gemm(zA, B, "bf16", "bf16", C=C, c_fmt="f32", beta=1.0, bias=bias)
    assert np.array_equal(ref3, C.view(np.float32).astype(np.float64) + oracle.decode(bias, "bf16")[None, :])


@pytest.mark.parametrize("fa,fb", [("bf16", "bf16"), ("f16", "f16"), ("e4m3", "e4m3"), ("e4m3", "e5m2")])
def test_integer_inputs_exact(fa, fb):
    M, N, K = 40, 24, 200
    A = _rand_codes((M, K), fa, 51, kind="int")
    B = _rand_codes((N, K), fb, 52, kind="int")
    ref, _ = oracle.gemm(A, B, fa, fb)
    ai = oracle.decode(A, fa).astype(np.int64)
    bi = oracle.decode(B, fb).astype(np.int64)
    assert np.array_equal(ref, (ai @ bi.T).astype(np.float64))


def test_leading_dimension_padding_ignored():
    M, N, K, pad = 20, 12, 64, 16
    A = _rand_codes((M, K + pad), "bf16", 61)
    B = _rand_codes((N, K + pad), "bf16", 62)
    ref, _ = oracle.gemm(A, B, "bf16", "bf16", K=K)
    ref2, _ = oracle.gemm(np.ascontiguousarray(A[:, :K]), np.ascontiguousarray(B[:, :K]), "bf16", "bf16")
    assert np.array_equal(ref, ref2)


def test_sampled_equals_full():
    M, N, K = 70, 50, 64
    A = _rand_codes((M, K), "bf16", 71)
    B = _rand_codes((N, K), "bf16", 72)
    C = _rand_codes((M, N), "f32", 73, kind="uniform")
    full, Sf = oracle.gemm(A, B, "bf16", "bf16", C=C, beta=0.5)
    g = np.random.default_rng(0)
    r = g.integers(0, M, 300)
    c = g.integers(0, N, 300)
    samp, Ss = oracle.gemm(A, B, "bf16", "bf16", C=C, beta=0.5, rows=r, cols=c)
    assert np.array_equal(samp, full[r, c]) and np.array_equal(Ss, Sf[r, c])


def test_bad_arguments_rejected():
    A = _rand_codes((4, 32), "bf16", 1)
    with pytest.raises(ValueError):
        oracle.gemm(A, A, "bf16", "bf16", rows=[0, 9], cols=[0, 0])
    with pytest.raises(ValueError):
        oracle.sp_compress(_rand_codes((4, 24), "bf16", 1), "bf16")


# ---------------------------------------------------------------- tolerance

def test_bound_accepts_exact_and_rejects_outside():
    ref = np.array([1.0, -3.0, 1e-3])
    S = np.array([10.0, 20.0, 0.0])
    b = oracle.bound(ref, S, "bf16")
    exact = si.codes(torch.tensor(ref, dtype=torch.bfloat16))
    assert oracle.err_over_bound(exact, "bf16", ref, S) <= 1.0
    far = si.codes(torch.tensor(ref + 2.5 * b, dtype=torch.float32))
    assert oracle.err_over_bound(far, "f32", ref, S) > 1.0
    nan = si.codes(torch.tensor([np.nan, 0, 0], dtype=torch.float32))
    assert oracle.err_over_bound(nan, "f32", ref, S) == np.inf


# ---------------------------------------------------------------- 2:4 sparsity

def _bf16_codes(vals):
    return si.codes(torch.tensor(vals, dtype=torch.bfloat16))


def test_sparse_worked_example_from_page():
    spec = json.load(open(os.path.join(GOLDEN, "sp24_worked_example.json")))
    for case in spec["cases"]:
        logical = case["logical"] * 8  # K = 32: the example repeated over 8 groups
        Ac, meta = oracle.sp_compress(_bf16_codes([logical]), "bf16")
        assert oracle.decode(Ac, "bf16")[0, :2].tolist() == case["values"]
        i0, i1 = case["positions"]
        assert meta[0, 0] == sum((i0 | (i1 << 2)) << (4 * g) for g in range(8))
        back = oracle.sp_decompress(Ac, meta, "bf16")
        assert oracle.decode(back, "bf16")[0].tolist() == logical


def _brute_keep(vals):
    """Top two positions by (|v| descending, index ascending), returned ascending."""
    order = sorted(range(4), key=lambda q: (-abs(vals[q]), q))
    return sorted(order[:2])


def test_sparse_selection_exhaustive_small_alphabet():
    alphabet = [0.0, -0.0, 1.0, -1.0, 2.0, -2.0]
    groups = list(itertools.product(alphabet, repeat=4))
    while len(groups) % 8:
        groups.append((0.0, 0.0, 0.0, 0.0))
    row = [v for grp in groups for v in grp]
    Ac, meta = oracle.sp_compress(_bf16_codes([row]), "bf16")
    vals = oracle.decode(Ac, "bf16")[0]
    for g, grp in enumerate(groups):
        nib = (int(meta[0, g // 8]) >> (4 * (g % 8))) & 0xF
        i0, i1 = nib & 3, nib >> 2
        assert [i0, i1] == _brute_keep(grp), (grp, i0, i1)
        assert i0 < i1
        assert vals[2 * g] == grp[i0] and vals[2 * g + 1] == grp[i1]


def test_sparse_roundtrip_random():
    M, K = 64, 256
    A = _rand_codes((M, K), "bf16", 81)
    Ac, meta = oracle.sp_compress(A, "bf16")
    Ap = oracle.sp_decompress(Ac, meta, "bf16")
    # every group of the pruned matrix keeps exactly the brute-force pair
    Ad = oracle.decode(A, "bf16")
    Apd = oracle.decode(Ap, "bf16")
    for m in range(0, M, 7):
        for g in range(K // 4):
            keep = _brute_keep(Ad[m, 4 * g:4 * g + 4].tolist())
            for q in range(4):
                want = Ad[m, 4 * g + q] if q in keep else 0.0
                assert Apd[m, 4 * g + q] == want
    # compress of an already-pruned matrix reproduces values and metadata
    Ac2, meta2 = oracle.sp_compress(Ap, "bf16")
    assert np.array_equal(Ac2, Ac) and np.array_equal(meta2, meta)


def test_sparse_gemm_from_compressed_definition():
    """D = sum over kept values only (compressed form) == dense GEMM of decompressed A."""
    M, N, K = 6, 5, 64
    A = _rand_codes((M, K), "bf16", 91)
    B = _rand_codes((N, K), "bf16", 92)
    Ac, meta = oracle.sp_compress(A, "bf16")
    ref, _ = oracle.gemm(oracle.sp_decompress(Ac, meta, "bf16"), B, "bf16", "bf16")
    acd = oracle.decode(Ac, "bf16")
    bd = oracle.decode(B, "bf16")
    for m in range(M):
        for n in range(N):
            total = Fraction(0)
            for g in range(K // 4):
                nib = (int(meta[m, g // 8]) >> (4 * (g % 8))) & 0xF
                for t, q in enumerate((nib & 3, nib >> 2)):
                    total += Fraction(acd[m, 2 * g + t]) * Fraction(bd[n, 4 * g + q])
            assert abs(Fraction(ref[m, n]) - total) <= Fraction(2.0 ** -45) * (1 + abs(total))


def test_sparse_decompress_rejects_unordered_metadata():
    Ac = np.zeros((1, 16), dtype=np.uint16)
    meta = np.array([[0x33333333]], dtype=np.uint32)  # i0 = i1 = 3: not ascending
    with pytest.raises(ValueError):
        oracle.sp_decompress(Ac, meta, "bf16")


# ---------------------------------------------------------------- block-scaled (MX)

def test_decode_e8m0_exhaustive_closed_form():
    import math
    c = np.arange(256, dtype=np.uint8)
    got = oracle.decode(c, "e8m0")
    for e in range(255):
        assert got[e] == math.ldexp(1.0, e - 127)
    assert np.isnan(got[255])
    if hasattr(torch, "float8_e8m0fnu"):
        theirs = torch.from_numpy(c.copy()).view(torch.float8_e8m0fnu).to(torch.float64).numpy()
        assert _same(got, theirs)


def _mx_inputs(M, N, K, seed, fa="e4m3", fb="e4m3"):
    g = si.generator(seed)
    A, SA = si.mx_quantize(torch.randn((M, K), generator=g), fa)
    B, SB = si.mx_quantize(torch.randn((N, K), generator=g), fb)
    return si.codes(A), SA.numpy(), si.codes(B), SB.numpy()


def test_mx_ones_closed_form():
    """a = b = 1 everywhere, scales 2^u and 2^v per block: D = sum_g 32 * 2^(u_mg + v_ng)."""
    M, N, K = 6, 5, 128
    g = np.random.default_rng(4)
    u = g.integers(-6, 6, (M, K // 32))
    v = g.integers(-6, 6, (N, K // 32))
    ones_a = si.codes(torch.ones((M, K), dtype=torch.float8_e4m3fn))
    ones_b = si.codes(torch.ones((N, K), dtype=torch.float8_e4m3fn))
    ref, S = oracle.gemm_mx(ones_a, (u + 127).astype(np.uint8), ones_b, (v + 127).astype(np.uint8),
                            "e4m3", "e4m3")
    expect = (32.0 * 2.0 ** (u[:, None, :] + v[None, :, :])).sum(axis=2)
    assert np.array_equal(ref, expect) and np.array_equal(S, expect)


@pytest.mark.parametrize("fa,fb", [("e4m3", "e4m3"), ("e4m3", "e5m2"), ("e5m2", "e5m2")])
def test_mx_matches_numpy_expansion(fa, fb):
    """Expanding every block scale onto its 32 elements and multiplying (numpy fp64)."""
    M, N, K = 48, 40, 256
    A, SA, B, SB = _mx_inputs(M, N, K, 17, fa, fb)
    ref, S = oracle.gemm_mx(A, SA, B, SB, fa, fb)
    ea = oracle.decode(A, fa) * np.repeat(oracle.decode(SA, "e8m0"), 32, axis=1)
    eb = oracle.decode(B, fb) * np.repeat(oracle.decode(SB, "e8m0"), 32, axis=1)
    assert np.all(np.abs(ref - ea @ eb.T) <= 1e-12 * S)
    assert np.allclose(S, np.abs(ea) @ np.abs(eb).T, rtol=1e-12, atol=0)


def test_mx_scales_enter_per_block_exact():
    """Tiny case against exact rationals: each block's sum is scaled before it is added."""
    M, N, K = 3, 2, 96
    A, SA, B, SB = _mx_inputs(M, N, K, 23)
    SA[0, 1] = 127 + 5  # make the per-block scales differ strongly
    SB[1, 2] = 127 - 7
    ref, _ = oracle.gemm_mx(A, SA, B, SB, "e4m3", "e4m3", alpha=0.5, bias=si.codes(torch.tensor([1.0, -2.0],
                                                                                                  dtype=torch.bfloat16)))
    a = oracle.decode(A, "e4m3")
    b = oracle.decode(B, "e4m3")
    for m in range(M):
        for n in range(N):
            total = Fraction(0)
            for gi in range(K // 32):
                part = sum(Fraction(a[m, k]) * Fraction(b[n, k]) for k in range(32 * gi, 32 * gi + 32))
                total += part * Fraction(2) ** (int(SA[m, gi]) - 127) * Fraction(2) ** (int(SB[n, gi]) - 127)
            want = Fraction(1, 2) * total + [Fraction(1), Fraction(-2)][n]
            assert Fraction(ref[m, n]) == want


def test_mx_unit_scales_equal_plain_gemm():
    M, N, K = 20, 24, 160
    A, _, B, _ = _mx_inputs(M, N, K, 29)
    ones_a = np.full((M, K // 32), 127, dtype=np.uint8)
    ones_b = np.full((N, K // 32), 127, dtype=np.uint8)
    r1, s1 = oracle.gemm_mx(A, ones_a, B, ones_b, "e4m3", "e4m3")
    r2, s2 = oracle.gemm(A, B, "e4m3", "e4m3")
    assert np.array_equal(r1, r2) and np.array_equal(s1, s2)


def test_mx_sampled_equals_full():
    M, N, K = 30, 20, 64
    A, SA, B, SB = _mx_inputs(M, N, K, 31)
    full, Sf = oracle.gemm_mx(A, SA, B, SB, "e4m3", "e4m3")
    r = np.array([0, 5, 29, 7]); c = np.array([0, 19, 3, 3])
    samp, Ss = oracle.gemm_mx(A, SA, B, SB, "e4m3", "e4m3", rows=r, cols=c)
    assert np.array_equal(samp, full[r, c]) and np.array_equal(Ss, Sf[r, c])


# ---- blocked scale layout (a pure permutation defined by the library header)

def _pack_source(rows, K):
    nblk = K // 32
    r = np.arange(rows)[:, None]
    j = np.arange(nblk)[None, :]
    return ((r * 7 + j * 3) % 254).astype(np.uint8)  # never 127 at most positions, never 255


def test_mx_pack_hand_worked_positions():
    """rows = 130, K = 160: 2 row tiles x 2 K stages of 512-byte atoms; positions worked by hand."""
    SC = _pack_source(130, 160)
    out = oracle.mx_pack_scales(SC, 160)
    assert out.shape == (2048,)
    cases = {  # (row, block) -> byte offset
        (0, 0): 0, (1, 0): 16, (32, 0): 4, (33, 3): 23, (127, 2): 510,
        (0, 4): 512, (31, 4): 1008, (96, 4): 524, (128, 0): 1024, (129, 4): 1552,
    }
    for (r, j), pos in cases.items():
        assert out[pos] == SC[r, j], (r, j, pos)
    for pos in (513, 515, 1056, 2047, 1024 + 64):  # block 5+ of stage 1, rows 130+
        assert out[pos] == 127, pos


@pytest.mark.parametrize("rows,K", [(1, 32), (127, 96), (128, 128), (130, 160), (300, 1024)])
def test_mx_pack_is_a_permutation_with_unit_padding(rows, K):
    SC = _pack_source(rows, K)
    out = oracle.mx_pack_scales(SC, K)
    kt = (K + 127) // 128
    assert out.size == ((rows + 127) // 128) * kt * 512
    # a block-by-block view (tile, quarter, lane, stage, block) read back in row-major order
    rt = (rows + 127) // 128
    atoms = out.reshape(rt, kt, 32, 4, 4)  # (tile, stage, lane, quarter, block-in-stage)
    back = atoms.transpose(0, 3, 2, 1, 4).reshape(rt * 128, kt * 4)
    assert np.array_equal(back[:rows, :K // 32], SC)
    pad = np.ones_like(back, dtype=bool)
    pad[:rows, :K // 32] = False
    assert np.all(back[pad] == 127)


# ---- fused epilogue tail: activation, FP8 target, bound

def _phi_simpson(x, n=20000):
    """Standard normal distribution function by Simpson's rule on the density (independent of erf)."""
    import math
    if x == 0:
        return 0.5
    h = x / n
    s = 1.0 + math.exp(-0.5 * x * x)
    for i in range(1, n):
        t = i * h
        s += (4 if i % 2 else 2) * math.exp(-0.5 * t * t)
    return 0.5 + s * h / 3.0 / math.sqrt(2.0 * math.pi)


def test_gelu_is_x_times_normal_cdf():
    xs = np.array([-4.0, -1.5, -0.25, 0.3, 1.0, 2.5])
    got = oracle.activate(xs, "gelu")
    for x, g in zip(xs, got):
        assert abs(g - x * _phi_simpson(float(x))) <= 1e-12 * max(1.0, abs(x))
    # Phi(1) from the standard normal table
    assert abs(oracle.activate(np.array([1.0]), "gelu")[0] - 0.8413447460685429) < 1e-15


def test_gelu_odd_part_identity_and_limits():
    g = np.random.default_rng(3)
    x = g.normal(0, 3, 1000)
    assert np.allclose(oracle.activate(x, "gelu") - oracle.activate(-x, "gelu"), x, rtol=0, atol=1e-12)
    assert oracle.activate(np.array([0.0]), "gelu")[0] == 0.0
    big = oracle.activate(np.array([12.0, -12.0]), "gelu")
    assert big[0] == 12.0 and abs(big[1]) < 1e-30


def test_relu_definition():
    x = np.array([-2.0, -0.0, 0.0, 1e-300, 3.5, np.nan, -np.inf, np.inf])
    y = oracle.activate(x, "relu")
    assert list(y[:5]) == [0.0, 0.0, 0.0, 1e-300, 3.5]
    assert y[5] == 0.0 and y[6] == 0.0 and y[7] == np.inf
    assert np.array_equal(oracle.activate(x[:5], "none"), x[:5])


def test_fp8_target_divides_and_saturates():
    y = np.array([100.0, 896.0, 897.0, -1e9, 0.5, np.nan])
    t, *_ = oracle.fused_reference(y, np.zeros_like(y), None, "e4m3", d_scale=2.0)
    assert list(t[:5]) == [50.0, 448.0, 448.0, -448.0, 0.25] and np.isnan(t[5])
    t, *_ = oracle.fused_reference(np.array([1e6, -57344.0 * 4]), np.zeros(2), None, "e5m2", d_scale=4.0)
    assert list(t) == [57344.0, -57344.0]


def test_fused_bound_without_activation_covers_the_plain_bound():
    g = np.random.default_rng(5)
    ref = g.normal(0, 10, 200)
    S = np.abs(g.normal(0, 100, 200))
    for fmt in ("bf16", "f16", "f32"):
        t, b, y, ey = oracle.fused_reference(ref, S, None, fmt, scale=0.5)
        assert np.array_equal(t, ref) and np.array_equal(y, ref)
        assert np.all(b >= oracle.bound(ref, S, fmt, 0.5))
    _, b_relu, _, e_relu = oracle.fused_reference(ref, S, "relu", "bf16")
    _, b_gelu, _, e_gelu = oracle.fused_reference(ref, S, "gelu", "bf16")
    assert np.all(e_gelu >= e_relu)


# ---- FP4 E2M1 (OCP): decode, packing order, GEMM with packed operands

def test_e2m1_decode_all_codes():
    """The 16 E2M1 codes from the format definition: s | e(2, bias 1) | m(1), no inf/NaN."""
    table = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
    codes = np.array([(2 * i + 1) << 4 | (2 * i) for i in range(8)], dtype=np.uint8)  # codes 0..15 in order
    got = oracle.decode(codes, "e2m1")
    assert list(got[:8]) == table
    assert list(-got[8:]) == table and np.signbit(got[8])


def test_e2m1_packing_puts_element_2i_in_the_low_nibble():
    got = oracle.decode(np.array([[0x21, 0x7F]], dtype=np.uint8), "e2m1")
    assert got.tolist() == [[0.5, 1.0, -6.0, 6.0]]


def test_gemm_with_e2m1_operand_matches_numpy():
    g = np.random.default_rng(11)
    M, N, K = 20, 24, 96
    A = si.codes(si.fp8_per_tensor(torch.from_numpy(g.normal(size=(M, K)).astype(np.float32)), "e4m3")[0])
    B = g.integers(0, 256, (N, K // 2), dtype=np.uint8)
    ref, S = oracle.gemm(A, B, "e4m3", "e2m1", sa=0.5, sb=2.0)
    da, db = oracle.decode(A, "e4m3"), oracle.decode(B, "e2m1")
    assert db.shape == (N, K)
    assert np.all(np.abs(ref - da @ db.T) <= 1e-12 * np.maximum(S, 1e-300))
    # swapped roles: E2M1 A
    ref2, _ = oracle.gemm(B, A, "e2m1", "e4m3")
    assert np.allclose(ref2, db @ da.T, rtol=1e-12, atol=0)


def test_fp4_input_rounding_ties_to_even_and_saturates():
    x = torch.tensor([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, -5.0, 7.0, -0.3, 0.26, 100.0])
    vals = oracle.decode(si.pack_fp4(si.fp4_e2m1(x)).numpy(), "e2m1")
    assert vals.tolist() == [0.0, 1.0, 1.0, 2.0, 2.0, 4.0, 4.0, -4.0, 6.0, -0.5, 0.5, 6.0]


# ---- NVFP4: UE4M3 block scales per 16 over E2M1 elements

def test_ue4m3_decode():
    c = np.arange(128, dtype=np.uint8)
    got = oracle.decode(c, "ue4m3")
    theirs = torch.from_numpy(c.copy()).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    assert _same(got, theirs)
    assert got[0x38] == 1.0 and got[0x7E] == 448.0 and got[0x01] == 2.0 ** -9 and np.isnan(got[0x7F])


def test_nvfp4_ones_closed_form():
    """a = b = 1 (E2M1 code 2) everywhere, block scales 2^u, 2^v per 16: D = sum_g 16 * 2^(u + v)."""
    M, N, K = 5, 6, 128
    g = np.random.default_rng(9)
    u = g.integers(-5, 6, (M, K // 16))
    v = g.integers(-5, 6, (N, K // 16))
    ones_a = np.full((M, K // 2), 0x22, dtype=np.uint8)
    ones_b = np.full((N, K // 2), 0x22, dtype=np.uint8)
    ref, S = oracle.gemm_mx(ones_a, ((u + 7) << 3).astype(np.uint8), ones_b, ((v + 7) << 3).astype(np.uint8),
                            "e2m1", "e2m1", block=16, sf_fmt="ue4m3")
    expect = (16.0 * 2.0 ** (u[:, None, :] + v[None, :, :])).sum(axis=2)
    assert np.array_equal(ref, expect) and np.array_equal(S, expect)


def test_nvfp4_matches_numpy_expansion():
    c = si.nvfp4_case(40, 24, 192, seed=3)
    ref, S = oracle.gemm_mx(c["A"].numpy(), c["SA"].numpy(), c["B"].numpy(), c["SB"].numpy(), "e2m1", "e2m1",
                            block=16, sf_fmt="ue4m3", alpha=c["alpha"])
    ea = oracle.decode(c["A"].numpy(), "e2m1") * np.repeat(oracle.decode(c["SA"].numpy(), "ue4m3"), 16, axis=1)
    eb = oracle.decode(c["B"].numpy(), "e2m1") * np.repeat(oracle.decode(c["SB"].numpy(), "ue4m3"), 16, axis=1)
    assert np.all(np.abs(ref - c["alpha"] * (ea @ eb.T)) <= 1e-12 * c["alpha"] * np.maximum(S, 1e-300))


# ---- hardware-ordered 2:4 metadata (tensor-memory order of the sparse MMA)

def test_sp_meta_pack_hand_worked():
    """16 rows, K = 32: one canonical word per row, one stage, MMA 0 only; positions worked by hand."""
    meta = np.array([0xA0A1A2A3 + 0x01010101 * r for r in range(16)], dtype=np.uint32).reshape(16, 1)
    out = oracle.sp_meta_pack(meta, 32).view(np.uint32).reshape(128, 4)  # (lane, MMA k)
    assert out[0, 0] == (0xA2A3 | (0xAAAB << 16))          # lane 0: low halves of rows 0 and 8
    assert out[8, 0] == (0xA0A1 | (0xA8A9 << 16))          # lane 8: high halves of rows 0 and 8
    assert out[3, 0] == (0xA5A6 | (0xADAE << 16))          # lane 3: rows 3 and 11
    assert out[15, 0] == (0xA7A8 | (0xAFB0 << 16))         # lane 15: high halves of rows 7 and 15
    assert np.all(out[16:, 0] == 0x44444444)                # rows >= 16 read positions {0, 1}
    assert np.all(out[:, 1:] == 0x44444444)                 # MMAs 1..3: words past K/32


@pytest.mark.parametrize("M,K", [(128, 128), (130, 96), (300, 512)])
def test_sp_meta_pack_reads_back_to_the_canonical_words(M, K):
    g = np.random.default_rng(M + K)
    meta = g.integers(0, 2 ** 32, (M, K // 32), dtype=np.uint64).astype(np.uint32)
    words = oracle.sp_meta_pack(meta, K).view(np.uint32)
    kbs = (K + 127) // 128
    assert words.size == ((M + 127) // 128) * kbs * 128 * 4
    back = np.zeros_like(meta)
    for R in range(M):
        t, i = divmod(R, 128)
        a, rr = divmod(i, 16)
        half = 16 * (rr // 8)         # rows 16a+8.. sit in the high halves
        r = rr % 8
        for q in range(K // 32):
            base = (t * kbs + q // 4) * 128
            lo = (int(words[(base + 16 * a + r) * 4 + q % 4]) >> half) & 0xFFFF      # lane s = 0: nibbles 0..3
            hi = (int(words[(base + 16 * a + 8 + r) * 4 + q % 4]) >> half) & 0xFFFF  # lane s = 1: nibbles 4..7
            back[R, q] = lo | (hi << 16)
    assert np.array_equal(back, meta)


def test_pack_replicated_atoms_are_copies():
    """reps = 4 (NVFP4): each 512-byte atom four times in a row, otherwise the reps = 1 layout."""
    SC = _pack_source(130, 160)
    one = oracle.mx_pack_scales(SC, 160)
    four = oracle.mx_pack_scales(SC, 160, reps=4)
    assert four.size == 4 * one.size
    atoms = four.reshape(-1, 4, 512)
    for c in range(4):
        assert np.array_equal(atoms[:, c, :].reshape(-1), one)


# ---- MXFP4: E8M0 block scales per 32 over E2M1 elements

def test_mxfp4_ones_closed_form():
    """a = b = 1 (E2M1 code 2) everywhere, block scales 2^u, 2^v per 32: D = sum_g 32 * 2^(u + v)."""
    M, N, K = 5, 6, 256
    g = np.random.default_rng(19)
    u = g.integers(-6, 7, (M, K // 32))
    v = g.integers(-6, 7, (N, K // 32))
    ones_a = np.full((M, K // 2), 0x22, dtype=np.uint8)
    ones_b = np.full((N, K // 2), 0x22, dtype=np.uint8)
    ref, S = oracle.gemm_mx(ones_a, (u + 127).astype(np.uint8), ones_b, (v + 127).astype(np.uint8),
                            "e2m1", "e2m1", block=32, sf_fmt="e8m0")
    expect = (32.0 * 2.0 ** (u[:, None, :] + v[None, :, :])).sum(axis=2)
    assert np.array_equal(ref, expect) and np.array_equal(S, expect)


def test_mxfp4_matches_numpy_expansion():
    c = si.mxfp4_case(40, 24, 256, seed=3)
    ref, S = oracle.gemm_mx(c["A"].numpy(), c["SA"].numpy(), c["B"].numpy(), c["SB"].numpy(), "e2m1", "e2m1",
                            block=32, sf_fmt="e8m0")
    ea = oracle.decode(c["A"].numpy(), "e2m1") * np.repeat(oracle.decode(c["SA"].numpy(), "e8m0"), 32, axis=1)
    eb = oracle.decode(c["B"].numpy(), "e2m1") * np.repeat(oracle.decode(c["SB"].numpy(), "e8m0"), 32, axis=1)
    assert np.all(np.abs(ref - ea @ eb.T) <= 1e-12 * np.maximum(S, 1e-300))


def test_mxfp4_quantize_scale_rule_worked_by_hand():
    """OCP MX conversion with emax(E2M1) = 2: block amax 3 -> e = floor(log2 3) - 2 = -1 (code 126),
    elements x / 2^-1 rounded to E2M1; amax 40 -> e = 3 (code 130), 40 / 8 = 5 -> 4 (ties to even);
    an all-zero block -> code 0 (2^-127) and zero elements."""
    x = torch.zeros((1, 96))
    x[0, 0], x[0, 1], x[0, 2] = 3.0, -0.75, 1.25     # block 0: amax 3
    x[0, 32], x[0, 33] = 40.0, 7.0                    # block 1: amax 40
    q, sc = si.mxfp4_quantize(x)
    assert sc.tolist() == [[126, 130, 0]]
    vals = oracle.decode(q.numpy(), "e2m1")[0]
    assert vals[:3].tolist() == [6.0, -1.5, 2.0]      # 3/0.5 = 6; -0.75/0.5 = -1.5; 1.25/0.5 = 2.5 -> 2 (even)
    assert vals[32:34].tolist() == [4.0, 1.0]         # 40/8 = 5 -> 4 (tie to even), 7/8 = 0.875 -> 1
    assert not vals[64:].any()


def test_fp8_target_multiplies_by_the_rounded_reciprocal():
    """FP8 outputs hold y * RN32(1 / d_scale): for d_scale = 3 the multiplier is the fp32 value
    nearest 1/3 (0x3EAAAAAB = 11184811 * 2^-25), so y = 3 targets 3 * that, just above 1."""
    r = oracle.fp32_reciprocal(3.0)
    assert r == 11184811 * 2.0 ** -25 and np.float32(r).view(np.uint32) == 0x3EAAAAAB
    t, *_ = oracle.fused_reference(np.array([3.0, -6.0]), np.zeros(2), None, "e4m3", d_scale=3.0)
    assert list(t) == [3.0 * r, -6.0 * r] and t[0] > 1.0
    # exact reciprocals are unchanged; ties between fp32 neighbours cannot occur for 1/d, but
    # the choice between the neighbours is the nearest one
    for d in (2.0, 0.25, 448.0, 1e-3, 7.0, 1.0 / 3.0):
        rr = oracle.fp32_reciprocal(d)
        c = np.float32(rr)
        lo, hi = np.nextafter(c, np.float32(0)), np.nextafter(c, np.float32(np.inf))
        from fractions import Fraction
        ex = 1 / Fraction(d)
        assert abs(Fraction(float(c)) - ex) <= min(abs(Fraction(float(lo)) - ex), abs(Fraction(float(hi)) - ex))


# ---- INT8 x INT8 -> INT32 with .satfinite

def test_gemm_i8_brute_force_python_ints():
    """Every output of a ragged 7 x 5 x 37 case against a Python-integer triple loop, with C."""
    g = np.random.default_rng(21)
    A = g.integers(-128, 128, (7, 37), dtype=np.int8)
    B = g.integers(-128, 128, (5, 37), dtype=np.int8)
    C = g.integers(-2 ** 31, 2 ** 31, (7, 5), dtype=np.int64).astype(np.int32)
    got = oracle.gemm_i8(A, B, C)
    for i in range(7):
        for j in range(5):
            exact = sum(int(A[i, k]) * int(B[j, k]) for k in range(37)) + int(C[i, j])
            assert got[i, j] == max(-2 ** 31, min(2 ** 31 - 1, exact))


def test_gemm_i8_matches_numpy_int64_and_samples():
    g = np.random.default_rng(22)
    A = g.integers(-128, 128, (64, 300), dtype=np.int8)
    B = g.integers(-128, 128, (48, 300), dtype=np.int8)
    ref = A.astype(np.int64) @ B.astype(np.int64).T
    got = oracle.gemm_i8(A, B)
    assert np.array_equal(got, ref.astype(np.int32))
    rows, cols = g.integers(0, 64, 50), g.integers(0, 48, 50)
    assert np.array_equal(oracle.gemm_i8(A, B, rows=rows, cols=cols), got[rows, cols])


def test_gemm_i8_closed_forms_and_saturation():
    """a = b = -128: each output is 16384 K; at K = 131072 that is 2^31, clamped to 2^31 - 1.
    a = -128, b = 127: -16256 K; with C = -2^31 the sum clamps to -2^31.  Identity A picks rows of B."""
    K = 1024
    A = np.full((2, K), -128, dtype=np.int8)
    assert np.all(oracle.gemm_i8(A, A[:1]) == 16384 * K)
    K = 131072
    A = np.full((1, K), -128, dtype=np.int8)
    assert oracle.gemm_i8(A, A)[0, 0] == 2 ** 31 - 1
    B = np.full((1, 8), 127, dtype=np.int8)
    C = np.array([[-2 ** 31]], dtype=np.int32)
    assert oracle.gemm_i8(np.full((1, 8), -128, dtype=np.int8), B, C)[0, 0] == -2 ** 31
    assert oracle.gemm_i8(np.full((1, 8), -128, dtype=np.int8), B)[0, 0] == -16256 * 8
    I = np.eye(16, dtype=np.int8)
    Bm = np.random.default_rng(23).integers(-128, 128, (16, 16), dtype=np.int8)
    assert np.array_equal(oracle.gemm_i8(I, Bm), Bm.T.astype(np.int32))
