"""Pins for the CPU oracle: each checks it against something other than itself.

Sources of truth used here: numpy's own binary16 conversion, the definition
of bfloat16 as the top half of binary32, exact rational arithmetic
(fractions.Fraction), closed forms (identity, permutation, all-ones,
rank-1), exact integer matrix products, torch's fp64 CPU matmul, the
error-function GELU x*Phi(x), and constants the pages print after rounding.
"""
from __future__ import annotations

import math
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

import gemm_inputs
import oracle
from tests import tolerance

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ---------------------------------------------------------------- decoders --

def test_f16_decode_all_patterns_match_numpy():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ours = oracle.decode(bits, "f16")
    ref = bits.view(np.float16).astype(np.float64)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], ref[~nan])
    # sign of zero kept
    assert math.copysign(1.0, ours[0x8000]) == -1.0


def test_bf16_decode_all_patterns_match_binary32_top_half():
    bits = np.arange(65536, dtype=np.uint32)
    ours = oracle.decode(bits.astype(np.uint16), "bf16")
    with np.errstate(invalid="ignore"):
        ref = (bits << 16).astype(np.uint32).view(np.float32).astype(np.float64)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], ref[~nan])


# ---------------------------------------------------------------- rounding --

def _f16_sample(rng, n):
    # spans subnormals, normals, near-overflow and exact ties
    mags = np.ldexp(rng.uniform(1.0, 2.0, n), rng.integers(-30, 17, n))
    x = np.where(rng.random(n) < 0.5, -mags, mags)
    return x


def test_f16_round_matches_numpy_rne():
    rng = np.random.default_rng(1)
    x = _f16_sample(rng, 200000)
    # exact ties half-way between consecutive binary16 values
    h = rng.integers(0, 0x7bff, 20000).astype(np.uint16)
    lo = h.view(np.float16).astype(np.float64)
    hi = (h + 1).astype(np.uint16).view(np.float16).astype(np.float64)
    ties = (lo + hi) / 2
    x = np.concatenate([x, ties, -ties, [65504.0, 65519.99, 65520.0, 1e6, 2.0 ** -25,
                                         3 * 2.0 ** -25, 2.0 ** -26, 0.0, -0.0]])
    ours = oracle.round_to(x, "f16")
    with np.errstate(over="ignore"):
        ref = x.astype(np.float16).view(np.uint16)
    assert np.array_equal(ours, ref)


def test_rounding_of_nan_and_infinities():
    # IEEE 754: a NaN stays a NaN (the default quiet NaN), infinities keep
    # their sign.  fp16 against numpy's binary16 conversion; bf16 against the
    # upper half of numpy's binary32 patterns (bf16 is binary32's top 16 bits,
    # and these values need no rounding).
    x = np.array([np.nan, np.inf, -np.inf], dtype=np.float64)
    assert np.array_equal(oracle.round_to(x, "f16"), x.astype(np.float16).view(np.uint16))
    top = (x.astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    assert np.array_equal(oracle.round_to(x, "bf16"), top)
    for dt in ("f16", "bf16"):
        back = oracle.decode(oracle.round_to(x, dt), dt)
        assert np.isnan(back[0]) and back[1] == np.inf and back[2] == -np.inf


def test_bf16_round_is_nearest_even_by_enumeration():
    # All finite non-negative bf16 values, in increasing order of bit pattern.
    pos_bits = np.arange(0, 0x7f80, dtype=np.uint32)
    pos_vals = (pos_bits << 16).astype(np.uint32).view(np.float32).astype(np.float64)
    rng = np.random.default_rng(2)
    mags = np.ldexp(rng.uniform(1.0, 2.0, 50000), rng.integers(-135, 128, 50000))
    k = rng.integers(1, len(pos_vals) - 1, 5000)
    ties = (pos_vals[k] + pos_vals[k + 1]) / 2
    x = np.concatenate([mags, ties])
    ours = oracle.round_to(x, "bf16")
    idx = np.searchsorted(pos_vals, x)               # pos_vals[idx-1] < x <= pos_vals[idx]
    for xi, oi, i in zip(x, ours, idx):
        if i >= len(pos_vals):                       # above the largest finite value:
            # IEEE rounds as if the next binade existed; reaching 2^128 means inf.
            below, above = pos_vals[-1], 2.0 ** 128
            cand_bits = (0x7f7f, 0x7f80)
        else:
            below, above = pos_vals[i - 1], pos_vals[i]
            cand_bits = (i - 1, i)
        if xi == above:
            want = cand_bits[1]
        else:
            d0, d1 = xi - below, above - xi
            if d0 < d1:
                want = cand_bits[0]
            elif d1 < d0:
                want = cand_bits[1]
            else:
                want = cand_bits[0] if cand_bits[0] % 2 == 0 else cand_bits[1]
        assert oi == want, (xi, oi, want)


def test_rounding_reproduces_printed_gelu_constants():
    path = os.path.join(GOLDEN, "gelu_constants_printed.txt")
    n = 0
    with open(path) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            exact, dtype, printed, digits, _src = line.split()
            bits = oracle.round_to(np.array([float(exact)]), dtype)
            val = oracle.decode(bits, dtype)[0]
            assert float("%.*g" % (int(digits), val)) == pytest.approx(float(printed), rel=0, abs=0), \
                (exact, dtype, val, printed)
            n += 1
    assert n == 4


# -------------------------------------------------------------- GEMM pins --

def _exact_gemm(a_vals, b_vals):
    M, K = len(a_vals), len(a_vals[0]) if a_vals else 0
    N = len(b_vals)
    return [[sum((Fraction(a_vals[i][k]) * Fraction(b_vals[j][k]) for k in range(K)), Fraction(0))
             for j in range(N)] for i in range(M)]


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("shape", [(1, 1, 1), (2, 3, 5), (7, 5, 3), (8, 8, 8), (3, 1, 7), (5, 2, 1)])
def test_gemm_matches_exact_rational_arithmetic(dtype, shape):
    M, N, K = shape
    A, B = gemm_inputs.custom(M, N, K, dtype=dtype, seed=sum(shape))
    a = oracle.decode(A, dtype)
    b = oracle.decode(B, dtype)
    exact = _exact_gemm(a.tolist(), b.tolist())
    C = oracle.gemm_nt(A, B, dtype)
    assert C.shape == (M, N)
    for i in range(M):
        for j in range(N):
            bound = K * 2.0 ** -53 * float(sum(abs(Fraction(a[i, k]) * Fraction(b[j, k]))
                                               for k in range(K)))
            assert abs(Fraction(C[i, j]) - exact[i][j]) <= Fraction(bound)


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_gemm_bit_exact_on_a_dyadic_grid(dtype):
    # Entries are multiples of 2^-6 in [-2, 2]: every partial sum is exact in fp64,
    # so the oracle must equal the rational result bit for bit.
    rng = np.random.default_rng(5)
    M, N, K = 6, 4, 9
    a = rng.integers(-128, 129, (M, K)) / 64.0
    b = rng.integers(-128, 129, (N, K)) / 64.0
    A, B = oracle.round_to(a, dtype), oracle.round_to(b, dtype)
    assert np.array_equal(oracle.decode(A, dtype), a)
    C = oracle.gemm_nt(A, B, dtype)
    exact = _exact_gemm(a.tolist(), b.tolist())
    for i in range(M):
        for j in range(N):
            assert Fraction(C[i, j]) == exact[i][j]


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_identity_gives_transpose(dtype):
    K, N = 19, 11
    _, B = gemm_inputs.custom(1, N, K, dtype=dtype, seed=7)
    I = oracle.round_to(np.eye(K), dtype)
    C = oracle.gemm_nt(I, B, dtype)                  # C[i,j] = sum_k I[i,k] B[j,k] = B[j,i]
    assert np.array_equal(C, oracle.decode(B, dtype).T)


def test_permutation_gives_column_permutation():
    M, K = 9, 13
    A, _ = gemm_inputs.custom(M, 1, K, seed=8)
    perm = np.random.default_rng(8).permutation(K)
    P = np.zeros((K, K))
    P[np.arange(K), perm] = 1.0                      # B[j, perm[j]] = 1
    C = oracle.gemm_nt(A, oracle.round_to(P, "f16"), "f16")
    a = oracle.decode(A, "f16")
    assert np.array_equal(C, a[:, perm])


def test_all_ones_gives_k():
    M, N, K = 4, 6, 257
    ones_a = oracle.round_to(np.ones((M, K)), "f16")
    ones_b = oracle.round_to(np.ones((N, K)), "f16")
    assert np.array_equal(oracle.gemm_nt(ones_a, ones_b, "f16"), np.full((M, N), float(K)))


def test_rank_one_closed_form():
    M, N, K = 7, 5, 64
    rng = np.random.default_rng(9)
    u = oracle.decode(oracle.round_to(rng.uniform(-1, 1, M), "f16"), "f16")
    v = oracle.decode(oracle.round_to(rng.uniform(-1, 1, N), "f16"), "f16")
    A = oracle.round_to(np.repeat(u[:, None], K, axis=1), "f16")
    B = oracle.round_to(np.repeat(v[:, None], K, axis=1), "f16")
    C = oracle.gemm_nt(A, B, "f16")
    assert np.array_equal(C, K * np.outer(u, v))     # K a power of two: exact


def test_small_integers_exact_against_integer_matmul():
    A, B = gemm_inputs.make("gemm_256_f16_int")
    ai = A.to(torch.int64).numpy()
    bi = B.to(torch.int64).numpy()
    assert ai.min() >= -2 and ai.max() <= 2 and len(np.unique(ai)) == 5
    C = oracle.gemm_nt(A, B, "f16")
    assert np.array_equal(C, (ai @ bi.T).astype(np.float64))
    assert np.abs(C).max() <= 1024


def test_library_cross_check_torch_fp64():
    for dtype in ("f16", "bf16"):
        A, B = gemm_inputs.custom(64, 48, 300, dtype=dtype, dist="normal_scaled", seed=10)
        C = oracle.gemm_nt(A, B, dtype)
        ref = torch.matmul(A.to(torch.float64), B.to(torch.float64).T).numpy()
        assert np.max(np.abs(C - ref)) <= 1e-12 * np.max(np.abs(ref))


def test_entries_equal_full_product():
    A, B = gemm_inputs.custom(33, 29, 71, seed=11)
    full = oracle.gemm_nt(A, B, "f16", epilogue="gelu")
    rng = np.random.default_rng(11)
    r = rng.integers(0, 33, 200)
    c = rng.integers(0, 29, 200)
    ent = oracle.gemm_nt_entries(A, B, "f16", r, c, epilogue="gelu")
    assert np.array_equal(ent, full[r, c])


def test_empty_and_zero_k():
    A = np.zeros((3, 0), np.uint16)
    B = np.zeros((4, 0), np.uint16)
    assert np.array_equal(oracle.gemm_nt(A, B, "f16"), np.zeros((3, 4)))
    assert oracle.gemm_nt(np.zeros((0, 5), np.uint16), np.zeros((2, 5), np.uint16), "f16").shape == (0, 2)


def test_entries_reject_out_of_range():
    A, B = gemm_inputs.custom(4, 4, 4, seed=1)
    with pytest.raises(RuntimeError):
        oracle.gemm_nt_entries(A, B, "f16", [4], [0])


# -------------------------------------------------------------- GELU pins --

def test_gelu_zero_and_odd_even_identity():
    x = np.linspace(-9, 9, 2001)
    g = oracle.gelu_tanh(x)
    gm = oracle.gelu_tanh(-x)
    assert oracle.gelu_tanh(np.array([0.0]))[0] == 0.0
    # 0.5x(1+t(x)) - 0.5(-x)(1+t(-x)) = x because t is odd
    assert np.max(np.abs((g - gm) - x)) <= 1e-14 * 9


def test_gelu_slope_half_at_zero():
    h = 1e-6
    g = oracle.gelu_tanh(np.array([h, -h]))
    assert abs((g[0] - g[1]) / (2 * h) - 0.5) < 1e-9


def test_gelu_asymptotes_and_no_nan():
    big = np.array([50.0, 100.0, 1e4, 1e200])
    assert np.array_equal(oracle.gelu_tanh(big), big)
    neg = oracle.gelu_tanh(-big)
    assert np.all(neg == 0.0)
    mixed = np.concatenate([big, -big, [1e308, -1e308]])
    assert not np.any(np.isnan(oracle.gelu_tanh(mixed)))


def test_gelu_close_to_erf_gelu_with_known_max_error():
    # The tanh form approximates x*Phi(x); its largest deviation is about 4.73e-4
    # (near |x| = 2.7).  A wrong constant (e.g. the bf16-rounded 0.796875 or a
    # mistyped cubic coefficient) moves the maximum outside this window.
    xs = np.linspace(-8, 8, 160001)
    exact = np.array([0.5 * x * (1 + math.erf(x / math.sqrt(2))) for x in xs])
    d = np.abs(oracle.gelu_tanh(xs) - exact)
    assert 4.70e-4 <= d.max() <= 4.76e-4
    assert 2.6 <= abs(xs[int(np.argmax(d))]) <= 2.8


def test_gemm_gelu_epilogue_applies_after_sum():
    A, B = gemm_inputs.custom(5, 7, 40, dtype="bf16", dist="normal_xw", seed=12)
    plain = oracle.gemm_nt(A, B, "bf16")
    fused = oracle.gemm_nt(A, B, "bf16", epilogue="gelu")
    assert np.array_equal(fused, oracle.gelu_tanh(plain))


# ------------------------------------------------------ tolerance metric --

def test_tolerance_self_check_and_negative_control():
    A, B = gemm_inputs.custom(96, 80, 512, dist="normal_scaled", seed=13)
    ref = oracle.gemm_nt(A, B, "f16")
    rounded = oracle.decode(oracle.round_to(ref, "f16"), "f16")
    st = tolerance.compare(rounded, ref, "f16")
    assert st["ok"] and st["max_ulp"] <= 0.5
    bad = rounded.copy()
    bad[17, 23] = ref[17, 23] + 3 * tolerance.ulp(ref[17, 23], "f16") + 1.001e-3
    st = tolerance.compare(bad, ref, "f16")
    assert not st["ok"] and st["bad"] == 1 and st["first_bad"] == (17, 23)
    nanned = rounded.copy()
    nanned[0, 0] = np.nan
    assert not tolerance.compare(nanned, ref, "f16")["ok"]


def test_ulp_definition_matches_numpy_spacing():
    rng = np.random.default_rng(3)
    x16 = np.ldexp(rng.uniform(1, 2, 1000), rng.integers(-24, 15, 1000)).astype(np.float16)
    x16 = x16[x16 > 0]
    assert np.array_equal(tolerance.ulp(x16.astype(np.float64), "f16"),
                          np.spacing(x16).astype(np.float64))


def test_bf16_rounding_floor_exceeds_frobenius_bound():
    # The reason the bf16 Frobenius check is taken against the correctly rounded
    # result: rounding alone already costs more than 1e-3 relative.
    A, B = gemm_inputs.make("gelu_3072x16384x4096_bf16", M=128, N=256, K=256)
    ref = oracle.gemm_nt(A, B, "bf16", epilogue="gelu")
    rnd = oracle.decode(oracle.round_to(ref, "bf16"), "bf16")
    assert np.linalg.norm(rnd - ref) / np.linalg.norm(ref) > 1e-3
    st = tolerance.compare(rnd, ref, "bf16")
    assert st["ok"] and st["frob"] == 0.0
    # one element off by 3 ulps still fails per element
    bad = rnd.copy()
    bad[5, 7] += 3 * tolerance.ulp(ref[5, 7], "bf16") + 1.001e-3
    assert not tolerance.compare(bad, ref, "bf16")["ok"]


# -------------------------------------------------------------- ReLU pins --

def test_relu_epilogue_on_a_transposed_identity():
    # A = I makes C = B^T exactly; with the ReLU epilogue every negative entry
    # of B^T must become +0 and every positive one stay as it is.
    K, N = 24, 13
    _, B = gemm_inputs.custom(1, N, K, dist="int", lo=-3, hi=3, seed=17)
    I = oracle.round_to(np.eye(K), "f16")
    C = oracle.gemm_nt(I, B, "f16", epilogue="relu")
    bt = B.to(torch.float64).numpy().T
    want = np.where(bt > 0, bt, 0.0)
    assert np.array_equal(C, want)
    assert not np.any(np.signbit(C))           # no -0


def test_relu_epilogue_is_the_triton_clamp():
    # matmul_relu_kernel: acc = max(acc, 0) on the fp32 accumulator; in exact
    # arithmetic that is the positive part of the plain product, which the
    # integer case pins independently of the oracle (numpy int64 matmul).
    A, B = gemm_inputs.custom(40, 30, 64, dist="int", lo=-2, hi=2, seed=18)
    C = oracle.gemm_nt(A, B, "f16", epilogue="relu")
    exact = A.to(torch.int64).numpy() @ B.to(torch.int64).numpy().T
    assert np.array_equal(C, np.maximum(exact, 0).astype(np.float64))
    assert (exact < 0).any() and (exact > 0).any()


# ------------------------------------------------------------------ bias --
# No page defines a bias; the reading is a Linear layer's per-output-column
# bias, added to the exact sum before the epilogue.

def test_bias_alone_with_zero_a():
    # A = 0 leaves C[i,j] = epi(bias[j]) in every row.  M < N so that a bias
    # taken by row index instead of column index reads a different value.
    M, N, K = 3, 7, 5
    A = np.zeros((M, K), dtype=np.float16)
    _, B = gemm_inputs.custom(1, N, K, seed=19)
    bias = np.array([-2.5, -0.75, -0.0, 0.0, 0.5, 1.25, 3.0], dtype=np.float16)
    b = bias.astype(np.float64)
    for epi, f in ((None, lambda x: x), ("relu", lambda x: np.where(x > 0, x, 0.0)),
                   ("gelu", lambda x: 0.5 * x * (1 + np.tanh(0.7978845608 * (x + 0.044715 * x ** 3))))):
        C = oracle.gemm_nt(A, B, "f16", epilogue=epi, bias=bias)
        assert np.allclose(C, np.broadcast_to(f(b), (M, N)), rtol=1e-15, atol=0), epi


def test_bias_is_exact_on_integers():
    # Integer A, B and bias: C = A B^T + bias exactly (numpy int64 arithmetic),
    # for fp16 and bf16 patterns of the same integers.
    for dtype, td in (("f16", torch.float16), ("bf16", torch.bfloat16)):
        A, B = gemm_inputs.custom(9, 14, 32, dtype=dtype, dist="int", lo=-2, hi=2, seed=21)
        bias_i = np.arange(-7, 7, dtype=np.int64) * 3
        bias = torch.tensor(bias_i, dtype=td)
        C = oracle.gemm_nt(A, B, dtype, bias=bias)
        exact = A.to(torch.int64).numpy() @ B.to(torch.int64).numpy().T + bias_i[None, :]
        assert np.array_equal(C, exact.astype(np.float64)), dtype


def test_bias_is_added_before_the_epilogue():
    # Sums that are negative but become positive with the bias: ReLU must see
    # s + b (giving s + b), not s (giving b).
    A = np.full((2, 4), 1.0, dtype=np.float16)
    B = np.full((3, 4), -1.0, dtype=np.float16)          # every sum is -4
    bias = np.array([5.0, 4.0, 6.5], dtype=np.float16)
    C = oracle.gemm_nt(A, B, "f16", epilogue="relu", bias=bias)
    assert np.array_equal(C, np.broadcast_to(np.array([1.0, 0.0, 2.5]), (2, 3)))
    G = oracle.gemm_nt(A, B, "f16", epilogue="gelu", bias=bias)
    x = np.array([1.0, 0.0, 2.5])
    assert np.allclose(G[0], 0.5 * x * (1 + np.tanh(0.7978845608 * (x + 0.044715 * x ** 3))),
                       rtol=1e-15, atol=0)


def test_bias_entries_equal_the_full_product():
    A, B = gemm_inputs.custom(11, 17, 40, seed=22)
    bias = torch.linspace(-2, 2, 17).to(torch.float16)
    C = oracle.gemm_nt(A, B, "f16", epilogue="gelu", bias=bias)
    rows = np.array([0, 10, 5, 3], dtype=np.int64)
    cols = np.array([16, 0, 8, 11], dtype=np.int64)
    e = oracle.gemm_nt_entries(A, B, "f16", rows, cols, epilogue="gelu", bias=bias)
    assert np.array_equal(e, C[rows, cols])


def test_no_bias_is_a_zero_bias():
    A, B = gemm_inputs.custom(5, 6, 16, seed=23)   # M < N (see test_bias_alone_with_zero_a)
    z = torch.zeros(6, dtype=torch.float16)
    assert np.array_equal(oracle.gemm_nt(A, B, "f16", bias=z), oracle.gemm_nt(A, B, "f16"))


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_row_block_comparison_equals_whole_matrix_comparison(dtype):
    # The full-size parity tests compare 8192 x 8192 results a block of rows
    # at a time; the blocks must add up to exactly the whole-matrix verdict,
    # including a planted element error in the last, partial block.
    A, B = gemm_inputs.custom(203, 96, 300, dtype=dtype, dist="normal_scaled", seed=14)
    ref = oracle.gemm_nt(A, B, dtype)
    rnd = oracle.decode(oracle.round_to(ref, dtype), dtype)
    noisy = rnd + 0.4 * tolerance.ulp(ref, dtype) * np.sign(np.sin(np.arange(ref.size))).reshape(ref.shape)
    for got in (rnd, noisy):
        whole = tolerance.compare(got, ref, dtype)
        blocks = tolerance.compare_rows(lambda r0, r1: got[r0:r1], ref, dtype, chunk=64)
        assert blocks["ok"] == whole["ok"] and blocks["bad"] == whole["bad"]
        for key in ("frob", "frob_vs_exact", "max_abs", "max_ulp"):
            assert blocks[key] == pytest.approx(whole[key], rel=1e-12, abs=1e-300), key
    bad = rnd.copy()
    bad[200, 5] = ref[200, 5] + 3 * tolerance.ulp(ref[200, 5], dtype) + 1.001e-3
    blocks = tolerance.compare_rows(lambda r0, r1: bad[r0:r1], ref, dtype, chunk=64)
    assert not blocks["ok"] and blocks["bad"] == 1 and blocks["first_bad"] == (200, 5)
    bad[3, 3] = np.nan
    blocks = tolerance.compare_rows(lambda r0, r1: bad[r0:r1], ref, dtype, chunk=64)
    assert blocks["bad"] == 2 and blocks["first_bad"] == (3, 3) and not blocks["ok"]
