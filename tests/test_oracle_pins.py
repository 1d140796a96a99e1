"""Pins for the CPU oracle (no GPU).

Each test checks the oracle against something other than itself: exact
integer arithmetic (numpy int64 matmul / einsum on small-integer inputs,
which bf16 and fp64 represent exactly), hand-worked values, closed forms
(identity, permutation, rank-1), an exact rational brute force, and
identities of SiLU.  A dropped term, a wrong sign or index, or a transposed
operand in the oracle fails at least one of them.
"""
import math
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def bf16_bits(x: np.ndarray) -> np.ndarray:
    """Float array -> bf16 bit patterns (values must be exactly representable)."""
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16)
    back = t.to(torch.float32).numpy()
    assert np.array_equal(back, np.asarray(x, dtype=np.float32)), "not bf16-exact"
    return t.view(torch.int16).numpy().view(np.uint16)


def small_ints(rng, shape, lo=-8, hi=8):
    return rng.integers(lo, hi + 1, size=shape).astype(np.float64)


def read_golden(name):
    blocks = {}
    with open(os.path.join(GOLDEN, name)) as f:
        lines = [l.strip() for l in f if l.strip() and not l.startswith("#")]
    i = 0
    while i < len(lines):
        tag, r, c = lines[i].split()
        r, c = int(r), int(c)
        rows = [[float(v) for v in lines[i + 1 + j].split()] for j in range(r)]
        blocks[tag] = np.array(rows)
        i += 1 + r
    return blocks


# ----------------------------------------------------------------------------
# bf16 widening
# ----------------------------------------------------------------------------
def test_bf16_widening_known_patterns():
    # bit pattern -> value, from the bf16 format (sign, 8-bit exponent, 7-bit mantissa)
    cases = {0x3F80: 1.0, 0xC000: -2.0, 0x3F00: 0.5, 0x4049: 3.140625,
             0x0001: 2.0 ** -133, 0x7F7F: (2 - 2 ** -7) * 2.0 ** 127, 0x8000: -0.0}
    one = np.array([[0x3F80]], dtype=np.uint16)
    for bits, val in cases.items():
        a = np.array([[bits]], dtype=np.uint16)
        c = oracle.gemm(a, one)
        assert c[0, 0] == val, hex(bits)


# ----------------------------------------------------------------------------
# dense GEMM
# ----------------------------------------------------------------------------
def test_gemm_hand_worked_golden():
    g = read_golden("gemm_hand_2x2x3.txt")
    C = oracle.gemm(bf16_bits(g["A"]), bf16_bits(g["B"]))
    assert np.array_equal(C, g["C"])
    Cb = oracle.gemm(bf16_bits(g["A"]), bf16_bits(g["B"]),
                     bias=bf16_bits(g["bias"][0]), epi="bias")
    assert np.array_equal(Cb, g["C_bias"])


@pytest.mark.parametrize("M,N,K", [(1, 1, 1), (5, 7, 3), (13, 4, 9), (3, 17, 33)])
def test_gemm_exact_integer(M, N, K):
    rng = np.random.default_rng(M * 100 + N * 10 + K)
    A = small_ints(rng, (M, K))
    B = small_ints(rng, (N, K))
    C = oracle.gemm(bf16_bits(A), bf16_bits(B))
    ref = A.astype(np.int64) @ B.astype(np.int64).T
    assert np.array_equal(C, ref.astype(np.float64))


def test_gemm_identity_and_permutation():
    rng = np.random.default_rng(1)
    K = 24
    A = torch.randn(10, K, generator=torch.Generator().manual_seed(3)).to(torch.bfloat16)
    Af = A.float().numpy().astype(np.float64)
    I = np.eye(K)
    C = oracle.gemm(A, bf16_bits(I))
    assert np.array_equal(C, Af)
    perm = rng.permutation(K)
    P = I[perm]                     # row n of B selects column perm[n] of A
    C = oracle.gemm(A, bf16_bits(P))
    assert np.array_equal(C, Af[:, perm])
    # left identity: I_M . B^T = B^T
    Bm = torch.randn(7, K, generator=torch.Generator().manual_seed(4)).to(torch.bfloat16)
    C = oracle.gemm(bf16_bits(np.eye(K)), Bm)
    assert np.array_equal(C, Bm.float().numpy().astype(np.float64).T)


def test_gemm_rank1_closed_form():
    # A[m][k] = u_m for all k, B[n][k] = v_n for all k  =>  C = K u_m v_n
    M, N, K = 6, 5, 40
    u = np.array([1, -2, 0.5, 4, -0.25, 3])
    v = np.array([2, -1, 0.125, 8, -3])
    A = np.repeat(u[:, None], K, axis=1)
    B = np.repeat(v[:, None], K, axis=1)
    C = oracle.gemm(bf16_bits(A), bf16_bits(B))
    assert np.array_equal(C, K * np.outer(u, v))


def test_gemm_exact_rational_bruteforce():
    # fp64 accumulation of bf16 products over K=64 is exact to ~1e-15 relative;
    # check against exact rational arithmetic in pure Python.
    M, N, K = 3, 4, 64
    g = torch.Generator().manual_seed(11)
    A = torch.randn(M, K, generator=g).to(torch.bfloat16)
    B = torch.randn(N, K, generator=g).to(torch.bfloat16)
    C = oracle.gemm(A, B)
    Af = A.float().tolist()
    Bf = B.float().tolist()
    for m in range(M):
        for n in range(N):
            exact = sum(Fraction(Af[m][k]) * Fraction(Bf[n][k]) for k in range(K))
            scale = sum(abs(Fraction(Af[m][k]) * Fraction(Bf[n][k])) for k in range(K))
            assert abs(Fraction(C[m, n]) - exact) <= Fraction(1, 10 ** 14) * scale


def test_gemm_batched_strides_and_row_sample():
    rng = np.random.default_rng(5)
    batch, M, N, K = 3, 4, 6, 5
    A = small_ints(rng, (batch, M, K))
    B = small_ints(rng, (batch, N, K))
    C = oracle.gemm(bf16_bits(A), bf16_bits(B))
    for b in range(batch):
        assert np.array_equal(C[b], A[b] @ B[b].T)
    # a 2-D B is shared by every batch
    C = oracle.gemm(bf16_bits(A), bf16_bits(B[1]))
    for b in range(batch):
        assert np.array_equal(C[b], A[b] @ B[1].T)
    # row sample: listed rows computed, others untouched (NaN)
    C = oracle.gemm(bf16_bits(A), bf16_bits(B), rows=[2, 0])
    for b in range(batch):
        assert np.array_equal(C[b, [0, 2]], (A[b] @ B[b].T)[[0, 2]])
        assert np.isnan(C[b, [1, 3]]).all()


# ----------------------------------------------------------------------------
# epilogue: bias, SiLU
# ----------------------------------------------------------------------------
def test_bias_exact_integer():
    rng = np.random.default_rng(9)
    batch, M, N, K = 2, 3, 5, 4
    A = small_ints(rng, (batch, M, K))
    B = small_ints(rng, (batch, N, K))
    bias = small_ints(rng, (batch, N))
    C = oracle.gemm(bf16_bits(A), bf16_bits(B), bias=bf16_bits(bias), epi="bias")
    for b in range(batch):
        assert np.array_equal(C[b], A[b] @ B[b].T + bias[b][None, :])
    # a 1-D bias is shared by every batch
    C = oracle.gemm(bf16_bits(A), bf16_bits(B), bias=bf16_bits(bias[0]), epi="bias")
    for b in range(batch):
        assert np.array_equal(C[b], A[b] @ B[b].T + bias[0][None, :])


def test_silu_golden_values():
    pts = np.loadtxt(os.path.join(GOLDEN, "silu_values.txt"))
    x = pts[:, 0]
    # A = 0, so the pre-activation is exactly the bias
    A = np.zeros((1, 1))
    B = np.zeros((x.size, 1))
    C = oracle.gemm(bf16_bits(A), bf16_bits(B), bias=bf16_bits(x), epi="bias_silu")
    np.testing.assert_allclose(C[0], pts[:, 1], rtol=1e-15, atol=0)


def test_silu_identities():
    # silu(x) - silu(-x) = x  (since sigmoid(x) + sigmoid(-x) = 1);
    # silu(x) -> x for large x, -> 0 for very negative x; silu(0) = 0.
    g = torch.Generator().manual_seed(2)
    x = (torch.randn(64, generator=g) * 4).to(torch.bfloat16)
    xs = torch.cat([x, -x, torch.tensor([0.0, 40.0, -40.0]).to(torch.bfloat16)])
    A = np.zeros((1, 1))
    B = np.zeros((xs.numel(), 1))
    C = oracle.gemm(bf16_bits(A), bf16_bits(B), bias=xs, epi="bias_silu")[0]
    xf = xs.float().numpy().astype(np.float64)
    n = x.numel()
    np.testing.assert_allclose(C[:n] - C[n:2 * n], xf[:n], rtol=1e-13, atol=1e-13)
    assert C[2 * n] == 0.0
    assert abs(C[2 * n + 1] - 40.0) < 1e-15 * 40 + 40 * math.exp(-40) * 1.01
    assert -1e-15 < C[2 * n + 2] <= 0.0
    # SiLU is applied after the bias: with integer A.B^T = s and bias b, out = silu(s + b)
    A = np.array([[1.0, 2.0]])
    B = np.array([[1.0, -1.0]])      # s = -1
    C = oracle.gemm(bf16_bits(A), bf16_bits(B), bias=bf16_bits(np.array([2.0])), epi="bias_silu")
    np.testing.assert_allclose(C[0, 0], 0.7310585786300049, rtol=1e-15)


def test_gelu_golden_values():
    pts = np.loadtxt(os.path.join(GOLDEN, "gelu_values.txt"))
    x = pts[:, 0]
    A = np.zeros((1, 1))
    B = np.zeros((x.size, 1))
    C = oracle.gemm(bf16_bits(A), bf16_bits(B), bias=bf16_bits(x), epi="bias_gelu")
    np.testing.assert_allclose(C[0], pts[:, 1], rtol=2e-15, atol=1e-17)


def test_gelu_identities():
    # gelu(x) - gelu(-x) = x (since Phi(x) + Phi(-x) = 1); gelu(x) -> x for
    # large x and -> 0 from below for very negative x; gelu(0) = 0; the
    # activation acts on bias + A.B^T.
    g = torch.Generator().manual_seed(3)
    x = (torch.randn(64, generator=g) * 3).to(torch.bfloat16)
    xs = torch.cat([x, -x, torch.tensor([0.0, 40.0, -40.0]).to(torch.bfloat16)])
    A = np.zeros((1, 1))
    B = np.zeros((xs.numel(), 1))
    C = oracle.gemm(bf16_bits(A), bf16_bits(B), bias=xs, epi="bias_gelu")[0]
    xf = xs.float().numpy().astype(np.float64)
    n = x.numel()
    np.testing.assert_allclose(C[:n] - C[n:2 * n], xf[:n], rtol=1e-13, atol=1e-13)
    assert C[2 * n] == 0.0
    assert C[2 * n + 1] == 40.0
    assert -1e-300 <= C[2 * n + 2] <= 0.0
    A = np.array([[1.0, 2.0]])
    B = np.array([[1.0, -1.0]])      # s = -1, bias 2 -> gelu(1)
    C = oracle.gemm(bf16_bits(A), bf16_bits(B), bias=bf16_bits(np.array([2.0])), epi="bias_gelu")
    np.testing.assert_allclose(C[0, 0], 0.841344746068542948585, rtol=1e-15)


# ----------------------------------------------------------------------------
# grouped GEMM
# ----------------------------------------------------------------------------
def _int_grouped_case(rng, sizes, N, K):
    G = len(sizes)
    off = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int32)
    A = small_ints(rng, (int(off[-1]), K))
    B = small_ints(rng, (G, N, K))
    return A, B, off


@pytest.mark.parametrize("sizes", [[3, 0, 5, 1], [0, 0, 4], [7], [2, 2, 2, 2, 2]])
def test_grouped_exact_integer_blocks(sizes):
    rng = np.random.default_rng(sum(sizes) + len(sizes))
    N, K = 6, 5
    A, B, off = _int_grouped_case(rng, sizes, N, K)
    C = oracle.grouped(bf16_bits(A), bf16_bits(B), off)
    for g in range(len(sizes)):
        r0, r1 = off[g], off[g + 1]
        assert np.array_equal(C[r0:r1], A[r0:r1] @ B[g].T)
    assert not np.isnan(C).any()


def test_grouped_block_diagonal_equivalence():
    # grouped(A, B, off) == rows of the dense product A . [B_0; B_1; ...]^T
    # restricted to each group's own column block (block-diagonal selection).
    rng = np.random.default_rng(21)
    sizes = [4, 0, 3, 6]
    N, K = 5, 7
    A, B, off = _int_grouped_case(rng, sizes, N, K)
    C = oracle.grouped(bf16_bits(A), bf16_bits(B), off)
    full = A @ B.reshape(-1, K).T                     # [M_total, G*N]
    for g in range(len(sizes)):
        r0, r1 = off[g], off[g + 1]
        assert np.array_equal(C[r0:r1], full[r0:r1, g * N:(g + 1) * N])


def test_grouped_one_group_equals_dense_and_bias():
    rng = np.random.default_rng(22)
    A, B, off = _int_grouped_case(rng, [9], 4, 6)
    bias = small_ints(rng, (1, 4))
    C = oracle.grouped(bf16_bits(A), bf16_bits(B), off, bias=bf16_bits(bias), epi="bias")
    assert np.array_equal(C, A @ B[0].T + bias[0][None, :])


def test_grouped_rejects_bad_offsets():
    rng = np.random.default_rng(23)
    A, B, off = _int_grouped_case(rng, [2, 2], 3, 3)
    for bad in ([0, 3, 2], [1, 2, 4], [0, 2, 3]):
        with pytest.raises(ValueError):
            oracle.grouped(bf16_bits(A), bf16_bits(B), bad)


# ----------------------------------------------------------------------------
# IKBO linear compression
# ----------------------------------------------------------------------------
def _int_ikbo_case(rng, counts, Du, Dc, D, O):
    users = len(counts)
    off = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    U = small_ints(rng, (users, Du, D), -4, 4)
    C = small_ints(rng, (int(off[-1]), Dc, D), -4, 4)
    W = small_ints(rng, (O, Du + Dc), -4, 4)
    return U, C, W, off


@pytest.mark.parametrize("counts", [[3, 1, 2], [0, 4, 0, 1], [1]])
def test_ikbo_exact_integer_einsum(counts):
    rng = np.random.default_rng(len(counts) * 7 + sum(counts))
    Du, Dc, D, O = 6, 3, 5, 4
    U, C, W, off = _int_ikbo_case(rng, counts, Du, Dc, D, O)
    Y = oracle.ikbo(bf16_bits(U), bf16_bits(C), bf16_bits(W), off)
    user = np.repeat(np.arange(len(counts)), counts)
    X = np.concatenate([U[user], C], axis=1)          # [cand, Du+Dc, D]
    ref = np.einsum("of,cfd->cod", W.astype(np.int64), X.astype(np.int64))
    assert np.array_equal(Y, ref.astype(np.float64))


def test_ikbo_materialised_equals_decomposed():
    g = torch.Generator().manual_seed(31)
    users, Du, Dc, D, O = 3, 16, 8, 12, 5
    counts = [2, 0, 3]
    off = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    U = torch.randn(users, Du, D, generator=g).to(torch.bfloat16)
    C = torch.randn(int(off[-1]), Dc, D, generator=g).to(torch.bfloat16)
    W = torch.randn(O, Du + Dc, generator=g).to(torch.bfloat16)
    Y1 = oracle.ikbo(U, C, W, off)
    Y2 = oracle.ikbo_decomposed(U, C, W, off)
    scale = (U.float().abs().max() * W.float().abs().max()).item() * (Du + Dc)
    np.testing.assert_allclose(Y1, Y2, rtol=0, atol=1e-13 * scale)


def test_ikbo_zero_user_reduces_to_candidate_gemm():
    # U = 0  =>  Y[c] = W[:, Du:] . C[c]  (a plain GEMM per candidate)
    g = torch.Generator().manual_seed(32)
    users, Du, Dc, D, O = 2, 8, 4, 6, 3
    counts = [2, 1]
    off = np.array([0, 2, 3], dtype=np.int32)
    U = torch.zeros(users, Du, D).to(torch.bfloat16)
    C = torch.randn(3, Dc, D, generator=g).to(torch.bfloat16)
    W = torch.randn(O, Du + Dc, generator=g).to(torch.bfloat16)
    Y = oracle.ikbo(U, C, W, off)
    Wc = W[:, Du:].contiguous()
    for c in range(3):
        # C[c] is [Dc, D]; the gemm oracle takes B as [N, K] = [D, Dc]
        ref = oracle.gemm(Wc, C[c].t().contiguous())
        assert np.array_equal(Y[c], ref)


def test_ikbo_candidate_sample_and_bad_offsets():
    rng = np.random.default_rng(33)
    U, C, W, off = _int_ikbo_case(rng, [2, 2], 4, 2, 3, 2)
    full = oracle.ikbo(bf16_bits(U), bf16_bits(C), bf16_bits(W), off)
    part = oracle.ikbo(bf16_bits(U), bf16_bits(C), bf16_bits(W), off, cands=[3, 1])
    assert np.array_equal(part[[1, 3]], full[[1, 3]])
    assert np.isnan(part[[0, 2]]).all()
    with pytest.raises(ValueError):
        oracle.ikbo(bf16_bits(U), bf16_bits(C), bf16_bits(W), [0, 3, 2])


# ----------------------------------------------------------------------------
# GEMM on RMS-normalised rows of A
# ----------------------------------------------------------------------------
def test_rmsnorm_constant_rows_closed_form():
    # A row of constant value c has mean square c^2, so with eps = 0 the
    # normalised row is sign(c) * 1 and C[m][n] = sign(c) * sum_k B[n][k].
    K = 16
    u = np.array([2.0, -0.5, 4.0])
    A = np.repeat(u[:, None], K, axis=1)
    rng = np.random.default_rng(61)
    B = small_ints(rng, (5, K))
    C = oracle.gemm_rmsnorm(bf16_bits(A), bf16_bits(B), eps=0.0)
    ref = np.sign(u)[:, None] * B.sum(axis=1)[None, :]
    np.testing.assert_allclose(C, ref, rtol=1e-15, atol=0)


def test_rmsnorm_scale_invariance_and_unit_rows():
    g = torch.Generator().manual_seed(62)
    A = torch.randn(6, 32, generator=g).to(torch.bfloat16)
    B = torch.randn(7, 32, generator=g).to(torch.bfloat16)
    C1 = oracle.gemm_rmsnorm(A, B, eps=0.0)
    # scaling rows by powers of two is exact in bf16 and leaves C unchanged at eps = 0
    scale = torch.tensor([1, 2, 4, 0.5, 8, 0.25]).to(torch.bfloat16)[:, None]
    C2 = oracle.gemm_rmsnorm((A.float() * scale.float()).to(torch.bfloat16), B, eps=0.0)
    np.testing.assert_allclose(C1, C2, rtol=1e-13, atol=1e-13)
    # rows of +-1 have unit RMS: the normalised GEMM equals the plain GEMM
    S = torch.where(torch.randn(6, 32, generator=g) > 0, 1.0, -1.0).to(torch.bfloat16)
    np.testing.assert_allclose(oracle.gemm_rmsnorm(S, B, eps=0.0), oracle.gemm(S, B),
                               rtol=1e-15, atol=1e-15)


def test_rmsnorm_eps_and_epilogue():
    # A = 0: r = 1/sqrt(eps) multiplies a zero product; the output is the (SiLU of the) bias
    A = np.zeros((2, 8))
    B = np.ones((3, 8))
    bias = np.array([1.0, -2.0, 0.5])
    C = oracle.gemm_rmsnorm(bf16_bits(A), bf16_bits(B), eps=1e-6, bias=bf16_bits(bias), epi="bias")
    assert np.array_equal(C, np.tile(bias, (2, 1)))
    # large eps: r ~ 1/sqrt(eps), so C ~ (A.B^T)/sqrt(eps)
    rng = np.random.default_rng(63)
    A = small_ints(rng, (3, 8), -2, 2)
    B = small_ints(rng, (4, 8), -2, 2)
    C = oracle.gemm_rmsnorm(bf16_bits(A), bf16_bits(B), eps=1e12)
    np.testing.assert_allclose(C, (A @ B.T) / 1e6, rtol=1e-9, atol=1e-15)


# ----------------------------------------------------------------------------
# GEMM on LayerNorm-normalised rows of A
# ----------------------------------------------------------------------------
def test_layernorm_alternating_rows_closed_form():
    # Row m = c_m + d_m * (+1, -1, +1, -1, ...): mean c_m, variance d_m^2, so
    # the normalised row is (+-1) * d_m / sqrt(d_m^2 + eps), whatever c_m.
    K = 16
    sign = np.where(np.arange(K) % 2 == 0, 1.0, -1.0)
    c = np.array([0.0, 3.0, -5.0, 100.0])
    d = np.array([1.0, 2.0, 0.5, 4.0])
    A = c[:, None] + d[:, None] * sign[None, :]
    rng = np.random.default_rng(64)
    B = small_ints(rng, (5, K))
    for eps in (0.0, 0.25):
        C = oracle.gemm_layernorm(bf16_bits(A), bf16_bits(B), eps=eps)
        ref = (d / np.sqrt(d * d + eps))[:, None] * (B @ sign)[None, :]
        np.testing.assert_allclose(C, ref, rtol=1e-13, atol=1e-13)


def test_layernorm_shift_and_scale_invariance():
    # Adding a constant to a row changes nothing; scaling it by a power of two
    # changes nothing at eps = 0 (both exact in bf16 for these values).
    g = torch.Generator().manual_seed(65)
    A = torch.randint(-8, 9, (6, 32), generator=g).float()
    B = torch.randn(7, 32, generator=g).to(torch.bfloat16)
    C1 = oracle.gemm_layernorm(A.to(torch.bfloat16), B, eps=0.0)
    shift = torch.tensor([0.0, 16.0, -32.0, 64.0, 3.0, -7.0])[:, None]
    C2 = oracle.gemm_layernorm((A + shift).to(torch.bfloat16), B, eps=0.0)
    np.testing.assert_allclose(C1, C2, rtol=1e-12, atol=1e-12)
    scale = torch.tensor([1, 2, 4, 0.5, 8, 0.25])[:, None]
    C3 = oracle.gemm_layernorm((A * scale).to(torch.bfloat16), B, eps=0.0)
    np.testing.assert_allclose(C1, C3, rtol=1e-12, atol=1e-12)


def test_layernorm_constant_rows_and_zero_mean_rows():
    # A constant row normalises to zero: the output is exactly the (activated) bias.
    A = np.full((2, 8), 3.0)
    B = np.ones((3, 8))
    bias = np.array([1.0, -2.0, 0.5])
    C = oracle.gemm_layernorm(bf16_bits(A), bf16_bits(B), eps=1e-5, bias=bf16_bits(bias), epi="bias")
    assert np.array_equal(C, np.tile(bias, (2, 1)))
    # Rows with zero mean: LayerNorm is RMSNorm (two independent codings).
    g = torch.Generator().manual_seed(66)
    half = torch.randn(4, 12, generator=g)
    Z = torch.cat([half, -half], dim=1).to(torch.bfloat16)   # each row sums to zero exactly
    Bz = torch.randn(5, 24, generator=g).to(torch.bfloat16)
    np.testing.assert_allclose(oracle.gemm_layernorm(Z, Bz, eps=1e-3),
                               oracle.gemm_rmsnorm(Z, Bz, eps=1e-3), rtol=1e-12, atol=1e-12)
