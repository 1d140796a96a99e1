"""Pins of the IKBO attention oracle against closed forms and invariants.

The reading pinned here (the pages name IKBO FlashAttention but print no
formula): every query row q of candidate c attends over the keys/values of
its user u, per head: o = sum_j softmax_j(scale * q . k_j) v_j, no mask.
Each pin is chosen so that a plausible slip in the oracle (a dropped term, a
wrong sign, a swapped index, a wrong scale, a transposed operand) fails it.
"""
import math

import numpy as np
import pytest
import torch

import oracle


def bf16(x):
    return torch.as_tensor(np.asarray(x, dtype=np.float32)).to(torch.bfloat16)


def widen(t):
    return t.float().double().numpy()


def make(users_counts, Lq, H, Dh, Lkv, seed, dist="normal"):
    g = torch.Generator().manual_seed(seed)
    nc = sum(users_counts)
    shape_q = (nc * Lq, H, Dh)
    shape_kv = (len(users_counts), Lkv, H, Dh)
    if dist == "int":
        Q = torch.randint(-3, 4, shape_q, generator=g).to(torch.bfloat16)
        K = torch.randint(-3, 4, shape_kv, generator=g).to(torch.bfloat16)
        V = torch.randint(-8, 9, shape_kv, generator=g).to(torch.bfloat16)
    else:
        Q = torch.randn(shape_q, generator=g).to(torch.bfloat16)
        K = torch.randn(shape_kv, generator=g).to(torch.bfloat16)
        V = torch.randn(shape_kv, generator=g).to(torch.bfloat16)
    off = np.concatenate([[0], np.cumsum(users_counts)]).astype(np.int32)
    return Q, K, V, off


def both(Q, K, V, off, Lq, scale=None):
    a = oracle.ikbo_attention(Q, K, V, off, Lq, scale)
    b = oracle.ikbo_attention_grouped(Q, K, V, off, Lq, scale)
    return a, b


def owner_rows(off, Lq):
    """user index of every query row"""
    return np.repeat(np.arange(len(off) - 1), np.diff(off) * Lq)


def test_single_key_returns_its_value():
    Q, K, V, off = make([3, 0, 2], Lq=2, H=2, Dh=16, Lkv=1, seed=1)
    for O in both(Q, K, V, off, 2):
        u = owner_rows(off, 2)
        assert np.array_equal(O, widen(V)[u, 0])


def test_zero_query_averages_values():
    Q, K, V, off = make([2, 3], Lq=1, H=3, Dh=8, Lkv=7, seed=2)
    Q = torch.zeros_like(Q)
    mean = widen(V).mean(axis=1)  # [users, H, Dh]
    for O in both(Q, K, V, off, 1):
        np.testing.assert_allclose(O, mean[owner_rows(off, 1)], rtol=0, atol=1e-14)


def test_identical_keys_average_values_whatever_the_query():
    Q, K, V, off = make([4, 1], Lq=3, H=1, Dh=8, Lkv=5, seed=3)
    K = K[:, :1].expand(-1, 5, -1, -1).contiguous()
    mean = widen(V).mean(axis=1)
    for O in both(Q, K, V, off, 3):
        np.testing.assert_allclose(O, mean[owner_rows(off, 3)], rtol=0, atol=1e-14)


def test_two_keys_logistic_closed_form():
    # Small-integer q, k: every dot product is exact; with two keys the
    # softmax is the logistic function of the logit difference.
    Q, K, V, off = make([2, 2], Lq=1, H=2, Dh=8, Lkv=2, seed=4, dist="int")
    scale = 0.37
    q, k, v = widen(Q), widen(K), widen(V)
    u = owner_rows(off, 1)
    for O in both(Q, K, V, off, 1, scale):
        for r in range(q.shape[0]):
            for h in range(2):
                d = scale * (q[r, h] @ (k[u[r], 0, h] - k[u[r], 1, h]))
                p0 = 1.0 / (1.0 + math.exp(-d))
                want = p0 * v[u[r], 0, h] + (1.0 - p0) * v[u[r], 1, h]
                np.testing.assert_allclose(O[r, h], want, rtol=0, atol=1e-13)


def test_one_hot_values_expose_probabilities():
    # V[u, j] = e_j: the output row is the probability vector itself.  The
    # probabilities sum to one and their log-ratios are the scaled logit
    # differences scale * q . (k_0 - k_j) (exact for integer q, k).
    Lkv, Dh, scale = 6, 16, 0.25
    Q, K, _, off = make([3, 2], Lq=2, H=2, Dh=Dh, Lkv=Lkv, seed=5, dist="int")
    eye = np.zeros((2, Lkv, 2, Dh), np.float32)
    for j in range(Lkv):
        eye[:, j, :, j] = 1.0
    V = bf16(eye)
    q, k = widen(Q), widen(K)
    u = owner_rows(off, 2)
    for O in both(Q, K, V, off, 2, scale):
        p = O[..., :Lkv]
        assert (p > 0).all()
        np.testing.assert_allclose(p.sum(-1), 1.0, rtol=0, atol=1e-14)
        assert np.array_equal(O[..., Lkv:], np.zeros_like(O[..., Lkv:]))
        for r in range(q.shape[0]):
            for h in range(2):
                for j in range(1, Lkv):
                    want = scale * (q[r, h] @ (k[u[r], 0, h] - k[u[r], j, h]))
                    got = math.log(p[r, h, 0] / p[r, h, j])
                    assert abs(got - want) < 1e-12


def test_joint_key_value_permutation_is_invisible():
    Q, K, V, off = make([2, 3], Lq=2, H=2, Dh=8, Lkv=9, seed=6)
    perm = torch.randperm(9, generator=torch.Generator().manual_seed(7))
    a = oracle.ikbo_attention(Q, K, V, off, 2)
    b = oracle.ikbo_attention(Q, K[:, perm].contiguous(), V[:, perm].contiguous(), off, 2)
    np.testing.assert_allclose(a, b, rtol=0, atol=1e-13)
    # permuting only the values must change the result
    c = oracle.ikbo_attention(Q, K, V[:, perm].contiguous(), off, 2)
    assert np.abs(a - c).max() > 1e-3


def test_linear_in_the_values():
    Q, K, V1, off = make([2, 2], Lq=1, H=2, Dh=8, Lkv=5, seed=8, dist="int")
    V2 = torch.randint(-8, 9, V1.shape, generator=torch.Generator().manual_seed(9)).to(torch.bfloat16)
    Vs = (V1.float() + V2.float()).to(torch.bfloat16)  # exact: small integers
    assert torch.equal(Vs.float(), V1.float() + V2.float())
    a = oracle.ikbo_attention(Q, K, V1, off, 1)
    b = oracle.ikbo_attention(Q, K, V2, off, 1)
    c = oracle.ikbo_attention(Q, K, Vs, off, 1)
    np.testing.assert_allclose(a + b, c, rtol=0, atol=1e-12)


def test_candidates_see_only_their_users_context():
    # Two candidates with the same queries: equal outputs under one user,
    # different outputs under different users.
    Q, K, V, off = make([2, 1], Lq=2, H=1, Dh=8, Lkv=4, seed=10)
    Q[2:4] = Q[0:2]          # candidate 1 (user 0) copies candidate 0 (user 0)
    Q[4:6] = Q[0:2]          # candidate 2 (user 1) too
    for O in both(Q, K, V, off, 2):
        assert np.array_equal(O[0:2], O[2:4])
        assert np.abs(O[0:2] - O[4:6]).max() > 1e-3


def test_large_scale_is_hard_attention():
    Q, K, V, off = make([2, 2], Lq=1, H=1, Dh=8, Lkv=6, seed=11, dist="int")
    q, k, v = widen(Q), widen(K), widen(V)
    u = owner_rows(off, 1)
    O = oracle.ikbo_attention(Q, K, V, off, 1, scale=1e4)
    for r in range(q.shape[0]):
        s = k[u[r], :, 0] @ q[r, 0]
        if np.sort(s)[-1] - np.sort(s)[-2] < 1.0:
            continue  # tie: no unique winner
        np.testing.assert_allclose(O[r, 0], v[u[r], int(np.argmax(s)), 0], rtol=0, atol=1e-12)


def test_materialised_equals_grouped_coding():
    Q, K, V, off = make([5, 0, 3, 1], Lq=3, H=2, Dh=32, Lkv=37, seed=12)
    a, b = both(Q, K, V, off, 3, scale=0.2)
    assert not np.isnan(a).any()
    np.testing.assert_allclose(a, b, rtol=0, atol=1e-12)


def test_candidate_sample_matches_full():
    Q, K, V, off = make([4, 4], Lq=2, H=2, Dh=16, Lkv=10, seed=13)
    full = oracle.ikbo_attention(Q, K, V, off, 2)
    part = oracle.ikbo_attention(Q, K, V, off, 2, cands=[1, 6])
    rows = [2, 3, 12, 13]
    assert np.array_equal(part[rows], full[rows])
    assert np.isnan(np.delete(part, rows, axis=0)).all()


def test_bad_offsets_rejected():
    Q, K, V, off = make([2, 2], Lq=1, H=1, Dh=8, Lkv=3, seed=14)
    with pytest.raises(ValueError):
        oracle.ikbo_attention(Q, K, V, np.array([0, 3, 2], np.int32), 1)
    with pytest.raises(ValueError):
        oracle.ikbo_attention_grouped(Q, K, V, np.array([0, 1, 3], np.int32), 1)
