"""Seeded synthetic inputs shared by the tests, the smoke check and the benchmark.

This module holds NO arithmetic of the method: it only draws random numbers
(torch CPU generator, fp32 draws rounded to bf16 round-to-nearest-even) and
builds the routing / user-offset index arrays.  Both the CUDA path and the
CPU oracle consume exactly the bf16 bits produced here.

Workloads (sizes as named; every generator also takes smaller sizes for
parity cases):
  dense 256^3        A, B ~ U[-1, 1]; fp32 output          (seed 1000)
  dense 8192^3       A, B ~ N(0, 1)/sqrt(K); bf16 output   (seed 1001)
  grouped MoE        64 experts, 16384 tokens routed top-2 to distinct
                     experts uniformly at random, K=4096, N=1536 per expert,
                     N(0, 0.02); bf16 output               (seed 1002)
  IKBO               64 users x 128 candidates, U[64,256,128],
                     C[8192,64,128] ~ N(0,1), W[32,320] ~ N(0, 1/sqrt(320));
                     fp32 output                           (seed 1003)
  skinny batch       512 x (M=1024, N=256, K=512) ~ N(0,1)/sqrt(K),
                     bias ~ N(0, 0.1), bias+SiLU, bf16 out (seed 1004)
"""
from __future__ import annotations

import math

import torch

SEED_BASE = 1000


def _gen(seed: int) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    return g


def _normal(g, shape, std: float) -> torch.Tensor:
    x = torch.randn(*shape, generator=g, dtype=torch.float32)
    if std != 1.0:
        x.mul_(std)
    return x.to(torch.bfloat16)


def _uniform(g, shape, lo: float, hi: float) -> torch.Tensor:
    x = torch.rand(*shape, generator=g, dtype=torch.float32)
    x.mul_(hi - lo).add_(lo)
    return x.to(torch.bfloat16)


def dense(M: int, N: int, K: int, batch: int = 0, seed: int = SEED_BASE + 1,
          dist: str = "normal", bias: bool = False, bias_std: float = 0.1):
    """A [batch,M,K] (or [M,K] when batch == 0), B [batch,N,K] (K contiguous),
    optional bias [batch,N].  dist: 'normal' = N(0,1)/sqrt(K), 'uniform' =
    U[-1,1]."""
    g = _gen(seed)
    lead = (batch,) if batch else ()
    if dist == "normal":
        s = 1.0 / math.sqrt(K)
        A = _normal(g, lead + (M, K), s)
        B = _normal(g, lead + (N, K), s)
    elif dist == "uniform":
        A = _uniform(g, lead + (M, K), -1.0, 1.0)
        B = _uniform(g, lead + (N, K), -1.0, 1.0)
    else:
        raise ValueError(dist)
    out = {"A": A, "B": B}
    if bias:
        out["bias"] = _normal(g, lead + (N,), bias_std)
    return out


def top2_routing(tokens: int, experts: int, g: torch.Generator, k: int = 2):
    """Each token picks k DISTINCT experts uniformly at random.

    Returns (token_ids, offsets): token_ids[r] is the token whose features
    fill row r of the expert-sorted activation matrix (rows of expert e are
    [offsets[e], offsets[e+1]), tokens ascending within an expert)."""
    if k > experts:
        raise ValueError("k > experts")
    choice = torch.rand(tokens, experts, generator=g).argsort(dim=1)[:, :k]
    expert_of = choice.reshape(-1)                       # [tokens*k]
    token_of = torch.arange(tokens).repeat_interleave(k)  # [tokens*k]
    order = torch.argsort(expert_of * tokens + token_of)  # expert-major, token-minor
    counts = torch.bincount(expert_of, minlength=experts)
    offsets = torch.zeros(experts + 1, dtype=torch.int32)
    offsets[1:] = torch.cumsum(counts, 0).to(torch.int32)
    return token_of[order], offsets


def routing_table(tokens: int, experts: int, k: int, g: torch.Generator) -> torch.Tensor:
    """int32 [tokens, k]: each token's k DISTINCT experts, uniformly at random."""
    if k > experts:
        raise ValueError("k > experts")
    return torch.rand(tokens, experts, generator=g).argsort(dim=1)[:, :k].to(torch.int32).contiguous()


def moe_tokens(tokens: int, experts: int, K: int, N: int, topk: int = 2, std: float = 0.02,
               seed: int = SEED_BASE + 6):
    """Token-major MoE layer inputs (for the expert-parallel layout): X
    [tokens, K] bf16, routing int32 [tokens, topk] (distinct experts per
    token), B [experts, N, K] bf16 (K contiguous)."""
    g = _gen(seed)
    X = _normal(g, (tokens, K), std)
    routing = routing_table(tokens, experts, topk, g)
    B = _normal(g, (experts, N, K), std)
    return {"X": X, "routing": routing, "B": B}


def grouped(experts: int = 64, tokens: int = 16384, K: int = 4096, N: int = 1536,
            topk: int = 2, std: float = 0.02, seed: int = SEED_BASE + 2,
            group_sizes=None):
    """MoE expert up-projection inputs.

    A [sum M_g, K]: token features gathered in expert-sorted order (a token
    routed to two experts appears in both groups with the same features);
    B [experts, N, K] (K contiguous); offsets int32 [experts+1].
    ``group_sizes`` overrides the routing with explicit per-group row counts
    (rows then get fresh features), for edge cases such as empty groups."""
    g = _gen(seed)
    if group_sizes is None:
        X = _normal(g, (tokens, K), std)
        token_ids, offsets = top2_routing(tokens, experts, g, topk)
        A = X[token_ids].contiguous()
    else:
        sizes = torch.tensor(list(group_sizes), dtype=torch.int64)
        if sizes.numel() != experts or (sizes < 0).any():
            raise ValueError("group_sizes")
        offsets = torch.zeros(experts + 1, dtype=torch.int32)
        offsets[1:] = torch.cumsum(sizes, 0).to(torch.int32)
        A = _normal(g, (int(offsets[-1]), K), std)
    B = _normal(g, (experts, N, K), std)
    return {"A": A, "B": B, "offsets": offsets}


def ikbo(users: int = 64, cand_per_user=128, Du: int = 256, Dc: int = 64,
         D: int = 128, O: int = 32, seed: int = SEED_BASE + 3):
    """IKBO linear-compression inputs.

    cand_per_user: an int (same count for every user) or a list of counts
    (zeros allowed).  Candidates are contiguous per user; user_offsets int32
    [users+1]."""
    g = _gen(seed)
    if isinstance(cand_per_user, int):
        counts = [cand_per_user] * users
    else:
        counts = list(cand_per_user)
        if len(counts) != users:
            raise ValueError("cand_per_user")
    offsets = torch.zeros(users + 1, dtype=torch.int32)
    offsets[1:] = torch.cumsum(torch.tensor(counts, dtype=torch.int64), 0).to(torch.int32)
    ncand = int(offsets[-1])
    U = _normal(g, (users, Du, D), 1.0)
    C = _normal(g, (ncand, Dc, D), 1.0)
    W = _normal(g, (O, Du + Dc), 1.0 / math.sqrt(Du + Dc))
    return {"U": U, "C": C, "W": W, "user_offsets": offsets}


def ikbo_attention(users: int = 32, cand_per_user=256, Lq: int = 2, H: int = 4,
                   Dh: int = 128, Lkv: int = 2048, seed: int = SEED_BASE + 5):
    """IKBO attention inputs: every query row of a candidate attends over its
    user's context.

    Q [num_cand*Lq, H, Dh] (candidate c owns rows [c*Lq, (c+1)*Lq)), K and V
    [users, Lkv, H, Dh], all N(0, 1) in bf16; user_offsets int32 [users+1]
    over candidates (cand_per_user: an int or a list of counts, zeros
    allowed)."""
    g = _gen(seed)
    counts = [cand_per_user] * users if isinstance(cand_per_user, int) else list(cand_per_user)
    if len(counts) != users:
        raise ValueError("cand_per_user")
    offsets = torch.zeros(users + 1, dtype=torch.int32)
    offsets[1:] = torch.cumsum(torch.tensor(counts, dtype=torch.int64), 0).to(torch.int32)
    ncand = int(offsets[-1])
    Q = _normal(g, (ncand * Lq, H, Dh), 1.0)
    K = _normal(g, (users, Lkv, H, Dh), 1.0)
    V = _normal(g, (users, Lkv, H, Dh), 1.0)
    return {"Q": Q, "K": K, "V": V, "user_offsets": offsets, "Lq": Lq}


# The named workloads at full size.
def workload(name: str):
    if name == "dense256":
        return dense(256, 256, 256, seed=SEED_BASE + 0, dist="uniform")
    if name == "dense8192":
        return dense(8192, 8192, 8192, seed=SEED_BASE + 1)
    if name == "grouped_moe":
        return grouped(seed=SEED_BASE + 2)
    if name == "ikbo":
        return ikbo(seed=SEED_BASE + 3)
    if name == "skinny_batch":
        return dense(1024, 256, 512, batch=512, seed=SEED_BASE + 4, bias=True)
    if name == "ikbo_attention":
        return ikbo_attention(seed=SEED_BASE + 5)
    raise KeyError(name)


WORKLOADS = ("dense256", "dense8192", "grouped_moe", "ikbo", "skinny_batch", "ikbo_attention")
