"""GPU parity: GEMM on LayerNorm-normalised rows of A (row statistics fused
into the GEMM, column sums of B from a first kernel) vs the fp64 oracle.

Tolerance: the general GEMM bound of oracle.compare with max|A| replaced by
max_m r_m max_k |A[m][k]| (r_m = 1/sqrt(var_m + eps)), which bounds both
the normalised operand and the mean term r mu s[n] that the kernel subtracts.
"""
import numpy as np
import pytest
import torch

import oracle
import synthetic
from gpu_util import amax
from oracle import compare

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def wst():
    import warp_specialized_tensor_gb300 as w
    w.load_library()
    return w


def shifted_rows(M, N, K, batch=0, seed=0, bias=False, shared_b=False):
    """Rows of A with their own spread 2^e (e in [-3, 3]) and a mean of up to
    four spreads, so that both halves of the normalisation matter."""
    d = synthetic.dense(M, N, K, batch=batch, seed=seed, bias=bias)
    g = torch.Generator().manual_seed(seed + 1)
    lead = (batch,) if batch else ()
    sig = torch.exp2(torch.randint(-3, 4, lead + (M, 1), generator=g).float())
    mu = sig * (torch.rand(lead + (M, 1), generator=g) * 8.0 - 4.0)
    d["A"] = (d["A"].float() * K ** 0.5 * sig + mu).to(torch.bfloat16)
    if shared_b and batch:
        d["B"] = d["B"][0].contiguous()
        if bias:
            d["bias"] = d["bias"][0].contiguous()
    return d


def a_eff(A, eps):
    a = A.float().numpy().astype(np.float64)
    var = a.var(axis=-1)
    r = 1.0 / np.sqrt(var + eps)
    return float((r * np.abs(a).max(axis=-1)).max())


def run(wst, d, out, eps, epi="none", B=None):
    A = d["A"].cuda()
    B = d["B"].cuda() if B is None else B
    lead = (A.shape[0],) if A.dim() == 3 else ()
    C = torch.full(lead + (A.shape[-2], B.shape[-2]), float("nan"), dtype=out, device="cuda")
    bias = d["bias"].cuda() if epi != "none" else None
    ws = wst.layernorm_workspace(B)
    wst.wst_gemm_layernorm_bf16(A, B, C, eps=eps, bias=bias, epi=epi, workspace=ws)
    assert wst.wst_sync_status(ws) == 0
    return C


def check(C, d, eps, K, epi="none", rows=None, B=None):
    B = d["B"] if B is None else B
    ref = oracle.gemm_layernorm(d["A"], B, eps=eps, bias=d.get("bias"), epi=epi, rows=rows)
    g = C.float().cpu().numpy()
    if rows is not None:
        g, ref = g[..., rows, :], ref[..., rows, :]
    ok, metric, detail = compare.check(g, ref, K, a_eff(d["A"], eps), amax(B),
                                       C.dtype == torch.bfloat16)
    assert ok, detail
    return metric


@pytest.mark.parametrize("M,N,K,out", [
    (128, 256, 64, torch.float32),     # one single-CTA tile
    (300, 520, 200, torch.bfloat16),   # CTA pairs, ragged M and N
    (513, 264, 1000, torch.float32),   # ragged everywhere, 16 K blocks
    (1, 8, 8, torch.float32),          # smallest
    (129, 40, 8, torch.bfloat16),      # one K block, N not a multiple of 32
])
def test_layernorm_shapes(wst, M, N, K, out):
    d = shifted_rows(M, N, K, seed=M + N + K)
    C = run(wst, d, out, 1e-5)
    check(C, d, 1e-5, K)


@pytest.mark.parametrize("shared_b", [False, True])
@pytest.mark.parametrize("epi,out", [("bias", torch.float32), ("bias_silu", torch.bfloat16),
                                     ("bias_gelu", torch.bfloat16)])
def test_layernorm_batched_epilogue(wst, epi, out, shared_b):
    d = shifted_rows(300, 264, 512, batch=3, seed=81, bias=True, shared_b=shared_b)
    C = run(wst, d, out, 1e-5, epi=epi)
    check(C, d, 1e-5, 512, epi=epi)


def test_layernorm_padded_rows(wst):
    # A and B rows with leading dimensions larger than K = 100, the padding
    # filled with 100.0, and K not a multiple of the column-sum kernel's
    # 8-element vectors: statistics and sums must read exactly K elements.
    K = 100
    d = shifted_rows(200, 132, K, seed=82)
    Apad = torch.full((200, 104), 100.0, dtype=torch.bfloat16)
    Apad[:, :K] = d["A"]
    Bpad = torch.full((132, 128), 100.0, dtype=torch.bfloat16)
    Bpad[:, :K] = d["B"]
    Bv = Bpad.cuda()[:, :K]
    C = torch.full((200, 132), float("nan"), device="cuda")
    ws = wst.layernorm_workspace(Bv)
    wst.wst_gemm_layernorm_bf16(Apad.cuda()[:, :K], Bv, C, eps=1e-5, workspace=ws)
    assert wst.wst_sync_status(ws) == 0
    check(C, d, 1e-5, K)


def test_layernorm_constant_rows(wst):
    # A constant row has zero variance: its normalised row is 0 and C is the
    # bias alone (the epilogue applied to it).
    d = shifted_rows(256, 128, 256, seed=83, bias=True)
    A = d["A"].float()
    A[5] = 2.0
    A[200] = -0.75
    d["A"] = A.to(torch.bfloat16)
    for eps in (1e-5, 1.0):
        C = run(wst, d, torch.float32, eps, epi="bias")
        check(C, d, eps, 256, epi="bias")


def test_layernorm_sign_and_scale_symmetry_bit_exact(wst):
    # LayerNorm(-a) = -LayerNorm(a) and, with eps = 0, LayerNorm(2a) =
    # LayerNorm(a); the kernel's arithmetic commutes with both exactly.
    d = shifted_rows(256, 256, 320, seed=84)
    C1 = run(wst, d, torch.float32, 0.0)
    dn = dict(d, A=(-d["A"].float()).to(torch.bfloat16))
    d2 = dict(d, A=(d["A"].float() * 2.0).to(torch.bfloat16))
    assert torch.equal(run(wst, dn, torch.float32, 0.0), -C1)
    assert torch.equal(run(wst, d2, torch.float32, 0.0), C1)


def test_layernorm_matches_rmsnorm_on_centred_rows(wst):
    # Rows whose bf16 values sum to exactly 0 (each value paired with its
    # negation): mean 0, so LayerNorm and RMSNorm agree up to rounding.
    d = synthetic.dense(256, 256, 128, seed=85)
    A = d["A"].float()
    A[:, 64:] = -A[:, :64]
    d["A"] = A.to(torch.bfloat16)
    C_ln = run(wst, d, torch.float32, 1e-5)
    ws = wst.workspace()
    C_rms = torch.empty_like(C_ln)
    wst.wst_gemm_rmsnorm_bf16(d["A"].cuda(), d["B"].cuda(), C_rms, eps=1e-5, workspace=ws)
    assert wst.wst_sync_status(ws) == 0
    s = compare.scale(128, a_eff(d["A"], 1e-5), amax(d["B"]))
    assert float((C_ln - C_rms).abs().max()) <= 1e-4 * s


def test_layernorm_dense8192_sampled_rows(wst):
    d = synthetic.workload("dense8192")
    g = torch.Generator().manual_seed(86)
    d = dict(d, A=(d["A"].float() + 0.05 * torch.randn(8192, 1, generator=g)).to(torch.bfloat16))
    C = run(wst, d, torch.bfloat16, 1e-5)
    rows = sorted(set(torch.randperm(8192, generator=g)[:12].tolist() + [0, 8191]))
    check(C, d, 1e-5, 8192, rows=rows)
