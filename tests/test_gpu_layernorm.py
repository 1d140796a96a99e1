"""GPU parity: GEMM on LayerNorm-normalised rows of A (the norm applied in
the GEMM's epilogue, column sums of B from a first kernel) vs the fp64
oracle, with the row statistics gathered in the GEMM from the A tiles and
with them taken by a separate pass over A (every test runs under both).

Tolerance: the general GEMM bound of oracle.compare applied to the
contraction the definition states, C = x_hat . B^T with the normalised rows
x_hat = (A - mu) / sqrt(var + eps): s = sqrt(K) max|x_hat| max|B| (plus one
bf16 ulp of the oracle for bf16 output).  It does not depend on how large a
row's mean is against its spread, so rows with means of hundreds of spreads
(where a one-pass E[a^2] - mu^2 variance in fp32 would cancel) must meet the
same bound as centred ones.
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


@pytest.fixture(autouse=True, params=["fused", "pass"])
def stats(request, wst):
    mode = wst.NORM_STATS_FUSED if request.param == "fused" else wst.NORM_STATS_PASS
    with wst.option(wst.OPT_NORM_STATS, mode):
        yield request.param


def shifted_rows(M, N, K, batch=0, seed=0, bias=False, shared_b=False, spreads=(-4.0, 4.0)):
    """Rows of A with their own spread 2^e (e in [-3, 3]) and a mean drawn
    uniformly from spreads[0]..spreads[1] times the spread, with a random
    sign when the range is positive (so both halves of the normalisation
    matter)."""
    d = synthetic.dense(M, N, K, batch=batch, seed=seed, bias=bias)
    g = torch.Generator().manual_seed(seed + 1)
    lead = (batch,) if batch else ()
    sig = torch.exp2(torch.randint(-3, 4, lead + (M, 1), generator=g).float())
    lo, hi = spreads
    mu = sig * (torch.rand(lead + (M, 1), generator=g) * (hi - lo) + lo)
    if lo >= 0:
        mu = mu * (torch.randint(0, 2, lead + (M, 1), generator=g).float() * 2 - 1)
    d["A"] = (d["A"].float() * K ** 0.5 * sig + mu).to(torch.bfloat16)
    if shared_b and batch:
        d["B"] = d["B"][0].contiguous()
        if bias:
            d["bias"] = d["bias"][0].contiguous()
    return d


def xhat_max(A, eps, rows=None):
    """max |x_hat| over the rows (fp64): the max|A| of the normalised operand."""
    a = A.float().numpy().astype(np.float64)
    if rows is not None:
        a = a[..., rows, :]
    mu = a.mean(axis=-1, keepdims=True)
    var = ((a - mu) ** 2).mean(axis=-1, keepdims=True)
    return float((np.abs(a - mu) / np.sqrt(var + eps)).max())


def run(wst, d, out, eps, epi="none", B=None):
    A = d["A"].cuda()
    B = d["B"].cuda() if B is None else B
    lead = (A.shape[0],) if A.dim() == 3 else ()
    C = torch.full(lead + (A.shape[-2], B.shape[-2]), float("nan"), dtype=out, device="cuda")
    bias = d["bias"].cuda() if epi != "none" else None
    ws = wst.norm_workspace(A, B, layernorm=True)
    wst.wst_gemm_layernorm_bf16(A, B, C, eps=eps, bias=bias, epi=epi, workspace=ws)
    assert wst.wst_sync_status(ws) == 0
    return C


def check(C, d, eps, K, epi="none", rows=None, B=None):
    B = d["B"] if B is None else B
    ref = oracle.gemm_layernorm(d["A"], B, eps=eps, bias=d.get("bias"), epi=epi, rows=rows)
    g = C.float().cpu().numpy()
    if rows is not None:
        g, ref = g[..., rows, :], ref[..., rows, :]
    ok, metric, detail = compare.check(g, ref, K, xhat_max(d["A"], eps, rows), amax(B),
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
    Av = Apad.cuda()[:, :K]
    C = torch.full((200, 132), float("nan"), device="cuda")
    ws = wst.norm_workspace(Av, Bv, layernorm=True)
    wst.wst_gemm_layernorm_bf16(Av, Bv, C, eps=1e-5, workspace=ws)
    assert wst.wst_sync_status(ws) == 0
    check(C, d, 1e-5, K)


def test_layernorm_batched_b_ragged_n(wst):
    # A batch stride on B and N = 101, not a multiple of 4: each batch
    # entry's column sums start on a padded row of 104 floats (the epilogue
    # reads them as float4), so entries past the first must land there.
    # C is a view with a padded row (ldc = 104) to meet the 16-byte rule.
    M, N, K = 200, 101, 256
    d = shifted_rows(M, N, K, batch=3, seed=88)
    A, B = d["A"].cuda(), d["B"].cuda()
    Cfull = torch.full((3, M, 104), float("nan"), device="cuda")
    C = Cfull[..., :N]
    ws = wst.norm_workspace(A, B, layernorm=True)
    wst.wst_gemm_layernorm_bf16(A, B, C, eps=1e-5, workspace=ws)
    assert wst.wst_sync_status(ws) == 0
    check(C, d, 1e-5, K)
    assert torch.isnan(Cfull[..., N:]).all()   # the padding is never written


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
    A, B = d["A"].cuda(), d["B"].cuda()
    ws = wst.norm_workspace(A, B)
    C_rms = torch.empty_like(C_ln)
    wst.wst_gemm_rmsnorm_bf16(A, B, C_rms, eps=1e-5, workspace=ws)
    assert wst.wst_sync_status(ws) == 0
    s = compare.scale(128, xhat_max(d["A"], 1e-5), amax(d["B"]))
    assert float((C_ln - C_rms).abs().max()) <= 1e-4 * s


def test_layernorm_dense8192_sampled_rows(wst):
    d = synthetic.workload("dense8192")
    g = torch.Generator().manual_seed(86)
    d = dict(d, A=(d["A"].float() + 0.05 * torch.randn(8192, 1, generator=g)).to(torch.bfloat16))
    C = run(wst, d, torch.bfloat16, 1e-5)
    rows = sorted(set(torch.randperm(8192, generator=g)[:12].tolist() + [0, 8191]))
    check(C, d, 1e-5, 8192, rows=rows)


@pytest.mark.parametrize("M,N,K,out", [
    (300, 264, 200, torch.float32),     # small K, CTA pairs, ragged
    (100, 72, 72, torch.bfloat16),      # single-CTA tile, ragged K block
    (256, 256, 8192, torch.float32),    # long rows
])
def test_layernorm_mean_far_above_spread(wst, M, N, K, out):
    # Row means of 256 to 288 row spreads (either sign): a one-pass fp32
    # variance E[a^2] - mu^2 would lose ~16 of its 24 bits here.  (Much
    # larger ratios stop meaning anything for bf16 rows: at 256 spreads the
    # bf16 spacing near the mean is already one to two spreads.)
    d = shifted_rows(M, N, K, seed=M + K + 7, spreads=(256.0, 288.0))
    C = run(wst, d, out, 1e-5)
    check(C, d, 1e-5, K)


def test_layernorm_pass_needs_workspace_room(wst, stats):
    # Column sums (one row of N floats) and then 8 bytes per row of A: the
    # minimal LayerNorm workspace holds only the sums, so the forced pass is
    # refused and the automatic choice keeps the statistics in the GEMM.
    d = shifted_rows(200, 1536, 256, seed=87)
    A, B = d["A"].cuda(), d["B"].cuda()
    C = torch.full((200, 1536), float("nan"), device="cuda")
    small = wst.layernorm_workspace(B)
    assert wst.wst_gemm_norm_workspace_size(1, 200, 1536, 0, 0, True) == 256 + 1536 * 4 + 200 * 8
    if stats == "pass":
        with pytest.raises(wst.WstError, match="precomputed statistics"):
            wst.wst_gemm_layernorm_bf16(A, B, C, eps=1e-5, workspace=small)
    with wst.option(wst.OPT_NORM_STATS, wst.NORM_STATS_AUTO):
        wst.wst_gemm_layernorm_bf16(A, B, C, eps=1e-5, workspace=small)
        assert wst.wst_sync_status(small) == 0
        check(C, d, 1e-5, 256)
        C2 = torch.full_like(C, float("nan"))
        ws = wst.norm_workspace(A, B, layernorm=True)
        wst.wst_gemm_layernorm_bf16(A, B, C2, eps=1e-5, workspace=ws)
        assert wst.wst_sync_status(ws) == 0
        check(C2, d, 1e-5, 256)
