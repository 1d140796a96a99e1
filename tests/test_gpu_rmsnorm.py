"""GPU parity: GEMM on RMS-normalised rows of A (the norm applied in the
GEMM's epilogue) vs the fp64 oracle, with the row statistics gathered in the
GEMM from the A tiles and with them taken by a separate pass over A (every
test runs under both forms)."""
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


def normed_max(A, eps, rows=None):
    """max |r_m A[m][k]| (fp64): the max|A| of the normalised operand the
    definition contracts, r_m = 1/sqrt(mean_k A[m][k]^2 + eps)."""
    a = A.float().numpy().astype(np.float64)
    if rows is not None:
        a = a[..., rows, :]
    r = 1.0 / np.sqrt((a * a).mean(axis=-1, keepdims=True) + eps)
    return float(np.abs(r * a).max())


def scaled_rows(M, N, K, batch=0, seed=0, bias=False):
    """Rows of A with very different magnitudes, so the normalisation matters."""
    d = synthetic.dense(M, N, K, batch=batch, seed=seed, bias=bias)
    g = torch.Generator().manual_seed(seed + 1)
    lead = (batch,) if batch else ()
    s = torch.exp2(torch.randint(-4, 5, lead + (M, 1), generator=g).float())
    d["A"] = (d["A"].float() * s).to(torch.bfloat16)
    return d


def run(wst, d, out, eps, epi="none"):
    A, B = d["A"].cuda(), d["B"].cuda()
    lead = (A.shape[0],) if A.dim() == 3 else ()
    C = torch.full(lead + (A.shape[-2], B.shape[-2]), float("nan"), dtype=out, device="cuda")
    bias = d["bias"].cuda() if epi != "none" else None
    ws = wst.norm_workspace(A, B)
    wst.wst_gemm_rmsnorm_bf16(A, B, C, eps=eps, bias=bias, epi=epi, workspace=ws)
    assert wst.wst_sync_status(ws) == 0
    return C


def check(C, d, eps, K, epi="none", rows=None):
    ref = oracle.gemm_rmsnorm(d["A"], d["B"], eps=eps, bias=d.get("bias"), epi=epi, rows=rows)
    g = C.float().cpu().numpy()
    if rows is not None:
        g, ref = g[..., rows, :], ref[..., rows, :]
    ok, metric, detail = compare.check(g, ref, K, normed_max(d["A"], eps, rows), amax(d["B"]),
                                       C.dtype == torch.bfloat16)
    assert ok, detail


@pytest.mark.parametrize("M,N,K,out", [
    (128, 256, 64, torch.float32),
    (300, 520, 200, torch.bfloat16),
    (513, 264, 1000, torch.float32),
    (1, 8, 8, torch.float32),
])
def test_rmsnorm_shapes(wst, M, N, K, out):
    d = scaled_rows(M, N, K, seed=M + N)
    C = run(wst, d, out, 1e-6)
    check(C, d, 1e-6, K)


@pytest.mark.parametrize("epi,out", [("bias", torch.float32), ("bias_silu", torch.bfloat16),
                                     ("bias_gelu", torch.bfloat16)])
def test_rmsnorm_batched_epilogue(wst, epi, out):
    d = scaled_rows(300, 256, 512, batch=4, seed=71, bias=True)
    C = run(wst, d, out, 1e-5, epi=epi)
    check(C, d, 1e-5, 512, epi=epi)


def test_rmsnorm_row_scale_invariance_bit_exact(wst):
    # With eps = 0, doubling a row of A (exact in bf16) must leave C unchanged.
    d = synthetic.dense(256, 256, 320, seed=72)
    C1 = run(wst, d, torch.float32, 0.0)
    d2 = dict(d)
    d2["A"] = (d["A"].float() * 2.0).to(torch.bfloat16)
    C2 = run(wst, d2, torch.float32, 0.0)
    assert torch.equal(C1, C2)


def test_rmsnorm_dense8192_sampled_rows(wst):
    d = synthetic.workload("dense8192")
    C = run(wst, d, torch.bfloat16, 1e-6)
    rows = sorted(set(torch.randperm(8192, generator=torch.Generator().manual_seed(9))[:12].tolist() + [0, 8191]))
    check(C, d, 1e-6, 8192, rows=rows)


def test_rmsnorm_pass_needs_workspace_room(wst, stats):
    # The separate statistics pass writes 8 bytes per row of A after the
    # header: forced, it refuses a workspace without that room; automatic,
    # the same call falls back to the in-GEMM statistics and matches.
    d = scaled_rows(256, 4096, 128, seed=73)
    A, B = d["A"].cuda(), d["B"].cuda()
    C = torch.full((256, 4096), float("nan"), device="cuda")
    small = wst.workspace()
    assert wst.wst_gemm_norm_workspace_size(1, 256, 4096) == 256 + 256 * 8
    if stats == "pass":
        with pytest.raises(wst.WstError, match="precomputed statistics"):
            wst.wst_gemm_rmsnorm_bf16(A, B, C, eps=1e-6, workspace=small)
    with wst.option(wst.OPT_NORM_STATS, wst.NORM_STATS_AUTO):
        wst.wst_gemm_rmsnorm_bf16(A, B, C, eps=1e-6, workspace=small)     # in the GEMM
        assert wst.wst_sync_status(small) == 0
        check(C, d, 1e-6, 128)
        C2 = torch.full_like(C, float("nan"))
        ws = wst.norm_workspace(A, B)
        wst.wst_gemm_rmsnorm_bf16(A, B, C2, eps=1e-6, workspace=ws)        # N > 2048: the pass
        assert wst.wst_sync_status(ws) == 0
        check(C2, d, 1e-6, 128)


@pytest.mark.parametrize("layernorm", [False, True])
def test_norm_shared_a_batched_b_through_abi(wst, stats, layernorm):
    # batch = 3 with strideA = 0 (one A shared by the batch) and a batched B,
    # through the C ABI (the Python binding takes the batch from A): the
    # separate pass then computes one batch's row statistics and every batch
    # entry's epilogue reads them.
    M, N, K, batch = 200, 256, 320, 3
    d = scaled_rows(M, N, K, seed=74)
    Bb = synthetic.dense(M, N, K, batch=batch, seed=75)["B"]
    A, B = d["A"].cuda(), Bb.cuda()
    C = torch.full((batch, M, N), float("nan"), device="cuda")
    nbytes = wst.wst_gemm_norm_workspace_size(batch, M, N, 0, B.stride(0), layernorm)
    assert nbytes == 256 + (batch * N * 4 if layernorm else 0) + M * 8
    ws = torch.zeros(nbytes, dtype=torch.uint8, device="cuda")
    lib = wst.load_library()
    fn = lib.wst_gemm_layernorm_bf16 if layernorm else lib.wst_gemm_rmsnorm_bf16
    st = fn(batch, M, N, K, A.data_ptr(), K, 0, B.data_ptr(), K, B.stride(0), 1e-5, None, 0,
            C.data_ptr(), N, M * N, wst.F32, wst.EPI_NONE, ws.data_ptr(), nbytes, None)
    assert st == 0, lib.wst_last_error()
    assert wst.wst_sync_status(ws) == 0
    A3 = d["A"].expand(batch, M, K).contiguous()
    ref = (oracle.gemm_layernorm if layernorm else oracle.gemm_rmsnorm)(A3, Bb, eps=1e-5)
    a = A3.float().numpy().astype(np.float64)
    if layernorm:
        mu = a.mean(axis=-1, keepdims=True)
        amax_n = float((np.abs(a - mu) / np.sqrt(((a - mu) ** 2).mean(axis=-1, keepdims=True) + 1e-5)).max())
    else:
        amax_n = normed_max(A3, 1e-5)
    ok, metric, detail = compare.check(C.cpu().numpy(), ref, K, amax_n, amax(Bb), False)
    assert ok, detail
