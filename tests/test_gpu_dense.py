"""GPU parity: dense / strided-batched GEMM (through the C ABI) vs the fp64 oracle."""
import numpy as np
import pytest
import torch

import oracle
import synthetic
from gpu_util import amax, assert_parity, dense_run

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def wst():
    import warp_specialized_tensor_gb300 as w
    w.load_library()
    return w


def test_dense256_fp32_out(wst):
    d = synthetic.workload("dense256")
    C = dense_run(wst, d["A"], d["B"], torch.float32)
    ref = oracle.gemm(d["A"], d["B"])
    assert_parity(C, ref, 256, amax(d["A"]), amax(d["B"]), False, what="dense256")


def test_identity_operand_exact(wst):
    # A . I = A exactly (fp32 output): pins descriptor layout / transposition.
    K = 192
    A = synthetic.dense(256, 8, K, seed=7, dist="uniform")["A"]
    B = torch.eye(K, dtype=torch.float32).to(torch.bfloat16)  # N = K
    C = dense_run(wst, A, B, torch.float32)
    assert torch.equal(C.cpu(), A.float()), "A . I != A"
    # permutation of columns
    perm = torch.randperm(K, generator=torch.Generator().manual_seed(1))
    P = torch.eye(K)[perm].to(torch.bfloat16)
    C = dense_run(wst, A, P, torch.float32)
    assert torch.equal(C.cpu(), A.float()[:, perm])


@pytest.mark.parametrize("M,N,K,out", [
    (128, 256, 64, torch.bfloat16),     # exactly one tile, one K-block
    (300, 520, 200, torch.bfloat16),    # ragged M, N and K tails
    (1, 8, 8, torch.float32),           # degenerate
    (513, 264, 1000, torch.float32),    # several tiles, ragged everything
    (1024, 1024, 512, torch.bfloat16),  # 32 tiles, 8 K-blocks
])
def test_dense_shapes(wst, M, N, K, out):
    d = synthetic.dense(M, N, K, seed=M + N + K)
    C = dense_run(wst, d["A"], d["B"], out)
    ref = oracle.gemm(d["A"], d["B"])
    assert_parity(C, ref, K, amax(d["A"]), amax(d["B"]), out == torch.bfloat16,
                  what="dense %dx%dx%d" % (M, N, K))


def test_dense_padded_leading_dims(wst):
    # N = 257 needs a padded ldc (16-byte rule); A and B with padded rows too.
    M, N, K = 257, 257, 136
    d = synthetic.dense(M, N, K, seed=3)
    Ab = torch.zeros(M, K + 8, dtype=torch.bfloat16)
    Ab[:, :K] = d["A"]
    Bb = torch.zeros(N, K + 24, dtype=torch.bfloat16)
    Bb[:, :K] = d["B"]
    dA, dB = Ab.cuda()[:, :K], Bb.cuda()[:, :K]
    Cb = torch.full((M, 264), float("nan"), dtype=torch.bfloat16, device="cuda")
    C = Cb[:, :N]
    ws = wst.workspace()
    wst.wst_gemm_bf16(dA, dB, C, workspace=ws)
    assert wst.wst_sync_status(ws) == 0
    ref = oracle.gemm(d["A"], d["B"])
    assert_parity(C, ref, K, amax(d["A"]), amax(d["B"]), True, what="padded")
    assert torch.isnan(Cb[:, N:].float()).all(), "padding columns were written"


def test_dense_k_tail_with_nan_padding(wst):
    # K = 100 is not a multiple of 8: the rows are padded to 104 elements and
    # the padding holds NaN, which must never enter the sums.
    M, N, K, ld = 200, 136, 100, 104
    d = synthetic.dense(M, N, K, seed=12)
    Ab = torch.full((M, ld), float("nan"), dtype=torch.bfloat16)
    Ab[:, :K] = d["A"]
    Bb = torch.full((N, ld), float("nan"), dtype=torch.bfloat16)
    Bb[:, :K] = d["B"]
    C = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
    ws = wst.workspace()
    wst.wst_gemm_bf16(Ab.cuda()[:, :K], Bb.cuda()[:, :K], C, workspace=ws)
    assert wst.wst_sync_status(ws) == 0
    ref = oracle.gemm(d["A"], d["B"])
    assert_parity(C, ref, K, amax(d["A"]), amax(d["B"]), False, what="K tail")


@pytest.mark.parametrize("epi", ["bias", "bias_silu", "bias_gelu"])
@pytest.mark.parametrize("out", [torch.bfloat16, torch.float32])
def test_batched_epilogues(wst, epi, out):
    # the skinny recsys batch, scaled down: 6 GEMMs of 300 x 256 x 512
    d = synthetic.dense(300, 256, 512, batch=6, seed=1004, bias=True)
    C = dense_run(wst, d["A"], d["B"], out, bias=d["bias"], epi=epi)
    ref = oracle.gemm(d["A"], d["B"], bias=d["bias"], epi=epi)
    assert_parity(C, ref, 512, amax(d["A"]), amax(d["B"]), out == torch.bfloat16,
                  what="batched %s" % epi)


def test_batched_shared_operand_and_bias(wst):
    d = synthetic.dense(200, 136, 264, batch=3, seed=9, bias=True)
    B2 = d["B"][1].contiguous()       # one B shared by the batch
    b1 = d["bias"][2].contiguous()    # one bias row shared by the batch
    C = dense_run(wst, d["A"], B2, torch.bfloat16, bias=b1, epi="bias_silu")
    ref = oracle.gemm(d["A"], B2, bias=b1, epi="bias_silu")
    assert_parity(C, ref, 264, amax(d["A"]), amax(B2), True, what="shared B/bias")


def test_skinny_batch_full_size_every_gemm(wst):
    # All 512 GEMMs (1024 x 256 x 512, bias + SiLU) element by element.
    d = synthetic.workload("skinny_batch")
    C = dense_run(wst, d["A"], d["B"], torch.bfloat16, bias=d["bias"], epi="bias_silu")
    ref = oracle.gemm(d["A"], d["B"], bias=d["bias"], epi="bias_silu")
    assert_parity(C, ref, 512, amax(d["A"]), amax(d["B"]), True, what="skinny batch")


def test_dense8192_full_size_sampled_rows(wst):
    # 512 rows: 16 in every one of the 32 row tiles of 256 (CTA pairs), at
    # offsets that differ between tiles and cover both CTAs' 128-row halves,
    # plus the first and last row; all 8192 columns of each.
    d = synthetic.workload("dense8192")
    C = dense_run(wst, d["A"], d["B"], torch.bfloat16)
    rows = sorted({t * 256 + j * 16 + (t * 5) % 16 for t in range(32) for j in range(16)} |
                  {0, 8191})
    ref = oracle.gemm(d["A"], d["B"], rows=rows)
    assert_parity(C.cpu()[rows], ref[rows], 8192, amax(d["A"]), amax(d["B"]), True,
                  what="dense8192 rows")


def test_repeated_calls_same_workspace(wst):
    d = synthetic.dense(256, 256, 128, seed=11)
    ws = wst.workspace()
    ref = oracle.gemm(d["A"], d["B"])
    for _ in range(3):
        C = dense_run(wst, d["A"], d["B"], torch.float32, ws=ws)
        assert_parity(C, ref, 128, amax(d["A"]), amax(d["B"]), False, what="repeat")


@pytest.mark.parametrize("cg", [1, 2])
def test_dense_cta_group_forced(wst, cg):
    # The 1-CTA tile path for shapes that would otherwise use CTA pairs, and
    # the pair path for a shape of at most 128 rows, chosen through the
    # process-wide option WST_OPT_DENSE_CTA_GROUP.
    shape = (300, 264, 200) if cg == 1 else (100, 264, 200)
    d = synthetic.dense(*shape, batch=3, seed=31 + cg, bias=True)
    with wst.option(wst.OPT_DENSE_CTA_GROUP, cg):
        C = dense_run(wst, d["A"], d["B"], torch.bfloat16, bias=d["bias"], epi="bias_silu")
    ref = oracle.gemm(d["A"], d["B"], bias=d["bias"], epi="bias_silu")
    assert_parity(C, ref, 200, amax(d["A"]), amax(d["B"]), True, what="CTA group %d forced" % cg)


@pytest.mark.parametrize("epi", ["bias_silu", "bias_gelu"])
def test_single_cta_activation_ragged(wst, epi):
    # M <= 128 runs on single-CTA tiles; N and K ragged
    d = synthetic.dense(100, 520, 200, seed=1010, bias=True, batch=1)
    C = dense_run(wst, d["A"], d["B"], torch.float32, bias=d["bias"], epi=epi)
    ref = oracle.gemm(d["A"], d["B"], bias=d["bias"], epi=epi)
    assert_parity(C, ref, 200, amax(d["A"]), amax(d["B"]), False, what="single-CTA %s" % epi)
