"""GPU: the expert-parallel grouped GEMM at world size 1 (the whole path:
plans, the permute kernel for every row move, the grouped GEMM kernel),
checked against the oracle's grouped GEMM on the same problem; and the
permute kernel's index checks."""
import os
import sys

import numpy as np
import pytest
import torch

import synthetic
from oracle import compare

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, os.path.join(ROOT, "tests"))


@pytest.fixture(scope="module")
def wst():
    import warp_specialized_tensor_gb300 as w
    w.load_library()
    return w


@pytest.mark.parametrize("tokens,experts,K,N,k", [
    (300, 8, 256, 384, 2),     # ragged groups, N of 1.5 tiles
    (1000, 16, 136, 256, 3),   # K not a multiple of 64, top-3
    (5, 64, 64, 256, 2),       # most experts empty
])
def test_ep_world1_matches_oracle(wst, tokens, experts, K, N, k):
    from ep_ops import reference
    from warp_specialized_tensor_gb300.expert_parallel import ep_grouped_gemm
    d = synthetic.moe_tokens(tokens=tokens, experts=experts, K=K, N=N, topk=k, seed=tokens + K)
    out = ep_grouped_gemm(d["X"].cuda(), d["routing"], d["B"].cuda(), experts)
    torch.cuda.synchronize()
    ref = reference(d["X"], d["routing"], d["B"])
    amax = lambda t: float(t.float().abs().max())
    ok, metric, detail = compare.check(out.float().cpu().numpy(), ref, K, amax(d["X"]), amax(d["B"]),
                                       True)
    assert ok, detail


def test_permute_rows_gather_scatter_exact(wst):
    ws = wst.workspace()
    src = torch.randn(100, 72, device="cuda").to(torch.bfloat16)   # 144-byte rows
    idx = torch.randperm(100)[:60].to(torch.int32)
    dst = torch.zeros(60, 72, dtype=torch.bfloat16, device="cuda")
    wst.wst_permute_rows(src, dst, src_index=idx.cuda(), workspace=ws)
    assert wst.wst_sync_status(ws) == 0
    assert torch.equal(dst.cpu(), src.cpu()[idx.long()])
    back = torch.zeros(100, 72, dtype=torch.bfloat16, device="cuda")
    wst.wst_permute_rows(dst, back, dst_index=idx.cuda(), workspace=ws)
    assert wst.wst_sync_status(ws) == 0
    want = torch.zeros(100, 72, dtype=torch.bfloat16)
    want[idx.long()] = src.cpu()[idx.long()]
    assert torch.equal(back.cpu(), want)


def test_permute_rows_bad_index_latched(wst):
    # An index past the source's rows skips that row and latches
    # WST_ERR_INVALID_ARG; the other rows move.
    ws = wst.workspace()
    src = torch.arange(8 * 8, dtype=torch.float32, device="cuda").reshape(8, 8)
    dst = torch.full((3, 8), -1.0, device="cuda")
    idx = torch.tensor([2, 9, 0], dtype=torch.int32, device="cuda")
    wst.wst_permute_rows(src, dst, src_index=idx, workspace=ws)
    assert wst.wst_sync_status(ws) == wst.WST_ERR_INVALID_ARG
    d = dst.cpu()
    assert torch.equal(d[0], src.cpu()[2]) and torch.equal(d[2], src.cpu()[0])
    assert (d[1] == -1.0).all()
