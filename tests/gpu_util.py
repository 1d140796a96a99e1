"""Shared helpers for the GPU parity tests: move seeded inputs to the device,
run the oracle on the same bf16 bits, and assert the tolerance."""
import numpy as np
import torch

import oracle
from oracle import compare


def amax(*ts):
    return max(float(t.float().abs().max()) if t.numel() else 0.0 for t in ts)


def assert_parity(gpu, ref, K, a_max, b_max, out_bf16, mask=None, what=""):
    g = gpu.float().cpu().numpy() if isinstance(gpu, torch.Tensor) else gpu
    ok, metric, detail = compare.check(g, ref, K, a_max, b_max, out_bf16, mask=mask)
    assert ok, "%s parity failed: %s" % (what, detail)
    return metric


def dense_run(wst, A, B, out_dtype, bias=None, epi="none", ws=None):
    dA, dB = A.cuda(), B.cuda()
    M, N = A.shape[-2], B.shape[-2]
    lead = (A.shape[0],) if A.dim() == 3 else ()
    C = torch.full(lead + (M, N), float("nan"), dtype=out_dtype, device="cuda")
    dbias = bias.cuda() if bias is not None else None
    ws = ws if ws is not None else wst.workspace()
    wst.wst_gemm_bf16(dA, dB, C, bias=dbias, epi=epi, workspace=ws)
    assert wst.wst_sync_status(ws) == 0
    return C
