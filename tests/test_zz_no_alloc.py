"""GPU test of wst_ikbo_linear_compress_noalloc, the allocation-free IKBO entry point.

Callers that cannot allocate device memory at call time (a fixed memory
budget, an allocator they must not bypass, a host framework that owns every
allocation) use this form: its scratch lives in a fixed device array inside
the library.  This file is collected last so that a run stopping at the first
failure has already run every other test.  It must pass alone in a fresh
process and after the other tests.
"""
import ctypes

import numpy as np
import pytest
import torch

import synthetic
from oracle import compare

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    import warp_specialized_tensor_gb300 as w
    return w.load_library()


def _dev(d):
    return {k: v.cuda() for k, v in d.items()}


def _call_noalloc(lib, d, Y, status):
    U, C, W, off = d["U"], d["C"], d["W"], d["user_offsets"]
    users, Du, D = U.shape
    return lib.wst_ikbo_linear_compress_noalloc(
        users, C.shape[0], Du, C.shape[1], D, W.shape[0], U.data_ptr(), C.data_ptr(),
        W.data_ptr(), off.data_ptr(), Y.data_ptr(), status.data_ptr(),
        torch.cuda.current_stream().cuda_stream)


def _call_workspace(lib, d, Y, ws):
    U, C, W, off = d["U"], d["C"], d["W"], d["user_offsets"]
    users, Du, D = U.shape
    return lib.wst_ikbo_linear_compress(
        users, C.shape[0], Du, C.shape[1], D, W.shape[0], U.data_ptr(), C.data_ptr(),
        W.data_ptr(), off.data_ptr(), Y.data_ptr(), ws.data_ptr(),
        torch.cuda.current_stream().cuda_stream)


def test_noalloc_matches_workspace_entry_point_twice(lib):
    import warp_specialized_tensor_gb300 as w
    cases = [synthetic.ikbo(users=5, cand_per_user=[3, 40, 0, 128, 7], seed=41),
             synthetic.ikbo(seed=1003)]  # then the full 64 x 128 workload, new inputs
    for d_host in cases:
        d = _dev(d_host)
        users, _, D = d["U"].shape
        O = d["W"].shape[0]
        nc = d["C"].shape[0]
        ws = w.workspace(users, O, D)
        Y_ref = torch.full((nc, O, D), float("nan"), device="cuda")
        assert _call_workspace(lib, d, Y_ref, ws) == 0
        assert w.wst_sync_status(ws) == 0
        Y = torch.full((nc, O, D), float("nan"), device="cuda")
        status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
        assert _call_noalloc(lib, d, Y, status) == 0, lib.wst_last_error()
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        K = d["W"].shape[1]
        ok, metric, detail = compare.check(
            Y.cpu().numpy(), Y_ref.cpu().numpy().astype(np.float64), K,
            float(d_host["W"].float().abs().max()),
            max(float(d_host["U"].float().abs().max()), float(d_host["C"].float().abs().max())),
            False)
        assert ok, detail


def test_noalloc_rejects_oversize_request(lib):
    # 300 users x O=32 x D=128 need ~4.8 MB of scratch: more than the array holds.
    d = _dev(synthetic.ikbo(users=300, cand_per_user=1, seed=42))
    Y = torch.empty((300, 32, 128), device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    assert _call_noalloc(lib, d, Y, status) == 1  # WST_ERR_INVALID_ARG
    assert b"scratch" in lib.wst_last_error()
