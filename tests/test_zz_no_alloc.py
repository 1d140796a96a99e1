"""GPU test of wst_ikbo_linear_compress_noalloc, the allocation-free IKBO entry point.

Some callers cannot allocate device memory when they call: code that runs
under a fixed memory budget, behind an allocator it must not bypass, or as a
plugin whose host framework owns every allocation.  This entry point serves
them: its scratch (error word, ready flags, per-user partial products) lives
in a fixed device array inside the library instead of a caller workspace.

Checks, each through the C ABI unless stated:
  - the result equals the fp64 oracle within the parity tolerance, and equals
    the workspace entry point's result bit for bit (same kernel, same inputs);
  - two calls in a row, and a small case run again after the full 64 x 128
    one, so partial products a larger call left in the shared array would
    show;
  - the Python wrapper runs, and rejects a non-contiguous Y;
  - inconsistent offsets land WST_ERR_BAD_OFFSETS in the caller's status
    word, and the next call reports 0 again;
  - a request larger than the array is refused before anything is enqueued.

This file is collected last, so a run that stops at the first failure has
already run every other test; it passes alone in a fresh process as well.
"""
import numpy as np
import pytest
import torch

import oracle
import synthetic
from gpu_util import amax, assert_parity

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


def _check_oracle(d_host, Y, cands=None):
    ref = oracle.ikbo(d_host["U"], d_host["C"], d_host["W"], d_host["user_offsets"], cands=cands)
    mask = None
    if cands is not None:
        mask = np.zeros(ref.shape[0], dtype=bool)
        mask[cands] = True
    assert_parity(Y, ref, d_host["W"].shape[1], amax(d_host["W"]),
                  amax(d_host["U"], d_host["C"]), False, mask=mask, what="ikbo noalloc")


def test_noalloc_matches_oracle_and_workspace_entry_point(lib):
    import warp_specialized_tensor_gb300 as w
    small = synthetic.ikbo(users=5, cand_per_user=[3, 40, 0, 128, 7], seed=41)
    full = synthetic.ikbo(seed=1003)  # 64 users x 128 candidates
    g = torch.Generator().manual_seed(43)
    full_cands = sorted(set(torch.randperm(8192, generator=g)[:96].tolist() + [0, 127, 8191]))
    # small, full, then small again: a stale partial product from the 64-user
    # call in the shared array would corrupt the second small call
    for d_host, cands in ((small, None), (full, full_cands), (small, None)):
        d = _dev(d_host)
        users, _, D = d["U"].shape
        O = d["W"].shape[0]
        nc = d["C"].shape[0]
        ws = w.workspace(users, O, D)
        Y_ref = torch.full((nc, O, D), float("nan"), device="cuda")
        assert _call_workspace(lib, d, Y_ref, ws) == 0
        assert w.wst_sync_status(ws) == 0
        for _ in range(2):  # two calls in a row on the shared array
            Y = torch.full((nc, O, D), float("nan"), device="cuda")
            status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
            assert _call_noalloc(lib, d, Y, status) == 0, lib.wst_last_error()
            torch.cuda.synchronize()
            assert int(status.item()) == 0
            assert torch.equal(Y, Y_ref), "noalloc differs from the workspace entry point"
            _check_oracle(d_host, Y, cands)


def test_noalloc_python_wrapper_and_layout_checks(lib):
    import warp_specialized_tensor_gb300 as w
    d_host = synthetic.ikbo(users=3, cand_per_user=[9, 1, 30], seed=44)
    d = _dev(d_host)
    Y = torch.full((40, 32, 128), float("nan"), device="cuda")
    status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    w.wst_ikbo_linear_compress_noalloc(d["U"], d["C"], d["W"], d["user_offsets"], Y, status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    _check_oracle(d_host, Y)
    # a permuted view of the right shape must be refused, not written through
    Yt = torch.empty((40, 128, 32), device="cuda").transpose(1, 2)
    with pytest.raises(ValueError):
        w.wst_ikbo_linear_compress_noalloc(d["U"], d["C"], d["W"], d["user_offsets"], Yt, status)


def test_noalloc_bad_offsets_reported_then_cleared(lib):
    d_host = synthetic.ikbo(users=3, cand_per_user=[4, 4, 4], seed=45)
    good = _dev(d_host)
    bad = dict(good, user_offsets=torch.tensor([0, 9, 2, 12], dtype=torch.int32, device="cuda"))
    Y = torch.full((12, 32, 128), float("nan"), device="cuda")
    status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    assert _call_noalloc(lib, bad, Y, status) == 0, lib.wst_last_error()
    torch.cuda.synchronize()
    assert int(status.item()) == 6  # WST_ERR_BAD_OFFSETS
    status.fill_(-1)
    assert _call_noalloc(lib, good, Y, status) == 0, lib.wst_last_error()
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    _check_oracle(d_host, Y)


def test_noalloc_rejects_oversize_request(lib):
    # 300 users x O=32 x D=128 need ~4.8 MB of scratch: more than the array holds.
    d = _dev(synthetic.ikbo(users=300, cand_per_user=1, seed=42))
    Y = torch.empty((300, 32, 128), device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    assert _call_noalloc(lib, d, Y, status) == 1  # WST_ERR_INVALID_ARG
    assert b"scratch" in lib.wst_last_error()
