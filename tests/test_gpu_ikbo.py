"""GPU parity: IKBO linear compression (in-kernel user broadcast) vs the
materialised-broadcast fp64 oracle, under both candidate schedules."""
import numpy as np
import pytest
import torch

import oracle
import synthetic
from gpu_util import amax, assert_parity

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def wst():
    import warp_specialized_tensor_gb300 as w
    w.load_library()
    return w


@pytest.fixture(autouse=True, params=["static", "clc"])
def sched(request, wst):
    # Every test under both candidate schedules: the static persistent split
    # and hardware cluster launch control (WST_OPT_IKBO_SCHEDULE).
    value = wst.SCHED_CLC if request.param == "clc" else wst.SCHED_STATIC
    with wst.option(wst.OPT_IKBO_SCHEDULE, value):
        yield request.param


def run_ikbo(wst, d, ws=None):
    U, Cf, W, off = d["U"].cuda(), d["C"].cuda(), d["W"].cuda(), d["user_offsets"].cuda()
    users, Du, D = U.shape
    O = W.shape[0]
    Y = torch.full((Cf.shape[0], O, D), float("nan"), dtype=torch.float32, device="cuda")
    if ws is None:
        ws = wst.workspace(users, O, D)
    wst.wst_ikbo_linear_compress(U, Cf, W, off, Y, ws)
    return Y, wst.wst_sync_status(ws), ws


def check(d, Y, cands=None):
    K = d["W"].shape[1]
    ref = oracle.ikbo(d["U"], d["C"], d["W"], d["user_offsets"], cands=cands)
    mask = None
    if cands is not None:
        mask = np.zeros(ref.shape[0], dtype=bool)
        mask[cands] = True
    assert_parity(Y, ref, K, amax(d["W"]), amax(d["U"], d["C"]), False, mask=mask, what="ikbo")


@pytest.mark.parametrize("counts", [
    [3, 0, 17, 1, 130],        # ragged users, an empty one, a >128 one
    [128] * 6,                 # the production shape, fewer users
    [1],                       # one user, one candidate
    [0, 0, 5],                 # leading users without candidates
])
def test_ikbo_counts(wst, counts):
    d = synthetic.ikbo(users=len(counts), cand_per_user=counts, seed=sum(counts) + 1)
    Y, st, _ = run_ikbo(wst, d)
    assert st == 0
    check(d, Y)


@pytest.mark.parametrize("Du,Dc,O", [(256, 64, 64), (72, 40, 32), (128, 128, 128)])
def test_ikbo_dims(wst, Du, Dc, O):
    d = synthetic.ikbo(users=3, cand_per_user=[7, 40, 2], Du=Du, Dc=Dc, O=O, seed=Du + Dc + O)
    Y, st, _ = run_ikbo(wst, d)
    assert st == 0
    check(d, Y)


def test_ikbo_many_users_more_than_ctas(wst):
    # more users than CTAs: some CTAs own several user items
    counts = [(i * 7) % 5 for i in range(400)]
    d = synthetic.ikbo(users=400, cand_per_user=counts, seed=400)
    Y, st, _ = run_ikbo(wst, d)
    assert st == 0
    check(d, Y)


def test_ikbo_back_to_back_calls_new_inputs(wst):
    # The per-user ready flags carry an epoch: a second call on the same
    # workspace must not pick up the first call's partial products.
    d1 = synthetic.ikbo(users=4, cand_per_user=[30, 2, 50, 9], seed=1)
    d2 = synthetic.ikbo(users=4, cand_per_user=[30, 2, 50, 9], seed=2)
    Y1, st, ws = run_ikbo(wst, d1)
    assert st == 0
    check(d1, Y1)
    Y2, st, _ = run_ikbo(wst, d2, ws=ws)
    assert st == 0
    check(d2, Y2)
    Y3, st, _ = run_ikbo(wst, d1, ws=ws)
    assert st == 0
    check(d1, Y3)


def test_ikbo_full_size_sampled(wst):
    d = synthetic.workload("ikbo")
    Y, st, _ = run_ikbo(wst, d)
    assert st == 0
    assert not torch.isnan(Y).any(), "unwritten outputs"
    g = torch.Generator().manual_seed(4)
    cands = sorted(set(torch.randperm(8192, generator=g)[:160].tolist() + [0, 127, 128, 8191]))
    check(d, Y, cands=cands)


def test_ikbo_bad_offsets_latched(wst):
    d = synthetic.ikbo(users=3, cand_per_user=[4, 4, 4], seed=6)
    d["user_offsets"] = torch.tensor([0, 9, 2, 12], dtype=torch.int32)
    Y, st, _ = run_ikbo(wst, d)
    assert st == wst.WST_ERR_BAD_OFFSETS
