"""GPU parity: IKBO attention (candidate queries over their user's context)
against the fp64 oracle.

Tolerance, from the kernel's arithmetic: the probabilities are rounded to
bf16 (relative error <= 2^-9) before the product with V, while the row sums,
maxima and the output accumulate in fp32, so |O_gpu - O_ref| <= 2^-9 max|V|
plus fp32 rounding.  The test allows 2^-8 max|V| (a factor 2 of margin),
plus one bf16 ulp of the reference for bf16 outputs.  Merging split items
(the stream-K tail) adds fp32 rounding only.

Every test runs under both schedules: whole items only (a header-only
workspace) and the split last wave (a full attention workspace).
"""
import math

import numpy as np
import pytest
import torch

import oracle
import synthetic
from oracle import compare

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def wst():
    import warp_specialized_tensor_gb300 as w
    w.load_library()
    return w


SCHED = {"sched": "split"}


@pytest.fixture(autouse=True, params=["whole", "split"])
def sched(request):
    SCHED["sched"] = request.param
    yield request.param


_WS = {}


def workspace(wst):
    # one workspace per schedule, reused across calls (the split schedule's
    # flags carry a per-call epoch)
    k = SCHED["sched"]
    if k not in _WS:
        _WS[k] = wst.attention_workspace() if k == "split" else wst.workspace()
    return _WS[k]


def run(wst, d, out_dtype=torch.float32, scale=None):
    Q, K, V, off = d["Q"].cuda(), d["K"].cuda(), d["V"].cuda(), d["user_offsets"].cuda()
    O = torch.full(Q.shape, float("nan"), dtype=out_dtype, device="cuda")
    ws = workspace(wst)
    wst.wst_ikbo_attention_bf16(Q, K, V, off, O, Lq=d["Lq"], scale=scale, workspace=ws)
    return O, wst.wst_sync_status(ws)


def check(O, ref, V, out_bf16, rows=None, what=""):
    g = O.float().cpu().numpy().astype(np.float64)
    if rows is not None:
        g, ref = g[rows], ref[rows]
    assert not np.isnan(ref).any()
    tol = 2.0 ** -8 * float(V.float().abs().max())
    bound = tol + (compare.ulp_bf16(ref) if out_bf16 else 0.0)
    err = np.abs(g - ref)
    bad = ~(err <= bound)
    assert not bad.any(), "%s: %d elements out of tolerance, max err %.3g (tol %.3g) at %s" % (
        what, int(bad.sum()), float(np.nanmax(err)), tol, np.argwhere(bad)[:3].tolist())
    return float(err.max()) / tol


@pytest.mark.parametrize("counts,Lq,H,Lkv", [
    ([40, 0, 130, 7], 2, 2, 200),   # ragged users (one empty), 3 key blocks + 8
    ([64], 2, 1, 64),               # exactly one query tile and one key block
    ([1, 3, 2], 1, 3, 1),           # a single key: O = V[u, 0]
    ([100, 28], 1, 2, 65),          # one key past a block edge
    ([300], 3, 1, 130),             # 900 query rows of one user: 8 tiles
])
@pytest.mark.parametrize("out", [torch.float32, torch.bfloat16])
def test_attention_parity(wst, counts, Lq, H, Lkv, out):
    d = synthetic.ikbo_attention(users=len(counts), cand_per_user=counts, Lq=Lq, H=H, Lkv=Lkv,
                                 seed=len(counts) * 100 + Lkv)
    O, st = run(wst, d, out)
    assert st == 0
    ref = oracle.ikbo_attention(d["Q"], d["K"], d["V"], d["user_offsets"], Lq)
    check(O, ref, d["V"], out == torch.bfloat16, what="attention %s" % (counts,))


def test_attention_single_key_is_exact_value(wst):
    d = synthetic.ikbo_attention(users=2, cand_per_user=[5, 9], Lq=2, H=2, Lkv=1, seed=3)
    O, st = run(wst, d, torch.float32)
    assert st == 0
    users = np.repeat([0, 1], np.array([5, 9]) * 2)
    want = d["V"].float()[users, 0]
    assert torch.equal(O.cpu(), want)


def test_attention_scale_argument(wst):
    d = synthetic.ikbo_attention(users=2, cand_per_user=[20, 30], Lq=1, H=2, Lkv=150, seed=4)
    O, st = run(wst, d, torch.float32, scale=0.5)
    assert st == 0
    ref = oracle.ikbo_attention(d["Q"], d["K"], d["V"], d["user_offsets"], 1, scale=0.5)
    check(O, ref, d["V"], False, what="scale 0.5")


def test_attention_full_size_sampled(wst):
    # Every candidate of eight users: the last four users (whose items fill
    # the persistent grid's partial last wave, split by key blocks over all
    # CTAs and merged when the workspace allows) and four drawn at random.
    d = synthetic.workload("ikbo_attention")
    O, st = run(wst, d, torch.bfloat16)
    assert st == 0
    off = d["user_offsets"].tolist()
    Lq = d["Lq"]
    users = len(off) - 1
    g = torch.Generator().manual_seed(5)
    pick = set(range(users - 4, users)) | set(torch.randperm(users - 4, generator=g)[:4].tolist())
    cands = sorted(c for u in pick for c in range(off[u], off[u + 1]))
    ref = oracle.ikbo_attention(d["Q"], d["K"], d["V"], d["user_offsets"], Lq, cands=cands)
    rows = [c * Lq + r for c in cands for r in range(Lq)]
    check(O, ref, d["V"], True, rows=rows, what="full size")
    assert not torch.isnan(O.float()).any(), "unwritten rows"


def test_attention_bad_offsets_latched(wst):
    d = synthetic.ikbo_attention(users=3, cand_per_user=[10, 10, 10], Lq=1, H=1, Lkv=70, seed=6)
    d["user_offsets"] = torch.tensor([0, 20, 5, 30], dtype=torch.int32)
    O, st = run(wst, d)
    assert st == wst.WST_ERR_BAD_OFFSETS


def test_attention_rescale_path(wst):
    # Keys of later blocks scaled up so that row maxima grow by far more than
    # 2^8 between blocks: the kernel must rescale O in tensor memory (the
    # N(0,1) cases above never take that branch).
    d = synthetic.ikbo_attention(users=2, cand_per_user=[70, 9], Lq=2, H=2, Lkv=400, seed=8)
    K = d["K"].float()
    K[:, 128:256] *= 6.0
    K[:, 256:] *= 14.0
    d["K"] = K.to(torch.bfloat16)
    for out in (torch.float32, torch.bfloat16):
        O, st = run(wst, d, out)
        assert st == 0
        ref = oracle.ikbo_attention(d["Q"], d["K"], d["V"], d["user_offsets"], 2)
        check(O, ref, d["V"], out == torch.bfloat16, what="rescale")


def test_attention_large_row_sum_without_growth(wst):
    # After a fragment's first block the kernel skips the row maximum while
    # the block's row sum stays <= 2^8; here every later key scores ~6.0
    # (base 2) above the first block's maximum, so the sums are ~128 x 2^6
    # while no single weight exceeds 2^8: the kernel must take its reload
    # path, find that the maximum need not grow, and still produce the exact
    # softmax (weights 1 in the first block, ~2^6 after it).
    d = synthetic.ikbo_attention(users=2, cand_per_user=[70, 9], Lq=2, H=2, Lkv=520, seed=10)
    Q = torch.zeros(d["Q"].shape)
    Q[..., 0] = 1.0
    K = torch.zeros(d["K"].shape)
    K[:, 128:, :, 0] = 6.0 / math.log2(math.e)  # raw score 4.16: 2^(log2(e) * 4.16) ~ 2^6
    K[:, 300:310, :, 0] = -3.0                   # and a few low ones
    d["Q"], d["K"] = Q.to(torch.bfloat16), K.to(torch.bfloat16)
    for out in (torch.float32, torch.bfloat16):
        O, st = run(wst, d, out, scale=1.0)
        assert st == 0
        ref = oracle.ikbo_attention(d["Q"], d["K"], d["V"], d["user_offsets"], 2, scale=1.0)
        check(O, ref, d["V"], out == torch.bfloat16, what="large row sums")


@pytest.mark.parametrize("scale", [-0.3, 0.0])
def test_attention_negative_and_zero_scale(wst, scale):
    # scale < 0: the row extremum is the minimum of the raw scores; scale = 0:
    # uniform weights over the context (the mean of V).
    d = synthetic.ikbo_attention(users=3, cand_per_user=[20, 0, 45], Lq=1, H=2, Lkv=300, seed=9)
    O, st = run(wst, d, torch.float32, scale=scale)
    assert st == 0
    ref = oracle.ikbo_attention(d["Q"], d["K"], d["V"], d["user_offsets"], 1, scale=scale)
    check(O, ref, d["V"], False, what="scale %g" % scale)


def test_attention_one_item_over_many_ctas(wst):
    # One item of 16 key blocks: under the split schedule each block runs on
    # its own CTA and the CTA holding block 0 merges 15 partials.
    d = synthetic.ikbo_attention(users=1, cand_per_user=[10], Lq=3, H=1, Lkv=2000, seed=10)
    for out in (torch.float32, torch.bfloat16):
        O, st = run(wst, d, out)
        assert st == 0
        ref = oracle.ikbo_attention(d["Q"], d["K"], d["V"], d["user_offsets"], 3)
        check(O, ref, d["V"], out == torch.bfloat16, what="one item")


def test_attention_one_wave_plus_tail(wst):
    # SMs + 8 items: one full round-robin wave and a tail of 8 items split
    # over all CTAs; sampled rows of the first, a middle and the tail items.
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    n_items = sms + 8
    d = synthetic.ikbo_attention(users=2, cand_per_user=[128 * (n_items // 2), 128 * (n_items - n_items // 2)],
                                 Lq=1, H=1, Lkv=700, seed=11)
    O, st = run(wst, d, torch.float32)
    assert st == 0
    nq = d["Q"].shape[0]
    tiles = [0, 1, sms // 2, sms - 1, sms, sms + 3, n_items - 1]
    cands = sorted({min(nq - 1, 128 * t + r) for t in tiles for r in (0, 77, 127)})
    ref = oracle.ikbo_attention(d["Q"], d["K"], d["V"], d["user_offsets"], 1, cands=cands)
    check(O, ref, d["V"], False, rows=cands, what="wave + tail")
    assert not torch.isnan(O).any(), "unwritten rows"


def test_attention_repeated_calls_same_workspace(wst):
    # The per-call epoch: back-to-back calls on one workspace with different
    # inputs must not read each other's partials.
    d1 = synthetic.ikbo_attention(users=2, cand_per_user=[30, 50], Lq=2, H=2, Lkv=500, seed=12)
    d2 = synthetic.ikbo_attention(users=2, cand_per_user=[30, 50], Lq=2, H=2, Lkv=500, seed=13)
    for d in (d1, d2, d1, d2):
        O, st = run(wst, d, torch.float32)
        assert st == 0
        ref = oracle.ikbo_attention(d["Q"], d["K"], d["V"], d["user_offsets"], 2)
        check(O, ref, d["V"], False, what="repeat")
