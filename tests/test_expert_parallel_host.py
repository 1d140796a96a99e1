"""Expert-parallel grouped GEMM on CPU: the libwst host plans (no GPU needed)
and the whole dispatch / exchange / combine path over two and four gloo
ranks, with the GPU operations replaced by test stand-ins (numpy row moves,
the fp64 oracle's grouped GEMM) and the result checked against the oracle's
grouped GEMM on the unsharded problem."""
import multiprocessing as mp
import os
import socket
import sys

import numpy as np
import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def wst():
    import warp_specialized_tensor_gb300 as w
    w.load_library()
    return w


def test_dispatch_plan_hand_example(wst):
    # pairs p = t*k + s: p0->e0 p1->e3 p2->e2 p3->e1 p4->e3 p5->e0; rank 0
    # owns e0, e1 and rank 1 owns e2, e3
    r = np.array([[0, 3], [2, 1], [3, 0]], dtype=np.int32)
    counts, group_counts, pairs = wst.wst_ep_dispatch_plan(r, 4, 2)
    assert counts.tolist() == [3, 3]
    assert group_counts.tolist() == [2, 1, 1, 2]
    assert pairs.tolist() == [0, 5, 3, 2, 1, 4]


def test_receive_plan_hand_example(wst):
    # source 0 sends 1 row for e0 and 2 for e1; source 1 sends 3 for e1
    offsets, rows = wst.wst_ep_receive_plan(np.array([[1, 2], [0, 3]]))
    assert offsets.tolist() == [0, 1, 6]
    assert rows.tolist() == [0, 1, 2, 3, 4, 5]
    # source-major blocks interleave when both sources send to both experts
    offsets, rows = wst.wst_ep_receive_plan(np.array([[2, 1], [1, 2]]))
    # received rows: s0e0 = 0,1; s0e1 = 2; s1e0 = 3; s1e1 = 4,5
    assert offsets.tolist() == [0, 3, 6]
    assert rows.tolist() == [0, 1, 3, 2, 4, 5]


@pytest.mark.parametrize("world,experts,tokens,k", [(1, 8, 50, 2), (4, 16, 300, 3), (8, 64, 1000, 2)])
def test_dispatch_plan_properties(wst, world, experts, tokens, k):
    g = torch.Generator().manual_seed(world + tokens)
    import synthetic
    r = synthetic.routing_table(tokens, experts, k, g).numpy()
    counts, group_counts, pairs = wst.wst_ep_dispatch_plan(r, experts, world)
    flat = r.reshape(-1)
    # a permutation of all pairs, ordered by expert then pair id
    assert sorted(pairs.tolist()) == list(range(tokens * k))
    e = flat[pairs]
    assert (np.diff(e) >= 0).all()
    for ex in range(experts):
        sel = pairs[e == ex]
        assert (np.diff(sel) > 0).all()
    assert group_counts.tolist() == np.bincount(flat, minlength=experts).tolist()
    per = experts // world
    assert counts.tolist() == [int(group_counts[d * per:(d + 1) * per].sum()) for d in range(world)]


def test_plans_reject_bad_input(wst):
    with pytest.raises(wst.WstError):
        wst.wst_ep_dispatch_plan(np.array([[0, 4]], dtype=np.int32), 4, 2)   # id out of range
    with pytest.raises(wst.WstError):
        wst.wst_ep_dispatch_plan(np.array([[0, 1]], dtype=np.int32), 6, 4)   # 6 experts over 4 ranks
    with pytest.raises(wst.WstError):
        wst.wst_ep_receive_plan(np.array([[1, -1]]))


def test_single_rank_path_matches_oracle(wst):
    sys.path.insert(0, os.path.join(ROOT, "tests"))
    import synthetic
    from ep_ops import CpuTestOps, reference
    from warp_specialized_tensor_gb300.expert_parallel import ep_grouped_gemm
    d = synthetic.moe_tokens(tokens=40, experts=4, K=64, N=32, topk=2, seed=7)
    out = ep_grouped_gemm(d["X"], d["routing"], d["B"], 4, ops=CpuTestOps())
    ref = reference(d["X"], d["routing"], d["B"])
    assert np.abs(out.double().numpy() - ref).max() <= 2.0 ** -7 * np.abs(ref).max() + 1e-12


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q, tokens_per_rank, experts, K, N, k):
    sys.path.insert(0, ROOT)
    sys.path.insert(0, os.path.join(ROOT, "tests"))
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    import torch.distributed as dist
    import synthetic
    from ep_ops import CpuTestOps, reference
    from warp_specialized_tensor_gb300.expert_parallel import ep_grouped_gemm
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # every rank draws the same global problem and keeps its share:
        # tokens [rank*T, (rank+1)*T) and experts [rank*E/R, (rank+1)*E/R)
        d = synthetic.moe_tokens(tokens=tokens_per_rank * world, experts=experts, K=K, N=N,
                                 topk=k, seed=11)
        lo, hi = rank * tokens_per_rank, (rank + 1) * tokens_per_rank
        per = experts // world
        out = ep_grouped_gemm(d["X"][lo:hi].contiguous(), d["routing"][lo:hi],
                              d["B"][rank * per:(rank + 1) * per].contiguous(), experts,
                              ops=CpuTestOps())
        ref = reference(d["X"], d["routing"], d["B"])[lo:hi]
        err = float(np.abs(out.double().numpy() - ref).max())
        q.put((rank, err, float(np.abs(ref).max()), bool(torch.isnan(out.float()).any())))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world,tokens_per_rank,experts", [(2, 60, 8), (4, 33, 8)])
def test_expert_parallel_gloo(world, tokens_per_rank, experts):
    # The plans, both count and row all-to-alls and the combine over gloo
    # ranks; a rank may receive no rows for some expert.
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    args = (world, port, q, tokens_per_rank, experts, 64, 32, 2)
    procs = [ctx.Process(target=_worker, args=(r,) + args) for r in range(world)]
    for p in procs:
        p.start()
    got = [q.get(timeout=180) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, err, amax, has_nan in got:
        assert not has_nan, "rank %d left outputs unwritten" % rank
        # bf16 output of an fp64 product: within one bf16 rounding of the max
        assert err <= 2.0 ** -7 * amax, (rank, err, amax)
