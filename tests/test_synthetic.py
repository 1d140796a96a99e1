"""Host logic of the seeded input generators (routing, offsets, seeds)."""
import torch

import synthetic


def test_top2_routing_distinct_and_sorted():
    g = torch.Generator().manual_seed(0)
    tok, off = synthetic.top2_routing(1000, 16, g)
    assert off[0] == 0 and off[-1] == 2000 and (off[1:] >= off[:-1]).all()
    # every token appears exactly twice, in two different experts
    assert torch.equal(torch.bincount(tok, minlength=1000), torch.full((1000,), 2))
    expert = torch.repeat_interleave(torch.arange(16), (off[1:] - off[:-1]).long())
    pairs = {}
    for e, t in zip(expert.tolist(), tok.tolist()):
        pairs.setdefault(t, []).append(e)
    assert all(len(set(v)) == 2 for v in pairs.values())
    # ascending token order inside each expert
    for e in range(16):
        seg = tok[off[e]:off[e + 1]]
        assert (seg[1:] > seg[:-1]).all()


def test_moe_workload_statistics():
    d = synthetic.grouped(experts=64, tokens=16384, K=8, N=8, seed=1002)
    sizes = (d["offsets"][1:] - d["offsets"][:-1])
    assert int(sizes.sum()) == 32768
    assert 400 < int(sizes.min()) and int(sizes.max()) < 640


def test_seeded_determinism_and_dtypes():
    a = synthetic.dense(16, 8, 32, seed=5)
    b = synthetic.dense(16, 8, 32, seed=5)
    assert torch.equal(a["A"], b["A"]) and a["A"].dtype == torch.bfloat16
    d = synthetic.ikbo(users=3, cand_per_user=[1, 0, 2], seed=1)
    assert d["user_offsets"].tolist() == [0, 1, 1, 3]
    assert d["C"].shape == (3, 64, 128) and d["W"].shape == (32, 320)
