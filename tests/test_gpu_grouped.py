"""GPU parity: grouped (MoE expert) GEMM with device offsets vs the fp64 oracle.

Every test runs under both tile schedules: the static persistent walk and
hardware cluster launch control, chosen through wst_set_option
(WST_OPT_GROUPED_SCHEDULE).
"""
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
    value = wst.SCHED_CLC if request.param == "clc" else wst.SCHED_STATIC
    with wst.option(wst.OPT_GROUPED_SCHEDULE, value):
        yield request.param


def run_grouped(wst, d, out_dtype=torch.bfloat16, bias=None, epi="none", extra_rows=128):
    A, B, off = d["A"].cuda(), d["B"].cuda(), d["offsets"].cuda()
    M_total, N = d["A"].shape[0], d["B"].shape[1]
    # poison-filled buffer with rows past M_total that no group owns
    Cb = torch.full((M_total + extra_rows, N), float("nan"), dtype=out_dtype, device="cuda")
    C = Cb[:M_total]
    ws = wst.workspace()
    wst.wst_grouped_gemm_bf16(A, B, off, C, bias=None if bias is None else bias.cuda(),
                              epi=epi, workspace=ws)
    st = wst.wst_sync_status(ws)
    return Cb, C, st


@pytest.mark.parametrize("experts,tokens,K,N", [
    (8, 600, 256, 384),      # ragged groups, N = 1.5 tiles
    (16, 1000, 136, 256),    # K not a multiple of 64
    (4, 300, 512, 520),      # N ragged past two tiles
])
def test_grouped_routed(wst, experts, tokens, K, N):
    d = synthetic.grouped(experts=experts, tokens=tokens, K=K, N=N, seed=experts + tokens)
    Cb, C, st = run_grouped(wst, d)
    assert st == 0
    ref = oracle.grouped(d["A"], d["B"], d["offsets"])
    assert_parity(C, ref, K, amax(d["A"]), amax(d["B"]), True, what="grouped")
    assert torch.isnan(Cb[C.shape[0]:].float()).all(), "rows past M_total were written"


@pytest.mark.parametrize("sizes", [
    [0, 200, 0, 0, 77, 0],            # empty groups around ragged ones
    [513, 0],                         # one group, trailing empty group
    [0, 0, 0, 130],                   # leading empty groups
    [1, 1, 1, 1, 127, 129, 128, 256],  # tiny and tile-edge groups
])
def test_grouped_edge_sizes(wst, sizes):
    d = synthetic.grouped(experts=len(sizes), K=192, N=256, seed=sum(sizes), group_sizes=sizes)
    Cb, C, st = run_grouped(wst, d)
    assert st == 0
    ref = oracle.grouped(d["A"], d["B"], d["offsets"])
    assert_parity(C, ref, 192, amax(d["A"]), amax(d["B"]), True, what="grouped edge")
    assert torch.isnan(Cb[C.shape[0]:].float()).all()


@pytest.mark.parametrize("G", [255, 300])
def test_grouped_many_groups(wst, G):
    # 255 groups: their 256 offsets fill the kernel's shared-memory offset
    # table exactly; 300: past it, the tile walks read the offsets from
    # global memory.  Small ragged groups, a third of them empty.
    rng = np.random.default_rng(G)
    sizes = rng.integers(1, 40, size=G)
    sizes[rng.choice(G, size=G // 3, replace=False)] = 0
    d = synthetic.grouped(experts=G, K=128, N=256, seed=G, group_sizes=sizes.tolist())
    Cb, C, st = run_grouped(wst, d)
    assert st == 0
    ref = oracle.grouped(d["A"], d["B"], d["offsets"])
    assert_parity(C, ref, 128, amax(d["A"]), amax(d["B"]), True, what="grouped many groups")
    assert torch.isnan(Cb[C.shape[0]:].float()).all()


def test_grouped_all_tokens_one_expert(wst):
    sizes = [0] * 7 + [700]
    d = synthetic.grouped(experts=8, K=256, N=256, seed=5, group_sizes=sizes)
    Cb, C, st = run_grouped(wst, d)
    assert st == 0
    ref = oracle.grouped(d["A"], d["B"], d["offsets"])
    assert_parity(C, ref, 256, amax(d["A"]), amax(d["B"]), True, what="one expert")


@pytest.mark.parametrize("epi,out", [("bias", torch.float32), ("bias_silu", torch.bfloat16),
                                     ("bias_gelu", torch.bfloat16), ("bias_gelu", torch.float32)])
def test_grouped_epilogue(wst, epi, out):
    d = synthetic.grouped(experts=6, tokens=500, K=128, N=256, seed=77)
    bias = synthetic._normal(torch.Generator().manual_seed(78), (6, 256), 0.1)
    Cb, C, st = run_grouped(wst, d, out_dtype=out, bias=bias, epi=epi)
    assert st == 0
    ref = oracle.grouped(d["A"], d["B"], d["offsets"], bias=bias, epi=epi)
    assert_parity(C, ref, 128, amax(d["A"]), amax(d["B"]), out == torch.bfloat16, what="grouped epi")


_MOE = {}


def _moe_inputs_and_oracle():
    # The full-size oracle (4.1e11 multiply-adds in fp64) is computed once per
    # module and compared with both schedules' results.
    if not _MOE:
        d = synthetic.workload("grouped_moe")
        _MOE["d"] = d
        _MOE["ref"] = oracle.grouped(d["A"], d["B"], d["offsets"])
    return _MOE["d"], _MOE["ref"]


def test_grouped_moe_full_size_every_row(wst):
    # Every one of the 32768 rows (64 experts, top-2 routing of 16384 tokens,
    # K 4096, N 1536): full 256-token tiles and every expert's remainder tile.
    d, ref = _moe_inputs_and_oracle()
    Cb, C, st = run_grouped(wst, d)
    assert st == 0
    assert_parity(C, ref, 4096, amax(d["A"]), amax(d["B"]), True, what="moe full size")
    assert torch.isnan(Cb[C.shape[0]:].float()).all()


def test_grouped_bad_offsets_latched(wst):
    # Non-monotone offsets: the kernel clamps them (stays in bounds) and
    # latches WST_ERR_BAD_OFFSETS for wst_sync_status.
    d = synthetic.grouped(experts=3, K=64, N=256, seed=8, group_sizes=[100, 100, 100])
    d["offsets"] = torch.tensor([0, 250, 120, 300], dtype=torch.int32)
    Cb, C, st = run_grouped(wst, d)
    assert st == wst.WST_ERR_BAD_OFFSETS
    assert torch.isnan(Cb[300:].float()).all()
