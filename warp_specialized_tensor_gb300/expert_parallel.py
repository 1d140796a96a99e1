"""Expert-parallel grouped GEMM: the experts of a mixture-of-experts layer
spread over the ranks (one GPU each) of a node.

"How We Built TLX: A Hardware-Native GPU Compiler for Production ML at Scale"
(Meta Engineering), "Case Study 3: Distributed Grouped GEMM for LLM
Pretraining" and "TLX in Production": every routed (token, expert) pair is
sent to the rank that owns the expert, multiplied there by that rank's
grouped GEMM, and sent back to the token's rank.

For rank r of R with G experts (G divisible by R; rank r owns experts
[r*G/R, (r+1)*G/R)) and local tokens x [T, K] routed to top_k experts each:

    out[t, s] = x[t] . W[routing[t, s]]^T          out: [T, top_k, N]

Steps (the index plans are libwst host functions, every row movement is
libwst's permute kernel, the products are libwst's grouped GEMM, and the two
exchanges are torch.distributed all-to-alls, NCCL on GPUs):

    dispatch plan -> count exchange -> gather send rows -> row all-to-all ->
    receive plan -> gather by expert -> grouped GEMM -> scatter to received
    order -> reverse row all-to-all -> scatter to the pairs

``ops`` replaces the three GPU operations (permute, grouped GEMM, buffer
allocation); only tests use it, to run the plans and the exchanges over
gloo on CPU against the CPU oracle.  The default is the CUDA library, which
raises if it is not available: there is no CPU path in the product.
"""
from __future__ import annotations

import numpy as np
import torch

from . import (wst_ep_dispatch_plan, wst_ep_receive_plan, wst_grouped_gemm_bf16,
               wst_permute_rows, workspace as _workspace)

__all__ = ["ep_grouped_gemm", "CudaOps"]


class CudaOps:
    """The GPU operations of the expert-parallel layer (libwst kernels)."""

    def __init__(self, device=None, ws=None):
        self.device = torch.device(device or "cuda")
        self.ws = ws if ws is not None else _workspace(device=self.device)

    def empty(self, shape, dtype):
        return torch.empty(shape, dtype=dtype, device=self.device)

    def index(self, a: np.ndarray) -> torch.Tensor:
        return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).to(self.device)

    def permute(self, src, dst, src_index=None, dst_index=None, n_rows=None):
        wst_permute_rows(src, dst, src_index=src_index, dst_index=dst_index, n_rows=n_rows,
                         workspace=self.ws)

    def grouped(self, A, B, offsets, C):
        wst_grouped_gemm_bf16(A, B, offsets, C, workspace=self.ws)


def _all_to_all(out, inp, out_splits, in_splits, group):
    import torch.distributed as dist
    dist.all_to_all_single(out, inp, output_split_sizes=[int(v) for v in out_splits],
                           input_split_sizes=[int(v) for v in in_splits], group=group)


def _exchange_counts(send_group_counts: np.ndarray, world: int, group, device) -> np.ndarray:
    """All-to-all of the per-(rank, local expert) counts: returns
    recv[s][e] = rows source s sends for this rank's local expert e."""
    if world == 1:
        return send_group_counts.reshape(1, -1).copy()
    import torch.distributed as dist
    per = send_group_counts.size // world
    send = torch.from_numpy(send_group_counts.astype(np.int64)).to(device)
    recv = torch.empty_like(send)
    dist.all_to_all_single(recv, send, output_split_sizes=[per] * world,
                           input_split_sizes=[per] * world, group=group)
    return recv.cpu().numpy().astype(np.int32).reshape(world, per)


def ep_grouped_gemm(x, routing, w_local, num_experts: int, group=None, out=None, ops=None):
    """Expert-parallel grouped GEMM of this rank's tokens.

    x:        bf16 [T, K] this rank's token features (on the ops' device)
    routing:  int32 [T, top_k] expert ids in [0, num_experts) (host array or
              tensor; it is read on the host to build the plans)
    w_local:  bf16 [num_experts / world, N, K] this rank's experts
    group:    torch.distributed process group (None: the default group if
              initialised, else a single rank)
    Returns out [T, top_k, N] bf16 with out[t, s] = x[t] . W[routing[t, s]]^T.
    """
    import torch.distributed as dist
    ops = ops or CudaOps(device=x.device)
    world = dist.get_world_size(group) if dist.is_available() and dist.is_initialized() else 1
    r = np.asarray(routing.cpu() if isinstance(routing, torch.Tensor) else routing, dtype=np.int32)
    T, k = r.shape
    K = x.shape[1]
    e_local, N, K2 = w_local.shape
    if K2 != K or e_local * world != num_experts:
        raise ValueError("w_local must be [num_experts / world, N, K]")
    if out is None:
        out = ops.empty((T, k, N), torch.bfloat16)
    if out.shape != (T, k, N):
        raise ValueError("out must be [T, top_k, N]")

    # 1-2: what goes where, and what arrives from where
    send_counts, send_group_counts, send_pairs = wst_ep_dispatch_plan(r, num_experts, world)
    recv_group_counts = _exchange_counts(send_group_counts, world, group, x.device)
    recv_counts = recv_group_counts.sum(axis=1)
    n_send, n_recv = int(send_counts.sum()), int(recv_counts.sum())

    # 3: the token row of every pair, in send order
    send = ops.empty((n_send, K), torch.bfloat16)
    if n_send:
        ops.permute(x, send, src_index=ops.index(send_pairs // k))
    # 4: rows to the experts' ranks
    if world > 1:
        recv = ops.empty((n_recv, K), torch.bfloat16)
        _all_to_all(recv, send, recv_counts, send_counts, group)
    else:
        recv = send
    # 5: expert-major order and this rank's grouped GEMM
    offsets, expert_rows = wst_ep_receive_plan(recv_group_counts)
    A = ops.empty((n_recv, K), torch.bfloat16)
    rows_dev = ops.index(expert_rows) if n_recv else None
    if n_recv:
        ops.permute(recv, A, src_index=rows_dev)
    C = ops.empty((n_recv, N), torch.bfloat16)
    if n_recv:
        ops.grouped(A, w_local, ops.index(offsets), C)
    # 6: products back to received order, back to their ranks, to their pairs
    back_src = ops.empty((n_recv, N), torch.bfloat16)
    if n_recv:
        ops.permute(C, back_src, dst_index=rows_dev)
    if world > 1:
        back = ops.empty((n_send, N), torch.bfloat16)
        _all_to_all(back, back_src, send_counts, recv_counts, group)
    else:
        back = back_src
    if n_send:
        ops.permute(back, out.view(T * k, N), dst_index=ops.index(send_pairs))
    return out
