"""CPU stand-ins for the expert-parallel layer's three GPU operations, used
only by the tests that run the plans and the exchanges over gloo on CPU: row
moves by numpy indexing and the grouped GEMM by the fp64 oracle (rounded to
bf16, as the GPU path stores it)."""
import numpy as np
import torch

import oracle


class CpuTestOps:
    device = torch.device("cpu")

    def empty(self, shape, dtype):
        return torch.full(shape, float("nan"), dtype=dtype)

    def index(self, a):
        return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int64))

    def permute(self, src, dst, src_index=None, dst_index=None, n_rows=None):
        n = n_rows if n_rows is not None else (
            (src_index if src_index is not None else dst_index).numel())
        si = src_index if src_index is not None else torch.arange(n)
        di = dst_index if dst_index is not None else torch.arange(n)
        dst[di[:n]] = src[si[:n]]

    def grouped(self, A, B, offsets, C):
        C[:] = torch.from_numpy(oracle.grouped(A, B, offsets.to(torch.int32))).to(C.dtype)


def reference(X, routing, B):
    """out[t, s] = X[t] . B[routing[t, s]]^T through oracle.grouped on the
    unsharded problem: the pairs sorted by expert (stable), one group per
    expert."""
    T, k = routing.shape
    E = B.shape[0]
    pairs = routing.reshape(-1).to(torch.int64)
    order = torch.argsort(pairs, stable=True)
    A = X[order // k]
    counts = torch.bincount(pairs, minlength=E)
    offsets = torch.zeros(E + 1, dtype=torch.int32)
    offsets[1:] = torch.cumsum(counts, 0).to(torch.int32)
    rows = oracle.grouped(A, B, offsets)
    out = np.empty((T * k, B.shape[1]))
    out[order.numpy()] = rows
    return out.reshape(T, k, B.shape[1])
