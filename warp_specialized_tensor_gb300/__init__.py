"""Python binding of libwst, the GB300 (sm_103a) warp-specialized contraction
library.  Argument marshalling only: every step of the computation runs in the
CUDA kernels behind the C ABI declared in ``include/wst.h``; there is no CPU
or PyTorch fallback.  PyTorch supplies device memory and streams.

The functions carry the C ABI's names and take torch tensors; sizes, leading
dimensions and batch strides are read from the tensors' shapes and strides.
A non-OK status raises :class:`WstError`.
"""
from __future__ import annotations

import ctypes
import math
import os
import threading

import torch

from . import _build

__all__ = [
    "WstError", "EPI_NONE", "EPI_BIAS", "EPI_BIAS_SILU", "EPI_BIAS_GELU", "F32", "BF16",
    "load_library", "library_path", "wst_workspace_size", "wst_workspace_init",
    "workspace", "wst_gemm_bf16", "wst_gemm_rmsnorm_bf16", "wst_gemm_layernorm_bf16",
    "wst_gemm_layernorm_workspace_size", "layernorm_workspace", "wst_gemm_norm_workspace_size",
    "norm_workspace", "wst_grouped_gemm_bf16",
    "wst_ikbo_linear_compress", "wst_ikbo_linear_compress_noalloc", "wst_ikbo_attention_bf16",
    "wst_ikbo_attention_workspace_size", "attention_workspace",
    "wst_sync_status", "wst_status_string", "wst_set_option", "wst_get_option", "option",
    "OPT_GROUPED_SCHEDULE", "OPT_DENSE_CTA_GROUP", "OPT_IKBO_SCHEDULE", "OPT_NORM_STATS",
    "SCHED_STATIC", "SCHED_CLC", "NORM_STATS_AUTO", "NORM_STATS_FUSED", "NORM_STATS_PASS",
    "wst_version", "wst_ep_dispatch_plan", "wst_ep_receive_plan", "wst_permute_rows",
]

# enums of include/wst.h
WST_OK, WST_ERR_INVALID_ARG, WST_ERR_ALIGNMENT, WST_ERR_UNSUPPORTED = 0, 1, 2, 3
WST_ERR_CUDA, WST_ERR_TIMEOUT, WST_ERR_BAD_OFFSETS = 4, 5, 6
F32, BF16 = 0, 1
EPI_NONE, EPI_BIAS, EPI_BIAS_SILU, EPI_BIAS_GELU = 0, 1, 2, 3
OPT_GROUPED_SCHEDULE, OPT_DENSE_CTA_GROUP, OPT_IKBO_SCHEDULE, OPT_NORM_STATS = 0, 1, 2, 3
SCHED_STATIC, SCHED_CLC = 0, 1
NORM_STATS_AUTO, NORM_STATS_FUSED, NORM_STATS_PASS = 0, 1, 2
_EPI_NAMES = {"none": EPI_NONE, "bias": EPI_BIAS, "bias_silu": EPI_BIAS_SILU,
              "bias_gelu": EPI_BIAS_GELU}

_lock = threading.Lock()
_lib = None


class WstError(RuntimeError):
    def __init__(self, status: int, where: str, detail: str):
        self.status = status
        super().__init__("%s: %s%s" % (where, wst_status_string(status),
                                       (" -- " + detail) if detail else ""))


def library_path() -> str:
    return _build.LIB


def load_library(build_if_missing: bool = True) -> ctypes.CDLL:
    """Load libwst.so (building it in-tree with nvcc when absent or stale)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if build_if_missing and not _build.up_to_date():
            _build.build()
        if not os.path.exists(_build.LIB):
            raise ImportError("libwst.so is not built; run warp_specialized_tensor_gb300._build.build()")
        lib = ctypes.CDLL(_build.LIB)
        P, I, L, Z = ctypes.c_void_p, ctypes.c_int, ctypes.c_long, ctypes.c_size_t
        lib.wst_workspace_size.argtypes = [I, I, I]
        lib.wst_workspace_size.restype = Z
        lib.wst_workspace_init.argtypes = [P, Z, P]
        lib.wst_workspace_init.restype = I
        lib.wst_gemm_bf16.argtypes = [I, I, I, I, P, L, L, P, L, L, P, L, P, L, L, I, I, P, P]
        lib.wst_gemm_bf16.restype = I
        lib.wst_gemm_rmsnorm_bf16.argtypes = [I, I, I, I, P, L, L, P, L, L, ctypes.c_float, P, L,
                                              P, L, L, I, I, P, Z, P]
        lib.wst_gemm_rmsnorm_bf16.restype = I
        lib.wst_gemm_layernorm_bf16.argtypes = [I, I, I, I, P, L, L, P, L, L, ctypes.c_float, P,
                                                L, P, L, L, I, I, P, Z, P]
        lib.wst_gemm_layernorm_bf16.restype = I
        lib.wst_gemm_layernorm_workspace_size.argtypes = [I, I, L]
        lib.wst_gemm_layernorm_workspace_size.restype = Z
        lib.wst_gemm_norm_workspace_size.argtypes = [I, I, I, L, L, I]
        lib.wst_gemm_norm_workspace_size.restype = Z
        lib.wst_grouped_gemm_bf16.argtypes = [I, I, I, I, P, L, P, L, L, P, P, L, P, L, I, I, P, P]
        lib.wst_grouped_gemm_bf16.restype = I
        lib.wst_ikbo_linear_compress.argtypes = [I, I, I, I, I, I, P, P, P, P, P, P, P]
        lib.wst_ikbo_linear_compress.restype = I
        lib.wst_ikbo_linear_compress_noalloc.argtypes = [I, I, I, I, I, I, P, P, P, P, P, P, P]
        lib.wst_ikbo_linear_compress_noalloc.restype = I
        lib.wst_ikbo_attention_bf16.argtypes = [I, I, I, I, I, I, P, P, P, P, ctypes.c_float,
                                                P, I, P, Z, P]
        lib.wst_ikbo_attention_bf16.restype = I
        lib.wst_ikbo_attention_workspace_size.argtypes = []
        lib.wst_ikbo_attention_workspace_size.restype = Z
        IP = ctypes.POINTER(ctypes.c_int)
        lib.wst_ep_dispatch_plan.argtypes = [I, I, IP, I, I, IP, IP, IP]
        lib.wst_ep_dispatch_plan.restype = I
        lib.wst_ep_receive_plan.argtypes = [I, I, IP, IP, IP]
        lib.wst_ep_receive_plan.restype = I
        lib.wst_permute_rows.argtypes = [I, Z, P, Z, P, I, P, Z, P, I, P, P]
        lib.wst_permute_rows.restype = I
        lib.wst_set_option.argtypes = [I, I]
        lib.wst_set_option.restype = I
        lib.wst_get_option.argtypes = [I, ctypes.POINTER(ctypes.c_int)]
        lib.wst_get_option.restype = I
        lib.wst_sync_status.argtypes = [P, P]
        lib.wst_sync_status.restype = I
        lib.wst_status_string.argtypes = [I]
        lib.wst_status_string.restype = ctypes.c_char_p
        lib.wst_last_error.argtypes = []
        lib.wst_last_error.restype = ctypes.c_char_p
        lib.wst_version.argtypes = []
        lib.wst_version.restype = ctypes.c_char_p
        _lib = lib
        return lib


def wst_status_string(status: int) -> str:
    return load_library().wst_status_string(int(status)).decode()


def wst_version() -> str:
    return load_library().wst_version().decode()


def _check(status: int, where: str):
    if status != WST_OK:
        detail = load_library().wst_last_error().decode()
        raise WstError(status, where, detail)


def _stream_handle(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return int(stream.cuda_stream) if hasattr(stream, "cuda_stream") else int(stream)


def _ptr(t) -> int | None:
    return None if t is None else t.data_ptr()


def _epi(epi) -> int:
    return _EPI_NAMES[epi] if isinstance(epi, str) else int(epi)


def _ctype(C) -> int:
    if C.dtype == torch.float32:
        return F32
    if C.dtype == torch.bfloat16:
        return BF16
    raise TypeError("C must be float32 or bfloat16")


def _need(t, name, dtype=None, dims=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError("%s must be a torch tensor" % name)
    if not t.is_cuda:
        raise ValueError("%s must be a CUDA tensor" % name)
    if dtype is not None and t.dtype != dtype:
        raise TypeError("%s must be %s" % (name, dtype))
    if dims is not None and t.dim() not in dims:
        raise ValueError("%s must have %s dimensions" % (name, dims))
    if t.stride(-1) != 1:
        raise ValueError("%s must have a contiguous last dimension" % name)


# ----------------------------------------------------------------------------
# process-wide options
# ----------------------------------------------------------------------------
def wst_set_option(opt: int, value: int) -> None:
    """Set a process-wide tuning option (OPT_GROUPED_SCHEDULE and
    OPT_IKBO_SCHEDULE: SCHED_STATIC or SCHED_CLC; OPT_DENSE_CTA_GROUP: 0
    automatic, 1 single-CTA tiles, 2 pairs; OPT_NORM_STATS: NORM_STATS_AUTO,
    NORM_STATS_FUSED or NORM_STATS_PASS)."""
    _check(load_library().wst_set_option(int(opt), int(value)), "wst_set_option")


def wst_get_option(opt: int) -> int:
    v = ctypes.c_int(0)
    _check(load_library().wst_get_option(int(opt), ctypes.byref(v)), "wst_get_option")
    return int(v.value)


class option:
    """Context manager: set an option for the duration of a block, then restore it."""

    def __init__(self, opt: int, value: int):
        self.opt, self.value, self.old = opt, value, None

    def __enter__(self):
        self.old = wst_get_option(self.opt)
        wst_set_option(self.opt, self.value)
        return self

    def __exit__(self, *exc):
        wst_set_option(self.opt, self.old)
        return False


# ----------------------------------------------------------------------------
# workspace
# ----------------------------------------------------------------------------
def wst_workspace_size(num_users: int = 0, O: int = 0, D: int = 0) -> int:
    return int(load_library().wst_workspace_size(num_users, O, D))


def wst_workspace_init(ws: torch.Tensor, stream=None) -> None:
    _check(load_library().wst_workspace_init(ws.data_ptr(), ws.numel() * ws.element_size(),
                                             _stream_handle(stream)), "wst_workspace_init")


def workspace(num_users: int = 0, O: int = 0, D: int = 0, device=None, stream=None) -> torch.Tensor:
    """Allocate (through PyTorch) and zero-fill a workspace for these sizes."""
    n = wst_workspace_size(num_users, O, D)
    ws = torch.empty(n, dtype=torch.uint8, device=device or "cuda")
    wst_workspace_init(ws, stream)
    return ws


# ----------------------------------------------------------------------------
# the three operations
# ----------------------------------------------------------------------------
def wst_gemm_bf16(A, B, C, bias=None, epi="none", workspace=None, stream=None) -> None:
    """C[b] = epi(A[b] . B[b]^T (+ bias[b])) on the GPU.

    A: bf16 [M,K] or [batch,M,K]; B: bf16 [N,K] or [batch,N,K] (a 2-D B is
    shared by the batch); C: bf16/fp32 [M,N] or [batch,M,N]; bias: bf16 [N]
    (shared) or [batch,N]."""
    _need(A, "A", torch.bfloat16, (2, 3))
    _need(B, "B", torch.bfloat16, (2, 3))
    _need(C, "C", None, (2, 3))
    if workspace is None:
        raise ValueError("workspace is required (see workspace())")
    batch = A.shape[0] if A.dim() == 3 else 1
    M, K = A.shape[-2], A.shape[-1]
    N = B.shape[-2]
    if B.shape[-1] != K or C.shape[-2:] != (M, N):
        raise ValueError("shape mismatch: A %s B %s C %s" % (tuple(A.shape), tuple(B.shape), tuple(C.shape)))
    if C.dim() == 3 and C.shape[0] != batch:
        raise ValueError("C batch mismatch")
    sA = A.stride(0) if A.dim() == 3 else 0
    sB = B.stride(0) if B.dim() == 3 else 0
    if B.dim() == 3 and B.shape[0] != batch:
        raise ValueError("B batch mismatch")
    sC = C.stride(0) if C.dim() == 3 else 0
    e = _epi(epi)
    sBias = 0
    if e != EPI_NONE:
        _need(bias, "bias", torch.bfloat16, (1, 2))
        sBias = bias.stride(0) if bias.dim() == 2 else 0
    st = load_library().wst_gemm_bf16(
        batch, M, N, K, A.data_ptr(), A.stride(-2), sA, B.data_ptr(), B.stride(-2), sB,
        _ptr(bias) if e else None, sBias, C.data_ptr(), C.stride(-2), sC, _ctype(C), e,
        workspace.data_ptr(), _stream_handle(stream))
    _check(st, "wst_gemm_bf16")


def _norm_gemm_args(A, B, C, bias, epi, workspace):
    _need(A, "A", torch.bfloat16, (2, 3))
    _need(B, "B", torch.bfloat16, (2, 3))
    _need(C, "C", None, (2, 3))
    if workspace is None:
        raise ValueError("workspace is required (see workspace())")
    batch = A.shape[0] if A.dim() == 3 else 1
    M, K = A.shape[-2], A.shape[-1]
    N = B.shape[-2]
    if B.shape[-1] != K or C.shape[-2:] != (M, N):
        raise ValueError("shape mismatch")
    if (B.dim() == 3 and B.shape[0] != batch) or (C.dim() == 3 and C.shape[0] != batch):
        raise ValueError("batch mismatch")
    sA = A.stride(0) if A.dim() == 3 else 0
    sB = B.stride(0) if B.dim() == 3 else 0
    sC = C.stride(0) if C.dim() == 3 else 0
    e = _epi(epi)
    sBias = 0
    if e != EPI_NONE:
        _need(bias, "bias", torch.bfloat16, (1, 2))
        sBias = bias.stride(0) if bias.dim() == 2 else 0
    return batch, M, N, K, sA, sB, sC, e, sBias


def wst_gemm_rmsnorm_bf16(A, B, C, eps=1e-6, bias=None, epi="none", workspace=None,
                          stream=None) -> None:
    """C[b] = epi(diag(r[b]) . A[b] . B[b]^T (+ bias[b])), r = 1/sqrt(mean(A^2, -1) + eps).

    Same tensor conventions as wst_gemm_bf16.  Any workspace() works; one of
    norm_workspace(A, B) bytes also lets the row statistics come from a
    separate pass over A (faster for wide N)."""
    batch, M, N, K, sA, sB, sC, e, sBias = _norm_gemm_args(A, B, C, bias, epi, workspace)
    st = load_library().wst_gemm_rmsnorm_bf16(
        batch, M, N, K, A.data_ptr(), A.stride(-2), sA, B.data_ptr(), B.stride(-2), sB,
        float(eps), _ptr(bias) if e else None, sBias, C.data_ptr(), C.stride(-2), sC, _ctype(C),
        e, workspace.data_ptr(), workspace.numel() * workspace.element_size(),
        _stream_handle(stream))
    _check(st, "wst_gemm_rmsnorm_bf16")


def wst_gemm_layernorm_workspace_size(batch: int, N: int, strideB: int = 0) -> int:
    return int(load_library().wst_gemm_layernorm_workspace_size(batch, N, strideB))


def layernorm_workspace(B, device=None, stream=None) -> torch.Tensor:
    """A zero-filled workspace large enough for wst_gemm_layernorm_bf16 with this B."""
    batch = B.shape[0] if B.dim() == 3 else 1
    n = wst_gemm_layernorm_workspace_size(batch, B.shape[-2], B.stride(0) if B.dim() == 3 else 0)
    ws = torch.empty(n, dtype=torch.uint8, device=device or B.device)
    wst_workspace_init(ws, stream)
    return ws


def wst_gemm_norm_workspace_size(batch: int, M: int, N: int, strideA: int = 0, strideB: int = 0,
                                 layernorm: bool = False) -> int:
    return int(load_library().wst_gemm_norm_workspace_size(batch, M, N, strideA, strideB,
                                                           1 if layernorm else 0))


def norm_workspace(A, B, layernorm=False, device=None, stream=None) -> torch.Tensor:
    """A zero-filled workspace with which wst_gemm_rmsnorm_bf16 (or, with
    layernorm=True, wst_gemm_layernorm_bf16) can take either form of the row
    statistics for these A and B."""
    batch = A.shape[0] if A.dim() == 3 else 1
    n = wst_gemm_norm_workspace_size(batch, A.shape[-2], B.shape[-2], A.stride(0) if A.dim() == 3 else 0,
                                     B.stride(0) if B.dim() == 3 else 0, layernorm)
    ws = torch.empty(n, dtype=torch.uint8, device=device or A.device)
    wst_workspace_init(ws, stream)
    return ws


def wst_gemm_layernorm_bf16(A, B, C, eps=1e-5, bias=None, epi="none", workspace=None,
                            stream=None) -> None:
    """C[b] = epi(LayerNorm(A[b]) . B[b]^T (+ bias[b])), the rows of A normalised
    to zero mean and unit (biased) variance, eps inside the square root.

    Same tensor conventions as wst_gemm_bf16; the workspace must hold
    wst_gemm_layernorm_workspace_size(...) bytes (see layernorm_workspace());
    one of norm_workspace(A, B, layernorm=True) bytes also lets the row
    statistics come from a separate pass over A."""
    batch, M, N, K, sA, sB, sC, e, sBias = _norm_gemm_args(A, B, C, bias, epi, workspace)
    st = load_library().wst_gemm_layernorm_bf16(
        batch, M, N, K, A.data_ptr(), A.stride(-2), sA, B.data_ptr(), B.stride(-2), sB,
        float(eps), _ptr(bias) if e else None, sBias, C.data_ptr(), C.stride(-2), sC, _ctype(C),
        e, workspace.data_ptr(), workspace.numel() * workspace.element_size(),
        _stream_handle(stream))
    _check(st, "wst_gemm_layernorm_bf16")


def wst_grouped_gemm_bf16(A, B, offsets, C, bias=None, epi="none", workspace=None,
                          stream=None) -> None:
    """Rows [off[g], off[g+1]) of C = epi(rows of A . B[g]^T (+ bias[g])).

    A: bf16 [M_total,K]; B: bf16 [G,N,K]; offsets: device int32 [G+1];
    C: bf16/fp32 [M_total,N]; bias: bf16 [G,N]."""
    _need(A, "A", torch.bfloat16, (2,))
    _need(B, "B", torch.bfloat16, (3,))
    _need(C, "C", None, (2,))
    _need(offsets, "offsets", torch.int32, (1,))
    if workspace is None:
        raise ValueError("workspace is required (see workspace())")
    G, N, K = B.shape
    M_total = A.shape[0]
    if A.shape[1] != K or C.shape != (M_total, N) or offsets.numel() != G + 1:
        raise ValueError("shape mismatch")
    e = _epi(epi)
    sBias = 0
    if e != EPI_NONE:
        _need(bias, "bias", torch.bfloat16, (2,))
        sBias = bias.stride(0)
    st = load_library().wst_grouped_gemm_bf16(
        G, M_total, N, K, A.data_ptr(), A.stride(0), B.data_ptr(), B.stride(1), B.stride(0),
        offsets.data_ptr(), _ptr(bias) if e else None, sBias, C.data_ptr(), C.stride(0),
        _ctype(C), e, workspace.data_ptr(), _stream_handle(stream))
    _check(st, "wst_grouped_gemm_bf16")


def wst_ikbo_linear_compress(U, Cf, W, user_offsets, Y, workspace, stream=None) -> None:
    """Y[c] = W . concat(U[user(c)], Cf[c]) with the user part computed once per user.

    U: bf16 [users,Du,D]; Cf: bf16 [cand,Dc,D]; W: bf16 [O,Du+Dc];
    user_offsets: device int32 [users+1]; Y: fp32 [cand,O,D]; workspace of
    wst_workspace_size(users, O, D) bytes."""
    for t, n, d in ((U, "U", 3), (Cf, "Cf", 3), (W, "W", 2)):
        _need(t, n, torch.bfloat16, (d,))
        if not t.is_contiguous():
            raise ValueError("%s must be contiguous" % n)
    _need(Y, "Y", torch.float32, (3,))
    _need(user_offsets, "user_offsets", torch.int32, (1,))
    if not Y.is_contiguous():
        raise ValueError("Y must be contiguous")
    if not user_offsets.is_contiguous():
        raise ValueError("user_offsets must be contiguous")
    users, Du, D = U.shape
    cand, Dc, D2 = Cf.shape
    O, F = W.shape
    if D2 != D or F != Du + Dc or Y.shape != (cand, O, D) or user_offsets.numel() != users + 1:
        raise ValueError("shape mismatch")
    need = wst_workspace_size(users, O, D)
    if workspace.numel() * workspace.element_size() < need:
        raise ValueError("workspace too small: %d < %d bytes" % (workspace.numel(), need))
    st = load_library().wst_ikbo_linear_compress(
        users, cand, Du, Dc, D, O, U.data_ptr(), Cf.data_ptr(), W.data_ptr(),
        user_offsets.data_ptr(), Y.data_ptr(), workspace.data_ptr(), _stream_handle(stream))
    _check(st, "wst_ikbo_linear_compress")


def wst_ikbo_attention_bf16(Q, K, V, user_offsets, O, Lq: int = 1, scale=None, workspace=None,
                            stream=None) -> None:
    """IKBO attention: every query row of a candidate of user u attends over
    u's context, per head: O[r][h] = softmax(scale * Q[r][h] . K[u][:, h]^T) V[u][:, h].

    Q: bf16 [cand*Lq, H, Dh]; K, V: bf16 [users, Lkv, H, Dh];
    user_offsets: device int32 [users+1] (candidates per user);
    O: fp32 or bf16 [cand*Lq, H, Dh]; scale defaults to 1/sqrt(Dh).
    workspace: attention_workspace() splits the last partial wave of items by
    key blocks over all SMs; a smaller one (workspace()) schedules whole
    items only."""
    for t, n in ((Q, "Q"), (K, "K"), (V, "V")):
        _need(t, n, torch.bfloat16, (3,) if n == "Q" else (4,))
        if not t.is_contiguous():
            raise ValueError("%s must be contiguous" % n)
    _need(user_offsets, "user_offsets", torch.int32, (1,))
    if O.dtype not in (torch.float32, torch.bfloat16) or not O.is_contiguous():
        raise ValueError("O must be a contiguous fp32 or bf16 tensor")
    users, Lkv, H, Dh = K.shape
    nq = Q.shape[0]
    if V.shape != K.shape or Q.shape[1:] != (H, Dh) or O.shape != Q.shape or nq % Lq:
        raise ValueError("shape mismatch")
    if user_offsets.numel() != users + 1:
        raise ValueError("user_offsets needs users+1 entries")
    if scale is None:
        scale = 1.0 / math.sqrt(Dh)
    if workspace is None:
        raise ValueError("workspace is required")
    st = load_library().wst_ikbo_attention_bf16(
        users, nq // Lq, Lq, H, Dh, Lkv, Q.data_ptr(), K.data_ptr(), V.data_ptr(),
        user_offsets.data_ptr(), float(scale), O.data_ptr(),
        F32 if O.dtype == torch.float32 else BF16, workspace.data_ptr(),
        workspace.numel() * workspace.element_size(), _stream_handle(stream))
    _check(st, "wst_ikbo_attention_bf16")


def wst_ikbo_attention_workspace_size() -> int:
    return int(load_library().wst_ikbo_attention_workspace_size())


def attention_workspace(device=None, stream=None) -> torch.Tensor:
    """A zero-filled workspace for wst_ikbo_attention_bf16's split schedule."""
    ws = torch.empty(wst_ikbo_attention_workspace_size(), dtype=torch.uint8,
                     device=device or "cuda")
    wst_workspace_init(ws, stream)
    return ws


def wst_ikbo_linear_compress_noalloc(U, Cf, W, user_offsets, Y, status=None,
                                     stream=None) -> None:
    """wst_ikbo_linear_compress without a workspace, for callers that cannot
    allocate device memory at call time: the scratch lives in a fixed 4 MiB
    device array inside the library (shared by every call on the device, so
    overlapping calls race).  status: optional device int32 tensor that
    receives the call's device-side status code."""
    for t, n, d in ((U, "U", 3), (Cf, "Cf", 3), (W, "W", 2)):
        _need(t, n, torch.bfloat16, (d,))
        if not t.is_contiguous():
            raise ValueError("%s must be contiguous" % n)
    _need(Y, "Y", torch.float32, (3,))
    _need(user_offsets, "user_offsets", torch.int32, (1,))
    if not Y.is_contiguous():
        raise ValueError("Y must be contiguous")
    if not user_offsets.is_contiguous():
        raise ValueError("user_offsets must be contiguous")
    if status is not None:
        _need(status, "status", torch.int32, (1,))
        if not status.is_contiguous():
            raise ValueError("status must be contiguous")
    users, Du, D = U.shape
    cand, Dc, D2 = Cf.shape
    O, F = W.shape
    if D2 != D or F != Du + Dc or Y.shape != (cand, O, D) or user_offsets.numel() != users + 1:
        raise ValueError("shape mismatch")
    st = load_library().wst_ikbo_linear_compress_noalloc(
        users, cand, Du, Dc, D, O, U.data_ptr(), Cf.data_ptr(), W.data_ptr(),
        user_offsets.data_ptr(), Y.data_ptr(), _ptr(status), _stream_handle(stream))
    _check(st, "wst_ikbo_linear_compress_noalloc")


def wst_sync_status(workspace, stream=None) -> int:
    """Synchronize the stream; return (and clear) the first device-side error code."""
    return int(load_library().wst_sync_status(workspace.data_ptr(), _stream_handle(stream)))


# ----------------------------------------------------------------------------
# expert parallelism: host plans and GPU row movement
# ----------------------------------------------------------------------------
def _i32p(a):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_int))


def wst_ep_dispatch_plan(routing, num_experts: int, world_size: int):
    """Host plan of the pairs this rank sends (see include/wst.h).

    routing: int32 array [tokens, top_k] of expert ids (numpy or CPU tensor).
    Returns numpy int32 arrays (send_counts [world_size], send_group_counts
    [num_experts], send_pairs [tokens*top_k])."""
    import numpy as np
    r = np.ascontiguousarray(np.asarray(routing, dtype=np.int32))
    if r.ndim != 2:
        raise ValueError("routing must be [tokens, top_k]")
    T, k = r.shape
    send_counts = np.zeros(world_size, dtype=np.int32)
    group_counts = np.zeros(num_experts, dtype=np.int32)
    pairs = np.zeros(max(T * k, 1), dtype=np.int32)
    _check(load_library().wst_ep_dispatch_plan(T, k, _i32p(r), num_experts, world_size,
                                               _i32p(send_counts), _i32p(group_counts), _i32p(pairs)),
           "wst_ep_dispatch_plan")
    return send_counts, group_counts, pairs[:T * k]


def wst_ep_receive_plan(recv_group_counts):
    """Host plan ordering received rows by local expert.

    recv_group_counts: int32 [world_size, experts_per_rank].  Returns numpy
    int32 arrays (group_offsets [experts_per_rank+1], expert_rows [rows])."""
    import numpy as np
    c = np.ascontiguousarray(np.asarray(recv_group_counts, dtype=np.int32))
    if c.ndim != 2:
        raise ValueError("recv_group_counts must be [world_size, experts_per_rank]")
    R, E = c.shape
    offsets = np.zeros(E + 1, dtype=np.int32)
    rows = np.zeros(max(int(c.astype(np.int64).sum()), 1), dtype=np.int32)
    _check(load_library().wst_ep_receive_plan(R, E, _i32p(c), _i32p(offsets), _i32p(rows)),
           "wst_ep_receive_plan")
    return offsets, rows[:int(offsets[-1])]


def wst_permute_rows(src, dst, src_index=None, dst_index=None, n_rows=None, workspace=None,
                     stream=None) -> None:
    """dst[dst_index[i] (or i)] = src[src_index[i] (or i)] for i < n_rows, on the GPU.

    src, dst: CUDA tensors of rows (2-D, last dimension contiguous, the same
    bytes per row); src_index / dst_index: CUDA int32 tensors or None;
    n_rows defaults to the index length (else the source's rows)."""
    for t, n in ((src, "src"), (dst, "dst")):
        _need(t, n, None, (2,))
    row_bytes = src.shape[1] * src.element_size()
    if dst.shape[1] * dst.element_size() != row_bytes:
        raise ValueError("src and dst rows differ in size")
    for t, n in ((src_index, "src_index"), (dst_index, "dst_index")):
        if t is not None:
            _need(t, n, torch.int32, (1,))
    if n_rows is None:
        idx = src_index if src_index is not None else dst_index
        n_rows = idx.numel() if idx is not None else src.shape[0]
    if workspace is None:
        raise ValueError("workspace is required (see workspace())")
    st = load_library().wst_permute_rows(
        int(n_rows), row_bytes, src.data_ptr(), src.stride(0) * src.element_size(), _ptr(src_index),
        src.shape[0], dst.data_ptr(), dst.stride(0) * dst.element_size(), _ptr(dst_index),
        dst.shape[0], workspace.data_ptr(), _stream_handle(stream))
    _check(st, "wst_permute_rows")
