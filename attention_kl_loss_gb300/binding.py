"""ctypes binding of the C ABI in ``include/streamkl.h``.

Argument marshalling only: every step of the computation runs in the CUDA
library. PyTorch provides device memory and the current stream. The library
must have been built in-tree (``__graft_entry__.build()`` or
``python -m attention_kl_loss_gb300.build``); there is no fallback.
"""
from __future__ import annotations

import contextlib
import ctypes
import math
import os
from typing import Optional

import torch

from . import build as _build

STREAMKL_OK = 0
STREAMKL_ERR_INVALID_ARG = 1
STREAMKL_ERR_UNSUPPORTED = 2
STREAMKL_ERR_CUDA = 3
STREAMKL_ERR_TIMEOUT = 4
STREAMKL_ERR_DEVICE_CHECK = 5

_STATUS_NAMES = {0: "OK", 1: "INVALID_ARG", 2: "UNSUPPORTED", 3: "CUDA", 4: "TIMEOUT",
                 5: "DEVICE_CHECK"}

# loaded libraries: False = release build, True = debug build (device checks)
_libs: dict = {}
_use_debug = False

_P = ctypes.c_void_p
_I = ctypes.c_int
_F = ctypes.c_float
_Z = ctypes.c_size_t

_SIGNATURES = {
    "streamkl_status_string": (ctypes.c_char_p, [_I]),
    "streamkl_last_error": (ctypes.c_char_p, []),
    "streamkl_choose_splits": (_I, [_I, _I, _I, _I, _I, _I]),
    "streamkl_fwd_workspace_size": (_Z, [_I, _I, _I, _I, _I, _I, _I]),
    "streamkl_bwd_workspace_size": (_Z, [_I, _I, _I, _I, _I, _I, _I]),
    "streamkl_workspace_size": (_Z, [_I, _I, _I, _I, _I, _I, _I]),
    "streamkl_fwd": (_I, [_P, _P, _P, _P, _I, _I, _I, _I, _I, _F, _I, _I, _P, _P, _P, _P, _Z,
                          _P, _P]),
    "streamkl_bwd": (_I, [_P, _P, _P, _P, _I, _I, _I, _I, _I, _F, _I, _P, _P, _P, _P, _P, _P,
                          _P, _P, _P, _Z, _P, _P]),
    "streamkl_fwd_reverse": (_I, [_P, _P, _P, _P, _I, _I, _I, _I, _I, _F, _I, _I, _P, _P, _P,
                                  _P, _Z, _P, _P]),
    "streamkl_bwd_reverse": (_I, [_P, _P, _P, _P, _I, _I, _I, _I, _I, _F, _I, _P, _P, _P, _P, _P,
                                  _P, _P, _P, _P, _Z, _P, _P]),
    "streamkl_selftest_wait_timeout": (_I, [_P, ctypes.c_uint, _P]),
    "streamkl_selftest_device_check": (_I, [_P, _P]),
    "streamkl_fwd_pairs": (_I, [_I, _I, _I, _I, _I, _I, _I]),
    "streamkl_set_fwd_pairs": (_I, [_I]),
    "streamkl_bwd_algorithm": (_I, [_I, _I, _I, _I, _I, _I, _I]),
    "streamkl_set_bwd_algorithm": (_I, [_I]),
    "streamkl_bwd_dq_splits": (_I, [_I, _I, _I, _I, _I, _I, _I]),
    "streamkl_set_bwd_dq_splits": (_I, [_I]),
    "streamkl_bwd_dk_persist": (_I, [_I, _I, _I, _I, _I, _I]),
    "streamkl_set_bwd_dk_persist": (_I, [_I]),
    "streamkl_fwd_noalloc": (_I, [_P, _P, _P, _P, _I, _I, _I, _I, _I, _F, _I, _I, _P, _P, _P,
                                  _P, _P]),
    "streamkl_fwd_varlen": (_I, [_P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _F, _I,
                                 _P, _P, _P, _P, _P]),
    "streamkl_bwd_varlen": (_I, [_P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _F, _I,
                                 _P, _P, _P, _P, _P, _P, _P, _P, _P, _P]),
}


class StreamKLError(RuntimeError):
    def __init__(self, status: int, where: str, detail: str = ""):
        self.status = status
        name = _STATUS_NAMES.get(status, "?")
        super().__init__(f"{where}: STREAMKL_ERR_{name} ({status}) {detail}".strip())


def library_path(debug: bool = False) -> str:
    return _build.lib_path(debug)


def _load_variant(debug: bool) -> ctypes.CDLL:
    if debug in _libs:
        return _libs[debug]
    path = library_path(debug)
    if not os.path.exists(path):
        how = ("`python -m attention_kl_loss_gb300.build --debug`" if debug
               else "`python -c 'import __graft_entry__ as g; g.build()'`")
        raise RuntimeError(f"StreamKL CUDA library not found at {path}; build it with {how}")
    lib = ctypes.CDLL(path)
    for name, (res, args) in _SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _libs[debug] = lib
    return lib


def load(debug: Optional[bool] = None) -> ctypes.CDLL:
    """Load the in-tree library (raises if it has not been built): the one the
    binding's calls use (the debug build inside ``use_debug_library()``), or
    the release / debug build when ``debug`` is given."""
    return _load_variant(_use_debug if debug is None else debug)


@contextlib.contextmanager
def use_debug_library():
    """Route this module's calls to the debug build (device-side range checks
    that report STREAMKL_ERR_DEVICE_CHECK) for the duration of the block."""
    global _use_debug
    prev = _use_debug
    lib = _load_variant(True)
    _use_debug = True
    try:
        yield lib
    finally:
        _use_debug = prev


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream_handle(stream: Optional[torch.cuda.Stream]):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _check(status: int, where: str):
    if status != STREAMKL_OK:
        detail = load().streamkl_last_error().decode(errors="replace")
        raise StreamKLError(status, where, detail)


def _dims(q1, k1, q2, k2):
    for name, t in (("q1", q1), ("k1", k1), ("q2", q2), ("k2", k2)):
        if not isinstance(t, torch.Tensor) or t.dim() != 4:
            raise ValueError(f"{name} must be a 4-D tensor [B, H, N, d]")
        if t.dtype != torch.bfloat16 or not t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous bf16 CUDA tensor")
    B, H, NQ, d = q1.shape
    NK = k1.shape[2]
    if q2.shape != q1.shape or k1.shape != (B, H, NK, d) or k2.shape != k1.shape:
        raise ValueError("shape mismatch: Q1,Q2 must be [B,H,NQ,d] and K1,K2 [B,H,NK,d]")
    return B, H, NQ, NK, d


def choose_splits(B, H, NQ, NK, d, causal) -> int:
    return int(load().streamkl_choose_splits(B, H, NQ, NK, d, int(causal)))


def streamkl_fwd_workspace_size(B, H, NQ, NK, d, causal, num_splits=0) -> int:
    return int(load().streamkl_fwd_workspace_size(B, H, NQ, NK, d, int(causal), int(num_splits)))


def streamkl_bwd_workspace_size(B, H, NQ, NK, d, causal, want_grad1) -> int:
    return int(load().streamkl_bwd_workspace_size(B, H, NQ, NK, d, int(causal), int(want_grad1)))


def streamkl_workspace_size(B, H, NQ, NK, d, causal, want_grad1) -> int:
    return int(load().streamkl_workspace_size(B, H, NQ, NK, d, int(causal), int(want_grad1)))


BWD_SEPARATE = 0
BWD_FUSED = 1


def bwd_algorithm(B, H, NQ, NK, d, causal, want_grad1=False) -> int:
    """0 = separate dK/dQ kernels, 1 = fused kernel with dQ atomics."""
    return int(load().streamkl_bwd_algorithm(B, H, NQ, NK, d, int(causal), int(want_grad1)))


def bwd_dq_splits(B, H, NQ, NK, d, causal, want_grad1=False) -> int:
    """Key splits of the separate backward's dQ kernel for these sizes."""
    return int(load().streamkl_bwd_dq_splits(B, H, NQ, NK, d, int(causal), int(want_grad1)))


def set_bwd_dq_splits(splits: Optional[int]) -> None:
    """Force the dQ kernel's key splits (None or 0: automatic)."""
    if load().streamkl_set_bwd_dq_splits(0 if splits is None else int(splits)) != 0:
        raise ValueError(f"invalid dQ split count {splits!r}")


def bwd_dk_persist(B, H, NQ, NK, d, causal) -> int:
    """Persistent dK CTAs the backward launches for these sizes (0: none)."""
    return int(load().streamkl_bwd_dk_persist(B, H, NQ, NK, d, int(causal)))


def set_bwd_dk_persist(ctas: Optional[int]) -> None:
    """Force the persistent dK kernel (n CTAs), turn it off (-1), or None/0: automatic."""
    if load().streamkl_set_bwd_dk_persist(0 if ctas is None else int(ctas)) != 0:
        raise ValueError(f"invalid persistent dK CTA count {ctas!r}")


def fwd_pairs(B, H, NQ, NK, d, causal, num_splits=0) -> bool:
    """Whether streamkl_fwd runs as CTA pairs (cta_group::2) for these sizes."""
    return int(load().streamkl_fwd_pairs(B, H, NQ, NK, d, int(causal), int(num_splits))) == 1


def set_fwd_pairs(enabled: Optional[bool]) -> None:
    """Use CTA pairs in the forward where the sizes allow (True), or not
    (False / None: the default), for this process."""
    load().streamkl_set_fwd_pairs(1 if enabled else 0)


def set_bwd_algorithm(algo: Optional[int]) -> None:
    """Force the backward algorithm process-wide (None = automatic)."""
    v = -1 if algo is None else int(algo)
    if load().streamkl_set_bwd_algorithm(v) != 0:
        raise ValueError(f"invalid backward algorithm {algo!r}")


def new_status(device=None) -> torch.Tensor:
    """A zeroed device status word for the kernels' bounded waits."""
    return torch.zeros(1, dtype=torch.int32, device=device or "cuda")


def _workspace(nbytes: int, device, workspace):
    if nbytes == 0:
        return None
    if workspace is not None:
        if workspace.numel() * workspace.element_size() < nbytes:
            raise ValueError(f"workspace too small: need {nbytes} bytes")
        return workspace
    return torch.empty(nbytes, dtype=torch.uint8, device=device)


def _fwd_call(entry, q1, k1, q2, k2, scale, causal, num_splits, out, workspace, dev_status,
              stream):
    lib = load()
    B, H, NQ, NK, d = _dims(q1, k1, q2, k2)
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    dev = q1.device
    if out is None:
        out = tuple(torch.empty((B, H, NQ), dtype=torch.float32, device=dev) for _ in range(3))
    kl, lse1, lse2 = out
    need = streamkl_fwd_workspace_size(B, H, NQ, NK, d, causal, num_splits)
    ws = _workspace(need, dev, workspace)
    status = dev_status if dev_status is not None else new_status(dev)
    st = getattr(lib, entry)(_ptr(q1), _ptr(k1), _ptr(q2), _ptr(k2), B, H, NQ, NK, d, scale,
                             int(causal), int(num_splits), _ptr(kl), _ptr(lse1), _ptr(lse2),
                             _ptr(ws), need if ws is not None else 0, _ptr(status),
                             _stream_handle(stream))
    _check(st, entry)
    return kl, lse1, lse2


def streamkl_fwd(q1, k1, q2, k2, scale: Optional[float] = None, causal: bool = False,
                 num_splits: int = 0, out=None, workspace=None, dev_status=None, stream=None):
    """Per-row KL(P1||P2), lse1, lse2 (fp32 [B, H, N_Q]) via the CUDA library."""
    return _fwd_call("streamkl_fwd", q1, k1, q2, k2, scale, causal, num_splits, out, workspace,
                     dev_status, stream)


def streamkl_fwd_reverse(q1, k1, q2, k2, scale: Optional[float] = None, causal: bool = False,
                         num_splits: int = 0, out=None, workspace=None, dev_status=None,
                         stream=None):
    """Per-row KL(P2||P1) (the reverse direction), lse1, lse2 (fp32 [B, H, N_Q])."""
    return _fwd_call("streamkl_fwd_reverse", q1, k1, q2, k2, scale, causal, num_splits, out,
                     workspace, dev_status, stream)


def streamkl_fwd_noalloc(q1, k1, q2, k2, out, scale: Optional[float] = None,
                         causal: bool = False, num_splits: int = 0, dev_status=None, stream=None):
    """Forward pass through the library's allocation-free entry point.

    For callers that cannot allocate device memory: the outputs ``out`` =
    (kl, lse1, lse2) must be given, and the split scratch is the library's
    built-in 16 MiB array (shared by every call on the device)."""
    lib = load()
    B, H, NQ, NK, d = _dims(q1, k1, q2, k2)
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    kl, lse1, lse2 = out
    if dev_status is None:
        raise ValueError("dev_status must be given (this path allocates nothing)")
    st = lib.streamkl_fwd_noalloc(_ptr(q1), _ptr(k1), _ptr(q2), _ptr(k2), B, H, NQ, NK, d, scale,
                                  int(causal), int(num_splits), _ptr(kl), _ptr(lse1), _ptr(lse2),
                                  _ptr(dev_status), _stream_handle(stream))
    _check(st, "streamkl_fwd_noalloc")
    return kl, lse1, lse2


def _bwd_call(entry, q1, k1, q2, k2, kl, lse1, lse2, dkl, scale, causal, grad1, grad2, out,
              workspace, dev_status, stream):
    if not (grad1 or grad2):
        raise ValueError("no gradient requested (grad1 and grad2 both False)")
    lib = load()
    B, H, NQ, NK, d = _dims(q1, k1, q2, k2)
    for name, t in (("kl", kl), ("lse1", lse1), ("lse2", lse2), ("dkl", dkl)):
        if t.dtype != torch.float32 or not t.is_cuda or not t.is_contiguous() or t.shape != (B, H, NQ):
            raise ValueError(f"{name} must be a contiguous fp32 CUDA tensor [B, H, N_Q]")
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    dev = q1.device
    if out is None:
        dq2 = torch.empty_like(q2) if grad2 else None
        dk2 = torch.empty_like(k2) if grad2 else None
        dq1 = torch.empty_like(q1) if grad1 else None
        dk1 = torch.empty_like(k1) if grad1 else None
    else:
        dq2, dk2, dq1, dk1 = out
    # sized for the sets requested (want_grad1 = both), which covers either
    # direction: the fused kernel's accumulators or the dQ split's partials
    need = streamkl_bwd_workspace_size(B, H, NQ, NK, d, causal, grad1 and grad2)
    ws = _workspace(need, dev, workspace)
    status = dev_status if dev_status is not None else new_status(dev)
    st = getattr(lib, entry)(_ptr(q1), _ptr(k1), _ptr(q2), _ptr(k2), B, H, NQ, NK, d, scale,
                             int(causal), _ptr(kl), _ptr(lse1), _ptr(lse2), _ptr(dkl), _ptr(dq2),
                             _ptr(dk2), _ptr(dq1), _ptr(dk1), _ptr(ws), need, _ptr(status),
                             _stream_handle(stream))
    _check(st, entry)
    return dq2, dk2, dq1, dk1


def streamkl_bwd(q1, k1, q2, k2, kl, lse1, lse2, dkl, scale: Optional[float] = None,
                 causal: bool = False, grad1: bool = False, out=None, workspace=None,
                 dev_status=None, stream=None, grad2: bool = True):
    """Gradients of sum(dkl * KL): (dq2, dk2, dq1, dk1), bf16. dq2/dk2
    (configuration 1, P1 fixed) unless ``grad2`` is False; dq1/dk1
    (configuration 2, P2 fixed) only with ``grad1``; skipped ones are None."""
    return _bwd_call("streamkl_bwd", q1, k1, q2, k2, kl, lse1, lse2, dkl, scale, causal, grad1,
                     grad2, out, workspace, dev_status, stream)


def streamkl_bwd_reverse(q1, k1, q2, k2, kl, lse1, lse2, dkl, scale: Optional[float] = None,
                         causal: bool = False, grad1: bool = False, out=None, workspace=None,
                         dev_status=None, stream=None, grad2: bool = True):
    """Gradients of sum(dkl * KL(P2||P1)), with kl, lse1, lse2 from
    streamkl_fwd_reverse: (dq2, dk2, dq1, dk1), bf16. dq2/dk2 (the student's,
    P1 fixed) unless ``grad2`` is False; dq1/dk1 (the teacher's, P2 fixed)
    only with ``grad1``; skipped ones are None."""
    return _bwd_call("streamkl_bwd_reverse", q1, k1, q2, k2, kl, lse1, lse2, dkl, scale, causal,
                     grad1, grad2, out, workspace, dev_status, stream)


def _packed_dims(q1, k1, q2, k2, cu_seqlens_q, cu_seqlens_k):
    for name, t in (("q1", q1), ("k1", k1), ("q2", q2), ("k2", k2)):
        if not isinstance(t, torch.Tensor) or t.dim() != 3:
            raise ValueError(f"{name} must be a 3-D packed tensor [total, H, d]")
        if t.dtype != torch.bfloat16 or not t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous bf16 CUDA tensor")
    TQ, H, d = q1.shape
    TK = k1.shape[0]
    if q2.shape != q1.shape or k1.shape != (TK, H, d) or k2.shape != k1.shape:
        raise ValueError("shape mismatch: Q1,Q2 must be [total_q,H,d] and K1,K2 [total_k,H,d]")
    for name, t in (("cu_seqlens_q", cu_seqlens_q), ("cu_seqlens_k", cu_seqlens_k)):
        if t.dtype != torch.int32 or not t.is_cuda or t.dim() != 1 or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous int32 CUDA vector [B + 1]")
    if cu_seqlens_k.numel() != cu_seqlens_q.numel() or cu_seqlens_q.numel() < 2:
        raise ValueError("cu_seqlens_q and cu_seqlens_k must both have B + 1 >= 2 entries")
    return cu_seqlens_q.numel() - 1, H, TQ, TK, d


def streamkl_fwd_varlen(q1, k1, q2, k2, cu_seqlens_q, cu_seqlens_k, max_seqlen_q: int,
                        max_seqlen_k: int, scale: Optional[float] = None, causal: bool = False,
                        out=None, dev_status=None, stream=None):
    """Forward for a packed variable-length batch: q1/q2 [total_q, H, d],
    k1/k2 [total_k, H, d] bf16, cu_seqlens_* int32 device offsets [B + 1].
    Returns (kl, lse1, lse2), fp32 [total_q, H]."""
    lib = load()
    B, H, TQ, TK, d = _packed_dims(q1, k1, q2, k2, cu_seqlens_q, cu_seqlens_k)
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    dev = q1.device
    if out is None:
        out = tuple(torch.empty((TQ, H), dtype=torch.float32, device=dev) for _ in range(3))
    kl, lse1, lse2 = out
    status = dev_status if dev_status is not None else new_status(dev)
    st = lib.streamkl_fwd_varlen(_ptr(q1), _ptr(k1), _ptr(q2), _ptr(k2), _ptr(cu_seqlens_q),
                                 _ptr(cu_seqlens_k), B, H, TQ, TK, int(max_seqlen_q),
                                 int(max_seqlen_k), d, scale, int(causal), _ptr(kl), _ptr(lse1),
                                 _ptr(lse2), _ptr(status), _stream_handle(stream))
    _check(st, "streamkl_fwd_varlen")
    return kl, lse1, lse2


def streamkl_bwd_varlen(q1, k1, q2, k2, cu_seqlens_q, cu_seqlens_k, max_seqlen_q: int,
                        max_seqlen_k: int, kl, lse1, lse2, dkl, scale: Optional[float] = None,
                        causal: bool = False, grad1: bool = False, grad2: bool = True, out=None,
                        dev_status=None, stream=None):
    """Backward for a packed variable-length batch; returns (dq2, dk2, dq1,
    dk1) shaped like the inputs, None where not requested."""
    if not (grad1 or grad2):
        raise ValueError("no gradient requested (grad1 and grad2 both False)")
    lib = load()
    B, H, TQ, TK, d = _packed_dims(q1, k1, q2, k2, cu_seqlens_q, cu_seqlens_k)
    for name, t in (("kl", kl), ("lse1", lse1), ("lse2", lse2), ("dkl", dkl)):
        if t.dtype != torch.float32 or not t.is_cuda or not t.is_contiguous() or t.shape != (TQ, H):
            raise ValueError(f"{name} must be a contiguous fp32 CUDA tensor [total_q, H]")
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    if out is None:
        dq2 = torch.empty_like(q2) if grad2 else None
        dk2 = torch.empty_like(k2) if grad2 else None
        dq1 = torch.empty_like(q1) if grad1 else None
        dk1 = torch.empty_like(k1) if grad1 else None
    else:
        dq2, dk2, dq1, dk1 = out
    status = dev_status if dev_status is not None else new_status(q1.device)
    st = lib.streamkl_bwd_varlen(_ptr(q1), _ptr(k1), _ptr(q2), _ptr(k2), _ptr(cu_seqlens_q),
                                 _ptr(cu_seqlens_k), B, H, TQ, TK, int(max_seqlen_q),
                                 int(max_seqlen_k), d, scale, int(causal), _ptr(kl), _ptr(lse1),
                                 _ptr(lse2), _ptr(dkl), _ptr(dq2), _ptr(dk2), _ptr(dq1), _ptr(dk1),
                                 _ptr(status), _stream_handle(stream))
    _check(st, "streamkl_bwd_varlen")
    return dq2, dk2, dq1, dk1


def selftest_wait_timeout(timeout_us: int = 20000, dev_status=None, stream=None) -> torch.Tensor:
    """Run the bounded-wait self-test kernel; returns the status tensor."""
    lib = load()
    status = dev_status if dev_status is not None else new_status()
    _check(lib.streamkl_selftest_wait_timeout(_ptr(status), int(timeout_us), _stream_handle(stream)),
           "streamkl_selftest_wait_timeout")
    return status


def selftest_device_check(dev_status=None, stream=None) -> torch.Tensor:
    """Run the range-check self-test kernel; returns the status tensor
    (STREAMKL_ERR_DEVICE_CHECK from the debug build, unchanged from the
    release build)."""
    lib = load()
    status = dev_status if dev_status is not None else new_status()
    _check(lib.streamkl_selftest_device_check(_ptr(status), _stream_handle(stream)),
           "streamkl_selftest_device_check")
    return status


def raise_on_device_status(dev_status: torch.Tensor, where: str = "kernel"):
    """Synchronise and raise if a kernel recorded a failure in ``dev_status``."""
    torch.cuda.synchronize(dev_status.device)
    v = int(dev_status.item())
    if v != 0:
        why = {STREAMKL_ERR_TIMEOUT: "a bounded wait inside the kernel gave up",
               STREAMKL_ERR_INVALID_ARG: "malformed sequence offsets or causal rows without a key",
               STREAMKL_ERR_DEVICE_CHECK: "a device-side range check failed (debug build)"}
        raise StreamKLError(v, where, why.get(v, "kernel failure"))
