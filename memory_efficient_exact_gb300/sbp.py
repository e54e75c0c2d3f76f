"""Python binding of libsbp.so (argument marshalling only).

Every function here checks shapes, takes raw device pointers from PyTorch tensors,
and calls the C entry point of the same name (see ``include/sbp.h``).  All
arithmetic runs in the library's CUDA kernels; PyTorch only provides device memory
and the current stream.  Importing this module loads the library and raises if it
has not been built (``__graft_entry__.build()``) -- there is no other code path.
"""
from __future__ import annotations

import ctypes
import os
import re

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
# SBP_LIBRARY_VARIANT selects a build of the same sources: "" (default), "checked" (guard
# zones around workspace regions) or "nvtx" (NVTX ranges); see _build.py
VARIANT = os.environ.get("SBP_LIBRARY_VARIANT", "")
if VARIANT not in ("", "checked", "nvtx"):
    raise ImportError(f"SBP_LIBRARY_VARIANT={VARIANT!r}: one of '', 'checked', 'nvtx'")
LIB_PATH = os.path.join(_HERE, f"libsbp_{VARIANT}.so" if VARIANT else "libsbp.so")
HEADER = os.path.join(os.path.dirname(_HERE), "include", "sbp.h")

(OK, ERR_INVALID_ARG, ERR_ALIGNMENT, ERR_WORKSPACE, ERR_LABEL_RANGE, ERR_TIMEOUT, ERR_CUDA, ERR_UNSUPPORTED,
 ERR_SCRATCH_LIMIT, ERR_WORKSPACE_OVERRUN) = range(10)
NOALLOC_SCRATCH_BYTES = 64 * 1024 * 1024
BF16, FP32 = 0, 1
MODE_SFT, MODE_GRPO, MODE_DPO1, MODE_DPO2 = 0, 1, 2, 3
IGNORE_INDEX = -100


class SbpError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {status_string(code)} ({code})")


def _load() -> ctypes.CDLL:
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"{LIB_PATH} is missing: build it with __graft_entry__.build() "
                          "(the LM-head kernels have no other implementation)")
    lib = ctypes.CDLL(LIB_PATH)
    P, I64, I32, F, SZ = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_float, ctypes.c_size_t
    C = ctypes.c_int
    lib.sbp_lmhead_workspace_bytes.restype = SZ
    lib.sbp_lmhead_workspace_bytes.argtypes = [I64, I64, I64, I64, C, C]
    lib.sbp_lmhead_workspace_bytes_lean.restype = SZ
    lib.sbp_lmhead_workspace_bytes_lean.argtypes = [I64, I64, I64, I64, C, C]
    lib.sbp_lmhead_sft.restype = C
    lib.sbp_lmhead_sft.argtypes = [P, P, P, I64, I64, I64, I64, I32, C, P, P, P, P, P, C, P, SZ, P, P]
    lib.sbp_lmhead_grpo.restype = C
    lib.sbp_lmhead_grpo.argtypes = [P, P, P, P, P, F, F, I64, I64, I64, I64, I32, C, P, P, P, P, P, C, P, SZ, P, P]
    lib.sbp_lmhead_grpo_ext.restype = C
    lib.sbp_lmhead_grpo_ext.argtypes = [P, P, P, P, P, F, F, P, F, P, I32, I64, I64, I64, I64, I32, C, P, P, P, P, P,
                                        C, P, SZ, P, P]
    lib.sbp_lmhead_dpo_pass1.restype = C
    lib.sbp_lmhead_dpo_pass1.argtypes = [P, P, P, P, I32, I64, I64, I64, I64, I32, C, P, P, P, P, SZ, P, P]
    lib.sbp_lmhead_dpo_pass2.restype = C
    lib.sbp_lmhead_dpo_pass2.argtypes = [P, P, P, P, I32, P, P, F, I64, I64, I64, I64, I32, C, P, P, P, P, C, P,
                                         SZ, P, P]
    lib.sbp_lmhead_sft_noalloc.restype = C
    lib.sbp_lmhead_sft_noalloc.argtypes = [P, P, P, I64, I64, I64, I64, I32, C, P, P, P, P, P, C, P, P]
    lib.sbp_lmhead_sft_host_workspace_bytes.restype = SZ
    lib.sbp_lmhead_sft_host_workspace_bytes.argtypes = [I64, I64, I64, I64, C]
    lib.sbp_lmhead_sft_host.restype = C
    lib.sbp_lmhead_sft_host.argtypes = [P, P, P, I64, I64, I64, I64, I32, C, P, P, P, P, C, P, SZ, P, P]
    lib.sbp_mlp_workspace_bytes.restype = SZ
    lib.sbp_mlp_workspace_bytes.argtypes = [I64, I64, I64, I64]
    lib.sbp_mlp_swiglu_backward.restype = C
    lib.sbp_mlp_swiglu_backward.argtypes = [P, P, P, P, I64, I64, I64, I64, P, P, P, C, P, SZ, P, P]
    lib.sbp_attn_workspace_bytes.restype = SZ
    lib.sbp_attn_workspace_bytes.argtypes = [I64, I64, I64, I64]
    lib.sbp_attn_causal_backward.restype = C
    lib.sbp_attn_causal_backward.argtypes = [P, P, P, P, P, P, I64, I64, I64, F, I64, P, P, P, C, P, SZ, P, P]
    lib.sbp_attn_causal_backward_gqa.restype = C
    lib.sbp_attn_causal_backward_gqa.argtypes = [P, P, P, P, P, P, I64, I64, I64, I64, F, I64, P, P, P, C, P, SZ, P,
                                                 P]
    lib.sbp_status_string.restype = ctypes.c_char_p
    lib.sbp_status_string.argtypes = [C]
    lib.sbp_last_launch_count.restype = C
    lib.sbp_last_launch_count.argtypes = []
    lib.sbp_profile_enable.restype = C
    lib.sbp_profile_enable.argtypes = [C]
    lib.sbp_profile_read.restype = C
    lib.sbp_profile_read.argtypes = [P, P, C]
    return lib


_lib = _load()


def header_functions() -> list[str]:
    """Names of the functions ``include/sbp.h`` declares."""
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(sbp_[a-z0-9_]+)\s*\(", src)))


def status_string(code: int) -> str:
    return _lib.sbp_status_string(int(code)).decode()


def last_launch_count() -> int:
    return int(_lib.sbp_last_launch_count())


KERNEL_CLASSES = ("forward_gemm", "backward_gemm", "logit_grad", "other")


def profile_enable(on: bool = True) -> None:
    _lib.sbp_profile_enable(1 if on else 0)


def profile_read() -> dict:
    """Per kernel class: (total ms, launches) recorded since the last read."""
    n = len(KERNEL_CLASSES)
    ms = (ctypes.c_double * n)()
    cnt = (ctypes.c_int64 * n)()
    r = _lib.sbp_profile_read(ctypes.cast(ms, ctypes.c_void_p), ctypes.cast(cnt, ctypes.c_void_p), n)
    if r < 0:
        raise SbpError(-r, "sbp_profile_read")
    return {k: (ms[i], cnt[i]) for i, k in enumerate(KERNEL_CLASSES)}


def workspace_bytes(T: int, d: int, V: int, chunk: int, dtype: int, mode: int) -> int:
    return int(_lib.sbp_lmhead_workspace_bytes(T, d, V, chunk, dtype, mode))


def workspace_bytes_lean(T: int, d: int, V: int, chunk: int, dtype: int, mode: int) -> int:
    """The smallest accepted workspace (one chunk buffer: the one-buffer schedule)."""
    return int(_lib.sbp_lmhead_workspace_bytes_lean(T, d, V, chunk, dtype, mode))


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _code(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return BF16
    if t.dtype == torch.float32:
        return FP32
    raise TypeError(f"unsupported dtype {t.dtype}: bf16 or fp32")


def _dev(*ts):
    for t in ts:
        if t is not None and (not t.is_cuda or not t.is_contiguous()):
            raise ValueError("tensors must be contiguous CUDA tensors")


def _stream(stream):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _check(code: int, where: str):
    if code != OK:
        raise SbpError(code, where)


def make_workspace(T, d, V, chunk, dtype, mode, device=None, lean=False) -> torch.Tensor:
    n = (workspace_bytes_lean if lean else workspace_bytes)(T, d, V, chunk, dtype, mode)
    if n == 0:
        raise SbpError(ERR_INVALID_ARG, "workspace_bytes")
    return torch.empty(n, dtype=torch.uint8, device=device or "cuda")


def _prep(H, W, labels, chunk, mode, workspace):
    _dev(H, W, labels)
    if labels.dtype != torch.int32:
        raise TypeError("labels must be int32")
    T, d = H.shape
    V = W.shape[0]
    if W.shape[1] != d or H.dtype != W.dtype or labels.shape != (T,):
        raise ValueError("shape/dtype mismatch between H [T,d], W [V,d], labels [T]")
    dt = _code(H)
    if workspace is None:
        workspace = make_workspace(T, d, V, chunk, dt, mode, H.device)
    return T, d, V, dt, workspace


def _grad_out(H, W, dH, dW):
    if dH is None:
        dH = torch.empty_like(H)
    if dW is None:
        dW = torch.empty(W.shape, dtype=torch.float32, device=W.device)
    _dev(dH, dW)
    return dH, dW


def sft(H, W, labels, chunk, ignore_index=IGNORE_INDEX, *, dH=None, dW=None, accumulate_dW=False,
        logp=True, workspace=None, status=None, stream=None) -> dict:
    """SFT cross-entropy forward + backward (``sbp_lmhead_sft``).  Returns device tensors."""
    T, d, V, dt, ws = _prep(H, W, labels, chunk, MODE_SFT, workspace)
    dH, dW = _grad_out(H, W, dH, dW)
    dev = H.device
    loss = torch.empty((), dtype=torch.float32, device=dev)
    nv = torch.empty((), dtype=torch.int64, device=dev)
    lp = torch.empty(T, dtype=torch.float32, device=dev) if logp else None
    st = torch.empty((), dtype=torch.int32, device=dev) if status is None else status
    _check(_lib.sbp_lmhead_sft(_p(H), _p(W), _p(labels), T, d, V, chunk, ignore_index, dt, _p(loss), _p(nv),
                               _p(lp), _p(dH), _p(dW), int(bool(accumulate_dW)), _p(ws), ws.numel(), _p(st),
                               _stream(stream)), "sbp_lmhead_sft")
    return dict(loss=loss, n_valid=nv, logp=lp, dH=dH, dW=dW, status=st)


def sft_noalloc(H, W, labels, chunk, ignore_index=IGNORE_INDEX, *, dH=None, dW=None, accumulate_dW=False,
                logp=True, status=None, stream=None) -> dict:
    """SFT forward + backward without a workspace (``sbp_lmhead_sft_noalloc``): for
    callers that cannot allocate device scratch.  The library works in its own fixed
    64 MiB device array, shared by all calls (overlapping calls race).  Output tensors
    are still the caller's."""
    _dev(H, W, labels)
    if labels.dtype != torch.int32:
        raise TypeError("labels must be int32")
    T, d = H.shape
    V = W.shape[0]
    if W.shape[1] != d or H.dtype != W.dtype or labels.shape != (T,):
        raise ValueError("shape/dtype mismatch between H [T,d], W [V,d], labels [T]")
    dt = _code(H)
    dH, dW = _grad_out(H, W, dH, dW)
    dev = H.device
    loss = torch.empty((), dtype=torch.float32, device=dev)
    nv = torch.empty((), dtype=torch.int64, device=dev)
    lp = torch.empty(T, dtype=torch.float32, device=dev) if logp else None
    st = torch.empty((), dtype=torch.int32, device=dev) if status is None else status
    _check(_lib.sbp_lmhead_sft_noalloc(_p(H), _p(W), _p(labels), T, d, V, chunk, ignore_index, dt, _p(loss),
                                       _p(nv), _p(lp), _p(dH), _p(dW), int(bool(accumulate_dW)), _p(st),
                                       _stream(stream)), "sbp_lmhead_sft_noalloc")
    return dict(loss=loss, n_valid=nv, logp=lp, dH=dH, dW=dW, status=st)


def host_workspace_bytes(T: int, d: int, V: int, chunk: int, dtype: int) -> int:
    """Workspace of ``sft_host``: the SFT workspace plus the row slots and the labels."""
    return int(_lib.sbp_lmhead_sft_host_workspace_bytes(T, d, V, chunk, dtype))


def sft_host(H, W, labels, chunk, ignore_index=IGNORE_INDEX, *, dH=None, dW=None, accumulate_dW=False,
             loss=None, n_valid=None, workspace=None, status=None, stream=None) -> dict:
    """SFT forward + backward with H, labels, dH, loss and N in host memory
    (``sbp_lmhead_sft_host``): the call streams the rows chunk by chunk.  H, labels and
    the host outputs should be pinned for the copies to overlap the GEMMs; W, dW, the
    workspace and the status are device tensors.  The host outputs are valid once the
    stream has been synchronised."""
    for t in (H, labels):
        if t.is_cuda or not t.is_contiguous():
            raise ValueError("H and labels must be contiguous host tensors")
    _dev(W)
    if labels.dtype != torch.int32:
        raise TypeError("labels must be int32")
    T, d = H.shape
    V = W.shape[0]
    if W.shape[1] != d or H.dtype != W.dtype or labels.shape != (T,):
        raise ValueError("shape/dtype mismatch between H [T,d], W [V,d], labels [T]")
    dt = _code(H)
    pin = H.is_pinned()
    if dH is None:
        dH = torch.empty(H.shape, dtype=H.dtype, pin_memory=pin)
    if dH.is_cuda or not dH.is_contiguous() or dH.shape != H.shape or dH.dtype != H.dtype:
        raise ValueError("dH must be a contiguous host tensor shaped and typed like H")
    if dW is None:
        dW = torch.empty(W.shape, dtype=torch.float32, device=W.device)
    _dev(dW)
    if loss is None:
        loss = torch.empty((), dtype=torch.float32, pin_memory=pin)
    if n_valid is None:
        n_valid = torch.empty((), dtype=torch.int64, pin_memory=pin)
    if workspace is None:
        n = host_workspace_bytes(T, d, V, chunk, dt)
        if n == 0:
            raise SbpError(ERR_INVALID_ARG, "sbp_lmhead_sft_host_workspace_bytes")
        workspace = torch.empty(n, dtype=torch.uint8, device=W.device)
    _dev(workspace)
    st = torch.empty((), dtype=torch.int32, device=W.device) if status is None else status
    _check(_lib.sbp_lmhead_sft_host(_p(H), _p(W), _p(labels), T, d, V, chunk, ignore_index, dt, _p(loss),
                                    _p(n_valid), _p(dH), _p(dW), int(bool(accumulate_dW)), _p(workspace),
                                    workspace.numel(), _p(st), _stream(stream)), "sbp_lmhead_sft_host")
    return dict(loss=loss, n_valid=n_valid, dH=dH, dW=dW, status=st)


def grpo(H, W, labels, advantages, logp_old, chunk, clip_lo=0.8, clip_hi=1.2, ignore_index=IGNORE_INDEX, *,
         dH=None, dW=None, accumulate_dW=False, logp=True, workspace=None, status=None, stream=None) -> dict:
    """GRPO / PPO-clip forward + backward (``sbp_lmhead_grpo``)."""
    T, d, V, dt, ws = _prep(H, W, labels, chunk, MODE_GRPO, workspace)
    _dev(advantages, logp_old)
    if advantages.dtype != torch.float32 or logp_old.dtype != torch.float32:
        raise TypeError("advantages and logp_old must be float32")
    dH, dW = _grad_out(H, W, dH, dW)
    dev = H.device
    loss = torch.empty((), dtype=torch.float32, device=dev)
    nv = torch.empty((), dtype=torch.int64, device=dev)
    lp = torch.empty(T, dtype=torch.float32, device=dev) if logp else None
    st = torch.empty((), dtype=torch.int32, device=dev) if status is None else status
    _check(_lib.sbp_lmhead_grpo(_p(H), _p(W), _p(labels), _p(advantages), _p(logp_old), clip_lo, clip_hi, T, d, V,
                                chunk, ignore_index, dt, _p(loss), _p(nv), _p(lp), _p(dH), _p(dW),
                                int(bool(accumulate_dW)), _p(ws), ws.numel(), _p(st), _stream(stream)),
           "sbp_lmhead_grpo")
    return dict(loss=loss, n_valid=nv, logp=lp, dH=dH, dW=dW, status=st)


def grpo_ext(H, W, labels, advantages, logp_old, chunk, clip_lo=0.8, clip_hi=1.2, ref_logp=None, kl_coef=0.0,
             cu_seqlens=None, ignore_index=IGNORE_INDEX, *, dH=None, dW=None, accumulate_dW=False, logp=True,
             workspace=None, status=None, stream=None) -> dict:
    """GRPO / PPO-clip with an optional KL penalty and per-sequence mean (``sbp_lmhead_grpo_ext``)."""
    T, d, V, dt, ws = _prep(H, W, labels, chunk, MODE_GRPO, workspace)
    _dev(advantages, logp_old, ref_logp, cu_seqlens)
    if advantages.dtype != torch.float32 or logp_old.dtype != torch.float32:
        raise TypeError("advantages and logp_old must be float32")
    if ref_logp is not None and ref_logp.dtype != torch.float32:
        raise TypeError("ref_logp must be float32")
    n_seq = 0 if cu_seqlens is None else cu_seqlens.numel() - 1
    dH, dW = _grad_out(H, W, dH, dW)
    dev = H.device
    loss = torch.empty((), dtype=torch.float32, device=dev)
    nv = torch.empty((), dtype=torch.int64, device=dev)
    lp = torch.empty(T, dtype=torch.float32, device=dev) if logp else None
    st = torch.empty((), dtype=torch.int32, device=dev) if status is None else status
    _check(_lib.sbp_lmhead_grpo_ext(_p(H), _p(W), _p(labels), _p(advantages), _p(logp_old), clip_lo, clip_hi,
                                    _p(ref_logp), float(kl_coef), _p(cu_seqlens), n_seq, T, d, V, chunk,
                                    ignore_index, dt, _p(loss), _p(nv), _p(lp), _p(dH), _p(dW),
                                    int(bool(accumulate_dW)), _p(ws), ws.numel(), _p(st), _stream(stream)),
           "sbp_lmhead_grpo_ext")
    return dict(loss=loss, n_valid=nv, logp=lp, dH=dH, dW=dW, status=st)


def dpo_pass1(H, W, labels, cu_seqlens, chunk, ignore_index=IGNORE_INDEX, *, logp=True, workspace=None,
              status=None, stream=None) -> dict:
    """DPO first pass: per-sequence summed label log-probs (``sbp_lmhead_dpo_pass1``)."""
    T, d, V, dt, ws = _prep(H, W, labels, chunk, MODE_DPO1, workspace)
    _dev(cu_seqlens)
    n_seq = cu_seqlens.numel() - 1
    dev = H.device
    S = torch.empty(max(n_seq, 0), dtype=torch.float64, device=dev)
    nv = torch.empty((), dtype=torch.int64, device=dev)
    lp = torch.empty(T, dtype=torch.float32, device=dev) if logp else None
    st = torch.empty((), dtype=torch.int32, device=dev) if status is None else status
    _check(_lib.sbp_lmhead_dpo_pass1(_p(H), _p(W), _p(labels), _p(cu_seqlens), n_seq, T, d, V, chunk,
                                     ignore_index, dt, _p(S), _p(lp), _p(nv), _p(ws), ws.numel(), _p(st),
                                     _stream(stream)), "sbp_lmhead_dpo_pass1")
    return dict(seq_logp=S, logp=lp, n_valid=nv, status=st)


def dpo_pass2(H, W, labels, cu_seqlens, seq_logp, ref_seq_logp, beta, chunk, ignore_index=IGNORE_INDEX, *,
              dH=None, dW=None, accumulate_dW=False, workspace=None, status=None, stream=None) -> dict:
    """DPO second pass: loss and gradients given the sequence sums (``sbp_lmhead_dpo_pass2``)."""
    T, d, V, dt, ws = _prep(H, W, labels, chunk, MODE_DPO2, workspace)
    _dev(cu_seqlens, seq_logp, ref_seq_logp)
    n_seq = cu_seqlens.numel() - 1
    dH, dW = _grad_out(H, W, dH, dW)
    dev = H.device
    loss = torch.empty((), dtype=torch.float32, device=dev)
    margins = torch.empty(max(n_seq // 2, 1), dtype=torch.float64, device=dev)
    st = torch.empty((), dtype=torch.int32, device=dev) if status is None else status
    _check(_lib.sbp_lmhead_dpo_pass2(_p(H), _p(W), _p(labels), _p(cu_seqlens), n_seq, _p(seq_logp),
                                     _p(ref_seq_logp), float(beta), T, d, V, chunk, ignore_index, dt, _p(loss),
                                     _p(margins), _p(dH), _p(dW), int(bool(accumulate_dW)), _p(ws), ws.numel(),
                                     _p(st), _stream(stream)), "sbp_lmhead_dpo_pass2")
    return dict(loss=loss, margins=margins[: n_seq // 2], dH=dH, dW=dW, status=st)


def check_status(status: torch.Tensor, where: str = "device") -> None:
    """Raise if a call's device status word (read after synchronising) is not SBP_OK."""
    code = int(status.item())
    if code != OK:
        raise SbpError(code, where)


def mlp_workspace_bytes(T: int, d: int, f: int, chunk: int) -> int:
    return int(_lib.sbp_mlp_workspace_bytes(T, d, f, chunk))


def mlp_swiglu_backward(X, Wgu, Wd, dY, chunk, *, dX=None, dWgu=None, dWd=None, accumulate=False, workspace=None,
                        status=None, stream=None) -> dict:
    """Chunked backward of the SwiGLU MLP sublayer (``sbp_mlp_swiglu_backward``).

    X, dY [T, d] bf16; Wgu [2f, d] bf16 (gate rows then up rows); Wd [d, f] bf16."""
    _dev(X, Wgu, Wd, dY)
    T, d = X.shape
    f = Wd.shape[1]
    if Wgu.shape != (2 * f, d) or Wd.shape != (d, f) or dY.shape != (T, d):
        raise ValueError("shapes: X, dY [T, d]; Wgu [2f, d]; Wd [d, f]")
    if any(t.dtype != torch.bfloat16 for t in (X, Wgu, Wd, dY)):
        raise TypeError("the MLP sublayer takes bf16 operands")
    dev = X.device
    if workspace is None:
        n = mlp_workspace_bytes(T, d, f, chunk)
        if n == 0:
            raise SbpError(ERR_INVALID_ARG, "mlp_workspace_bytes")
        workspace = torch.empty(n, dtype=torch.uint8, device=dev)
    dX = torch.empty_like(X) if dX is None else dX
    dWgu = torch.empty((2 * f, d), dtype=torch.float32, device=dev) if dWgu is None else dWgu
    dWd = torch.empty((d, f), dtype=torch.float32, device=dev) if dWd is None else dWd
    _dev(dX, dWgu, dWd)
    st = torch.empty((), dtype=torch.int32, device=dev) if status is None else status
    _check(_lib.sbp_mlp_swiglu_backward(_p(X), _p(Wgu), _p(Wd), _p(dY), T, d, f, chunk, _p(dX), _p(dWgu), _p(dWd),
                                        int(bool(accumulate)), _p(workspace), workspace.numel(), _p(st),
                                        _stream(stream)), "sbp_mlp_swiglu_backward")
    return dict(dX=dX, dWgu=dWgu, dWd=dWd, status=st)


def attn_workspace_bytes(H: int, T: int, hd: int, chunk: int) -> int:
    return int(_lib.sbp_attn_workspace_bytes(H, T, hd, chunk))


def attn_causal_backward(Q, K, V, O, dO, lse, scale, chunk, *, dQ=None, dK=None, dV=None, accumulate=False,
                         workspace=None, status=None, stream=None) -> dict:
    """Chunked causal-attention backward (``sbp_attn_causal_backward``, or
    ``sbp_attn_causal_backward_gqa`` when K and V have fewer heads than Q).

    Q, O, dO [H, T, hd] bf16; K, V [Hkv, T, hd] bf16 (Hkv divides H; Hkv = H is plain
    multi-head attention); lse [H, T] fp32 (the forward's row log-sum-exp).  dK, dV are
    [Hkv, T, hd] fp32."""
    _dev(Q, K, V, O, dO, lse)
    H, T, hd = Q.shape
    Hkv = K.shape[0]
    for t in (O, dO):
        if t.shape != (H, T, hd) or t.dtype != torch.bfloat16:
            raise ValueError("Q, O, dO must be bf16 [H, T, hd]")
    for t in (K, V):
        if t.shape != (Hkv, T, hd) or t.dtype != torch.bfloat16:
            raise ValueError("K, V must be bf16 [Hkv, T, hd]")
    if Q.dtype != torch.bfloat16 or lse.shape != (H, T) or lse.dtype != torch.float32:
        raise ValueError("Q bf16 [H, T, hd]; lse fp32 [H, T]")
    dev = Q.device
    if workspace is None:
        n = attn_workspace_bytes(H, T, hd, chunk)
        if n == 0:
            raise SbpError(ERR_INVALID_ARG, "attn_workspace_bytes")
        workspace = torch.empty(n, dtype=torch.uint8, device=dev)
    dQ = torch.empty_like(Q) if dQ is None else dQ
    dK = torch.empty((Hkv, T, hd), dtype=torch.float32, device=dev) if dK is None else dK
    dV = torch.empty((Hkv, T, hd), dtype=torch.float32, device=dev) if dV is None else dV
    _dev(dQ, dK, dV)
    st = torch.empty((), dtype=torch.int32, device=dev) if status is None else status
    if Hkv == H:
        _check(_lib.sbp_attn_causal_backward(_p(Q), _p(K), _p(V), _p(O), _p(dO), _p(lse), H, T, hd, float(scale),
                                             chunk, _p(dQ), _p(dK), _p(dV), int(bool(accumulate)), _p(workspace),
                                             workspace.numel(), _p(st), _stream(stream)), "sbp_attn_causal_backward")
    else:
        _check(_lib.sbp_attn_causal_backward_gqa(_p(Q), _p(K), _p(V), _p(O), _p(dO), _p(lse), H, Hkv, T, hd,
                                                 float(scale), chunk, _p(dQ), _p(dK), _p(dV), int(bool(accumulate)),
                                                 _p(workspace), workspace.numel(), _p(st), _stream(stream)),
               "sbp_attn_causal_backward_gqa")
    return dict(dQ=dQ, dK=dK, dV=dV, status=st)
