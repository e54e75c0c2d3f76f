"""Shared helpers of the GPU parity tests: tolerances, transfers, comparisons."""
import numpy as np

# Tolerances of the CUDA path against the float64 oracle, on the same inputs.
#   fp32 operands: loss relative error <= 1e-5, dH / dW relative Frobenius error <= 1e-4;
#   bf16 operands with fp32 accumulation: loss <= 1e-3, dH / dW <= 2e-2;
#   the ignore mask and the token count: exact.
TOL = {"fp32": dict(loss=1e-5, grad=1e-4, logp=1e-5, seq=1e-6),
       "bf16": dict(loss=1e-3, grad=2e-2, logp=2e-3, seq=1e-4)}


def rel_fro(a, b) -> float:
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    n = np.linalg.norm(b)
    return float(np.linalg.norm(a - b) / (n if n > 0 else 1.0))


def rel(a: float, b: float) -> float:
    return abs(float(a) - float(b)) / max(abs(float(b)), 1e-30)


def to_dev(torch, H, W, y, dtype):
    td = torch.bfloat16 if dtype == "bf16" else torch.float32
    Ht = torch.from_numpy(np.ascontiguousarray(H)).to("cuda").to(td).contiguous()
    Wt = torch.from_numpy(np.ascontiguousarray(W)).to("cuda").to(td).contiguous()
    yt = torch.from_numpy(np.ascontiguousarray(y, dtype=np.int32)).to("cuda")
    return Ht, Wt, yt


def host(t):
    return t.detach().float().cpu().numpy().astype(np.float64) if t.dtype != np.float64 else t
