"""GPU parity of the chunked SwiGLU-MLP backward against the float64 oracle.

Shapes span several 256-row pairs, several chunks with a ragged last chunk, and more
than one tile along d and f; bf16 operands, fp32 accumulation (dX / dW relative
Frobenius error <= 2e-2, the bf16 tolerance of the LM-head tests).
"""
import numpy as np
import pytest

from oracle import mlp as M
from memory_efficient_exact_gb300 import inputs as I
from parity_util import TOL, rel_fro

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def sbp():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    from memory_efficient_exact_gb300 import _build
    _build.build_library()
    from memory_efficient_exact_gb300 import sbp as mod
    return mod


def make(T, d, f, seed):
    g = np.random.default_rng(seed)
    X = I.round_bf16(g.standard_normal((T, d), dtype=np.float32))
    Wgu = I.round_bf16((g.standard_normal((2 * f, d), dtype=np.float32) / np.sqrt(d)).astype(np.float32))
    Wd = I.round_bf16((g.standard_normal((d, f), dtype=np.float32) / np.sqrt(f)).astype(np.float32))
    dY = I.round_bf16(g.standard_normal((T, d), dtype=np.float32))
    return X, Wgu, Wd, dY


def dev(x):
    return torch.from_numpy(x).cuda().to(torch.bfloat16).contiguous()


@pytest.mark.parametrize("T,d,f,chunk", [(300, 256, 512, 128), (513, 128, 768, 200), (1000, 512, 1024, 384),
                                         (256, 64, 256, 256)])
def test_mlp_backward_parity(sbp, T, d, f, chunk):
    X, Wgu, Wd, dY = make(T, d, f, seed=T + d)
    out = sbp.mlp_swiglu_backward(dev(X), dev(Wgu), dev(Wd), dev(dY), chunk)
    torch.cuda.synchronize()
    sbp.check_status(out["status"])
    ref = M.backward(X, Wgu[:f], Wgu[f:], Wd, dY)
    tol = TOL["bf16"]["grad"]
    e = {"dX": rel_fro(out["dX"].float().cpu().numpy(), ref["dx"]),
         "dWg": rel_fro(out["dWgu"][:f].cpu().numpy(), ref["dWg"]),
         "dWu": rel_fro(out["dWgu"][f:].cpu().numpy(), ref["dWu"]),
         "dWd": rel_fro(out["dWd"].cpu().numpy(), ref["dWd"])}
    assert max(e.values()) <= tol, e


def test_mlp_accumulate_and_determinism(sbp):
    T, d, f, chunk = 300, 128, 512, 128
    X, Wgu, Wd, dY = (dev(a) for a in make(T, d, f, seed=5))
    a = sbp.mlp_swiglu_backward(X, Wgu, Wd, dY, chunk)
    b = sbp.mlp_swiglu_backward(X, Wgu, Wd, dY, chunk)
    torch.cuda.synchronize()
    assert torch.equal(a["dX"], b["dX"]) and torch.equal(a["dWgu"], b["dWgu"]) and torch.equal(a["dWd"], b["dWd"])
    acc_gu, acc_d = a["dWgu"].clone(), a["dWd"].clone()
    sbp.mlp_swiglu_backward(X, Wgu, Wd, dY, chunk, dWgu=acc_gu, dWd=acc_d, accumulate=True)
    torch.cuda.synchronize()
    # the accumulated sum is ((a + c1) + c2) + c3 against 2 (c1 + c2 + c3): equal up to fp32
    # rounding of the chunk terms, which cancel in part
    for acc, ref in ((acc_gu, a["dWgu"]), (acc_d, a["dWd"])):
        assert torch.allclose(acc, 2 * ref, rtol=1e-5, atol=1e-6 * ref.abs().max().item())


def test_mlp_under_graph_capture(sbp):
    """The dWd GEMMs run on the library's side stream, forked from and joined back into
    the caller's stream: a call captured into a CUDA graph and replayed gives the same
    bits as a plain call."""
    T, d, f, chunk = 300, 128, 512, 128
    X, Wgu, Wd, dY = (dev(a) for a in make(T, d, f, seed=9))
    ref = sbp.mlp_swiglu_backward(X, Wgu, Wd, dY, chunk)
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    ws = torch.empty(sbp.mlp_workspace_bytes(T, d, f, chunk), dtype=torch.uint8, device="cuda")
    dX, dWgu, dWd = torch.empty_like(ref["dX"]), torch.empty_like(ref["dWgu"]), torch.empty_like(ref["dWd"])
    st = torch.zeros((), dtype=torch.int32, device="cuda")
    kw = dict(dX=dX, dWgu=dWgu, dWd=dWd, workspace=ws, status=st, stream=s)
    with torch.cuda.stream(s):
        sbp.mlp_swiglu_backward(X, Wgu, Wd, dY, chunk, **kw)
    s.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        sbp.mlp_swiglu_backward(X, Wgu, Wd, dY, chunk, **kw)
    for x in (dX, dWgu, dWd):
        x.zero_()
    g.replay()
    torch.cuda.synchronize()
    sbp.check_status(st)
    assert torch.equal(dX, ref["dX"]) and torch.equal(dWgu, ref["dWgu"]) and torch.equal(dWd, ref["dWd"])
