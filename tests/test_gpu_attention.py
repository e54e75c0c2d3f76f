"""GPU parity of the chunked causal-attention backward against the float64 oracle.

Inputs: Q, K, V, dO ~ N(0, 1) rounded to bf16; O and lse from the oracle's forward on the
same values (O rounded to bf16, lse kept in fp32, as a forward saves them); the expected
gradients are the oracle's unchunked backward on exactly the values the GPU sees.
Shapes span several heads, several chunks with a ragged last one, row pairs and 256-key
tiles; dQ / dK / dV relative Frobenius error <= 2e-2 (the bf16 tolerance of the other
tests).
"""
import numpy as np
import pytest

from oracle import attention as A
from memory_efficient_exact_gb300 import inputs as I
from parity_util import rel_fro

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


def make(H, T, hd, seed):
    g = np.random.default_rng(seed)
    Q, K, V, dO = (I.round_bf16(g.standard_normal((H, T, hd), dtype=np.float32)) for _ in range(4))
    scale = 1.0 / np.sqrt(hd)
    f = A.forward(Q, K, V, scale)
    O = I.round_bf16(f["O"].astype(np.float32))
    lse = f["lse"].astype(np.float32)
    return Q, K, V, O, dO, lse, scale


def dev(x, dt=torch.bfloat16):
    return torch.from_numpy(np.ascontiguousarray(x)).cuda().to(dt).contiguous()


@pytest.mark.parametrize("H,T,hd,chunk", [(2, 300, 64, 128), (4, 640, 128, 256), (3, 513, 128, 200),
                                          (1, 1024, 64, 1024), (2, 96, 128, 40)])
def test_attention_backward_parity(sbp, H, T, hd, chunk):
    Q, K, V, O, dO, lse, scale = make(H, T, hd, seed=H * 1000 + T)
    out = sbp.attn_causal_backward(dev(Q), dev(K), dev(V), dev(O), dev(dO), dev(lse, torch.float32), scale, chunk)
    torch.cuda.synchronize()
    sbp.check_status(out["status"])
    ref = A.backward(Q, K, V, O, dO, lse, scale)
    e = {"dQ": rel_fro(out["dQ"].float().cpu().numpy(), ref["dQ"]),
         "dK": rel_fro(out["dK"].cpu().numpy(), ref["dK"]),
         "dV": rel_fro(out["dV"].cpu().numpy(), ref["dV"])}
    assert max(e.values()) <= 2e-2, e


def test_attention_accumulate_and_determinism(sbp):
    H, T, hd, chunk = 2, 300, 64, 128
    Q, K, V, O, dO, lse, scale = make(H, T, hd, seed=7)
    args = [dev(Q), dev(K), dev(V), dev(O), dev(dO), dev(lse, torch.float32), scale, chunk]
    a = sbp.attn_causal_backward(*args)
    b = sbp.attn_causal_backward(*args)
    torch.cuda.synchronize()
    assert torch.equal(a["dQ"], b["dQ"]) and torch.equal(a["dK"], b["dK"]) and torch.equal(a["dV"], b["dV"])
    dK, dV = a["dK"].clone(), a["dV"].clone()
    sbp.attn_causal_backward(*args, dK=dK, dV=dV, accumulate=True)
    torch.cuda.synchronize()
    for acc, ref in ((dK, a["dK"]), (dV, a["dV"])):
        assert torch.allclose(acc, 2 * ref, rtol=1e-5, atol=1e-6 * ref.abs().max().item())
