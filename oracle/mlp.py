"""CPU oracle for the chunked backward of a position-wise SwiGLU MLP sublayer (float64).

TEST INFRASTRUCTURE ONLY (see ``oracle/lmhead.py``): only the tests, the smoke check
and the benchmark's CPU leg use it.

StreamBP applies the same linear decomposition of the chain rule along the sequence
to the transformer layers, layer by layer (chatpaper.ai / fugumt.com abstract;
atlas.scime.ai summary, "Approach").  The MLP sublayer is position-wise, so its
backward splits over row chunks exactly as the LM head does: each chunk recomputes its
activations from its inputs and adds its share of the weight gradients.

Reading (the pages give no layer formula): the Qwen3-style gated MLP on its already
normalised input x,
    g = x Wg^T,  u = x Wu^T,  a = silu(g) * u,  y = a Wd^T,
Wg, Wu [f, d], Wd [d, f], silu(t) = t sigmoid(t).  Given dY = dL/dy:
    da = dY Wd,  dg = da * u * silu'(g),  du = da * silu(g),
    dx = dg Wg + du Wu,  dWd = dY^T a,  dWg = dg^T x,  dWu = du^T x,
silu'(t) = sigmoid(t) (1 + t (1 - sigmoid(t))).
"""
from __future__ import annotations

import numpy as np


def _f64(x):
    return np.asarray(x, dtype=np.float64)


def sigmoid(t):
    t = _f64(t)
    return np.exp(-np.logaddexp(0.0, -t))


def silu(t):
    return _f64(t) * sigmoid(t)


def dsilu(t):
    s = sigmoid(t)
    return s * (1.0 + _f64(t) * (1.0 - s))


def forward(x, Wg, Wu, Wd) -> dict:
    x, Wg, Wu, Wd = _f64(x), _f64(Wg), _f64(Wu), _f64(Wd)
    g = x @ Wg.T
    u = x @ Wu.T
    a = silu(g) * u
    return dict(g=g, u=u, a=a, y=a @ Wd.T)


def backward(x, Wg, Wu, Wd, dY) -> dict:
    """Unchunked backward of the sublayer (all T rows at once)."""
    x, Wg, Wu, Wd, dY = _f64(x), _f64(Wg), _f64(Wu), _f64(Wd), _f64(dY)
    f = forward(x, Wg, Wu, Wd)
    da = dY @ Wd
    dg = da * f["u"] * dsilu(f["g"])
    du = da * silu(f["g"])
    return dict(dx=dg @ Wg + du @ Wu, dWg=dg.T @ x, dWu=du.T @ x, dWd=dY.T @ f["a"], y=f["y"])


def backward_chunked(x, Wg, Wu, Wd, dY, chunk: int) -> dict:
    """The same backward one row chunk at a time (recomputing the chunk's activations)."""
    x, dY = _f64(x), _f64(dY)
    T, d = x.shape
    fdim = Wg.shape[0]
    out = dict(dx=np.zeros((T, d)), dWg=np.zeros((fdim, d)), dWu=np.zeros((fdim, d)), dWd=np.zeros((d, fdim)))
    for r0 in range(0, T, chunk):
        b = backward(x[r0:r0 + chunk], Wg, Wu, Wd, dY[r0:r0 + chunk])
        out["dx"][r0:r0 + chunk] = b["dx"]
        for k in ("dWg", "dWu", "dWd"):
            out[k] += b[k]
    return out
