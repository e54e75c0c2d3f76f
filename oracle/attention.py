"""CPU oracle for the chunked backward of causal multi-head self-attention (float64).

TEST INFRASTRUCTURE ONLY (see ``oracle/lmhead.py``): only the tests, the smoke check
and the benchmark's CPU leg use it.

StreamBP decomposes the chain rule along the sequence layer by layer and uses the causal
structure: a chunk of queries only needs the keys and values up to its own position
(chatpaper.ai / fugumt.com abstract; atlas.scime.ai summary, "Approach").  So the
attention backward can run one query chunk at a time: chunk c (rows [c0, c1)) touches
keys [0, c1) only, writes its dQ rows, and adds its share to dK and dV of those keys.

Reading (the pages give no layer formula): per head, with scale s,
    S = s Q K^T (causal: S_ij = -inf for j > i),  P = softmax_rows(S) = exp(S - lse),
    O = P V;   given dO:  D_i = sum_k dO_ik O_ik,  dP = dO V^T,  dS = P * (dP - D),
    dQ = s dS K,  dK = s dS^T Q,  dV = P^T dO.
The forward's per-row log-sum-exp (lse) and output O are inputs, as a
FlashAttention-style forward saves them.  Tensors are [H, T, hd].

Grouped-query attention (the Qwen3 models of the pages' experiments share each key /
value head among H / Hkv query heads): K and V are [Hkv, T, hd]; query head h reads
key / value head h // (H / Hkv), and dK, dV of a key / value head sum over its group.
Hkv = H is plain multi-head attention.
"""
from __future__ import annotations

import numpy as np


def _f64(x):
    return np.asarray(x, dtype=np.float64)


def _group(Q, K) -> int:
    H, Hkv = Q.shape[0], K.shape[0]
    if Hkv < 1 or H % Hkv:
        raise ValueError("the query heads must be a multiple of the key / value heads")
    return H // Hkv


def forward(Q, K, V, scale: float) -> dict:
    """O and lse per query head, causal, unchunked."""
    Q, K, V = _f64(Q), _f64(K), _f64(V)
    H, T, _ = Q.shape
    grp = _group(Q, K)
    mask = np.triu(np.ones((T, T), dtype=bool), k=1)
    O = np.empty_like(Q)
    lse = np.empty((H, T))
    for h in range(H):
        hk = h // grp
        S = scale * (Q[h] @ K[hk].T)
        S[mask] = -np.inf
        m = S.max(axis=1)
        lse[h] = m + np.log(np.exp(S - m[:, None]).sum(axis=1))
        O[h] = np.exp(S - lse[h][:, None]) @ V[hk]
    return dict(O=O, lse=lse)


def backward(Q, K, V, O, dO, lse, scale: float) -> dict:
    """dQ, dK, dV, unchunked (all queries at once)."""
    Q, K, V, O, dO, lse = (_f64(a) for a in (Q, K, V, O, dO, lse))
    H, T, _ = Q.shape
    grp = _group(Q, K)
    mask = np.triu(np.ones((T, T), dtype=bool), k=1)
    dQ, dK, dV = np.zeros_like(Q), np.zeros_like(K), np.zeros_like(V)
    for h in range(H):
        hk = h // grp
        S = scale * (Q[h] @ K[hk].T)
        P = np.exp(S - lse[h][:, None])
        P[mask] = 0.0
        D = (dO[h] * O[h]).sum(axis=1)
        dP = dO[h] @ V[hk].T
        dS = P * (dP - D[:, None])
        dQ[h] = scale * (dS @ K[hk])
        dK[hk] += scale * (dS.T @ Q[h])
        dV[hk] += P.T @ dO[h]
    return dict(dQ=dQ, dK=dK, dV=dV)


def backward_chunked(Q, K, V, O, dO, lse, scale: float, chunk: int) -> dict:
    """The same backward one query chunk at a time: chunk [c0, c1) uses keys [0, c1)."""
    Q, K, V, O, dO, lse = (_f64(a) for a in (Q, K, V, O, dO, lse))
    H, T, _ = Q.shape
    grp = _group(Q, K)
    dQ, dK, dV = np.zeros_like(Q), np.zeros_like(K), np.zeros_like(V)
    for h in range(H):
        hk = h // grp
        for c0 in range(0, T, chunk):
            c1 = min(T, c0 + chunk)
            S = scale * (Q[h, c0:c1] @ K[hk, :c1].T)
            P = np.exp(S - lse[h, c0:c1][:, None])
            P[np.arange(c0, c1)[:, None] < np.arange(c1)[None, :]] = 0.0
            D = (dO[h, c0:c1] * O[h, c0:c1]).sum(axis=1)
            dS = P * (dO[h, c0:c1] @ V[hk, :c1].T - D[:, None])
            dQ[h, c0:c1] = scale * (dS @ K[hk, :c1])
            dK[hk, :c1] += scale * (dS.T @ Q[h, c0:c1])
            dV[hk, :c1] += P.T @ dO[h, c0:c1]
    return dict(dQ=dQ, dK=dK, dV=dV)


def rows_dQ(Q, K, V, O, dO, lse, scale: float, h: int, rows) -> np.ndarray:
    """dQ[h, t] for the listed query rows t, each from its own score row over keys
    0..t (the causal row of the backward above; cost O(T hd) per row)."""
    Q, K, V, O, dO, lse = (_f64(a) for a in (Q, K, V, O, dO, lse))
    hk = h // _group(Q, K)
    out = np.empty((len(rows), Q.shape[2]))
    for i, t in enumerate(rows):
        p = np.exp(scale * (K[hk, :t + 1] @ Q[h, t]) - lse[h, t])
        ds = p * (V[hk, :t + 1] @ dO[h, t] - dO[h, t] @ O[h, t])
        out[i] = scale * (ds @ K[hk, :t + 1])
    return out


def keys_dKdV(Q, K, V, O, dO, lse, scale: float, hk: int, keys):
    """dK[hk, k] and dV[hk, k] of key / value head hk for the listed keys k, each from its
    own score columns over queries k..T-1 of the query heads of its group (the causal
    column of the backward above; cost O(group T hd) per key)."""
    Q, K, V, O, dO, lse = (_f64(a) for a in (Q, K, V, O, dO, lse))
    grp = _group(Q, K)
    hd = Q.shape[2]
    dK, dV = np.zeros((len(keys), hd)), np.zeros((len(keys), hd))
    for h in range(hk * grp, (hk + 1) * grp):
        for i, k in enumerate(keys):
            p = np.exp(scale * (Q[h, k:] @ K[hk, k]) - lse[h, k:])
            D = (dO[h, k:] * O[h, k:]).sum(axis=1)
            ds = p * (dO[h, k:] @ V[hk, k] - D)
            dK[i] += scale * (ds @ Q[h, k:])
            dV[i] += p @ dO[h, k:]
    return dK, dV
