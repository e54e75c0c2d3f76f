"""Pins of the causal-attention oracle (CPU only): finite differences of sum(O * dO)
through the forward, PyTorch's scaled_dot_product_attention with autograd in float64
(library routine), the forward against a plain softmax, and chunked == unchunked
(the causal chunk decomposition is exact)."""
import numpy as np
import pytest

from oracle import attention as A


def tiny(H=2, T=7, hd=4, seed=0):
    g = np.random.default_rng(seed)
    return (g.standard_normal((H, T, hd)), g.standard_normal((H, T, hd)), g.standard_normal((H, T, hd)),
            g.standard_normal((H, T, hd)))


def test_forward_matches_plain_softmax():
    sp = pytest.importorskip("scipy.special")
    Q, K, V, _ = tiny(seed=1)
    f = A.forward(Q, K, V, 0.5)
    for h in range(2):
        S = 0.5 * Q[h] @ K[h].T
        S[np.triu(np.ones((7, 7), bool), 1)] = -np.inf
        np.testing.assert_allclose(f["O"][h], sp.softmax(S, axis=1) @ V[h], rtol=1e-13, atol=1e-14)
        np.testing.assert_allclose(f["lse"][h], sp.logsumexp(S, axis=1), rtol=1e-14)


def test_fd_of_sum_O_dO():
    Q, K, V, dO = tiny(seed=2)
    s = 0.7
    f = A.forward(Q, K, V, s)
    b = A.backward(Q, K, V, f["O"], dO, f["lse"], s)

    def loss():
        return float((A.forward(Q, K, V, s)["O"] * dO).sum())

    for X, key in ((Q, "dQ"), (K, "dK"), (V, "dV")):
        G = np.zeros_like(X)
        it = np.nditer(X, flags=["multi_index"])
        for _ in it:
            i = it.multi_index
            old = X[i]
            X[i] = old + 1e-6
            lp = loss()
            X[i] = old - 1e-6
            lm = loss()
            X[i] = old
            G[i] = (lp - lm) / 2e-6
        np.testing.assert_allclose(b[key], G, rtol=1e-6, atol=1e-8)


def test_matches_torch_sdpa_autograd_fp64():
    torch = pytest.importorskip("torch")
    Q, K, V, dO = tiny(H=3, T=9, hd=5, seed=3)
    s = 0.4
    f = A.forward(Q, K, V, s)
    b = A.backward(Q, K, V, f["O"], dO, f["lse"], s)
    q, k, v = (torch.tensor(x, dtype=torch.float64, requires_grad=True) for x in (Q, K, V))
    o = torch.nn.functional.scaled_dot_product_attention(q[None], k[None], v[None], is_causal=True, scale=s)[0]
    o.backward(torch.tensor(dO))
    np.testing.assert_allclose(f["O"], o.detach().numpy(), rtol=1e-12, atol=1e-13)
    for t, key in ((q, "dQ"), (k, "dK"), (v, "dV")):
        np.testing.assert_allclose(b[key], t.grad.numpy(), rtol=1e-11, atol=1e-12)


@pytest.mark.parametrize("chunk", [1, 3, 7])
def test_chunked_equals_unchunked(chunk):
    Q, K, V, dO = tiny(H=2, T=7, hd=3, seed=4)
    f = A.forward(Q, K, V, 0.6)
    a = A.backward(Q, K, V, f["O"], dO, f["lse"], 0.6)
    b = A.backward_chunked(Q, K, V, f["O"], dO, f["lse"], 0.6, chunk)
    for k in ("dQ", "dK", "dV"):
        np.testing.assert_allclose(b[k], a[k], rtol=1e-12, atol=1e-13)


def test_planted_missing_causal_mask_is_caught(monkeypatch):
    Q, K, V, dO = tiny(seed=5)
    f = A.forward(Q, K, V, 0.5)
    real = np.triu

    def no_mask(m, k=0):                 # the backward forgets the causal mask
        return np.zeros_like(real(m, k))
    monkeypatch.setattr(np, "triu", no_mask)
    b = A.backward(Q, K, V, f["O"], dO, f["lse"], 0.5)
    monkeypatch.setattr(np, "triu", real)
    ref = A.backward(Q, K, V, f["O"], dO, f["lse"], 0.5)
    assert np.abs(b["dV"] - ref["dV"]).max() > 1e-3


def test_row_and_column_functions_match_the_full_backward():
    # the sampled-row forms the full-size GPU test uses, against the pinned full backward
    g = np.random.default_rng(11)
    H, T, hd, s = 2, 23, 6, 0.45
    Q, K, V, dO = (g.standard_normal((H, T, hd)) for _ in range(4))
    f = A.forward(Q, K, V, s)
    b = A.backward(Q, K, V, f["O"], dO, f["lse"], s)
    rows, keys = [0, 1, 11, 22], [0, 5, 21, 22]
    for h in range(H):
        np.testing.assert_allclose(A.rows_dQ(Q, K, V, f["O"], dO, f["lse"], s, h, rows), b["dQ"][h, rows],
                                   rtol=1e-12, atol=1e-13)
        dK, dV = A.keys_dKdV(Q, K, V, f["O"], dO, f["lse"], s, h, keys)
        np.testing.assert_allclose(dK, b["dK"][h, keys], rtol=1e-12, atol=1e-13)
        np.testing.assert_allclose(dV, b["dV"][h, keys], rtol=1e-12, atol=1e-13)


def test_gqa_equals_mha_with_repeated_heads():
    # grouped-query attention is multi-head attention with each key / value head repeated
    # over its group; dK, dV of a shared head are the sums over the group (chain rule)
    g = np.random.default_rng(21)
    H, Hkv, T, hd, s = 6, 2, 9, 4, 0.5
    Q, dO = g.standard_normal((H, T, hd)), g.standard_normal((H, T, hd))
    K, V = g.standard_normal((Hkv, T, hd)), g.standard_normal((Hkv, T, hd))
    Kr, Vr = np.repeat(K, H // Hkv, axis=0), np.repeat(V, H // Hkv, axis=0)
    f, fr = A.forward(Q, K, V, s), A.forward(Q, Kr, Vr, s)
    np.testing.assert_allclose(f["O"], fr["O"], rtol=1e-13, atol=1e-14)
    b = A.backward(Q, K, V, f["O"], dO, f["lse"], s)
    br = A.backward(Q, Kr, Vr, fr["O"], dO, fr["lse"], s)
    np.testing.assert_allclose(b["dQ"], br["dQ"], rtol=1e-12, atol=1e-13)
    for key in ("dK", "dV"):
        summed = br[key].reshape(Hkv, H // Hkv, T, hd).sum(axis=1)
        np.testing.assert_allclose(b[key], summed, rtol=1e-12, atol=1e-13)
    c = A.backward_chunked(Q, K, V, f["O"], dO, f["lse"], s, 4)
    for key in ("dQ", "dK", "dV"):
        np.testing.assert_allclose(c[key], b[key], rtol=1e-12, atol=1e-13)
    dK, dV = A.keys_dKdV(Q, K, V, f["O"], dO, f["lse"], s, 1, [0, 4, 8])
    np.testing.assert_allclose(dK, b["dK"][1, [0, 4, 8]], rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(dV, b["dV"][1, [0, 4, 8]], rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(A.rows_dQ(Q, K, V, f["O"], dO, f["lse"], s, 5, [0, 8]), b["dQ"][5, [0, 8]],
                               rtol=1e-12, atol=1e-13)


def test_gqa_matches_torch_sdpa_autograd_fp64():
    torch = pytest.importorskip("torch")
    g = np.random.default_rng(22)
    H, Hkv, T, hd, s = 4, 1, 8, 5, 0.4
    Q, dO = g.standard_normal((H, T, hd)), g.standard_normal((H, T, hd))
    K, V = g.standard_normal((Hkv, T, hd)), g.standard_normal((Hkv, T, hd))
    f = A.forward(Q, K, V, s)
    b = A.backward(Q, K, V, f["O"], dO, f["lse"], s)
    q, k, v = (torch.tensor(x, dtype=torch.float64, requires_grad=True) for x in (Q, K, V))
    try:
        o = torch.nn.functional.scaled_dot_product_attention(q[None], k[None], v[None], is_causal=True, scale=s,
                                                             enable_gqa=True)[0]
    except TypeError:
        pytest.skip("this torch has no grouped-query scaled_dot_product_attention")
    o.backward(torch.tensor(dO))
    np.testing.assert_allclose(f["O"], o.detach().numpy(), rtol=1e-12, atol=1e-13)
    for t, key in ((q, "dQ"), (k, "dK"), (v, "dV")):
        np.testing.assert_allclose(b[key], t.grad.numpy(), rtol=1e-11, atol=1e-12)


def test_gqa_finite_differences():
    g = np.random.default_rng(23)
    H, Hkv, T, hd, s = 4, 2, 5, 3, 0.7
    Q, dO = g.standard_normal((H, T, hd)), g.standard_normal((H, T, hd))
    K, V = g.standard_normal((Hkv, T, hd)), g.standard_normal((Hkv, T, hd))
    f = A.forward(Q, K, V, s)
    b = A.backward(Q, K, V, f["O"], dO, f["lse"], s)

    def loss():
        return float((A.forward(Q, K, V, s)["O"] * dO).sum())

    for X, key in ((K, "dK"), (V, "dV")):
        G = np.zeros_like(X)
        it = np.nditer(X, flags=["multi_index"])
        for _ in it:
            i = it.multi_index
            old = X[i]
            X[i] = old + 1e-6
            lp = loss()
            X[i] = old - 1e-6
            lm = loss()
            X[i] = old
            G[i] = (lp - lm) / 2e-6
        np.testing.assert_allclose(b[key], G, rtol=1e-6, atol=1e-8)


# randomised shapes: query / key-value head counts (grouped-query included), lengths,
# widths, scales and chunks, each against PyTorch's SDPA autograd in float64 and against
# the chunked decomposition
@pytest.mark.parametrize("seed", range(16))
def test_random_shapes_against_sdpa_and_chunking(seed):
    torch = pytest.importorskip("torch")
    g = np.random.default_rng(1000 + seed)
    Hkv = int(g.integers(1, 4))
    H = Hkv * int(g.integers(1, 4))
    T = int(g.integers(1, 12))
    hd = int(g.integers(1, 7))
    s = float(g.uniform(0.2, 1.0))
    chunk = int(g.integers(1, T + 2))
    Q, dO = g.standard_normal((H, T, hd)), g.standard_normal((H, T, hd))
    K, V = g.standard_normal((Hkv, T, hd)), g.standard_normal((Hkv, T, hd))
    f = A.forward(Q, K, V, s)
    b = A.backward(Q, K, V, f["O"], dO, f["lse"], s)
    q, k, v = (torch.tensor(x, dtype=torch.float64, requires_grad=True) for x in (Q, K, V))
    o = torch.nn.functional.scaled_dot_product_attention(q[None], k[None], v[None], is_causal=True, scale=s,
                                                         enable_gqa=True)[0]
    o.backward(torch.tensor(dO))
    np.testing.assert_allclose(f["O"], o.detach().numpy(), rtol=1e-11, atol=1e-12)
    for t, key in ((q, "dQ"), (k, "dK"), (v, "dV")):
        np.testing.assert_allclose(b[key], t.grad.numpy(), rtol=1e-10, atol=1e-11)
    c = A.backward_chunked(Q, K, V, f["O"], dO, f["lse"], s, chunk)
    for key in ("dQ", "dK", "dV"):
        np.testing.assert_allclose(c[key], b[key], rtol=1e-12, atol=1e-12)
