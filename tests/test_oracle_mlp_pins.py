"""Pins of the MLP-sublayer oracle (CPU only): finite differences of a scalar loss
through the sublayer, PyTorch autograd in float64 (library routine), the closed-form
derivative of silu, and chunked == unchunked (the exactness of the row decomposition).
"""
import numpy as np
import pytest

from oracle import mlp as M


def tiny(T=5, d=4, f=6, seed=0):
    g = np.random.default_rng(seed)
    return (g.standard_normal((T, d)), 0.5 * g.standard_normal((f, d)), 0.5 * g.standard_normal((f, d)),
            0.5 * g.standard_normal((d, f)), g.standard_normal((T, d)))


def test_dsilu_matches_finite_difference():
    t = np.linspace(-8, 8, 33)
    h = 1e-6
    np.testing.assert_allclose(M.dsilu(t), (M.silu(t + h) - M.silu(t - h)) / (2 * h), rtol=1e-8, atol=1e-10)


def test_fd_of_the_loss_sum_y_times_dY():
    x, Wg, Wu, Wd, dY = tiny()
    b = M.backward(x, Wg, Wu, Wd, dY)

    def loss():
        return float((M.forward(x, Wg, Wu, Wd)["y"] * dY).sum())

    for X, key in ((x, "dx"), (Wg, "dWg"), (Wu, "dWu"), (Wd, "dWd")):
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


def test_matches_torch_autograd_fp64():
    torch = pytest.importorskip("torch")
    x, Wg, Wu, Wd, dY = tiny(T=7, d=5, f=9, seed=1)
    b = M.backward(x, Wg, Wu, Wd, dY)
    t = [torch.tensor(v, dtype=torch.float64, requires_grad=True) for v in (x, Wg, Wu, Wd)]
    y = (torch.nn.functional.silu(t[0] @ t[1].T) * (t[0] @ t[2].T)) @ t[3].T
    y.backward(torch.tensor(dY))
    for tt, key in zip(t, ("dx", "dWg", "dWu", "dWd")):
        np.testing.assert_allclose(b[key], tt.grad.numpy(), rtol=1e-12, atol=1e-14)


@pytest.mark.parametrize("chunk", [1, 3, 7])
def test_chunked_equals_unchunked(chunk):
    x, Wg, Wu, Wd, dY = tiny(T=7, d=5, f=9, seed=2)
    a = M.backward(x, Wg, Wu, Wd, dY)
    b = M.backward_chunked(x, Wg, Wu, Wd, dY, chunk)
    for k in ("dx", "dWg", "dWu", "dWd"):
        np.testing.assert_allclose(b[k], a[k], rtol=1e-13, atol=1e-15)


def test_planted_missing_gate_derivative_is_caught(monkeypatch):
    monkeypatch.setattr(M, "dsilu", M.sigmoid)          # a plausible slip: sigmoid for silu'
    x, Wg, Wu, Wd, dY = tiny(seed=3)
    with pytest.raises(AssertionError):
        _fd_dx(x, Wg, Wu, Wd, dY)


def _fd_dx(x, Wg, Wu, Wd, dY):
    b = M.backward(x, Wg, Wu, Wd, dY)
    G = np.zeros_like(x)
    for i in range(x.shape[0]):
        for j in range(x.shape[1]):
            old = x[i, j]
            x[i, j] = old + 1e-6
            lp = float((M.forward(x, Wg, Wu, Wd)["y"] * dY).sum())
            x[i, j] = old - 1e-6
            lm = float((M.forward(x, Wg, Wu, Wd)["y"] * dY).sum())
            x[i, j] = old
            G[i, j] = (lp - lm) / 2e-6
    np.testing.assert_allclose(b["dx"], G, rtol=1e-6, atol=1e-8)


# randomised shapes and weight scales against PyTorch autograd in float64, and the row
# decomposition at a random chunk
@pytest.mark.parametrize("seed", range(16))
def test_random_shapes_against_autograd_and_chunking(seed):
    torch = pytest.importorskip("torch")
    g = np.random.default_rng(2000 + seed)
    T, d, f = int(g.integers(1, 10)), int(g.integers(1, 7)), int(g.integers(1, 9))
    sc = float(g.uniform(0.2, 1.5))
    x, dY = g.standard_normal((T, d)), g.standard_normal((T, d))
    Wg, Wu, Wd = sc * g.standard_normal((f, d)), sc * g.standard_normal((f, d)), sc * g.standard_normal((d, f))
    b = M.backward(x, Wg, Wu, Wd, dY)
    xt, gt, ut, dt = (torch.tensor(a, dtype=torch.float64, requires_grad=True) for a in (x, Wg, Wu, Wd))
    y = (torch.nn.functional.silu(xt @ gt.T) * (xt @ ut.T)) @ dt.T
    y.backward(torch.tensor(dY))
    np.testing.assert_allclose(b["y"], y.detach().numpy(), rtol=1e-12, atol=1e-12)
    for t, key in ((xt, "dx"), (gt, "dWg"), (ut, "dWu"), (dt, "dWd")):
        np.testing.assert_allclose(b[key], t.grad.numpy(), rtol=1e-11, atol=1e-11)
    c = M.backward_chunked(x, Wg, Wu, Wd, dY, int(g.integers(1, T + 2)))
    for key in ("dx", "dWg", "dWu", "dWd"):
        np.testing.assert_allclose(c[key], b[key], rtol=1e-12, atol=1e-12)
