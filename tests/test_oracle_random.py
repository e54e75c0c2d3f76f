"""Randomised pins of the CPU oracle (CPU only): many small seeded shapes instead of a few
fixed ones.

For every drawn case (T, d, V, chunk, ignored positions, objective) the oracle must meet
what the mathematics fixes, checked against something other than itself:
  - the method's exactness claim: the chunked computation equals the unchunked one
    (ziziman.com article, LM-head paragraphs; atlas.scime.ai summary, "Approach");
  - central finite differences of the loss for every entry of dH and dW (tiny cases);
  - PyTorch's float64 cross-entropy and its autograd for SFT (a library routine);
  - the closed form of the CE logit gradient: rows sum to zero, ignored rows are zero;
  - GRPO with every ratio equal to one and A = 1 has SFT's gradient and loss -1; DPO
    at zero margins has loss log 2.
"""
import math

import numpy as np
import pytest

from oracle import lmhead as L

IGN = -100
CASES = 24


def draw(seed):
    g = np.random.default_rng(seed)
    T = int(g.integers(1, 13))
    d = int(g.integers(1, 7))
    V = int(g.integers(1, 10))
    chunk = int(g.integers(1, T + 2))
    H = g.standard_normal((T, d))
    W = float(g.uniform(0.2, 1.2)) * g.standard_normal((V, d))
    y = g.integers(0, V, T)
    y[g.random(T) < 0.25] = IGN
    return g, H, W, y, chunk


def central_fd(fun, X, h=1e-6):
    G = np.zeros_like(X)
    for i in np.ndindex(X.shape):
        old = X[i]
        X[i] = old + h
        fp = fun()
        X[i] = old - h
        fm = fun()
        X[i] = old
        G[i] = (fp - fm) / (2 * h)
    return G


def rel(a, b):
    a, b = np.asarray(a, np.float64), np.asarray(b, np.float64)
    n = np.linalg.norm(b)
    return float(np.linalg.norm(a - b) / (n if n > 0 else 1.0))


def grpo_inputs(g, H, W, y):
    T = H.shape[0]
    A = g.standard_normal(T)
    # ratios drawn away from the clip edges (0.8, 1.2) by at least 0.1, so that the
    # finite differences never straddle a kink
    r = g.choice([0.5, 0.7, 0.9, 1.0, 1.1, 1.3, 1.6], size=T)
    lpo = L.forward(H, W, y, IGN)["logp"] - np.log(r)
    return A, lpo


def dpo_inputs(g, T):
    # an even number of sequences covering [0, T)
    n = 2 * int(g.integers(1, max(2, T // 2) + 1)) if T >= 2 else 0
    if n == 0:
        return np.array([0, T], dtype=np.int64)[:1], np.zeros(0)
    cuts = np.sort(g.choice(np.arange(1, T), size=min(n - 1, T - 1), replace=False)) if T > 1 else np.array([])
    cu = np.concatenate([[0], cuts, [T]]).astype(np.int64)
    if (len(cu) - 1) % 2:
        cu = np.concatenate([cu[:-2], [T]])
    ref = -3.0 + g.standard_normal(len(cu) - 1)
    return cu, ref


@pytest.mark.parametrize("seed", range(CASES))
def test_chunked_equals_unchunked(seed):
    g, H, W, y, chunk = draw(seed)
    ref = L.sft(H, W, y, IGN)
    ch = L.chunked("sft", H, W, y, chunk, IGN)
    assert abs(ch["loss"] - ref["loss"]) <= 1e-12 * max(1.0, abs(ref["loss"]))
    assert rel(ch["dH"], ref["dH"]) <= 1e-12 and rel(ch["dW"], ref["dW"]) <= 1e-12
    A, lpo = grpo_inputs(g, H, W, y)
    ref = L.grpo(H, W, y, A, lpo, IGN)
    ch = L.chunked("grpo", H, W, y, chunk, IGN, advantages=A, logp_old=lpo)
    assert abs(ch["loss"] - ref["loss"]) <= 1e-12 * max(1.0, abs(ref["loss"]))
    assert rel(ch["dH"], ref["dH"]) <= 1e-12 and rel(ch["dW"], ref["dW"]) <= 1e-12
    cu, rf = dpo_inputs(g, H.shape[0])
    if len(cu) >= 3:
        ref = L.dpo(H, W, y, cu, rf, 0.4, IGN)
        ch = L.chunked("dpo", H, W, y, chunk, IGN, cu_seqlens=cu, ref_seq_logp=rf, beta=0.4)
        assert abs(ch["loss"] - ref["loss"]) <= 1e-12 * max(1.0, abs(ref["loss"]))
        assert rel(ch["dH"], ref["dH"]) <= 1e-12 and rel(ch["dW"], ref["dW"]) <= 1e-12


@pytest.mark.parametrize("seed", range(CASES))
def test_finite_differences(seed):
    g, H, W, y, _ = draw(100 + seed)
    for fn in (lambda: L.sft(H, W, y, IGN),):
        out = fn()
        assert rel(out["dH"], central_fd(lambda: fn()["loss"], H)) <= 1e-6
        assert rel(out["dW"], central_fd(lambda: fn()["loss"], W)) <= 1e-6
    A, lpo = grpo_inputs(g, H, W, y)
    fn = lambda: L.grpo(H, W, y, A, lpo, IGN)  # noqa: E731
    out = fn()
    assert rel(out["dH"], central_fd(lambda: fn()["loss"], H)) <= 1e-6
    assert rel(out["dW"], central_fd(lambda: fn()["loss"], W)) <= 1e-6
    cu, rf = dpo_inputs(g, H.shape[0])
    if len(cu) >= 3:
        fn = lambda: L.dpo(H, W, y, cu, rf, 0.4, IGN)  # noqa: E731
        out = fn()
        assert rel(out["dH"], central_fd(lambda: fn()["loss"], H)) <= 1e-6
        assert rel(out["dW"], central_fd(lambda: fn()["loss"], W)) <= 1e-6


@pytest.mark.parametrize("seed", range(CASES))
def test_sft_against_torch_and_closed_form(seed):
    torch = pytest.importorskip("torch")
    g, H, W, y, _ = draw(200 + seed)
    out = L.sft(H, W, y, IGN)
    valid = y != IGN
    assert out["n_valid"] == int(valid.sum())
    Ht = torch.tensor(H, dtype=torch.float64, requires_grad=True)
    Wt = torch.tensor(W, dtype=torch.float64, requires_grad=True)
    if valid.any():
        loss = torch.nn.functional.cross_entropy(Ht @ Wt.T, torch.tensor(y), ignore_index=IGN)
        loss.backward()
        assert abs(out["loss"] - loss.item()) <= 1e-12 * max(1.0, abs(loss.item()))
        assert rel(out["dH"], Ht.grad.numpy()) <= 1e-12 and rel(out["dW"], Wt.grad.numpy()) <= 1e-12
    else:
        assert out["loss"] == 0.0 and not out["dH"].any() and not out["dW"].any()
    # logit gradient: rows sum to zero, ignored rows are zero
    assert np.all(np.abs(out["G"].sum(axis=1)) <= 1e-14)
    assert not out["G"][~valid].any()


@pytest.mark.parametrize("seed", range(8))
def test_special_cases(seed):
    g, H, W, y, _ = draw(300 + seed)
    f = L.forward(H, W, y, IGN)
    # ratios of one and A = 1: the GRPO gradient is SFT's, and the loss is -mean(r A) = -1
    a = L.grpo(H, W, y, np.ones(H.shape[0]), f["logp"], IGN)
    s = L.sft(H, W, y, IGN)
    assert a["loss"] == pytest.approx(-1.0 if f["n_valid"] else 0.0, abs=1e-12)
    assert rel(a["dH"], s["dH"]) <= 1e-12 and rel(a["dW"], s["dW"]) <= 1e-12
    # DPO with references equal to the policy's own sums: every margin is 0, loss log 2
    cu, _ = dpo_inputs(g, H.shape[0])
    if len(cu) >= 3:
        S = L.dpo_pass1(H, W, y, cu, IGN)["seq_logp"]
        d = L.dpo(H, W, y, cu, S, 0.7, IGN)
        assert abs(d["loss"] - math.log(2.0)) <= 1e-12
        assert np.all(np.abs(d["margins"]) <= 1e-12)
