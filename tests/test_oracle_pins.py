"""Pins of the CPU oracle to things other than itself (CPU only).

Each test checks the oracle against mathematics the method fixes: finite
differences of the loss, the closed form of the cross-entropy logit gradient
(rows sum to zero, ignored rows zero), library routines (scipy log-sum-exp,
PyTorch autograd of cross-entropy in float64), special cases with closed forms
(W = 0, V = 1, N = 0, GRPO with r = 1, DPO at zero margin) and the exactness
claim of the method (chunked == unchunked, ziziman.com article, LM-head
paragraphs; atlas.scime.ai summary, "Approach").  The last tests plant typical
mistakes in a copy of the oracle and check that a pin catches each of them.
"""
import math

import numpy as np
import pytest

import oracle
from oracle import lmhead as L

IGN = -100


def tiny(T=6, d=4, V=7, seed=0, n_ignore=2, scale_w=0.7):
    g = np.random.default_rng(seed)
    H = g.standard_normal((T, d))
    W = scale_w * g.standard_normal((V, d))
    y = g.integers(0, V, T)
    if n_ignore:
        y[g.permutation(T)[:n_ignore]] = IGN
    return H, W, y


def central_fd(fun, X, h=1e-6):
    """Central finite differences of the scalar fun at X, entry by entry."""
    G = np.zeros_like(X)
    it = np.nditer(X, flags=["multi_index"])
    for _ in it:
        i = it.multi_index
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
    return np.linalg.norm(a - b) / (n if n > 0 else 1.0)


# ----------------------------------------------------------------------------- library

def test_lse_and_logp_match_scipy():
    sp = pytest.importorskip("scipy.special")
    H, W, y = tiny(T=9, d=5, V=11, seed=1)
    f = L.forward(H, W, y, IGN)
    Z = H @ W.T
    np.testing.assert_allclose(f["lse"], sp.logsumexp(Z, axis=1), rtol=1e-14, atol=1e-14)
    ls = sp.log_softmax(Z, axis=1)
    v = y != IGN
    np.testing.assert_allclose(f["logp"][v], ls[np.arange(9)[v], y[v]], rtol=1e-13, atol=1e-14)
    assert np.all(f["logp"][~v] == 0)


def test_sft_matches_torch_autograd_fp64():
    torch = pytest.importorskip("torch")
    H, W, y = tiny(T=12, d=5, V=9, seed=2, n_ignore=3)
    o = L.sft(H, W, y, IGN)
    Ht = torch.tensor(H, dtype=torch.float64, requires_grad=True)
    Wt = torch.tensor(W, dtype=torch.float64, requires_grad=True)
    loss = torch.nn.functional.cross_entropy(Ht @ Wt.T, torch.tensor(y, dtype=torch.long),
                                             ignore_index=IGN, reduction="mean")
    loss.backward()
    assert abs(o["loss"] - loss.item()) <= 1e-14 * abs(loss.item())
    np.testing.assert_allclose(o["dH"], Ht.grad.numpy(), rtol=1e-12, atol=1e-15)
    np.testing.assert_allclose(o["dW"], Wt.grad.numpy(), rtol=1e-12, atol=1e-15)


# ----------------------------------------------------------------------------- closed form

def test_ce_grad_rows_sum_to_zero_and_ignored_rows_zero():
    H, W, y = tiny(T=20, d=6, V=13, seed=3, n_ignore=5)
    o = L.sft(H, W, y, IGN)
    v = y != IGN
    N = v.sum()
    G = o["G"]
    assert np.all(G[~v] == 0.0)
    assert np.max(np.abs(G[v].sum(axis=1))) <= 1e-15 * 13
    # softmax minus onehot, divided by N: the target entry is the only negative one
    sp = pytest.importorskip("scipy.special")
    P = sp.softmax(H @ W.T, axis=1)
    E = np.zeros_like(P)
    E[np.arange(20)[v], y[v]] = 1.0
    np.testing.assert_allclose(G[v], (P[v] - E[v]) / N, rtol=1e-12, atol=1e-17)


# ----------------------------------------------------------------------------- finite differences

def _fd_check(loss_fn, H, W, tol=1e-7):
    out = loss_fn()
    dH_fd = central_fd(lambda: loss_fn()["loss"], H)
    dW_fd = central_fd(lambda: loss_fn()["loss"], W)
    assert rel(out["dH"], dH_fd) <= tol, rel(out["dH"], dH_fd)
    assert rel(out["dW"], dW_fd) <= tol, rel(out["dW"], dW_fd)
    # entry-wise too (every entry of dH and dW)
    np.testing.assert_allclose(out["dH"], dH_fd, rtol=1e-6, atol=1e-9)
    np.testing.assert_allclose(out["dW"], dW_fd, rtol=1e-6, atol=1e-9)


def test_fd_sft():
    H, W, y = tiny(seed=4)
    _fd_check(lambda: L.sft(H, W, y, IGN), H, W)


def _grpo_inputs(seed=5):
    H, W, y = tiny(seed=seed)
    f = L.forward(H, W, y, IGN)
    g = np.random.default_rng(seed + 100)
    # ratios r = exp(logp - logp_old) placed >= 1e-3 away from the clip edges 0.8/1.2:
    # inside the interval, below it, above it, with both signs of A
    target_r = np.array([1.05, 0.7, 1.5, 0.95, 1.3, 0.6])
    logp_old = f["logp"] - np.log(target_r)
    A = np.array([0.8, -1.3, 1.1, -0.4, -0.9, 0.5])
    return H, W, y, A, logp_old


def test_fd_grpo():
    H, W, y, A, lpo = _grpo_inputs()
    _fd_check(lambda: L.grpo(H, W, y, A, lpo, IGN), H, W)


def test_fd_dpo():
    H, W, y = tiny(T=8, d=4, V=7, seed=6, n_ignore=2)
    cu = np.array([0, 3, 8])          # one pair: sequence 0 chosen, sequence 1 rejected
    ref = np.array([-1.5, -2.5])
    _fd_check(lambda: L.dpo(H, W, y, cu, ref, 0.7, IGN), H, W)


def test_fd_dpo_two_pairs():
    H, W, y = tiny(T=10, d=3, V=5, seed=7, n_ignore=1)
    cu = np.array([0, 2, 5, 7, 10])
    ref = np.array([-3.0, -1.0, -2.0, -4.0])
    _fd_check(lambda: L.dpo(H, W, y, cu, ref, 0.3, IGN), H, W)


# ----------------------------------------------------------------------------- exactness of chunking

@pytest.mark.parametrize("chunk", [1, 3, 16])
@pytest.mark.parametrize("objective", ["sft", "grpo", "dpo"])
def test_chunked_equals_unchunked(objective, chunk):
    T = 16
    H, W, y = tiny(T=T, d=5, V=9, seed=8, n_ignore=4)
    kw = {}
    if objective == "sft":
        ref = L.sft(H, W, y, IGN)
    elif objective == "grpo":
        g = np.random.default_rng(9)
        A = g.standard_normal(T)
        lpo = L.forward(H, W, y, IGN)["logp"] + 0.1 * g.standard_normal(T)
        kw = dict(advantages=A, logp_old=lpo)
        ref = L.grpo(H, W, y, A, lpo, IGN)
    else:
        cu = np.array([0, 5, 9, 12, 16])
        rf = np.array([-10.0, -11.0, -9.5, -12.0])
        kw = dict(cu_seqlens=cu, ref_seq_logp=rf, beta=0.5)
        ref = L.dpo(H, W, y, cu, rf, 0.5, IGN)
    ch = L.chunked(objective, H, W, y, chunk, IGN, **kw)
    assert abs(ch["loss"] - ref["loss"]) <= 1e-13 * max(1.0, abs(ref["loss"]))
    assert rel(ch["dH"], ref["dH"]) <= 1e-13
    assert rel(ch["dW"], ref["dW"]) <= 1e-12
    np.testing.assert_allclose(ch["logp"], ref["logp"], rtol=1e-14, atol=1e-15)


# ----------------------------------------------------------------------------- special cases

def test_w_zero_closed_form():
    T, d, V = 10, 4, 6
    H, _, y = tiny(T=T, d=d, V=V, seed=10, n_ignore=3)
    W = np.zeros((V, d))
    o = L.sft(H, W, y, IGN)
    v = y != IGN
    N = v.sum()
    assert o["loss"] == pytest.approx(math.log(V), rel=1e-15)
    assert np.all(o["dH"] == 0.0)
    onehot = np.zeros((T, V))
    onehot[np.arange(T)[v], y[v]] = 1.0
    Gc = (np.where(v[:, None], 1.0 / V, 0.0) - onehot) / N
    np.testing.assert_allclose(o["dW"], Gc.T @ H, rtol=1e-13, atol=1e-16)


def test_vocab_of_one():
    H, W, y = tiny(T=5, d=3, V=1, seed=11, n_ignore=1)
    y[y != IGN] = 0
    o = L.sft(H, W, y, IGN)
    assert o["loss"] == 0.0
    assert np.all(o["dH"] == 0.0) and np.all(o["dW"] == 0.0)


def test_all_ignored_gives_zero():
    H, W, y = tiny(T=5, d=3, V=4, seed=12, n_ignore=0)
    y[:] = IGN
    for o in (L.sft(H, W, y, IGN), L.grpo(H, W, y, np.ones(5), np.zeros(5), IGN)):
        assert o["n_valid"] == 0 and o["loss"] == 0.0
        assert np.all(o["dH"] == 0.0) and np.all(o["dW"] == 0.0)


def test_empty_batch():
    W = np.ones((4, 3))
    o = L.sft(np.zeros((0, 3)), W, np.zeros(0, np.int32), IGN)
    assert o["loss"] == 0.0 and o["dH"].shape == (0, 3) and np.all(o["dW"] == 0.0)


def test_label_out_of_range_rejected():
    H, W, y = tiny(T=4, d=3, V=5, seed=13, n_ignore=0)
    y[1] = 5
    with pytest.raises(ValueError):
        L.sft(H, W, y, IGN)
    y[1] = -1
    with pytest.raises(ValueError):
        L.sft(H, W, y, IGN)


# ----------------------------------------------------------------------------- GRPO reductions

def test_grpo_unit_ratio_equals_sft():
    H, W, y = tiny(T=9, d=4, V=6, seed=14, n_ignore=2)
    lp = L.forward(H, W, y, IGN)["logp"]
    s = L.sft(H, W, y, IGN)
    gp = L.grpo(H, W, y, np.ones(9), lp, IGN)
    gm = L.grpo(H, W, y, -np.ones(9), lp, IGN)
    np.testing.assert_array_equal(gp["dH"], s["dH"])
    np.testing.assert_array_equal(gp["dW"], s["dW"])
    np.testing.assert_array_equal(gm["dH"], -s["dH"])
    # objective at r = 1 is A, so the loss is -mean(A) = -1 / +1
    assert gp["loss"] == pytest.approx(-1.0) and gm["loss"] == pytest.approx(1.0)


def test_grpo_clipped_tokens_have_zero_gradient():
    H, W, y = tiny(T=6, d=4, V=6, seed=15, n_ignore=0)
    lp = L.forward(H, W, y, IGN)["logp"]
    A = np.array([1.0, 1.0, -1.0, -1.0, 1.0, -1.0])
    r = np.array([1.3, 1.0, 0.7, 1.0, 1.19, 0.81])
    o = L.grpo(H, W, y, A, lp - np.log(r), IGN)
    G = o["G"]
    assert np.all(G[0] == 0) and np.all(G[2] == 0)              # clipped: r>hi with A>0, r<lo with A<0
    for t in (1, 3, 4, 5):
        assert np.abs(G[t]).max() > 0


# ----------------------------------------------------------------------------- DPO closed form

def test_dpo_zero_margin_closed_form():
    T, beta = 12, 0.25
    H, W, y = tiny(T=T, d=4, V=7, seed=16, n_ignore=3)
    cu = np.array([0, 3, 7, 9, 12])
    S = L.dpo_pass1(H, W, y, cu, IGN)["seq_logp"]
    P = 2
    # choose references so that every margin is exactly zero
    ref = np.concatenate([S[:P] - 1.0, S[P:] - 1.0])
    o = L.dpo(H, W, y, cu, ref, beta, IGN)
    assert np.allclose(o["margins"], 0.0, atol=1e-12)
    assert o["loss"] == pytest.approx(math.log(2.0), rel=1e-12)
    np.testing.assert_allclose(o["seq_weight"], [beta / (2 * P)] * P + [-beta / (2 * P)] * P, rtol=1e-12)
    # G = -beta sigma(-m) grad logp with sign +-1: scale times the per-sequence sum gradient
    f = L.forward(H, W, y, IGN)
    v = f["valid"]
    sid = L.seq_index(cu, T)
    E = np.zeros_like(f["P"])
    E[np.arange(T)[v], y[v]] = 1.0
    sign = np.where(sid < P, 1.0, -1.0)
    G_expect = np.where(v[:, None], (beta * 0.5 / P) * sign[:, None] * (f["P"] - E), 0.0)
    np.testing.assert_allclose(o["G"], G_expect, rtol=1e-12, atol=1e-17)


def test_dpo_margin_sweep_is_finite_and_matches_scipy():
    sp = pytest.importorskip("scipy.special")
    for m in np.linspace(-30, 30, 61):
        S = np.array([m / 0.5, 0.0])
        ref = np.zeros(2)
        mm, loss, w = L.dpo_scales(S, ref, 0.5)
        assert np.isfinite(loss) and np.all(np.isfinite(w))
        assert mm[0] == pytest.approx(m)
        assert loss == pytest.approx(-math.log(sp.expit(m)) if m > -30 else -sp.log_expit(m), rel=1e-12)
        assert w[0] == pytest.approx(0.5 * sp.expit(-m), rel=1e-12)
        assert w[1] == pytest.approx(-0.5 * sp.expit(-m), rel=1e-12)


# ----------------------------------------------------------------------------- row-wise helpers

def test_rowwise_helpers_agree_with_full_oracle():
    H, W, y = tiny(T=30, d=6, V=17, seed=17, n_ignore=6)
    o = L.sft(H, W, y, IGN)
    lse, lp = L.rows_lse_logp(H, W, y, None, IGN, block=7)
    np.testing.assert_allclose(lse, o["lse"], rtol=1e-14)
    np.testing.assert_allclose(lp, o["logp"], rtol=1e-13, atol=1e-15)
    rows = np.array([0, 4, 5, 29])
    w = np.where(y != IGN, 1.0 / (y != IGN).sum(), 0.0)
    np.testing.assert_allclose(L.rows_dH(H, W, y, w, rows, IGN, block=3), o["dH"][rows], rtol=1e-12, atol=1e-16)
    vocab = np.array([0, 3, 16])
    np.testing.assert_allclose(L.cols_dW(H, W, y, w, o["lse"], vocab, IGN), o["dW"][vocab],
                               rtol=1e-12, atol=1e-16)


# ----------------------------------------------------------------------------- planted mistakes

def _mutant(monkeypatch, name, fn):
    monkeypatch.setattr(L, name, fn)


def test_planted_dropped_onehot_is_caught(monkeypatch):
    def bad(f, w):
        G = f["P"] * w[:, None]
        G[~f["valid"]] = 0.0
        return G                      # forgot "- e_y"
    _mutant(monkeypatch, "_logit_grad", bad)
    H, W, y = tiny(seed=18)
    with pytest.raises(AssertionError):
        _fd_check(lambda: L.sft(H, W, y, IGN), H, W)


def test_planted_transposed_backward_is_caught(monkeypatch):
    def bad(G, H, W):
        return G @ L._f64(W), (G.T @ L._f64(H))[::-1].copy()     # wrong vocab row order
    _mutant(monkeypatch, "_backward", bad)
    H, W, y = tiny(seed=19)
    with pytest.raises(AssertionError):
        _fd_check(lambda: L.sft(H, W, y, IGN), H, W)


def test_planted_grpo_wrong_clip_side_is_caught(monkeypatch):
    real = L.grpo_weight

    def bad(logp, logp_old, A, valid, clip_lo=0.8, clip_hi=1.2):
        o, _ = real(logp, logp_old, A, valid, clip_lo, clip_hi)
        r = np.exp(L._f64(logp) - L._f64(logp_old))
        g = (r >= clip_lo) & (r <= clip_hi)          # ignores the sign of A
        return o, np.where(valid & g, L._f64(A) * r, 0.0)
    _mutant(monkeypatch, "grpo_weight", bad)
    H, W, y, A, lpo = _grpo_inputs()
    with pytest.raises(AssertionError):
        _fd_check(lambda: L.grpo(H, W, y, A, lpo, IGN), H, W)


def test_planted_dpo_sign_is_caught(monkeypatch):
    real = L.dpo_scales

    def bad(S, R, beta):
        m, loss, w = real(S, R, beta)
        return m, loss, -w
    _mutant(monkeypatch, "dpo_scales", bad)
    H, W, y = tiny(T=8, d=4, V=7, seed=6, n_ignore=2)
    cu = np.array([0, 3, 8])
    ref = np.array([-1.5, -2.5])
    with pytest.raises(AssertionError):
        _fd_check(lambda: L.dpo(H, W, y, cu, ref, 0.7, IGN), H, W)


def test_planted_per_chunk_mean_is_caught():
    # a chunked loop that divides by the chunk's own count instead of the global N
    H, W, y = tiny(T=12, d=4, V=6, seed=20, n_ignore=4)
    ref = L.sft(H, W, y, IGN)
    dH = np.zeros_like(H)
    for r0 in range(0, 12, 4):
        s = L.sft(H[r0:r0 + 4], W, y[r0:r0 + 4], IGN)
        dH[r0:r0 + 4] = s["dH"]
    assert rel(dH, ref["dH"]) > 1e-3


# ----------------------------------------------------------------------------- GRPO variants

def _ext_inputs(seed=30):
    H, W, y, A, lpo = _grpo_inputs(seed)
    f = L.forward(H, W, y, IGN)
    ref = f["logp"] + np.array([0.3, -0.2, 0.5, -0.4, 0.1, 0.25])
    return H, W, y, A, lpo, ref


@pytest.mark.parametrize("cu", [None, np.array([0, 2, 6])])
def test_fd_grpo_with_kl_and_reduction(cu):
    H, W, y, A, lpo, ref = _ext_inputs()
    _fd_check(lambda: L.grpo_ext(H, W, y, A, lpo, IGN, ref_logp=ref, kl_coef=0.7, cu_seqlens=cu), H, W)


def test_grpo_ext_reduces_to_grpo():
    H, W, y, A, lpo, ref = _ext_inputs(31)
    a = L.grpo(H, W, y, A, lpo, IGN)
    b = L.grpo_ext(H, W, y, A, lpo, IGN)
    assert b["loss"] == pytest.approx(a["loss"], rel=1e-14)
    np.testing.assert_allclose(b["dH"], a["dH"], rtol=1e-13, atol=1e-17)
    np.testing.assert_allclose(b["dW"], a["dW"], rtol=1e-13, atol=1e-17)


def test_kl_term_vanishes_at_the_reference():
    H, W, y, A, lpo, _ = _ext_inputs(32)
    f = L.forward(H, W, y, IGN)
    a = L.grpo(H, W, y, A, lpo, IGN)
    b = L.grpo_ext(H, W, y, A, lpo, IGN, ref_logp=f["logp"], kl_coef=3.0)
    assert b["loss"] == pytest.approx(a["loss"], rel=1e-12)
    np.testing.assert_allclose(b["dH"], a["dH"], rtol=1e-11, atol=1e-15)
    # k3 is non-negative and second order in q
    q = np.linspace(-2, 2, 41)
    k = L.kl_k3(np.zeros_like(q), q)
    assert np.all(k >= 0) and abs(L.kl_k3(0.0, 1e-4) - 0.5e-8) < 1e-12


def test_sequence_mean_equals_token_mean_for_equal_counts():
    H, W, y = tiny(T=12, d=4, V=6, seed=33, n_ignore=0)
    A = np.random.default_rng(1).standard_normal(12)
    lpo = L.forward(H, W, y, IGN)["logp"] + 0.05
    cu = np.array([0, 4, 8, 12])
    a = L.grpo_ext(H, W, y, A, lpo, IGN)
    b = L.grpo_ext(H, W, y, A, lpo, IGN, cu_seqlens=cu)
    assert b["loss"] == pytest.approx(a["loss"], rel=1e-13)
    np.testing.assert_allclose(b["dW"], a["dW"], rtol=1e-12, atol=1e-17)
    # with unequal counts the two reductions differ
    c = L.grpo_ext(H, W, y, A, lpo, IGN, cu_seqlens=np.array([0, 2, 12]))
    assert abs(c["loss"] - a["loss"]) > 1e-6


def test_planted_kl_sign_is_caught(monkeypatch):
    real = L.kl_k3
    monkeypatch.setattr(L, "kl_k3", lambda lp, ref: -real(lp, ref))
    H, W, y, A, lpo, ref = _ext_inputs()
    with pytest.raises(AssertionError):
        _fd_check(lambda: L.grpo_ext(H, W, y, A, lpo, IGN, ref_logp=ref, kl_coef=0.7), H, W)
