"""CPU oracle for the StreamBP language-model head: plain, unchunked, float64.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path may import, call or execute
this module: only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` /
``--impl reference`` legs of ``bench.py`` use it.  It shares no code with the CUDA
path; the one module both sides use is the seeded input generator.

Source of the method: "StreamBP: Memory-Efficient Exact Backpropagation for Long
Sequence Training of LLMs" (Luo, Li, Zhao, Li; arXiv 2506.03077), as summarised on
the ziziman.com article (the LM-head paragraphs on SFT/GRPO and on DPO), the
chatpaper.ai / fugumt.com abstract pages and the atlas.scime.ai summary
("Approach").  The pages fix the principle only: the LM-head gradient is computed
chunk by chunk along the sequence, and the result is *exactly* the unchunked
gradient.  So this oracle is the plain unchunked definition:

    Z = H W^T (all T x V logits, materialised), lse_t = log sum_v exp Z_tv,
    logp_t = Z_{t, y_t} - lse_t, P = exp(Z - lse),
    G = dL/dZ, dH = G W, dW = G^T H.

The objectives (SFT cross-entropy, GRPO/PPO-clip, DPO) follow their standard
definitions; the readings taken where the pages are silent are listed at each
function.  Every function here is pinned by ``tests/test_oracle_pins.py`` to
something other than itself (finite differences, closed forms, library routines,
special cases).  Parity pins that rest only on a reading of the pages (the N = 0
convention, the GRPO token mean, the DPO pair layout) are marked "reading" below.
"""
from __future__ import annotations

import numpy as np

IGNORE_INDEX = -100


def _f64(x) -> np.ndarray:
    return np.asarray(x, dtype=np.float64)


def check_labels(y: np.ndarray, V: int, ignore_index: int) -> None:
    y = np.asarray(y)
    bad = (y != ignore_index) & ((y < 0) | (y >= V))
    if bad.any():
        raise ValueError("label outside [0, V) that is not ignore_index")


def logits(H, W) -> np.ndarray:
    """Z = H W^T in float64, the full T x V matrix (LM-head forward)."""
    return _f64(H) @ _f64(W).T


def row_lse(Z: np.ndarray) -> np.ndarray:
    """lse_t = m_t + log sum_v exp(Z_tv - m_t), m_t = max_v Z_tv (stable log-sum-exp)."""
    m = Z.max(axis=1)
    return m + np.log(np.exp(Z - m[:, None]).sum(axis=1))


def forward(H, W, y, ignore_index: int = IGNORE_INDEX) -> dict:
    """Logits, row log-sum-exp, per-token label log-prob and the softmax, unchunked.

    Label alignment (reading): labels[t] is the target of row H[t]; the caller shifts.
    Ignored tokens get logp = 0 and take no part in any sum.
    """
    H, W = _f64(H), _f64(W)
    y = np.asarray(y).astype(np.int64)
    T, V = H.shape[0], W.shape[0]
    check_labels(y, V, ignore_index)
    valid = y != ignore_index
    if T == 0:
        Z = np.zeros((0, V))
        return dict(Z=Z, lse=np.zeros(0), logp=np.zeros(0), P=Z, valid=valid, y=y, n_valid=0)
    Z = logits(H, W)
    lse = row_lse(Z)
    yc = np.where(valid, y, 0)
    logp = np.where(valid, Z[np.arange(T), yc] - lse, 0.0)
    P = np.exp(Z - lse[:, None])
    return dict(Z=Z, lse=lse, logp=logp, P=P, valid=valid, y=y, n_valid=int(valid.sum()))


def _logit_grad(f: dict, w: np.ndarray) -> np.ndarray:
    """G_t = w_t (P_t - e_{y_t}) for valid t, 0 for ignored t.

    This is dL/dZ for any loss whose dependence on row t is through logp_t, with
    w_t = -dL/dlogp_t, because dlogp_t/dZ_tv = [v = y_t] - P_tv.
    """
    G = f["P"] * w[:, None]
    idx = np.nonzero(f["valid"])[0]
    G[idx, f["y"][idx]] -= w[idx]
    G[~f["valid"]] = 0.0
    return G


def _backward(G, H, W):
    return G @ _f64(W), G.T @ _f64(H)


def sft(H, W, y, ignore_index: int = IGNORE_INDEX) -> dict:
    """SFT cross-entropy, mean over the non-ignored tokens of the whole call.

    L = -(1/N) sum_{valid t} logp_t, G_t = (P_t - e_{y_t}) / N.
    Reading: N is the count over the whole call (not per chunk).  N = 0 gives
    loss 0 and zero gradients (PyTorch would give NaN).
    """
    f = forward(H, W, y, ignore_index)
    N = f["n_valid"]
    inv = 1.0 / N if N else 0.0
    loss = -float(f["logp"][f["valid"]].sum()) * inv
    w = np.where(f["valid"], inv, 0.0)
    G = _logit_grad(f, w)
    dH, dW = _backward(G, H, W)
    return dict(loss=loss, n_valid=N, logp=f["logp"], lse=f["lse"], G=G, dH=dH, dW=dW)


def grpo_weight(logp, logp_old, A, valid, clip_lo=0.8, clip_hi=1.2):
    """Per-token GRPO/PPO-clip objective and its logit-gradient weight.

    r_t = exp(logp_t - logp_old_t); o_t = min(r_t A_t, clip(r_t, lo, hi) A_t).
    The derivative of o_t with respect to r_t is A_t when the unclipped branch is
    active and 0 otherwise.  Active branch (closed at the clip edges, matching the
    min/clamp subgradient convention): A >= 0 and r <= hi, or A < 0 and r >= lo.
    do_t/dlogp_t = g_t A_t r_t.  Returns (o, g A r).
    """
    r = np.exp(_f64(logp) - _f64(logp_old))
    A = _f64(A)
    o = np.minimum(r * A, np.clip(r, clip_lo, clip_hi) * A)
    g = ((A >= 0) & (r <= clip_hi)) | ((A < 0) & (r >= clip_lo))
    return np.where(valid, o, 0.0), np.where(valid & g, A * r, 0.0)


def grpo(H, W, y, advantages, logp_old, ignore_index: int = IGNORE_INDEX,
         clip_lo: float = 0.8, clip_hi: float = 1.2) -> dict:
    """GRPO/PPO-clip per-token objective, token mean over the non-ignored tokens.

    L = -(1/N) sum_{valid t} min(r_t A_t, clip(r_t, lo, hi) A_t), r_t = exp(logp_t - logp_old_t).
    G_t = (g_t A_t r_t / N) (P_t - e_{y_t}).
    Reading: one token mean over all responses of the call (the workload's
    "-mean_t"); no KL or entropy term.
    """
    f = forward(H, W, y, ignore_index)
    N = f["n_valid"]
    inv = 1.0 / N if N else 0.0
    o, gar = grpo_weight(f["logp"], logp_old, advantages, f["valid"], clip_lo, clip_hi)
    loss = -float(o.sum()) * inv
    G = _logit_grad(f, gar * inv)
    dH, dW = _backward(G, H, W)
    return dict(loss=loss, n_valid=N, logp=f["logp"], lse=f["lse"], G=G, dH=dH, dW=dW)


def kl_k3(logp, ref_logp):
    """Per-token KL estimate to a reference policy, k3 form: exp(q) - q - 1 with
    q = ref_logp - logp (non-negative, zero when the two agree)."""
    q = _f64(ref_logp) - _f64(logp)
    return np.exp(q) - q - 1.0


def grpo_ext(H, W, y, advantages, logp_old, ignore_index: int = IGNORE_INDEX, clip_lo: float = 0.8,
             clip_hi: float = 1.2, ref_logp=None, kl_coef: float = 0.0, cu_seqlens=None) -> dict:
    """GRPO / PPO-clip with an optional KL penalty and an optional per-sequence mean.

    Per-token term  l_t = -min(r_t A_t, clip(r_t) A_t) + kl_coef * KL_t,
    KL_t = exp(q_t) - q_t - 1, q_t = ref_logp_t - logp_t (k3 estimator).
    Reduction (reading): with cu_seqlens None, the token mean over the N non-ignored
    tokens; otherwise the mean over the S sequences of each sequence's token mean,
    L = (1/S) sum_i (1/N_i) sum_{t in i, valid} l_t, where a sequence without a valid
    token contributes 0 (and still counts in S); tokens outside every sequence get no
    weight.  dl_t/dlogp_t = -g_t A_t r_t + kl_coef (1 - exp(q_t)), so the logit-gradient
    weight is w_t = f_t (g_t A_t r_t - kl_coef (1 - exp(q_t))) with f_t the token's
    share of the mean.
    """
    f = forward(H, W, y, ignore_index)
    T = f["P"].shape[0]
    valid = f["valid"]
    o, gar = grpo_weight(f["logp"], logp_old, advantages, valid, clip_lo, clip_hi)
    if ref_logp is not None and kl_coef != 0.0:
        kl = np.where(valid, kl_k3(f["logp"], ref_logp), 0.0)
        dkl = np.where(valid, 1.0 - np.exp(_f64(ref_logp) - f["logp"]), 0.0)
    else:
        kl = np.zeros(T)
        dkl = np.zeros(T)
    term = np.where(valid, -o + kl_coef * kl, 0.0)
    if cu_seqlens is None:
        N = f["n_valid"]
        fac = np.where(valid, 1.0 / N if N else 0.0, 0.0)
    else:
        cu = np.asarray(cu_seqlens, dtype=np.int64)
        S = len(cu) - 1
        sid = seq_index(cu, T)
        Ni = np.array([int(valid[cu[i]:cu[i + 1]].sum()) for i in range(S)])
        per = np.where(Ni > 0, 1.0 / (S * np.maximum(Ni, 1)), 0.0)
        fac = np.where(valid & (sid >= 0), per[np.maximum(sid, 0)] if S else 0.0, 0.0)
    loss = float((term * fac).sum())
    w = fac * (gar - kl_coef * dkl)
    G = _logit_grad(f, w)
    dH, dW = _backward(G, H, W)
    return dict(loss=loss, n_valid=f["n_valid"], logp=f["logp"], lse=f["lse"], G=G, dH=dH, dW=dW, weight=w)


def seq_index(cu_seqlens, T: int) -> np.ndarray:
    """Sequence id of every token; tokens outside [cu[0], cu[-1]) get -1."""
    cu = np.asarray(cu_seqlens, dtype=np.int64)
    s = np.searchsorted(cu, np.arange(T), side="right") - 1
    s[(np.arange(T) < cu[0]) | (np.arange(T) >= cu[-1])] = -1
    return s


def seq_sums(logp, valid, cu_seqlens) -> np.ndarray:
    """S_i = sum of the label log-probs of the non-ignored tokens of sequence i."""
    cu = np.asarray(cu_seqlens, dtype=np.int64)
    lv = np.where(valid, logp, 0.0)
    return np.array([lv[cu[i]:cu[i + 1]].sum() for i in range(len(cu) - 1)], dtype=np.float64)


def dpo_pass1(H, W, y, cu_seqlens, ignore_index: int = IGNORE_INDEX) -> dict:
    """DPO first pass: per-sequence summed label log-probs (DPO paragraph of the
    ziziman.com article: the sigmoid couples positions, so the sums come first)."""
    f = forward(H, W, y, ignore_index)
    return dict(seq_logp=seq_sums(f["logp"], f["valid"], cu_seqlens), logp=f["logp"],
                lse=f["lse"], n_valid=f["n_valid"])


def softplus(x):
    return np.logaddexp(0.0, _f64(x))


def sigmoid(x):
    return np.exp(-np.logaddexp(0.0, -_f64(x)))


def dpo_scales(seq_logp, ref_seq_logp, beta: float):
    """Margins, loss and per-sequence logit-gradient weights of DPO.

    Reading: sequences [0, P) are the chosen answers, [P, 2P) the rejected ones,
    pair i = (i, i + P); the loss is the mean over pairs; no label smoothing.
    m_i = beta [(S_i - S_i^ref) - (S_{i+P} - S_{i+P}^ref)],  L = (1/P) sum softplus(-m_i),
    dL/dS_i = -beta sigma(-m_i)/P,  dL/dS_{i+P} = +beta sigma(-m_i)/P.
    The weight of the logit gradient of a token of sequence j is -dL/dS_j.
    """
    S, R = _f64(seq_logp), _f64(ref_seq_logp)
    n = S.shape[0]
    if n % 2:
        raise ValueError("DPO needs an even number of sequences")
    P = n // 2
    m = beta * ((S[:P] - R[:P]) - (S[P:] - R[P:]))
    loss = float(softplus(-m).sum() / P) if P else 0.0
    s = beta * sigmoid(-m) / P if P else np.zeros(0)
    w = np.concatenate([s, -s])
    return m, loss, w


def dpo(H, W, y, cu_seqlens, ref_seq_logp, beta: float, ignore_index: int = IGNORE_INDEX) -> dict:
    """DPO loss and gradients (both passes, unchunked): G_t = w_{seq(t)} (P_t - e_{y_t})."""
    f = forward(H, W, y, ignore_index)
    S = seq_sums(f["logp"], f["valid"], cu_seqlens)
    m, loss, wseq = dpo_scales(S, ref_seq_logp, beta)
    T = f["P"].shape[0]
    sid = seq_index(cu_seqlens, T)
    w = np.where((sid >= 0) & f["valid"], wseq[np.maximum(sid, 0)] if len(wseq) else 0.0, 0.0)
    G = _logit_grad(f, w)
    dH, dW = _backward(G, H, W)
    return dict(loss=loss, seq_logp=S, margins=m, seq_weight=wseq, logp=f["logp"],
                lse=f["lse"], G=G, dH=dH, dW=dW, n_valid=f["n_valid"])


# --------------------------------------------------------------------------------------
# The chunked form of the same computation (the method itself, in float64), used only
# to pin "chunked == unchunked".  Chunks are contiguous row ranges of `chunk` rows.
# --------------------------------------------------------------------------------------

def chunked(objective: str, H, W, y, chunk: int, ignore_index: int = IGNORE_INDEX, **kw) -> dict:
    """The LM-head gradient computed one row chunk at a time (ziziman.com article,
    LM-head paragraph): only one chunk's logits and logit gradient exist at a time;
    dH_c = G_c W is written per chunk and dW accumulates G_c^T H_c.

    The global quantities that the weights need (N; for DPO the sequence sums)
    are computed first, as the method requires."""
    H, W = _f64(H), _f64(W)
    y = np.asarray(y).astype(np.int64)
    T, d = H.shape
    V = W.shape[0]
    check_labels(y, V, ignore_index)
    valid = y != ignore_index
    N = int(valid.sum())
    inv = 1.0 / N if N else 0.0
    dH = np.zeros((T, d))
    dW = np.zeros((V, d))
    logp = np.zeros(T)
    out = {}
    if objective == "dpo":
        # pass 1: sequence sums from chunked forwards
        for r0 in range(0, T, chunk):
            f = forward(H[r0:r0 + chunk], W, y[r0:r0 + chunk], ignore_index)
            logp[r0:r0 + chunk] = f["logp"]
        S = seq_sums(logp, valid, kw["cu_seqlens"])
        m, loss, wseq = dpo_scales(S, kw["ref_seq_logp"], kw["beta"])
        sid = seq_index(kw["cu_seqlens"], T)
        out.update(seq_logp=S, margins=m)
    loss_acc = 0.0
    for r0 in range(0, T, chunk):
        sl = slice(r0, min(T, r0 + chunk))
        f = forward(H[sl], W, y[sl], ignore_index)
        logp[sl] = f["logp"]
        if objective == "sft":
            w = np.where(f["valid"], inv, 0.0)
            loss_acc += -float(f["logp"][f["valid"]].sum()) * inv
        elif objective == "grpo":
            o, gar = grpo_weight(f["logp"], kw["logp_old"][sl], kw["advantages"][sl], f["valid"],
                                 kw.get("clip_lo", 0.8), kw.get("clip_hi", 1.2))
            w = gar * inv
            loss_acc += -float(o.sum()) * inv
        elif objective == "dpo":
            s = sid[sl]
            w = np.where((s >= 0) & f["valid"], wseq[np.maximum(s, 0)], 0.0)
        else:
            raise ValueError(objective)
        G = _logit_grad(f, w)
        dH[sl] = G @ W
        dW += G.T @ H[sl]
    if objective != "dpo":
        loss = loss_acc
    out.update(loss=loss, logp=logp, dH=dH, dW=dW, n_valid=N)
    return out


# --------------------------------------------------------------------------------------
# Row-wise evaluation of the same definitions for workloads too large to materialise:
# every quantity of row t depends on H[t], W and the row's label only, so rows can be
# evaluated one at a time (grouped into blocks of rows purely for BLAS speed).
# --------------------------------------------------------------------------------------

def rows_lse_logp(H, W, y, rows=None, ignore_index: int = IGNORE_INDEX, block: int = 256):
    """lse_t and logp_t (0 for ignored t) for the given rows (all rows if None)."""
    H = np.asarray(H)
    W64 = _f64(W)
    y = np.asarray(y).astype(np.int64)
    rows = np.arange(H.shape[0]) if rows is None else np.asarray(rows)
    lse = np.empty(len(rows))
    logp = np.zeros(len(rows))
    for b in range(0, len(rows), block):
        r = rows[b:b + block]
        Z = _f64(H[r]) @ W64.T
        l = row_lse(Z)
        lse[b:b + block] = l
        yr = y[r]
        v = yr != ignore_index
        logp[b:b + block] = np.where(v, Z[np.arange(len(r)), np.where(v, yr, 0)] - l, 0.0)
    return lse, logp


def rows_dH(H, W, y, w, rows, ignore_index: int = IGNORE_INDEX, block: int = 256):
    """dH_t = w_t (P_t - e_{y_t}) W for the given rows, with per-row weights w[rows]."""
    W64 = _f64(W)
    y = np.asarray(y).astype(np.int64)
    out = np.empty((len(rows), W64.shape[1]))
    for b in range(0, len(rows), block):
        r = np.asarray(rows[b:b + block])
        Z = _f64(np.asarray(H)[r]) @ W64.T
        P = np.exp(Z - row_lse(Z)[:, None])
        wr = _f64(w)[r]
        yr = y[r]
        v = yr != ignore_index
        G = P * wr[:, None]
        idx = np.nonzero(v)[0]
        G[idx, yr[idx]] -= wr[idx]
        G[~v] = 0.0
        out[b:b + block] = G @ W64
    return out


def cols_dW(H, W, y, w, lse, vocab, ignore_index: int = IGNORE_INDEX):
    """dW_v = sum_t w_t (P_tv - [y_t = v]) H_t for the given vocabulary rows v,
    given every row's lse_t (P_tv = exp(H_t . W_v - lse_t))."""
    H64 = _f64(H)
    W64 = _f64(W)
    y = np.asarray(y).astype(np.int64)
    vocab = np.asarray(vocab)
    valid = y != ignore_index
    Zc = H64 @ W64[vocab].T                        # [T, k]
    Pc = np.exp(Zc - _f64(lse)[:, None])
    Gc = Pc * _f64(w)[:, None]
    Gc -= (y[:, None] == vocab[None, :]) * _f64(w)[:, None]
    Gc[~valid] = 0.0
    return Gc.T @ H64
