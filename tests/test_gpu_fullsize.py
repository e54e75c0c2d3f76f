"""GPU parity at the workloads' full sizes, in the launch configuration of the bench.

The oracle cannot materialise T x V float64 logits at these sizes, so it evaluates
the same definitions row by row: every row's lse / logp (all rows: the loss and the
DPO sums need them), dH on seeded sampled rows, dW on seeded sampled vocabulary rows
(which needs every row's lse).  The 65536-token workload follows its own recipe:
per-token loss and dH on sampled rows of the full run, and the full dW of the
4096-token prefix sub-problem; the GRPO and DPO workloads add the same kind of
sub-problem check (full dH and dW of 4096 of their tokens, unchunked in the oracle).
"""
import numpy as np
import pytest

from oracle import lmhead as O
from memory_efficient_exact_gb300 import inputs as I
from parity_util import TOL, rel, rel_fro

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu
IGN = -100
BF = TOL["bf16"]


@pytest.fixture(scope="module")
def sbp():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    from memory_efficient_exact_gb300 import _build
    _build.build_library()
    from memory_efficient_exact_gb300 import sbp as mod
    return mod


def dev_inputs(H, W, y):
    return (torch.from_numpy(H).cuda().to(torch.bfloat16), torch.from_numpy(W).cuda().to(torch.bfloat16),
            torch.from_numpy(y).cuda())


def vocab_sample(y, V, seed, k=48):
    g = np.random.default_rng(seed)
    lab = np.unique(y[y != IGN])
    pick = np.concatenate([g.choice(lab, size=min(k // 2, len(lab)), replace=False), g.choice(V, size=k // 2)])
    return np.unique(pick)


def check_sampled(H, W, y, w, lse, out, rows, vocab, extra=""):
    dH = out["dH"]
    ign = torch.from_numpy(y == IGN).cuda()
    assert torch.count_nonzero(dH[ign]).item() == 0, "ignored rows of dH must be exactly zero"
    ref_dh = O.rows_dH(H, W, y, w, rows, IGN)
    got_dh = dH[torch.from_numpy(rows).cuda()].float().cpu().numpy()
    e = rel_fro(got_dh, ref_dh)
    assert e <= BF["grad"], f"dH sampled rows {e}{extra}"
    ref_dw = O.cols_dW(H, W, y, w, lse, vocab, IGN)
    got_dw = out["dW"][torch.from_numpy(vocab).cuda()].cpu().numpy()
    e = rel_fro(got_dw, ref_dw)
    assert e <= BF["grad"], f"dW sampled vocab rows {e}{extra}"


@pytest.fixture(scope="module")
def c2():
    x = I.make_workload("sft_bf16_T8192_d2560_V151936")
    lse, logp = O.rows_lse_logp(x["H"], x["W"], x["labels"], None, IGN)
    x["lse"], x["logp"] = lse, logp
    return x


@pytest.mark.parametrize("chunk", [512, 1024, 2048])
def test_sft_T8192_d2560(sbp, c2, chunk):
    H, W, y = c2["H"], c2["W"], c2["labels"]
    valid = y != IGN
    N = int(valid.sum())
    ref_loss = -c2["logp"][valid].sum() / N
    Ht, Wt, yt = dev_inputs(H, W, y)
    out = sbp.sft(Ht, Wt, yt, chunk)
    torch.cuda.synchronize()
    sbp.check_status(out["status"])
    assert int(out["n_valid"].item()) == N
    assert rel(out["loss"].item(), ref_loss) <= BF["loss"]
    lp = out["logp"].cpu().numpy()
    assert np.max(np.abs(lp - c2["logp"])) <= BF["logp"] * np.abs(c2["logp"]).max()
    w = np.where(valid, 1.0 / N, 0.0)
    rows = I.sample_rows(len(y), 256, 1001)
    check_sampled(H, W, y, w, c2["lse"], out, rows, vocab_sample(y, W.shape[0], chunk), f" chunk={chunk}")


def test_sft_T8192_d2560_prefix_full_dW(sbp, c2):
    """The first 4096 tokens as a problem of their own at chunk 1024: the first chunk is the
    1024-token prompt, every label ignored, so one whole chunk contributes nothing while
    the later ones accumulate into dW; full dH and full dW against the unchunked oracle."""
    Tp = 4096
    H, W = np.ascontiguousarray(c2["H"][:Tp]), c2["W"]
    y = np.ascontiguousarray(c2["labels"][:Tp])
    assert np.all(y[:1024] == IGN)
    Ht, Wt, yt = dev_inputs(H, W, y)
    out = sbp.sft(Ht, Wt, yt, 1024)
    torch.cuda.synchronize()
    sbp.check_status(out["status"])
    ref = O.sft(H, W, y, IGN)
    assert int(out["n_valid"].item()) == ref["n_valid"]
    assert rel(out["loss"].item(), ref["loss"]) <= BF["loss"]
    dH = out["dH"].float().cpu().numpy()
    assert rel_fro(dH, ref["dH"]) <= BF["grad"]
    assert rel_fro(out["dW"].cpu().numpy(), ref["dW"]) <= BF["grad"]
    assert np.all(dH[:1024] == 0.0)


@pytest.fixture(scope="module")
def c3():
    return I.make_workload("grpo_bf16_8x2048_d4096_V151936")


def test_grpo_8x2048_d4096(sbp, c3):
    x = c3
    H, W, y = x["H"], x["W"], x["labels"]
    lse, logp = O.rows_lse_logp(H, W, y, None, IGN)
    valid = y != IGN
    lpo = (logp + x["logp_noise"]).astype(np.float32)      # old log-probs fixed at generation
    A = x["advantages"].astype(np.float32)
    N = int(valid.sum())
    o, gar = O.grpo_weight(logp, lpo.astype(np.float64), A.astype(np.float64), valid)
    ref_loss = -o.sum() / N
    Ht, Wt, yt = dev_inputs(H, W, y)
    out = sbp.grpo(Ht, Wt, yt, torch.from_numpy(A).cuda(), torch.from_numpy(lpo).cuda(), 2048)
    torch.cuda.synchronize()
    sbp.check_status(out["status"])
    assert int(out["n_valid"].item()) == N
    assert rel(out["loss"].item(), ref_loss) <= BF["loss"]
    check_sampled(H, W, y, gar / N, lse, out, I.sample_rows(len(y), 256, 1002), vocab_sample(y, W.shape[0], 3))


def test_grpo_8x2048_d4096_prefix_full_dW(sbp, c3):
    """The first two responses (4096 tokens) as a problem of their own, in the bench's
    chunking (two chunks of 2048): full dH and full dW against the unchunked oracle."""
    Tp = 4096
    H, W = np.ascontiguousarray(c3["H"][:Tp]), c3["W"]
    y = np.ascontiguousarray(c3["labels"][:Tp])
    _, logp = O.rows_lse_logp(H, W, y, None, IGN)
    lpo = (logp + c3["logp_noise"][:Tp]).astype(np.float32)
    A = np.ascontiguousarray(c3["advantages"][:Tp]).astype(np.float32)
    Ht, Wt, yt = dev_inputs(H, W, y)
    out = sbp.grpo(Ht, Wt, yt, torch.from_numpy(A).cuda(), torch.from_numpy(lpo).cuda(), 2048)
    torch.cuda.synchronize()
    sbp.check_status(out["status"])
    ref = O.grpo(H, W, y, A.astype(np.float64), lpo.astype(np.float64), IGN)
    assert int(out["n_valid"].item()) == ref["n_valid"]
    assert rel(out["loss"].item(), ref["loss"]) <= BF["loss"]
    dH = out["dH"].float().cpu().numpy()
    assert rel_fro(dH, ref["dH"]) <= BF["grad"]
    assert rel_fro(out["dW"].cpu().numpy(), ref["dW"]) <= BF["grad"]
    assert np.all(dH[y == IGN] == 0.0)


@pytest.fixture(scope="module")
def c4():
    return I.make_workload("dpo_bf16_8x4096_d4096_V151936")


def test_dpo_8x4096_d4096(sbp, c4):
    x = c4
    H, W, y, cu, Sref = x["H"], x["W"], x["labels"], x["cu_seqlens"], x["ref_seq_logp"]
    lse, logp = O.rows_lse_logp(H, W, y, None, IGN)
    valid = y != IGN
    S = O.seq_sums(logp, valid, cu)
    m, ref_loss, wseq = O.dpo_scales(S, Sref, 0.1)
    sid = O.seq_index(cu, len(y))
    w = np.where(valid & (sid >= 0), wseq[np.maximum(sid, 0)], 0.0)
    Ht, Wt, yt = dev_inputs(H, W, y)
    cut = torch.from_numpy(cu).cuda()
    p1 = sbp.dpo_pass1(Ht, Wt, yt, cut, 2048)
    p2 = sbp.dpo_pass2(Ht, Wt, yt, cut, p1["seq_logp"], torch.from_numpy(Sref).cuda(), 0.1, 2048)
    torch.cuda.synchronize()
    sbp.check_status(p1["status"])
    sbp.check_status(p2["status"])
    Sg = p1["seq_logp"].cpu().numpy()
    assert np.max(np.abs(Sg - S) / np.abs(S)) <= BF["seq"]
    assert rel(p2["loss"].item(), ref_loss) <= BF["loss"]
    check_sampled(H, W, y, w, lse, p2, I.sample_rows(len(y), 256, 1003), vocab_sample(y, W.shape[0], 4))


def test_dpo_8x4096_d4096_prefix_full_dW(sbp, c4):
    """One preference pair as a problem of its own: the first 2048 tokens of the chosen
    sequence 0 and of its rejected partner, sequence 4 (each with its 1024-token head
    masked, as in the workload), with their reference sums.  Pass 1's sums go through
    pass 2 on the device, in the bench's chunking; full dH and full dW against the
    unchunked oracle."""
    L, Lw = 2048, 4096
    rows = np.concatenate([np.arange(0, L), np.arange(4 * Lw, 4 * Lw + L)])
    H, W = np.ascontiguousarray(c4["H"][rows]), c4["W"]
    y = np.ascontiguousarray(c4["labels"][rows])
    cu = np.array([0, L, 2 * L], dtype=np.int32)
    Sref = np.ascontiguousarray(c4["ref_seq_logp"][[0, 4]])
    Ht, Wt, yt = dev_inputs(H, W, y)
    cut = torch.from_numpy(cu).cuda()
    p1 = sbp.dpo_pass1(Ht, Wt, yt, cut, 2048)
    p2 = sbp.dpo_pass2(Ht, Wt, yt, cut, p1["seq_logp"], torch.from_numpy(Sref).cuda(), 0.1, 2048)
    torch.cuda.synchronize()
    sbp.check_status(p1["status"])
    sbp.check_status(p2["status"])
    ref = O.dpo(H, W, y, cu, Sref, 0.1, IGN)
    Sg = p1["seq_logp"].cpu().numpy()
    assert np.max(np.abs(Sg - ref["seq_logp"]) / np.abs(ref["seq_logp"])) <= BF["seq"]
    assert rel(p2["loss"].item(), ref["loss"]) <= BF["loss"]
    dH = p2["dH"].float().cpu().numpy()
    assert rel_fro(dH, ref["dH"]) <= BF["grad"]
    assert rel_fro(p2["dW"].cpu().numpy(), ref["dW"]) <= BF["grad"]
    assert np.all(dH[y == IGN] == 0.0)


@pytest.fixture(scope="module")
def c5():
    x = I.make_workload("sft_bf16_T65536_d5120_V151936")
    H, W, y = x["H"], x["W"], x["labels"]
    valid = y != IGN
    x["rows"] = I.sample_rows(H.shape[0], 4096, 1004)
    x["lse_s"], x["logp_s"] = O.rows_lse_logp(H, W, y, x["rows"], IGN)
    x["sub"] = x["rows"][::8]
    x["ref_dh"] = O.rows_dH(H, W, y, np.where(valid, 1.0 / int(valid.sum()), 0.0), x["sub"], IGN)
    return x


@pytest.mark.parametrize("chunk", [512, 1024, 2048, 4096, 8192])
def test_sft_T65536_d5120_sampled(sbp, c5, chunk):
    H, W, y = c5["H"], c5["W"], c5["labels"]
    valid = y != IGN
    N = int(valid.sum())
    Ht, Wt, yt = dev_inputs(H, W, y)
    torch.cuda.reset_peak_memory_stats()
    base = torch.cuda.memory_allocated()
    out = sbp.sft(Ht, Wt, yt, chunk)
    torch.cuda.synchronize()
    sbp.check_status(out["status"])
    peak_extra = torch.cuda.max_memory_allocated() - base
    T, V, d = H.shape[0], W.shape[0], H.shape[1]
    # device memory beyond the inputs: dH, dW, the outputs and one chunk's workspace --
    # far below the unchunked fp32 logits (T x V x 4 = 39.8 GB)
    ws = sbp.workspace_bytes(T, d, V, chunk, sbp.BF16, sbp.MODE_SFT)
    assert peak_extra <= T * d * 2 + V * d * 4 + ws + 64 * T + (1 << 24)
    assert peak_extra < T * V * 4 / 4
    assert int(out["n_valid"].item()) == N
    rows, logp_s = c5["rows"], c5["logp_s"]
    lp = out["logp"].cpu().numpy()
    assert np.max(np.abs(lp[rows] - logp_s)) <= BF["logp"] * np.abs(logp_s).max()
    # the loss is the mean of the per-token terms (a property at any size) ...
    assert rel(out["loss"].item(), -lp[valid].astype(np.float64).sum() / N) <= 1e-5
    # ... and over the sampled rows that mean agrees with the oracle's
    vs = valid[rows]
    assert rel(-lp[rows][vs].astype(np.float64).mean(), -logp_s[vs].mean()) <= BF["loss"]
    got = out["dH"][torch.from_numpy(c5["sub"]).cuda()].float().cpu().numpy()
    assert rel_fro(got, c5["ref_dh"]) <= BF["grad"]
    assert torch.count_nonzero(out["dH"][torch.from_numpy(~valid).cuda()]).item() == 0


def test_sft_T65536_d5120_prefix_full_dW(sbp, c5):
    Tp = 4096
    H, W, y = c5["H"][:Tp], c5["W"], c5["labels"][:Tp]
    Ht, Wt, yt = dev_inputs(np.ascontiguousarray(H), W, np.ascontiguousarray(y))
    out = sbp.sft(Ht, Wt, yt, 2048)
    torch.cuda.synchronize()
    sbp.check_status(out["status"])
    ref = O.sft(H, W, y, IGN)
    assert rel(out["loss"].item(), ref["loss"]) <= BF["loss"]
    assert rel_fro(out["dH"].float().cpu().numpy(), ref["dH"]) <= BF["grad"]
    assert rel_fro(out["dW"].cpu().numpy(), ref["dW"]) <= BF["grad"]
