"""GPU parity: the CUDA path through the C ABI against the float64 oracle.

Small and medium shapes that the oracle finishes in seconds but that still span
several 128x256 tiles, several chunks and ragged tails in T, d, V and the chunk;
every objective; the edge cases (empty batch, all tokens ignored, a chunk larger
than T, chunk = 1, accumulation into dW, labels out of range) and determinism.
"""
import numpy as np
import pytest

from oracle import lmhead as O
from memory_efficient_exact_gb300 import inputs as I
from parity_util import TOL, rel, rel_fro, to_dev

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu
IGN = -100


@pytest.fixture(scope="module")
def sbp():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    from memory_efficient_exact_gb300 import _build
    _build.build_library()
    from memory_efficient_exact_gb300 import sbp as mod
    return mod


def make_case(T, d, V, dtype, seed, w_std=0.02, frac=0.1):
    H, W = I.make_hw(T, d, V, seed, dtype, w_std=w_std)
    y = I.make_labels(T, V, seed, "frac", frac)
    return H, W, y


def check_grads(dtype, out, ref, y):
    tol = TOL[dtype]
    dH = out["dH"].float().cpu().numpy()
    dW = out["dW"].cpu().numpy()
    assert rel_fro(dH, ref["dH"]) <= tol["grad"], rel_fro(dH, ref["dH"])
    assert rel_fro(dW, ref["dW"]) <= tol["grad"], rel_fro(dW, ref["dW"])
    ign = np.asarray(y) == IGN
    assert np.all(dH[ign] == 0.0), "rows of ignored tokens must be exactly zero"
    return dH, dW


SFT_CASES = [
    # dtype, T, d, V, chunk, w_std
    ("fp32", 256, 64, 1000, 64, 0.02),      # the fp32 workload of the spec
    ("fp32", 77, 36, 531, 16, 0.3),          # ragged everything
    ("fp32", 40, 16, 97, 1, 0.5),            # chunk = 1
    ("bf16", 300, 256, 2000, 128, 0.05),    # several chunks, ragged last chunk and V tail
    ("bf16", 517, 192, 1304, 200, 0.08),    # d < one 256-wide N tile; V not a tile multiple
    ("bf16", 130, 72, 264, 64, 0.2),        # K tail (72 = 64 + 8)
    ("bf16", 1000, 512, 4096, 384, 0.04),   # many tiles in every dimension
    ("bf16", 640, 1024, 8200, 640, 0.03),   # d spans 4 N tiles, V spans 33 (tail of 8)
    ("bf16", 96, 128, 262144, 64, 0.05),    # a vocabulary of 2^18 (2048 statistics tiles per row)
    ("bf16", 300, 8192, 4096, 256, 0.01),   # d = 8192 (32 N tiles, 128 k-blocks per forward tile)
]


@pytest.mark.parametrize("dtype,T,d,V,chunk,w_std", SFT_CASES)
def test_sft_parity(sbp, dtype, T, d, V, chunk, w_std):
    H, W, y = make_case(T, d, V, dtype, seed=11 + T, w_std=w_std)
    Ht, Wt, yt = to_dev(torch, H, W, y, dtype)
    out = sbp.sft(Ht, Wt, yt, chunk)
    torch.cuda.synchronize()
    sbp.check_status(out["status"])
    ref = O.sft(H, W, y, IGN)
    tol = TOL[dtype]
    assert int(out["n_valid"].item()) == ref["n_valid"]
    assert rel(out["loss"].item(), ref["loss"]) <= tol["loss"], (out["loss"].item(), ref["loss"])
    lp = out["logp"].cpu().numpy()
    assert np.max(np.abs(lp - ref["logp"])) <= tol["logp"] * max(1.0, np.abs(ref["logp"]).max())
    assert np.all(lp[np.asarray(y) == IGN] == 0.0)
    check_grads(dtype, out, ref, y)


@pytest.mark.parametrize("dtype,T,d,V,chunk", [("fp32", 64, 32, 200, 16), ("bf16", 300, 256, 2000, 128),
                                                ("bf16", 520, 128, 1000, 256)])
def test_grpo_parity(sbp, dtype, T, d, V, chunk):
    H, W, y = make_case(T, d, V, dtype, seed=7 + T, w_std=0.1)
    f = O.forward(H, W, y, IGN)
    n_resp = 4
    L = (T + n_resp - 1) // n_resp
    A = I.make_advantages(n_resp, L, seed=T)[:T].astype(np.float32)
    lpo = (f["logp"] + I.make_logp_noise(T, seed=T)).astype(np.float32)
    Ht, Wt, yt = to_dev(torch, H, W, y, dtype)
    out = sbp.grpo(Ht, Wt, yt, torch.from_numpy(A).cuda(), torch.from_numpy(lpo).cuda(), chunk)
    torch.cuda.synchronize()
    sbp.check_status(out["status"])
    ref = O.grpo(H, W, y, A.astype(np.float64), lpo.astype(np.float64), IGN)
    tol = TOL[dtype]
    assert int(out["n_valid"].item()) == ref["n_valid"]
    assert rel(out["loss"].item(), ref["loss"]) <= tol["loss"]
    check_grads(dtype, out, ref, y)


@pytest.mark.parametrize("dtype,T,d,V,chunk,per_seq,kl", [("fp32", 64, 32, 200, 16, True, 0.3),
                                                            ("bf16", 300, 256, 2000, 128, True, 0.1),
                                                            ("bf16", 520, 128, 1000, 256, False, 0.5)])
def test_grpo_variants_parity(sbp, dtype, T, d, V, chunk, per_seq, kl):
    H, W, y = make_case(T, d, V, dtype, seed=17 + T, w_std=0.1)
    f = O.forward(H, W, y, IGN)
    lens = [T // 4, T // 3, T // 6, T - (T // 4 + T // 3 + T // 6)]
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    A = I.make_advantages(len(lens), T, seed=T)[:T].astype(np.float32)
    lpo = (f["logp"] + I.make_logp_noise(T, seed=T)).astype(np.float32)
    ref = (f["logp"] + 0.3 * I.make_logp_noise(T, seed=T + 1)).astype(np.float32)
    Ht, Wt, yt = to_dev(torch, H, W, y, dtype)
    At, lpot, reft = (torch.from_numpy(x).cuda() for x in (A, lpo, ref))
    cut = torch.from_numpy(cu).cuda() if per_seq else None
    out = sbp.grpo_ext(Ht, Wt, yt, At, lpot, chunk, ref_logp=reft, kl_coef=kl, cu_seqlens=cut)
    torch.cuda.synchronize()
    sbp.check_status(out["status"])
    refo = O.grpo_ext(H, W, y, A.astype(np.float64), lpo.astype(np.float64), IGN, ref_logp=ref.astype(np.float64),
                      kl_coef=kl, cu_seqlens=cu if per_seq else None)
    tol = TOL[dtype]
    assert int(out["n_valid"].item()) == refo["n_valid"]
    assert rel(out["loss"].item(), refo["loss"]) <= tol["loss"], (out["loss"].item(), refo["loss"])
    check_grads(dtype, out, refo, y)
    # without the extras the variant is the plain GRPO call, bit for bit
    a = sbp.grpo_ext(Ht, Wt, yt, At, lpot, chunk)
    b = sbp.grpo(Ht, Wt, yt, At, lpot, chunk)
    torch.cuda.synchronize()
    assert torch.equal(a["dH"], b["dH"]) and torch.equal(a["dW"], b["dW"]) and torch.equal(a["loss"], b["loss"])


@pytest.mark.parametrize("dtype,lens,d,V,chunk", [("fp32", [30, 20, 25, 21], 32, 200, 40),
                                                   ("bf16", [200, 96, 150, 74], 256, 2000, 128),
                                                   ("bf16", [128, 256, 64, 192, 100, 100], 128, 1024, 100)])
def test_dpo_parity(sbp, dtype, lens, d, V, chunk):
    T = sum(lens)
    H, W = I.make_hw(T, d, V, 99 + T, dtype, w_std=0.1)
    y = I.make_labels(T, V, 99 + T, "frac", 0.2)
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    n = len(lens)
    f = O.dpo_pass1(H, W, y, cu, IGN)
    # references close to the policy's own sums so that the margins spread around 0
    ref_S = f["seq_logp"] + np.linspace(-3, 3, n)
    beta = 0.5
    Ht, Wt, yt = to_dev(torch, H, W, y, dtype)
    cut = torch.from_numpy(cu).cuda()
    p1 = sbp.dpo_pass1(Ht, Wt, yt, cut, chunk)
    p2 = sbp.dpo_pass2(Ht, Wt, yt, cut, p1["seq_logp"], torch.from_numpy(ref_S).cuda(), beta, chunk)
    torch.cuda.synchronize()
    sbp.check_status(p1["status"])
    sbp.check_status(p2["status"])
    tol = TOL[dtype]
    S = p1["seq_logp"].cpu().numpy()
    assert np.max(np.abs(S - f["seq_logp"]) / np.abs(f["seq_logp"])) <= tol["seq"]
    assert int(p1["n_valid"].item()) == f["n_valid"]
    ref = O.dpo(H, W, y, cu, ref_S, beta, IGN)
    assert rel(p2["loss"].item(), ref["loss"]) <= tol["loss"]
    np.testing.assert_allclose(p2["margins"].cpu().numpy(), ref["margins"], rtol=0, atol=50 * tol["seq"])
    check_grads(dtype, p2, ref, y)


@pytest.mark.parametrize("dtype", ["fp32", "bf16"])
def test_dpo_saturated_margins(sbp, dtype):
    """DPO with the sigmoid far in both tails: the references are set so that the pairs'
    margins are about +5000, -500, +30 and 0 (beta = 0.5).  sigma(-m) underflows to 0 for
    the first, is 1 to fp64 precision for the second; the loss is log(1 + e^-m) summed
    stably (about 500 + 2e-13 + log 2 here, mean over pairs) and the gradient scales
    -beta sigma(-m) must stay finite.  Loss, margins and full dH / dW against the oracle."""
    lens = [60, 50, 40, 30, 60, 50, 40, 30]   # pairs (0, 4), (1, 5), (2, 6), (3, 7)
    d, V, chunk = 64, 704, 64   # V a multiple of 8 (bf16 rows of W 16-byte aligned)
    T = sum(lens)
    H, W = I.make_hw(T, d, V, 4242, dtype, w_std=0.1)
    y = I.make_labels(T, V, 4242, "frac", 0.1)
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    beta = 0.5
    f = O.dpo_pass1(H, W, y, cu, IGN)
    x = np.array([1e4, -1e3, 60.0, 0.0])          # margins beta * x
    ref_S = f["seq_logp"].copy()
    ref_S[:4] -= x                                 # chosen: S_c - ref_c = x, rejected: 0
    Ht, Wt, yt = to_dev(torch, H, W, y, dtype)
    cut = torch.from_numpy(cu).cuda()
    p1 = sbp.dpo_pass1(Ht, Wt, yt, cut, chunk)
    p2 = sbp.dpo_pass2(Ht, Wt, yt, cut, p1["seq_logp"], torch.from_numpy(ref_S).cuda(), beta, chunk)
    torch.cuda.synchronize()
    sbp.check_status(p1["status"])
    sbp.check_status(p2["status"])
    tol = TOL[dtype]
    ref = O.dpo(H, W, y, cu, ref_S, beta, IGN)
    m = p2["margins"].cpu().numpy()
    assert np.all(np.isfinite(m)) and np.isfinite(p2["loss"].item())
    np.testing.assert_allclose(m, ref["margins"], rtol=0, atol=50 * tol["seq"] * np.abs(f["seq_logp"]).max())
    assert m[0] > 4000 and m[1] < -400 and abs(m[3]) < 1
    assert rel(p2["loss"].item(), ref["loss"]) <= tol["loss"]
    dH, dW = p2["dH"].float().cpu().numpy(), p2["dW"].cpu().numpy()
    assert np.all(np.isfinite(dH)) and np.all(np.isfinite(dW))
    check_grads(dtype, p2, ref, y)


@pytest.mark.parametrize("dtype", ["fp32", "bf16"])
def test_accumulate_dw_and_determinism(sbp, dtype):
    T, d, V, chunk = 200, 128, 1000, 64
    H, W, y = make_case(T, d, V, dtype, seed=5, w_std=0.1)
    Ht, Wt, yt = to_dev(torch, H, W, y, dtype)
    a = sbp.sft(Ht, Wt, yt, chunk)
    b = sbp.sft(Ht, Wt, yt, chunk)
    torch.cuda.synchronize()
    assert torch.equal(a["dH"], b["dH"]) and torch.equal(a["dW"], b["dW"]) and torch.equal(a["loss"], b["loss"])
    acc = a["dW"].clone()
    sbp.sft(Ht, Wt, yt, chunk, dW=acc, accumulate_dW=True)
    torch.cuda.synchronize()
    assert torch.allclose(acc, 2 * a["dW"], rtol=1e-6, atol=1e-9)


def test_lean_workspace_same_bits(sbp):
    # the one-buffer schedule (the smallest workspace) forms each chunk's logit gradient
    # in its own pass instead of inside the next chunk's forward: same arithmetic, so the
    # same bits, for SFT and GRPO over several chunks
    T, d, V, chunk = 700, 256, 3000, 128
    H, W, y = make_case(T, d, V, "bf16", seed=11, w_std=0.08)
    Ht, Wt, yt = to_dev(torch, H, W, y, "bf16")
    lean = sbp.make_workspace(T, d, V, chunk, sbp.BF16, sbp.MODE_SFT, lean=True)
    assert lean.numel() < sbp.workspace_bytes(T, d, V, chunk, sbp.BF16, sbp.MODE_SFT)
    a = sbp.sft(Ht, Wt, yt, chunk)
    b = sbp.sft(Ht, Wt, yt, chunk, workspace=lean)
    adv = torch.from_numpy(I.make_advantages(T // 4, 4, 11)).cuda()
    lpo = torch.randn(T, device="cuda") * 0.1 - 8.0
    c = sbp.grpo(Ht, Wt, yt, adv, lpo, chunk)
    e = sbp.grpo(Ht, Wt, yt, adv, lpo, chunk, workspace=lean)
    torch.cuda.synchronize()
    sbp.check_status(b["status"])
    for x, z in ((a, b), (c, e)):
        assert torch.equal(x["dH"], z["dH"]) and torch.equal(x["dW"], z["dW"]) and torch.equal(x["loss"], z["loss"])
    small = torch.empty(lean.numel() - 256, dtype=torch.uint8, device="cuda")
    with pytest.raises(sbp.SbpError):
        sbp.sft(Ht, Wt, yt, chunk, workspace=small)


@pytest.mark.parametrize("dtype", ["fp32", "bf16"])
def test_edge_cases(sbp, dtype):
    d, V = 64, 512
    # all tokens ignored -> loss 0, zero gradients, N = 0
    H, W, y = make_case(50, d, V, dtype, seed=3)
    y[:] = IGN
    Ht, Wt, yt = to_dev(torch, H, W, y, dtype)
    o = sbp.sft(Ht, Wt, yt, 16)
    torch.cuda.synchronize()
    assert o["loss"].item() == 0.0 and int(o["n_valid"].item()) == 0
    assert torch.count_nonzero(o["dH"]).item() == 0 and torch.count_nonzero(o["dW"]).item() == 0
    # empty batch: dW overwritten with zeros, loss 0
    He = torch.empty((0, d), dtype=Ht.dtype, device="cuda")
    ye = torch.empty((0,), dtype=torch.int32, device="cuda")
    dW = torch.full((V, d), 7.0, device="cuda")
    o = sbp.sft(He, Wt, ye, 16, dW=dW)
    torch.cuda.synchronize()
    assert o["loss"].item() == 0.0 and torch.count_nonzero(dW).item() == 0
    # a chunk larger than T equals one chunk
    H, W, y = make_case(50, d, V, dtype, seed=4, w_std=0.2)
    Ht, Wt, yt = to_dev(torch, H, W, y, dtype)
    o1 = sbp.sft(Ht, Wt, yt, 4096)
    o2 = sbp.sft(Ht, Wt, yt, 50)
    torch.cuda.synchronize()
    assert torch.equal(o1["dH"], o2["dH"]) and torch.equal(o1["dW"], o2["dW"])
    ref = O.sft(H, W, y, IGN)
    check_grads(dtype, o1, ref, y)


@pytest.mark.parametrize("dtype,T,d,V,chunk,label", [
    ("bf16", 1, 128, 1000, 1, None),          # a single token
    ("bf16", 64, 16, 256, 16, None),          # d far below one 64-wide k-block
    ("bf16", 700, 256, 2000, 320, None),      # last chunk of 60 rows
    ("bf16", 100, 128, 1000, 64, "last"),     # every label on the last column (V-tail tile)
    ("fp32", 100, 32, 333, 64, "last"),
    ("bf16", 300, 128, 1000, 128, "zero"),    # every label on column 0
    ("fp32", 40, 64, 1, 8, None),             # V = 1: loss 0 and zero gradients exactly
    ("fp32", 50, 64, 7, 16, None),            # V inside one 8-column vector of the gradient pass
    ("bf16", 50, 64, 8, 16, None),            # the smallest bf16 vocabulary (rows of 16 bytes)
])
def test_edge_shapes_and_labels(sbp, dtype, T, d, V, chunk, label):
    H, W, y = make_case(T, d, V, dtype, seed=23 + T + d, w_std=0.2)
    if label == "last":
        y[y != IGN] = V - 1
    elif label == "zero":
        y[y != IGN] = 0
    Ht, Wt, yt = to_dev(torch, H, W, y, dtype)
    out = sbp.sft(Ht, Wt, yt, chunk)
    torch.cuda.synchronize()
    sbp.check_status(out["status"])
    ref = O.sft(H, W, y, IGN)
    tol = TOL[dtype]
    assert int(out["n_valid"].item()) == ref["n_valid"]
    if V == 1:
        assert out["loss"].item() == 0.0 and torch.count_nonzero(out["dH"]).item() == 0
        assert torch.count_nonzero(out["dW"]).item() == 0
        return
    assert rel(out["loss"].item(), ref["loss"]) <= tol["loss"]
    check_grads(dtype, out, ref, y)


def test_label_out_of_range_sets_device_status(sbp):
    H, W, y = make_case(40, 64, 256, "bf16", seed=8)
    y[5] = 256
    Ht, Wt, yt = to_dev(torch, H, W, y, "bf16")
    o = sbp.sft(Ht, Wt, yt, 16)
    torch.cuda.synchronize()
    assert int(o["status"].item()) == sbp.ERR_LABEL_RANGE
    y[5] = -7
    Ht, Wt, yt = to_dev(torch, H, W, y, "fp32")
    o = sbp.sft(Ht, Wt, yt, 16)
    torch.cuda.synchronize()
    assert int(o["status"].item()) == sbp.ERR_LABEL_RANGE


HOST_CASES = [
    # dtype, T, d, V, chunk, pinned
    ("bf16", 700, 256, 3000, 128, True),     # 6 chunks: both slot rings wrap; ragged last chunk
    ("bf16", 517, 192, 1304, 200, True),     # 3 chunks; chunk not a multiple of the 256-row tile
    ("bf16", 300, 256, 2000, 1000, True),    # one chunk (chunk > T)
    ("bf16", 1000, 512, 4096, 384, False),   # pageable host memory: same results
    ("fp32", 77, 36, 531, 16, True),         # fp32 path, 5 chunks, ragged everything
]


@pytest.mark.parametrize("dtype,T,d,V,chunk,pinned", HOST_CASES)
def test_sft_host_same_bits(sbp, dtype, T, d, V, chunk, pinned):
    # H, labels and dH in host memory, streamed chunk by chunk through device slots: the
    # same kernels on the same rows, so the same bits as the device-resident call
    H, W, y = make_case(T, d, V, dtype, seed=21, w_std=0.08)
    Ht, Wt, yt = to_dev(torch, H, W, y, dtype)
    ref = sbp.sft(Ht, Wt, yt, chunk, logp=False)
    Hh, yh = Ht.cpu(), yt.cpu()
    if pinned:
        Hh, yh = Hh.pin_memory(), yh.pin_memory()
    out = sbp.sft_host(Hh, Wt, yh, chunk)
    torch.cuda.synchronize()
    sbp.check_status(out["status"])
    assert torch.equal(out["dH"], ref["dH"].cpu())
    assert torch.equal(out["dW"], ref["dW"])
    assert out["loss"].item() == ref["loss"].item()
    assert int(out["n_valid"]) == int(ref["n_valid"].item())
    # and against the oracle, as the device-resident call
    o = O.sft(H, W, y, IGN)
    assert rel(out["loss"].item(), o["loss"]) <= TOL[dtype]["loss"], (out["loss"].item(), o["loss"])


def test_sft_host_lean_accumulate_and_empty(sbp):
    T, d, V, chunk = 700, 256, 3000, 128
    H, W, y = make_case(T, d, V, "bf16", seed=23, w_std=0.08)
    Ht, Wt, yt = to_dev(torch, H, W, y, "bf16")
    Hh, yh = Ht.cpu().pin_memory(), yt.cpu().pin_memory()
    ref = sbp.sft(Ht, Wt, yt, chunk, logp=False)
    # one-buffer schedule: the smallest accepted host workspace
    full = sbp.host_workspace_bytes(T, d, V, chunk, sbp.BF16)
    lean_dev = sbp.workspace_bytes_lean(T, d, V, chunk, sbp.BF16, sbp.MODE_SFT)
    dev_full = sbp.workspace_bytes(T, d, V, chunk, sbp.BF16, sbp.MODE_SFT)
    lean = torch.empty(full - (dev_full - lean_dev), dtype=torch.uint8, device="cuda")
    out = sbp.sft_host(Hh, Wt, yh, chunk, workspace=lean)
    # accumulation into dW: twice the same batch
    dW = torch.zeros(V, d, device="cuda")
    sbp.sft_host(Hh, Wt, yh, chunk, dW=dW)
    acc = sbp.sft_host(Hh, Wt, yh, chunk, dW=dW, accumulate_dW=True)
    torch.cuda.synchronize()
    sbp.check_status(out["status"])
    assert torch.equal(out["dH"], ref["dH"].cpu()) and torch.equal(out["dW"], ref["dW"])
    assert out["loss"].item() == ref["loss"].item()
    ref2 = sbp.sft(Ht, Wt, yt, chunk, logp=False, dW=ref["dW"].clone(), accumulate_dW=True)
    torch.cuda.synchronize()
    assert torch.equal(acc["dW"], ref2["dW"])
    # empty batch: dW overwritten with zeros, loss 0, N 0
    He = torch.empty((0, d), dtype=torch.bfloat16).pin_memory()
    ye = torch.empty((0,), dtype=torch.int32).pin_memory()
    dW.fill_(7.0)
    e = sbp.sft_host(He, Wt, ye, chunk, dW=dW)
    torch.cuda.synchronize()
    sbp.check_status(e["status"])
    assert e["loss"].item() == 0.0 and int(e["n_valid"]) == 0
    assert torch.count_nonzero(dW).item() == 0


@pytest.mark.parametrize("chunk", [1, 3, 16])
def test_fp32_golden_fixtures(sbp, chunk):
    # the stored oracle fixtures (tests/golden/, tiny odd sizes: d = 5, V = 11) through the
    # fp32 path, in several chunks and with a chunk larger than T
    import json
    import os
    gdir = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
    tol = TOL["fp32"]

    def load(name):
        fx = json.load(open(os.path.join(gdir, name)))
        a = {k: (np.asarray(v) if isinstance(v, list) else v) for k, v in fx["inputs"].items()}
        Ht, Wt, yt = to_dev(torch, a["H"].astype(np.float32), a["W"].astype(np.float32), a["labels"], "fp32")
        return a, fx["outputs"], Ht, Wt, yt

    def grads(out, want):
        assert rel_fro(out["dH"].cpu().numpy(), want["dH"]) <= tol["grad"]
        assert rel_fro(out["dW"].cpu().numpy(), want["dW"]) <= tol["grad"]

    a, want, Ht, Wt, yt = load("lmhead_sft_T7_d5_V11.json")
    o = sbp.sft(Ht, Wt, yt, chunk)
    torch.cuda.synchronize()
    sbp.check_status(o["status"])
    assert int(o["n_valid"].item()) == want["n_valid"]
    assert rel(o["loss"].item(), want["loss"]) <= tol["loss"]
    assert np.max(np.abs(o["logp"].cpu().numpy() - np.asarray(want["logp"]))) <= tol["logp"]
    grads(o, want)

    a, want, Ht, Wt, yt = load("lmhead_grpo_T7_d5_V11.json")
    At = torch.from_numpy(a["advantages"].astype(np.float32)).cuda()
    lpo = torch.from_numpy(a["logp_old"].astype(np.float32)).cuda()
    o = sbp.grpo(Ht, Wt, yt, At, lpo, chunk, a["clip_lo"], a["clip_hi"])
    torch.cuda.synchronize()
    sbp.check_status(o["status"])
    assert int(o["n_valid"].item()) == want["n_valid"]
    assert rel(o["loss"].item(), want["loss"]) <= tol["loss"]
    grads(o, want)

    a, want, Ht, Wt, yt = load("lmhead_dpo_T8_d5_V11.json")
    cut = torch.from_numpy(a["cu_seqlens"].astype(np.int32)).cuda()
    p1 = sbp.dpo_pass1(Ht, Wt, yt, cut, chunk)
    p2 = sbp.dpo_pass2(Ht, Wt, yt, cut, p1["seq_logp"], torch.from_numpy(a["ref_seq_logp"]).cuda(), a["beta"],
                       chunk)
    torch.cuda.synchronize()
    sbp.check_status(p2["status"])
    S = np.asarray(want["seq_logp"])
    assert np.max(np.abs(p1["seq_logp"].cpu().numpy() - S) / np.abs(S)) <= tol["seq"]
    assert rel(p2["loss"].item(), want["loss"]) <= tol["loss"]
    grads(p2, want)


def test_lmhead_calls_under_graph_capture(sbp):
    """The LM-head calls only enqueue work on the caller's stream (the host-buffer call also
    forks the library's side stream from it and joins it back): each can be captured into
    a CUDA graph and replayed, and a replay gives the bits of a plain call.  SFT, GRPO, both
    DPO passes in one graph, and the host-buffer SFT call with page-locked host arrays."""
    T, d, V, chunk = 700, 256, 2000, 256
    H, W, y = make_case(T, d, V, "bf16", seed=91, w_std=0.1)
    Ht, Wt, yt = to_dev(torch, H, W, y, "bf16")
    f = O.forward(H, W, y, IGN)
    A = torch.from_numpy(I.make_advantages(4, (T + 3) // 4, 91)[:T].astype(np.float32)).cuda()
    lpo = torch.from_numpy((f["logp"] + I.make_logp_noise(T, 91)).astype(np.float32)).cuda()
    cu = torch.tensor([0, 200, 350, 550, 700], dtype=torch.int32, device="cuda")
    sref = torch.tensor([-7000.0, -5000.0, -7100.0, -4900.0], dtype=torch.float64, device="cuda")
    s = torch.cuda.Stream()
    mk = lambda mode: sbp.make_workspace(T, d, V, chunk, sbp.BF16, mode)
    ws = {m: mk(m) for m in (sbp.MODE_SFT, sbp.MODE_GRPO, sbp.MODE_DPO1, sbp.MODE_DPO2)}
    st = torch.zeros((), dtype=torch.int32, device="cuda")
    dH, dW = torch.empty_like(Ht), torch.empty((V, d), dtype=torch.float32, device="cuda")
    Hh = torch.from_numpy(H).to(torch.bfloat16).pin_memory()
    yh = torch.from_numpy(y).pin_memory()
    dHh = torch.empty(Hh.shape, dtype=torch.bfloat16).pin_memory()
    lossh = torch.empty((), dtype=torch.float32).pin_memory()
    nvh = torch.empty((), dtype=torch.int64).pin_memory()
    hws = torch.empty(sbp.host_workspace_bytes(T, d, V, chunk, sbp.BF16), dtype=torch.uint8, device="cuda")
    calls = {
        "sft": lambda: sbp.sft(Ht, Wt, yt, chunk, dH=dH, dW=dW, workspace=ws[sbp.MODE_SFT], status=st, stream=s),
        "grpo": lambda: sbp.grpo(Ht, Wt, yt, A, lpo, chunk, dH=dH, dW=dW, workspace=ws[sbp.MODE_GRPO], status=st,
                                 stream=s),
        "dpo": lambda: sbp.dpo_pass2(Ht, Wt, yt, cu, sbp.dpo_pass1(Ht, Wt, yt, cu, chunk, workspace=ws[sbp.MODE_DPO1],
                                                                  status=st, stream=s)["seq_logp"],
                                     sref, 0.5, chunk, dH=dH, dW=dW, workspace=ws[sbp.MODE_DPO2], status=st,
                                     stream=s),
        "host": lambda: sbp.sft_host(Hh, Wt, yh, chunk, dH=dHh, dW=dW, loss=lossh, n_valid=nvh, workspace=hws,
                                     status=st, stream=s),
    }
    for name, call in calls.items():
        # a plain call (which also sets up the library's per-device state), then a capture
        with torch.cuda.stream(s):
            out = call()
        s.synchronize()
        sbp.check_status(st, name)
        ref = {"dH": (dHh if name == "host" else dH).clone(), "dW": dW.clone(),
               "loss": (lossh if name == "host" else out["loss"]).clone()}
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            out = call()
        for _ in range(2):
            dW.zero_()
            (dHh if name == "host" else dH).zero_()
            g.replay()
            torch.cuda.synchronize()
            sbp.check_status(st, name)
            assert torch.equal((dHh if name == "host" else dH), ref["dH"]), name
            assert torch.equal(dW, ref["dW"]), name
            assert torch.equal((lossh if name == "host" else out["loss"]), ref["loss"]), name


def test_host_buffer_calls_from_two_threads(sbp):
    """Host-buffer calls from two host threads on two streams share the library's
    per-device side stream (taken under its lock for each call's enqueue): each gives the
    bits of a call made alone."""
    import threading
    T, d, V, chunk = 900, 256, 2000, 256
    cases = []
    for seed in (5, 6):
        H, W, y = make_case(T, d, V, "bf16", seed=seed, w_std=0.1)
        Wt = torch.from_numpy(W).cuda().to(torch.bfloat16)
        Hh = torch.from_numpy(H).to(torch.bfloat16).pin_memory()
        yh = torch.from_numpy(y).pin_memory()
        ref = sbp.sft_host(Hh, Wt, yh, chunk)
        torch.cuda.synchronize()
        sbp.check_status(ref["status"])
        cases.append((Hh, Wt, yh, {k: v.clone() for k, v in ref.items() if k in ("dH", "dW", "loss")}))
    outs = [None, None]

    def run(i):
        Hh, Wt, yh, _ = cases[i]
        si = torch.cuda.Stream()
        for _ in range(3):   # repeated, so the two threads' calls interleave
            outs[i] = sbp.sft_host(Hh, Wt, yh, chunk, stream=si)
        si.synchronize()
    th = [threading.Thread(target=run, args=(i,)) for i in range(2)]
    for t in th:
        t.start()
    for t in th:
        t.join()
    torch.cuda.synchronize()
    for i in range(2):
        sbp.check_status(outs[i]["status"])
        for k in ("dH", "dW", "loss"):
            assert torch.equal(outs[i][k], cases[i][3][k]), (i, k)
