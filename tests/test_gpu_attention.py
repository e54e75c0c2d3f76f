"""GPU parity of the chunked causal-attention backward against the float64 oracle.

Inputs: Q, K, V, dO ~ N(0, 1) rounded to bf16; O and lse from the oracle's forward on the
same values (O rounded to bf16, lse kept in fp32, as a forward saves them); the expected
gradients are the oracle's unchunked backward on exactly the values the GPU sees.
Shapes span several heads, several chunks with a ragged last one, row pairs and 256-key
tiles; the benchmark's size (T=8192) and the long-sequence one (T=32768, grouped heads) on
sampled rows and keys; dQ / dK / dV relative Frobenius error <= 2e-2 (the bf16 tolerance
of the other tests).
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


def make(H, T, hd, seed, Hkv=None):
    g = np.random.default_rng(seed)
    Hkv = H if Hkv is None else Hkv
    Q, dO = (I.round_bf16(g.standard_normal((H, T, hd), dtype=np.float32)) for _ in range(2))
    K, V = (I.round_bf16(g.standard_normal((Hkv, T, hd), dtype=np.float32)) for _ in range(2))
    scale = 1.0 / np.sqrt(hd)
    f = A.forward(Q, K, V, scale)
    O = I.round_bf16(f["O"].astype(np.float32))
    lse = f["lse"].astype(np.float32)
    return Q, K, V, O, dO, lse, scale


def dev(x, dt=torch.bfloat16):
    return torch.from_numpy(np.ascontiguousarray(x)).cuda().to(dt).contiguous()


# hd = 128 runs the fused kernels (P and dS on chip), other widths the chunk-buffer path.
# The hd = 128 cases cover one token, chunks of one token, chunks that are not multiples
# of the 128-query block, a chunk equal to T, several 256-key units per head, and more
# units than SM pairs (H = 48), so that every barrier crosses unit boundaries.
@pytest.mark.parametrize("H,T,hd,chunk", [(2, 300, 64, 128), (4, 640, 128, 256), (3, 513, 128, 200),
                                          (1, 1024, 64, 1024), (2, 96, 128, 40), (1, 1, 128, 1),
                                          (2, 5, 128, 3), (2, 67, 128, 1), (1, 700, 128, 700),
                                          (2, 1100, 128, 384), (48, 1024, 128, 512), (1, 260, 192, 100)])
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


# grouped-query attention (key / value heads shared by H / Hkv query heads, the Qwen3
# layout): head dimension 128, groups of 2 to 8 (8: the Qwen3-32B ratio, 5: Qwen3-14B),
# one shared head (multi-query), ragged chunks, and more units than SM pairs
@pytest.mark.parametrize("H,Hkv,T,chunk", [(8, 2, 640, 256), (4, 1, 513, 200), (6, 3, 96, 40),
                                           (48, 8, 1024, 512), (2, 1, 1, 1),
                                           (16, 2, 520, 200), (10, 2, 384, 384)])
def test_attention_gqa_parity(sbp, H, Hkv, T, chunk):
    hd = 128
    Q, K, V, O, dO, lse, scale = make(H, T, hd, seed=H * 100 + Hkv * 10 + T, Hkv=Hkv)
    out = sbp.attn_causal_backward(dev(Q), dev(K), dev(V), dev(O), dev(dO), dev(lse, torch.float32), scale, chunk)
    torch.cuda.synchronize()
    sbp.check_status(out["status"])
    assert out["dK"].shape == (Hkv, T, hd) and out["dV"].shape == (Hkv, T, hd)
    ref = A.backward(Q, K, V, O, dO, lse, scale)
    e = {"dQ": rel_fro(out["dQ"].float().cpu().numpy(), ref["dQ"]),
         "dK": rel_fro(out["dK"].cpu().numpy(), ref["dK"]),
         "dV": rel_fro(out["dV"].cpu().numpy(), ref["dV"])}
    assert max(e.values()) <= 2e-2, e


def test_attention_gqa_needs_hd128(sbp):
    Q, K, V, O, dO, lse, scale = make(4, 64, 64, seed=3, Hkv=2)
    with pytest.raises(sbp.SbpError):
        sbp.attn_causal_backward(dev(Q), dev(K), dev(V), dev(O), dev(dO), dev(lse, torch.float32), scale, 32)


@pytest.mark.parametrize("hd", [64, 128])
def test_attention_accumulate_and_determinism(sbp, hd):
    H, T, chunk = 2, 300, 128
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


@pytest.mark.parametrize("Hkv", [32, 8])
def test_attention_fullsize_sampled(sbp, Hkv):
    """The benchmark's workload and launch configuration (H=32 query heads, T=8192,
    hd=128, chunk 4096; and chunk 1024 on the same inputs), with 32 key / value heads (multi-head) and with 8 (grouped, the
    Qwen3-8B layout): dQ on sampled query rows and dK, dV on sampled keys of the first and
    last key / value heads against the oracle's row and column forms (chunk starts and
    ends, the first and last token, random picks).  The O and lse of every query head in
    those heads' groups come from the oracle's forward; the other heads' from a plain
    fp32 torch forward (they only have to be valid inputs)."""
    H, T, hd = 32, 8192, 128
    g = np.random.default_rng(81920 + Hkv)
    Q, dO = (I.round_bf16(g.standard_normal((H, T, hd), dtype=np.float32)) for _ in range(2))
    K, V = (I.round_bf16(g.standard_normal((Hkv, T, hd), dtype=np.float32)) for _ in range(2))
    grp = H // Hkv
    scale = 1.0 / np.sqrt(hd)
    tq, tk, tv, tdo = dev(Q), dev(K), dev(V), dev(dO)
    O = torch.empty_like(tq)
    lse = torch.empty((H, T), dtype=torch.float32, device="cuda")
    mask = torch.ones((T, T), dtype=torch.bool, device="cuda").triu(1)
    for h in range(H):
        S = (tq[h].float() @ tk[h // grp].float().T) * scale
        S.masked_fill_(mask, float("-inf"))
        lse[h] = torch.logsumexp(S, dim=1)
        O[h] = (torch.exp(S - lse[h][:, None]) @ tv[h // grp].float()).to(torch.bfloat16)
    del S, mask
    # query heads whose rows are checked, and the key / value heads whose dK, dV are: all
    # query heads of a checked key / value head's group need oracle O and lse
    kv_heads = (0, Hkv - 1)
    heads = sorted({h for hk in kv_heads for h in range(hk * grp, (hk + 1) * grp)})
    On = O.float().cpu().numpy()
    lsen = lse.cpu().numpy()
    for h in heads:
        f = A.forward(Q[h:h + 1], K[h // grp:h // grp + 1], V[h // grp:h // grp + 1], scale)
        On[h] = I.round_bf16(f["O"][0].astype(np.float32))
        lsen[h] = f["lse"][0].astype(np.float32)
        O[h] = dev(On[h])
        lse[h] = torch.from_numpy(lsen[h]).cuda()
    edges = [0, 1, 127, 128, 255, 256, 1023, 1024, 1025, 4095, 4096, 7167, 7168, 8190, 8191]
    rows = sorted(set(edges) | set(g.integers(0, T, 20).tolist()))
    keys = sorted(set(edges) | set(g.integers(0, T, 20).tolist()))
    rq = {h: A.rows_dQ(Q, K, V, On, dO, lsen, scale, h, rows) for h in (heads[0], heads[-1])}
    rkv = {hk: A.keys_dKdV(Q, K, V, On, dO, lsen, scale, hk, keys) for hk in kv_heads}
    for chunk in (4096, 1024):
        out = sbp.attn_causal_backward(tq, tk, tv, O, tdo, lse, scale, chunk)
        torch.cuda.synchronize()
        sbp.check_status(out["status"])
        dQ = out["dQ"].float().cpu().numpy()
        dK, dV = out["dK"].cpu().numpy(), out["dV"].cpu().numpy()
        del out
        for h, r in rq.items():
            assert rel_fro(dQ[h][rows], r) <= 2e-2, (chunk, h, rel_fro(dQ[h][rows], r))
        for hk, (rk, rv) in rkv.items():
            e = {"dK": rel_fro(dK[hk][keys], rk), "dV": rel_fro(dV[hk][keys], rv)}
            assert max(e.values()) <= 2e-2, (chunk, hk, e)


def test_side_stream_under_graph_capture_and_threads(sbp):
    """The hd = 128 path runs its dQ kernels on the library's side stream, forked from the
    caller's stream and joined back into it: a call captured into a CUDA graph and
    replayed, and calls from two host threads on two streams, give the same bits as a
    plain call."""
    import threading
    H, T, hd, chunk = 4, 640, 128, 256
    Q, K, V, O, dO, lse, scale = make(H, T, hd, seed=77)
    args = [dev(Q), dev(K), dev(V), dev(O), dev(dO), dev(lse, torch.float32), scale, chunk]
    ref = sbp.attn_causal_backward(*args)
    torch.cuda.synchronize()
    # graph capture on a side stream of the caller's
    s = torch.cuda.Stream()
    ws = torch.empty(sbp.attn_workspace_bytes(H, T, hd, chunk), dtype=torch.uint8, device="cuda")
    dQ, dK, dV = torch.empty_like(ref["dQ"]), torch.empty_like(ref["dK"]), torch.empty_like(ref["dV"])
    st = torch.zeros((), dtype=torch.int32, device="cuda")
    with torch.cuda.stream(s):   # warm the library's per-device state outside the capture
        sbp.attn_causal_backward(*args, dQ=dQ, dK=dK, dV=dV, workspace=ws, status=st, stream=s)
    s.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        sbp.attn_causal_backward(*args, dQ=dQ, dK=dK, dV=dV, workspace=ws, status=st, stream=s)
    for x in (dQ, dK, dV):
        x.zero_()
    g.replay()
    torch.cuda.synchronize()
    sbp.check_status(st)
    for k, x in (("dQ", dQ), ("dK", dK), ("dV", dV)):
        assert torch.equal(x, ref[k]), k
    # two host threads, two streams, two workspaces
    outs = [None, None]

    def run(i):
        si = torch.cuda.Stream()
        with torch.cuda.stream(si):
            outs[i] = sbp.attn_causal_backward(*args, stream=si)
        si.synchronize()
    th = [threading.Thread(target=run, args=(i,)) for i in range(2)]
    for t in th:
        t.start()
    for t in th:
        t.join()
    torch.cuda.synchronize()
    for o in outs:
        sbp.check_status(o["status"])
        for k in ("dQ", "dK", "dV"):
            assert torch.equal(o[k], ref[k]), k


def test_attention_long_T32768_gqa_sampled(sbp):
    """The long-sequence workload of the attention measurements: T=32768, 32 query heads on
    8 key / value heads, hd=128, at chunks 4096 and 8192.  O and lse come from a plain fp32
    torch forward on the device (O rounded to bf16, as a forward saves it); the oracle's
    row and column forms take exactly those values, so the check is of the backward alone:
    dQ on sampled query rows of the first and last query heads, dK / dV on sampled keys of
    the first and last key / value heads (chunk edges, the first and last token, random
    picks), each against the float64 oracle."""
    H, Hkv, T, hd = 32, 8, 32768, 128
    grp = H // Hkv
    g = np.random.default_rng(327680)
    Q, dO = (I.round_bf16(g.standard_normal((H, T, hd), dtype=np.float32)) for _ in range(2))
    K, V = (I.round_bf16(g.standard_normal((Hkv, T, hd), dtype=np.float32)) for _ in range(2))
    scale = 1.0 / np.sqrt(hd)
    tq, tk, tv, tdo = dev(Q), dev(K), dev(V), dev(dO)
    O = torch.empty_like(tq)
    lse = torch.empty((H, T), dtype=torch.float32, device="cuda")
    mask = torch.ones((T, T), dtype=torch.bool, device="cuda").triu(1)
    for h in range(H):
        S = (tq[h].float() @ tk[h // grp].float().T) * scale
        S.masked_fill_(mask, float("-inf"))
        lse[h] = torch.logsumexp(S, dim=1)
        S.sub_(lse[h][:, None]).exp_()
        O[h] = (S @ tv[h // grp].float()).to(torch.bfloat16)
    del S, mask
    torch.cuda.empty_cache()
    On = O.float().cpu().numpy()
    lsen = lse.cpu().numpy()
    edges = [0, 1, 127, 128, 4095, 4096, 8191, 8192, 16383, 16384, 24576, 32766, 32767]
    rows = sorted(set(edges) | set(g.integers(0, T, 16).tolist()))
    keys = sorted(set(edges) | set(g.integers(0, T, 16).tolist()))
    # the oracle on the heads it checks only (each call takes one query head, or one key /
    # value head with its group)
    rq = {h: A.rows_dQ(Q[h:h + 1], K[h // grp:h // grp + 1], V[h // grp:h // grp + 1], On[h:h + 1],
                       dO[h:h + 1], lsen[h:h + 1], scale, 0, rows) for h in (0, H - 1)}
    rkv = {}
    for hk in (0, Hkv - 1):
        qs = slice(hk * grp, (hk + 1) * grp)
        rkv[hk] = A.keys_dKdV(Q[qs], K[hk:hk + 1], V[hk:hk + 1], On[qs], dO[qs], lsen[qs], scale, 0, keys)
    for chunk in (4096, 8192):
        out = sbp.attn_causal_backward(tq, tk, tv, O, tdo, lse, scale, chunk)
        torch.cuda.synchronize()
        sbp.check_status(out["status"])
        dQ = out["dQ"].float().cpu().numpy()
        dK, dV = out["dK"].cpu().numpy(), out["dV"].cpu().numpy()
        del out
        for h, r in rq.items():
            assert rel_fro(dQ[h][rows], r) <= 2e-2, (chunk, h, rel_fro(dQ[h][rows], r))
        for hk, (rk, rv) in rkv.items():
            e = {"dK": rel_fro(dK[hk][keys], rk), "dV": rel_fro(dV[hk][keys], rv)}
            assert max(e.values()) <= 2e-2, (chunk, hk, e)
