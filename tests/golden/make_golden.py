"""Writes the regression fixtures of this folder from the float64 oracle.

The pages print no worked example (no small case with its numbers), so none of these
fixtures holds a value of the pages.  Each holds tiny seeded inputs and the oracle's
outputs on them, written by this script and by nothing else; ``tests/test_golden.py``
recomputes the outputs from the stored inputs and compares.  A later change to the
oracle's arithmetic therefore fails that test until the fixture is rewritten here, in
a commit that names the passage (or the reading of it) that justifies the change.

Every fixture names the oracle function it records and the passage that function
follows.  Inputs come from ``memory_efficient_exact_gb300.inputs`` (random draws only)
and are stored in the fixture, so the comparison does not depend on the generator.

    python tests/golden/make_golden.py        # rewrites the *.json files here
"""
from __future__ import annotations

import json
import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(os.path.dirname(HERE))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from memory_efficient_exact_gb300 import inputs as I  # noqa: E402
from oracle import attention as OA  # noqa: E402
from oracle import lmhead as O  # noqa: E402
from oracle import mlp as OM  # noqa: E402

SOURCE = "written by tests/golden/make_golden.py from the float64 oracle (no page prints a worked example)"


def _lists(d: dict) -> dict:
    out = {}
    for k, v in d.items():
        if isinstance(v, np.ndarray):
            out[k] = v.tolist()
        elif isinstance(v, (np.floating, np.integer)):
            out[k] = v.item()
        else:
            out[k] = v
    return out


def lmhead_inputs(seed: int, T: int = 7, d: int = 5, V: int = 11):
    H, W = I.make_hw(T, d, V, seed, "fp32", w_std=0.5)
    y = I.make_labels(T, V, seed, "frac", 0.3)
    return H.astype(np.float64), W.astype(np.float64), y


def case_sft():
    H, W, y = lmhead_inputs(2001)
    r = O.sft(H, W, y)
    return dict(
        function="oracle.lmhead.sft",
        passage="SFT cross-entropy: ziziman.com article, LM-head paragraph on SFT/GRPO",
        inputs=_lists(dict(H=H, W=W, labels=y, ignore_index=O.IGNORE_INDEX)),
        outputs=_lists(dict(loss=r["loss"], n_valid=r["n_valid"], logp=r["logp"], lse=r["lse"], dH=r["dH"],
                            dW=r["dW"])))


def case_grpo():
    H, W, y = lmhead_inputs(2002)
    T = H.shape[0]
    A = I.make_advantages(T, 1, 2002)[:T]
    # old log-probs: the current ones shifted so that some ratios leave [0.8, 1.2]
    cur = O.forward(H, W, y)["logp"]
    shift = np.array([0.0, 0.5, -0.5, 0.1, -0.1, 0.3, -0.3])[:T]
    logp_old = np.where(np.asarray(y) == O.IGNORE_INDEX, 0.0, cur + shift)
    r = O.grpo(H, W, y, A, logp_old)
    return dict(
        function="oracle.lmhead.grpo",
        passage="GRPO / PPO-clip per-token objective: ziziman.com article, LM-head paragraph on SFT/GRPO",
        inputs=_lists(dict(H=H, W=W, labels=y, advantages=A, logp_old=logp_old, clip_lo=0.8, clip_hi=1.2,
                           ignore_index=O.IGNORE_INDEX)),
        outputs=_lists(dict(loss=r["loss"], n_valid=r["n_valid"], logp=r["logp"], dH=r["dH"], dW=r["dW"])))


def case_dpo():
    H, W, y = lmhead_inputs(2003, T=8)
    cu = I.cu_seqlens(4, 2)
    ref = np.array([-20.0, -21.5, -19.0, -22.0])
    r = O.dpo(H, W, y, cu, ref, 0.1)
    return dict(
        function="oracle.lmhead.dpo",
        passage="DPO, two passes (sequence sums first): ziziman.com article, DPO paragraph",
        inputs=_lists(dict(H=H, W=W, labels=y, cu_seqlens=cu, ref_seq_logp=ref, beta=0.1,
                           ignore_index=O.IGNORE_INDEX)),
        outputs=_lists(dict(loss=r["loss"], seq_logp=r["seq_logp"], margins=r["margins"], dH=r["dH"],
                            dW=r["dW"])))


def case_attention():
    g = np.random.default_rng(np.random.SeedSequence([2004, 1]))
    Hq, Hkv, T, hd = 2, 1, 5, 4
    Q, K, V, dO = (g.standard_normal(s) for s in ((Hq, T, hd), (Hkv, T, hd), (Hkv, T, hd), (Hq, T, hd)))
    scale = 0.5
    f = OA.forward(Q, K, V, scale)
    b = OA.backward(Q, K, V, f["O"], dO, f["lse"], scale)
    return dict(
        function="oracle.attention.forward / backward",
        passage="causal attention, a chunk of queries reads keys up to its own position: "
                "atlas.scime.ai summary, Approach",
        inputs=_lists(dict(Q=Q, K=K, V=V, dO=dO, scale=scale)),
        outputs=_lists(dict(O=f["O"], lse=f["lse"], dQ=b["dQ"], dK=b["dK"], dV=b["dV"])))


def case_mlp():
    g = np.random.default_rng(np.random.SeedSequence([2005, 1]))
    T, d, f = 3, 4, 6
    x, Wg, Wu, Wd, dY = (g.standard_normal(s) for s in ((T, d), (f, d), (f, d), (d, f), (T, d)))
    b = OM.backward(x, Wg, Wu, Wd, dY)
    return dict(
        function="oracle.mlp.backward",
        passage="layer-wise linear decomposition of the chain rule along the sequence: "
                "chatpaper.ai / fugumt.com abstract",
        inputs=_lists(dict(x=x, Wg=Wg, Wu=Wu, Wd=Wd, dY=dY)),
        outputs=_lists(dict(y=b["y"], dx=b["dx"], dWg=b["dWg"], dWu=b["dWu"], dWd=b["dWd"])))


CASES = {
    "lmhead_sft_T7_d5_V11.json": case_sft,
    "lmhead_grpo_T7_d5_V11.json": case_grpo,
    "lmhead_dpo_T8_d5_V11.json": case_dpo,
    "attention_gqa_H2_Hkv1_T5_hd4.json": case_attention,
    "mlp_swiglu_T3_d4_f6.json": case_mlp,
}


def main() -> None:
    for name, fn in CASES.items():
        d = fn()
        d = dict(source=SOURCE, **d)
        with open(os.path.join(HERE, name), "w") as fh:
            json.dump(d, fh, indent=1)
            fh.write("\n")
        print("wrote", name)


if __name__ == "__main__":
    main()
