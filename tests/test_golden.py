"""The oracle against its stored regression fixtures (``tests/golden/``, CPU only).

The fixtures hold tiny inputs and the oracle's outputs on them, written by
``tests/golden/make_golden.py``; the pages print no worked example to store instead.
Here the outputs are recomputed from the stored inputs and must agree to float64
rounding: a change to the oracle's arithmetic fails until the fixture is rewritten.
"""
import json
import os

import numpy as np
import pytest

from oracle import attention as OA
from oracle import lmhead as O
from oracle import mlp as OM

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
NAMES = sorted(f for f in os.listdir(GOLDEN) if f.endswith(".json"))


def recompute(fx: dict) -> dict:
    a = {k: (np.asarray(v) if isinstance(v, list) else v) for k, v in fx["inputs"].items()}
    fn = fx["function"]
    if fn == "oracle.lmhead.sft":
        return O.sft(a["H"], a["W"], a["labels"].astype(np.int32), a["ignore_index"])
    if fn == "oracle.lmhead.grpo":
        return O.grpo(a["H"], a["W"], a["labels"].astype(np.int32), a["advantages"], a["logp_old"],
                      a["ignore_index"], a["clip_lo"], a["clip_hi"])
    if fn == "oracle.lmhead.dpo":
        return O.dpo(a["H"], a["W"], a["labels"].astype(np.int32), a["cu_seqlens"], a["ref_seq_logp"], a["beta"],
                     a["ignore_index"])
    if fn == "oracle.attention.forward / backward":
        f = OA.forward(a["Q"], a["K"], a["V"], a["scale"])
        b = OA.backward(a["Q"], a["K"], a["V"], f["O"], a["dO"], f["lse"], a["scale"])
        return dict(O=f["O"], lse=f["lse"], **b)
    if fn == "oracle.mlp.backward":
        return OM.backward(a["x"], a["Wg"], a["Wu"], a["Wd"], a["dY"])
    raise KeyError(fn)


def test_every_fixture_is_listed():
    assert len(NAMES) == 5, NAMES


@pytest.mark.parametrize("name", NAMES)
def test_oracle_matches_fixture(name):
    fx = json.load(open(os.path.join(GOLDEN, name)))
    assert fx["source"].startswith("written by tests/golden/make_golden.py")
    assert fx["passage"]
    got = recompute(fx)
    for k, want in fx["outputs"].items():
        g = np.asarray(got[k], dtype=np.float64)
        w = np.asarray(want, dtype=np.float64)
        assert g.shape == w.shape, (k, g.shape, w.shape)
        if k == "n_valid":
            assert int(g) == int(w)
            continue
        # float64 rounding only (a different BLAS may sum in another order)
        assert np.allclose(g, w, rtol=1e-12, atol=1e-14), (name, k, float(np.max(np.abs(g - w))))
