"""Failure detection on the GPU without a fault: a bounded wait that runs out.

A child process sets SBP_FAULT_STALL=1, so the forward kernel's MMA thread first waits
on a barrier nothing arrives on, and SBP_WAIT_LIMIT_MS=200.  Every role of the SM pair
must then leave through the bounded-abort path: the call's device status reads
SBP_ERR_TIMEOUT, and after the knob is switched off the same process runs a correct call
(the context stays usable).  Nothing here faults, traps or hangs the GPU.
"""
import json
import os
import subprocess
import sys

import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = r"""
import json, os, sys
sys.path.insert(0, sys.argv[1])
import numpy as np, torch
from memory_efficient_exact_gb300 import _build
_build.build_library()
from memory_efficient_exact_gb300 import sbp, inputs as I
from oracle import lmhead as O
H, W = I.make_hw(300, 256, 2000, 3, "bf16", w_std=0.05)
y = I.make_labels(300, 2000, 3, "frac", 0.1)
Ht = torch.from_numpy(H).cuda().bfloat16(); Wt = torch.from_numpy(W).cuda().bfloat16(); yt = torch.from_numpy(y).cuda()
a = sbp.sft(Ht, Wt, yt, 128); torch.cuda.synchronize()
st1 = int(a["status"].item())
os.environ["SBP_FAULT_STALL"] = "0"
b = sbp.sft(Ht, Wt, yt, 128); torch.cuda.synchronize()
st2 = int(b["status"].item())
ref = O.sft(H, W, y)
e = float(np.linalg.norm(b["dW"].cpu().numpy() - ref["dW"]) / np.linalg.norm(ref["dW"]))
print(json.dumps({"first": st1, "second": st2, "dW_err": e, "loss_err": abs(b["loss"].item() - ref["loss"]) / abs(ref["loss"])}))
"""


def test_bounded_wait_runs_out_and_context_survives():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    env = dict(os.environ, SBP_FAULT_STALL="1", SBP_WAIT_LIMIT_MS="200")
    r = subprocess.run([sys.executable, "-c", CHILD, ROOT], env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    res = json.loads(r.stdout.strip().splitlines()[-1])
    from memory_efficient_exact_gb300 import sbp
    assert res["first"] == sbp.ERR_TIMEOUT
    assert res["second"] == sbp.OK
    assert res["dW_err"] <= 2e-2 and res["loss_err"] <= 1e-3
