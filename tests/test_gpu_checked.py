"""The checked and NVTX builds on the GPU (child processes, one per build).

Checked build (``SBP_LIBRARY_VARIANT=checked``): every workspace region is followed by a
guard zone that each call fills before its first kernel and verifies after its last one.
Every entry point runs on shapes with several chunks and ragged tails (SFT in both
schedules, GRPO with its extras, both DPO passes, the host-buffer and allocation-free
calls, the MLP and both attention paths); every call must end with status OK (no kernel
wrote past its workspace region) and agree with the oracle.  The output tensors are views
into larger buffers whose padding must come back untouched (no write past an output).
Then the ``SBP_FAULT_GUARD`` knob plants a wrong word in one guard zone, standing in for
an overrun, and the call must report SBP_ERR_WORKSPACE_OVERRUN; without the knob the same
process runs a clean call again.  Nothing here faults, traps or hangs the GPU.

NVTX build: one SFT call agrees with the oracle (the ranges change nothing on the device).
"""
import json
import os
import subprocess
import sys

import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD_CHECKED = r"""
import json, os, sys
sys.path.insert(0, sys.argv[1])
import numpy as np, torch
from memory_efficient_exact_gb300 import _build
_build.build_library()
from memory_efficient_exact_gb300 import sbp, inputs as I
from oracle import lmhead as O, attention as OA, mlp as OM
assert sbp.LIB_PATH.endswith("libsbp_checked.so"), sbp.LIB_PATH
res = {}

def rel(a, b):
    return float(np.linalg.norm(np.asarray(a, np.float64) - b) / max(np.linalg.norm(b), 1e-30))

def padded(shape, dtype, pad=64):
    # an output view with `pad` guard elements after it, filled with 7
    n = int(np.prod(shape))
    buf = torch.full((n + pad,), 7.0, dtype=dtype, device="cuda")
    return buf, buf[:n].view(*shape)

def pad_ok(buf, pad=64):
    return bool(torch.all(buf[-pad:] == 7.0).item())

T, d, V, chunk = 700, 256, 3000, 128
H, W = I.make_hw(T, d, V, 31, "bf16", w_std=0.08)
y = I.make_labels(T, V, 31, "frac", 0.1)
Ht = torch.from_numpy(H).cuda().bfloat16(); Wt = torch.from_numpy(W).cuda().bfloat16(); yt = torch.from_numpy(y).cuda()
ref = O.sft(H, W, y)
bH, dH = padded((T, d), torch.bfloat16); bW, dW = padded((V, d), torch.float32)
for lean in (False, True):
    ws = sbp.make_workspace(T, d, V, chunk, sbp.BF16, sbp.MODE_SFT, lean=lean)
    o = sbp.sft(Ht, Wt, yt, chunk, dH=dH, dW=dW, workspace=ws); torch.cuda.synchronize()
    res[f"sft_lean{int(lean)}"] = [int(o["status"].item()), rel(o["dH"].float().cpu(), ref["dH"]),
                                   rel(o["dW"].cpu(), ref["dW"]), pad_ok(bH) and pad_ok(bW)]
A = I.make_advantages(T, 1, 5)[:T].astype(np.float32)
lpo = (ref["logp"] + I.make_logp_noise(T, 5)).astype(np.float32)
cu = np.array([0, 200, 450, 700], dtype=np.int32)
o = sbp.grpo_ext(Ht, Wt, yt, torch.from_numpy(A).cuda(), torch.from_numpy(lpo).cuda(), chunk,
                 ref_logp=torch.from_numpy(lpo).cuda(), kl_coef=0.2, cu_seqlens=torch.from_numpy(cu).cuda())
torch.cuda.synchronize()
g = O.grpo_ext(H, W, y, A.astype(np.float64), lpo.astype(np.float64), ref_logp=lpo.astype(np.float64), kl_coef=0.2,
               cu_seqlens=cu)
res["grpo_ext"] = [int(o["status"].item()), rel(o["dH"].float().cpu(), g["dH"]), rel(o["dW"].cpu(), g["dW"]), True]
cu4 = np.array([0, 150, 350, 500, 700], dtype=np.int32)
p1 = O.dpo_pass1(H, W, y, cu4)
rS = p1["seq_logp"] + np.array([-2.0, 1.0, 0.5, -1.0])
q1 = sbp.dpo_pass1(Ht, Wt, yt, torch.from_numpy(cu4).cuda(), chunk)
q2 = sbp.dpo_pass2(Ht, Wt, yt, torch.from_numpy(cu4).cuda(), q1["seq_logp"], torch.from_numpy(rS).cuda(), 0.5, chunk)
torch.cuda.synchronize()
r2 = O.dpo(H, W, y, cu4, rS, 0.5)
res["dpo"] = [max(int(q1["status"].item()), int(q2["status"].item())), rel(q2["dH"].float().cpu(), r2["dH"]),
              rel(q2["dW"].cpu(), r2["dW"]), True]
o = sbp.sft_host(Ht.cpu().pin_memory(), Wt, yt.cpu().pin_memory(), chunk); torch.cuda.synchronize()
res["sft_host"] = [int(o["status"].item()), rel(o["dH"].float(), ref["dH"]), rel(o["dW"].cpu(), ref["dW"]), True]
o = sbp.sft_noalloc(Ht[:300], Wt, yt[:300], 64); torch.cuda.synchronize()
r3 = O.sft(H[:300], W, y[:300])
res["sft_noalloc"] = [int(o["status"].item()), rel(o["dH"].float().cpu(), r3["dH"]), rel(o["dW"].cpu(), r3["dW"]), True]

g_ = np.random.default_rng(3)
Tm, dm, fm = 300, 256, 512
X = I.round_bf16(g_.standard_normal((Tm, dm), dtype=np.float32))
Wgu = I.round_bf16((g_.standard_normal((2 * fm, dm), dtype=np.float32) / 16).astype(np.float32))
Wd = I.round_bf16((g_.standard_normal((dm, fm), dtype=np.float32) / 22).astype(np.float32))
dY = I.round_bf16(g_.standard_normal((Tm, dm), dtype=np.float32))
bf = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda().bfloat16()
bX, dX = padded((Tm, dm), torch.bfloat16)
o = sbp.mlp_swiglu_backward(bf(X), bf(Wgu), bf(Wd), bf(dY), 128, dX=dX); torch.cuda.synchronize()
m = OM.backward(X, Wgu[:fm], Wgu[fm:], Wd, dY)
res["mlp"] = [int(o["status"].item()), rel(o["dX"].float().cpu(), m["dx"]), rel(o["dWd"].cpu(), m["dWd"]), pad_ok(bX)]

for (Hq, Hkv, Ta, hd, ch) in ((4, 2, 300, 128, 128), (2, 2, 300, 64, 128)):
    Q, dO = (I.round_bf16(g_.standard_normal((Hq, Ta, hd), dtype=np.float32)) for _ in range(2))
    K, Vv = (I.round_bf16(g_.standard_normal((Hkv, Ta, hd), dtype=np.float32)) for _ in range(2))
    sc = hd ** -0.5
    f = OA.forward(Q, K, Vv, sc)
    Oo = I.round_bf16(f["O"].astype(np.float32)); lse = f["lse"].astype(np.float32)
    bQ, dQ = padded((Hq, Ta, hd), torch.bfloat16)
    bK, dK = padded((Hkv, Ta, hd), torch.float32)
    o = sbp.attn_causal_backward(bf(Q), bf(K), bf(Vv), bf(Oo), bf(dO), torch.from_numpy(lse).cuda(), sc, ch,
                                 dQ=dQ, dK=dK)
    torch.cuda.synchronize()
    a = OA.backward(Q, K, Vv, Oo, dO, lse, sc)
    res[f"attn_hd{hd}"] = [int(o["status"].item()), rel(o["dQ"].float().cpu(), a["dQ"]), rel(o["dK"].cpu(), a["dK"]),
                           pad_ok(bQ) and pad_ok(bK)]

os.environ["SBP_FAULT_GUARD"] = "1"
o = sbp.sft(Ht, Wt, yt, chunk); torch.cuda.synchronize()
res["planted"] = int(o["status"].item())
os.environ["SBP_FAULT_GUARD"] = "0"
o = sbp.sft(Ht, Wt, yt, chunk); torch.cuda.synchronize()
res["after"] = int(o["status"].item())
print(json.dumps(res))
"""

CHILD_NVTX = r"""
import json, sys
sys.path.insert(0, sys.argv[1])
import numpy as np, torch
from memory_efficient_exact_gb300 import _build
_build.build_library()
from memory_efficient_exact_gb300 import sbp, inputs as I
from oracle import lmhead as O
assert sbp.LIB_PATH.endswith("libsbp_nvtx.so"), sbp.LIB_PATH
H, W = I.make_hw(300, 256, 2000, 7, "bf16", w_std=0.05)
y = I.make_labels(300, 2000, 7, "frac", 0.1)
o = sbp.sft(torch.from_numpy(H).cuda().bfloat16(), torch.from_numpy(W).cuda().bfloat16(), torch.from_numpy(y).cuda(), 128)
torch.cuda.synchronize()
r = O.sft(H, W, y)
e = float(np.linalg.norm(o["dW"].cpu().numpy() - r["dW"]) / np.linalg.norm(r["dW"]))
print(json.dumps({"status": int(o["status"].item()), "dW": e, "loss": abs(o["loss"].item() - r["loss"]) / abs(r["loss"])}))
"""


def _run(code, variant):
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    env = dict(os.environ, SBP_LIBRARY_VARIANT=variant, SBP_WAIT_LIMIT_MS="2000")
    env.pop("SBP_FAULT_GUARD", None)
    r = subprocess.run([sys.executable, "-c", code, ROOT], capture_output=True, text=True, env=env, timeout=600)
    assert r.returncode == 0, r.stderr[-3000:]
    return json.loads(r.stdout.strip().splitlines()[-1])


def test_checked_build_guard_zones_and_output_padding():
    res = _run(CHILD_CHECKED, "checked")
    for name, (status, e1, e2, pads) in ((k, v) for k, v in res.items() if isinstance(v, list)):
        assert status == 0, (name, status)
        assert e1 <= 2e-2 and e2 <= 2e-2, (name, e1, e2)
        assert pads, name
    assert res["planted"] == 9          # SBP_ERR_WORKSPACE_OVERRUN
    assert res["after"] == 0


def test_nvtx_build():
    res = _run(CHILD_NVTX, "nvtx")
    assert res["status"] == 0 and res["dW"] <= 2e-2 and res["loss"] <= 1e-3
