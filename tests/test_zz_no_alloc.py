"""The allocation-free SFT entry point, ``sbp_lmhead_sft_noalloc``.

Some callers cannot allocate device memory: code running inside a host framework or
plugin that owns every allocation and hands none to extensions, runtimes with a fixed
memory budget that forbid allocating on their hot path (an allocation can also
synchronise the device), or plain C callers with no allocator at hand.  For them the
library offers this entry point: it takes no workspace and works in one fixed 64 MiB
device array of its own.  Here it is called through the C ABI twice in a row, and
each result is checked against the workspace entry point ``sbp_lmhead_sft`` on the
same inputs, within the parity tolerances of the other tests.  Sizes whose workspace
exceeds the array must be refused on the host with SBP_ERR_SCRATCH_LIMIT.
"""
import numpy as np
import pytest

from memory_efficient_exact_gb300 import inputs as I
from parity_util import TOL, rel, rel_fro, to_dev

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


@pytest.mark.parametrize("dtype,T,d,V,chunk", [("bf16", 200, 4096, 151936, 32), ("fp32", 256, 64, 1000, 64)])
def test_noalloc_matches_workspace_entry_point(sbp, dtype, T, d, V, chunk):
    assert sbp.workspace_bytes(T, d, V, chunk, sbp.BF16 if dtype == "bf16" else sbp.FP32,
                               sbp.MODE_SFT) <= sbp.NOALLOC_SCRATCH_BYTES
    H, W = I.make_hw(T, d, V, 21, dtype, w_std=0.02)
    y = I.make_labels(T, V, 21, "frac", 0.1)
    Ht, Wt, yt = to_dev(torch, H, W, y, dtype)
    ref = sbp.sft(Ht, Wt, yt, chunk)
    torch.cuda.synchronize()
    sbp.check_status(ref["status"])
    tol = TOL[dtype]
    for _ in range(2):
        out = sbp.sft_noalloc(Ht, Wt, yt, chunk)
        torch.cuda.synchronize()
        sbp.check_status(out["status"])
        assert int(out["n_valid"].item()) == int(ref["n_valid"].item())
        assert rel(out["loss"].item(), ref["loss"].item()) <= tol["loss"]
        assert rel_fro(out["dH"].float().cpu().numpy(), ref["dH"].float().cpu().numpy()) <= tol["grad"]
        assert rel_fro(out["dW"].cpu().numpy(), ref["dW"].cpu().numpy()) <= tol["grad"]
        lp, lr = out["logp"].cpu().numpy(), ref["logp"].cpu().numpy()
        assert np.max(np.abs(lp - lr)) <= tol["logp"] * max(1.0, np.abs(lr).max())


def test_noalloc_refuses_sizes_beyond_its_scratch(sbp):
    T, d, V, chunk = 4096, 4096, 151936, 2048
    assert sbp.workspace_bytes(T, d, V, chunk, sbp.BF16, sbp.MODE_SFT) > sbp.NOALLOC_SCRATCH_BYTES
    H = torch.zeros((T, d), dtype=torch.bfloat16, device="cuda")
    W = torch.zeros((V, d), dtype=torch.bfloat16, device="cuda")
    y = torch.zeros((T,), dtype=torch.int32, device="cuda")
    with pytest.raises(sbp.SbpError) as e:
        sbp.sft_noalloc(H, W, y, chunk)
    assert e.value.code == sbp.ERR_SCRATCH_LIMIT
