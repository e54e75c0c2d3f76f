"""The allocation-free SFT entry point, ``sbp_lmhead_sft_noalloc``.

Some callers cannot allocate device memory: code running inside a host framework or
plugin that owns every allocation and hands none to extensions, runtimes with a fixed
memory budget that forbid allocating on their hot path (an allocation can also
synchronise the device), or plain C callers with no allocator at hand.  For them the
library offers this entry point: it takes no workspace and works in one fixed 64 MiB
device array of its own, on the one-buffer schedule.

Checked here, through the C ABI:
  * two calls in a row give the results of ``sbp_lmhead_sft`` with a one-buffer
    workspace on the same inputs, bit for bit (the same kernels on the same rows; the
    second call also shows that nothing left in the shared array by the first leaks
    into the next result);
  * the second call changes neither torch's allocation count nor the device's free
    memory (it allocates nothing);
  * at a shape the oracle finishes at once, the result agrees with the float64 oracle
    within the parity tolerances of the other tests;
  * the largest chunk whose one-buffer workspace fits the array runs, and the next one
    up is refused on the host with SBP_ERR_SCRATCH_LIMIT.

The file is collected last, so a run that stops at the first failure has already run
every other test; it also passes alone in a fresh process.
"""
import ctypes

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


def raw_noalloc(sbp, Ht, Wt, yt, chunk, outs):
    """One call of the C entry point with every output already allocated."""
    T, d = Ht.shape
    V = Wt.shape[0]
    p = sbp._p
    code = sbp._lib.sbp_lmhead_sft_noalloc(
        p(Ht), p(Wt), p(yt), T, d, V, chunk, IGN, sbp._code(Ht), p(outs["loss"]), p(outs["n_valid"]),
        p(outs["logp"]), p(outs["dH"]), p(outs["dW"]), 0, p(outs["status"]),
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    return code


def alloc_outs(Ht, Wt):
    T = Ht.shape[0]
    return dict(loss=torch.empty((), dtype=torch.float32, device="cuda"),
                n_valid=torch.empty((), dtype=torch.int64, device="cuda"),
                logp=torch.empty(T, dtype=torch.float32, device="cuda"),
                dH=torch.empty_like(Ht), dW=torch.empty(Wt.shape, dtype=torch.float32, device="cuda"),
                status=torch.empty((), dtype=torch.int32, device="cuda"))


def assert_same(out, ref):
    for k in ("loss", "n_valid", "logp", "dH", "dW"):
        assert torch.equal(out[k], ref[k]), k


@pytest.mark.parametrize("dtype,T,d,V,chunk", [("bf16", 300, 4096, 151936, 64), ("bf16", 517, 192, 1304, 200),
                                                ("fp32", 256, 64, 1000, 64)])
def test_noalloc_same_bits_as_lean_workspace_call(sbp, dtype, T, d, V, chunk):
    dt = sbp.BF16 if dtype == "bf16" else sbp.FP32
    assert sbp.workspace_bytes_lean(T, d, V, chunk, dt, sbp.MODE_SFT) <= sbp.NOALLOC_SCRATCH_BYTES
    H, W = I.make_hw(T, d, V, 21, dtype, w_std=0.02)
    y = I.make_labels(T, V, 21, "frac", 0.1)
    Ht, Wt, yt = to_dev(torch, H, W, y, dtype)
    ws = sbp.make_workspace(T, d, V, chunk, dt, sbp.MODE_SFT, lean=True)
    ref = sbp.sft(Ht, Wt, yt, chunk, workspace=ws)
    torch.cuda.synchronize()
    sbp.check_status(ref["status"])
    # first call through the binding
    out = sbp.sft_noalloc(Ht, Wt, yt, chunk)
    torch.cuda.synchronize()
    sbp.check_status(out["status"])
    assert_same(out, ref)
    # second call straight through the C ABI, outputs allocated beforehand: same bits,
    # and neither torch's allocator nor the device's free memory moves
    outs = alloc_outs(Ht, Wt)
    torch.cuda.synchronize()
    a0, f0 = torch.cuda.memory_allocated(), torch.cuda.mem_get_info()[0]
    assert raw_noalloc(sbp, Ht, Wt, yt, chunk, outs) == sbp.OK
    torch.cuda.synchronize()
    a1, f1 = torch.cuda.memory_allocated(), torch.cuda.mem_get_info()[0]
    sbp.check_status(outs["status"])
    assert a1 == a0 and f1 == f0, (a0, a1, f0, f1)
    assert_same(outs, ref)


def test_noalloc_against_oracle(sbp):
    T, d, V, chunk = 256, 64, 1000, 64
    H, W = I.make_hw(T, d, V, 1000, "fp32")
    y = I.make_labels(T, V, 1000, "frac", 0.1)
    Ht, Wt, yt = to_dev(torch, H, W, y, "fp32")
    out = sbp.sft_noalloc(Ht, Wt, yt, chunk)
    torch.cuda.synchronize()
    sbp.check_status(out["status"])
    ref = O.sft(H, W, y, IGN)
    tol = TOL["fp32"]
    assert int(out["n_valid"].item()) == ref["n_valid"]
    assert rel(out["loss"].item(), ref["loss"]) <= tol["loss"]
    dH = out["dH"].cpu().numpy()
    assert rel_fro(dH, ref["dH"]) <= tol["grad"]
    assert rel_fro(out["dW"].cpu().numpy(), ref["dW"]) <= tol["grad"]
    assert np.all(dH[y == IGN] == 0.0)


def test_noalloc_size_boundary(sbp):
    """The largest chunk whose one-buffer workspace fits the array runs (same bits as the
    workspace call); the next chunk up is refused before anything is enqueued."""
    T, d, V = 1024, 4096, 151936
    lim = sbp.NOALLOC_SCRATCH_BYTES
    sizes = {c: sbp.workspace_bytes_lean(T, d, V, c, sbp.BF16, sbp.MODE_SFT) for c in range(1, 513)}
    fit = max(c for c, n in sizes.items() if n <= lim)
    assert fit < 512 and sizes[fit + 1] > lim
    H, W = I.make_hw(T, d, V, 23, "bf16")
    y = I.make_labels(T, V, 23, "frac", 0.1)
    Ht, Wt, yt = to_dev(torch, H, W, y, "bf16")
    ws = sbp.make_workspace(T, d, V, fit, sbp.BF16, sbp.MODE_SFT, lean=True)
    ref = sbp.sft(Ht, Wt, yt, fit, workspace=ws)
    out = sbp.sft_noalloc(Ht, Wt, yt, fit)
    torch.cuda.synchronize()
    sbp.check_status(ref["status"])
    sbp.check_status(out["status"])
    assert_same(out, ref)
    before = [t.clone() for t in (out["dH"], out["dW"])]
    with pytest.raises(sbp.SbpError) as e:
        sbp.sft_noalloc(Ht, Wt, yt, fit + 1, dH=out["dH"], dW=out["dW"])
    assert e.value.code == sbp.ERR_SCRATCH_LIMIT
    torch.cuda.synchronize()
    assert torch.equal(before[0], out["dH"]) and torch.equal(before[1], out["dW"])
