#!/usr/bin/env python3
"""Benchmark of the StreamBP language-model head on GB300 (one JSON line on stdout).

Workload: SFT cross-entropy forward + backward of the LM head through the C ABI
(``sbp_lmhead_sft``), bf16 operands with fp32 accumulation, T = 16384 tokens
(8 x 2048), d = 4096, V = 151936, chunk = 4096; H ~ N(0,1), W ~ N(0, 0.02^2),
labels uniform with 10% ignored -- synthetic, Qwen3-shaped.  One step = one call =
the whole hot path (label scan, 4 x [forward GEMM + statistics, combine, logit
gradient, dH/dW GEMMs, dH reduce], loss reduction) over one batch.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

N > 1 runs under torchrun, one rank per GPU; every rank processes its own batch
(weak scaling, no collective on the data path); the timing is the max over ranks.
``--impl reference`` times the float64 CPU oracle on a bounded sample of the same
workload instead (rank 0 only).

The plain invocation also measures the other workloads -- GRPO, DPO, the two chunk
sweeps and the two sublayers, each in its own process after the main line's measurement --
and folds their JSON lines under "other_workloads" (`--no-other-workloads` skips that).
Other lines (each its own JSON line when run by itself):
  --objective grpo|dpo [--chunk C]   the other objectives (8 x 2048 / 8 x 4096 tokens,
                                chunk 2048 unless given)
  --workload sft_T8192_d2560|sft_T65536_d5120 [--chunk C]   the chunk-sweep workloads
  --workload profile            a small case of the same kernels for ncu captures
  --lean                        the one-buffer workspace schedule
  --sublayer mlp [--d D --f F]  the chunked SwiGLU-MLP backward
  --sublayer attn [--heads H --kv-heads K --hd 64..256 --tokens T --chunk C]
                                the chunked causal-attention backward
  --comparator torch            the same chunked LM head in eager PyTorch (timing only)
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

WORKLOAD = dict(workload="sft_ce_lmhead_bf16_T16384_d4096_V151936_chunk4096", objective="sft", T=16384, d=4096,
                V=151936, chunk=4096, dtype="bf16", seed=1002, mask="frac", frac=0.1)
METRIC = "lm_head fwd+bwd tokens/s (SFT CE, d=4096, V=151936) and % BF16 tensor peak"
UNIT = "tokens/s"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
# A small case of the same kernels for ncu captures: the bench's chunk and d, V = 32768
# (W 268 MB, larger than L2), about 1.6 GB on the device in total; two chunks, so that the second launch of the
# backward kernel accumulates into dW as every launch but the first of a call does.
PROFILE_WORKLOAD = dict(workload="sft_ce_lmhead_bf16_T8192_d4096_V32768_chunk4096", objective="sft", T=8192,
                        d=4096, V=32768, chunk=4096, dtype="bf16", seed=1002, mask="frac", frac=0.1)
# The two chunk-sweep workloads (sizes and label masks of the named input recipes):
# T = 8192 at d = 2560 with the first 1024 tokens masked as prompt, and the long-sequence
# stress case T = 65536 at d = 5120 with 5% of the tokens ignored.
SWEEP_WORKLOADS = {
    "sft_T8192_d2560": dict(T=8192, d=2560, chunk=2048, seed=1001, mask="prefix", n=1024, frac=0.0),
    "sft_T65536_d5120": dict(T=65536, d=5120, chunk=4096, seed=1004, mask="frac", frac=0.05),
}
CPU_SAMPLE_TOKENS = 384
# DRAM bytes (read + write) of one accumulating k_bwd launch, from an ncu capture of the
# profile workload (d = 4096, chunk 4096, V = 32768: 2.160 GB read + 0.565 GB written),
# scaled to V = 151936 by the units processed (every operand but H_c grows with V).  Only
# valid for the main workload's shape and the kernel version it was captured on (dH units
# in bands of 8 row tiles).
K_BWD_TRAFFIC_BYTES = (2.160e9 + 0.565e9) * 151936 / 32768


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        try:
            d = json.load(open(path))
            out = {}
            for k in FALLBACK_PEAKS:
                v = d.get(k)
                if isinstance(v, dict):
                    v = v.get("value")
                if v is not None:
                    out[k] = float(v)
            if "bf16_tflops" in out:
                out.setdefault("bf16_tflops_sustained", out["bf16_tflops"])
                out.setdefault("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"])
                return out, "measured"
        except Exception:
            pass
    return dict(FALLBACK_PEAKS), "fallback"


# ------------------------------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi clock / throttle-reason samples every 200 ms while running."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str | None):
        self.proc = None
        self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "200"]
        if gpu_id is not None:
            cmd += ["-i", gpu_id]
        try:
            self.proc = subprocess.Popen(cmd, stdout=self.file, stderr=subprocess.DEVNULL)
        except (OSError, ValueError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.file.flush()
        rows = []
        with open(self.file.name) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.file.name)
        if not rows:
            return None
        sm = [float(r[1]) for r in rows if r[1].replace(".", "", 1).isdigit()]
        smax = [float(r[2]) for r in rows if r[2].replace(".", "", 1).isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower().startswith("active")})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": reasons, "samples": len(rows)}


def gpu_id_for(torch, dev) -> str | None:
    try:
        u = torch.cuda.get_device_properties(dev).uuid
        s = str(u)
        return s if s.startswith("GPU-") else "GPU-" + s
    except Exception:
        vis = os.environ.get("CUDA_VISIBLE_DEVICES")
        return vis.split(",")[dev] if vis else str(dev)


# ------------------------------------------------------------------------------- distributed

def dist_env():
    return int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)), int(os.environ.get("LOCAL_RANK", 0))


def aggregate(torch, dist, tokens_local: float, ms_local: float, device) -> tuple[float, float]:
    """Whole-job tokens (sum over ranks) and the step time (max over ranks)."""
    if dist is None or not dist.is_initialized():
        return tokens_local, ms_local
    t = torch.tensor([tokens_local], dtype=torch.float64, device=device)
    m = torch.tensor([ms_local], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    dist.all_reduce(m, op=dist.ReduceOp.MAX)
    return float(t.item()), float(m.item())


# ------------------------------------------------------------------------------------ inputs

def make_inputs(rank: int, T: int | None = None):
    from memory_efficient_exact_gb300 import inputs as I
    w = WORKLOAD
    T = w["T"] if T is None else T
    H, W = I.make_hw(T, w["d"], w["V"], w["seed"] + rank, w["dtype"])
    y = I.make_labels(T, w["V"], w["seed"] + rank, w["mask"], w["frac"], w.get("n", 0), w.get("seq_len", 0))
    return H, W, y


def cpu_oracle_sample(H, W, y, tokens: int):
    """Times the float64 oracle (as it stands) on the first `tokens` tokens."""
    from oracle import lmhead as O
    t0 = time.perf_counter()
    O.sft(H[:tokens], W, y[:tokens])
    return time.perf_counter() - t0


def cpu_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def blas_info() -> str:
    """The BLAS numpy (and so the oracle) uses, and its thread limit where set."""
    import numpy as np
    try:
        b = np.show_config(mode="dicts")["Build Dependencies"]["blas"]
        name = f"{b.get('name', '?')} {b.get('version', '')}".strip()
    except Exception:
        name = "unknown"
    threads = os.environ.get("OPENBLAS_NUM_THREADS") or os.environ.get("OMP_NUM_THREADS") or "default (all cores)"
    return f"{name}, threads {threads}"


# --------------------------------------------------------------------------------- reference

def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    w = WORKLOAD
    H, W, y = make_inputs(0, T=CPU_SAMPLE_TOKENS)
    cpu_oracle_sample(H, W, y, 16)  # warm-up: BLAS threads, page-in
    times = [cpu_oracle_sample(H, W, y, CPU_SAMPLE_TOKENS) for _ in range(args.steps)]
    sec = sum(times)
    value = CPU_SAMPLE_TOKENS * args.steps / sec
    sample = (f"first {CPU_SAMPLE_TOKENS} tokens of the workload per step (full V and d), "
              "numpy float64 with BLAS on all host cores")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1000 * sec / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": {k: w[k] for k in ("workload", "T", "d", "V", "chunk")},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cpu_cores(), "kind": "oracle", "sample": sample,
                         "blas": blas_info()},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# --------------------------------------------------------------------------------------- ours

# The other workloads of the input recipes and the two sublayers, each measured by its own
# bench process after the main line (the plain invocation only); their JSON lines are
# folded into the main line under "other_workloads", so that one run records them all.
OTHER_WORKLOADS = [
    ("grpo_8x2048_d4096_chunk2048", ["--objective", "grpo", "--steps", "10"]),
    ("grpo_8x2048_d4096_chunk4096", ["--objective", "grpo", "--chunk", "4096", "--steps", "10"]),
    ("dpo_8x4096_d4096_chunk2048", ["--objective", "dpo", "--steps", "5"]),
    ("dpo_8x4096_d4096_chunk4096", ["--objective", "dpo", "--chunk", "4096", "--steps", "5"]),
    ("sft_T8192_d2560_chunk512", ["--workload", "sft_T8192_d2560", "--chunk", "512", "--steps", "10"]),
    ("sft_T8192_d2560_chunk1024", ["--workload", "sft_T8192_d2560", "--chunk", "1024", "--steps", "10"]),
    ("sft_T8192_d2560_chunk2048", ["--workload", "sft_T8192_d2560", "--chunk", "2048", "--steps", "10"]),
    ("sft_T65536_d5120_chunk4096", ["--workload", "sft_T65536_d5120", "--chunk", "4096", "--steps", "3"]),
    ("attn_H32_T8192_hd128_chunk4096", ["--sublayer", "attn", "--steps", "5"]),
    ("attn_H32_Hkv8_T8192_hd128_chunk4096", ["--sublayer", "attn", "--steps", "5", "--kv-heads", "8"]),
    ("mlp_T16384_d4096_f12288_chunk4096", ["--sublayer", "mlp", "--steps", "5"]),
]
OTHER_KEYS = ("metric", "value", "unit", "ms_per_step", "steps", "dtype", "config", "roofline", "pct_bf16_peak",
              "pct_bf16_peak_executed", "peak_mem_gb", "e2e", "clocks", "gpu_launches")


def run_other_workloads(timeout_s: float = 240.0) -> dict:
    out = {}
    for name, extra in OTHER_WORKLOADS:
        cmd = [sys.executable, os.path.abspath(__file__), *extra, "--no-cpu-baseline", "--no-other-workloads"]
        try:
            r = subprocess.run(cmd, capture_output=True, text=True, timeout=timeout_s, cwd=ROOT)
            lines = [x for x in r.stdout.strip().splitlines() if x.startswith("{")]
            if r.returncode != 0 or not lines:
                out[name] = {"error": f"rc={r.returncode}: " + (r.stderr.strip().splitlines() or [""])[-1][:200]}
                continue
            d = json.loads(lines[-1])
            out[name] = {k: d[k] for k in OTHER_KEYS if k in d}
            out[name]["command"] = "python bench.py " + " ".join(extra)
        except (subprocess.TimeoutExpired, OSError, ValueError) as e:
            out[name] = {"error": f"{type(e).__name__}: {e}"[:200]}
    return out


def run_ours(args):
    import numpy as np
    import torch
    rank, world, local_rank = dist_env()
    dist = None
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl")
    dev = torch.device("cuda", local_rank if world > 1 else torch.cuda.current_device())
    torch.cuda.set_device(dev)

    from memory_efficient_exact_gb300 import _build
    _build.build_library()
    from memory_efficient_exact_gb300 import sbp

    w = WORKLOAD
    T, d, V, chunk = w["T"], w["d"], w["V"], w["chunk"]
    H, W, y = make_inputs(rank)
    Ht = torch.from_numpy(H).to(dev).to(torch.bfloat16)
    Wt = torch.from_numpy(W).to(dev).to(torch.bfloat16)
    yt = torch.from_numpy(y).to(dev)
    lean = bool(getattr(args, "lean", False))
    ws = sbp.make_workspace(T, d, V, chunk, sbp.BF16, sbp.MODE_SFT, dev, lean=lean)
    dH = torch.empty_like(Ht)
    dW = torch.empty((V, d), dtype=torch.float32, device=dev)
    st = torch.zeros((), dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream(dev)

    objective = w.get("objective", "sft")
    if objective == "grpo":
        # per-response advantages A ~ N(0, 1); old log-probs = the exact current label
        # log-probs plus N(0, 0.1^2) noise, fixed at generation: computed once here, before
        # the timed region, by one forward-only library call (the first DPO pass over a
        # single sequence returns every token's log-prob and forms no gradient)
        from memory_efficient_exact_gb300 import inputs as I
        n_resp = max(1, T // 2048)
        At = torch.from_numpy(I.make_advantages(n_resp, (T + n_resp - 1) // n_resp, w["seed"])[:T]).to(dev)
        ws = sbp.make_workspace(T, d, V, chunk, sbp.BF16, sbp.MODE_GRPO, dev, lean=lean)
        ws1 = sbp.make_workspace(T, d, V, chunk, sbp.BF16, sbp.MODE_DPO1, dev)
        one = torch.tensor([0, T], dtype=torch.int32, device=dev)
        cur = sbp.dpo_pass1(Ht, Wt, yt, one, chunk, workspace=ws1, status=st, logp=True, stream=stream)
        torch.cuda.synchronize(dev)
        sbp.check_status(st, "old log-probs")
        lpo = (cur["logp"].double() + torch.from_numpy(I.make_logp_noise(T, w["seed"])).to(dev)).float()
        del ws1, cur

        def step():
            return sbp.grpo(Ht, Wt, yt, At, lpo, chunk, dH=dH, dW=dW, workspace=ws, status=st, logp=False,
                            stream=stream)
    elif objective == "dpo":
        from memory_efficient_exact_gb300 import inputs as I
        n_seq = max(2, T // w.get("seq_len", 4096))
        cu = torch.from_numpy(I.cu_seqlens(n_seq, T // n_seq)).to(dev)
        sref = torch.from_numpy(I.make_ref_seq_logp(n_seq, w["seed"])).to(dev)
        ws = sbp.make_workspace(T, d, V, chunk, sbp.BF16, sbp.MODE_DPO2, dev, lean=lean)

        def step():
            p1 = sbp.dpo_pass1(Ht, Wt, yt, cu, chunk, workspace=ws, status=st, logp=False, stream=stream)
            return sbp.dpo_pass2(Ht, Wt, yt, cu, p1["seq_logp"], sref, 0.1, chunk, dH=dH, dW=dW, workspace=ws,
                                 status=st, stream=stream)
    else:
        def step():
            return sbp.sft(Ht, Wt, yt, chunk, dH=dH, dW=dW, workspace=ws, status=st, logp=False, stream=stream)

    torch.cuda.reset_peak_memory_stats(dev)
    for _ in range(args.warmup):
        out = step()
    torch.cuda.synchronize(dev)
    sbp.check_status(st, "warm-up")
    launches_per_call = sbp.last_launch_count()
    if objective == "dpo":
        launches_per_call *= 2   # (pass 2 and pass 1 enqueue the same number of launches)

    # ---- device-timed region: inputs resident in HBM (larger than L2: W is 1.24 GB) ----
    clocks = ClockSampler(gpu_id_for(torch, dev))
    time.sleep(0.3)
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize(dev)
    sbp.profile_read()
    sbp.profile_enable(True)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        out = step()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    sbp.profile_enable(False)
    if dist is not None:
        dist.barrier()
    clk = clocks.stop()
    prof = sbp.profile_read()
    sbp.check_status(st, "timed region")
    ms_local = e0.elapsed_time(e1)
    # torch's peak plus the library's one static device array (the scratch of the
    # allocation-free entry point), which every GPU that loads the library holds
    peak_mem = torch.cuda.max_memory_allocated(dev) + sbp.NOALLOC_SCRATCH_BYTES
    loss = float(out["loss"].item())

    tokens_all, ms = aggregate(torch, dist, float(T * args.steps), ms_local, dev)
    value = tokens_all / (ms / 1000.0)
    ms_per_step = ms / args.steps

    # ---- end to end through the C ABI with host buffers (pinned), copies inside ----
    # SFT: the host-buffer entry point, which streams H in and dH out chunk by chunk
    # beside the GEMMs; for the other objectives the same copies wrap their step
    Hh = torch.from_numpy(H).to(torch.bfloat16).pin_memory()
    yh = torch.from_numpy(y).pin_memory()
    dHh = torch.empty(Hh.shape, dtype=torch.bfloat16).pin_memory()
    lossh = torch.empty((), dtype=torch.float32).pin_memory()
    nvh = torch.empty((), dtype=torch.int64).pin_memory()
    if objective == "sft":
        nh = sbp.host_workspace_bytes(T, d, V, chunk, sbp.BF16)
        if lean:
            nh -= sbp.workspace_bytes(T, d, V, chunk, sbp.BF16, sbp.MODE_SFT) - \
                sbp.workspace_bytes_lean(T, d, V, chunk, sbp.BF16, sbp.MODE_SFT)
        hws = torch.empty(nh, dtype=torch.uint8, device=dev)
    else:
        Hd = torch.empty_like(Ht)
        yd = torch.empty_like(yt)

    def e2e_step():
        if objective == "sft":
            sbp.sft_host(Hh, Wt, yh, chunk, dH=dHh, dW=dW, loss=lossh, n_valid=nvh, workspace=hws, status=st,
                         stream=stream)
            return
        Hd.copy_(Hh, non_blocking=True)
        yd.copy_(yh, non_blocking=True)
        Ht.copy_(Hd)
        o = step()
        dHh.copy_(o["dH"], non_blocking=True)
        lossh.copy_(o["loss"], non_blocking=True)

    for _ in range(2):
        e2e_step()
    torch.cuda.synchronize(dev)
    if dist is not None:
        dist.barrier()
    e2 = torch.cuda.Event(enable_timing=True)
    e3 = torch.cuda.Event(enable_timing=True)
    e2.record(stream)
    for _ in range(args.steps):
        e2e_step()
    e3.record(stream)
    torch.cuda.synchronize(dev)
    sbp.check_status(st, "e2e region")
    e2e_tokens, e2e_ms = aggregate(torch, dist, float(T * args.steps), e2.elapsed_time(e3), dev)
    h2d = Hh.numel() * Hh.element_size() + yh.numel() * yh.element_size()
    d2h = dHh.numel() * dHh.element_size() + lossh.element_size() + (nvh.element_size() if objective == "sft" else 0)

    if rank != 0:
        if dist is not None:
            dist.destroy_process_group()
        return 0

    peaks, peak_src = load_peaks()
    n_chunks = (T + chunk - 1) // chunk
    bwd_ms, bwd_n = prof["backward_gemm"]
    fwd_ms, fwd_n = prof["forward_gemm"]
    grad_ms, grad_n = prof["logit_grad"]
    oth_ms, oth_n = prof["other"]
    # algorithmic FLOPs per launch (average over the chunks of a call): dH and dW GEMMs
    # of one chunk = 4 rows d V; the forward GEMM = 2 rows d V
    flops_bwd_launch = 4.0 * T * d * V / n_chunks
    flops_fwd_launch = 2.0 * T * d * V / n_chunks
    # (DPO launches the forward twice per chunk, once per pass: the per-launch averages
    # below divide by the launch counts, and the useful rate credits 6 d V per token)
    bwd_avg_s = bwd_ms / max(bwd_n, 1) / 1000.0
    fwd_avg_s = fwd_ms / max(fwd_n, 1) / 1000.0
    bwd_tf = flops_bwd_launch / bwd_avg_s / 1e12 if bwd_n else None
    fwd_tf = flops_fwd_launch / fwd_avg_s / 1e12 if fwd_n else None
    peak_tf = peaks["bf16_tflops_sustained"]
    useful_tf = 6.0 * d * V * value / 1e12
    gtb = 4.0 * (T / n_chunks) * V / 1e9  # logit gradient: read e (fp16) + write G (bf16), GB per launch
    grad_gbs = gtb / (grad_ms / max(grad_n, 1) / 1000.0) if grad_n else None

    cpu = None
    if world == 1 and not args.no_cpu_baseline and objective == "sft":
        Ts = CPU_SAMPLE_TOKENS
        sec = cpu_oracle_sample(H, W, y, Ts)
        cpu = {"value": Ts / sec, "unit": UNIT, "cores": cpu_cores(), "kind": "oracle",
               "sample": f"first {Ts} of the {T} tokens (full V={V}, d={d}), float64 numpy/BLAS, one run",
               "blas": blas_info()}

    metric = METRIC if (objective, d, V) == ("sft", 4096, 151936) else \
        f"lm_head fwd+bwd tokens/s ({objective}, d={d}, V={V})"
    line = {
        "metric": metric, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": w["workload"], "objective": objective, "T": T, "d": d, "V": V, "chunk": chunk,
                   "schedule": "one chunk buffer" if lean else "two chunk buffers",
                   "tokens_per_gpu_per_step": T, "ignored_frac": float(np.mean(y == -100)),
                   "l2": f"inputs larger than L2 (W {V * d * 2 / 1e9:.2f} GB; chunk logits "
                         f"{chunk * V * 2 / 1e9:.2f} GB per chunk)",
                   "parallelism": f"dp{world} replicas (no collective)"},
        "roofline": {"kernel": "k_bwd (dH and dW GEMMs of one chunk)", "bound": "tensor",
                     "achieved": bwd_tf, "peak": peak_tf, "unit": "TFLOP/s",
                     "frac": (bwd_tf / peak_tf) if bwd_tf else None,
                     "traffic": K_BWD_TRAFFIC_BYTES if (d, V, chunk) == (4096, 151936, 4096) and
                     objective == "sft" else None,
                     "peak_source": f"bf16 dense, sustained, {peak_src}",
                     "algorithmic_flops_per_launch": flops_bwd_launch, "launches": bwd_n,
                     "avg_launch_ms": bwd_avg_s * 1e3},
        "kernels": {
            "k_fwd": {"achieved_tflops": fwd_tf, "avg_launch_ms": fwd_avg_s * 1e3, "launches": fwd_n,
                      "share": fwd_ms / ms_local if ms_local else None},
            "k_bwd": {"achieved_tflops": bwd_tf, "avg_launch_ms": bwd_avg_s * 1e3, "launches": bwd_n,
                      "share": bwd_ms / ms_local if ms_local else None},
            "k_grad": {"achieved_gbs": grad_gbs, "avg_launch_ms": grad_ms / max(grad_n, 1),
                       "launches": grad_n, "share": grad_ms / ms_local if ms_local else None},
            "other": {"ms": oth_ms, "launches": oth_n, "share": oth_ms / ms_local if ms_local else None},
        },
        "step_tflops_useful": useful_tf / world,
        "pct_bf16_peak": 100.0 * useful_tf / world / peaks["bf16_tflops"],
        "pct_bf16_peak_sustained": 100.0 * useful_tf / world / peaks["bf16_tflops_sustained"],
        "peak_source": peak_src,
        "peak_mem_gb": peak_mem / 1e9,
        "unchunked_fp32_logits_gb": T * V * 4 / 1e9,
        "e2e": {"value": e2e_tokens / (e2e_ms / 1000.0), "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h,
                "call": ("sbp_lmhead_sft_host (H in and dH out per chunk, beside the GEMMs)" if objective == "sft"
                         else "H2D copy, device call, D2H copy")},
        "gpu_launches": launches_per_call * args.steps,
        "clocks": clk,
        "loss": loss,
        "cpu_baseline": cpu,
    }
    if getattr(args, "other_workloads", False) and world == 1:
        # the other lines run in their own processes (this one keeps under 7 GB meanwhile)
        torch.cuda.empty_cache()
        line["other_workloads"] = run_other_workloads()
    print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()
    return 0


# ------------------------------------------------------------------------ MLP sublayer

MLP_WORKLOAD = dict(workload="swiglu_mlp_bwd_bf16_T16384_d4096_f12288_chunk4096", T=16384, d=4096, f=12288,
                    chunk=4096, seed=1005)
MLP_METRIC = "mlp sublayer bwd tokens/s (SwiGLU, d=4096, f=12288) and % BF16 tensor peak"


def make_mlp_inputs(T, d, f, seed):
    from memory_efficient_exact_gb300 import inputs as I
    import numpy as np
    g = np.random.default_rng(np.random.SeedSequence([seed, 11]))
    X = I.round_bf16(g.standard_normal((T, d), dtype=np.float32))
    Wgu = I.round_bf16(g.standard_normal((2 * f, d), dtype=np.float32) * np.float32(d ** -0.5))
    Wd = I.round_bf16(g.standard_normal((d, f), dtype=np.float32) * np.float32(f ** -0.5))
    dY = I.round_bf16(g.standard_normal((T, d), dtype=np.float32))
    return X, Wgu, Wd, dY


def run_mlp_bench(args):
    import torch
    from memory_efficient_exact_gb300 import _build
    _build.build_library()
    from memory_efficient_exact_gb300 import sbp
    w = dict(MLP_WORKLOAD)
    if args.chunk:
        w["chunk"] = args.chunk
    if args.tokens:
        w["T"] = args.tokens
    if args.d:
        w["d"] = args.d
    if args.f:
        w["f"] = args.f
    T, d, f, chunk = w["T"], w["d"], w["f"], w["chunk"]
    w["workload"] = f"swiglu_mlp_bwd_bf16_T{T}_d{d}_f{f}_chunk{chunk}"
    dev = torch.device("cuda", torch.cuda.current_device())
    X, Wgu, Wd, dY = make_mlp_inputs(T, d, f, w["seed"])
    bf = lambda a: torch.from_numpy(a).to(dev).to(torch.bfloat16)
    Xt, Wgut, Wdt, dYt = bf(X), bf(Wgu), bf(Wd), bf(dY)
    ws = torch.empty(sbp.mlp_workspace_bytes(T, d, f, chunk), dtype=torch.uint8, device=dev)
    dX = torch.empty_like(Xt)
    dWgu = torch.empty((2 * f, d), dtype=torch.float32, device=dev)
    dWd = torch.empty((d, f), dtype=torch.float32, device=dev)
    st = torch.zeros((), dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step():
        return sbp.mlp_swiglu_backward(Xt, Wgut, Wdt, dYt, chunk, dX=dX, dWgu=dWgu, dWd=dWd, workspace=ws,
                                       status=st, stream=stream)
    torch.cuda.reset_peak_memory_stats(dev)
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    sbp.check_status(st, "warm-up")
    launches = sbp.last_launch_count()
    clocks = ClockSampler(gpu_id_for(torch, dev))
    time.sleep(0.3)
    sbp.profile_read()
    sbp.profile_enable(True)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        step()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    sbp.profile_enable(False)
    clk = clocks.stop()
    prof = sbp.profile_read()
    sbp.check_status(st, "timed region")
    ms = e0.elapsed_time(e1)
    value = T * args.steps / (ms / 1000.0)
    peaks, src = load_peaks()
    n_chunks = (T + chunk - 1) // chunk
    up_ms, up_n = prof["forward_gemm"]      # recompute of g, u and the da GEMM (2 launches per chunk)
    bw_ms, bw_n = prof["backward_gemm"]     # dX + [dWg; dWu] and dWd (2 launches per chunk)
    executed = 16.0 * d * f                  # per token: recompute 4, da 2, dX 4, dWgu 4, dWd 2 (x d f)
    bw_tf = 10.0 * d * f * T * args.steps / (bw_ms / 1000.0) / 1e12 if bw_n else None
    gemm_ms = ms - prof["other"][0]
    gemm_tf = executed * T * args.steps / (gemm_ms / 1000.0) / 1e12
    fw_tf = 6.0 * d * f * T * args.steps / (up_ms / 1000.0) / 1e12 if up_n else None
    cpu = None
    if not args.no_cpu_baseline:
        from oracle import mlp as OM
        Ts = 128
        t0 = time.perf_counter()
        OM.backward(X[:Ts], Wgu[:f], Wgu[f:], Wd, dY[:Ts])
        sec = time.perf_counter() - t0
        cpu = {"value": Ts / sec, "unit": UNIT, "cores": cpu_cores(), "kind": "oracle",
               "sample": f"first {Ts} tokens (full d={d}, f={f}), float64 numpy/BLAS, one run"}
    line = {
        "metric": MLP_METRIC if (d, f) == (4096, 12288) else f"mlp sublayer bwd tokens/s (SwiGLU, d={d}, f={f})",
        "value": value, "unit": UNIT, "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": ms / args.steps, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16", "data": "synthetic",
        "config": {"workload": w["workload"], "T": T, "d": d, "f": f, "chunk": chunk},
        # the dWd GEMM runs on the library's second stream beside the chunk's k_mlp and k_bwd
        # launches, so their event durations overlap: the GEMM kernels are timed together, as
        # the step's time less the small kernels that run alone
        "roofline": {"kernel": "k_mlp x2 + k_bwd x2 per chunk (concurrent on two streams, timed together)",
                     "bound": "tensor", "achieved": gemm_tf, "peak": peaks["bf16_tflops_sustained"],
                     "unit": "TFLOP/s", "frac": gemm_tf / peaks["bf16_tflops_sustained"], "traffic": None,
                     "peak_source": f"bf16 dense, sustained, {src}",
                     "flops_per_token": executed, "gemm_ms_per_step": gemm_ms / args.steps},
        "kernels": {"k_mlp (recompute + da)": {"achieved_tflops": fw_tf, "ms": up_ms, "launches": up_n},
                    "k_bwd": {"achieved_tflops": bw_tf, "ms": bw_ms, "launches": bw_n},
                    "other": {"ms": prof["other"][0], "launches": prof["other"][1]},
                    "note": "per-kernel event durations include the overlap with the second stream"},
        "executed_tflops": executed * value / 1e12,
        "pct_bf16_peak_executed": 100.0 * executed * value / 1e12 / peaks["bf16_tflops"],
        "pct_bf16_peak_credited_12dF": 100.0 * 12.0 * d * f * value / 1e12 / peaks["bf16_tflops"],
        "peak_source": src, "peak_mem_gb": (torch.cuda.max_memory_allocated(dev) + sbp.NOALLOC_SCRATCH_BYTES) / 1e9,
        "unchunked_activations_gb": 3 * T * f * 2 / 1e9,
        "gpu_launches": launches * args.steps, "clocks": clk, "cpu_baseline": cpu,
    }
    print(json.dumps(line), flush=True)
    return 0


# ------------------------------------------------------------------- causal attention

# chunk 4096: on the fused path (hd 128) the chunk changes no memory, and larger chunks
# run faster (3.66M / 3.80M / 4.04M tokens/s at chunks 1024 / 2048 / 4096, 32 heads)
ATTN_WORKLOAD = dict(H=32, T=8192, hd=128, chunk=4096, seed=1006)
ATTN_METRIC = "attention bwd tokens/s (causal, H=32, hd=128, T=8192)"


def attn_pairs(T: int, chunk: int):
    """(causal, rectangles): the (query, key) pairs of one head that the method's GEMMs
    cover, q >= k, T (T + 1) / 2 of them whatever the chunk; and the pairs of the chunk
    rectangles (each chunk's queries x every key up to the chunk's end, the diagonal
    blocks' masked half included), what the chunk-buffer path computes and stores."""
    rect = sum(min(chunk, T - c0) * min(T, c0 + chunk) for c0 in range(0, T, chunk))
    return T * (T + 1) // 2, rect


def attn_forward_inputs(torch, Q, K, V, scale):
    """O and the row log-sum-exp of the causal forward, head by head in fp32 (input set-up
    with plain torch ops, outside the timed region); K, V may have H / group heads."""
    H, T, hd = Q.shape
    grp = H // K.shape[0]
    O = torch.empty_like(Q)
    lse = torch.empty((H, T), dtype=torch.float32, device=Q.device)
    mask = torch.ones((T, T), dtype=torch.bool, device=Q.device).triu(1)
    for h in range(H):
        S = (Q[h].float() @ K[h // grp].float().T) * scale
        S.masked_fill_(mask, float("-inf"))
        l = torch.logsumexp(S, dim=1)
        lse[h] = l
        O[h] = (torch.exp(S - l[:, None]) @ V[h // grp].float()).to(Q.dtype)
    return O, lse


def run_attn_bench(args):
    import numpy as np
    import torch
    from memory_efficient_exact_gb300 import _build
    _build.build_library()
    from memory_efficient_exact_gb300 import sbp
    w = dict(ATTN_WORKLOAD)
    if args.chunk:
        w["chunk"] = args.chunk
    if args.tokens:
        w["T"] = args.tokens
    if args.heads:
        w["H"] = args.heads
    if args.hd:
        w["hd"] = args.hd
    H, T, hd, chunk = w["H"], w["T"], w["hd"], w["chunk"]
    Hkv = args.kv_heads or H
    dev = torch.device("cuda", torch.cuda.current_device())
    g = torch.Generator(device=dev).manual_seed(w["seed"])
    Q, dO = (torch.randn((H, T, hd), device=dev, generator=g).to(torch.bfloat16) for _ in range(2))
    K, V = (torch.randn((Hkv, T, hd), device=dev, generator=g).to(torch.bfloat16) for _ in range(2))
    scale = hd ** -0.5
    O, lse = attn_forward_inputs(torch, Q, K, V, scale)
    ws = torch.empty(sbp.attn_workspace_bytes(H, T, hd, chunk), dtype=torch.uint8, device=dev)
    dQ = torch.empty_like(Q)
    dK = torch.empty((Hkv, T, hd), dtype=torch.float32, device=dev)
    dV = torch.empty((Hkv, T, hd), dtype=torch.float32, device=dev)
    st = torch.zeros((), dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step():
        return sbp.attn_causal_backward(Q, K, V, O, dO, lse, scale, chunk, dQ=dQ, dK=dK, dV=dV, workspace=ws,
                                        status=st, stream=stream)
    torch.cuda.reset_peak_memory_stats(dev)
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    sbp.check_status(st, "warm-up")
    launches = sbp.last_launch_count()
    clocks = ClockSampler(gpu_id_for(torch, dev))
    time.sleep(0.3)
    sbp.profile_read()
    sbp.profile_enable(True)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        step()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    sbp.profile_enable(False)
    clk = clocks.stop()
    prof = sbp.profile_read()
    sbp.check_status(st, "timed region")
    ms = e0.elapsed_time(e1)
    value = T * args.steps / (ms / 1000.0)
    peaks, src = load_peaks()
    # algorithmic FLOPs: five GEMMs (S, dP, dQ, dK, dV) of 2 hd per causal (query, key)
    # pair; the chunk rectangles are what the chunk-buffer path computes and stores
    causal, rowkeys = attn_pairs(T, chunk)
    flops = 5 * 2 * hd * H * causal
    fused = hd == 128   # P and dS stay on chip (k_attn_kv, k_attn_q); else chunk buffers in HBM
    # chunk buffers: P and dS written once and read twice each (2 bytes an element)
    pds_bytes = 0 if fused else 12 * H * rowkeys
    sp_ms, sp_n = prof["forward_gemm"]
    bw_ms, bw_n = prof["backward_gemm"]
    if fused:   # k_attn_kv forms S, dP and accumulates dV, dK; k_attn_q forms S, dP and accumulates dQ
        names, gemms = ("k_attn_kv (S, dP, dV, dK)", "k_attn_q (S, dP, dQ)"), (4, 3)
    else:
        names, gemms = ("k_attn (P, dS)", "k_bwd (dQ + dK, dV)"), (2, 3)
    if fused:
        # k_attn_q runs on the library's second stream beside the next chunk's k_attn_kv, so
        # their event durations overlap: the pair is timed together, as the step's time less
        # the small kernels that run alone; algorithmic FLOPs = the five GEMMs of the method
        # (the pair executes seven: S and dP are formed in both kernels), causal pairs only
        pair_ms = ms - prof["other"][0]
        pair_tf = flops * args.steps / (pair_ms / 1000.0) / 1e12
        roof = {"kernel": "k_attn_kv + k_attn_q (concurrent on two streams, timed together)", "bound": "tensor",
                "achieved": pair_tf, "peak": peaks["bf16_tflops_sustained"], "unit": "TFLOP/s", "traffic": None,
                "peak_source": f"bf16 dense, sustained, {src}",
                "flops": "5 GEMMs x 2 hd per causal (q >= k) pair", "tflops_7_gemms": pair_tf * 7 / 5,
                "pair_ms_per_step": pair_ms / args.steps}
    else:
        # the dominant kernel of the path against the tensor roofline (its own GEMMs over
        # the causal pairs)
        roof = {"kernel": names[0] if sp_ms >= bw_ms else names[1], "bound": "tensor",
                "achieved": (2 * gemms[0] * hd * H * causal * args.steps / (sp_ms / 1000.0) / 1e12
                             if sp_ms >= bw_ms else
                             2 * gemms[1] * hd * H * causal * args.steps / (bw_ms / 1000.0) / 1e12)
                if (sp_n and bw_n) else None, "flops": "the kernel's GEMMs x 2 hd per causal (q >= k) pair",
                "peak": peaks["bf16_tflops_sustained"], "unit": "TFLOP/s", "traffic": None,
                "peak_source": f"bf16 dense, sustained, {src}"}
    line = {
        "metric": ATTN_METRIC if (H, Hkv, T, hd) == (32, 32, 8192, 128) else
        f"attention bwd tokens/s (causal, H={H}, Hkv={Hkv}, hd={hd}, T={T})",
        "value": value, "unit": UNIT, "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": f"causal_attn_bwd_bf16_H{H}" + (f"_Hkv{Hkv}" if Hkv != H else "") +
                   f"_T{T}_hd{hd}_chunk{chunk}", "H": H, "Hkv": Hkv, "T": T, "hd": hd, "chunk": chunk},
        "tflops": flops * args.steps / (ms / 1000.0) / 1e12,
        "pct_bf16_peak": 100.0 * flops * args.steps / (ms / 1000.0) / 1e12 / peaks["bf16_tflops"],
        "flops": "5 GEMMs x 2 hd per causal (q >= k) pair",
        "tflops_chunk_rectangles": 5 * 2 * hd * H * rowkeys * args.steps / (ms / 1000.0) / 1e12,
        "chunk_buffer_gbs": pds_bytes * args.steps / (ms / 1000.0) / 1e9 if pds_bytes else None,
        "roofline": roof,
        "kernels": {names[0]: {"ms": sp_ms, "launches": sp_n,
                               "tflops": 2 * gemms[0] * hd * H * causal * args.steps / (sp_ms / 1000.0) / 1e12
                               if sp_n else None},
                    names[1]: {"ms": bw_ms, "launches": bw_n,
                               "tflops": 2 * gemms[1] * hd * H * causal * args.steps / (bw_ms / 1000.0) / 1e12
                               if bw_n else None},
                    "other": {"ms": prof["other"][0], "launches": prof["other"][1]}},
        "peak_source": src, "peak_mem_gb": (torch.cuda.max_memory_allocated(dev) + sbp.NOALLOC_SCRATCH_BYTES) / 1e9,
        "unchunked_scores_gb": H * T * T * 2 * 2 / 1e9,
        "gpu_launches": launches * args.steps, "clocks": clk,
    }
    rf = line["roofline"]
    rf["frac"] = rf["achieved"] / rf["peak"] if rf["achieved"] else None
    if fused:
        line["kernels"]["note"] = "per-kernel event durations include the overlap with the second stream"
    print(json.dumps(line), flush=True)
    return 0


# ------------------------------------------------------- timing comparator (opt-in only)

def run_torch_comparator(args):
    """The same chunked SFT LM head written as plain eager PyTorch (cuBLAS bf16 GEMMs,
    fp32 softmax), timed on the same workload: what the hand-written kernels buy over an
    idiomatic implementation of the method.  A timing comparison only: nothing of the
    library's path runs here, and nothing of this runs in the library."""
    import torch
    w = WORKLOAD
    T, d, V, chunk = w["T"], w["d"], w["V"], w["chunk"]
    dev = torch.device("cuda", torch.cuda.current_device())
    H, W, y = make_inputs(0)
    Ht = torch.from_numpy(H).to(dev).to(torch.bfloat16)
    Wt = torch.from_numpy(W).to(dev).to(torch.bfloat16)
    yt = torch.from_numpy(y).to(dev).long()
    dH = torch.empty_like(Ht)
    dW = torch.empty((V, d), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step():
        valid_all = yt != -100
        n = valid_all.sum().clamp_min(1).float()
        dW.zero_()
        loss = torch.zeros((), dtype=torch.float32, device=dev)
        for c0 in range(0, T, chunk):
            h, yc, vc = Ht[c0:c0 + chunk], yt[c0:c0 + chunk], valid_all[c0:c0 + chunk]
            z = (h @ Wt.T).float()
            lse = torch.logsumexp(z, dim=1)
            logp = z.gather(1, yc.clamp_min(0)[:, None])[:, 0] - lse
            loss -= (logp * vc).sum() / n
            g = torch.exp(z - lse[:, None])
            g[torch.arange(g.shape[0], device=dev), yc.clamp_min(0)] -= 1.0
            g *= (vc.float() / n)[:, None]
            gb = g.to(torch.bfloat16)
            dH[c0:c0 + chunk] = gb @ Wt
            dW.add_((gb.T @ h).float())
        return loss

    torch.cuda.reset_peak_memory_stats(dev)
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(gpu_id_for(torch, dev))
    time.sleep(0.3)
    e0.record(stream)
    for _ in range(args.steps):
        step()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    clk = clocks.stop()
    ms = e0.elapsed_time(e1)
    peaks, src = load_peaks()
    value = T * args.steps / (ms / 1000.0)
    line = {
        "comparator": "eager PyTorch (cuBLAS bf16 GEMMs, fp32 softmax), same chunking",
        "metric": METRIC if (d, V) == (4096, 151936) else f"lm_head fwd+bwd tokens/s (sft, d={d}, V={V})",
        "value": value, "unit": UNIT, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms / args.steps,
        "pct_bf16_peak": 100.0 * 6.0 * d * V * value / 1e12 / peaks["bf16_tflops"], "peak_source": src,
        "config": {k: w[k] for k in ("workload", "T", "d", "V", "chunk")},
        "peak_mem_gb": torch.cuda.max_memory_allocated(dev) / 1e9, "clocks": clk,
    }
    print(json.dumps(line), flush=True)
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-other-workloads", action="store_true",
                    help="plain invocation: skip the other workloads' lines folded into the main line")
    ap.add_argument("--comparator", choices=["torch"], default=None,
                    help="time the same chunked LM head in eager PyTorch instead (a comparison line only)")
    ap.add_argument("--workload", choices=["main", "profile"] + sorted(SWEEP_WORKLOADS), default="main",
                    help="profile: a small case of the same kernels for ncu captures; "
                         "sft_T8192_d2560 / sft_T65536_d5120: the chunk-sweep workloads (with --chunk)")
    ap.add_argument("--chunk", type=int, default=None, help="override the chunk size (sweeps)")
    ap.add_argument("--tokens", type=int, default=None, help="override T (sweeps)")
    ap.add_argument("--hd", type=int, default=None, help="override the attention head width (--sublayer attn)")
    ap.add_argument("--kv-heads", type=int, default=None,
                    help="--sublayer attn: key / value heads (grouped-query attention; default = query heads)")
    ap.add_argument("--lean", action="store_true",
                    help="LM head: the smallest workspace (one chunk buffer, gradient as its own pass)")
    ap.add_argument("--d", type=int, default=None, help="override the hidden size (sweeps; --sublayer mlp too)")
    ap.add_argument("--f", type=int, default=None, help="--sublayer mlp: the intermediate size")
    ap.add_argument("--heads", type=int, default=None, help="--sublayer attn: query heads")
    ap.add_argument("--sublayer", choices=["lmhead", "mlp", "attn"], default="lmhead",
                    help="mlp / attn: the chunked SwiGLU-MLP or causal-attention backward (own JSON line)")
    ap.add_argument("--objective", choices=["sft", "grpo", "dpo"], default="sft",
                    help="grpo: 8 responses of 2048 tokens; dpo: 8 sequences of 4096 tokens, both passes per "
                         "step; chunk 2048 for both unless --chunk is given")
    args = ap.parse_args(argv)
    if args.workload == "profile":
        WORKLOAD.clear()
        WORKLOAD.update(PROFILE_WORKLOAD)
        args.no_cpu_baseline = True
    if args.workload in SWEEP_WORKLOADS:
        WORKLOAD.update(SWEEP_WORKLOADS[args.workload])
        WORKLOAD["workload"] = "x"   # renamed below from the final sizes
        if args.chunk is None:
            args.chunk = WORKLOAD["chunk"]
    WORKLOAD["objective"] = args.objective
    if args.objective == "dpo" and args.workload == "main":
        # the DPO input recipe: 8 sequences of 4096 tokens, the first 1024 of each masked
        WORKLOAD.update(T=32768, seed=1003, mask="seqhead", n=1024, seq_len=4096, frac=0.0)
    if args.objective != "sft" and args.workload == "main":
        WORKLOAD["chunk"] = 2048   # the GRPO and DPO workloads' own chunk
    for key, val in (("chunk", args.chunk), ("T", args.tokens), ("d", args.d)):
        if val is not None:
            WORKLOAD[key] = val
    if args.chunk is not None or args.tokens is not None or args.d is not None or args.objective != "sft":
        tag = {"sft": "sft_ce", "grpo": "grpo_clip", "dpo": "dpo_two_pass"}[args.objective]
        WORKLOAD["workload"] = (f"{tag}_lmhead_bf16_T{WORKLOAD['T']}_d{WORKLOAD['d']}_V{WORKLOAD['V']}"
                                f"_chunk{WORKLOAD['chunk']}")
    if args.warmup < 3 and args.impl == "ours":
        args.warmup = 3
    # the other workloads' lines ride along with the main line of a plain invocation only
    args.other_workloads = (not args.no_other_workloads and args.workload == "main" and args.objective == "sft"
                            and args.sublayer == "lmhead" and args.comparator is None and args.chunk is None
                            and args.tokens is None and args.d is None and not args.lean)
    if args.impl == "reference":
        return run_reference(args)
    if args.comparator == "torch":
        return run_torch_comparator(args)
    if args.sublayer == "mlp":
        return run_mlp_bench(args)
    if args.sublayer == "attn":
        return run_attn_bench(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
