"""Seeded synthetic inputs for the LM-head workloads.

This module only draws random numbers and rounds them to the storage dtype. It holds
none of the method's arithmetic (no logits, no softmax, no gradients), so both the
CUDA path and the CPU oracle can take their inputs from it.

Recipe (numpy PCG64, one independent stream per quantity):
  H ~ N(0, 1), W ~ N(0, 0.02^2), drawn in float32 then rounded to bfloat16
  (round-to-nearest-even) for the bf16 workloads; labels ~ U[0, V) int32;
  ignored positions set to ``ignore_index`` by one of three masks:
    - "frac":    exactly floor(frac * T) positions, chosen by a permutation,
    - "prefix":  the first ``n`` positions of the whole batch,
    - "seqhead": the first ``n`` positions of every sequence.
  GRPO advantages A ~ N(0, 1) per response, broadcast to its tokens; the noise
  added to the old log-probs ~ N(0, 0.1^2); DPO reference sequence log-probs
  ~ N(-2000, 50^2), float64.

Peaked (confident-token) inputs, ``make_peaked``: W ~ N(0, (sigma_z / sqrt(d))^2) so that
a row's logits spread with standard deviation about sigma_z, and every row of H is
nudged towards its label's row of W, H_t += a_t W_{y_t} / (w_std^2 d) with a_t ~ U[lo, hi],
which raises the label's logit by about a_t while moving the others by about
a_t / sqrt(d).  With a_t well above the largest of V Gaussian logits most tokens are
predicted with probability close to 1, the regime of a trained language-model head.
The nudge is applied to the float32 draws, then both matrices are rounded.
"""
from __future__ import annotations

import numpy as np

IGNORE_INDEX = -100

# one stream id per quantity so that changing one shape never shifts another draw
_STREAM = {"H": 1, "W": 2, "labels": 3, "mask": 4, "adv": 5, "noise": 6, "ref": 7, "rows": 8, "lift": 9}


def rng_for(seed: int, what: str) -> np.random.Generator:
    return np.random.default_rng(np.random.SeedSequence([int(seed), _STREAM[what]]))


def round_bf16(x: np.ndarray) -> np.ndarray:
    """Round float32 values to the nearest bfloat16 (ties to even); returns float32."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    u = x.view(np.uint32)
    u = (u + np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))) & np.uint32(0xFFFF0000)
    return u.view(np.float32)


def _normal(seed: int, what: str, shape, std: float, bf16: bool, block_rows: int = 8192) -> np.ndarray:
    """float32 normal draws, generated in row blocks (one child stream per block) so
    that very large matrices are drawn with bounded temporary memory."""
    rows = shape[0]
    out = np.empty(shape, dtype=np.float32)
    nblk = max(1, (rows + block_rows - 1) // block_rows)
    children = np.random.SeedSequence([int(seed), _STREAM[what]]).spawn(nblk)
    for b in range(nblk):
        r0, r1 = b * block_rows, min(rows, (b + 1) * block_rows)
        g = np.random.default_rng(children[b])
        blk = g.standard_normal((r1 - r0,) + tuple(shape[1:]), dtype=np.float32)
        if std != 1.0:
            blk *= np.float32(std)
        out[r0:r1] = round_bf16(blk) if bf16 else blk
    return out


def make_hw(T: int, d: int, V: int, seed: int, dtype: str, w_std: float = 0.02):
    """H [T, d] ~ N(0, 1) and W [V, d] ~ N(0, w_std^2) as float32 arrays holding values
    exact in ``dtype``."""
    if dtype not in ("bf16", "fp32"):
        raise ValueError(dtype)
    H = _normal(seed, "H", (T, d), 1.0, dtype == "bf16")
    W = _normal(seed, "W", (V, d), w_std, dtype == "bf16")
    return H, W


def make_peaked(T: int, d: int, V: int, seed: int, dtype: str, sigma_z: float, lift_lo: float,
                lift_hi: float, frac: float = 0.1, copies=(), labels=None):
    """H [T, d], W [V, d] and labels [T] of the confident-token regime (see the module
    docstring): the label's logit lifted by a_t ~ U[lift_lo, lift_hi] above a N(0,
    sigma_z^2) background, ``frac`` of the tokens ignored by a permutation mask.

    ``copies``: pairs (dst, src) of vocabulary rows; row dst of W becomes an exact copy of
    row src before anything else, so the two logits are equal in every row.  ``labels``:
    [T] labels to use (before the ignore mask) instead of the uniform draw."""
    if dtype not in ("bf16", "fp32"):
        raise ValueError(dtype)
    w_std = sigma_z / np.sqrt(d)
    H = _normal(seed, "H", (T, d), 1.0, False)
    W = _normal(seed, "W", (V, d), w_std, False)
    for dst, src in copies:
        W[dst] = W[src]
    y = make_labels(T, V, seed, "frac" if frac > 0 else "none", frac)
    lab = rng_for(seed, "labels").integers(0, V, size=T, dtype=np.int64)   # the labels before masking
    if labels is not None:
        lab = np.asarray(labels, dtype=np.int64)
        y = np.where(y == IGNORE_INDEX, y, lab).astype(np.int32)
    a = rng_for(seed, "lift").uniform(lift_lo, lift_hi, size=T).astype(np.float32)
    H += (a / np.float32(w_std * w_std * d))[:, None] * W[lab]
    if dtype == "bf16":
        H, W = round_bf16(H), round_bf16(W)
    return H, W, y


def make_labels(T: int, V: int, seed: int, mask: str = "none", frac: float = 0.0,
                n: int = 0, seq_len: int = 0, ignore_index: int = IGNORE_INDEX) -> np.ndarray:
    y = rng_for(seed, "labels").integers(0, V, size=T, dtype=np.int64).astype(np.int32)
    if mask == "frac":
        k = int(np.floor(frac * T))
        pos = rng_for(seed, "mask").permutation(T)[:k]
        y[pos] = ignore_index
    elif mask == "prefix":
        y[: min(n, T)] = ignore_index
    elif mask == "seqhead":
        for s in range(0, T, seq_len):
            y[s: s + min(n, seq_len)] = ignore_index
    elif mask != "none":
        raise ValueError(mask)
    return y


def make_advantages(n_resp: int, resp_len: int, seed: int) -> np.ndarray:
    a = rng_for(seed, "adv").standard_normal(n_resp).astype(np.float32)
    return np.repeat(a, resp_len)


def make_logp_noise(T: int, seed: int, std: float = 0.1) -> np.ndarray:
    return (rng_for(seed, "noise").standard_normal(T) * std).astype(np.float64)


def make_ref_seq_logp(n_seq: int, seed: int, mean: float = -2000.0, std: float = 50.0) -> np.ndarray:
    return mean + std * rng_for(seed, "ref").standard_normal(n_seq)


def sample_rows(T: int, k: int, seed: int) -> np.ndarray:
    k = min(k, T)
    return np.sort(rng_for(seed, "rows").choice(T, size=k, replace=False))


def cu_seqlens(n_seq: int, seq_len: int) -> np.ndarray:
    return (np.arange(n_seq + 1, dtype=np.int64) * seq_len).astype(np.int32)


# Workloads.  Seeds are 1000 + the workload's index.
WORKLOADS = {
    "sft_fp32_T256_d64_V1000": dict(
        objective="sft", T=256, d=64, V=1000, chunks=(64,), dtype="fp32", seed=1000,
        mask="frac", frac=0.1),
    "sft_bf16_T8192_d2560_V151936": dict(
        objective="sft", T=8192, d=2560, V=151936, chunks=(512, 1024, 2048), dtype="bf16",
        seed=1001, mask="prefix", n=1024),
    "grpo_bf16_8x2048_d4096_V151936": dict(
        objective="grpo", T=16384, d=4096, V=151936, chunks=(2048,), dtype="bf16", seed=1002,
        mask="frac", frac=0.1, n_resp=8, resp_len=2048),
    "dpo_bf16_8x4096_d4096_V151936": dict(
        objective="dpo", T=32768, d=4096, V=151936, chunks=(2048,), dtype="bf16", seed=1003,
        mask="seqhead", n=1024, n_seq=8, seq_len=4096, beta=0.1),
    "sft_bf16_T65536_d5120_V151936": dict(
        objective="sft", T=65536, d=5120, V=151936, chunks=(512, 1024, 2048, 4096, 8192),
        dtype="bf16", seed=1004, mask="frac", frac=0.05),
}


def make_workload(name: str, T: int | None = None):
    """All inputs of a named workload (optionally truncated to the first T tokens)."""
    w = WORKLOADS[name]
    T = w["T"] if T is None else T
    H, W = make_hw(T, w["d"], w["V"], w["seed"], w["dtype"])
    seq_len = w.get("seq_len", 0)
    y = make_labels(T, w["V"], w["seed"], w["mask"], w.get("frac", 0.0), w.get("n", 0), seq_len)
    out = dict(H=H, W=W, labels=y)
    if w["objective"] == "grpo":
        out["advantages"] = make_advantages(w["n_resp"], w["resp_len"], w["seed"])[:T]
        out["logp_noise"] = make_logp_noise(T, w["seed"])
    if w["objective"] == "dpo":
        out["cu_seqlens"] = cu_seqlens(w["n_seq"], w["seq_len"])
        out["ref_seq_logp"] = make_ref_seq_logp(w["n_seq"], w["seed"])
    return out
