"""The multi-rank bench path on CPU: world size 2 over gloo.

Every rank runs its own batch (weak scaling, no collective on the data path); the
bench reports whole-job tokens (sum over ranks) over the step time (max over ranks).
"""
import os
import socket
import sys

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    r, w, lr = bench.dist_env()
    tokens, ms = bench.aggregate(torch, dist, 1000.0 * (rank + 1), 10.0 + 5.0 * rank, "cpu")
    # per-rank inputs differ (seed + rank) but have the same shape
    from memory_efficient_exact_gb300 import inputs as I
    y = I.make_labels(64, 100, 1002 + rank, "frac", 0.1)
    q.put((rank, r, w, tokens, ms, int((y == -100).sum()), y[:8].tolist()))
    dist.destroy_process_group()


def test_two_rank_aggregation_over_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, r, w, tokens, ms, n_ign, head in res:
        assert r == rank and w == 2
        assert tokens == 3000.0          # sum over ranks
        assert ms == 15.0                # max over ranks
        assert n_ign == 6                # floor(0.1 * 64) on every rank
    assert res[0][6] != res[1][6]        # each rank draws its own batch


def _args_of(argv):
    """The workload bench.main() would run for argv (the run is replaced by a recorder)."""
    import importlib.util
    spec = importlib.util.spec_from_file_location("bench_args_probe", os.path.join(ROOT, "bench.py"))
    b = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(b)
    seen = {}

    def rec(args):
        seen.update(dict(b.WORKLOAD), chunk_arg=args.chunk, sublayer=args.sublayer,
                    other=getattr(args, "other_workloads", None), others=list(b.OTHER_WORKLOADS))
        return 0
    b.run_ours = b.run_mlp_bench = b.run_attn_bench = rec
    b.run_reference = rec
    assert b.main(argv) == 0
    return seen


def test_other_workloads_ride_only_with_the_plain_invocation():
    # the plain invocation folds the other workloads' lines into its own; any flag that
    # picks another workload, schedule or sublayer measures that one alone
    assert _args_of([])["other"] is True and _args_of(["--steps", "2"])["other"] is True
    for argv in (["--no-other-workloads"], ["--chunk", "2048"], ["--objective", "grpo"], ["--workload", "profile"],
                 ["--lean"], ["--sublayer", "mlp"], ["--tokens", "8192"]):
        assert _args_of(argv)["other"] is False, argv
    others = _args_of([])["others"]
    names = [n for n, _ in others]
    assert len(set(names)) == len(names) and len(names) == 11
    # each folded line's name carries the chunk its command runs
    for name, argv in others:
        if name.startswith(("grpo", "dpo", "sft")):
            assert name.endswith(f"_chunk{_args_of(argv)['chunk']}"), (name, argv)


def test_bench_workload_selection():
    # default: the SFT workload the metric is quoted on
    w = _args_of([])
    assert (w["T"], w["d"], w["V"], w["chunk"], w["objective"]) == (16384, 4096, 151936, 4096, "sft")
    assert w["workload"] == "sft_ce_lmhead_bf16_T16384_d4096_V151936_chunk4096"
    # the two chunk-sweep workloads keep their sizes and label masks
    w = _args_of(["--workload", "sft_T8192_d2560", "--chunk", "512"])
    assert (w["T"], w["d"], w["chunk"], w["mask"], w["n"]) == (8192, 2560, 512, "prefix", 1024)
    assert w["workload"] == "sft_ce_lmhead_bf16_T8192_d2560_V151936_chunk512"
    w = _args_of(["--workload", "sft_T65536_d5120"])
    assert (w["T"], w["d"], w["chunk"], w["mask"], w["frac"]) == (65536, 5120, 4096, "frac", 0.05)
    # DPO defaults to 8 sequences of 4096 tokens, GRPO to 8 x 2048, both at chunk 2048
    assert (_args_of(["--objective", "dpo"])["T"], _args_of(["--objective", "dpo"])["chunk"]) == (32768, 2048)
    assert (_args_of(["--objective", "grpo"])["T"], _args_of(["--objective", "grpo"])["chunk"]) == (16384, 2048)
    w = _args_of(["--objective", "grpo", "--chunk", "4096"])
    assert w["chunk"] == 4096 and w["workload"] == "grpo_clip_lmhead_bf16_T16384_d4096_V151936_chunk4096"
    # the profile case for ncu captures
    w = _args_of(["--workload", "profile"])
    assert (w["T"], w["V"], w["chunk"]) == (8192, 32768, 4096)
    assert _args_of(["--sublayer", "attn"])["sublayer"] == "attn"


def test_attention_pair_counts():
    """The attention line's FLOP accounting: causal pairs T (T + 1) / 2 whatever the chunk;
    chunk rectangles (n + 1) / n times that, n = T / chunk, when the chunk divides T (the
    chunks' sum of c (i + 1) c over i < n), and equal to the full square for one chunk."""
    import importlib.util
    spec = importlib.util.spec_from_file_location("bench_pairs_probe", os.path.join(ROOT, "bench.py"))
    b = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(b)
    for T, chunk in ((8192, 1024), (8192, 4096), (4096, 4096), (32768, 4096)):
        causal, rect = b.attn_pairs(T, chunk)
        n = T // chunk
        assert causal == T * (T + 1) // 2
        assert rect == chunk * chunk * n * (n + 1) // 2
    assert b.attn_pairs(8192, 8192)[1] == 8192 * 8192
    # a ragged last chunk: chunks of 3 over T = 7 -> rows 3, 3, 1 reading keys 3, 6, 7
    assert b.attn_pairs(7, 3) == (28, 3 * 3 + 3 * 6 + 1 * 7)
    # brute force on a small case: the causal pairs q >= k, counted one by one
    assert b.attn_pairs(37, 5)[0] == sum(1 for q in range(37) for k in range(q + 1))
