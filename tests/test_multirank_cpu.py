"""The N > 1 host paths of the benchmark, on CPU.

Batch-1 decode runs as independent replicas, one per GPU, so ranks exchange only the
timing: the slowest rank's time (a MAX all-reduce) and the whole-job rate over all
ranks' units.  Here two gloo ranks run that reduction, and the reference arm runs under
torchrun with two processes: only rank 0 works and prints its single JSON line.

The batched workload partitions its streams over the ranks (each stream is an
independent decoder, "Qwen3-TTS ncnn port", section "Talker: non-standard structure and
two-level generation"): two gloo ranks each decode their slice of a small batched
workload with the oracle, and the slices put back together equal one rank decoding
every stream.
"""
import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    ms = bench.max_over_ranks(10.0 * (rank + 1), world)
    rate = bench.whole_job_rate(100, world, ms)
    with open(os.path.join(out_dir, f"r{rank}.json"), "w") as f:
        json.dump({"ms": ms, "rate": rate}, f)
    dist.barrier()
    dist.destroy_process_group()


def test_max_over_ranks_and_whole_job_rate_with_two_gloo_ranks(tmp_path):
    import torch.multiprocessing as mp
    port = _free_port()
    mp.start_processes(_rank_main, args=(2, port, str(tmp_path)), nprocs=2, join=True, start_method="spawn")
    got = [json.load(open(tmp_path / f"r{r}.json")) for r in range(2)]
    assert all(g["ms"] == 20.0 for g in got)                 # both ranks see the slowest rank's time
    assert all(g["rate"] == pytest.approx(2 * 100 / 0.020) for g in got)


def test_single_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(12.5, 1) == 12.5
    assert bench.whole_job_rate(300, 1, 50.0) == pytest.approx(6000.0)


def test_reference_arm_under_torchrun_prints_one_line_from_rank_0():
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), "bench.py", "--impl", "reference",
           "--workload", "tiny", "--steps", "2", "--warmup", "1"]
    env = dict(os.environ, OMP_NUM_THREADS="2")
    r = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-3000:]
    lines = [json.loads(x) for x in r.stdout.splitlines() if x.startswith("{")]
    assert len(lines) == 1, r.stdout
    line = lines[0]
    assert line["impl"] == "reference" and line["n_gpus"] == 2 and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle"


def _small_batch():
    import workloads as W
    s = W.scaled(W.TALKER, name="talker_kv", hidden=128, n_layers=2, n_q_heads=4, n_kv_heads=2, head_dim=32,
                 ffn=256, vocab=96, embed_rows=96, buckets=(32, 64), prefill=20)
    n = 5                                                       # not a multiple of the ranks
    lens = W.uniform_int("multirank/L0", n, 3, 40)
    toks = W.batch_first_tokens(n, s.vocab)
    return s, n, lens, toks


def _decode_streams(streams, steps=6):
    """The oracle's greedy ids of the given streams of the small batched workload."""
    import oracle as O
    import workloads as W
    s, _, lens, toks = _small_batch()
    w = W.model_weights(s)
    out = {}
    for b in streams:
        o = O.Oracle(s, w)
        o.set_kv(W.batch_stream_kv(s, b, int(lens[b])), int(lens[b]))
        tok, ids = int(toks[b]), []
        for _ in range(steps):
            tok, _, _, _ = o.step(token=tok, want_logits=False)
            ids.append(int(tok))
        o.close()
        out[b] = ids
    return out


def _shard_rank_main(rank, world, port, out_dir):
    sys.path.insert(0, ROOT)
    sys.path.insert(0, os.path.join(ROOT, "tests"))
    os.environ["OMP_NUM_THREADS"] = "1"
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    _, n, _, _ = _small_batch()
    lo, hi = bench.stream_shard(n, rank, world)
    mine = _decode_streams(range(lo, hi))
    parts = [None] * world
    dist.all_gather_object(parts, {"lo": lo, "hi": hi, "ids": mine})
    if rank == 0:
        with open(os.path.join(out_dir, "shards.json"), "w") as f:
            json.dump(parts, f)
    dist.barrier()
    dist.destroy_process_group()


def test_stream_shards_cover_every_stream_once():
    sys.path.insert(0, ROOT)
    import bench
    for n in (1, 5, 64):
        for ws in (1, 2, 3, 4, 8):
            got = [bench.stream_shard(n, r, ws) for r in range(ws)]
            assert got[0][0] == 0 and got[-1][1] == n
            assert all(got[r][1] == got[r + 1][0] for r in range(ws - 1))
            assert max(h - l for l, h in got) - min(h - l for l, h in got) <= 1


def test_batched_streams_partitioned_over_two_gloo_ranks_equal_one_rank(tmp_path):
    import torch.multiprocessing as mp
    port = _free_port()
    mp.start_processes(_shard_rank_main, args=(2, port, str(tmp_path)), nprocs=2, join=True, start_method="spawn")
    parts = json.load(open(tmp_path / "shards.json"))
    _, n, _, _ = _small_batch()
    assert [p["lo"] for p in parts] == [0, parts[0]["hi"]] and parts[-1]["hi"] == n
    joined = {int(k): v for p in parts for k, v in p["ids"].items()}
    assert sorted(joined) == list(range(n))
    assert joined == _decode_streams(range(n))
