"""The benchmark's multi-replica logic on CPU: two gloo ranks (world size 2).

The path has no data exchange (every (sequence, KV head) is independent), so
several GPUs run independent replicas; what the ranks share is the timing
reduction (the slowest replica sets the job time), the per-rank seeds and the
rank-0-only output of the reference arm."""
import os
import subprocess
import sys

import numpy as np
import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)


def _rank_main(rank, world, port, out):
    import torch
    import torch.distributed as dist
    import bench
    from sparse_attention_decode_pages_gb300 import workloads as wl
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        local = [1.0 + rank, 5.0 - rank, 2.5 * (rank + 1)]
        got = bench.max_over_ranks(local, world, torch.device("cpu"))
        spec = wl.spec("tiny")
        spec.seed = bench.replica_seed(spec.seed, rank)
        w = wl.make(spec)
        qsum = float(np.asarray(w.q, dtype=np.float64).sum())
        dist.barrier()
        out.put((rank, got, spec.seed, qsum, bench.job_tokens_per_s(world, w.B, got[0])))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_reduce_timings_and_use_distinct_batches():
    world, port = 2, 29500 + os.getpid() % 1000
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = dict((r, (g, s, qs, v)) for r, g, s, qs, v in (q.get(timeout=120) for _ in range(world)))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    # every rank sees the maximum over ranks of each timing
    assert res[0][0] == res[1][0] == [2.0, 5.0, 5.0]
    # replicas draw different batches from different seeds
    assert res[0][1] != res[1][1] and res[0][2] != res[1][2]
    # the job's throughput counts both replicas' batches over the slowest time
    assert res[0][3] == pytest.approx(2 * 2 / 2.0e-3)


def test_reference_arm_prints_on_rank_zero_only():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "3", "--config", "tiny"], env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0 and r.stdout.strip() == ""


def test_reference_arm_line_on_rank_zero():
    import json
    env = dict(os.environ, RANK="0", WORLD_SIZE="1", LOCAL_RANK="0")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "2",
                        "--warmup", "3", "--config", "tiny"], env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-500:]
    line = json.loads(r.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["value"] > 0 and line["cpu_baseline"]["kind"] == "oracle"
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["higher_is_better"] is True


def test_staged_inputs_are_views_of_one_buffer():
    """The benchmark's e2e copies a step's inputs in one transfer: staged() packs the
    tensors at 256-byte offsets of one buffer, as views with their shapes, dtypes and
    values."""
    import torch
    import bench
    ts = [torch.arange(10, dtype=torch.int32), torch.randn(3, 5).to(torch.bfloat16),
          torch.ones(70, dtype=torch.float32), torch.arange(6, dtype=torch.int32).reshape(2, 3)]
    buf, views = bench.staged(torch, "cpu", ts)
    assert buf.dtype == torch.uint8 and buf.numel() == 256 + 256 + 512 + 256
    base = buf.data_ptr()
    for t, v in zip(ts, views):
        assert v.dtype == t.dtype and v.shape == t.shape and torch.equal(v, t)
        assert (v.data_ptr() - base) % 256 == 0
    views[0].fill_(7)  # a view: writes land in the buffer
    assert torch.equal(buf[:40].view(torch.int32), torch.full((10,), 7, dtype=torch.int32))


def test_gpus_flag_runs_replicas_under_a_launcher():
    """`bench.py --gpus 2` without a launcher re-runs itself under torch.distributed.run
    with two processes: here the reference arm, so rank 0 alone prints one line."""
    import json
    env = {k: v for k, v in os.environ.items() if k not in ("RANK", "WORLD_SIZE", "LOCAL_RANK")}
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--gpus", "2", "--impl", "reference",
                        "--steps", "1", "--warmup", "3", "--config", "tiny"], env=env, capture_output=True,
                       text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-800:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    assert json.loads(lines[0])["n_gpus"] == 2


def test_replica_launch_command():
    import bench
    cmd = bench.replica_launch_cmd(["--gpus", "4", "--steps", "3"], 4, 12345)
    assert cmd[1:4] == ["-m", "torch.distributed.run", "--nnodes=1"] and "--nproc-per-node=4" in cmd
    assert cmd[cmd.index("--master-addr") + 1] == "127.0.0.1" and cmd[cmd.index("--master-port") + 1] == "12345"
    assert cmd[-4:] == ["--gpus", "4", "--steps", "3"]


def test_retrieval_recall_and_byte_breakdown():
    """Recall counts, per KV head, the planted tokens whose page is selected; the step's
    algorithmic bytes are the sum of their parts, with a summary read per page."""
    import bench
    from sparse_attention_decode_pages_gb300 import workloads as wl
    w = wl.named("q17b", B=2, len_lo=600, len_hi=900, threads=2)
    assert all(len(p) == 8 for p in w.planted)
    ps = w.page_size
    sel = np.full((w.B, w.H_kv, 4), -1, np.int32)
    nsel = np.zeros((w.B, w.H_kv), np.int32)
    pos = w.planted[0][0] // ps
    sel[0, :, 0] = pos                       # every head of sequence 0 keeps one planted page
    nsel[0, :] = 1
    want = sum(1 for t in w.planted[0] if t // ps == pos) * w.H_kv / (8 * w.B * w.H_kv)
    assert bench.retrieval_recall(w, sel, nsel) == pytest.approx(want)
    chosen = [[[0, w.pages(b) - 1] for _ in range(w.H_kv)] for b in range(w.B)]
    nb = bench.algorithmic_bytes(w, chosen)
    assert nb["step"] == nb["selected_kv"] + nb["summaries"] + nb["q_o_lse"] + nb["append"]
    assert nb["summaries"] == sum(w.pages(b) for b in range(w.B)) * w.H_kv * 4 * w.D
    full_last = [min(ps, int(w.seq_lens[b]) - (w.pages(b) - 1) * ps) for b in range(w.B)]
    assert nb["selected_kv"] == sum((ps + full_last[b]) * w.H_kv * 4 * w.D for b in range(w.B))
