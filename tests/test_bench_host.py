"""bench.py host logic on CPU: the multi-rank aggregation (gloo ranks stand
in for GPU ranks: every rank runs an independent replica, the job's time is
the slowest rank's and its throughput counts every rank's tokens) and the
reference arm's JSON line, alone and under torchrun with two ranks."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, times, out):
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms = bench.max_over_ranks(times[rank], "cpu")
        rate = bench.whole_job_rate(4, 10, world, ms)
        out.put((rank, ms, rate))
    finally:
        dist.destroy_process_group()


def test_slowest_rank_sets_the_time_and_every_rank_counts():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    times = [12.5, 20.0]
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, times, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, ms, rate in res:
        assert ms == 20.0                                   # max over ranks, on every rank
        assert rate == pytest.approx(4 * 10 * 2 / 20e-3)    # all ranks' tokens / slowest time


def test_single_rank_is_unchanged():
    assert bench.max_over_ranks(7.0) == 7.0
    assert bench.whole_job_rate(1, 1000, 1, 80.0) == pytest.approx(12500.0)


def _json_lines(out: str):
    return [json.loads(l) for l in out.splitlines() if l.startswith("{")]


def test_reference_arm_prints_one_line():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--config", "tiny-fp32", "--steps", "3", "--warmup", "1"],
                       capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = _json_lines(r.stdout)
    assert len(lines) == 1
    j = lines[0]
    assert j["impl"] == "reference" and j["unit"] == "tokens/s" and j["value"] > 0
    assert j["metric"] == bench.METRIC and j["higher_is_better"] is True
    assert j["cpu_baseline"]["kind"] == "oracle" and j["cpu_baseline"]["cores"] >= 1
    assert j["e2e"] == {"value": j["value"], "unit": "tokens/s", "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}


def test_reference_arm_under_torchrun_prints_on_rank_zero_only():
    r = subprocess.run([sys.executable, "-m", "torch.distributed.run", "--nnodes=1",
                        "--nproc-per-node", "2", "--master-addr", "127.0.0.1",
                        "--master-port", str(_free_port()),
                        os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2",
                        "--config", "tiny-fp32", "--steps", "2", "--warmup", "1"],
                       capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = _json_lines(r.stdout)
    assert len(lines) == 1 and lines[0]["impl"] == "reference" and lines[0]["n_gpus"] == 2


def test_work_model_matches_closed_forms():
    """The roofline numerators at DeepSeek-V2 widths (d = 5120, 128 heads of
    128, d_c = 512, d_R = 64): weight bytes read once, one 576-wide bf16 row
    per cached token, 2 FLOP per multiply-add."""
    from synth import workloads as W
    k, tot_bytes, tot_flops, cache_bytes = bench.work_model(W.config("b1-l4096"))
    assert k["out_proj"][0] == 5120 * 16384 * 2 + 16384 * 2 + 5120 * 2   # W_O + o + u
    assert k["out_proj"][1] == 2 * 5120 * 16384
    assert k["compress_append"][0] == 576 * 5120 * 2 + 5120 * 2 + 576 * 2
    assert k["absorb_q"][1] == 2 * 128 * 128 * 512
    assert cache_bytes == 4096 * 576 * 2
    # attention: every query token sees its 4096 rows; S over 576 features
    # and O over 512 latent columns for each of 128 heads
    assert k["attend"][1] == 2 * 4096 * 128 * (576 + 512)
    assert k["append_absorb"] == tuple(a + b for a, b in zip(k["compress_append"], k["absorb_q"]))
    weights = (576 * 5120 + 128 * 128 * 512 + 128 * 128 * 512 + 5120 * 16384) * 2
    assert tot_bytes == weights + cache_bytes + (5120 + 128 * 192 + 5120) * 2
    # causal T = 2: the first new token does not see the second
    k2, _, _, _ = bench.work_model(W.config("b128-l16k-t2"))
    vis = sum(2 * S - 1 for S in W.config("b128-l16k-t2").seq_lens)
    assert k2["attend"][1] == 2 * vis * 128 * (576 + 512)


def test_work_model_query_path():
    """With the query path the step reads W^DQ [1536, 5120], W^UQ [16384,
    1536] and W^QR [8192, 5120] instead of taking the queries as input."""
    from synth import workloads as W
    wl = W.config("b1-l4096")
    _, b0, f0, _ = bench.work_model(wl)
    k, b1, f1, _ = bench.work_model(wl, query_path=True)
    assert k["query_down"][1] == 2 * 1536 * 5120
    assert k["query_up"][1] == 2 * 16384 * 1536
    assert k["query_rope"][1] == 2 * 8192 * 5120
    assert b1 - b0 == (1536 * 5120 + 16384 * 1536 + 8192 * 5120) * 2 - 128 * 192 * 2
    assert f1 - f0 == 2 * (1536 * 5120 + 16384 * 1536 + 8192 * 5120)


def test_work_model_layer_stack():
    """A stack reads every layer's weights and cache once per step, plus the
    residual's h and u reads and h write."""
    import dataclasses
    from synth import workloads as W
    one = dataclasses.replace(W.config("b1-l4096-x60"), layers=1)
    _, b1, f1, c1 = bench.work_model(one, query_path=True)
    k, b60, f60, c60 = bench.work_model(W.config("b1-l4096-x60"), query_path=True)
    assert k["residual"] == (3 * 5120 * 2, 5120.0)
    assert b60 == 60 * (b1 + 3 * 5120 * 2)
    assert f60 == 60 * (f1 + 5120)
    assert c60 == 60 * c1 == 60 * 4096 * 576 * 2


def test_work_model_prefill_explicit():
    """The explicit prefill form: K^C and V of every cached row up-projected
    once (2 * 512 * 16384 FLOP each), 2 * (192 + 128) FLOP per head and
    visible (query, key) pair, and the causal count T (T + 1) / 2 for a chunk
    with an empty prefix."""
    from synth import workloads as W
    wl = W.config("prefill-b4-t4096")
    k, b, f, c = bench.work_model(wl, form="explicit")
    n = 4 * 4096
    assert k["key_up"][1] == k["value_up"][1] == 2 * n * 16384 * 512
    assert k["prefill_attend"][1] == 2 * (4 * 4096 * 4097 // 2) * 128 * (192 + 128)
    assert k["gather"][0] == 2 * n * 576 * 2
    assert f == sum(k[x][1] for x in ("compress_append", "key_up", "value_up", "prefill_attend",
                                      "out_proj"))
    assert c == n * 576 * 2
    # the same chunk in the absorbed form: 2 * (576 + 512) FLOP per pair
    ka, _, fa, _ = bench.work_model(wl)
    assert ka["attend"][1] == 2 * (4 * 4096 * 4097 // 2) * 128 * (576 + 512)
    assert fa > f
