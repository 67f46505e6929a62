"""CPU-only: the multi-rank path of bench.py (one replica per rank, barrier,
max of the ranks' times, whole-job throughput) on two gloo ranks."""

import os
import socket
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        bench.barrier(world)
        mine = 1.5 + rank          # rank 1 is the slower one
        slowest = bench.max_over_ranks(mine, world, torch.device("cpu"))
        value = bench.whole_job_tokens_per_s(4096, world, slowest)
        bench.barrier(world)
        q.put((rank, slowest, value))
    finally:
        dist.destroy_process_group()


def test_two_rank_timing_uses_the_slowest_rank():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=5) for _ in range(2))
    for rank, slowest, value in got:
        assert slowest == 2.5
        assert value == pytest.approx(2 * 4096 * 1000.0 / 2.5)


def test_reference_arm_other_ranks_print_nothing(capsys):
    sys.path.insert(0, ROOT)
    import bench

    class A:
        config, rows, steps, warmup, gpus = "tiny", 8, 1, 0, 2
    bench.run_reference(A, 2, 1)      # rank 1 of 2: exits without work
    assert capsys.readouterr().out == ""


def test_reference_arm_rank0_line(capsys):
    """Rank 0 of the reference arm prints one JSON line: the oracle on every
    host core, with the contract's keys."""
    import json
    sys.path.insert(0, ROOT)
    import bench

    class A:
        config, rows, steps, warmup, gpus = "tiny", 64, 1, 0, 1
    bench.run_reference(A, 1, 0)
    out = capsys.readouterr().out.strip().splitlines()
    assert len(out) == 1
    d = json.loads(out[0])
    assert d["impl"] == "reference" and d["value"] > 0 and d["higher_is_better"] is True
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"]
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0
    # the same config keys as the GPU arm's line (workload_desc + parallelism)
    assert d["config"]["parallelism"] == "single GPU"
    for k in ("workload", "N", "V", "active_rows", "temperature", "l2"):
        assert k in d["config"]


def test_cpu_baseline_all_cores_runs_every_thread():
    sys.path.insert(0, ROOT)
    import bench
    from vocab_selected_token_gb300 import workloads as W
    inp = W.make_logits_inputs("tiny", device="cpu", N=64)
    v, rows, secs, cores = bench.oracle_rows_per_second_all_cores(inp, 0.2, rows_per_thread=4)
    assert cores >= 1 and rows >= 4 * cores and v > 0 and secs >= 0.2


def test_fused_timing_builds_each_workload_at_its_own_size(monkeypatch):
    """time_fused builds every workload with its recipe's own row count (or
    the one override it is given), not with the row count of the workload
    timed before it."""
    sys.path.insert(0, ROOT)
    import bench
    from vocab_selected_token_gb300 import _lib
    from vocab_selected_token_gb300 import workloads as W

    seen = []

    class Stop(Exception):
        pass

    def fake(name, device="cpu", N=None, V=None, seed=None):
        seen.append((name, N))
        if len(seen) == 3:
            raise Stop()
        x = torch.zeros((W.WORKLOADS[name]["N"] if N is None else N, 8), dtype=torch.bfloat16)
        return W.LogitsInputs(x=x, t=torch.zeros(x.shape[0], dtype=torch.int32), mask=None,
                              T=1.0, g=torch.zeros(x.shape[0]), name=name)

    class FakeLib:
        def slp_forward_backward(self, *a):
            return 0

    monkeypatch.setattr(W, "make_logits_inputs", fake)
    monkeypatch.setattr(_lib, "load", lambda: FakeLib())
    monkeypatch.setattr(torch.cuda, "synchronize", lambda *a, **k: None)

    class Ev:
        def __init__(self, **k):
            pass

        def record(self, *a):
            pass

        def elapsed_time(self, other):
            return 1.0

    class St:
        cuda_stream = 0

    monkeypatch.setattr(torch.cuda, "Event", Ev)
    monkeypatch.setattr(torch.cuda, "current_stream", lambda *a: St())
    monkeypatch.setattr(torch.cuda, "empty_cache", lambda: None)
    with pytest.raises(Stop):
        bench.time_fused(torch.device("cpu"), 1.0, steps=1, warmup=1)
    assert seen == [("c151k", None), ("packed", None), ("stability", None)]
    seen.clear()
    with pytest.raises(Stop):
        bench.time_fused(torch.device("cpu"), 1.0, steps=1, warmup=1,
                         names=("c151k", "packed", "stability"), rows=7, vocab=None)
    assert seen == [("c151k", 7), ("packed", 7), ("stability", 7)]


def test_code_hash_ignores_comments_only():
    """The DRAM-traffic record is keyed on the kernels' code: comments and
    blank lines do not change the hash, code and string contents do."""
    sys.path.insert(0, ROOT)
    import bench
    a = 'int f() { return 1; }  // one\n/* block\n comment */\nconst char* s = "x//y";\n'
    b = '// header\nint f() { return 1; }\n\n\nconst char* s = "x//y";   \n'
    c = 'int f() { return 2; }\nconst char* s = "x//y";\n'
    d = 'int f() { return 1; }\nconst char* s = "x/y";\n'
    assert bench.code_text(a) == bench.code_text(b)
    assert bench.code_text(a) != bench.code_text(c)
    assert bench.code_text(a) != bench.code_text(d)
